"""GPU parity of the backward (attention.fkc.md, "attention_flash_backward")
against the float64 oracle ``oracle.attn_bwd`` on the same 16-bit inputs.

Bar, per gradient tensor X in (dQ, dK, dV), with s = max(1, max |X_oracle|):
    max |X_gpu - X_oracle| <= 2e-2 s   and   mean |X_gpu - X_oracle| <= 2e-3 s.
For gradients of order one this is the forward's 16-bit bar; above that it
grows with the tensor, because the kernel's own error is relative: P and dS
enter the tensor cores as 16-bit values (relative rounding 2^-9 for bf16),
Delta = dO . O is taken from the forward's 16-bit output, and the result is
rounded to 16 bits (half an ulp, 2^-9 relative).  Rows with no admissible key
have exactly zero dQ on both sides.  Reruns are bitwise identical (no atomics).

fp32 inputs run the SIMT path in fp32 throughout; its bar is that of the fp32
forward, relative the same way: max |err| <= 1e-4 s and mean |err| <= 1e-5 s.
"""
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu
BF16 = torch.bfloat16


def _inputs(B, Hq, Hkv, Sq, Sk, D, seed, dtype=BF16):
    return (synth.normal((B, Hq, Sq, D), seed, synth.STREAM_Q, dtype),
            synth.normal((B, Hkv, Sk, D), seed, synth.STREAM_K, dtype),
            synth.normal((B, Hkv, Sk, D), seed, synth.STREAM_V, dtype),
            synth.normal((B, Hq, Sq, D), seed, synth.STREAM_DO, dtype))


def check_grad(got, ref, what):
    g = got.detach().to("cpu", torch.float64).reshape(ref.shape)
    assert torch.isfinite(g).all(), f"{what}: non-finite gradient"
    err = (g - ref).abs()
    s = max(1.0, ref.abs().max().item())
    mx, mean = err.max().item(), err.mean().item()
    bar_max, bar_mean = (1e-4, 1e-5) if got.dtype == torch.float32 else (2e-2, 2e-3)
    assert mx <= bar_max * s, f"{what}: max abs err {mx:.3e} > {bar_max} x {s:.3g}"
    assert mean <= bar_mean * s, f"{what}: mean abs err {mean:.3e} > {bar_mean} x {s:.3g}"
    return mx, mean


def _run(cuda_device, B, Hq, Hkv, Sq, Sk, D, seed=0, dtype=BF16, causal=False, wl=None, wr=None, cap=None,
         alibi=False, rowb=None, given_fwd=False):
    import tiled_scaled_dot_gb300 as g
    q, k, v, do = _inputs(B, Hq, Hkv, Sq, Sk, D, seed, dtype)
    slopes = synth.alibi_slopes(Hq) if alibi else None
    kw = dict(causal=causal, window_left=wl, window_right=wr, softcap=cap)
    ref = oracle.attn_bwd(q, k, v, do, alibi_slopes=slopes, row_kv_bounds=rowb, **kw)
    dev = [t.to(cuda_device) for t in (q, k, v, do)]
    sl = None if slopes is None else slopes.to(cuda_device)
    rb = None if rowb is None else rowb.to(cuda_device)
    out = lse = None
    if given_fwd:
        lse = torch.empty(B, Hq, Sq, dtype=torch.float32, device=cuda_device)
        out = g.attn_fwd(dev[0], dev[1], dev[2], sl, lse=lse, row_kv_bounds=rb, **kw)
    grads = g.attn_bwd(*dev, out, lse, sl, row_kv_bounds=rb, **kw)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    what = f"bwd B{B} H{Hq}/{Hkv} S{Sq}x{Sk} D{D} {dtype} {kw} alibi{alibi} rowb{rowb is not None}"
    for name, got, want in zip(("dq", "dk", "dv"), grads, ref):
        check_grad(got, want, f"{what} {name}")
    return grads, ref


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_bwd_tiles_and_ragged_tail(cuda_device, D, causal):
    # 300 rows: two full 128-row tiles and a ragged third, on both axes
    _run(cuda_device, 1, 4, 2, 300, 300, D, seed=1, causal=causal)


@pytest.mark.parametrize("Sq,Sk", [(200, 333), (333, 200), (1, 257), (129, 1)])
def test_bwd_unequal_lengths(cuda_device, Sq, Sk):
    _run(cuda_device, 2, 2, 1, Sq, Sk, 128, seed=2, causal=True)


@pytest.mark.parametrize("G", [1, 2, 4])
def test_bwd_gqa_groups(cuda_device, G):
    _run(cuda_device, 2, 2 * G, 2, 256, 256, 128, seed=3, causal=True)


@pytest.mark.parametrize("D", [64, 128])
def test_bwd_softcap_alibi_window(cuda_device, D):
    _run(cuda_device, 1, 4, 4, 384, 384, D, seed=4, causal=True, wl=100, wr=0, cap=30.0, alibi=True)


def test_bwd_two_sided_window_noncausal_alibi(cuda_device):
    _run(cuda_device, 2, 4, 2, 320, 320, 64, seed=5, wl=70, wr=40, alibi=True)


def test_bwd_row_bounds_with_empty_rows(cuda_device):
    B, S = 2, 384
    rowb = synth.row_kv_bounds_with_empty_rows(B, S, S, 0.05, seed=6)
    grads, ref = _run(cuda_device, B, 4, 2, S, S, 128, seed=6, causal=True, rowb=rowb)
    empty = rowb[..., 0] > rowb[..., 1]  # [B, S]
    assert empty.any()
    dq = grads[0].cpu()
    assert (dq.permute(0, 2, 1, 3)[empty] == 0).all()


def test_bwd_random_row_bounds(cuda_device):
    # arbitrary per-row key ranges: the dK / dV kernel masks column by column
    B, S = 2, 300
    lo = synth.randint(B * S, S, 9, synth.STREAM_AUX).view(B, S)
    span = synth.randint(B * S, S, 10, synth.STREAM_AUX).view(B, S)
    rowb = torch.stack([lo, torch.clamp(lo + span - S // 3, max=S - 1)], dim=-1).to(torch.int32)
    assert (rowb[..., 0] > rowb[..., 1]).any() and (rowb[..., 0] <= rowb[..., 1]).any()
    _run(cuda_device, B, 4, 2, S, S, 64, seed=9, rowb=rowb, alibi=True)


def test_bwd_fp16(cuda_device):
    _run(cuda_device, 1, 4, 2, 300, 300, 128, seed=7, dtype=torch.float16, causal=True, cap=20.0, alibi=True)


def test_bwd_given_forward_equals_recompute(cuda_device):
    import tiled_scaled_dot_gb300 as g
    B, Hq, Hkv, S, D = 2, 4, 2, 256, 128
    q, k, v, do = (t.to(cuda_device) for t in _inputs(B, Hq, Hkv, S, S, D, 8))
    lse = torch.empty(B, Hq, S, dtype=torch.float32, device=cuda_device)
    out = g.attn_fwd(q, k, v, causal=True, lse=lse)
    a = g.attn_bwd(q, k, v, do, out, lse, causal=True)
    b = g.attn_bwd(q, k, v, do, causal=True)
    c = g.attn_bwd(q, k, v, do, causal=True)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    for x, y, z in zip(a, b, c):
        assert torch.equal(x, y) and torch.equal(y, z)


def test_bwd_full_size_sampled_groups(cuda_device):
    """The causal B4 Hq32 Hkv8 S2048 D128 shape: every gradient of two
    seeded (batch, kv group) slices, each computed whole by the oracle."""
    import tiled_scaled_dot_gb300 as g
    B, Hq, Hkv, S, D = 4, 32, 8, 2048, 128
    G = Hq // Hkv
    q, k, v, do = _inputs(B, Hq, Hkv, S, S, D, 0)
    dq, dk, dv = g.attn_bwd(*(t.to(cuda_device) for t in (q, k, v, do)), causal=True)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    for b, kh in ((0, 0), (3, 5)):
        hs = slice(kh * G, (kh + 1) * G)
        ref = oracle.attn_bwd(q[b:b + 1, hs], k[b:b + 1, kh:kh + 1], v[b:b + 1, kh:kh + 1],
                              do[b:b + 1, hs], causal=True)
        for name, got, want in zip(("dq", "dk", "dv"),
                                   (dq[b:b + 1, hs], dk[b:b + 1, kh:kh + 1], dv[b:b + 1, kh:kh + 1]), ref):
            check_grad(got, want, f"full size b{b} group{kh} {name}")


def test_bwd_outputs_16_byte_aligned(cuda_device):
    # gradient buffers 16 bytes past a 32-byte boundary take the 16-byte store
    # path; the result is bitwise that of aligned buffers
    import tiled_scaled_dot_gb300 as g
    B, Hq, Hkv, S, D = 1, 4, 2, 200, 128
    q, k, v, do = (t.to(cuda_device) for t in _inputs(B, Hq, Hkv, S, S, D, 10))

    def offset_like(t):
        buf = torch.empty(t.numel() + 8, dtype=t.dtype, device=cuda_device)
        out = buf[8:].view(t.shape)
        assert out.data_ptr() % 32 == 16
        return out

    a = g.attn_bwd(q, k, v, do, causal=True)
    dq, dk, dv = offset_like(q), offset_like(k), offset_like(v)
    b = g.attn_bwd(q, k, v, do, causal=True, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    for x, y in zip(a, b):
        assert torch.equal(x, y)


F32 = torch.float32


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_bwd_fp32_tiles_and_ragged_tail(cuda_device, D, causal):
    _run(cuda_device, 1, 4, 2, 150, 150, D, seed=11, dtype=F32, causal=causal)


@pytest.mark.parametrize("Sq,Sk", [(70, 133), (133, 70), (1, 65)])
def test_bwd_fp32_unequal_lengths(cuda_device, Sq, Sk):
    _run(cuda_device, 2, 4, 1, Sq, Sk, 64, seed=12, dtype=F32, causal=True)


def test_bwd_fp32_softcap_alibi_window(cuda_device):
    _run(cuda_device, 1, 4, 2, 160, 160, 128, seed=13, dtype=F32, causal=True, wl=40, wr=0, cap=20.0, alibi=True)


def test_bwd_fp32_row_bounds_given_forward(cuda_device):
    B, S = 2, 96
    rowb = synth.row_kv_bounds_with_empty_rows(B, S, S, 0.05, seed=14)
    grads, _ = _run(cuda_device, B, 2, 2, S, S, 64, seed=14, dtype=F32, rowb=rowb, alibi=True, given_fwd=True)
    empty = rowb[..., 0] > rowb[..., 1]
    assert empty.any() and (grads[0].cpu().permute(0, 2, 1, 3)[empty] == 0).all()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_bwd_phase_times_form(cuda_device, dtype):
    """attn_bwd_phase_times writes the same gradients as attn_bwd and four phase
    times in the order (forward recompute, prep, dK / dV, dQ), whatever order
    the launches run in (the 16-bit path runs dQ first)."""
    import tiled_scaled_dot_gb300 as g
    B, Hq, Hkv, S, D = 2, 8, 2, 512, 128
    q, k, v, do = (t.to(cuda_device) for t in _inputs(B, Hq, Hkv, S, S, D, 9, dtype))
    lse = torch.empty(B, Hq, S, dtype=torch.float32, device=cuda_device)
    out = g.attn_fwd(q, k, v, causal=True, lse=lse)
    ref = g.attn_bwd(q, k, v, do, out, lse, causal=True)
    *grads, phases = g.attn_bwd(q, k, v, do, out, lse, causal=True, phase_times_reps=3)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    for x, y in zip(ref, grads):
        assert torch.equal(x, y)
    assert len(phases) == 4 and all(t >= 0.0 for t in phases)
    fwd, prep, dkdv, dq = phases
    assert fwd < 0.05 and dkdv > 0.0 and dq > 0.0  # out and lse given: no recompute
