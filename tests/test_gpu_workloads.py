"""The five benchmark workloads at full size, in the launch configuration the
benchmark times (same entry points, default split choice, default stream).

Outputs are compared with the float64 oracle on sampled rows (the oracle
computes each sampled row on its own): the first and last rows of every
tile boundary class, every fully-masked row, and a seeded random sample.
The fp32 workload is small enough to compare in full.
"""
import pytest
import torch

import oracle
import synth
from synth.workloads import WORKLOADS, make_inputs
from tests._parity import check_lse, check_out

pytestmark = pytest.mark.gpu


def _sample_rows(w, rb, n=384):
    Sq = w.Sq
    total = w.B * w.Hq * Sq
    picks = set(synth.randint(n, total, 9, 7).tolist())
    for b in range(w.B):
        for h in (0, w.Hq - 1):
            for qi in (0, 1, 127, 128, 129, Sq // 2, Sq - 129, Sq - 128, Sq - 2, Sq - 1):
                if 0 <= qi < Sq:
                    picks.add((b * w.Hq + h) * Sq + qi)
    if rb is not None:
        empty = (rb[..., 0] > rb[..., 1]).nonzero().tolist()
        for b, qi in empty:
            for h in range(w.Hq):
                picks.add((b * w.Hq + h) * Sq + qi)
    return torch.tensor(sorted(picks), dtype=torch.int64)


@pytest.mark.parametrize("name", [n for n in WORKLOADS if not WORKLOADS[n].decode])
def test_prefill_workload(cuda_device, name):
    import tiled_scaled_dot_gb300 as g
    w = WORKLOADS[name]
    x = make_inputs(w, "cpu")
    dev = {k: (None if t is None else t.to(cuda_device)) for k, t in x.items()}
    lse = torch.empty(w.B, w.Hq, w.Sq, dtype=torch.float32, device=cuda_device)
    out = g.attn_fwd(dev["q"], dev["k"], dev["v"], dev["alibi_slopes"], softmax_scale=w.scale, causal=w.causal,
                     window_left=w.window_left, window_right=w.window_right, softcap=w.softcap,
                     row_kv_bounds=dev["row_kv_bounds"], lse=lse)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    kw = dict(scale=w.scale, causal=w.causal, window_left=w.window_left, window_right=w.window_right,
              softcap=w.softcap, alibi_slopes=x["alibi_slopes"], row_kv_bounds=x["row_kv_bounds"])
    if w.dtype == torch.float32:
        ref, ref_lse = oracle.attn(x["q"], x["k"], x["v"], return_lse=True, **kw)
        check_out(out, ref, w.dtype, name)
        check_lse(lse, ref_lse, w.dtype, name)
        return
    rows = _sample_rows(w, x["row_kv_bounds"])
    ref, ref_lse = oracle.attn(x["q"], x["k"], x["v"], rows=rows, return_lse=True, **kw)
    got = out.view(-1, w.D)[rows.to(cuda_device)]
    check_out(got, ref, w.dtype, name)
    check_lse(lse.view(-1)[rows.to(cuda_device)], ref_lse, w.dtype, name)
    if x["row_kv_bounds"] is not None:
        rb = x["row_kv_bounds"]
        empty = rb[..., 0] > rb[..., 1]
        o = out.float().cpu().view(w.B, w.Hq, w.Sq, w.D)
        assert (o.permute(0, 2, 1, 3)[empty] == 0).all()


def test_decode_workload(cuda_device):
    import tiled_scaled_dot_gb300 as g
    w = WORKLOADS["bf16_decode_b64_h32_sk8192_d128"]
    x = make_inputs(w, cuda_device)
    lse = torch.empty(w.B, w.Hq, dtype=torch.float32, device=cuda_device)
    out = g.attn_decode(x["q"], x["k"], x["v"], softmax_scale=w.scale, lse=lse)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    # sampled (b, h) rows; the oracle needs only their kv heads
    rows = sorted(set(synth.randint(48, w.B * w.Hq, 9, 8).tolist()) | {0, w.B * w.Hq - 1})
    for r in rows:
        b, h = divmod(r, w.Hq)
        kv = h // (w.Hq // w.Hkv)
        q = x["q"][b:b + 1, h:h + 1].cpu()
        k = x["k"][b:b + 1, kv:kv + 1].cpu()
        v = x["v"][b:b + 1, kv:kv + 1].cpu()
        ref, ref_lse = oracle.decode(q, k, v, scale=w.scale, return_lse=True)
        check_out(out[b:b + 1, h:h + 1], ref, torch.bfloat16, f"decode row {r}")
        check_lse(lse[b:b + 1, h:h + 1].reshape(1, 1, 1), ref_lse, torch.bfloat16, f"decode row {r}")


@pytest.mark.parametrize("shape", [(8, 16, 8, 4096, 128), (16, 8, 8, 4096, 64)], ids=["gqa2_d128", "mha_d64"])
def test_dense_prefill_with_kv_beyond_l2(cuda_device, shape):
    """Dense problems whose K and V (134 MB here) do not fit in L2: more work
    items than one pass of the persistent grid, both GQA pairings; sampled rows
    against the oracle."""
    import tiled_scaled_dot_gb300 as g
    from synth.workloads import scaled
    B, Hq, Hkv, S, D = shape
    w = scaled(WORKLOADS["bf16_causal_b4_h32_s2048_d128"], name=f"banded_{B}_{Hq}_{Hkv}_{S}_{D}", B=B, Hq=Hq,
               Hkv=Hkv, Sq=S, Sk=S, D=D)
    assert 2 * B * Hkv * S * D * 2 > 64 * 2**20
    x = make_inputs(w, cuda_device)
    lse = torch.empty(B, Hq, S, dtype=torch.float32, device=cuda_device)
    out = g.attn_fwd(x["q"], x["k"], x["v"], causal=True, lse=lse)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    rows = _sample_rows(w, None, n=256)
    ref, ref_lse = oracle.attn(x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), causal=True, rows=rows, return_lse=True)
    check_out(out.view(-1, D)[rows.to(cuda_device)], ref, torch.bfloat16, w.name)
    check_lse(lse.view(-1)[rows.to(cuda_device)], ref_lse, torch.bfloat16, w.name)


def test_varlen_bench_workload(cuda_device):
    """The benchmark's packed workload at full size (32 causal sequences of
    512..4096 tokens, Hq 32, Hkv 8, D 128: 8 bands of sequences), as the
    benchmark launches it.  Each checked sequence is compared on sampled rows
    with the dense oracle over that sequence alone (queries = keys, where the
    bottom-right causal alignment is the top-left one)."""
    import tiled_scaled_dot_gb300 as g
    B, Hq, Hkv, D = 32, 32, 8, 128
    lens = (512 + synth.randint(B, 4096 - 512 + 1, 0, 7)).tolist()
    cu = torch.tensor([0] + [sum(lens[:i + 1]) for i in range(B)], dtype=torch.int32)
    T = int(cu[-1])
    q = synth.normal((T, Hq, D), 0, synth.STREAM_Q, torch.bfloat16, cuda_device)
    k = synth.normal((T, Hkv, D), 0, synth.STREAM_K, torch.bfloat16, cuda_device)
    v = synth.normal((T, Hkv, D), 0, synth.STREAM_V, torch.bfloat16, cuda_device)
    cud = cu.to(cuda_device)
    lse = torch.empty(Hq, T, dtype=torch.float32, device=cuda_device)
    out = g.attn_fwd_varlen(q, k, v, cud, cud, max(lens), causal=True, lse=lse)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    order = sorted(range(B), key=lambda i: lens[i])
    picks = sorted(set([order[0], order[-1]] + synth.randint(4, B, 5, 9).tolist()))
    for b in picks:
        a0, n = int(cu[b]), lens[b]
        qs = q[a0:a0 + n].permute(1, 0, 2).unsqueeze(0).cpu()
        ks = k[a0:a0 + n].permute(1, 0, 2).unsqueeze(0).cpu()
        vs = v[a0:a0 + n].permute(1, 0, 2).unsqueeze(0).cpu()
        w = synth.randint(48, Hq * n, 6, b).tolist()
        edge = [(h * n + i) for h in (0, Hq - 1) for i in (0, 1, 127, 128, n // 2, n - 129, n - 2, n - 1) if 0 <= i < n]
        rows = torch.tensor(sorted(set(w + edge)), dtype=torch.int64)
        ref, ref_lse = oracle.attn(qs, ks, vs, causal=True, rows=rows, return_lse=True)
        h, i = rows // n, rows % n
        got = out[a0 + i.to(cuda_device), h.to(cuda_device)]
        check_out(got, ref, torch.bfloat16, f"varlen bench sequence {b} ({n} tokens)")
        check_lse(lse[h.to(cuda_device), a0 + i.to(cuda_device)], ref_lse, torch.bfloat16, f"varlen sequence {b}")
