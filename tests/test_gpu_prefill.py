"""GPU parity of the prefill entry (attn_fwd / attn_fwd_ex through the C ABI)
against the float64 oracle, element by element, on seeded inputs.

Small cases span several 128-row / 128-key tiles with ragged tails, both GQA
pairings (Hq/Hkv even: two heads per work item; odd: two row tiles), every
flag (causal, windows, softcap, ALiBi, per-row bounds with empty rows) and
the degenerate sizes (one row, one key, Sq != Sk).
"""
import pytest
import torch

import oracle
import synth
from tests._parity import check_lse, check_out

pytestmark = pytest.mark.gpu


def _inputs(B, Hq, Hkv, Sq, Sk, D, dtype, seed=1):
    q = synth.normal((B, Hq, Sq, D), seed, synth.STREAM_Q, dtype)
    k = synth.normal((B, Hkv, Sk, D), seed, synth.STREAM_K, dtype)
    v = synth.normal((B, Hkv, Sk, D), seed, synth.STREAM_V, dtype)
    return q, k, v


def _rowb(B, Sq, Sk, seed=4):
    lo = synth.randint(B * Sq, Sk, seed, 5).view(B, Sq)
    hi = synth.randint(B * Sq, Sk, seed, 6).view(B, Sq)
    rb = torch.stack((torch.minimum(lo, hi), torch.maximum(lo, hi)), -1).to(torch.int32)
    empty = synth.empty_rows(B, Sq, 0.05, seed)
    for f in empty:
        b, i = divmod(f, Sq)
        rb[b, i] = torch.tensor([1, 0], dtype=torch.int32)
    return rb


def run_case(dev, B, Hq, Hkv, Sq, Sk, D, dtype=torch.bfloat16, causal=False, wl=None, wr=None, softcap=None,
             alibi=False, rowb=False, scale=None, lse=True):
    import tiled_scaled_dot_gb300 as g
    q, k, v = _inputs(B, Hq, Hkv, Sq, Sk, D, dtype)
    slopes = synth.alibi_slopes(Hq) if alibi else None
    rb = _rowb(B, Sq, Sk) if rowb else None
    kw = dict(causal=causal, window_left=wl, window_right=wr, softcap=softcap, alibi_slopes=slopes,
              row_kv_bounds=rb)
    ref, ref_lse = oracle.attn(q, k, v, scale=scale, return_lse=True, **kw)
    gl = torch.empty(B, Hq, Sq, dtype=torch.float32, device=dev) if lse else None
    out = g.attn_fwd(q.to(dev), k.to(dev), v.to(dev), None if slopes is None else slopes.to(dev),
                     softmax_scale=scale, causal=causal, window_left=wl, window_right=wr, softcap=softcap,
                     row_kv_bounds=None if rb is None else rb.to(dev), lse=gl)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    what = f"B{B} Hq{Hq} Hkv{Hkv} Sq{Sq} Sk{Sk} D{D} {dtype} {kw if not rowb else 'rowb'}"
    check_out(out, ref, dtype, what)
    if lse:
        check_lse(gl, ref_lse, dtype, what)
    return out


SMALL = [
    # (B, Hq, Hkv, Sq, Sk, D)
    (1, 2, 1, 128, 128, 128),
    (1, 4, 2, 300, 300, 128),
    (2, 4, 1, 257, 257, 64),
    (1, 3, 3, 200, 333, 64),
    (1, 2, 2, 1, 1, 128),
    (1, 2, 1, 65, 1, 64),
    (1, 2, 2, 1, 500, 128),
    (1, 6, 2, 384, 130, 128),
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_plain(cuda_device, shape, causal):
    run_case(cuda_device, *shape, causal=causal)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("flags", [
    dict(causal=True, wl=100, wr=0),
    dict(causal=False, wl=70, wr=40),
    dict(causal=True, softcap=5.0),
    dict(causal=True, alibi=True),
    dict(causal=True, wl=150, wr=0, softcap=50.0, alibi=True),
    dict(causal=False, softcap=2.0, alibi=True),
    dict(causal=True, rowb=True),
    dict(causal=False, wl=64, wr=64, rowb=True, alibi=True, softcap=30.0),
], ids=lambda f: "-".join(f"{k}{v}" for k, v in f.items()))
def test_bf16_flags(cuda_device, D, flags):
    run_case(cuda_device, 2, 4, 2, 391, 391, D, **flags)
    run_case(cuda_device, 1, 3, 1, 260, 260, D, **flags)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("softcap", [21.0, 23.0, 25.0])
def test_bf16_softcap_moderate_caps(cuda_device, D, softcap):
    # Scores scale * q.k are about N(0, 1) and reach 4 to 5 in a 128 x 128 tile:
    # caps of 21..25 bend the largest scores by a few percent, with and without
    # ALiBi and windows.
    run_case(cuda_device, 2, 4, 2, 520, 520, D, causal=True, softcap=softcap)
    run_case(cuda_device, 1, 4, 4, 300, 300, D, softcap=softcap, alibi=True, wl=200, wr=50)


def test_bf16_window_masks_every_key_of_some_rows(cuda_device):
    # window_right = 0, window_left = 0 and causal off, plus Sq > Sk: rows past Sk see no key
    run_case(cuda_device, 1, 2, 2, 300, 100, 128, wl=0, wr=0)


def test_bf16_scale_not_default(cuda_device):
    run_case(cuda_device, 1, 2, 1, 200, 200, 128, causal=True, scale=0.02)
    run_case(cuda_device, 1, 2, 1, 200, 200, 64, causal=True, scale=0.3)


def test_bf16_large_logits_stay_finite(cuda_device):
    import tiled_scaled_dot_gb300 as g
    q, k, v = _inputs(1, 2, 1, 256, 256, 128, torch.bfloat16)
    q = (q.float() * 6).to(torch.bfloat16)
    ref = oracle.attn(q, k, v, causal=True)
    out = g.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    check_out(out, ref, torch.bfloat16, "large logits")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("flags", [dict(), dict(causal=True), dict(causal=True, wl=20, wr=0, softcap=3.0,
                                                                     alibi=True, rowb=True)])
def test_fp32(cuda_device, D, flags):
    run_case(cuda_device, 1, 4, 2, 150, 150, D, dtype=torch.float32, **flags)
    run_case(cuda_device, 2, 3, 1, 33, 70, D, dtype=torch.float32, **flags)


def test_reruns_are_bitwise_identical(cuda_device):
    import tiled_scaled_dot_gb300 as g
    q, k, v = _inputs(2, 8, 2, 700, 700, 128, torch.bfloat16)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    a = g.attn_fwd(q, k, v, causal=True)
    b = g.attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_stream_argument_is_used(cuda_device):
    import tiled_scaled_dot_gb300 as g
    q, k, v = _inputs(1, 2, 1, 256, 256, 64, torch.bfloat16)
    ref = oracle.attn(q, k, v)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
        out = g.attn_fwd(qd, kd, vd, stream=s)
    s.synchronize()
    check_out(out, ref, torch.bfloat16, "side stream")
