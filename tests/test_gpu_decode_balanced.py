"""GPU parity of the balanced decode launch against the float64 oracles.

An automatic multi-split plan (num_splits = 0) runs the balanced kernel: the
CTAs take equal shares of all (sequence, kv head, head chunk) streams' 64-key
tiles laid end to end, so one stream's tiles may be split across several CTAs
and one CTA may finish one stream and start the next.  Each run writes a
partial (o / l, base-2 lse) into the stream's next workspace slot; the last run
of a stream marks the stream's unused slots empty; the combine merges them in
slot order (gfx942 page, section 8: split-KV decode and its log-sum-exp
combine).  Cases: empty paged contexts between long ones (rows of zeros, lse
-inf), one long context among many short ones (the share floor that keeps a
stream within the workspace's slots), contexts much shorter than the table,
windows, head chunks (G = 8 at D = 128), D = 64 with GC = 8, and reruns that
must agree bitwise.
"""
import pytest
import torch

import oracle
import synth
from synth.workloads import make_paged_inputs
from tests._parity import check_lse, check_out

pytestmark = pytest.mark.gpu


def run_paged(dev, B, Hq, Hkv, D, ctx, bs, wl=None, alibi=False, softcap=None, seed=51, max_blocks=None):
    import tiled_scaled_dot_gb300 as g
    x = make_paged_inputs(B, Hq, Hkv, D, ctx, bs, seed=seed, max_blocks=max_blocks)
    slopes = synth.alibi_slopes(Hq) if alibi else None
    ref, ref_lse = oracle.attn_paged(x["q"], x["k_cache"], x["v_cache"], x["block_table"], x["context_lens"],
                                     softcap=softcap, alibi_slopes=slopes, window_left=wl, return_lse=True)
    args = [x[n].to(dev) for n in ("q", "k_cache", "v_cache", "block_table", "context_lens")]
    sl = None if slopes is None else slopes.to(dev)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)
    out = g.attn_decode_paged(*args, sl, softcap=softcap, window_left=wl, lse=lse)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    what = f"balanced paged B{B} Hq{Hq} Hkv{Hkv} D{D} ctx{list(ctx)[:6]} bs{bs} wl{wl}"
    check_out(out, ref, torch.bfloat16, what)
    check_lse(lse.view(B, Hq, 1), ref_lse, torch.bfloat16, what)
    again = g.attn_decode_paged(*args, sl, softcap=softcap, window_left=wl)
    torch.cuda.synchronize()
    assert torch.equal(out, again), what + ": rerun differs"


def run_dense(dev, B, Hq, Hkv, Sk, D, wl=None, alibi=False, seed=52):
    import tiled_scaled_dot_gb300 as g
    q = synth.normal((B, Hq, 1, D), seed, synth.STREAM_Q, torch.bfloat16)
    k = synth.normal((B, Hkv, Sk, D), seed, synth.STREAM_K, torch.bfloat16)
    v = synth.normal((B, Hkv, Sk, D), seed, synth.STREAM_V, torch.bfloat16)
    slopes = synth.alibi_slopes(Hq) if alibi else None
    ref, ref_lse = oracle.decode(q, k, v, alibi_slopes=slopes, window_left=wl, return_lse=True)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    sl = None if slopes is None else slopes.to(dev)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)
    out = g.attn_decode(qd, kd, vd, sl, window_left=wl, lse=lse)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    what = f"balanced dense B{B} Hq{Hq} Hkv{Hkv} Sk{Sk} D{D} wl{wl} alibi{alibi}"
    check_out(out, ref, torch.bfloat16, what)
    check_lse(lse.view(B, Hq, 1), ref_lse, torch.bfloat16, what)
    # the fixed-split kernel (an explicit split count) agrees within the bar
    fixed = g.attn_decode(qd, kd, vd, sl, window_left=wl, num_splits=3)
    torch.cuda.synchronize()
    check_out(fixed, ref, torch.bfloat16, what + " (3 fixed splits)")
    again = g.attn_decode(qd, kd, vd, sl, window_left=wl)
    torch.cuda.synchronize()
    assert torch.equal(out, again), what + ": rerun differs"


def test_paged_empty_contexts_between_long_ones(cuda_device):
    run_paged(cuda_device, 9, 8, 2, 128, [0, 3000, 0, 1, 0, 64, 2049, 0, 3], 64, alibi=True)


def test_paged_one_long_context_among_short_ones(cuda_device):
    # the share floor keeps the long stream within the workspace's slots
    ctx = [5] * 39 + [6000]
    run_paged(cuda_device, 40, 4, 1, 128, ctx, 32)


def test_paged_contexts_much_shorter_than_the_table(cuda_device):
    ctx = (1 + synth.randint(24, 100, 7, 1)).tolist()
    run_paged(cuda_device, 24, 8, 2, 64, ctx, 16, max_blocks=512)


@pytest.mark.parametrize("wl", [0, 70, 500])
def test_paged_windows(cuda_device, wl):
    run_paged(cuda_device, 6, 8, 2, 128, [4000, 10, 0, 700, 129, 2500], 64, wl=wl, softcap=20.0)


@pytest.mark.parametrize("B,Hq,Hkv,Sk,D", [(1, 32, 8, 20000, 128), (3, 16, 2, 3000, 128), (2, 16, 2, 1500, 64),
                                           (5, 8, 8, 777, 64)])
def test_dense_shapes(cuda_device, B, Hq, Hkv, Sk, D):
    run_dense(cuda_device, B, Hq, Hkv, Sk, D)


def test_dense_window_and_alibi(cuda_device):
    run_dense(cuda_device, 2, 8, 2, 5000, 128, wl=900, alibi=True)
