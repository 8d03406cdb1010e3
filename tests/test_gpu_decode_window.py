"""GPU parity of the sliding window in the decode entries (attn_decode and
attn_decode_paged through the C ABI) against the float64 oracles.

The decode query is the newest token, at position Sk - 1 (paged: its context
length - 1); the dense contract's window (attention.fkc.md, header:
window_size_left/right) admits keys j >= pos - window_left, and ALiBi adds
slope (j - pos).  Cases: windows shorter than one 64-key tile, than one split
and longer than the sequence; windows starting on and off a tile boundary;
automatic and explicit split counts; bf16 and fp16; softcap and ALiBi; paged
contexts of uneven lengths, including empty and shorter-than-window ones.
"""
import pytest
import torch

import oracle
import synth
from synth.workloads import make_paged_inputs
from tests._parity import check_lse, check_out

pytestmark = pytest.mark.gpu


def run_window(dev, B, Hq, Hkv, Sk, D, wl, splits=0, dtype=torch.bfloat16, softcap=None, alibi=False, wr=None,
               seed=41):
    import tiled_scaled_dot_gb300 as g
    q = synth.normal((B, Hq, 1, D), seed, synth.STREAM_Q, dtype)
    k = synth.normal((B, Hkv, Sk, D), seed, synth.STREAM_K, dtype)
    v = synth.normal((B, Hkv, Sk, D), seed, synth.STREAM_V, dtype)
    slopes = synth.alibi_slopes(Hq) if alibi else None
    ref, ref_lse = oracle.decode(q, k, v, softcap=softcap, alibi_slopes=slopes, window_left=wl, window_right=wr,
                                 return_lse=True)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)
    out = g.attn_decode(q.to(dev), k.to(dev), v.to(dev), None if slopes is None else slopes.to(dev),
                        softcap=softcap, window_left=wl, window_right=wr, num_splits=splits, lse=lse)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    what = f"decode window B{B} Hq{Hq} Hkv{Hkv} Sk{Sk} D{D} wl{wl} splits{splits} {dtype} cap{softcap} alibi{alibi}"
    check_out(out, ref, dtype, what)
    check_lse(lse.view(B, Hq, 1), ref_lse, dtype, what)
    return out


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("wl", [0, 1, 63, 64, 100, 777, 5000])
@pytest.mark.parametrize("splits", [0, 1, 3, 8])
def test_decode_window(cuda_device, D, wl, splits):
    run_window(cuda_device, 2, 8, 2, 3001, D, wl, splits)


@pytest.mark.parametrize("flags", [dict(softcap=30.0), dict(alibi=True), dict(softcap=5.0, alibi=True, wr=0),
                                   dict(dtype=torch.float16), dict(dtype=torch.float16, alibi=True, softcap=20.0)])
def test_decode_window_flags(cuda_device, flags):
    run_window(cuda_device, 3, 8, 2, 2048, 128, 300, 0, **flags)
    run_window(cuda_device, 2, 4, 4, 1000, 64, 130, 4, **flags)


def test_decode_window_shorter_than_one_split(cuda_device):
    # 64 explicit splits of a 40-key window: most splits are empty
    run_window(cuda_device, 1, 4, 1, 4096, 128, 40, 64)


def test_decode_window_tiles_before_the_window_are_not_read(cuda_device):
    """NaN in every key and value before the window's first tile: the output
    is still finite and equal to the clean inputs' output, bitwise."""
    import tiled_scaled_dot_gb300 as g
    B, Hq, Hkv, Sk, D, wl = 2, 8, 2, 2000, 128, 200
    q = synth.normal((B, Hq, 1, D), 5, 0, torch.bfloat16).cuda()
    k = synth.normal((B, Hkv, Sk, D), 5, 1, torch.bfloat16).cuda()
    v = synth.normal((B, Hkv, Sk, D), 5, 2, torch.bfloat16).cuda()
    clean = g.attn_decode(q, k, v, window_left=wl, num_splits=3)
    first_tile = (Sk - 1 - wl) // 64 * 64
    k2, v2 = k.clone(), v.clone()
    k2[:, :, :first_tile] = float("nan")
    v2[:, :, :first_tile] = float("nan")
    dirty = g.attn_decode(q, k2, v2, window_left=wl, num_splits=3)
    torch.cuda.synchronize()
    assert torch.equal(clean, dirty)


def run_paged_window(dev, B, Hq, Hkv, D, ctx, bs, wl, splits=0, dtype=torch.bfloat16, softcap=None, alibi=False,
                     seed=43):
    import tiled_scaled_dot_gb300 as g
    x = make_paged_inputs(B, Hq, Hkv, D, ctx, bs, dtype=dtype, seed=seed)
    slopes = synth.alibi_slopes(Hq) if alibi else None
    ref, ref_lse = oracle.attn_paged(x["q"], x["k_cache"], x["v_cache"], x["block_table"], x["context_lens"],
                                     softcap=softcap, alibi_slopes=slopes, window_left=wl, return_lse=True)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)
    out = g.attn_decode_paged(x["q"].to(dev), x["k_cache"].to(dev), x["v_cache"].to(dev),
                              x["block_table"].to(dev), x["context_lens"].to(dev),
                              None if slopes is None else slopes.to(dev), softcap=softcap, window_left=wl,
                              num_splits=splits, lse=lse)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    what = f"paged window B{B} ctx{list(ctx)[:5]} bs{bs} wl{wl} splits{splits} {dtype} cap{softcap} alibi{alibi}"
    check_out(out, ref, dtype, what)
    check_lse(lse.view(B, Hq, 1), ref_lse, dtype, what)


@pytest.mark.parametrize("bs", [16, 64, 256])
@pytest.mark.parametrize("wl", [0, 50, 64, 700])
@pytest.mark.parametrize("splits", [0, 2, 9])
def test_paged_window(cuda_device, bs, wl, splits):
    run_paged_window(cuda_device, 5, 8, 2, 128, [0, 1, 64, 300, 1500], bs, wl, splits)


@pytest.mark.parametrize("flags", [dict(alibi=True, softcap=25.0), dict(dtype=torch.float16, alibi=True)])
def test_paged_window_flags(cuda_device, flags):
    run_paged_window(cuda_device, 3, 8, 2, 64, [1000, 129, 2048], 32, 333, 0, **flags)
