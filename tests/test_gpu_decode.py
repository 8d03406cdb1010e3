"""GPU parity of the split-KV decode entry (attn_decode through the C ABI)
against the float64 oracle (one query row, every key admissible)."""
import pytest
import torch

import oracle
import synth
from tests._parity import check_lse, check_out

pytestmark = pytest.mark.gpu


def run_decode(dev, B, Hq, Hkv, Sk, D, splits=0, softcap=None, alibi=False, seed=2):
    import tiled_scaled_dot_gb300 as g
    q = synth.normal((B, Hq, 1, D), seed, synth.STREAM_Q, torch.bfloat16)
    k = synth.normal((B, Hkv, Sk, D), seed, synth.STREAM_K, torch.bfloat16)
    v = synth.normal((B, Hkv, Sk, D), seed, synth.STREAM_V, torch.bfloat16)
    slopes = synth.alibi_slopes(Hq) if alibi else None
    ref, ref_lse = oracle.decode(q, k, v, softcap=softcap, alibi_slopes=slopes, return_lse=True)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)
    out = g.attn_decode(q.to(dev), k.to(dev), v.to(dev), None if slopes is None else slopes.to(dev),
                        softcap=softcap, num_splits=splits, lse=lse)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    what = f"decode B{B} Hq{Hq} Hkv{Hkv} Sk{Sk} D{D} splits{splits} cap{softcap} alibi{alibi}"
    check_out(out, ref, torch.bfloat16, what)
    check_lse(lse.view(B, Hq, 1), ref_lse, torch.bfloat16, what)
    return out


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Sk", [1, 64, 100, 1000, 4097])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_decode_shapes(cuda_device, D, Sk, splits):
    run_decode(cuda_device, 2, 8, 2, Sk, D, splits)


@pytest.mark.parametrize("G", [1, 2, 3, 4, 6, 8])
def test_decode_group_sizes(cuda_device, G):
    run_decode(cuda_device, 2, 2 * G, 2, 777, 128, 0)
    run_decode(cuda_device, 1, G, 1, 300, 64, 2)


@pytest.mark.parametrize("flags", [dict(softcap=30.0), dict(alibi=True), dict(softcap=5.0, alibi=True)])
def test_decode_flags(cuda_device, flags):
    run_decode(cuda_device, 2, 8, 2, 2000, 128, 0, **flags)
    run_decode(cuda_device, 2, 8, 2, 500, 64, 4, **flags)


def test_decode_many_splits_more_than_keys(cuda_device):
    run_decode(cuda_device, 1, 4, 1, 130, 128, 64)


def test_decode_reruns_bitwise(cuda_device):
    import tiled_scaled_dot_gb300 as g
    q = synth.normal((4, 8, 1, 128), 3, 0, torch.bfloat16).cuda()
    k = synth.normal((4, 2, 3000, 128), 3, 1, torch.bfloat16).cuda()
    v = synth.normal((4, 2, 3000, 128), 3, 2, torch.bfloat16).cuda()
    a = g.attn_decode(q, k, v, num_splits=5)
    b = g.attn_decode(q, k, v, num_splits=5)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
