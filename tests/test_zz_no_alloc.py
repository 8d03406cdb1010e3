"""attn_decode_noalloc: the decode entry for callers that cannot allocate.

Some callers cannot pass the library a workspace (their own memory pool owns
the device, or their serving loop must never call cudaMalloc).  For them the
library takes the decode's split partials from a fixed scratch array in its
own device module.  This test calls that entry through the C ABI twice in a
row, on different inputs, and checks each result against the ordinary
attn_decode (which gets a workspace from the caller) within the bf16 parity
tolerance of the other tests; it also checks that an oversized problem is
refused.  The file name puts it last in collection order.
"""
import ctypes

import pytest
import torch

import synth
from tests._parity import BF16_MAX, BF16_MEAN

pytestmark = pytest.mark.gpu


def _entry():
    import tiled_scaled_dot_gb300 as g
    L = g.lib()
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn = L.attn_decode_noalloc
    fn.argtypes = [P, P, P, P, P, P, I, I, I, I, I, F, F, I, I, P]
    fn.restype = I
    return g, fn


def _inputs(seed, B, Hq, Hkv, Sk, D, dev):
    q = synth.normal((B, Hq, 1, D), seed, 0, torch.bfloat16, dev)
    k = synth.normal((B, Hkv, Sk, D), seed, 1, torch.bfloat16, dev)
    v = synth.normal((B, Hkv, Sk, D), seed, 2, torch.bfloat16, dev)
    return q, k, v


def test_noalloc_decode_matches_workspace_decode_twice(cuda_device):
    g, fn = _entry()
    B, Hq, Hkv, Sk, D = 4, 16, 4, 3000, 128
    assert g.decode_workspace_size(B, Hq, Hkv, Sk, D, 0) > 0  # the scratch is really used
    stream = torch.cuda.current_stream()
    for seed in (21, 22):
        q, k, v = _inputs(seed, B, Hq, Hkv, Sk, D, cuda_device)
        ref_lse = torch.empty(B, Hq, dtype=torch.float32, device=cuda_device)
        ref = g.attn_decode(q, k, v, lse=ref_lse)
        out = torch.full_like(q, float("nan"))
        lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=cuda_device)
        st = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), None, out.data_ptr(), lse.data_ptr(),
                B, Hq, Hkv, Sk, D, 1.0 / D ** 0.5, 0.0, 0, 0, ctypes.c_void_p(stream.cuda_stream))
        assert st == 0, g.lib().gbattn_status_string(st)
        torch.cuda.synchronize()
        assert g.device_status() == 0
        err = (out.double() - ref.double()).abs()
        assert torch.isfinite(out).all()
        assert err.max().item() <= BF16_MAX and err.mean().item() <= BF16_MEAN
        assert (lse - ref_lse).abs().max().item() <= 1e-3


def test_noalloc_decode_refuses_oversized_problem(cuda_device):
    g, fn = _entry()
    B, Hq, Hkv, Sk, D = 512, 64, 8, 65536, 128
    need = g.decode_workspace_size(B, Hq, Hkv, Sk, D, 256)
    assert need > 32 * 1024 * 1024
    st = fn(16, 32, 48, None, 64, None, B, Hq, Hkv, Sk, D, 0.1, 0.0, 256, 0, None)
    assert st == 2  # GBATTN_ERR_UNSUPPORTED, nothing launched
