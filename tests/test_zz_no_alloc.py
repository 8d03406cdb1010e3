"""attn_decode_noalloc: the decode entry for callers that cannot allocate.

Some callers cannot pass the library a workspace (their own memory pool owns
the device, or their serving loop must never call cudaMalloc).  For them the
library takes the decode's split partials from a fixed scratch array in its
own device module.  This test calls that entry through the C ABI twice in a
row, on different inputs, with the automatic split count and with 8 explicit
splits.  The entry runs the same split plan and the same fixed-order combine
as the ordinary attn_decode (which gets a workspace from the caller), so each
output and lse must be bitwise equal to attn_decode's; each output is also
checked against the float64 oracle within the bf16 parity tolerance of the
other tests.  An oversized problem must be refused.  The file name puts it
last in collection order.
"""
import ctypes

import pytest
import torch

import oracle
import synth
from tests._parity import check_lse, check_out

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


@pytest.mark.parametrize("num_splits", [0, 8])
def test_noalloc_decode_matches_workspace_decode_twice(cuda_device, num_splits):
    g, fn = _entry()
    B, Hq, Hkv, Sk, D = 4, 16, 4, 3000, 128
    assert g.decode_workspace_size(B, Hq, Hkv, Sk, D, num_splits) > 0  # the scratch is really used
    stream = torch.cuda.current_stream()
    for seed in (21, 22):
        q, k, v = _inputs(seed, B, Hq, Hkv, Sk, D, cuda_device)
        ref_lse = torch.empty(B, Hq, dtype=torch.float32, device=cuda_device)
        ref = g.attn_decode(q, k, v, lse=ref_lse, num_splits=num_splits)
        out = torch.full_like(q, float("nan"))
        lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=cuda_device)
        st = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), None, out.data_ptr(), lse.data_ptr(),
                B, Hq, Hkv, Sk, D, 1.0 / D ** 0.5, 0.0, num_splits, 0, ctypes.c_void_p(stream.cuda_stream))
        assert st == 0, g.lib().gbattn_status_string(st)
        torch.cuda.synchronize()
        assert g.device_status() == 0
        # same kernels, same split plan, same combine order: bitwise equal
        assert torch.equal(out, ref), f"seed {seed}: output differs from attn_decode"
        assert torch.equal(lse, ref_lse), f"seed {seed}: lse differs from attn_decode"
        want, want_lse = oracle.decode(q.cpu(), k.cpu(), v.cpu(), scale=1.0 / D ** 0.5, return_lse=True)
        check_out(out, want, torch.bfloat16, f"noalloc seed {seed} splits {num_splits}")
        check_lse(lse, want_lse, torch.bfloat16, f"noalloc seed {seed} splits {num_splits}")


def test_noalloc_decode_refuses_oversized_problem(cuda_device):
    g, fn = _entry()
    B, Hq, Hkv, Sk, D = 512, 64, 8, 65536, 128
    need = g.decode_workspace_size(B, Hq, Hkv, Sk, D, 256)
    assert need > 32 * 1024 * 1024
    st = fn(16, 32, 48, None, 64, None, B, Hq, Hkv, Sk, D, 0.1, 0.0, 256, 0, None)
    assert st == 2  # GBATTN_ERR_UNSUPPORTED, nothing launched
