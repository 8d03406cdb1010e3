"""The plain prefill entry attn_fwd, called directly through the C ABI.

The binding's attn_fwd goes through attn_fwd_ex; these cases call the
library's attn_fwd symbol itself with ctypes (device pointers, sizes, the
scalar flags and the stream, exactly as a C caller would) and compare its
output with the float64 oracle element by element:
  * the fp32 workload shape (B 1, Hq 2, Hkv 1, S 64, D 64, non-causal), bar 1e-4;
  * bf16 causal with softcap and ALiBi (attention.fkc.md, attention_naive:
    scale, then softcap, then ALiBi, then the mask), bf16 bars;
  * bf16 and fp16 with a two-sided window, Sq != Sk.
"""
import ctypes

import pytest
import torch

import oracle
import synth
from tests._parity import check_out

pytestmark = pytest.mark.gpu

_DT = {torch.bfloat16: 0, torch.float32: 1, torch.float16: 2}


def _call_attn_fwd(q, k, v, slopes, out, scale, causal, wl, wr, softcap, stream):
    import tiled_scaled_dot_gb300 as g
    L = g.lib()
    B, Hq, Sq, D = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    return L.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), None if slopes is None else slopes.data_ptr(),
                      out.data_ptr(), B, Hq, Hkv, Sq, Sk, D, ctypes.c_float(scale), int(causal),
                      -1 if wl is None else wl, -1 if wr is None else wr, ctypes.c_float(softcap or 0.0),
                      _DT[q.dtype], ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.parametrize("case", [
    # (B, Hq, Hkv, Sq, Sk, D, dtype, causal, wl, wr, softcap, alibi)
    (1, 2, 1, 64, 64, 64, torch.float32, False, None, None, None, False),
    (2, 8, 2, 300, 300, 128, torch.bfloat16, True, None, None, 50.0, True),
    (1, 4, 4, 260, 260, 64, torch.bfloat16, True, None, None, 20.0, True),
    (1, 4, 2, 200, 333, 128, torch.bfloat16, False, 90, 30, None, False),
    (1, 4, 2, 200, 333, 64, torch.float16, False, 90, 30, 10.0, True),
], ids=["fp32_b1_h2_s64_d64", "bf16_causal_softcap_alibi_d128", "bf16_causal_softcap_alibi_d64",
        "bf16_window_sq_ne_sk", "fp16_window_softcap_alibi"])
def test_attn_fwd_symbol_matches_oracle(cuda_device, case):
    import tiled_scaled_dot_gb300 as g
    B, Hq, Hkv, Sq, Sk, D, dtype, causal, wl, wr, softcap, alibi = case
    seed = 0 if dtype == torch.float32 else 3
    q = synth.normal((B, Hq, Sq, D), seed, synth.STREAM_Q, dtype)
    k = synth.normal((B, Hkv, Sk, D), seed, synth.STREAM_K, dtype)
    v = synth.normal((B, Hkv, Sk, D), seed, synth.STREAM_V, dtype)
    slopes = synth.alibi_slopes(Hq) if alibi else None
    scale = 1.0 / D ** 0.5
    ref = oracle.attn(q, k, v, scale=scale, causal=causal, window_left=wl, window_right=wr, softcap=softcap,
                      alibi_slopes=slopes)
    qd, kd, vd = q.to(cuda_device), k.to(cuda_device), v.to(cuda_device)
    sd = None if slopes is None else slopes.to(cuda_device)
    out = torch.full_like(qd, float("nan"))
    stream = torch.cuda.current_stream()
    st = _call_attn_fwd(qd, kd, vd, sd, out, scale, causal, wl, wr, softcap, stream)
    assert st == 0, g.lib().gbattn_status_string(st)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    check_out(out, ref, dtype, f"attn_fwd {case}")


def test_attn_fwd_symbol_rejects_before_launch(cuda_device):
    # Hq not a multiple of Hkv: an argument error, nothing launched
    import tiled_scaled_dot_gb300 as g
    q = torch.zeros(1, 3, 64, 64, dtype=torch.bfloat16, device=cuda_device)
    k = torch.zeros(1, 2, 64, 64, dtype=torch.bfloat16, device=cuda_device)
    out = torch.empty_like(q)
    st = _call_attn_fwd(q, k, k, None, out, 0.125, False, None, None, None, torch.cuda.current_stream())
    assert st == 1
    torch.cuda.synchronize()
    assert g.device_status() == 0
