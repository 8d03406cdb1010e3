"""GPU parity of the fp16 paths (tcgen05 prefill with fp16 operands and P,
split-KV decode and paged decode reading fp16) against the float64 oracle,
which decodes binary16 itself.  The bars are those of the other 16-bit
storage type, bf16: max-abs <= 2e-2, mean-abs <= 2e-3."""
import pytest
import torch

import oracle
import synth
from synth.workloads import make_paged_inputs
from tests._parity import check_lse, check_out

pytestmark = pytest.mark.gpu
F16 = torch.float16


def _qkv(B, Hq, Hkv, Sq, Sk, D, seed):
    return (synth.normal((B, Hq, Sq, D), seed, synth.STREAM_Q, F16),
            synth.normal((B, Hkv, Sk, D), seed, synth.STREAM_K, F16),
            synth.normal((B, Hkv, Sk, D), seed, synth.STREAM_V, F16))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2])
@pytest.mark.parametrize("causal,wl,wr,cap,alibi", [(True, None, None, None, False), (False, None, None, None, False),
                                                    (True, 100, 0, 30.0, True), (False, 50, 70, None, True)])
def test_fp16_prefill(cuda_device, D, G, causal, wl, wr, cap, alibi):
    import tiled_scaled_dot_gb300 as g
    B, Hkv, S = 2, 2, 300
    Hq = G * Hkv
    q, k, v = _qkv(B, Hq, Hkv, S, S, D, 21)
    slopes = synth.alibi_slopes(Hq) if alibi else None
    ref, ref_lse = oracle.attn(q, k, v, causal=causal, window_left=wl, window_right=wr, softcap=cap,
                               alibi_slopes=slopes, return_lse=True)
    lse = torch.empty(B, Hq, S, dtype=torch.float32, device=cuda_device)
    out = g.attn_fwd(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                     None if slopes is None else slopes.to(cuda_device), causal=causal, window_left=wl,
                     window_right=wr, softcap=cap, lse=lse)
    torch.cuda.synchronize()
    assert out.dtype == F16
    assert g.device_status() == 0
    what = f"fp16 prefill D{D} G{G} causal{causal} w({wl},{wr}) cap{cap} alibi{alibi}"
    check_out(out, ref, F16, what)
    check_lse(lse, ref_lse, F16, what)


def test_fp16_prefill_full_size_sampled(cuda_device):
    """The causal B4 H32/8 S2048 D128 shape in fp16, 512 seeded rows."""
    import tiled_scaled_dot_gb300 as g
    B, Hq, Hkv, S, D = 4, 32, 8, 2048, 128
    q, k, v = _qkv(B, Hq, Hkv, S, S, D, 0)
    out = g.attn_fwd(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device), causal=True)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    rows = torch.unique(synth.randint(512, B * Hq * S, 13, 3))
    ref = oracle.attn(q, k, v, causal=True, rows=rows)
    check_out(out.reshape(-1, D)[rows.to(cuda_device)], ref, F16, "fp16 prefill full size")


@pytest.mark.parametrize("splits", [0, 3])
@pytest.mark.parametrize("cap,alibi", [(None, False), (25.0, True)])
def test_fp16_decode(cuda_device, splits, cap, alibi):
    import tiled_scaled_dot_gb300 as g
    B, Hq, Hkv, Sk, D = 3, 8, 2, 1000, 128
    q, k, v = _qkv(B, Hq, Hkv, 1, Sk, D, 22)
    slopes = synth.alibi_slopes(Hq) if alibi else None
    ref, ref_lse = oracle.decode(q, k, v, softcap=cap, alibi_slopes=slopes, return_lse=True)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=cuda_device)
    out = g.attn_decode(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                        None if slopes is None else slopes.to(cuda_device), softcap=cap, num_splits=splits, lse=lse)
    torch.cuda.synchronize()
    assert out.dtype == F16
    assert g.device_status() == 0
    check_out(out, ref, F16, f"fp16 decode splits{splits}")
    check_lse(lse.view(B, Hq, 1), ref_lse, F16, f"fp16 decode splits{splits}")


@pytest.mark.parametrize("bs", [16, 64])
def test_fp16_paged_decode(cuda_device, bs):
    import tiled_scaled_dot_gb300 as g
    x = make_paged_inputs(3, 8, 2, 128, [100, 1, 777], bs, dtype=F16, seed=23)
    slopes = synth.alibi_slopes(8)
    ref = oracle.attn_paged(x["q"], x["k_cache"], x["v_cache"], x["block_table"], x["context_lens"],
                            alibi_slopes=slopes)
    out = g.attn_decode_paged(*(x[n].to(cuda_device) for n in ("q", "k_cache", "v_cache", "block_table",
                                                               "context_lens")), slopes.to(cuda_device))
    torch.cuda.synchronize()
    assert out.dtype == F16
    assert g.device_status() == 0
    check_out(out, ref, F16, f"fp16 paged bs{bs}")
