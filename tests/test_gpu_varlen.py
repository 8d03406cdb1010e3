"""GPU parity of packed variable-length attention (attn_fwd_varlen through the
C ABI) against the float64 varlen oracle ("gfx942 unified attention",
sections 4-5: packed queries, seqused_k, bottom-right causal alignment)."""
import pytest
import torch

import oracle
import synth
from tests._parity import check_lse, check_out

pytestmark = pytest.mark.gpu


def _cu(lens):
    c = [0]
    for n in lens:
        c.append(c[-1] + n)
    return torch.tensor(c, dtype=torch.int32)


def run_varlen(dev, Hq, Hkv, D, lens_q, lens_k, used=None, causal=True, wl=None, wr=None, softcap=None, alibi=False,
               seed=12, extra_k=0, dtype=torch.bfloat16):
    import tiled_scaled_dot_gb300 as g
    cq, ck = _cu(lens_q), _cu(lens_k)
    total_q, total_k = int(cq[-1]), int(ck[-1]) + extra_k
    q = synth.normal((max(total_q, 1), Hq, D), seed, synth.STREAM_Q, dtype)[:total_q]
    k = synth.normal((total_k, Hkv, D), seed, synth.STREAM_K, dtype)
    v = synth.normal((total_k, Hkv, D), seed, synth.STREAM_V, dtype)
    slopes = synth.alibi_slopes(Hq) if alibi else None
    su = None if used is None else torch.tensor(used, dtype=torch.int32)
    ref, ref_lse = oracle.attn_varlen(q, k, v, cq, ck, seqused_k=su, causal=causal, window_left=wl, window_right=wr,
                                      softcap=softcap, alibi_slopes=slopes, return_lse=True)
    lse = torch.empty(Hq, total_q, dtype=torch.float32, device=dev)
    out = g.attn_fwd_varlen(q.to(dev), k.to(dev), v.to(dev), cq.to(dev), ck.to(dev), max(lens_q),
                            None if su is None else su.to(dev), None if slopes is None else slopes.to(dev),
                            causal=causal, window_left=wl, window_right=wr, softcap=softcap, lse=lse)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    what = f"varlen {dtype} Hq{Hq} Hkv{Hkv} D{D} q{lens_q[:5]} k{lens_k[:5]} c{causal} w({wl},{wr}) cap{softcap} alibi{alibi}"
    assert out.dtype == dtype
    check_out(out, ref, dtype, what)
    check_lse(lse, ref_lse, dtype, what)
    return out


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 4])
@pytest.mark.parametrize("causal", [True, False])
def test_varlen_equal_lengths(cuda_device, D, G, causal):
    lens = [1, 100, 128, 129, 700]
    run_varlen(cuda_device, 2 * G, 2, D, lens, lens, causal=causal)


@pytest.mark.parametrize("G", [1, 2])
def test_varlen_bottom_right_causal(cuda_device, G):
    """Fewer queries than keys (prefill of a chunk after cached history, or
    decode rows): query i sits at kv_len - q_len + i."""
    run_varlen(cuda_device, 2 * G, 2, 128, [1, 64, 300, 129], [1000, 64, 2000, 130], causal=True, alibi=True)


@pytest.mark.parametrize("cap,alibi,wl,wr", [(30.0, False, None, None), (None, True, 200, 0), (25.0, True, 100, 50),
                                             (None, False, 0, 0)])
def test_varlen_flags(cuda_device, cap, alibi, wl, wr):
    run_varlen(cuda_device, 4, 2, 64, [257, 3, 640], [300, 3, 1024], causal=True, wl=wl, wr=wr, softcap=cap,
               alibi=alibi)


def test_varlen_seqused_k_and_empty_sequences(cuda_device):
    """Live-key prefixes shorter than the packed key ranges, a sequence with no
    queries, one with no live keys, and more queries than keys (rows before the
    first key are zero)."""
    run_varlen(cuda_device, 4, 4, 128, [50, 0, 20, 300], [400, 10, 30, 200], used=[333, 10, 0, 120],
               causal=True, extra_k=37)


def test_varlen_equal_lengths_match_dense_kernel_bitwise(cuda_device):
    """B equal-length sequences packed: the same rows, tiles and arithmetic as
    the dense kernel on [B, H, S, D], so the outputs are bitwise equal."""
    import tiled_scaled_dot_gb300 as g
    B, Hq, Hkv, S, D = 3, 8, 2, 384, 128
    q = synth.normal((B, Hq, S, D), 9, synth.STREAM_Q, torch.bfloat16).to(cuda_device)
    k = synth.normal((B, Hkv, S, D), 9, synth.STREAM_K, torch.bfloat16).to(cuda_device)
    v = synth.normal((B, Hkv, S, D), 9, synth.STREAM_V, torch.bfloat16).to(cuda_device)
    dense = g.attn_fwd(q, k, v, causal=True)
    pack = lambda t: t.permute(0, 2, 1, 3).reshape(B * S, t.shape[1], D).contiguous()
    cu = _cu([S] * B).to(cuda_device)
    out = g.attn_fwd_varlen(pack(q), pack(k), pack(v), cu, cu, S, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(out, pack(dense))
    assert g.device_status() == 0


def test_varlen_many_sequences_mixed_lengths(cuda_device):
    """A serving-like mix: 24 sequences of 1 .. 2048 queries, GQA 4."""
    lens = (1 + synth.randint(24, 2048, 3, 6)).tolist()
    run_varlen(cuda_device, 16, 4, 128, lens, lens, causal=True)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("flags", [dict(), dict(softcap=20.0, alibi=True, wl=300, wr=0)],
                         ids=["plain", "softcap-alibi-window"])
def test_varlen_fp16(cuda_device, D, flags):
    """fp16 packed sequences: fp16 operands and P on the tensor cores, fp16 output
    (attention.fkc.md lists F16 among the input types); the 16-bit bars."""
    run_varlen(cuda_device, 8, 2, D, [1, 300, 129, 700], [1, 300, 200, 700], causal=True, dtype=torch.float16,
               **flags)
    lens = (1 + synth.randint(12, 1500, 4, 6)).tolist()
    run_varlen(cuda_device, 8, 4, D, lens, lens, causal=True, dtype=torch.float16, **flags)
