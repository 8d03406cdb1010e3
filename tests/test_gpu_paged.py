"""GPU parity of the paged-cache decode entry (attn_decode_paged through the C
ABI) against the float64 paged oracle (attention.fkc.md,
"attention_paged_naive")."""
import pytest
import torch

import oracle
import synth
from synth.workloads import make_paged_inputs
from tests._parity import check_lse, check_out

pytestmark = pytest.mark.gpu


def run_paged(dev, B, Hq, Hkv, D, ctx, bs, splits=0, softcap=None, alibi=False, seed=3, extra_blocks=0):
    import tiled_scaled_dot_gb300 as g
    x = make_paged_inputs(B, Hq, Hkv, D, ctx, bs, seed=seed)
    if extra_blocks:  # a wider table whose unused entries must never be read
        bt = torch.full((B, x["block_table"].shape[1] + extra_blocks), x["num_blocks"] + 7, dtype=torch.int32)
        bt[:, :x["block_table"].shape[1]] = x["block_table"]
        x["block_table"] = bt
    slopes = synth.alibi_slopes(Hq) if alibi else None
    ref, ref_lse = oracle.attn_paged(x["q"], x["k_cache"], x["v_cache"], x["block_table"], x["context_lens"],
                                     softcap=softcap, alibi_slopes=slopes, return_lse=True)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)
    out = g.attn_decode_paged(x["q"].to(dev), x["k_cache"].to(dev), x["v_cache"].to(dev),
                              x["block_table"].to(dev), x["context_lens"].to(dev),
                              None if slopes is None else slopes.to(dev), softcap=softcap, num_splits=splits, lse=lse)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    what = f"paged B{B} Hq{Hq} Hkv{Hkv} D{D} ctx{list(ctx)[:4]} bs{bs} splits{splits} cap{softcap} alibi{alibi}"
    check_out(out, ref, torch.bfloat16, what)
    check_lse(lse.view(B, Hq, 1), ref_lse, torch.bfloat16, what)
    return out


@pytest.mark.parametrize("bs", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("D", [64, 128])
def test_paged_block_sizes(cuda_device, bs, D):
    run_paged(cuda_device, 3, 8, 2, D, [100, 1, 333], bs)


@pytest.mark.parametrize("splits", [0, 1, 2, 5])
@pytest.mark.parametrize("cap,alibi", [(None, False), (30.0, False), (None, True), (25.0, True)])
def test_paged_flags_and_splits(cuda_device, splits, cap, alibi):
    run_paged(cuda_device, 2, 8, 2, 128, [700, 129], 32, splits=splits, softcap=cap, alibi=alibi)


@pytest.mark.parametrize("G", [1, 2, 3, 4, 8])
def test_paged_group_sizes(cuda_device, G):
    run_paged(cuda_device, 2, 2 * G, 2, 128, [257, 64], 64)


def test_paged_empty_and_ragged_contexts(cuda_device):
    """Context 0 (zero row, lse -inf), 1 key, exact block multiples, a ragged
    tail, and a table wider than any context (unused entries never read)."""
    run_paged(cuda_device, 5, 4, 4, 64, [0, 1, 64, 65, 1000], 64, alibi=True, extra_blocks=3)


def test_paged_identity_layout_equals_contiguous_decode(cuda_device):
    """Blocks laid out in order with a full context: the same kernel arithmetic
    as the contiguous decode, so the outputs are bitwise equal."""
    import tiled_scaled_dot_gb300 as g
    B, Hq, Hkv, Sk, D, bs = 2, 8, 2, 512, 128, 64
    q = synth.normal((B, Hq, 1, D), 4, synth.STREAM_Q, torch.bfloat16).to(cuda_device)
    k = synth.normal((B, Hkv, Sk, D), 4, synth.STREAM_K, torch.bfloat16).to(cuda_device)
    v = synth.normal((B, Hkv, Sk, D), 4, synth.STREAM_V, torch.bfloat16).to(cuda_device)
    pool = lambda t: t.permute(0, 2, 1, 3).reshape(B * Sk // bs, bs, Hkv, D).contiguous()
    table = torch.arange(B * Sk // bs, dtype=torch.int32, device=cuda_device).reshape(B, Sk // bs)
    lens = torch.full((B,), Sk, dtype=torch.int32, device=cuda_device)
    a = g.attn_decode(q, k, v, num_splits=4)
    b = g.attn_decode_paged(q, pool(k), pool(v), table, lens, num_splits=4)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert g.device_status() == 0


def test_paged_bad_block_index_sets_status(cuda_device):
    """A physical block index past the pool is reported in the device status
    word (bit 10) without reading outside the pool; the context stays usable."""
    import tiled_scaled_dot_gb300 as g
    x = make_paged_inputs(2, 4, 2, 64, [200, 90], 64, seed=6)
    bt = x["block_table"].clone()
    bt[0, 1] = x["num_blocks"] + 100
    g.device_status()
    g.attn_decode_paged(x["q"].to(cuda_device), x["k_cache"].to(cuda_device), x["v_cache"].to(cuda_device),
                        bt.to(cuda_device), x["context_lens"].to(cuda_device))
    st = g.device_status()
    assert st & (1 << 10), f"status {st:#x}"
    run_paged(cuda_device, 2, 4, 2, 64, [200, 90], 64, seed=6)


def test_paged_reruns_are_bitwise_identical(cuda_device):
    import tiled_scaled_dot_gb300 as g
    x = make_paged_inputs(4, 8, 2, 128, [1500, 3, 800, 4096], 16, seed=7)
    args = [x[k].to(cuda_device) for k in ("q", "k_cache", "v_cache", "block_table", "context_lens")]
    a = g.attn_decode_paged(*args)
    b = g.attn_decode_paged(*args)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_paged_serving_shape_sampled(cuda_device):
    """The benchmark's paged workload shape (B64 Hq32 Hkv8 D128, contexts of
    4096..8192 keys, block size 64), every row against the oracle."""
    B = 64
    ctx = (4096 + synth.randint(B, 4097, 0, 5)).tolist()
    run_paged(cuda_device, B, 32, 8, 128, ctx, 64, seed=0)
