"""Pins of the paged-cache oracle (attention.fkc.md, "attention_paged_naive")
against things other than itself: the independent C oracle of the contiguous
definition, closed forms, and invariances the contract fixes."""
import math

import pytest
import torch

import oracle
import synth
from synth.workloads import make_paged_inputs


def _rand(shape, stream, seed=21):
    return synth.normal(shape, seed, stream, torch.float64)


def _identity_pool(k, bs):
    """[B, Hkv, Sk, D] -> pool [B * Sk / bs, bs, Hkv, D] with sequence b's blocks in order."""
    B, Hkv, Sk, D = k.shape
    return k.permute(0, 2, 1, 3).reshape(B * Sk // bs, bs, Hkv, D).contiguous()


def _identity_table(B, Sk, bs):
    nb = Sk // bs
    return torch.arange(B * nb, dtype=torch.int32).reshape(B, nb)


@pytest.mark.parametrize("bs", [16, 64])
@pytest.mark.parametrize("cap,alibi", [(None, False), (30.0, False), (None, True), (20.0, True)])
def test_identity_table_equals_contiguous_decode(bs, cap, alibi):
    """With blocks laid out in order and context = Sk, paged decode is the
    contiguous decode: both put the query at position Sk - 1, so outputs and
    lse agree (the paged oracle is torch float64 code, the contiguous decode
    the C oracle)."""
    B, Hq, Hkv, Sk, D = 2, 4, 2, 128, 16
    q, k, v = _rand((B, Hq, 1, D), 0), _rand((B, Hkv, Sk, D), 1), _rand((B, Hkv, Sk, D), 2)
    slopes = synth.alibi_slopes(Hq) if alibi else None
    for wl in (None, 0, 37, 200):
        ref, ref_lse = oracle.decode(q, k, v, softcap=cap, alibi_slopes=slopes, window_left=wl, return_lse=True)
        out, lse = oracle.attn_paged(q, _identity_pool(k, bs), _identity_pool(v, bs), _identity_table(B, Sk, bs),
                                     torch.full((B,), Sk, dtype=torch.int32), softcap=cap, alibi_slopes=slopes,
                                     window_left=wl, return_lse=True)
        assert (out - ref).abs().max().item() < 1e-12
        assert (lse - ref_lse).abs().max().item() < 1e-10


def test_implicit_causal_is_bottom_right_causal():
    """Sq > 1: query q_pos sits at abs_pos = ctx - Sq + q_pos, so the paged rows
    equal the last Sq rows of a causal contiguous problem of length ctx (C oracle)."""
    B, Hq, Hkv, ctx, D, Sq, bs = 1, 2, 1, 96, 8, 5, 32
    k, v = _rand((B, Hkv, ctx, D), 1), _rand((B, Hkv, ctx, D), 2)
    qfull = _rand((B, Hq, ctx, D), 0)
    slopes = synth.alibi_slopes(Hq)
    ref = oracle.attn(qfull, k, v, causal=True, alibi_slopes=slopes)[:, :, ctx - Sq:, :]
    out = oracle.attn_paged(qfull[:, :, ctx - Sq:, :].contiguous(), _identity_pool(k, bs), _identity_pool(v, bs),
                            _identity_table(B, ctx, bs), torch.tensor([ctx], dtype=torch.int32),
                            alibi_slopes=slopes)
    assert (out - ref).abs().max().item() < 1e-12


def test_block_placement_does_not_matter_bitwise():
    """Moving physical blocks (and the table with them) changes nothing."""
    x = make_paged_inputs(3, 4, 2, 16, [70, 1, 130], 16, dtype=torch.float64, seed=5)
    ref = oracle.attn_paged(x["q"], x["k_cache"], x["v_cache"], x["block_table"], x["context_lens"])
    perm = torch.randperm(x["num_blocks"], generator=torch.Generator().manual_seed(3))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(perm.numel())
    k2 = torch.empty_like(x["k_cache"])
    v2 = torch.empty_like(x["v_cache"])
    k2[inv] = x["k_cache"]
    v2[inv] = x["v_cache"]
    bt = x["block_table"].clone().long()
    live = bt < x["num_blocks"]
    bt[live] = inv[bt[live]]
    out = oracle.attn_paged(x["q"], k2, v2, bt.to(torch.int32), x["context_lens"])
    assert torch.equal(out, ref)


def test_keys_past_the_context_have_no_effect():
    """NaN planted in the pool rows after a sequence's last key and in spare
    blocks: outputs are unchanged bitwise."""
    bs = 16
    x = make_paged_inputs(2, 2, 1, 8, [21, 40], bs, dtype=torch.float64, seed=8)
    ref = oracle.attn_paged(x["q"], x["k_cache"], x["v_cache"], x["block_table"], x["context_lens"])
    k, v = x["k_cache"].clone(), x["v_cache"].clone()
    used = set()
    for b, ctx in enumerate(x["context_lens"].tolist()):
        for kp in range(((ctx + bs - 1) // bs) * bs):
            blk = int(x["block_table"][b, kp // bs])
            if kp >= ctx:
                k[blk, kp % bs] = float("nan")
                v[blk, kp % bs] = float("nan")
            used.add(blk)
    for blk in range(x["num_blocks"]):
        if blk not in used:
            k[blk] = float("nan")
            v[blk] = float("nan")
    out = oracle.attn_paged(x["q"], k, v, x["block_table"], x["context_lens"])
    assert torch.equal(out, ref)


def test_empty_context_is_a_zero_row():
    x = make_paged_inputs(2, 2, 2, 8, [0, 5], 16, dtype=torch.float64, seed=9)
    out, lse = oracle.attn_paged(x["q"], x["k_cache"], x["v_cache"], x["block_table"], x["context_lens"],
                                 return_lse=True)
    assert torch.equal(out[0], torch.zeros_like(out[0]))
    assert torch.isinf(lse[0]).all() and (lse[0] < 0).all()
    assert torch.isfinite(out[1]).all()


def test_closed_form_two_keys():
    """Two keys in two different physical blocks (block_size 1): scores 0 and
    ln 3 give weights 1/4 and 3/4; ALiBi slope 1 with abs_pos = 1 adds -1 to
    key 0 and 0 to key 1."""
    D = 1
    q = torch.ones(1, 1, 1, D, dtype=torch.float64)
    k = torch.zeros(5, 1, 1, D, dtype=torch.float64)
    v = torch.zeros(5, 1, 1, D, dtype=torch.float64)
    k[3, 0, 0, 0], v[3, 0, 0, 0] = 0.0, 2.0          # logical key 0
    k[1, 0, 0, 0], v[1, 0, 0, 0] = math.log(3.0), 6.0  # logical key 1
    bt = torch.tensor([[3, 1]], dtype=torch.int32)
    cl = torch.tensor([2], dtype=torch.int32)
    out, lse = oracle.attn_paged(q, k, v, bt, cl, scale=1.0, return_lse=True)
    assert abs(out.item() - (0.25 * 2.0 + 0.75 * 6.0)) < 1e-12
    assert abs(lse.item() - math.log(4.0)) < 1e-12
    # with ALiBi slope 1: scores -1 and ln 3 (the scale is exact in float32 only for 1.0)
    slopes = torch.ones(1, dtype=torch.float32)
    out, lse = oracle.attn_paged(q, k, v, bt, cl, scale=1.0, alibi_slopes=slopes, return_lse=True)
    w0, w1 = math.exp(-1.0), 3.0
    assert abs(out.item() - (w0 * 2.0 + w1 * 6.0) / (w0 + w1)) < 1e-12
    assert abs(lse.item() - math.log(w0 + w1)) < 1e-12


def test_gqa_head_mapping():
    """Query head h reads kv head h // (Hq / Hkv): with kv head 1's values all
    equal to 5, heads 2 and 3 (group 2) output 5 exactly."""
    x = make_paged_inputs(1, 4, 2, 8, [33], 16, dtype=torch.float64, seed=4)
    v = x["v_cache"].clone()
    v[:, :, 1, :] = 5.0
    out = oracle.attn_paged(x["q"], x["k_cache"], v, x["block_table"], x["context_lens"])
    assert torch.allclose(out[0, 2:], torch.full_like(out[0, 2:], 5.0), atol=1e-12, rtol=0)


def test_rejects_out_of_range_blocks():
    x = make_paged_inputs(1, 2, 1, 8, [20], 16, dtype=torch.float64, seed=2)
    bt = x["block_table"].clone()
    bt[0, 1] = x["num_blocks"]
    with pytest.raises(ValueError):
        oracle.attn_paged(x["q"], x["k_cache"], x["v_cache"], bt, x["context_lens"])
