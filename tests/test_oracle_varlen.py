"""Pins of the packed variable-length oracle ("gfx942 unified attention",
sections 4-5) against the independent C oracle of the dense definition,
closed forms and invariances."""
import math

import pytest
import torch

import oracle
import synth


def _rand(shape, stream, seed=31):
    return synth.normal(shape, seed, stream, torch.float64)


def _pack(x):
    """[1, H, S, D] -> [S, H, D]"""
    return x[0].permute(1, 0, 2).contiguous()


@pytest.mark.parametrize("causal,wl,wr", [(False, None, None), (True, None, None), (True, 5, None),
                                          (False, 3, 4)])
@pytest.mark.parametrize("cap,alibi", [(None, False), (20.0, True)])
def test_equal_lengths_equal_dense_oracle(causal, wl, wr, cap, alibi):
    """q_len == kv_len for every sequence: bottom-right is top-left, so each
    packed sequence equals the dense C oracle on that sequence alone."""
    Hq, Hkv, D = 4, 2, 8
    lens = [17, 1, 40]
    cu = torch.tensor([0] + [sum(lens[:i + 1]) for i in range(len(lens))])
    q, k, v = _rand((cu[-1].item(), Hq, D), 0), _rand((cu[-1].item(), Hkv, D), 1), _rand((cu[-1].item(), Hkv, D), 2)
    slopes = synth.alibi_slopes(Hq) if alibi else None
    out, lse = oracle.attn_varlen(q, k, v, cu, cu, causal=causal, window_left=wl, window_right=wr, softcap=cap,
                                  alibi_slopes=slopes, return_lse=True)
    for b, n in enumerate(lens):
        a, e = int(cu[b]), int(cu[b + 1])
        qd = q[a:e].permute(1, 0, 2)[None]
        kd = k[a:e].permute(1, 0, 2)[None]
        vd = v[a:e].permute(1, 0, 2)[None]
        ref, ref_lse = oracle.attn(qd, kd, vd, causal=causal, window_left=wl, window_right=wr, softcap=cap,
                                   alibi_slopes=slopes, return_lse=True)
        assert (out[a:e] - _pack(ref)).abs().max().item() < 1e-12
        assert (lse[:, a:e] - ref_lse[0]).abs().max().item() < 1e-12


@pytest.mark.parametrize("q_len", [1, 7, 30])
def test_bottom_right_causal_is_the_tail_of_a_dense_causal_problem(q_len):
    """q_len < kv_len: query i sits at kv_len - q_len + i, so the rows equal the
    last q_len rows of the dense causal problem of length kv_len (with ALiBi
    and a left window relative to the same positions)."""
    Hq, Hkv, D, kv_len = 2, 1, 8, 30
    qfull = _rand((1, Hq, kv_len, D), 0)
    kd, vd = _rand((1, Hkv, kv_len, D), 1), _rand((1, Hkv, kv_len, D), 2)
    slopes = synth.alibi_slopes(Hq)
    ref = oracle.attn(qfull, kd, vd, causal=True, window_left=9, alibi_slopes=slopes)[:, :, kv_len - q_len:]
    out = oracle.attn_varlen(_pack(qfull[:, :, kv_len - q_len:]), _pack(kd), _pack(vd), torch.tensor([0, q_len]),
                             torch.tensor([0, kv_len]), causal=True, window_left=9, alibi_slopes=slopes)
    assert (out - _pack(ref)).abs().max().item() < 1e-12


def test_seqused_k_ignores_the_keys_after_it():
    """Keys past seqused_k (NaN planted) have no effect, and the sequence is
    the one with kv_len = seqused_k."""
    Hq, Hkv, D = 2, 2, 8
    cq, ck = torch.tensor([0, 5, 9]), torch.tensor([0, 20, 32])
    used = torch.tensor([12, 3])
    q, k, v = _rand((9, Hq, D), 0), _rand((32, Hkv, D), 1), _rand((32, Hkv, D), 2)
    ref = oracle.attn_varlen(q, k[torch.tensor(list(range(12)) + list(range(20, 23)))],
                             v[torch.tensor(list(range(12)) + list(range(20, 23)))], cq, torch.tensor([0, 12, 15]),
                             causal=True)
    k2, v2 = k.clone(), v.clone()
    k2[12:20] = float("nan")
    v2[12:20] = float("nan")
    k2[23:] = float("nan")
    v2[23:] = float("nan")
    out = oracle.attn_varlen(q, k2, v2, cq, ck, seqused_k=used, causal=True)
    assert torch.equal(out, ref)


def test_rows_without_keys_are_zero():
    """A sequence with no live keys, and causal rows of a sequence with more
    queries than keys (abs_i < 0), are zero rows with lse -inf."""
    Hq, Hkv, D = 2, 1, 4
    cq, ck = torch.tensor([0, 3, 8]), torch.tensor([0, 0, 2])
    q, k, v = _rand((8, Hq, D), 0), _rand((2, Hkv, D), 1), _rand((2, Hkv, D), 2)
    out, lse = oracle.attn_varlen(q, k, v, cq, ck, causal=True, return_lse=True)
    assert torch.equal(out[:3], torch.zeros_like(out[:3]))
    # sequence 1: q_len 5, kv_len 2 -> abs = -3, -2, -1, 0, 1: the first three rows see no key
    assert torch.equal(out[3:6], torch.zeros_like(out[3:6]))
    assert torch.isneginf(lse[:, :6]).all()
    assert torch.isfinite(lse[:, 6:]).all()
    # row abs 0 sees key 0 only: its output is V[key 0]
    assert (out[6] - v[0, 0]).abs().max().item() < 1e-12


def test_closed_form_two_keys():
    """One query at abs 1 (q_len 1, kv_len 2), scores 0 and ln 3: weights 1/4, 3/4."""
    q = torch.ones(1, 1, 1, dtype=torch.float64)
    k = torch.tensor([[[0.0]], [[math.log(3.0)]]], dtype=torch.float64)
    v = torch.tensor([[[2.0]], [[6.0]]], dtype=torch.float64)
    out, lse = oracle.attn_varlen(q, k, v, torch.tensor([0, 1]), torch.tensor([0, 2]), scale=1.0, causal=True,
                                  return_lse=True)
    assert abs(out.item() - 5.0) < 1e-12
    assert abs(lse.item() - math.log(4.0)) < 1e-12
