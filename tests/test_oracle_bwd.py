"""Pins of the float64 backward oracle (attention.fkc.md, "attention_flash_backward").

The backward is pinned to things other than itself:
  * central finite differences of the forward oracle (``oracle.attn``, itself
    pinned by test_oracle_pins.py) on tiny float64 problems, for every
    element of dQ, dK and dV, with each flag the forward has;
  * closed forms with uniform scores (Q = 0): dV and dK exactly;
  * invariants of the softmax Jacobian: without softcap the rows of dS sum to
    zero, so the keys' dK sum to zero, and the keys' dV sum to the live rows' dO;
  * a fully-masked row contributes nothing and gets a zero dQ row;
  * GQA: the grouped result equals the per-head result with K and V repeated,
    with dK / dV summed over the group.
"""
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


def _inputs(B, Hq, Hkv, Sq, Sk, D, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, Sq, D, generator=g, dtype=torch.float64)
    k = torch.randn(B, Hkv, Sk, D, generator=g, dtype=torch.float64)
    v = torch.randn(B, Hkv, Sk, D, generator=g, dtype=torch.float64)
    do = torch.randn(B, Hq, Sq, D, generator=g, dtype=torch.float64)
    return q, k, v, do


def _loss(q, k, v, do, kw):
    # L = sum(O * dO), so dL/dX is the backward of dO through the forward
    return float((oracle.attn(q, k, v, **kw) * do).sum())


def _finite_diff(q, k, v, do, kw, eps=1e-6):
    grads = []
    for idx in range(3):
        xs = [q.clone(), k.clone(), v.clone()]
        x = xs[idx]
        gr = torch.zeros_like(x)
        flat, gflat = x.view(-1), gr.view(-1)
        for e in range(flat.numel()):
            x0 = float(flat[e])
            flat[e] = x0 + eps
            lp = _loss(*xs, do, kw)
            flat[e] = x0 - eps
            lm = _loss(*xs, do, kw)
            flat[e] = x0
            gflat[e] = (lp - lm) / (2 * eps)
        grads.append(gr)
    return grads


CASES = [
    # (B, Hq, Hkv, Sq, Sk, D), flags
    ((1, 2, 1, 5, 6, 4), dict(causal=True)),
    ((1, 2, 1, 5, 6, 4), dict(causal=True, softcap=2.5)),
    ((1, 2, 2, 4, 7, 3), dict(alibi=True)),
    ((2, 4, 2, 6, 6, 4), dict(causal=True, window_left=2, softcap=4.0, alibi=True)),
    ((1, 2, 1, 6, 5, 4), dict(window_left=1, window_right=1)),
    ((2, 2, 1, 5, 6, 3), dict(rowb=True, softcap=3.0)),
]


def _kw(flags, Hq, B, Sq, Sk, seed=7):
    kw = dict(scale=0.37)
    for name in ("causal", "window_left", "window_right", "softcap"):
        if name in flags:
            kw[name] = flags[name]
    if flags.get("alibi"):
        kw["alibi_slopes"] = torch.tensor([0.5 ** (h + 1) for h in range(Hq)], dtype=torch.float32)
    if flags.get("rowb"):
        g = torch.Generator().manual_seed(seed)
        lo = torch.randint(0, Sk, (B, Sq), generator=g)
        hi = torch.minimum(lo + torch.randint(0, Sk, (B, Sq), generator=g), torch.full_like(lo, Sk - 1))
        rb = torch.stack([lo, hi], dim=-1).to(torch.int32)
        rb[0, 1] = torch.tensor([1, 0], dtype=torch.int32)  # one empty row
        kw["row_kv_bounds"] = rb
    return kw


@pytest.mark.parametrize("shape,flags", CASES)
def test_bwd_matches_finite_differences_of_forward(shape, flags):
    B, Hq, Hkv, Sq, Sk, D = shape
    q, k, v, do = _inputs(*shape, seed=sum(shape))
    kw = _kw(flags, Hq, B, Sq, Sk)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, **kw)
    fq, fk, fv = _finite_diff(q, k, v, do, kw)
    for got, ref in ((dq, fq), (dk, fk), (dv, fv)):
        assert torch.allclose(got, ref, atol=1e-7, rtol=1e-6), (got - ref).abs().max()


def test_bwd_uniform_scores_closed_form():
    # Q = 0: every admissible score is 0, so P = 1 / Sk on every row.
    B, Hq, Hkv, Sq, Sk, D = 1, 4, 2, 5, 8, 6
    _, k, v, do = _inputs(B, Hq, Hkv, Sq, Sk, D, seed=3)
    q = torch.zeros(B, Hq, Sq, D, dtype=torch.float64)
    sc = 0.25
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, scale=sc)
    G = Hq // Hkv
    for g in range(Hkv):
        grp = do[0, g * G:(g + 1) * G]  # [G, Sq, D]
        # dV[j] = sum_i P dO[i] = (1 / Sk) sum over the group's rows, the same for every key
        want = grp.sum(dim=(0, 1)) / Sk
        assert torch.allclose(dv[0, g], want.expand(Sk, D), atol=1e-14)
        # dK[j] = scale sum_i dS[i, j] Q[i] = 0
        assert torch.all(dk[0, g] == 0)
        for hh in range(G):
            h = g * G + hh
            dP = do[0, h] @ v[0, g].T  # [Sq, Sk]
            dS = (dP - dP.mean(dim=1, keepdim=True)) / Sk
            assert torch.allclose(dq[0, h], sc * dS @ k[0, g], atol=1e-13)


@pytest.mark.parametrize("flags", [dict(causal=True, alibi=True), dict(window_left=1, rowb=True)])
def test_bwd_softmax_jacobian_invariants(flags):
    B, Hq, Hkv, Sq, Sk, D = 2, 4, 2, 9, 9, 5
    q, k, v, do = _inputs(B, Hq, Hkv, Sq, Sk, D, seed=11)
    kw = _kw(flags, Hq, B, Sq, Sk)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, **kw)
    # rows of dS sum to zero -> the keys' dK sum to zero
    assert dk.sum(dim=2).abs().max() < 1e-12
    # sum over keys of dV = sum over live rows of dO (rows of P sum to one);
    # a row is live when the forward's lse is finite
    _, lse = oracle.attn(q, k, v, return_lse=True, **kw)
    live = torch.isfinite(lse)
    G = Hq // Hkv
    dol = torch.where(live[..., None], do, torch.zeros_like(do))
    want = dol.view(B, Hkv, G, Sq, D).sum(dim=(2, 3))
    assert torch.allclose(dv.sum(dim=2), want, atol=1e-12)


def test_bwd_fully_masked_row_contributes_nothing():
    B, Hq, Hkv, Sq, Sk, D = 1, 2, 1, 6, 6, 4
    q, k, v, do = _inputs(B, Hq, Hkv, Sq, Sk, D, seed=5)
    rb = torch.tensor([[[0, 5]] * Sq], dtype=torch.int32)
    rb[0, 3] = torch.tensor([4, 2])  # row 3 admits no key
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal=True, row_kv_bounds=rb)
    assert torch.all(dq[0, :, 3] == 0)
    do2 = do.clone()
    do2[0, :, 3] = 100.0
    q2 = q.clone()
    q2[0, :, 3] = -7.0
    dq2, dk2, dv2 = oracle.attn_bwd(q2, k, v, do2, causal=True, row_kv_bounds=rb)
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2)
    assert torch.equal(dq[0, :, :3], dq2[0, :, :3]) and torch.equal(dq[0, :, 4:], dq2[0, :, 4:])


def test_bwd_gqa_equals_repeated_heads_summed():
    B, Hq, Hkv, Sq, Sk, D = 2, 6, 2, 5, 7, 4
    q, k, v, do = _inputs(B, Hq, Hkv, Sq, Sk, D, seed=9)
    kw = dict(causal=True, softcap=3.0, alibi_slopes=torch.linspace(0.1, 0.6, Hq, dtype=torch.float32))
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, **kw)
    G = Hq // Hkv
    kr, vr = k.repeat_interleave(G, dim=1), v.repeat_interleave(G, dim=1)
    dq_r, dk_r, dv_r = oracle.attn_bwd(q, kr, vr, do, **kw)
    assert torch.equal(dq, dq_r)
    assert torch.allclose(dk, dk_r.view(B, Hkv, G, Sk, D).sum(dim=2), atol=1e-13)
    assert torch.allclose(dv, dv_r.view(B, Hkv, G, Sk, D).sum(dim=2), atol=1e-13)
