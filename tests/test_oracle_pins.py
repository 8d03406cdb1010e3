"""Pins for the CPU oracle, against things other than itself.

Each test ties the oracle to a fact the pages or plain mathematics fix:
closed forms worked by hand, a brute force written separately in plain Python,
library routines on special cases, and invariants.  A plausible slip in the
oracle (a dropped scale, softcap after ALiBi, a flipped ALiBi sign, h % Hkv
instead of h / G, an off-by-one window, a missing max subtraction, a wrong
fully-masked row) fails at least one of them.
"""
import itertools
import math

import pytest
import torch

import oracle
import synth

NEG_INF = float("-inf")


def _rand(shape, stream, dtype=torch.float64, seed=11):
    return synth.normal(shape, seed, stream, dtype=dtype)


# --------------------------------------------------------------------------
# Closed forms worked by hand (definition: attention.fkc.md, attention_naive;
# softmax: "gfx942 unified attention", sections 1-2).
# --------------------------------------------------------------------------

def test_closed_form_two_keys_log3():
    # scores 0 and ln 3 -> weights 1/4, 3/4; O = 4/4 + 3*8/4 = 7; lse = ln 4.
    q = torch.tensor([1.0], dtype=torch.float64).view(1, 1, 1, 1)
    k = torch.tensor([0.0, math.log(3.0)], dtype=torch.float64).view(1, 1, 2, 1)
    v = torch.tensor([4.0, 8.0], dtype=torch.float64).view(1, 1, 2, 1)
    out, lse = oracle.attn(q, k, v, scale=1.0, return_lse=True)
    assert abs(out.item() - 7.0) < 1e-14
    assert abs(lse.item() - math.log(4.0)) < 1e-14


def test_closed_form_softcap_then_alibi():
    # qi = 1 attends keys 0, 1 (non-causal, Sk = 2), cap c = 1, slope 1.
    # key 0: raw 0 -> tanh(0) = 0, bias (0 - 1) = -1 -> s0 = -1
    # key 1: raw 100 -> tanh(100) = 1, bias 0        -> s1 = 1
    # O with v = (0, 1) is e / (e^-1 + e) = e^2 / (1 + e^2).
    # (ALiBi first, then cap, would give s0 = tanh(-1) instead.)
    q = torch.tensor([0.0, 1.0], dtype=torch.float64).view(1, 1, 2, 1)
    k = torch.tensor([0.0, 100.0], dtype=torch.float64).view(1, 1, 2, 1)
    v = torch.tensor([0.0, 1.0], dtype=torch.float64).view(1, 1, 2, 1)
    slopes = torch.tensor([1.0], dtype=torch.float32)
    out = oracle.attn(q, k, v, scale=1.0, softcap=1.0, alibi_slopes=slopes)
    e2 = math.exp(2.0)
    assert abs(out[0, 0, 1, 0].item() - e2 / (1.0 + e2)) < 1e-14


def test_closed_form_alibi_sign():
    # q = 0, slope ln 2, query 0 over keys 0..2: bias kj*ln2 -> weights 1:2:4.
    # v = (1, 0, 0) -> 1/7.  (-slope*|kj-qi| or the opposite sign would give 4/7.)
    q = torch.zeros(1, 1, 1, 1, dtype=torch.float64)
    k = torch.zeros(1, 1, 3, 1, dtype=torch.float64)
    v = torch.tensor([1.0, 0.0, 0.0], dtype=torch.float64).view(1, 1, 3, 1)
    ln2 = float(torch.tensor(math.log(2.0), dtype=torch.float32))
    slopes = torch.tensor([ln2], dtype=torch.float32)
    out = oracle.attn(q, k, v, scale=1.0, alibi_slopes=slopes)
    w = [math.exp(ln2 * j) for j in range(3)]
    assert abs(out.item() - w[0] / sum(w)) < 1e-14
    assert abs(out.item() - 1.0 / 7.0) < 1e-7


@pytest.mark.parametrize("causal,wl,wr,expect", [
    (True, 1, None, [1.0, 1.5, 3.0, 6.0]),          # keys [qi-1, qi]
    (False, 0, 1, [1.5, 3.0, 6.0, 8.0]),            # keys [qi, qi+1]
    (True, None, None, [1.0, 1.5, 7 / 3, 15 / 4]),  # keys [0, qi]
    (False, 0, 0, [1.0, 2.0, 4.0, 8.0]),            # key qi only
    (False, None, None, [15 / 4] * 4),              # every key
])
def test_closed_form_windows(causal, wl, wr, expect):
    # q = 0 makes every admissible score 0, so O is the mean of admitted V rows.
    q = torch.zeros(1, 1, 4, 1, dtype=torch.float64)
    k = torch.zeros(1, 1, 4, 1, dtype=torch.float64)
    v = torch.tensor([1.0, 2.0, 4.0, 8.0], dtype=torch.float64).view(1, 1, 4, 1)
    out = oracle.attn(q, k, v, scale=1.0, causal=causal, window_left=wl, window_right=wr)
    assert out.view(-1).tolist() == pytest.approx(expect, abs=1e-15)


def test_closed_form_gqa_mapping():
    # Hq = 4, Hkv = 2, one key: head h reads kv head h // 2 -> (10, 10, 20, 20).
    q = _rand((1, 4, 1, 3), 0)
    k = _rand((1, 2, 1, 3), 1)
    v = torch.tensor([10.0, 20.0], dtype=torch.float64).view(1, 2, 1, 1).expand(1, 2, 1, 3).contiguous()
    out = oracle.attn(q, k, v)
    assert out[0, :, 0, 0].tolist() == [10.0, 10.0, 20.0, 20.0]


def test_closed_form_lse_uniform():
    q = torch.zeros(1, 1, 1, 2, dtype=torch.float64)
    k = _rand((1, 1, 3, 2), 1)
    v = _rand((1, 1, 3, 2), 2)
    _, lse = oracle.attn(q, k, v, return_lse=True)
    assert abs(lse.item() - math.log(3.0)) < 1e-15


# --------------------------------------------------------------------------
# Brute force, written separately with Python floats and the math module.
# --------------------------------------------------------------------------

def _brute(q, k, v, scale, causal, wl, wr, softcap, slopes, rb):
    B, Hq, Sq, D = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    G = Hq // Hkv
    ql, kl, vl = q.double().tolist(), k.double().tolist(), v.double().tolist()
    sl = None if slopes is None else [float(x) for x in slopes.tolist()]
    out = [[[[0.0] * D for _ in range(Sq)] for _ in range(Hq)] for _ in range(B)]
    lse = [[[NEG_INF] * Sq for _ in range(Hq)] for _ in range(B)]
    for b, h, i in itertools.product(range(B), range(Hq), range(Sq)):
        g = h // G
        s = []
        for j in range(Sk):
            ok = True
            if causal and j > i:
                ok = False
            if wl is not None and j + wl < i:
                ok = False
            if wr is not None and j > i + wr:
                ok = False
            if rb is not None and not (rb[b][i][0] <= j <= rb[b][i][1]):
                ok = False
            if not ok:
                s.append(None)
                continue
            x = scale * math.fsum(ql[b][h][i][d] * kl[b][g][j][d] for d in range(D))
            if softcap:
                x = softcap * math.tanh(x / softcap)
            if sl is not None:
                x += sl[h] * (j - i)
            s.append(x)
        fin = [x for x in s if x is not None]
        if not fin:
            continue
        m = max(fin)
        w = [0.0 if x is None else math.exp(x - m) for x in s]
        L = math.fsum(w)
        for d in range(D):
            out[b][h][i][d] = math.fsum(w[j] * vl[b][g][j][d] for j in range(Sk)) / L
        lse[b][h][i] = m + math.log(L)
    return torch.tensor(out, dtype=torch.float64), torch.tensor(lse, dtype=torch.float64)


BRUTE_CASES = [
    # (B, Hq, Hkv, Sq, Sk, D, causal, wl, wr, softcap, alibi, rowb, dtype)
    (1, 2, 1, 5, 7, 3, False, None, None, None, False, False, torch.float32),
    (2, 4, 2, 6, 6, 4, True, None, None, None, False, False, torch.bfloat16),
    (1, 3, 3, 8, 8, 2, True, 2, 0, None, True, False, torch.float32),
    (1, 2, 2, 7, 5, 3, False, 1, 2, 3.0, True, False, torch.float64),
    (2, 2, 1, 8, 8, 4, True, 3, 0, 0.7, True, True, torch.bfloat16),
    (1, 4, 1, 3, 8, 5, False, None, 1, None, False, True, torch.float32),
]


@pytest.mark.parametrize("case", BRUTE_CASES)
def test_brute_force_tiny(case):
    B, Hq, Hkv, Sq, Sk, D, causal, wl, wr, cap, alibi, rowb, dt = case
    q = _rand((B, Hq, Sq, D), 0, dt)
    k = _rand((B, Hkv, Sk, D), 1, dt)
    v = _rand((B, Hkv, Sk, D), 2, dt)
    slopes = synth.alibi_slopes(Hq) * 3.0 if alibi else None
    rb = None
    if rowb:
        lo = synth.randint(B * Sq, Sk, 5, 3).view(B, Sq)
        hi = synth.randint(B * Sq, Sk, 5, 4).view(B, Sq)
        rb = torch.stack((torch.minimum(lo, hi), torch.maximum(lo, hi)), -1).to(torch.int32)
        rb[0, 0] = torch.tensor([1, 0])  # one empty row
    scale = 0.37
    out, lse = oracle.attn(q, k, v, scale=scale, causal=causal, window_left=wl, window_right=wr,
                           softcap=cap, alibi_slopes=slopes, row_kv_bounds=rb, return_lse=True)
    bo, bl = _brute(q, k, v, float(torch.tensor(scale, dtype=torch.float32)), causal, wl, wr,
                    None if cap is None else float(torch.tensor(cap, dtype=torch.float32)),
                    slopes, None if rb is None else rb.tolist())
    assert torch.allclose(out, bo, rtol=0, atol=1e-12)
    fin = torch.isfinite(bl)
    assert torch.equal(fin, torch.isfinite(lse))
    assert torch.allclose(lse[fin], bl[fin], rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# Library special case: torch float64 softmax on rows that are not fully masked.
# --------------------------------------------------------------------------

def _torch_ref(q, k, v, scale, causal, wl, wr, softcap, slopes):
    B, Hq, Sq, D = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    kk = k.double().repeat_interleave(Hq // Hkv, dim=1)
    vv = v.double().repeat_interleave(Hq // Hkv, dim=1)
    s = scale * (q.double() @ kk.transpose(-1, -2))
    if softcap:
        s = softcap * torch.tanh(s / softcap)
    i = torch.arange(Sq).view(Sq, 1)
    j = torch.arange(Sk).view(1, Sk)
    if slopes is not None:
        s = s + slopes.double().view(1, Hq, 1, 1) * (j - i).double()
    ok = torch.ones(Sq, Sk, dtype=torch.bool)
    if causal:
        ok &= j <= i
    if wl is not None:
        ok &= j + wl >= i
    if wr is not None:
        ok &= j <= i + wr
    s = s.masked_fill(~ok, NEG_INF)
    return torch.softmax(s, dim=-1) @ vv, ok.any(-1)


@pytest.mark.parametrize("causal,wl,wr,cap,alibi", [
    (False, None, None, None, False),
    (True, None, None, None, False),
    (True, 5, 0, None, True),
    (False, 3, 4, 2.5, True),
    (True, None, None, 5.0, False),
])
def test_matches_torch_float64(causal, wl, wr, cap, alibi):
    B, Hq, Hkv, Sq, Sk, D = 2, 4, 2, 33, 33, 16
    q = _rand((B, Hq, Sq, D), 0, torch.float32)
    k = _rand((B, Hkv, Sk, D), 1, torch.float32)
    v = _rand((B, Hkv, Sk, D), 2, torch.float32)
    slopes = synth.alibi_slopes(Hq) if alibi else None
    scale = 1.0 / math.sqrt(D)
    out = oracle.attn(q, k, v, scale=scale, causal=causal, window_left=wl, window_right=wr,
                      softcap=cap, alibi_slopes=slopes)
    f32 = lambda x: float(torch.tensor(x, dtype=torch.float32))
    ref, live = _torch_ref(q, k, v, f32(scale), causal, wl, wr, None if cap is None else f32(cap), slopes)
    assert live.all()
    assert torch.allclose(out, ref, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# Invariants from the definition.
# --------------------------------------------------------------------------

def test_uniform_scores_mean_of_admitted_values():
    B, Hq, Hkv, Sq, Sk, D = 1, 2, 1, 12, 12, 5
    q = torch.zeros(B, Hq, Sq, D, dtype=torch.float64)
    k = _rand((B, Hkv, Sk, D), 1)
    v = _rand((B, Hkv, Sk, D), 2)
    out = oracle.attn(q, k, v, causal=True, window_left=3)
    for i in range(Sq):
        lo = max(0, i - 3)
        mean = v[0, 0, lo:i + 1].mean(dim=0)
        assert torch.allclose(out[0, 0, i], mean, rtol=0, atol=1e-15)
        assert torch.allclose(out[0, 1, i], mean, rtol=0, atol=1e-15)


def test_dominant_key_selects_its_value_row():
    B, Hq, Hkv, Sq, Sk, D = 1, 1, 1, 4, 9, 8
    q = _rand((B, Hq, Sq, D), 0)
    k = _rand((B, Hkv, Sk, D), 1)
    v = _rand((B, Hkv, Sk, D), 2)
    j = 6
    qi = 2
    k[0, 0, j] = 60.0 * q[0, 0, qi] / q[0, 0, qi].norm()
    out = oracle.attn(q, k, v, scale=1.0)
    s = (q[0, 0, qi] @ k[0, 0].T)
    gap = (s[j] - torch.cat((s[:j], s[j + 1:])).max()).item()
    assert gap > 30
    bound = Sk * math.exp(-gap) * v.abs().max().item() * 2
    assert torch.allclose(out[0, 0, qi], v[0, 0, j], rtol=0, atol=bound)


def test_masked_positions_have_zero_weight_bitwise():
    B, Hq, Hkv, Sq, Sk, D = 1, 2, 1, 10, 10, 4
    q = _rand((B, Hq, Sq, D), 0)
    k = _rand((B, Hkv, Sk, D), 1)
    v = _rand((B, Hkv, Sk, D), 2)
    base = oracle.attn(q, k, v, causal=True)
    # keys after row qi are masked for that row: perturb keys/values beyond 4
    k2, v2 = k.clone(), v.clone()
    k2[:, :, 5:] += 1e3
    v2[:, :, 5:] = float("nan")
    got = oracle.attn(q, k2, v2, causal=True)
    assert torch.equal(got[:, :, :5], base[:, :, :5])


def test_fully_masked_rows_are_exact_zeros():
    B, Hq, Hkv, Sq, Sk, D = 2, 2, 2, 6, 6, 3
    q = _rand((B, Hq, Sq, D), 0)
    k = _rand((B, Hkv, Sk, D), 1)
    v = _rand((B, Hkv, Sk, D), 2)
    rb = torch.zeros(B, Sq, 2, dtype=torch.int32)
    rb[..., 1] = Sk - 1
    rb[1, 3] = torch.tensor([1, 0])
    rb[0, 0] = torch.tensor([4, 5])          # causal leaves only key 0 -> empty
    out, lse = oracle.attn(q, k, v, causal=True, row_kv_bounds=rb, return_lse=True)
    for b, i in ((1, 3), (0, 0)):
        assert torch.equal(out[b, :, i], torch.zeros(Hq, D, dtype=torch.float64))
        assert torch.isneginf(lse[b, :, i]).all()
    assert torch.isfinite(lse[0, :, 1]).all()


def test_gqa_equals_repeated_kv_bitwise():
    B, Hq, Hkv, Sq, Sk, D = 2, 6, 2, 7, 9, 4
    q = _rand((B, Hq, Sq, D), 0, torch.bfloat16)
    k = _rand((B, Hkv, Sk, D), 1, torch.bfloat16)
    v = _rand((B, Hkv, Sk, D), 2, torch.bfloat16)
    slopes = synth.alibi_slopes(Hq)
    a = oracle.attn(q, k, v, causal=True, alibi_slopes=slopes, softcap=4.0)
    b = oracle.attn(q, k.repeat_interleave(3, dim=1), v.repeat_interleave(3, dim=1),
                    causal=True, alibi_slopes=slopes, softcap=4.0)
    assert torch.equal(a, b)


@pytest.mark.parametrize("BR,BC", [(16, 16), (7, 13), (1, 64)])
@pytest.mark.parametrize("flags", [
    dict(),
    dict(causal=True),
    dict(causal=True, window_left=9, window_right=0, softcap=3.0, alibi=True, rowb=True),
    dict(window_left=4, window_right=6, alibi=True),
])
def test_tiled_online_recurrence_matches_materialised(BR, BC, flags):
    B, Hq, Hkv, Sq, Sk, D = 2, 4, 2, 37, 41, 8
    flags = dict(flags)
    q = _rand((B, Hq, Sq, D), 0, torch.bfloat16)
    k = _rand((B, Hkv, Sk, D), 1, torch.bfloat16)
    v = _rand((B, Hkv, Sk, D), 2, torch.bfloat16)
    if flags.pop("alibi", False):
        flags["alibi_slopes"] = synth.alibi_slopes(Hq)
    if flags.pop("rowb", False):
        flags["row_kv_bounds"] = synth.row_kv_bounds_with_empty_rows(B, Sq, Sk, 0.1, seed=3)
    a, la = oracle.attn(q, k, v, return_lse=True, **flags)
    b, lb = oracle.attn_tiled(q, k, v, BR=BR, BC=BC, return_lse=True, **flags)
    assert torch.allclose(a, b, rtol=0, atol=1e-12)
    fin = torch.isfinite(la)
    assert torch.equal(fin, torch.isfinite(lb))
    assert torch.allclose(la[fin], lb[fin], rtol=0, atol=1e-12)


def test_limits_reduce_to_plain_attention():
    B, Hq, Hkv, Sq, Sk, D = 1, 2, 1, 11, 11, 4
    q = _rand((B, Hq, Sq, D), 0)
    k = _rand((B, Hkv, Sk, D), 1)
    v = _rand((B, Hkv, Sk, D), 2)
    base = oracle.attn(q, k, v, causal=True)
    assert torch.allclose(oracle.attn(q, k, v, causal=True, softcap=1e30), base, rtol=0, atol=1e-12)
    assert torch.equal(oracle.attn(q, k, v, causal=True, alibi_slopes=torch.zeros(Hq)), base)
    assert torch.equal(oracle.attn(q, k, v, causal=True, window_left=Sk, window_right=Sk), base)


def test_key_permutation_invariance():
    B, Hq, Hkv, Sq, Sk, D = 1, 2, 2, 5, 13, 6
    q = _rand((B, Hq, Sq, D), 0)
    k = _rand((B, Hkv, Sk, D), 1)
    v = _rand((B, Hkv, Sk, D), 2)
    perm = torch.randperm(Sk, generator=torch.Generator().manual_seed(0))
    a = oracle.attn(q, k, v)
    b = oracle.attn(q, k[:, :, perm], v[:, :, perm])
    assert torch.allclose(a, b, rtol=0, atol=1e-13)


def test_row_subset_equals_full_problem():
    B, Hq, Hkv, Sq, Sk, D = 2, 4, 2, 9, 10, 4
    q = _rand((B, Hq, Sq, D), 0, torch.bfloat16)
    k = _rand((B, Hkv, Sk, D), 1, torch.bfloat16)
    v = _rand((B, Hkv, Sk, D), 2, torch.bfloat16)
    full, lfull = oracle.attn(q, k, v, causal=True, return_lse=True)
    rows = torch.tensor([0, 5, 17, B * Hq * Sq - 1])
    sub, lsub = oracle.attn(q, k, v, causal=True, rows=rows, return_lse=True)
    assert torch.equal(sub, full.view(-1, D)[rows])
    assert torch.equal(lsub, lfull.view(-1)[rows])


def test_decode_is_one_row_without_causal_mask():
    B, Hq, Hkv, Sk, D = 2, 4, 2, 17, 8
    q = _rand((B, Hq, 1, D), 0, torch.bfloat16)
    k = _rand((B, Hkv, Sk, D), 1, torch.bfloat16)
    v = _rand((B, Hkv, Sk, D), 2, torch.bfloat16)
    out = oracle.decode(q, k, v)
    ref, _ = _torch_ref(q, k, v, float(torch.tensor(1 / math.sqrt(D), dtype=torch.float32)),
                        False, None, None, None, None)
    assert torch.allclose(out, ref, rtol=0, atol=1e-12)


def test_rejects_bad_problems():
    q = torch.zeros(1, 3, 2, 4)
    k = torch.zeros(1, 2, 2, 4)
    with pytest.raises(ValueError):
        oracle.attn(q, k, k)


def test_fp16_inputs_widen_exactly():
    """fp16 inputs are read by the oracle's own binary16 decoding; it must
    agree bitwise with the same values widened to float64 by torch, including
    subnormals, zeros of both signs and the largest finite values."""
    q = synth.normal((1, 2, 9, 16), 17, 0, torch.float16)
    k = synth.normal((1, 1, 11, 16), 17, 1, torch.float16)
    v = synth.normal((1, 1, 11, 16), 17, 2, torch.float16)
    v[0, 0, 0, :4] = torch.tensor([6.0e-8, -0.0, 65504.0, -3.0e-5], dtype=torch.float16)
    k[0, 0, 1, :2] = torch.tensor([1.0e-6, -6.1e-5], dtype=torch.float16)
    for causal in (False, True):
        a, la = oracle.attn(q, k, v, causal=causal, softcap=10.0, return_lse=True)
        b, lb = oracle.attn(q.double(), k.double(), v.double(), causal=causal, softcap=10.0, return_lse=True)
        assert torch.equal(a, b) and torch.equal(la, lb)
