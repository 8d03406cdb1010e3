"""Pins of the decode oracle's query position and sliding window.

A decode row is the newest token of its sequence: it sits at position
Sk - 1, after every key ("gfx942 unified attention", section 4: decode runs
non-causal, which at the last position is the causal mask; attention.fkc.md,
attention_paged_naive: abs_pos = context_len - 1 for the decode query).  The
dense contract's window (attention.fkc.md, header: window_size_left/right,
position_admissible) then admits keys j with Sk - 1 - left <= j; no key lies
after the query, so the right window admits them all.  ALiBi adds
slope_h * (j - (Sk - 1)).

Each pin checks the decode oracle against something other than itself: the
dense C oracle with the query placed at row Sk - 1 (top-left alignment, the
position-0 path pinned elsewhere), the independent torch code of the packed
variable-length oracle with one query per sequence, closed forms, a Python
brute force, and invariances of the mask.
"""
import math

import pytest
import torch

import oracle
import synth

FLAGS = [
    dict(),
    dict(window_left=0),
    dict(window_left=5),
    dict(window_left=13, softcap=3.0),
    dict(window_left=9, alibi=True),
    dict(window_left=20, window_right=0, softcap=10.0, alibi=True),
    dict(alibi=True, softcap=7.0),
    dict(window_right=4, alibi=True),
]


def _qkv(B, Hq, Hkv, Sk, D, dtype=torch.bfloat16, seed=31):
    q = synth.normal((B, Hq, 1, D), seed, synth.STREAM_Q, dtype)
    k = synth.normal((B, Hkv, Sk, D), seed, synth.STREAM_K, dtype)
    v = synth.normal((B, Hkv, Sk, D), seed, synth.STREAM_V, dtype)
    return q, k, v


def _kw(f, Hq):
    return dict(window_left=f.get("window_left"), window_right=f.get("window_right"), softcap=f.get("softcap"),
                alibi_slopes=synth.alibi_slopes(Hq) if f.get("alibi") else None)


@pytest.mark.parametrize("flags", FLAGS, ids=lambda f: "-".join(f"{k}{v}" for k, v in f.items()) or "plain")
def test_decode_is_the_last_row_of_the_dense_problem(flags):
    """Row Sk - 1 of a dense Sq = Sk problem (top-left: row i at position i)
    whose query tensor holds the decode query in that row."""
    B, Hq, Hkv, Sk, D = 2, 4, 2, 23, 8
    q, k, v = _qkv(B, Hq, Hkv, Sk, D)
    kw = _kw(flags, Hq)
    out, lse = oracle.decode(q, k, v, return_lse=True, **kw)
    qfull = torch.zeros(B, Hq, Sk, D, dtype=q.dtype)
    qfull[:, :, Sk - 1] = q[:, :, 0]
    ref, ref_lse = oracle.attn(qfull, k, v, return_lse=True, **kw)
    assert (out[:, :, 0] - ref[:, :, Sk - 1]).abs().max().item() < 1e-12
    assert (lse[:, :, 0] - ref_lse[:, :, Sk - 1]).abs().max().item() < 1e-12


@pytest.mark.parametrize("flags", FLAGS, ids=lambda f: "-".join(f"{k}{v}" for k, v in f.items()) or "plain")
def test_decode_equals_one_packed_query_per_sequence(flags):
    """The packed-sequence oracle (torch float64, bottom-right: a sequence's
    single query sits at kv_len - 1) with q_len = 1 for every sequence."""
    B, Hq, Hkv, Sk, D = 3, 4, 1, 19, 16
    q, k, v = _qkv(B, Hq, Hkv, Sk, D, seed=33)
    kw = _kw(flags, Hq)
    out, lse = oracle.decode(q, k, v, return_lse=True, **kw)
    qp = q[:, :, 0, :].contiguous()                                   # [B, Hq, D] = [total_q, Hq, D]
    kp = k.permute(0, 2, 1, 3).reshape(B * Sk, Hkv, D).contiguous()   # [total_k, Hkv, D]
    vp = v.permute(0, 2, 1, 3).reshape(B * Sk, Hkv, D).contiguous()
    cq = torch.arange(B + 1, dtype=torch.int32)
    ck = torch.arange(B + 1, dtype=torch.int32) * Sk
    ref, ref_lse = oracle.attn_varlen(qp, kp, vp, cq, ck, return_lse=True, **kw)
    assert (out[:, :, 0] - ref).abs().max().item() < 1e-12
    assert (lse[:, :, 0] - ref_lse.T).abs().max().item() < 1e-12


def test_window_zero_selects_the_newest_key():
    """window_left = 0: only key Sk - 1 is admissible, so O = V[Sk - 1]
    exactly and lse = its score (the ALiBi term is 0 there)."""
    B, Hq, Hkv, Sk, D = 1, 2, 1, 40, 8
    q, k, v = _qkv(B, Hq, Hkv, Sk, D, dtype=torch.float64)
    out, lse = oracle.decode(q, k, v, window_left=0, alibi_slopes=synth.alibi_slopes(Hq), return_lse=True)
    scale = float(torch.tensor(1 / math.sqrt(D), dtype=torch.float32))
    for h in range(Hq):
        assert torch.equal(out[0, h, 0], v[0, 0, Sk - 1])
        s = scale * float((q[0, h, 0] * k[0, 0, Sk - 1]).sum())
        assert abs(lse[0, h, 0].item() - s) < 1e-12


def test_window_one_closed_form():
    """window_left = 1: keys Sk - 2 and Sk - 1 with scores 0 and ln 3 give
    weights 1/4 and 3/4; ALiBi with slope 1 adds -1 and 0."""
    Sk, D = 6, 1
    q = torch.ones(1, 1, 1, D, dtype=torch.float64)
    k = torch.full((1, 1, Sk, D), 9.0, dtype=torch.float64)  # outside the window: would dominate
    v = torch.full((1, 1, Sk, D), 100.0, dtype=torch.float64)
    k[0, 0, Sk - 2, 0], v[0, 0, Sk - 2, 0] = 0.0, 2.0
    k[0, 0, Sk - 1, 0], v[0, 0, Sk - 1, 0] = math.log(3.0), 6.0
    out, lse = oracle.decode(q, k, v, scale=1.0, window_left=1, return_lse=True)
    assert abs(out.item() - (0.25 * 2.0 + 0.75 * 6.0)) < 1e-12
    assert abs(lse.item() - math.log(4.0)) < 1e-12
    out, lse = oracle.decode(q, k, v, scale=1.0, window_left=1, alibi_slopes=torch.ones(1), return_lse=True)
    w0, w1 = math.exp(-1.0), 3.0
    assert abs(out.item() - (w0 * 2.0 + w1 * 6.0) / (w0 + w1)) < 1e-12
    assert abs(lse.item() - math.log(w0 + w1)) < 1e-12


def test_brute_force_tiny():
    """A Python-float brute force of the decode row at position Sk - 1."""
    B, Hq, Hkv, Sk, D = 1, 2, 1, 7, 3
    q, k, v = _qkv(B, Hq, Hkv, Sk, D, dtype=torch.float64, seed=35)
    slopes = synth.alibi_slopes(Hq)
    scale = float(torch.tensor(1 / math.sqrt(D), dtype=torch.float32))
    cap = float(torch.tensor(2.5, dtype=torch.float32))
    for wl in (None, 0, 2, 6, 50):
        out, lse = oracle.decode(q, k, v, softcap=2.5, alibi_slopes=slopes, window_left=wl, return_lse=True)
        p = Sk - 1
        for h in range(Hq):
            s = []
            for j in range(Sk):
                if wl is not None and j < p - wl:
                    continue
                x = scale * math.fsum(float(q[0, h, 0, d]) * float(k[0, 0, j, d]) for d in range(D))
                x = cap * math.tanh(x / cap) + float(slopes[h]) * (j - p)
                s.append((j, x))
            m = max(x for _, x in s)
            w = [(j, math.exp(x - m)) for j, x in s]
            L = math.fsum(x for _, x in w)
            for d in range(D):
                o = math.fsum(x * float(v[0, 0, j, d]) for j, x in w) / L
                assert abs(out[0, h, 0, d].item() - o) < 1e-12
            assert abs(lse[0, h, 0].item() - (m + math.log(L))) < 1e-12


def test_window_invariances():
    """A window wider than the sequence is no window; the right window never
    masks anything; NaN planted in keys and values outside the left window
    changes nothing, bitwise."""
    B, Hq, Hkv, Sk, D = 2, 4, 2, 30, 8
    q, k, v = _qkv(B, Hq, Hkv, Sk, D, seed=37)
    slopes = synth.alibi_slopes(Hq)
    base, lb = oracle.decode(q, k, v, alibi_slopes=slopes, return_lse=True)
    for wl, wr in ((Sk - 1, None), (Sk + 50, None), (None, 0), (None, 3)):
        o, l = oracle.decode(q, k, v, alibi_slopes=slopes, window_left=wl, window_right=wr, return_lse=True)
        assert torch.equal(o, base) and torch.equal(l, lb)
    wl = 11
    ref = oracle.decode(q, k, v, alibi_slopes=slopes, window_left=wl)
    k2, v2 = k.clone(), v.clone()
    k2[:, :, :Sk - 1 - wl] = float("nan")
    v2[:, :, :Sk - 1 - wl] = float("nan")
    assert torch.equal(oracle.decode(q, k2, v2, alibi_slopes=slopes, window_left=wl), ref)


@pytest.mark.parametrize("bs", [16, 64])
def test_paged_window_is_the_dense_last_row(bs):
    """Paged decode with a window over shuffled blocks and uneven contexts:
    each sequence's row equals row ctx - 1 of its dense problem (C oracle)."""
    from synth.workloads import make_paged_inputs
    ctx = [70, 1, 130, 64]
    x = make_paged_inputs(4, 4, 2, 16, ctx, bs, dtype=torch.float64, seed=12)
    slopes = synth.alibi_slopes(4)
    for wl in (0, 9, 63, 64, 500):
        out, lse = oracle.attn_paged(x["q"], x["k_cache"], x["v_cache"], x["block_table"], x["context_lens"],
                                     alibi_slopes=slopes, softcap=15.0, window_left=wl, return_lse=True)
        for b, n in enumerate(ctx):
            pos = torch.arange(n)
            blk = x["block_table"][b, pos // bs].long()
            kb = x["k_cache"][blk, pos % bs].permute(1, 0, 2).unsqueeze(0).contiguous()  # [1, Hkv, n, D]
            vb = x["v_cache"][blk, pos % bs].permute(1, 0, 2).unsqueeze(0).contiguous()
            qfull = torch.zeros(1, 4, n, 16, dtype=torch.float64)
            qfull[0, :, n - 1] = x["q"][b, :, 0]
            ref, ref_lse = oracle.attn(qfull, kb, vb, alibi_slopes=slopes, softcap=15.0, window_left=wl,
                                       return_lse=True)
            assert (out[b, :, 0] - ref[0, :, n - 1]).abs().max().item() < 1e-12
            assert (lse[b, :, 0] - ref_lse[0, :, n - 1]).abs().max().item() < 1e-12
