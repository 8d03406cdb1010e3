"""CPU oracle for tiled scaled-dot-product attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
Python binding) never touches it, and it never touches the product: the two
share no code.

``attn`` materialises each score row in float64 (attention.fkc.md,
"attention_naive"); ``attn_tiled`` runs the streaming online-softmax
recurrence (attention.fkc.md, "attention_flash"; "gfx942 unified attention",
section 3) in float64 and exists to cross-check the first.  Decode is the same
definition with one query row at the last position, Sk - 1 ("gfx942 unified
attention", section 4: decode runs non-causal, the same as causal at the last
row), so ``decode`` calls ``attn`` with Sq = 1 and that query position.

``attn_paged`` is paged-cache attention (attention.fkc.md,
"attention_paged_naive"): keys and values read through a per-sequence block
table from a pool [num_blocks, block_size, Hkv, D], per-sequence context
lengths, and the implicit causal mask at the query's absolute position.

``attn_varlen`` is attention over packed variable-length sequences
("gfx942 unified attention", section 5: queries packed [total_q, heads, D]
with a cu_seqlens_q prefix sum, seqused_k per sequence) with the causal mask
aligned bottom-right (section 4): query i of a sequence sits at absolute
position kv_len - q_len + i.

``attn_bwd`` is the backward by recompute (attention.fkc.md,
"attention_flash_backward"): dQ, dK, dV of the forward above, with the softcap
derivative, dK / dV summed over each GQA group.

Parity pins: every function here is pinned by tests/test_oracle_pins.py,
tests/test_oracle_varlen.py, tests/test_oracle_paged.py and
tests/test_oracle_bwd.py (closed forms, brute force, library special cases,
invariants, finite differences of the forward); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_DT = {torch.bfloat16: 0, torch.float32: 1, torch.float64: 2, torch.float16: 3}


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into liboracle.so next to it (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                        "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            L = ctypes.c_long
            Dd = ctypes.c_double
            lib.oracle_attn_rows.argtypes = [I, P, P, P, P, P, I, I, I, I, I, I, Dd, I, L, L, Dd, L,
                                             P, ctypes.c_int64, P, P, I]
            lib.oracle_attn_rows.restype = I
            lib.oracle_attn_tiled.argtypes = [I, P, P, P, P, P, I, I, I, I, I, I, Dd, I, L, L, Dd,
                                              I, I, P, P, I]
            lib.oracle_attn_tiled.restype = I
            lib.oracle_max_threads.restype = I
            _lib = lib
    return _lib


def max_threads() -> int:
    return _load().oracle_max_threads()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _prep(q, k, v, alibi_slopes, row_kv_bounds):
    if not (q.dtype == k.dtype == v.dtype) or q.dtype not in _DT:
        raise TypeError("q, k, v must share one of bf16 / f16 / f32 / f64")
    q, k, v = (t.detach().to("cpu").contiguous() for t in (q, k, v))
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4 or k.shape != v.shape:
        raise ValueError("q [B,Hq,Sq,D], k and v [B,Hkv,Sk,D]")
    B, Hq, Sq, D = q.shape
    Bk, Hkv, Sk, Dk = k.shape
    if Bk != B or Dk != D or Hq % Hkv:
        raise ValueError("shape mismatch or Hq not a multiple of Hkv")
    s = None if alibi_slopes is None else alibi_slopes.detach().to("cpu", torch.float32).contiguous()
    if s is not None and s.numel() != Hq:
        raise ValueError("alibi slopes must be [Hq]")
    rb = None if row_kv_bounds is None else row_kv_bounds.detach().to("cpu", torch.int32).contiguous()
    if rb is not None and tuple(rb.shape) != (B, Sq, 2):
        raise ValueError("row_kv_bounds must be [B, Sq, 2]")
    return q, k, v, s, rb, (B, Hq, Hkv, Sq, Sk, D)


def _f32(x: float) -> float:
    """The float32 value the GPU receives, as a Python float."""
    return float(torch.tensor(x, dtype=torch.float32))


def _win(w):
    return -1 if w is None or w < 0 else int(w)


def attn(q, k, v, *, scale=None, causal=False, window_left=None, window_right=None,
         softcap=None, alibi_slopes=None, row_kv_bounds=None, rows=None, threads=0,
         return_lse=False, query_pos0=0):
    """Materialised float64 attention.

    q [B,Hq,Sq,D], k/v [B,Hkv,Sk,D] (bf16, f32 or f64, any device: copied to
    the host).  ``rows`` (optional 1-D int64 of flat (b*Hq + h)*Sq + qi
    indices) restricts the work to those rows; the result is then [n, D].
    Query row qi sits at position ``query_pos0 + qi`` for the causal and
    window masks and the ALiBi term (0: the top-left alignment of
    position_admissible).  Returns float64 out (and lse if asked).
    """
    q, k, v, s, rb, (B, Hq, Hkv, Sq, Sk, D) = _prep(q, k, v, alibi_slopes, row_kv_bounds)
    if scale is None:
        scale = 1.0 / (D ** 0.5)
    if rows is None:
        out = torch.empty(B, Hq, Sq, D, dtype=torch.float64)
        lse = torch.empty(B, Hq, Sq, dtype=torch.float64)
        rr, n = None, 0
    else:
        rr = torch.as_tensor(rows, dtype=torch.int64).contiguous()
        n = rr.numel()
        if n and (int(rr.min()) < 0 or int(rr.max()) >= B * Hq * Sq):
            raise ValueError("row index out of range")
        out = torch.empty(n, D, dtype=torch.float64)
        lse = torch.empty(n, dtype=torch.float64)
    rc = _load().oracle_attn_rows(_DT[q.dtype], _ptr(q), _ptr(k), _ptr(v), _ptr(s), _ptr(rb),
                                  B, Hq, Hkv, Sq, Sk, D, _f32(scale), int(bool(causal)),
                                  _win(window_left), _win(window_right),
                                  0.0 if not softcap else _f32(softcap), int(query_pos0),
                                  _ptr(rr), n, _ptr(out), _ptr(lse), int(threads))
    if rc:
        raise ValueError("oracle rejected the problem")
    return (out, lse) if return_lse else out


def attn_tiled(q, k, v, *, BR=16, BC=16, scale=None, causal=False, window_left=None,
               window_right=None, softcap=None, alibi_slopes=None, row_kv_bounds=None,
               threads=0, return_lse=False):
    """Streaming (online-softmax) float64 attention over BR x BC tiles."""
    q, k, v, s, rb, (B, Hq, Hkv, Sq, Sk, D) = _prep(q, k, v, alibi_slopes, row_kv_bounds)
    if scale is None:
        scale = 1.0 / (D ** 0.5)
    out = torch.empty(B, Hq, Sq, D, dtype=torch.float64)
    lse = torch.empty(B, Hq, Sq, dtype=torch.float64)
    rc = _load().oracle_attn_tiled(_DT[q.dtype], _ptr(q), _ptr(k), _ptr(v), _ptr(s), _ptr(rb),
                                   B, Hq, Hkv, Sq, Sk, D, _f32(scale), int(bool(causal)),
                                   _win(window_left), _win(window_right),
                                   0.0 if not softcap else _f32(softcap),
                                   int(BR), int(BC), _ptr(out), _ptr(lse), int(threads))
    if rc:
        raise ValueError("oracle rejected the problem")
    return (out, lse) if return_lse else out


def decode(q, k, v, *, scale=None, softcap=None, alibi_slopes=None, window_left=None, window_right=None,
           rows=None, threads=0, return_lse=False):
    """Decode: one query row per (b, h), the newest token of its sequence.

    The row sits at position Sk - 1, after every key ("gfx942 unified
    attention", section 4: decode runs non-causal, which at the last position
    is the causal mask; attention_paged_naive puts the decode query at
    context_len - 1 the same way).  The ALiBi term is slope_h (j - (Sk - 1));
    a left window admits keys j >= Sk - 1 - window_left; a right window admits
    every key (none lies after the query).
    """
    if q.shape[2] != 1:
        raise ValueError("decode takes Sq == 1")
    return attn(q, k, v, scale=scale, causal=False, softcap=softcap, alibi_slopes=alibi_slopes,
                window_left=window_left, window_right=window_right, rows=rows, threads=threads,
                return_lse=return_lse, query_pos0=k.shape[2] - 1)


def attn_paged(q, k_cache, v_cache, block_table, context_lens, *, scale=None, softcap=None,
               alibi_slopes=None, window_left=None, window_right=None, return_lse=False):
    """Paged-cache attention in float64 (attention.fkc.md, "attention_paged_naive").

    q [B, Hq, Sq, D]; k_cache, v_cache [num_blocks, block_size, Hkv, D];
    block_table [B, max_blocks] and context_lens [B] (non-negative integers).
    For each (b, h, q_pos) the logical keys are k_pos = 0 .. context_lens[b] - 1,
    key k_pos living at pool block block_table[b, k_pos // block_size], row
    k_pos % block_size, kv head h // (Hq / Hkv).  The query's absolute position
    is abs_pos = max(context_lens[b] - Sq, 0) + q_pos (the saturating
    subtraction of the contract); keys after it are masked, and so are keys
    outside the optional sliding window [abs_pos - window_left, abs_pos +
    window_right] (the dense contract's window, at the query's absolute
    position; None or -1: unbounded).  Scores: scale q.k,
    then softcap c tanh(s / c), then + slope_h (k_pos - abs_pos); a stable
    softmax and the weighted sum of V rows.  A row with no admissible key is
    the zero row with lse = -inf.  A physical block index >= num_blocks is an
    error (ValueError), as in the contract.  Returns float64 out [B, Hq, Sq, D]
    (and lse [B, Hq, Sq]).
    """
    q = q.detach().to("cpu", torch.float64)
    K = k_cache.detach().to("cpu", torch.float64)
    V = v_cache.detach().to("cpu", torch.float64)
    bt = block_table.detach().to("cpu", torch.int64)
    cl = context_lens.detach().to("cpu", torch.int64)
    if q.dim() != 4 or K.dim() != 4 or K.shape != V.shape:
        raise ValueError("q [B,Hq,Sq,D], pools [num_blocks, block_size, Hkv, D]")
    B, Hq, Sq, D = q.shape
    nblk, bs, Hkv, Dk = K.shape
    if Dk != D or Hq % Hkv or bt.dim() != 2 or bt.shape[0] != B or tuple(cl.shape) != (B,):
        raise ValueError("shape mismatch")
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / (D ** 0.5)
    sc = _f32(scale)
    cap = 0.0 if not softcap else _f32(softcap)
    slopes = None if alibi_slopes is None else alibi_slopes.detach().to("cpu", torch.float32).double()
    out = torch.zeros(B, Hq, Sq, D, dtype=torch.float64)
    lse = torch.full((B, Hq, Sq), float("-inf"), dtype=torch.float64)
    for b in range(B):
        ctx = int(cl[b])
        if ctx > bt.shape[1] * bs:
            raise ValueError("context length beyond the block table")
        pos = torch.arange(ctx, dtype=torch.int64)
        blk = bt[b, pos // bs] if ctx else torch.zeros(0, dtype=torch.int64)
        if ctx and (int(blk.min()) < 0 or int(blk.max()) >= nblk):
            raise ValueError("physical block index out of range")
        off = pos % bs
        Kb, Vb = K[blk, off], V[blk, off]  # [ctx, Hkv, D]: the gathered keys in logical order
        abs_pos = max(ctx - Sq, 0) + torch.arange(Sq, dtype=torch.int64)  # [Sq]
        admissible = pos[None, :] <= abs_pos[:, None]  # [Sq, ctx]
        if window_left is not None and window_left >= 0:
            admissible &= pos[None, :] >= abs_pos[:, None] - window_left
        if window_right is not None and window_right >= 0:
            admissible &= pos[None, :] <= abs_pos[:, None] + window_right
        for h in range(Hq):
            g = h // G
            s = sc * (q[b, h] @ Kb[:, g, :].T)  # [Sq, ctx]
            if cap:
                s = cap * torch.tanh(s / cap)
            if slopes is not None:
                s = s + slopes[h] * (pos[None, :] - abs_pos[:, None]).double()
            s = torch.where(admissible, s, torch.full_like(s, float("-inf")))
            for i in range(Sq):
                m = s[i].max() if ctx else torch.tensor(float("-inf"), dtype=torch.float64)
                if m == float("-inf"):
                    continue
                w = torch.exp(s[i] - m)
                L = w.sum()
                out[b, h, i] = (w @ Vb[:, g, :]) / L
                lse[b, h, i] = m + torch.log(L)
    return (out, lse) if return_lse else out


def attn_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, *, seqused_k=None, scale=None, causal=False,
                window_left=None, window_right=None, softcap=None, alibi_slopes=None, return_lse=False):
    """Packed variable-length attention in float64.

    q [total_q, Hq, D], k / v [total_k, Hkv, D]; cu_seqlens_q / cu_seqlens_k
    [B + 1] prefix sums; seqused_k [B] (optional) the live keys of each
    sequence, a prefix of its cu_seqlens_k range.  For sequence b with q_len
    queries and kv_len live keys, query i sits at abs_i = kv_len - q_len + i
    ("gfx942 unified attention", section 4: bottom-right alignment); key j
    (0 .. kv_len - 1) is admissible iff (not causal or j <= abs_i) and
    (window_left is None or j >= abs_i - window_left) and (window_right is
    None or j <= abs_i + window_right).  Scores: scale q.k, softcap
    c tanh(s / c), + slope_h (j - abs_i); stable softmax; weighted V.  A row
    with no admissible key is the zero row, lse -inf.  Returns float64 out
    [total_q, Hq, D] (and lse [Hq, total_q]).
    """
    q = q.detach().to("cpu", torch.float64)
    k = k.detach().to("cpu", torch.float64)
    v = v.detach().to("cpu", torch.float64)
    cq = [int(x) for x in cu_seqlens_q.detach().to("cpu").tolist()]
    ck = [int(x) for x in cu_seqlens_k.detach().to("cpu").tolist()]
    B = len(cq) - 1
    if q.dim() != 3 or k.dim() != 3 or k.shape != v.shape or len(ck) != B + 1:
        raise ValueError("q [total_q, Hq, D], k / v [total_k, Hkv, D], cu_seqlens [B + 1]")
    total_q, Hq, D = q.shape
    total_k, Hkv, Dk = k.shape
    if Dk != D or Hq % Hkv or cq[0] != 0 or ck[0] != 0 or cq[-1] != total_q or ck[-1] > total_k:
        raise ValueError("shape mismatch")
    if any(b < a for a, b in zip(cq, cq[1:])) or any(b < a for a, b in zip(ck, ck[1:])):
        raise ValueError("cu_seqlens must be non-decreasing")
    used = None if seqused_k is None else [int(x) for x in seqused_k.detach().to("cpu").tolist()]
    G = Hq // Hkv
    sc = _f32(1.0 / (D ** 0.5) if scale is None else scale)
    cap = 0.0 if not softcap else _f32(softcap)
    slopes = None if alibi_slopes is None else alibi_slopes.detach().to("cpu", torch.float32).double()
    out = torch.zeros(total_q, Hq, D, dtype=torch.float64)
    lse = torch.full((Hq, total_q), float("-inf"), dtype=torch.float64)
    for b in range(B):
        q_len = cq[b + 1] - cq[b]
        kv_len = ck[b + 1] - ck[b]
        if used is not None:
            if not 0 <= used[b] <= kv_len:
                raise ValueError("seqused_k must be within the sequence's keys")
            kv_len = used[b]
        if q_len == 0:
            continue
        j = torch.arange(kv_len, dtype=torch.int64)
        abs_i = kv_len - q_len + torch.arange(q_len, dtype=torch.int64)
        adm = torch.ones(q_len, kv_len, dtype=torch.bool)
        if causal:
            adm &= j[None, :] <= abs_i[:, None]
        if window_left is not None and window_left >= 0:
            adm &= j[None, :] >= abs_i[:, None] - window_left
        if window_right is not None and window_right >= 0:
            adm &= j[None, :] <= abs_i[:, None] + window_right
        kb, vb = k[ck[b]:ck[b] + kv_len], v[ck[b]:ck[b] + kv_len]
        for h in range(Hq):
            g = h // G
            s = sc * (q[cq[b]:cq[b + 1], h, :] @ kb[:, g, :].T)  # [q_len, kv_len]
            if cap:
                s = cap * torch.tanh(s / cap)
            if slopes is not None:
                s = s + slopes[h] * (j[None, :] - abs_i[:, None]).double()
            s = torch.where(adm, s, torch.full_like(s, float("-inf")))
            for i in range(q_len):
                m = s[i].max() if kv_len else torch.tensor(float("-inf"), dtype=torch.float64)
                if m == float("-inf"):
                    continue
                w = torch.exp(s[i] - m)
                L = w.sum()
                out[cq[b] + i, h] = (w @ vb[:, g, :]) / L
                lse[h, cq[b] + i] = m + torch.log(L)
    return (out, lse) if return_lse else out


def attn_bwd(q, k, v, dout, *, scale=None, causal=False, window_left=None, window_right=None,
             softcap=None, alibi_slopes=None, row_kv_bounds=None):
    """Attention backward by recompute, in float64 (attention.fkc.md,
    "attention_flash_backward").

    q, dout [B, Hq, Sq, D]; k, v [B, Hkv, Sk, D]; the forward's flags as in
    ``attn``.  For each (b, h) the forward is recomputed: the pre-softcap score
    s_pre = scale q.k, the score s = c tanh(s_pre / c) (softcap) + slope_h (j - i)
    (ALiBi), -inf where key j is not admissible for row i, and the stable
    softmax P of each row.  Then, in the contract's order:
      dV[j]  += sum_i P[i, j] dO[i]
      dP[i, j] = dO[i] . V[j]
      dS[i, j] = (dP[i, j] - sum_j' P[i, j'] dP[i, j']) P[i, j],
                 times 1 - tanh^2(s_pre / c) when softcap is set
      dQ[i]  += scale sum_j dS[i, j] K[j]
      dK[j]  += scale sum_i dS[i, j] Q[i]
    dK and dV of kv head g sum the contributions of every query head of its
    group; a row with no admissible key contributes nothing.  Returns float64
    (dq [B, Hq, Sq, D], dk [B, Hkv, Sk, D], dv [B, Hkv, Sk, D]).
    """
    q, k, v, s_, rb, (B, Hq, Hkv, Sq, Sk, D) = _prep(q, k, v, alibi_slopes, row_kv_bounds)
    if dout.shape != q.shape:
        raise ValueError("dout must have q's shape")
    do = dout.detach().to("cpu", torch.float64)
    q, k, v = q.double(), k.double(), v.double()
    G = Hq // Hkv
    sc = _f32(1.0 / (D ** 0.5) if scale is None else scale)
    cap = 0.0 if not softcap else _f32(softcap)
    slopes = None if s_ is None else s_.double()
    wl, wr = _win(window_left), _win(window_right)
    i = torch.arange(Sq, dtype=torch.int64)[:, None]
    j = torch.arange(Sk, dtype=torch.int64)[None, :]
    adm0 = torch.ones(Sq, Sk, dtype=torch.bool)
    if causal:
        adm0 &= j <= i
    if wl >= 0:
        adm0 &= j + wl >= i
    if wr >= 0:
        adm0 &= j <= i + wr
    dq = torch.zeros(B, Hq, Sq, D, dtype=torch.float64)
    dk = torch.zeros(B, Hkv, Sk, D, dtype=torch.float64)
    dv = torch.zeros(B, Hkv, Sk, D, dtype=torch.float64)
    for b in range(B):
        adm = adm0.clone()
        if rb is not None:
            lo = rb[b, :, 0].long()[:, None]
            hi = rb[b, :, 1].long()[:, None]
            adm &= (j >= lo) & (j <= hi)
        live = adm.any(dim=1)  # rows with at least one admissible key
        for h in range(Hq):
            g = h // G
            s_pre = sc * (q[b, h] @ k[b, g].T)  # [Sq, Sk]
            s = cap * torch.tanh(s_pre / cap) if cap else s_pre.clone()
            if slopes is not None:
                s = s + slopes[h] * (j - i).double()
            s = torch.where(adm, s, torch.full_like(s, float("-inf")))
            m = torch.where(live, s.max(dim=1).values, torch.zeros(Sq, dtype=torch.float64))
            w = torch.where(adm, torch.exp(s - m[:, None]), torch.zeros_like(s))
            L = w.sum(dim=1)
            P = torch.where(live[:, None], w / torch.where(live, L, torch.ones_like(L))[:, None],
                            torch.zeros_like(w))
            dv[b, g] += P.T @ do[b, h]
            dP = do[b, h] @ v[b, g].T
            dS = (dP - (P * dP).sum(dim=1, keepdim=True)) * P
            if cap:
                dS = dS * (1.0 - torch.tanh(s_pre / cap) ** 2)
            dq[b, h] = sc * (dS @ k[b, g])
            dk[b, g] += sc * (dS.T @ q[b, h])
    return dq, dk, dv
