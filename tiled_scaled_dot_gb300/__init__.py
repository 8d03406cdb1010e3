"""tiled_scaled_dot_gb300 -- Python binding of libgbattn (GB300, sm_103a).

The binding only marshals arguments: it checks that tensors are CUDA,
contiguous and of the right dtype, turns them into device pointers and calls
the C ABI declared in include/gbattn.h.  Every step of the computation runs
in the library's CUDA kernels; there is no other code path.  If the library
has not been built, importing the entry points raises.

Operation (attention.fkc.md, attention_naive / attention_flash; "gfx942
unified attention, from the math up", sections 1-4 and 8):

    O = softmax(scale * Q K^T [softcap] [+ ALiBi] [causal / window mask]) V

with GQA (kv head h // (Hq // Hkv)), top-left causal alignment, and an
all-zero output row where no key is admissible.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

__all__ = ["attn_fwd", "attn_fwd_varlen", "attn_decode", "decode_workspace_size", "attn_decode_paged",
           "decode_paged_workspace_size", "attn_bwd", "bwd_workspace_size", "device_status", "set_wait_timeout_ns",
           "diag_umma", "diag_wait_timeout", "GbattnError", "lib", "LIB_PATH"]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgbattn.so")

GBATTN_BF16 = 0
GBATTN_F32 = 1
GBATTN_F16 = 2
_DT = {torch.bfloat16: GBATTN_BF16, torch.float32: GBATTN_F32, torch.float16: GBATTN_F16}
_DT16 = {torch.bfloat16: GBATTN_BF16, torch.float16: GBATTN_F16}  # the decode entries


class GbattnError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: status {status} ({_status_string(status)})")
        self.status = status


class _FwdParams(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("alibi_slopes", ctypes.c_void_p), ("row_kv_bounds", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("lse_out", ctypes.c_void_p),
                ("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("Sq", ctypes.c_int),
                ("Sk", ctypes.c_int), ("D", ctypes.c_int), ("softmax_scale", ctypes.c_float),
                ("causal", ctypes.c_int), ("window_left", ctypes.c_int), ("window_right", ctypes.c_int),
                ("softcap", ctypes.c_float), ("dtype", ctypes.c_int), ("stream", ctypes.c_void_p)]


class _BwdParams(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("dout", ctypes.c_void_p),
                ("alibi_slopes", ctypes.c_void_p), ("row_kv_bounds", ctypes.c_void_p),
                ("dq", ctypes.c_void_p), ("dk", ctypes.c_void_p), ("dv", ctypes.c_void_p),
                ("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("Sq", ctypes.c_int),
                ("Sk", ctypes.c_int), ("D", ctypes.c_int), ("softmax_scale", ctypes.c_float),
                ("causal", ctypes.c_int), ("window_left", ctypes.c_int), ("window_right", ctypes.c_int),
                ("softcap", ctypes.c_float), ("dtype", ctypes.c_int),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("stream", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libgbattn.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m tiled_scaled_dot_gb300.build`"
                                   " (or __graft_entry__.build()); there is no fallback path")
            L = ctypes.CDLL(LIB_PATH)
            P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
            L.attn_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, I, I, I, F, I, P]
            L.attn_fwd.restype = I
            L.attn_fwd_ex.argtypes = [ctypes.POINTER(_FwdParams)]
            L.attn_fwd_ex.restype = I
            L.attn_decode_workspace_size.argtypes = [I, I, I, I, I, I]
            L.attn_decode_workspace_size.restype = Z
            L.attn_decode.argtypes = [P, P, P, P, P, P, I, I, I, I, I, F, F, I, I, I, P, Z, I, P]
            L.attn_decode.restype = I
            L.attn_fwd_varlen.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, I, I, F, I, P]
            L.attn_fwd_varlen.restype = I
            L.attn_decode_paged_workspace_size.argtypes = [I, I, I, I, I, I, I]
            L.attn_decode_paged_workspace_size.restype = Z
            L.attn_decode_paged.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, F, I, I, I, P, Z, I, P]
            L.attn_decode_paged.restype = I
            L.attn_bwd_workspace_size.argtypes = [I, I, I, I, I, I, I, I]
            L.attn_bwd_workspace_size.restype = Z
            L.attn_bwd.argtypes = [ctypes.POINTER(_BwdParams)]
            L.attn_bwd.restype = I
            L.attn_bwd_phase_times.argtypes = [ctypes.POINTER(_BwdParams), I, ctypes.POINTER(ctypes.c_float)]
            L.attn_bwd_phase_times.restype = I
            L.gbattn_status_string.argtypes = [I]
            L.gbattn_status_string.restype = ctypes.c_char_p
            L.gbattn_device_status.argtypes = [P, I]
            L.gbattn_device_status.restype = ctypes.c_uint
            L.gbattn_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
            L.gbattn_set_wait_timeout_ns.restype = ctypes.c_uint64
            L.gbattn_version.restype = I
            L.gbattn_diag_umma.argtypes = [I, P, P, P, I, P]
            L.gbattn_diag_umma.restype = I
            L.gbattn_diag_wait_timeout.argtypes = [ctypes.c_ulonglong, P]
            L.gbattn_diag_wait_timeout.restype = I
            _lib = L
    return _lib


def _status_string(st: int) -> str:
    try:
        return lib().gbattn_status_string(st).decode()
    except Exception:  # pragma: no cover - only when the library is missing
        return "unknown"


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(t, name, dtype=None, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (layout [B, H, S, D], zero offset)")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions")


def _win(w) -> int:
    return -1 if w is None else int(w)


def attn_fwd(q, k, v, alibi_slopes=None, *, softmax_scale=None, causal=False, window_left=None,
             window_right=None, softcap=None, out=None, lse=None, row_kv_bounds=None, stream=None):
    """Attention forward.  q [B,Hq,Sq,D], k/v [B,Hkv,Sk,D] (bf16 or fp32, CUDA).

    alibi_slopes: fp32 [Hq] or None.  window_left/right: None = unbounded.
    softcap: None/0 = none.  lse: optional fp32 [B,Hq,Sq] output.
    row_kv_bounds: optional int32 [B,Sq,2] inclusive key range per query row.
    Returns out [B,Hq,Sq,D] of q's dtype.
    """
    if q.dtype not in _DT:
        raise TypeError("q must be bf16 or fp32")
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n, q.dtype, 4)
    B, Hq, Sq, D = q.shape
    Bk, Hkv, Sk, Dk = k.shape
    if tuple(v.shape) != tuple(k.shape) or Bk != B or Dk != D:
        raise ValueError("k and v must be [B, Hkv, Sk, D] with q's B and D")
    if alibi_slopes is not None:
        _check(alibi_slopes, "alibi_slopes", torch.float32, 1)
        if alibi_slopes.numel() != Hq:
            raise ValueError("alibi_slopes must be [Hq]")
    if row_kv_bounds is not None:
        _check(row_kv_bounds, "row_kv_bounds", torch.int32, 3)
        if tuple(row_kv_bounds.shape) != (B, Sq, 2):
            raise ValueError("row_kv_bounds must be [B, Sq, 2]")
    if out is None:
        out = torch.empty_like(q)
    else:
        _check(out, "out", q.dtype, 4)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    if lse is not None:
        _check(lse, "lse", torch.float32, 3)
        if tuple(lse.shape) != (B, Hq, Sq):
            raise ValueError("lse must be [B, Hq, Sq]")
    scale = (1.0 / math.sqrt(D)) if softmax_scale is None else float(softmax_scale)
    prm = _FwdParams(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                     alibi_slopes.data_ptr() if alibi_slopes is not None else None,
                     row_kv_bounds.data_ptr() if row_kv_bounds is not None else None,
                     out.data_ptr(), lse.data_ptr() if lse is not None else None,
                     B, Hq, Hkv, Sq, Sk, D, scale, int(bool(causal)), _win(window_left), _win(window_right),
                     float(softcap or 0.0), _DT[q.dtype], _stream_handle(stream).value)
    st = lib().attn_fwd_ex(ctypes.byref(prm))
    if st:
        raise GbattnError(st, "attn_fwd")
    return out


def decode_workspace_size(B, Hq, Hkv, Sk, D, num_splits=0) -> int:
    return int(lib().attn_decode_workspace_size(B, Hq, Hkv, Sk, D, num_splits))


def attn_decode(q, k, v, alibi_slopes=None, *, softmax_scale=None, softcap=None, window_left=None,
                window_right=None, num_splits=0, out=None, lse=None, workspace=None, stream=None):
    """Split-KV decode.  q [B,Hq,1,D], k/v [B,Hkv,Sk,D] bf16 or fp16 (CUDA).

    The query is the newest token, at position Sk - 1: ALiBi adds
    slope (j - (Sk - 1)); window_left admits keys j >= Sk - 1 - window_left.

    workspace: optional uint8 CUDA tensor of at least decode_workspace_size(...)
    bytes; allocated here (through torch) when None.  Returns out [B,Hq,1,D].
    """
    if q.dtype not in _DT16:
        raise TypeError(f"decode takes bf16 or fp16, got {q.dtype}")
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n, q.dtype, 4)
    B, Hq, Sq, D = q.shape
    Bk, Hkv, Sk, Dk = k.shape
    if Sq != 1:
        raise ValueError("decode takes one query row (Sq == 1)")
    if tuple(v.shape) != tuple(k.shape) or Bk != B or Dk != D:
        raise ValueError("k and v must be [B, Hkv, Sk, D] with q's B and D")
    if alibi_slopes is not None:
        _check(alibi_slopes, "alibi_slopes", torch.float32, 1)
    if out is None:
        out = torch.empty_like(q)
    else:
        _check(out, "out", q.dtype, 4)
    if lse is not None:
        _check(lse, "lse", torch.float32)
    need = decode_workspace_size(B, Hq, Hkv, Sk, D, num_splits)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    scale = (1.0 / math.sqrt(D)) if softmax_scale is None else float(softmax_scale)
    st = lib().attn_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(alibi_slopes), _ptr(out), _ptr(lse),
                           B, Hq, Hkv, Sk, D, scale, float(softcap or 0.0), _win(window_left),
                           _win(window_right), int(num_splits), _ptr(workspace), ws_bytes, _DT16[q.dtype],
                           _stream_handle(stream))
    if st:
        raise GbattnError(st, "attn_decode")
    return out


def attn_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, seqused_k=None, alibi_slopes=None, *,
                    softmax_scale=None, causal=False, window_left=None, window_right=None, softcap=None, out=None,
                    lse=None, stream=None):
    """Packed variable-length attention (see attn_fwd_varlen in gbattn.h).

    q [total_q, Hq, D], k / v [total_k, Hkv, D] bf16 or fp16; cu_seqlens_q / cu_seqlens_k
    int32 [B + 1] and seqused_k int32 [B] (optional), all CUDA; max_seqlen_q an
    int at least every sequence's query count.  Causal masks align bottom-right.
    lse (optional) fp32 [Hq, total_q].  Returns out [total_q, Hq, D].
    """
    if q.dtype not in _DT16:
        raise TypeError(f"packed sequences take bf16 or fp16, got {q.dtype}")
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n, q.dtype, 3)
    for t, n in ((cu_seqlens_q, "cu_seqlens_q"), (cu_seqlens_k, "cu_seqlens_k"), (seqused_k, "seqused_k")):
        if t is not None:
            _check(t, n, torch.int32, 1)
    total_q, Hq, D = q.shape
    total_k, Hkv, Dk = k.shape
    B = cu_seqlens_q.shape[0] - 1
    if tuple(v.shape) != tuple(k.shape) or Dk != D or cu_seqlens_k.shape[0] != B + 1:
        raise ValueError("k and v must be [total_k, Hkv, D] with q's D; cu_seqlens_* must be [B + 1]")
    if seqused_k is not None and seqused_k.shape[0] != B:
        raise ValueError("seqused_k must be [B]")
    if alibi_slopes is not None:
        _check(alibi_slopes, "alibi_slopes", torch.float32, 1)
    if out is None:
        out = torch.empty_like(q)
    else:
        _check(out, "out", q.dtype, 3)
    if lse is not None:
        _check(lse, "lse", torch.float32)
    scale = (1.0 / math.sqrt(D)) if softmax_scale is None else float(softmax_scale)
    st = lib().attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), _ptr(seqused_k),
                               _ptr(alibi_slopes), _ptr(out), _ptr(lse), B, Hq, Hkv, D, total_q, total_k,
                               int(max_seqlen_q), scale, 1 if causal else 0, _win(window_left), _win(window_right),
                               float(softcap or 0.0), _DT16[q.dtype], _stream_handle(stream))
    if st:
        raise GbattnError(st, "attn_fwd_varlen")
    return out


def decode_paged_workspace_size(B, Hq, Hkv, max_blocks_per_seq, block_size, D, num_splits=0) -> int:
    return int(lib().attn_decode_paged_workspace_size(B, Hq, Hkv, max_blocks_per_seq, block_size, D, num_splits))


def attn_decode_paged(q, k_cache, v_cache, block_table, context_lens, alibi_slopes=None, *, softmax_scale=None,
                      softcap=None, window_left=None, window_right=None, num_splits=0, out=None, lse=None,
                      workspace=None, stream=None):
    """Decode over a paged KV cache (see attn_decode_paged in gbattn.h).

    q [B,Hq,1,D] bf16 or fp16; k_cache / v_cache [num_blocks, block_size, Hkv, D] of the same type;
    block_table [B, max_blocks] and context_lens [B] int32 or uint32 (CUDA),
    read as uint32.  Returns out [B,Hq,1,D].
    """
    if q.dtype not in _DT16:
        raise TypeError(f"paged decode takes bf16 or fp16, got {q.dtype}")
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _check(t, n, q.dtype, 4)
    for t, n in ((block_table, "block_table"), (context_lens, "context_lens")):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous CUDA tensor")
        if t.dtype not in (torch.int32, torch.uint32):
            raise ValueError(f"{n} must be int32 or uint32")
    B, Hq, Sq, D = q.shape
    num_blocks, block_size, Hkv, Dk = k_cache.shape
    if Sq != 1:
        raise ValueError("paged decode takes one query row (Sq == 1)")
    if tuple(v_cache.shape) != tuple(k_cache.shape) or Dk != D:
        raise ValueError("k_cache and v_cache must be [num_blocks, block_size, Hkv, D] with q's D")
    if block_table.dim() != 2 or block_table.shape[0] != B or tuple(context_lens.shape) != (B,):
        raise ValueError("block_table [B, max_blocks], context_lens [B]")
    if alibi_slopes is not None:
        _check(alibi_slopes, "alibi_slopes", torch.float32, 1)
    if out is None:
        out = torch.empty_like(q)
    else:
        _check(out, "out", q.dtype, 4)
    if lse is not None:
        _check(lse, "lse", torch.float32)
    max_blocks = block_table.shape[1]
    need = decode_paged_workspace_size(B, Hq, Hkv, max_blocks, block_size, D, num_splits)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    scale = (1.0 / math.sqrt(D)) if softmax_scale is None else float(softmax_scale)
    st = lib().attn_decode_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(context_lens),
                                 _ptr(alibi_slopes), _ptr(out), _ptr(lse), B, Hq, Hkv, D, num_blocks, block_size,
                                 max_blocks, scale, float(softcap or 0.0), _win(window_left), _win(window_right),
                                 int(num_splits), _ptr(workspace), ws_bytes, _DT16[q.dtype],
                                 _stream_handle(stream))
    if st:
        raise GbattnError(st, "attn_decode_paged")
    return out


def bwd_workspace_size(B, Hq, Hkv, Sq, Sk, D, recompute=True, dtype=torch.bfloat16) -> int:
    return int(lib().attn_bwd_workspace_size(B, Hq, Hkv, Sq, Sk, D, _DT[dtype], int(bool(recompute))))


def attn_bwd(q, k, v, dout, out=None, lse=None, alibi_slopes=None, *, softmax_scale=None, causal=False,
             window_left=None, window_right=None, softcap=None, row_kv_bounds=None, dq=None, dk=None, dv=None,
             workspace=None, stream=None, phase_times_reps=0):
    """Attention backward by recompute.  q, dout [B,Hq,Sq,D], k/v [B,Hkv,Sk,D]
    (bf16, fp16 or fp32, CUDA); the forward's flags.

    out and lse: the forward's output and fp32 lse [B,Hq,Sq] (attn_fwd with
    lse=...), both or neither; when neither, the library recomputes them into
    the workspace.  workspace: optional uint8 CUDA tensor of at least
    bwd_workspace_size(...) bytes, allocated here (through torch) when None.
    Returns (dq [B,Hq,Sq,D], dk [B,Hkv,Sk,D], dv [B,Hkv,Sk,D]) of q's dtype.
    With phase_times_reps = n > 0 the call is the synchronous profiling form
    (attn_bwd_phase_times): it runs n times and returns, after the gradients,
    the mean milliseconds of (forward recompute, prep, dK/dV, dQ).
    """
    if q.dtype not in _DT:
        raise TypeError(f"attn_bwd takes bf16, fp16 or fp32, got {q.dtype}")
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (dout, "dout")):
        _check(t, n, q.dtype, 4)
    B, Hq, Sq, D = q.shape
    Bk, Hkv, Sk, Dk = k.shape
    if tuple(v.shape) != tuple(k.shape) or Bk != B or Dk != D or dout.shape != q.shape:
        raise ValueError("k, v [B, Hkv, Sk, D]; dout of q's shape")
    if (out is None) != (lse is None):
        raise ValueError("give both out and lse, or neither")
    if out is not None:
        _check(out, "out", q.dtype, 4)
        _check(lse, "lse", torch.float32, 3)
        if out.shape != q.shape or tuple(lse.shape) != (B, Hq, Sq):
            raise ValueError("out [B, Hq, Sq, D] and lse [B, Hq, Sq]")
    if alibi_slopes is not None:
        _check(alibi_slopes, "alibi_slopes", torch.float32, 1)
        if alibi_slopes.numel() != Hq:
            raise ValueError("alibi_slopes must be [Hq]")
    if row_kv_bounds is not None:
        _check(row_kv_bounds, "row_kv_bounds", torch.int32, 3)
        if tuple(row_kv_bounds.shape) != (B, Sq, 2):
            raise ValueError("row_kv_bounds must be [B, Sq, 2]")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for t, n, like in ((dq, "dq", q), (dk, "dk", k), (dv, "dv", v)):
        _check(t, n, q.dtype, 4)
        if t.shape != like.shape:
            raise ValueError(f"{n} must have the shape of its input")
    need = bwd_workspace_size(B, Hq, Hkv, Sq, Sk, D, out is None, q.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    else:
        _check(workspace, "workspace", torch.uint8, 1)
    scale = (1.0 / math.sqrt(D)) if softmax_scale is None else float(softmax_scale)
    prm = _BwdParams(q.data_ptr(), k.data_ptr(), v.data_ptr(), _ptr(out), _ptr(lse), dout.data_ptr(),
                     _ptr(alibi_slopes), _ptr(row_kv_bounds), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                     B, Hq, Hkv, Sq, Sk, D, scale, int(bool(causal)), _win(window_left), _win(window_right),
                     float(softcap or 0.0), _DT[q.dtype], workspace.data_ptr(), workspace.numel(),
                     _stream_handle(stream).value)
    if phase_times_reps:
        ms = (ctypes.c_float * 4)()
        st = lib().attn_bwd_phase_times(ctypes.byref(prm), int(phase_times_reps), ms)
        if st:
            raise GbattnError(st, "attn_bwd_phase_times")
        return dq, dk, dv, tuple(float(x) for x in ms)
    st = lib().attn_bwd(ctypes.byref(prm))
    if st:
        raise GbattnError(st, "attn_bwd")
    return dq, dk, dv


def device_status(stream=None, clear: bool = True) -> int:
    """Synchronise the stream and read (and clear) the device status word."""
    return int(lib().gbattn_device_status(_stream_handle(stream), 1 if clear else 0))


def set_wait_timeout_ns(ns: int) -> int:
    return int(lib().gbattn_set_wait_timeout_ns(int(ns)))


def diag_umma(mode: int, a, b, n: int, stream=None):
    """One tcgen05 tile product through the kernels' layouts (see gbattn_diag.h)."""
    _check(a, "a", torch.bfloat16, 2)
    _check(b, "b", torch.bfloat16, 2)
    c = torch.empty(128, n, dtype=torch.float32, device=a.device)
    st = lib().gbattn_diag_umma(int(mode), _ptr(a), _ptr(b), _ptr(c), int(n), _stream_handle(stream))
    if st:
        raise GbattnError(st, "gbattn_diag_umma")
    return c


def diag_wait_timeout(timeout_ns: int, stream=None) -> None:
    """Launch a bounded wait that nothing satisfies (see gbattn_diag.h); it
    gives up after timeout_ns and sets bit 16 of the device status word."""
    st = lib().gbattn_diag_wait_timeout(int(timeout_ns), _stream_handle(stream))
    if st:
        raise GbattnError(st, "gbattn_diag_wait_timeout")
