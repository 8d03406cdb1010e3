"""Host-side checks of the C ABI: the library builds, loads, exports every
symbol the headers declare, and rejects bad arguments before launching
anything (these calls never reach a kernel, so they need no GPU)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from tiled_scaled_dot_gb300 import build
    build.build()
    import tiled_scaled_dot_gb300 as g
    return g.lib()


def _declared_functions():
    names = []
    for h in sorted(glob.glob(os.path.join(ROOT, "include", "*.h"))):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        text = re.sub(r"^\s*#[^\n]*", "", text, flags=re.M)  # preprocessor lines
        for m in re.finditer(r"\b([A-Za-z_][A-Za-z0-9_]*)\s*\(([^;{}]*)\)\s*;", text):
            names.append(m.group(1))
    return names


def test_every_declared_symbol_is_exported(L):
    names = _declared_functions()
    for expected in ("attn_fwd", "attn_fwd_ex", "attn_decode", "attn_decode_workspace_size",
                     "gbattn_status_string", "gbattn_device_status", "gbattn_set_wait_timeout_ns",
                     "gbattn_version", "gbattn_diag_umma", "gbattn_diag_wait_timeout",
                     "attn_decode_paged", "attn_decode_paged_workspace_size", "attn_fwd_varlen"):
        assert expected in names
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    for st in range(0, 5):
        assert L.gbattn_status_string(st)
    assert L.gbattn_status_string(99) == b"unknown status"
    assert L.gbattn_version() >= 100


FAKE = 1 << 20  # a non-null, 16-byte aligned pseudo pointer; never dereferenced on these paths


def _fwd(L, **kw):
    a = dict(q=FAKE, k=FAKE * 2, v=FAKE * 3, alibi=None, out=FAKE * 4, B=1, Hq=2, Hkv=1, Sq=64, Sk=64, D=64,
             scale=0.125, causal=0, wl=-1, wr=-1, softcap=0.0, dtype=0, stream=None)
    a.update(kw)
    return L.attn_fwd(a["q"], a["k"], a["v"], a["alibi"], a["out"], a["B"], a["Hq"], a["Hkv"], a["Sq"], a["Sk"],
                      a["D"], a["scale"], a["causal"], a["wl"], a["wr"], a["softcap"], a["dtype"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(B=0), 1), (dict(Hq=3, Hkv=2), 1), (dict(Sq=0), 1), (dict(Sk=-1), 1),
    (dict(q=None), 1), (dict(out=None), 1), (dict(scale=0.0), 1), (dict(scale=float("nan")), 1),
    (dict(softcap=-1.0), 1), (dict(wl=-2), 1), (dict(causal=2), 1), (dict(dtype=7), 1),
    (dict(q=FAKE + 2), 1), (dict(out=FAKE), 1),  # misaligned; out aliasing q
    (dict(D=96), 2), (dict(D=256), 2),
])
def test_forward_rejects_bad_arguments(L, kw, status):
    assert _fwd(L, **kw) == status


def test_decode_rejects_bad_arguments(L):
    P = ctypes.c_void_p
    # q, k, v, slopes, out, lse, B, Hq, Hkv, Sk, D, scale, softcap, window_left, window_right,
    # splits, ws, ws_bytes, dtype, stream
    base = [P(FAKE), P(FAKE * 2), P(FAKE * 3), None, P(FAKE * 4), None, 2, 4, 2, 128, 128, 0.1, 0.0, -1, -1, 0,
            None, 0, 0, None]
    def call(i, val):
        a = list(base)
        a[i] = val
        return L.attn_decode(*a)
    assert call(6, 0) == 1          # B = 0
    assert call(8, 3) == 1          # Hq % Hkv
    assert call(10, 96) == 2        # D
    assert call(18, 1) == 2         # fp32 decode not built
    assert call(15, -1) == 1        # negative split count
    assert call(13, -2) == 1        # window_left below -1
    assert call(14, -3) == 1        # window_right below -1
    assert L.attn_decode_workspace_size(0, 4, 2, 128, 128, 0) == 0
    assert L.attn_decode_workspace_size(2, 4, 2, 8192, 128, 1) == 0
    n = L.attn_decode_workspace_size(2, 4, 2, 8192, 128, 4)
    assert n >= 2 * 4 * 4 * (128 + 1) * 4
    # a split count above the tile count is clamped to one split per 64 keys
    assert L.attn_decode_workspace_size(1, 1, 1, 128, 64, 1000) == L.attn_decode_workspace_size(1, 1, 1, 128, 64, 2)


def test_fwd_ex_null_params(L):
    assert L.attn_fwd_ex(None) == 1


def test_diag_wait_timeout_rejects_bad_limits(L):
    assert L.gbattn_diag_wait_timeout(0, None) == 1
    assert L.gbattn_diag_wait_timeout(10_000_000_001, None) == 1


def test_binding_refuses_cpu_tensors():
    import torch
    import tiled_scaled_dot_gb300 as g
    q = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        g.attn_fwd(q, q[:, :1], q[:, :1])


def test_paged_decode_rejects_bad_arguments(L):
    P = ctypes.c_void_p
    # q, k_cache, v_cache, block_table, context_lens, slopes, out, lse,
    # B, Hq, Hkv, D, num_blocks, block_size, max_blocks, scale, softcap, window_left, window_right,
    # splits, ws, ws_bytes, dtype, stream
    base = [P(FAKE), P(FAKE * 2), P(FAKE * 3), P(FAKE * 5), P(FAKE * 6), None, P(FAKE * 4), None,
            2, 4, 2, 128, 10, 64, 4, 0.1, 0.0, -1, -1, 1, None, 0, 0, None]
    def call(i, val):
        a = list(base)
        a[i] = val
        return L.attn_decode_paged(*a)
    assert call(13, 48) == 1          # block size not a power of two
    assert call(13, 8) == 1           # block size below 16
    assert call(12, 0) == 1           # no blocks
    assert call(14, 0) == 1           # empty table
    assert call(3, None) == 1         # no block table
    assert call(4, P(FAKE * 6 + 2)) == 1  # misaligned context lengths
    assert call(11, 96) == 2          # D
    assert call(22, 1) == 2           # fp32 not built
    assert call(22, 3) == 1           # no such type
    assert call(17, -2) == 1          # window_left below -1
    assert call(18, -2) == 1          # window_right below -1
    assert L.attn_decode_paged_workspace_size(2, 4, 2, 4, 48, 128, 0) == 0
    assert L.attn_decode_paged_workspace_size(2, 4, 2, 4, 64, 128, 1) == 0
    assert L.attn_decode_paged_workspace_size(2, 4, 2, 4, 64, 128, 2) == \
        L.attn_decode_workspace_size(2, 4, 2, 256, 128, 2)


def test_varlen_rejects_bad_arguments(L):
    P = ctypes.c_void_p
    # q, k, v, cu_q, cu_k, used_k, slopes, out, lse, B, Hq, Hkv, D, total_q, total_k, max_q,
    # scale, causal, wl, wr, softcap, dtype, stream
    base = [P(FAKE), P(FAKE * 2), P(FAKE * 3), P(FAKE * 5), P(FAKE * 6), None, None, P(FAKE * 4), None,
            2, 4, 2, 128, 100, 100, 64, 0.1, 1, -1, -1, 0.0, 0, None]
    def call(i, val):
        a = list(base)
        a[i] = val
        return L.attn_fwd_varlen(*a)
    assert call(13, 0) == 1           # total_q
    assert call(14, 0) == 1           # total_k
    assert call(15, 0) == 1           # max_seqlen_q
    assert call(3, None) == 1         # cu_seqlens_q
    assert call(5, P(FAKE * 7 + 2)) == 1  # misaligned seqused_k
    assert call(10, 3) == 1           # Hq % Hkv
    assert call(17, 2) == 1           # causal flag
    assert call(18, -2) == 1          # window
    assert call(12, 96) == 2          # D
    assert call(21, 1) == 2           # fp32 not built
    assert call(21, 7) == 1           # no such type
    assert call(7, P(FAKE)) == 1      # out aliasing q


def test_backward_rejects_bad_arguments(L):
    import tiled_scaled_dot_gb300 as g
    L.attn_bwd.argtypes = [ctypes.POINTER(g._BwdParams)]
    B, Hq, Hkv, S, D = 2, 4, 2, 256, 128
    ws_need = L.attn_bwd_workspace_size(B, Hq, Hkv, S, S, D, 0, 1)
    ws_given = L.attn_bwd_workspace_size(B, Hq, Hkv, S, S, D, 0, 0)
    assert ws_need > ws_given > 0
    # the recomputed fp32 output takes twice the 16-bit one's bytes
    assert L.attn_bwd_workspace_size(B, Hq, Hkv, S, S, D, 1, 1) - ws_given == 2 * (ws_need - ws_given) - B * Hq * S * 4
    assert L.attn_bwd_workspace_size(B, 3, Hkv, S, S, D, 0, 1) == 0  # Hq % Hkv
    assert L.attn_bwd_workspace_size(B, Hq, Hkv, S, S, D, 7, 1) == 0  # dtype
    nq, nkv = B * Hq * S * D * 2, B * Hkv * S * D * 2
    base = dict(q=FAKE, k=FAKE + nq, v=FAKE + nq + nkv, dout=FAKE + 2 * nq + 2 * nkv, dq=FAKE * 64,
                dk=FAKE * 64 + nq, dv=FAKE * 64 + nq + nkv, B=B, Hq=Hq, Hkv=Hkv, Sq=S, Sk=S, D=D,
                softmax_scale=0.088, causal=1, window_left=-1, window_right=-1, softcap=0.0, dtype=0,
                workspace=FAKE * 128, workspace_bytes=ws_need)

    def call(**change):
        a = dict(base)
        a.update(change)
        prm = g._BwdParams(**a)
        return L.attn_bwd(ctypes.byref(prm))

    assert L.attn_bwd(None) == 1
    assert call(q=None) == 1
    assert call(workspace=None) == 1
    assert call(workspace_bytes=ws_need - 1) == 1
    assert call(workspace=FAKE * 128 + 16) == 1          # workspace not 256-byte aligned
    assert call(out=FAKE * 256) == 1                     # out without lse
    assert call(Hkv=3) == 1                              # Hq % Hkv
    assert call(causal=2) == 1
    assert call(window_left=-2) == 1
    assert call(D=96) == 2
    assert call(dtype=3) == 1                            # no such dtype
    assert call(dq=FAKE) == 1                            # dq aliasing q
    assert call(dv=FAKE * 64 + 8) == 1                   # dv overlapping dq (and misaligned)
    assert call(dk=FAKE * 128) == 1                      # dk inside the workspace
