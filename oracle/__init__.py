"""CPU oracle for the verify-and-accept step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  It wraps ``sv_oracle.c`` (plain C, double
precision, its own Philox) through ctypes and shares no code with the CUDA
library.  ``build()`` compiles the C file with gcc; importing this module
builds it on demand when the shared object is missing or stale.

Every function here marshals numpy arrays; the arithmetic lives in the C file,
where each function cites the passage of the pages it follows.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sv_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

DRAW_ACCEPT, DRAW_SAMPLE, DRAW_DRAFT, DRAW_TREE = 0, 1, 2, 3
ROW_NAN, ROW_BAD_TOKEN, ROW_RESID_ZERO, ROW_P_ZERO, ROW_BAD_TREE = 1, 2, 4, 8, 16


def build(force: bool = False) -> str:
    """Compile sv_oracle.c into liboracle.so (gcc, -ffp-contract=off)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call([
        "gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
        "-Wall", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(build())
        _declare(_lib)
    return _lib


_f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
_u32p = np.ctypeslib.ndpointer(np.uint32, flags="C_CONTIGUOUS")
_u64p = np.ctypeslib.ndpointer(np.uint64, flags="C_CONTIGUOUS")
_u8p = np.ctypeslib.ndpointer(np.uint8, flags="C_CONTIGUOUS")


def _declare(L):
    L.orc_philox4x32_10.argtypes = [_u32p, _u32p, _u32p]
    L.orc_philox4x32_10.restype = None
    L.orc_u24.argtypes = [C.c_uint64, C.c_uint64, C.c_uint32, C.c_uint32, C.c_uint32]
    L.orc_u24.restype = C.c_uint32
    L.orc_row_stats.argtypes = [_f32p, C.c_int, C.c_double,
                                C.POINTER(C.c_double), C.POINTER(C.c_double)]
    L.orc_row_stats.restype = None
    L.orc_softmax.argtypes = [_f32p, C.c_int, C.c_double, _f64p]
    L.orc_softmax.restype = None
    L.orc_accept.argtypes = [C.c_double, C.c_double, C.c_double]
    L.orc_accept.restype = C.c_int
    L.orc_residual.argtypes = [_f64p, _f64p, C.c_int, _f64p]
    L.orc_residual.restype = None
    L.orc_invcdf_f64.argtypes = [_f64p, C.c_int, C.c_double]
    L.orc_invcdf_f64.restype = C.c_int
    L.orc_tree_expand.argtypes = [_f32p, C.c_int, C.c_int, C.c_float, _f32p, C.c_int,
                                  _i32p, _f64p]
    L.orc_tree_select.argtypes = [_f32p, _i32p, C.c_int, C.c_int, C.c_int, _i32p]
    L.orc_tree_attention.argtypes = [_f32p, _f32p, _i32p, _u64p, C.c_int, C.c_int, C.c_int,
                                     C.c_int, C.c_int, C.c_int, C.c_double, C.c_void_p,
                                     C.c_int, _f64p, _f64p]
    L.orc_tree_attention.restype = C.c_int
    L.orc_tree_finalize.argtypes = [_i32p, _i32p, _f32p, _i32p, C.c_int, C.c_int, C.c_int,
                                    _i32p, _i32p, _f32p]
    L.orc_argmax.argtypes = [_f32p, C.c_int]
    L.orc_argmax.restype = C.c_int
    L.orc_exp32.argtypes = [C.c_float]
    L.orc_exp32.restype = C.c_float
    L.orc_sample_repro.argtypes = [_f32p, C.c_void_p, C.c_int, C.c_float, C.c_uint32,
                                   C.POINTER(C.c_double), C.POINTER(C.c_int)]
    L.orc_sample_repro.restype = C.c_int
    L.orc_sample_repro_many.argtypes = [_f32p, C.c_void_p, C.c_int, C.c_float, _u32p, C.c_int,
                                        _i32p, _f64p, C.POINTER(C.c_int)]
    L.orc_sample_repro_many.restype = C.c_int
    L.orc_verify.argtypes = [
        _f32p, C.c_int64, _f32p, C.c_int64, C.c_int, C.c_int, C.c_float,
        C.c_void_p, C.c_int, _i32p, _i32p, C.c_int, C.c_uint64, C.c_uint64,
        C.c_void_p, C.c_int, C.c_void_p, C.c_void_p,
        _i32p, C.c_int, _i32p, _f64p, _f64p, _f64p, C.c_int, _f64p, _u32p]
    L.orc_verify.restype = C.c_int
    L.orc_verify_ex.argtypes = L.orc_verify.argtypes + [C.c_int]
    L.orc_verify_ex.restype = C.c_int
    L.orc_tree_valid.argtypes = [_i32p, C.c_void_p, C.c_int]
    L.orc_tree_valid.restype = C.c_int
    L.orc_tree_best_path.argtypes = [_i32p, _f32p, C.c_int, C.c_int, _i32p]
    L.orc_tree_best_path.restype = C.c_int
    L.orc_verify_tree.argtypes = [
        _f32p, _f32p, _i32p, _i32p, _f32p, C.c_int, C.c_int, C.c_int, C.c_int,
        C.c_float, C.c_uint64, C.c_uint64, C.c_void_p, _i32p, _i32p, _i32p, _f64p, _f64p,
        _f64p, _f64p, _u32p]
    L.orc_verify_tree.restype = C.c_int
    L.orc_tree_mask.argtypes = [_i32p, C.c_int, C.c_int, _u64p, _i32p]
    L.orc_tree_mask.restype = None
    L.orc_kv_compact.argtypes = [
        _u8p, _u8p, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int,
        _i32p, _i32p, _i32p, _i32p, C.c_int, _i32p]
    L.orc_kv_compact.restype = None
    L.orc_expected_tokens.argtypes = [C.c_double, C.c_int]
    L.orc_expected_tokens.restype = C.c_double
    L.orc_speedup.argtypes = [C.c_double, C.c_int, C.c_double]
    L.orc_speedup.restype = C.c_double


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


# ---------------------------------------------------------------- primitives
def philox4x32_10(ctr, key):
    out = np.zeros(4, np.uint32)
    lib().orc_philox4x32_10(np.asarray(ctr, np.uint32), np.asarray(key, np.uint32), out)
    return out


def u24(seed, step, seq, pos, draw):
    return int(lib().orc_u24(seed, step, seq, pos, draw))


def row_stats(x, T=1.0):
    m, s = C.c_double(), C.c_double()
    x = _f32(x)
    lib().orc_row_stats(x, x.size, T, C.byref(m), C.byref(s))
    return m.value, s.value


def softmax(x, T=1.0):
    x = _f32(x)
    out = np.empty(x.size, np.float64)
    lib().orc_softmax(x, x.size, T, out)
    return out


def accept(q_prob, p_prob, u):
    return bool(lib().orc_accept(q_prob, p_prob, u))


def residual(q, p):
    q = np.ascontiguousarray(q, np.float64)
    p = np.ascontiguousarray(p, np.float64)
    out = np.empty_like(q)
    lib().orc_residual(q, p, q.size, out)
    return out


def invcdf(w, t):
    w = np.ascontiguousarray(w, np.float64)
    return int(lib().orc_invcdf_f64(w, w.size, t))


def tree_expand(dlogits, fscore, K, T=1.0):
    """Per frontier row ([..., V] logits, [...] path scores): the K tokens with
    the largest logits (ties to the lower id) and their child scores.
    Returns (tokens [..., K] int32, scores [..., K] float64)."""
    x = _f32(dlogits)
    V = x.shape[-1]
    lead = x.shape[:-1]
    R = int(np.prod(lead)) if lead else 1
    fs = _f32(fscore).reshape(-1)
    tok = np.empty(R * K, np.int32)
    sc = np.empty(R * K, np.float64)
    rc = lib().orc_tree_expand(x.reshape(-1), R, V, float(T), fs, K, tok, sc)
    assert rc == 0
    return tok.reshape(lead + (K,)), sc.reshape(lead + (K,))


def tree_select(score, token, K):
    """Per sequence ([B][C]) the indices of the K best candidates."""
    s, t = _f32(score), _i32(token)
    B, Cn = s.shape
    out = np.empty((B, K), np.int32)
    assert lib().orc_tree_select(s.reshape(-1), t.reshape(-1), B, Cn, K, out.reshape(-1)) == 0
    return out


def tree_finalize(cparent, ctoken, cscore, clevel, Tn):
    """Per sequence ([B][C] candidates) the Tn-slot tree: parent, token, score."""
    cp, ct, cl = _i32(cparent), _i32(ctoken), _i32(clevel)
    cs = _f32(cscore)
    B, Cn = cp.shape
    parent = np.empty((B, Tn), np.int32)
    token = np.empty((B, Tn), np.int32)
    score = np.empty((B, Tn), np.float32)
    assert lib().orc_tree_finalize(cp.reshape(-1), ct.reshape(-1), cs.reshape(-1),
                                   cl.reshape(-1), B, Cn, Tn, parent.reshape(-1),
                                   token.reshape(-1), score.reshape(-1)) == 0
    return parent, token, score


def argmax(x):
    """Arg max of a row, ties to the lowest index (greedy verification)."""
    x = _f32(x)
    return int(lib().orc_argmax(x, x.size))


def exp32(a):
    return np.float32(lib().orc_exp32(float(a)))


def sample_repro(xq, xp, u24_, T=1.0):
    """Residual (xp given) or bonus (xp None) sample in the kernel arithmetic."""
    xq = _f32(xq)
    invT = np.float32(np.float32(1.0) / np.float32(T))
    gap, rz = C.c_double(), C.c_int()
    if xp is not None:
        xp = _f32(xp)
        k = lib().orc_sample_repro(xq, xp.ctypes.data, xq.size, float(invT), u24_,
                                   C.byref(gap), C.byref(rz))
    else:
        k = lib().orc_sample_repro(xq, None, xq.size, float(invT), u24_,
                                   C.byref(gap), C.byref(rz))
    return int(k), gap.value, bool(rz.value)


def sample_repro_many(xq, xp, u24s, T=1.0):
    """Many draws on one row (pair) in the kernel arithmetic: the weights are
    formed once.  Returns (tokens [n], gaps [n], resid_zero)."""
    xq = _f32(xq)
    u = np.ascontiguousarray(u24s, np.uint32)
    invT = np.float32(np.float32(1.0) / np.float32(T))
    tok = np.empty(u.size, np.int32)
    gaps = np.empty(u.size, np.float64)
    rz = C.c_int()
    keep = _f32(xp) if xp is not None else None  # holds the buffer during the call
    xpp = keep.ctypes.data if keep is not None else None
    rc = lib().orc_sample_repro_many(xq, xpp, xq.size, float(invT), u, u.size, tok, gaps,
                                     C.byref(rz))
    assert rc == 0
    return tok, gaps, bool(rz.value)


# ---------------------------------------------------------------- verify
def _verify_core(vlog, dlog, V, T, path, path_stride, npos, tok, tok_stride,
                 seed, step, u_acc=None, u_samp=None, v_bstride=None,
                 d_bstride=None, B=None, maxpos=None, seq_ids=None, early_exit=False):
    vlog = _f32(vlog).reshape(-1)
    dlog = _f32(dlog).reshape(-1)
    npos = _i32(npos)
    B = npos.size if B is None else B
    tok = _i32(tok)
    maxpos = int(npos.max()) if maxpos is None else maxpos
    out_tok = np.empty((B, maxpos + 1), np.int32)
    out_acc = np.empty(B, np.int32)
    out_q = np.empty((B, max(maxpos, 1)), np.float64)
    out_p = np.empty((B, max(maxpos, 1)), np.float64)
    out_m = np.empty((B, maxpos + 1), np.float64)
    out_gap = np.empty(B, np.float64)
    out_st = np.empty(B, np.uint32)
    keep = []
    pth = None
    if path is not None:
        pth = _i32(path)
        keep.append(pth)
    ua = None
    if u_acc is not None:
        ua = np.ascontiguousarray(u_acc, np.uint32)
        keep.append(ua)
    us = None
    if u_samp is not None:
        us = np.ascontiguousarray(u_samp, np.uint32)
        keep.append(us)
    sid = None
    if seq_ids is not None:
        sid = _i32(seq_ids)
        keep.append(sid)
    rc = lib().orc_verify_ex(
        vlog, v_bstride, dlog, d_bstride, B, V, T,
        pth.ctypes.data if pth is not None else None, path_stride, npos, tok,
        tok_stride, seed, step,
        ua.ctypes.data if ua is not None else None,
        ua.shape[-1] if ua is not None else 0,
        us.ctypes.data if us is not None else None,
        sid.ctypes.data if sid is not None else None,
        out_tok, maxpos + 1, out_acc, out_q, out_p, out_m, maxpos, out_gap, out_st,
        1 if early_exit else 0)
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return dict(tokens=out_tok, accept_len=out_acc, q_prob=out_q[:, :maxpos],
                p_prob=out_p[:, :maxpos], margin=out_m, gap=out_gap, status=out_st)


def verify_chain(vlogits, dlogits, draft_tokens, T=1.0, seed=0, step=0,
                 u_acc=None, u_samp=None, shared_rows=False, seq_ids=None,
                 early_exit=False):
    """Chain verify.  vlogits [B][N+1][V], dlogits [B][N][V], draft_tokens [B][N].

    With ``shared_rows`` the logits are a single [N+1][V] / [N][V] set used by
    every sequence (for enumeration tests).  With ``early_exit`` only the rows
    the walk reaches are checked and reported (T > 0): a bad row or token
    after the first rejection does not fault the sequence, and q(d), p(d) and
    the margin are NaN after the rejecting position."""
    draft_tokens = _i32(draft_tokens)
    B, N = draft_tokens.shape
    vl = _f32(vlogits)
    V = vl.shape[-1]
    vstride = 0 if shared_rows else (N + 1) * V
    dstride = 0 if shared_rows else N * V
    if N == 0:
        dl = np.zeros(1, np.float32)
    else:
        dl = _f32(dlogits)
    return _verify_core(vl, dl, V, T, None, 0, np.full(B, N, np.int32),
                        draft_tokens, N, seed, step, u_acc, u_samp,
                        v_bstride=vstride, d_bstride=dstride, B=B, maxpos=N,
                        seq_ids=seq_ids, early_exit=early_exit)


def verify_tree(vlogits, dlogits, parent, token, score, max_depth, T=1.0,
                seed=0, step=0, seq_ids=None):
    """Tree verify.  vlogits/dlogits [B][T][V]; parent/token/score [B][T]."""
    vl = _f32(vlogits)
    dl = _f32(dlogits)
    parent = _i32(parent)
    token = _i32(token)
    score = _f32(score)
    B, Tn = parent.shape
    V = vl.shape[-1]
    P = max_depth + 1
    out_path = np.empty((B, P), np.int32)
    out_tok = np.empty((B, P), np.int32)
    out_acc = np.empty(B, np.int32)
    out_q = np.empty((B, max(max_depth, 1)), np.float64)
    out_p = np.empty((B, max(max_depth, 1)), np.float64)
    out_m = np.empty((B, P), np.float64)
    out_gap = np.empty(B, np.float64)
    out_st = np.empty(B, np.uint32)
    sid = _i32(seq_ids) if seq_ids is not None else None
    lib().orc_verify_tree(vl.reshape(-1), dl.reshape(-1), parent.reshape(-1),
                          token.reshape(-1), score.reshape(-1), B, Tn, max_depth,
                          V, T, seed, step, sid.ctypes.data if sid is not None else None,
                          out_path, out_tok, out_acc, out_q,
                          out_p, out_m, out_gap, out_st)
    return dict(path=out_path, tokens=out_tok, accept_len=out_acc,
                q_prob=out_q[:, :max_depth], p_prob=out_p[:, :max_depth],
                margin=out_m, gap=out_gap, status=out_st)


def tree_valid(parent, score=None):
    parent = _i32(parent)
    sc = _f32(score) if score is not None else None
    return bool(lib().orc_tree_valid(parent, sc.ctypes.data if sc is not None else None,
                                     parent.size))


def tree_best_path(parent, score, max_depth):
    parent = _i32(parent)
    score = _f32(score)
    path = np.full(max_depth + 1, -1, np.int32)
    D = lib().orc_tree_best_path(parent, score, parent.size, max_depth, path)
    return path[:D + 1].copy()


def tree_mask(parent):
    parent = _i32(parent)
    if parent.ndim == 1:
        parent = parent[None]
    B, T = parent.shape
    W = (T + 63) // 64
    mask = np.empty((B, T, W), np.uint64)
    depth = np.empty((B, T), np.int32)
    lib().orc_tree_mask(parent, B, T, mask, depth)
    return mask, depth


def kv_compact(src, dst, L, B, S_src, S_dst, H, D, elem_bytes, src_base,
               dst_base, rows, n_rows):
    """KV compaction on byte buffers (numpy uint8).  ``dst`` is modified;
    pass ``dst is src`` for the in-place form.  Returns kv_len [B]."""
    rows = _i32(rows)
    P = rows.shape[-1] if rows.ndim == 2 else 0
    out = np.empty(B, np.int32)
    if P == 0:
        rows = np.zeros((B, 1), np.int32)
    lib().orc_kv_compact(src, dst, L, B, S_src, S_dst, H, D, elem_bytes,
                         _i32(src_base), _i32(dst_base), rows, _i32(n_rows), P, out)
    return out


def tree_attention(q, kv, base, mask, scale, sel=None):
    """Tree-masked attention of one layer in double precision.

    q [B][T][Hq][D] and kv [2][B][S][Hkv][D] (float32 arrays holding the
    bf16 values exactly), base [B], mask [B][T][W] uint64.  With ``sel``
    (an [n][3] array of (b, node, head)) only those rows are computed.
    Returns (out, lse): [B][T][Hq][D] and [B][T][Hq], or [n][D] and [n]."""
    q, kv = _f32(q), _f32(kv)
    B, T, Hq, D = q.shape
    _, B2, S, Hkv, D2 = kv.shape
    assert B2 == B and D2 == D
    mask = np.ascontiguousarray(mask, np.uint64)
    if sel is None:
        out = np.empty((B, T, Hq, D), np.float64)
        lse = np.empty((B, T, Hq), np.float64)
        sp, ns = None, 0
    else:
        sel = _i32(sel).reshape(-1, 3)
        out = np.empty((sel.shape[0], D), np.float64)
        lse = np.empty(sel.shape[0], np.float64)
        sp, ns = sel.ctypes.data, sel.shape[0]
    rc = lib().orc_tree_attention(q.reshape(-1), kv.reshape(-1), _i32(base), mask.reshape(-1),
                                  B, T, Hq, Hkv, D, S, float(scale), sp, ns,
                                  out.reshape(-1), lse.reshape(-1))
    assert rc == 0, rc
    return out, lse


def expected_tokens(alpha, N):
    return lib().orc_expected_tokens(alpha, N)


def speedup(alpha, N, c):
    return lib().orc_speedup(alpha, N, c)
