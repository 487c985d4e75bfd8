"""Python binding for libsv.so, the sm_103a verify-and-accept library.

Argument marshalling only: every step runs in the CUDA kernels behind the C
ABI declared in ``include/sv.h``.  The ``sv_*`` functions keep the C names and
take torch tensors (device memory, or page-locked host memory that the kernels
read in place) instead of raw pointers; the lower-case
helpers (``verify_chain`` ...) allocate the outputs and the workspace.  There
is no CPU fallback: if the shared library is missing, loading fails loudly.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsv.so")

SV_OK, SV_ERR_INVALID_ARG, SV_ERR_UNSUPPORTED, SV_ERR_CUDA, SV_ERR_TIMEOUT = 0, 1, 2, 3, 4
SV_F32, SV_BF16 = 0, 1
SV_ROW_NAN, SV_ROW_BAD_TOKEN, SV_ROW_RESID_ZERO, SV_ROW_P_ZERO, SV_ROW_BAD_TREE = 1, 2, 4, 8, 16
SV_ROW_BAD_BASE, SV_ROW_TIMEOUT = 32, 64
SV_MAX_VOCAB, SV_MAX_POSITIONS, SV_MAX_TREE_NODES = 1 << 22, 1024, 1024

EXPORTS = ("sv_verify_chain_workspace", "sv_verify_chain_workspace_host", "sv_verify_chain",
           "sv_verify_chain_early_exit",
           "sv_verify_chain_noalloc", "sv_verify_tree_workspace_host",
           "sv_verify_chain_noalloc_max_bytes", "sv_verify_tree_workspace",
           "sv_verify_tree", "sv_tree_build_mask", "sv_kv_compact", "sv_tree_attention", "sv_tree_attention_ex", "sv_last_error",
           "sv_launch_count", "sv_trace_enable", "sv_trace_collect", "sv_tree_expand",
           "sv_tree_select", "sv_tree_finalize", "sv_tree_level")


class SvError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"sv status {status}: {msg}")
        self.status = status


class TraceEntry(C.Structure):
    _fields_ = [("name", C.c_char * 40), ("launches", C.c_int64), ("total_ms", C.c_double)]


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libsv.so (no GPU needed) and declare every exported symbol."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with __graft_entry__.build() "
                          "(nvcc, sm_103a); there is no CPU fallback")
    L = C.CDLL(path)
    vp, i32, u64, f32, sz = C.c_void_p, C.c_int, C.c_uint64, C.c_float, C.c_size_t
    L.sv_verify_chain_workspace.argtypes = [i32, i32, i32]
    L.sv_verify_chain_workspace.restype = sz
    L.sv_verify_chain.argtypes = [vp, vp, i32, vp, i32, i32, i32, f32, u64, u64,
                                  vp, vp, vp, vp, vp, vp, vp, sz, vp, vp]
    L.sv_verify_chain.restype = i32
    L.sv_verify_chain_early_exit.argtypes = L.sv_verify_chain.argtypes
    L.sv_verify_chain_early_exit.restype = i32
    L.sv_verify_chain_noalloc_max_bytes.argtypes = []
    L.sv_verify_chain_noalloc_max_bytes.restype = sz
    L.sv_verify_chain_noalloc.argtypes = [vp, vp, i32, vp, i32, i32, i32, f32, u64, u64,
                                          vp, vp, vp, vp, vp, vp, vp, vp]
    L.sv_verify_chain_noalloc.restype = i32
    L.sv_verify_tree_workspace.argtypes = [i32, i32, i32, i32]
    L.sv_verify_tree_workspace.restype = sz
    L.sv_verify_tree_workspace_host.argtypes = [i32, i32, i32, i32, i32]
    L.sv_verify_tree_workspace_host.restype = sz
    L.sv_verify_chain_workspace_host.argtypes = [i32, i32, i32, i32]
    L.sv_verify_chain_workspace_host.restype = sz
    L.sv_verify_tree.argtypes = [vp, vp, i32, vp, vp, vp, i32, i32, i32, i32, f32, u64, u64,
                                 vp, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp]
    L.sv_verify_tree.restype = i32
    L.sv_tree_expand.argtypes = [vp, i32, i32, i32, i32, f32, vp, i32, vp, vp, vp]
    L.sv_tree_expand.restype = i32
    L.sv_tree_select.argtypes = [vp, vp, i32, i32, i32, vp, vp]
    L.sv_tree_select.restype = i32
    L.sv_tree_finalize.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp]
    L.sv_tree_finalize.restype = i32
    L.sv_tree_level.argtypes = [vp, i32, i32, i32, i32, f32, i32, i32, i32, i32, vp, vp, vp, vp,
                                vp, vp]
    L.sv_tree_level.restype = i32
    L.sv_tree_build_mask.argtypes = [vp, i32, i32, vp, vp, vp]
    L.sv_tree_build_mask.restype = i32
    L.sv_kv_compact.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp,
                                i32, i32, vp, vp]
    L.sv_kv_compact.restype = i32
    L.sv_tree_attention.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, vp, vp,
                                    vp, vp]
    L.sv_tree_attention.restype = i32
    L.sv_tree_attention_ex.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, vp, vp,
                                       vp, u64, vp]
    L.sv_tree_attention_ex.restype = i32
    L.sv_last_error.argtypes = []
    L.sv_last_error.restype = C.c_char_p
    L.sv_launch_count.argtypes = []
    L.sv_launch_count.restype = C.c_uint64
    L.sv_trace_enable.argtypes = [i32]
    L.sv_trace_enable.restype = i32
    L.sv_trace_collect.argtypes = [C.POINTER(TraceEntry), i32]
    L.sv_trace_collect.restype = i32
    _lib = L
    return L


def _p(t):
    if t is None:
        return None
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError("sv: tensors must be in device memory or page-locked host memory")
    return C.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def _event(ev):
    """A torch.cuda.Event (or None) as a cudaEvent_t.  torch creates the
    underlying event on its first record, so an unused one is recorded once."""
    if ev is None:
        return None
    if not ev.cuda_event:
        ev.record()
    return C.c_void_p(ev.cuda_event)


def _check(st):
    if st != SV_OK:
        raise SvError(st, load_library().sv_last_error().decode())
    return st


def _dtype(t):
    if t.dtype == torch.float32:
        return SV_F32
    if t.dtype == torch.bfloat16:
        return SV_BF16
    raise ValueError(f"unsupported logit dtype {t.dtype}")


# ------------------------------------------------------------------ C names
def sv_verify_chain_workspace(B, N, V):
    return int(load_library().sv_verify_chain_workspace(B, N, V))


def sv_verify_chain_workspace_host(B, N, V, dtype):
    """Workspace bytes with room for a device copy of the rows read (for
    logits in page-locked host memory); dtype: a torch dtype."""
    return int(load_library().sv_verify_chain_workspace_host(
        B, N, V, SV_BF16 if dtype == torch.bfloat16 else SV_F32))


def sv_verify_chain(vlogits, dlogits, draft_tokens, temperature, seed, step, out_tokens,
                    out_accept_len, out_q_prob, out_p_prob, out_margin, out_status, workspace,
                    stream=None, accept_event=None):
    B, R, V = vlogits.shape
    N = R - 1
    return _check(load_library().sv_verify_chain(
        _p(vlogits), _p(dlogits) if N > 0 else None, _dtype(vlogits),
        _p(draft_tokens) if N > 0 else None, B, N, V, float(temperature), int(seed), int(step),
        _p(out_tokens), _p(out_accept_len), _p(out_q_prob), _p(out_p_prob), _p(out_margin),
        _p(out_status), _p(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream), _event(accept_event)))


def sv_verify_chain_early_exit(vlogits, dlogits, draft_tokens, temperature, seed, step,
                               out_tokens, out_accept_len, out_q_prob, out_p_prob, out_margin,
                               out_status, workspace, stream=None, accept_event=None):
    B, R, V = vlogits.shape
    N = R - 1
    return _check(load_library().sv_verify_chain_early_exit(
        _p(vlogits), _p(dlogits) if N > 0 else None, _dtype(vlogits),
        _p(draft_tokens) if N > 0 else None, B, N, V, float(temperature), int(seed), int(step),
        _p(out_tokens), _p(out_accept_len), _p(out_q_prob), _p(out_p_prob), _p(out_margin),
        _p(out_status), _p(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream), _event(accept_event)))


def sv_verify_chain_noalloc_max_bytes():
    return int(load_library().sv_verify_chain_noalloc_max_bytes())


def sv_verify_chain_noalloc(vlogits, dlogits, draft_tokens, temperature, seed, step, out_tokens,
                            out_accept_len, out_q_prob, out_p_prob, out_margin, out_status,
                            stream=None, accept_event=None):
    """sv_verify_chain for callers that cannot allocate: scratch is the
    library's static device array (see include/sv.h)."""
    B, R, V = vlogits.shape
    N = R - 1
    return _check(load_library().sv_verify_chain_noalloc(
        _p(vlogits), _p(dlogits) if N > 0 else None, _dtype(vlogits),
        _p(draft_tokens) if N > 0 else None, B, N, V, float(temperature), int(seed), int(step),
        _p(out_tokens), _p(out_accept_len), _p(out_q_prob), _p(out_p_prob), _p(out_margin),
        _p(out_status), _stream(stream), _event(accept_event)))


def sv_verify_tree_workspace(B, T, max_depth, V):
    return int(load_library().sv_verify_tree_workspace(B, T, max_depth, V))


def sv_verify_tree_workspace_host(B, T, max_depth, V, dtype):
    """As sv_verify_chain_workspace_host, for trees."""
    return int(load_library().sv_verify_tree_workspace_host(
        B, T, max_depth, V, SV_BF16 if dtype == torch.bfloat16 else SV_F32))


def sv_verify_tree(vlogits, dlogits, parent, token, score, max_depth, temperature, seed, step,
                   out_path_nodes, out_tokens, out_accept_len, out_q_prob, out_p_prob,
                   out_margin, out_status, workspace, stream=None, accept_event=None):
    B, T, V = vlogits.shape
    return _check(load_library().sv_verify_tree(
        _p(vlogits), _p(dlogits), _dtype(vlogits), _p(parent), _p(token), _p(score), B, T,
        max_depth, V, float(temperature), int(seed), int(step), _p(out_path_nodes),
        _p(out_tokens), _p(out_accept_len), _p(out_q_prob), _p(out_p_prob), _p(out_margin),
        _p(out_status), _p(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream), _event(accept_event)))


def sv_tree_build_mask(parent, out_mask, out_depth, stream=None):
    B, T = parent.shape
    return _check(load_library().sv_tree_build_mask(_p(parent), B, T, _p(out_mask),
                                                    _p(out_depth), _stream(stream)))


def sv_kv_compact(src_kv, dst_kv, src_base, dst_base, rows, n_rows, n_rows_add, out_kv_len,
                  stream=None):
    """src_kv [L][2][B][S_src][H][D], dst_kv [L][2][B][S_dst][H][D] (any dtype)."""
    L, two, B, S_src, H, D = src_kv.shape
    S_dst = dst_kv.shape[3]
    P = rows.shape[1] if rows is not None else S_src
    return _check(load_library().sv_kv_compact(
        _p(src_kv), _p(dst_kv), L, B, S_src, S_dst, H, D, src_kv.element_size(),
        _p(src_base), _p(dst_base), _p(rows), _p(n_rows), int(n_rows_add), P,
        _p(out_kv_len), _stream(stream)))


def sv_tree_attention(q, kv, base, mask, scale, out, out_lse=None, out_status=None,
                      stream=None):
    """q [B][T][Hq][D] bf16, kv [2][B][S][Hkv][D] bf16 (one layer), base [B] int32,
    mask [B][T][W] (64-bit words), out like q."""
    B, T, Hq, D = q.shape
    S, Hkv = kv.shape[2], kv.shape[3]
    return _check(load_library().sv_tree_attention(
        _p(q), _p(kv), _p(base), _p(mask), B, T, Hq, Hkv, D, S, float(scale), _p(out),
        _p(out_lse), _p(out_status), _stream(stream)))


def sv_tree_attention_ex(q, kv, base, mask, scale, out, out_lse=None, out_status=None,
                         wait_ns=0, stream=None):
    """sv_tree_attention with the limit of each device wait in nanoseconds
    (0: the default 2 s)."""
    B, T, Hq, D = q.shape
    S, Hkv = kv.shape[2], kv.shape[3]
    return _check(load_library().sv_tree_attention_ex(
        _p(q), _p(kv), _p(base), _p(mask), B, T, Hq, Hkv, D, S, float(scale), _p(out),
        _p(out_lse), _p(out_status), int(wait_ns), _stream(stream)))


def sv_tree_expand(dlogits, frontier_score, K, out_token, out_score, temperature=1.0,
                   stream=None):
    """dlogits [B][F][V]; frontier_score [B][F]; out_token / out_score [B][F][K]."""
    B, F, V = dlogits.shape
    return _check(load_library().sv_tree_expand(
        _p(dlogits), _dtype(dlogits), B, F, V, float(temperature), _p(frontier_score), int(K),
        _p(out_token), _p(out_score), _stream(stream)))


def sv_tree_select(cand_score, cand_token, K, out_index, stream=None):
    B, Cn = cand_score.shape
    return _check(load_library().sv_tree_select(_p(cand_score), _p(cand_token), B, Cn, int(K),
                                                _p(out_index), _stream(stream)))


def sv_tree_finalize(cand_parent, cand_token, cand_score, cand_level, T, out_parent, out_token,
                     out_score, stream=None):
    """cand_* [B][C] with unit column stride and one common row stride (views
    of a wider candidate table are passed as they are)."""
    B, Cn = cand_parent.shape
    ld = cand_parent.stride(0) if B > 1 else Cn
    for a in (cand_parent, cand_token, cand_score, cand_level):
        if a.shape != (B, Cn) or (Cn > 1 and a.stride(1) != 1) or (B > 1 and a.stride(0) != ld):
            raise ValueError("candidate arrays need unit column stride and one row stride")
    return _check(load_library().sv_tree_finalize(
        _p(cand_parent), _p(cand_token), _p(cand_score), _p(cand_level), B, Cn, int(ld), int(T),
        _p(out_parent), _p(out_token), _p(out_score), _stream(stream)))


def sv_tree_level(dlogits, K, level, n0, frontier, cand_parent, cand_token, cand_score,
                  cand_level, temperature=1.0, stream=None):
    """One build level through the candidate table [B][ldc] (see include/sv.h)."""
    B, F, V = dlogits.shape
    return _check(load_library().sv_tree_level(
        _p(dlogits), _dtype(dlogits), B, F, V, float(temperature), int(K), int(level), int(n0),
        int(cand_parent.shape[1]), _p(frontier), _p(cand_parent), _p(cand_token),
        _p(cand_score), _p(cand_level), _stream(stream)))


def sv_last_error():
    return load_library().sv_last_error().decode()


def sv_launch_count():
    return int(load_library().sv_launch_count())


def sv_trace_enable(on=True):
    return _check(load_library().sv_trace_enable(1 if on else 0))


def sv_trace_collect(max_entries=64):
    buf = (TraceEntry * max_entries)()
    n = load_library().sv_trace_collect(buf, max_entries)
    if n < 0:
        raise SvError(SV_ERR_CUDA, sv_last_error())
    return {buf[i].name.decode(): (int(buf[i].launches), float(buf[i].total_ms)) for i in range(n)}


# ------------------------------------------------------------------ helpers
def _ws(nbytes, device):
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)


def _out_dev(t):
    """Outputs and workspace go to device memory: the input's device, or the
    current device when the input sits in page-locked host memory."""
    return t.device if t.is_cuda else torch.device("cuda", torch.cuda.current_device())


def verify_chain(vlogits, dlogits, draft_tokens, temperature=1.0, seed=0, step=0,
                 workspace=None, stream=None, probs=True, accept_event=None, early_exit=False):
    """Allocate outputs and run sv_verify_chain (sv_verify_chain_early_exit
    with ``early_exit``).  Returns a dict of tensors."""
    B, R, V = vlogits.shape
    N = R - 1
    dev = _out_dev(vlogits)
    out = dict(
        tokens=torch.empty(B, N + 1, dtype=torch.int32, device=dev),
        accept_len=torch.empty(B, dtype=torch.int32, device=dev),
        q_prob=torch.empty(B, max(N, 1), dtype=torch.float32, device=dev) if probs else None,
        p_prob=torch.empty(B, max(N, 1), dtype=torch.float32, device=dev) if probs else None,
        margin=torch.empty(B, N + 1, dtype=torch.float32, device=dev) if probs else None,
        status=torch.empty(B, dtype=torch.int32, device=dev))
    if workspace is None:
        workspace = _ws(sv_verify_chain_workspace(B, N, V) if vlogits.is_cuda
                        else sv_verify_chain_workspace_host(B, N, V, vlogits.dtype), dev)
    fn = sv_verify_chain_early_exit if early_exit else sv_verify_chain
    fn(vlogits, dlogits, draft_tokens, temperature, seed, step, out["tokens"],
       out["accept_len"], out["q_prob"], out["p_prob"], out["margin"],
       out["status"], workspace, stream, accept_event)
    return out


def verify_tree(vlogits, dlogits, parent, token, score, max_depth, temperature=1.0, seed=0,
                step=0, workspace=None, stream=None, probs=True, accept_event=None):
    B, T, V = vlogits.shape
    dev = _out_dev(vlogits)
    P = max_depth + 1
    out = dict(
        path=torch.empty(B, P, dtype=torch.int32, device=dev),
        tokens=torch.empty(B, P, dtype=torch.int32, device=dev),
        accept_len=torch.empty(B, dtype=torch.int32, device=dev),
        q_prob=torch.empty(B, max(max_depth, 1), dtype=torch.float32, device=dev) if probs else None,
        p_prob=torch.empty(B, max(max_depth, 1), dtype=torch.float32, device=dev) if probs else None,
        margin=torch.empty(B, P, dtype=torch.float32, device=dev) if probs else None,
        status=torch.empty(B, dtype=torch.int32, device=dev))
    if workspace is None:
        workspace = _ws(sv_verify_tree_workspace(B, T, max_depth, V) if vlogits.is_cuda
                        else sv_verify_tree_workspace_host(B, T, max_depth, V, vlogits.dtype), dev)
    sv_verify_tree(vlogits, dlogits, parent, token, score, max_depth, temperature, seed, step,
                   out["path"], out["tokens"], out["accept_len"], out["q_prob"], out["p_prob"],
                   out["margin"], out["status"], workspace, stream, accept_event)
    return out


def tree_expand(dlogits, frontier_score, K, temperature=1.0, stream=None):
    B, F, V = dlogits.shape
    dev = _out_dev(dlogits)
    tok = torch.empty(B, F, K, dtype=torch.int32, device=dev)
    sc = torch.empty(B, F, K, dtype=torch.float32, device=dev)
    sv_tree_expand(dlogits, frontier_score, K, tok, sc, temperature, stream)
    return tok, sc


def tree_select(cand_score, cand_token, K, stream=None):
    out = torch.empty(cand_score.shape[0], K, dtype=torch.int32, device=_out_dev(cand_score))
    sv_tree_select(cand_score, cand_token, K, out, stream)
    return out


def tree_finalize(cand_parent, cand_token, cand_score, cand_level, T, stream=None):
    B = cand_parent.shape[0]
    dev = _out_dev(cand_parent)
    parent = torch.empty(B, T, dtype=torch.int32, device=dev)
    token = torch.empty(B, T, dtype=torch.int32, device=dev)
    score = torch.empty(B, T, dtype=torch.float32, device=dev)
    sv_tree_finalize(cand_parent, cand_token, cand_score, cand_level, T, parent, token, score,
                     stream)
    return parent, token, score


TREE_TABLE_COLUMNS = 2048  # candidate table width (the finalize step's limit)


def build_tree(level_rows, K, T, temperature=1.0, stream=None, return_candidates=False):
    """EAGLE-2 dynamic tree from the draft rows of each level.  level_rows(l,
    frontier) -> [B][F][V] draft logits of the frontier's nodes (frontier:
    int32 [B][K] candidate ids, -1 for an empty entry; None at level 1, whose
    frontier is the root), or None to stop.  Every step -- each level's
    expansion and frontier selection through one candidate table, and the
    final pruning -- runs in the library's kernels; this loop allocates the
    table and tracks where the next level's candidates start.
    Returns (parent, token, score) [B][T] for sv_verify_tree (and the
    candidate table's used columns with return_candidates)."""
    frontier = None
    table = None
    n0, level = 1, 0
    while True:
        rows = level_rows(level + 1, None if level == 0 else frontier)
        if rows is None:
            break
        B, F, _ = rows.shape
        if table is None:
            dev = _out_dev(rows)
            C = TREE_TABLE_COLUMNS
            table = (torch.empty(B, C, dtype=torch.int32, device=dev),
                     torch.empty(B, C, dtype=torch.int32, device=dev),
                     torch.empty(B, C, dtype=torch.float32, device=dev),
                     torch.empty(B, C, dtype=torch.int32, device=dev))
            frontier = torch.empty(B, K, dtype=torch.int32, device=dev)
        level += 1
        sv_tree_level(rows, K, level, n0, frontier, *table, temperature=temperature,
                      stream=stream)
        n0 += F * K
    if table is None:
        raise ValueError("level_rows gave no level")
    cands = tuple(a[:, :n0] for a in table)
    tree = tree_finalize(*cands, T, stream=stream)
    return (tree, cands) if return_candidates else tree


def tree_build_mask(parent, stream=None):
    B, T = parent.shape
    W = (T + 63) // 64
    mask = torch.empty(B, T, W, dtype=torch.int64, device=_out_dev(parent))
    depth = torch.empty(B, T, dtype=torch.int32, device=_out_dev(parent))
    sv_tree_build_mask(parent, mask, depth, stream)
    return mask, depth


def tree_attention(q, kv, base, mask, scale=None, return_lse=False, stream=None, wait_ns=0):
    """Tree-masked attention of one layer: returns out (like q), and with
    return_lse the log-sum-exp [B][T][Hq] and the status words [B].
    wait_ns: limit of each device wait (0: the default 2 s)."""
    B, T, Hq, D = q.shape
    if scale is None:
        scale = D ** -0.5
    dev = _out_dev(q)
    out = torch.empty_like(q, device=dev)
    lse = torch.empty(B, T, Hq, dtype=torch.float32, device=dev) if return_lse else None
    status = torch.zeros(B, dtype=torch.int32, device=dev) if return_lse else None
    sv_tree_attention_ex(q, kv, base, mask, scale, out, lse, status, wait_ns, stream)
    return (out, lse, status) if return_lse else out


def kv_compact(src_kv, dst_kv, src_base, dst_base, rows, n_rows, n_rows_add=0, stream=None):
    B = src_kv.shape[2]
    kv_len = torch.empty(B, dtype=torch.int32, device=_out_dev(src_kv))
    sv_kv_compact(src_kv, dst_kv, src_base, dst_base, rows, n_rows, n_rows_add, kv_len, stream)
    return kv_len
