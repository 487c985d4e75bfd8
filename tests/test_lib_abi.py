"""CPU checks of the C ABI: the shared library loads, exports every entry point
that include/sv.h declares, and rejects bad arguments on the host without
touching a GPU."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_vocab_gb300 import _build
    _build.build()
    import speculative_decoding_verification_vocab_gb300 as sv
    return sv.load_library()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "sv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sv_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for name in ("sv_verify_chain", "sv_verify_tree", "sv_kv_compact", "sv_tree_build_mask",
                 "sv_verify_chain_workspace", "sv_verify_tree_workspace", "sv_last_error"):
        assert name in syms


def test_every_declared_symbol_is_exported(lib):
    import speculative_decoding_verification_vocab_gb300 as sv
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert name in sv.EXPORTS or name.endswith("_workspace") or name.startswith("sv_")


def test_binding_has_the_c_names():
    import speculative_decoding_verification_vocab_gb300 as sv
    for name in declared_symbols():
        assert callable(getattr(sv, name)), name


def test_host_argument_checks_need_no_gpu(lib):
    null = None
    # negative sizes, bad dtype, bad temperature: refused before any CUDA call
    assert lib.sv_verify_chain(null, null, 0, null, -1, 2, 10, 1.0, 0, 0, null, null, null, null,
                               null, null, null, 0, null, null) == 1
    assert lib.sv_verify_chain(null, null, 7, null, 1, 2, 10, 1.0, 0, 0, null, null, null, null,
                               null, null, null, 0, null, null) == 1
    assert lib.sv_verify_chain(null, null, 0, null, 1, 2, 10, -0.5, 0, 0, null, null, null, null,
                               null, null, null, 0, null, null) == 1
    assert b"temperature" in lib.sv_last_error()
    assert lib.sv_verify_chain(null, null, 0, null, 1, 2, (1 << 22) + 1, 1.0, 0, 0, null, null,
                               null, null, null, null, null, 0, null, null) == 2
    # B == 0 is a no-op
    assert lib.sv_verify_chain(null, null, 0, null, 0, 2, 10, 1.0, 0, 0, null, null, null, null,
                               null, null, null, 0, null, null) == 0
    assert lib.sv_verify_tree(null, null, 1, null, null, null, 1, 20, 3, 10, 1.0, 0, 0, null,
                              null, null, null, null, null, null, null, 0, null, null) == 1
    assert lib.sv_tree_build_mask(null, 1, 2000, null, null, null) == 2
    assert lib.sv_tree_build_mask(null, 1, 0, null, null, null) == 1
    assert lib.sv_kv_compact(null, null, 0, 1, 4, 4, 1, 1, 2, null, null, null, null, 0, 1,
                             null, null) == 1
    assert lib.sv_launch_count() >= 0


def test_workspace_queries(lib):
    assert lib.sv_verify_chain_workspace(4, 3, 1000) > 0
    assert lib.sv_verify_tree_workspace(4, 25, 5, 1000) > lib.sv_verify_chain_workspace(4, 0, 1000)
    assert lib.sv_verify_chain_workspace(-1, 3, 1000) == 0


def test_tree_attention_host_checks_need_no_gpu(lib):
    """sv_tree_attention refuses bad shapes and scales before any CUDA call."""
    f = lib.sv_tree_attention
    null = None
    # (q, kv, base, mask, B, T, Hq, Hkv, D, S, scale, out, lse, status, stream)
    assert f(null, null, null, null, 1, 4, 8, 2, 64, 16, 1.0, null, null, null, null) == 2
    assert b"head dimension" in lib.sv_last_error()
    assert f(null, null, null, null, 1, 4, 9, 3, 128, 16, 1.0, null, null, null, null) == 2
    assert f(null, null, null, null, 1, 4, 8, 3, 128, 16, 1.0, null, null, null, null) == 1
    assert f(null, null, null, null, 1, 4, 8, 2, 128, 16, 0.0, null, null, null, null) == 1
    assert f(null, null, null, null, 1, 4, 8, 2, 128, 16, float("nan"), null, null, null,
             null) == 1
    assert f(null, null, null, null, 1, 0, 8, 2, 128, 16, 1.0, null, null, null, null) == 1
    assert f(null, null, null, null, 1, 2000, 8, 2, 128, 4096, 1.0, null, null, null,
             null) == 2
    # B == 0 is a no-op; null pointers with B > 0 are refused
    assert f(null, null, null, null, 0, 4, 8, 2, 128, 16, 1.0, null, null, null, null) == 0
    assert f(null, null, null, null, 1, 4, 8, 2, 128, 16, 1.0, null, null, null, null) == 1
    assert b"null" in lib.sv_last_error()


def test_tree_level_host_checks_need_no_gpu(lib):
    """sv_tree_level refuses inconsistent levels and full tables before any
    CUDA call."""
    f = lib.sv_tree_level
    null = None
    # (dlogits, dt, B, F, V, T, K, level, n0, ldc, frontier, parent, token, score, level, stream)
    def call(B=1, F=1, V=100, T=1.0, K=10, level=1, n0=1, ldc=2048):
        return f(null, 1, B, F, V, T, K, level, n0, ldc, null, null, null, null, null, null)
    assert call(F=2) == 1 and b"root" in lib.sv_last_error()       # level 1 expands the root
    assert call(n0=3) == 1
    assert call(level=2, F=11, n0=11) == 1                         # F > K
    assert call(level=2, F=10, n0=1) == 1                          # n0 < 2 after level 1
    assert call(level=2, F=10, n0=2000, ldc=2048) == 1             # table full
    assert b"full" in lib.sv_last_error()
    assert call(ldc=4096) == 2                                     # wider than finalize takes
    assert call(K=17) == 2 and call(K=0) == 1 and call(T=-1.0) == 1
    assert call(level=0) == 1
    assert call(B=0) == 0                                          # no-op
    assert call() == 1 and b"null" in lib.sv_last_error()
    # finalize: the row stride must cover the columns used
    g = lib.sv_tree_finalize
    assert g(null, null, null, null, 1, 10, 9, 5, null, null, null, null) == 1
    assert b"ldc" in lib.sv_last_error()


def test_noalloc_capacity_and_argument_order(lib):
    """The allocation-free chain verify: the shape its documentation quotes
    (the large-vocabulary chain, B=256, N=7, V=128256) fits the static
    scratch, and bad arguments get sv_verify_chain's statuses before the
    capacity check (host-side only, no GPU)."""
    cap = lib.sv_verify_chain_noalloc_max_bytes()
    assert cap == 16 << 20
    assert lib.sv_verify_chain_workspace(256, 7, 128256) <= cap
    # the limit the documentation states: up to B = 447 at N = 7, V = 128256
    assert lib.sv_verify_chain_workspace(447, 7, 128256) <= cap
    assert lib.sv_verify_chain_workspace(448, 7, 128256) > cap
    null = None
    args = lambda B, N, V, dt=1, T=1.0: (null, null, dt, null, B, N, V, T, 0, 0, null, null, null,
                                         null, null, null, null, null)
    # an oversize request with a bad dtype / temperature / null outputs: the
    # argument error wins, exactly as sv_verify_chain reports it
    assert lib.sv_verify_chain_noalloc(*args(1 << 20, 7, 128256, dt=7)) == 1
    assert lib.sv_verify_chain_noalloc(*args(1 << 20, 7, 128256, T=-1.0)) == 1
    assert lib.sv_verify_chain_noalloc(*args(1 << 20, 7, 128256)) == 1      # null pointers
    assert b"null" in lib.sv_last_error()
    assert lib.sv_verify_chain_noalloc(*args(-1, 7, 128256)) == 1
    assert lib.sv_verify_chain_noalloc(*args(0, 7, 128256)) == 0            # B = 0: no-op
    assert lib.sv_verify_chain_noalloc(*args(4, 7, (1 << 22) + 1)) == 2     # V above the maximum
