"""Pins for the oracle's tree walk, ancestor mask, KV compaction and the
speedup model."""
import itertools
import math

import numpy as np
import pytest

import oracle

# [2,2,2] tree of the lesson's exercise 3: 1 + 2 + 4 + 8 = 15 nodes, BFS order
PARENT_222 = np.array([-1, 0, 0, 1, 1, 2, 2, 3, 3, 4, 4, 5, 5, 6, 6], np.int32)


def _brute_mask(parent):
    T = len(parent)
    m = np.zeros((T, T), bool)
    for n in range(T):
        if parent[n] == -2:
            continue
        for j in range(T):                      # j is visible to n iff j is on n's root chain
            k = n
            while k >= 0:
                if k == j:
                    m[n, j] = True
                k = parent[k]
    return m


def _unpack(mask, T):
    return np.array([[(int(mask[n, j // 64]) >> (j % 64)) & 1 for j in range(T)] for n in range(T)], bool)


def test_mask_222_tree():
    mask, depth = oracle.tree_mask(PARENT_222)
    m = _unpack(mask[0], 15)
    assert np.array_equal(m, _brute_mask(PARENT_222))
    assert np.array_equal(m.sum(1), depth[0] + 1)
    assert (depth[0] == 3).sum() == 8              # eight candidate paths
    # siblings never see each other
    for n in range(1, 15):
        for s in range(1, 15):
            if s != n and PARENT_222[s] == PARENT_222[n]:
                assert not m[n, s]
    # recursive form: mask(n) = mask(parent(n)) | {n}
    for n in range(1, 15):
        want = m[PARENT_222[n]].copy(); want[n] = True
        assert np.array_equal(m[n], want)


def test_mask_chain_is_lower_triangular_and_wide_trees():
    T = 70                                          # more than one 64-bit word
    parent = np.arange(-1, T - 1, dtype=np.int32)
    mask, depth = oracle.tree_mask(parent)
    assert mask.shape == (1, T, 2)
    assert np.array_equal(_unpack(mask[0], T), np.tril(np.ones((T, T), bool)))
    assert np.array_equal(depth[0], np.arange(T))
    # padded slots are empty; an invalid tree is all-empty
    p = PARENT_222.copy(); p = np.concatenate([p, [-2, -2]]).astype(np.int32)
    mask, depth = oracle.tree_mask(p)
    assert np.all(mask[0, 15:] == 0) and np.all(depth[0, 15:] == -1)
    bad = PARENT_222.copy(); bad[5] = 9
    mask, depth = oracle.tree_mask(bad)
    assert np.all(mask == 0) and np.all(depth == -1)


def _all_paths(parent):
    kids = {}
    for c in range(1, len(parent)):
        if parent[c] >= 0:
            kids.setdefault(parent[c], []).append(c)
    out = []
    def rec(n, acc):
        if n not in kids:
            out.append(acc)
            return
        for c in kids[n]:
            rec(c, acc + [c])
    rec(0, [0])
    return out


def test_best_path_is_lexicographic_max_over_root_to_leaf_paths():
    rng = np.random.default_rng(0)
    for trial in range(300):
        T = int(rng.integers(1, 18))
        parent = np.full(T, -2, np.int32); parent[0] = -1
        for c in range(1, T):
            if rng.random() < 0.85:
                parent[c] = rng.integers(0, c)
                while parent[parent[c]] == -2:
                    parent[c] = rng.integers(0, c)
        score = rng.integers(0, 4, T).astype(np.float32) / 4     # many ties
        paths = _all_paths(parent)
        key = lambda pth: [(score[n], -n) for n in pth[1:]]
        best = max(paths, key=key)
        got = oracle.tree_best_path(parent, score, 64)
        assert got.tolist() == best, (parent, score, got, best)
        # the depth cap truncates the same walk
        assert oracle.tree_best_path(parent, score, 1).tolist() == best[:2]


def test_single_path_tree_equals_chain_bit_exactly():
    rng = np.random.default_rng(1)
    B, N, V = 6, 5, 300
    vq = (rng.standard_normal((B, N + 1, V)) * 2).astype(np.float32)
    dp = (vq[:, :N] + rng.standard_normal((B, N, V)) * 0.3).astype(np.float32)
    toks = rng.integers(0, V, (B, N)).astype(np.int32)
    ch = oracle.verify_chain(vq, dp, toks, T=0.8, seed=7, step=3)
    parent = np.tile(np.arange(-1, N, dtype=np.int32), (B, 1))
    token = np.concatenate([np.zeros((B, 1), np.int32), toks], 1)
    score = np.ones((B, N + 1), np.float32)
    dtree = np.concatenate([dp, np.zeros((B, 1, V), np.float32)], 1)
    tr = oracle.verify_tree(vq, dtree, parent, token, score, max_depth=N, T=0.8, seed=7, step=3)
    for k in ("tokens", "accept_len", "status"):
        assert np.array_equal(ch[k], tr[k]), k
    for k in ("q_prob", "p_prob"):
        assert np.array_equal(ch[k], tr[k]), k
    assert np.array_equal(ch["margin"], tr["margin"], equal_nan=True)
    for b in range(B):
        a = tr["accept_len"][b]
        assert tr["path"][b, :a + 1].tolist() == list(range(a + 1))


def test_222_tree_walk_invariants():
    rng = np.random.default_rng(2)
    B, T, V = 40, 15, 50
    parent = np.tile(PARENT_222, (B, 1))
    vq = (rng.standard_normal((B, T, V)) * 2).astype(np.float32)
    dp = (vq + rng.standard_normal((B, T, V)) * 0.5).astype(np.float32)
    token = rng.integers(0, V, (B, T)).astype(np.int32)
    score = rng.random((B, T)).astype(np.float32)
    r = oracle.verify_tree(vq, dp, parent, token, score, max_depth=3, seed=1, step=9)
    for b in range(B):
        best = oracle.tree_best_path(PARENT_222, score[b], 3)
        a = r["accept_len"][b]
        assert len(best) == 4 and 0 <= a <= 3
        assert r["path"][b, :a + 1].tolist() == best[:a + 1].tolist()
        assert r["tokens"][b, :a].tolist() == token[b, best[1:a + 1]].tolist()
        assert r["tokens"][b, a] >= 0 and np.all(r["tokens"][b, a + 1:] == -1)


def test_invalid_tree_is_flagged():
    bad = PARENT_222.copy(); bad[3] = 7
    B, T, V = 1, 15, 8
    z = np.zeros((B, T, V), np.float32)
    r = oracle.verify_tree(z, z, bad[None], np.zeros((B, T), np.int32),
                           np.ones((B, T), np.float32), max_depth=3)
    assert r["status"][0] == oracle.ROW_BAD_TREE and r["accept_len"][0] == 0
    assert r["path"][0].tolist() == [0, -1, -1, -1]


# ---------------------------------------------------------------- KV
def _kv_numpy(src, dst, src_base, dst_base, rows, n_rows):
    out = dst.copy()
    for b in range(src.shape[2]):
        n = n_rows[b]
        idx = src_base[b] + rows[b, :n]
        out[:, :, b, dst_base[b]:dst_base[b] + n] = src[:, :, b, idx]   # fancy index copies first
    return out


def test_kv_compact_gather_matches_numpy():
    rng = np.random.default_rng(3)
    L, B, S, H, D = 3, 4, 40, 2, 8
    kv = rng.integers(0, 256, (L, 2, B, S, H, D * 2), dtype=np.uint8)    # bf16 = 2 bytes
    base = np.array([5, 0, 12, 20], np.int32)
    rows = np.array([[0, 2, 5, 9, 10], [0, 1, 2, 3, 4], [0, 3, 4, 8, 0], [0, 6, 7, 0, 0]], np.int32)
    n = np.array([5, 5, 4, 3], np.int32)
    want = _kv_numpy(kv, kv, base, base, rows, n)
    work = kv.copy()
    kl = oracle.kv_compact(work, work, L, B, S, S, H, D, 2, base, base, rows, n)
    assert np.array_equal(kl, base + n)
    assert np.array_equal(work, want)
    # prefix rows are untouched
    for b in range(B):
        assert np.array_equal(work[:, :, b, :base[b]], kv[:, :, b, :base[b]])


def test_kv_compact_has_no_row_limit():
    # [Lesson] "Reversão de KV cache" / Passo 4 bound nothing but the buffer:
    # a request for more rows than any kernel limit is still copied
    rng = np.random.default_rng(8)
    L, B, S, H, D, n = 1, 2, 5000, 1, 4, 4999
    src = rng.integers(0, 256, (L, 2, B, S, H, D * 2), dtype=np.uint8)
    dst = rng.integers(0, 256, (L, 2, B, S, H, D * 2), dtype=np.uint8)
    rows = np.stack([np.sort(rng.choice(S, n, replace=False)).astype(np.int32) for _ in range(B)])
    nn = np.array([n, 4097], np.int32)
    z = np.zeros(B, np.int32)
    want = _kv_numpy(src, dst, z, z, rows, nn)
    kl = oracle.kv_compact(src, dst, L, B, S, S, H, D, 2, z, z, rows, nn)
    assert kl.tolist() == [n, 4097]
    assert np.array_equal(dst, want)


def test_kv_exercise4_two_sequences_rollback_and_commit():
    # sequence A accepts every draft, sequence B rejects at position 2
    L, B, S, H, D, N, base = 2, 2, 64, 2, 64, 4, 32
    rng = np.random.default_rng(4)
    cache = rng.integers(0, 256, (L, 2, B, S, H, D * 2), dtype=np.uint8)
    accept = np.array([N, 1], np.int32)
    n_rows = accept + 1                                   # the round's input token + accepted drafts
    rows = np.tile(np.arange(N + 1, dtype=np.int32), (B, 1))
    bases = np.full(B, base, np.int32)
    before = cache.copy()
    kl = oracle.kv_compact(cache, cache, L, B, S, S, H, D, 2, bases, bases, rows, n_rows)
    assert kl.tolist() == [base + 1 + N, base + 1 + 1]
    assert np.array_equal(cache, before)                 # logical truncation moves nothing
    # scratch-then-commit form: rows 0..a of a scratch buffer land at base
    scratch = rng.integers(0, 256, (L, 2, B, N + 1, H, D * 2), dtype=np.uint8)
    kl = oracle.kv_compact(scratch, cache, L, B, N + 1, S, H, D, 2,
                           np.zeros(B, np.int32), bases, rows, n_rows)
    assert kl.tolist() == [base + 1 + N, base + 1 + 1]
    assert np.array_equal(cache[:, :, 0, base:base + N + 1], scratch[:, :, 0])
    assert np.array_equal(cache[:, :, 1, base:base + 2], scratch[:, :, 1, :2])
    assert np.array_equal(cache[:, :, 1, base + 2:], before[:, :, 1, base + 2:])


def test_kv_invalid_requests_move_nothing():
    L, B, S, H, D = 1, 3, 16, 1, 8
    kv = np.arange(L * 2 * B * S * H * D * 2, dtype=np.int64).astype(np.uint8).reshape(L, 2, B, S, H, D * 2)
    base = np.array([2, 2, 2], np.int32)
    rows = np.array([[0, 3, 2], [0, 20, 0], [1, 0, 0]], np.int32)   # decreasing / out of range / r<k
    n = np.array([3, 2, 2], np.int32)
    before = kv.copy()
    kl = oracle.kv_compact(kv, kv, L, B, S, S, H, D, 2, base, base, rows, n)
    assert kl.tolist() == [-1, -1, -1]
    assert np.array_equal(kv, before)


# ---------------------------------------------------------------- speedup
def test_expected_tokens_closed_forms():
    for a in (0.0, 0.3, 0.6, 0.8, 0.9, 0.95):
        for N in range(0, 12):
            assert abs(oracle.expected_tokens(a, N) - sum(a ** k for k in range(N + 1))) < 1e-12
    assert oracle.expected_tokens(1.0, 7) == 8.0
    assert abs(oracle.expected_tokens(0.6, 5) - 2.38336) < 1e-12
    assert abs(oracle.expected_tokens(0.9, 5) - 4.68559) < 1e-12
    assert abs(oracle.speedup(0.8, 8, 0.05) - (1 - 0.8 ** 9) / 0.2 / 1.4) < 1e-12
