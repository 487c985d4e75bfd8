"""Pins of the oracle's dynamic-tree builder (EAGLE-2 expansion, frontier
selection, pruning to the node budget) against numpy / scipy restatements
and the properties the builder must have."""
import numpy as np
import pytest

import oracle


@pytest.fixture(scope="module", autouse=True)
def _build():
    oracle.build()


def _bf16(rng, shape, sigma=3.0):
    x = (rng.standard_normal(shape) * sigma).astype(np.float32)
    return (x.view(np.uint32) & 0xFFFF0000).view(np.float32)


def _softmax(x, T):
    z = x.astype(np.float64) / T
    z -= z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def test_expand_top_k_and_scores():
    rng = np.random.default_rng(1)
    R, V, K = 40, 97, 7
    x = _bf16(rng, (R, V), sigma=1.0)  # bf16 values: many equal logits
    fs = rng.uniform(0.01, 1.0, R).astype(np.float32)
    tok, sc = oracle.tree_expand(x, fs, K, T=0.8)
    p = _softmax(x, 0.8)
    for r in range(R):
        order = np.lexsort((np.arange(V), -x[r]))  # logit desc, then id asc
        assert list(tok[r]) == list(order[:K])
        assert np.allclose(sc[r], fs[r].astype(np.float64) * p[r, order[:K]], rtol=1e-12)


def test_expand_greedy_and_faults():
    x = np.zeros((3, 5), np.float32)
    x[0] = [1, 3, 3, 2, 0]
    x[1, 2] = np.nan
    x[2] = -np.inf
    tok, sc = oracle.tree_expand(x, np.float32([0.5, 1, 1]), 3, T=0.0)
    assert list(tok[0]) == [1, 2, 3] and list(sc[0]) == [0.5, 0.0, 0.0]
    assert list(tok[1]) == [-1, -1, -1] and np.all(np.isneginf(sc[1]))
    assert list(tok[2]) == [-1, -1, -1]


def test_select_best_k():
    rng = np.random.default_rng(2)
    B, C, K = 16, 60, 10
    s = rng.choice(np.float32([0.1, 0.2, 0.3, 0.5]), (B, C))  # many equal scores
    t = rng.integers(-1, 50, (B, C)).astype(np.int32)
    sel = oracle.tree_select(s, t, K)
    for b in range(B):
        ok = np.nonzero(t[b] >= 0)[0]
        order = ok[np.lexsort((ok, -s[b, ok]))]
        want = list(order[:K]) + [-1] * max(0, K - len(order))
        assert list(sel[b]) == want


def _build_tree(rng, B, V, K, depth, Tn, T=1.0):
    """A full dynamic build with the oracle: rows drawn per level, as the
    draft model would produce them.  Returns the candidate lists, the rows
    of every candidate that was expanded, and the finalized tree."""
    cp = [np.full((B, 1), -1, np.int32)]
    ct = [np.zeros((B, 1), np.int32)]
    cs = [np.ones((B, 1), np.float32)]
    cl = [np.zeros((B, 1), np.int32)]
    rows = {}  # (b, candidate) -> logits row
    frontier = np.zeros((B, 1), np.int64)
    n = 1
    for lvl in range(1, depth + 1):
        F = frontier.shape[1]
        x = _bf16(rng, (B, F, V))
        for b in range(B):
            for f in range(F):
                rows[(b, int(frontier[b, f]))] = x[b, f]
        fs = np.take_along_axis(np.concatenate(cs, 1), frontier, 1)
        tok, sc = oracle.tree_expand(x, fs, K, T)
        cp.append(np.repeat(frontier, K, axis=1).astype(np.int32))
        ct.append(tok.reshape(B, F * K))
        cs.append(sc.reshape(B, F * K).astype(np.float32))
        cl.append(np.full((B, F * K), lvl, np.int32))
        ids = np.arange(n, n + F * K)
        n += F * K
        if lvl < depth:
            sel = oracle.tree_select(cs[-1], ct[-1], K)
            frontier = ids[sel]
    C = [np.concatenate(a, 1) for a in (cp, ct, cs, cl)]
    return C, rows, oracle.tree_finalize(*C, Tn)


def test_finalize_keeps_the_best_and_numbers_by_level():
    rng = np.random.default_rng(3)
    B, V, K, depth, Tn = 6, 31, 4, 4, 20
    (cp, ct, cs, cl), rows, (parent, token, score) = _build_tree(rng, B, V, K, depth, Tn)
    for b in range(B):
        Cn = cp.shape[1]
        valid = [c for c in range(Cn) if c == 0 or ct[b, c] >= 0]
        keep = sorted(valid, key=lambda c: (-cs[b, c], cl[b, c], c))[:Tn]
        slots = sorted(keep, key=lambda c: (cl[b, c], -cs[b, c], c))
        assert list(token[b]) == [int(ct[b, c]) for c in slots]
        assert np.array_equal(score[b], cs[b, slots])
        slot_of = {c: i for i, c in enumerate(slots)}
        assert parent[b, 0] == -1
        for i, c in enumerate(slots[1:], 1):
            assert parent[b, i] == slot_of[int(cp[b, c])]  # ancestor-closed
            assert parent[b, i] < i
        assert oracle.tree_valid(parent[b], score[b])


def test_built_scores_are_path_products():
    """Every kept node's score is the product of the draft probabilities of
    the tokens along its path (scipy-free restatement in float64)."""
    rng = np.random.default_rng(4)
    B, V, K, depth, Tn, T = 4, 23, 3, 3, 12, 0.7
    (cp, ct, cs, cl), rows, (parent, token, score) = _build_tree(rng, B, V, K, depth, Tn, T)
    for b in range(B):
        # candidate id of every slot, to find the rows expanded at each node
        Cn = cp.shape[1]
        valid = [c for c in range(Cn) if c == 0 or ct[b, c] >= 0]
        keep = sorted(valid, key=lambda c: (-cs[b, c], cl[b, c], c))[:Tn]
        slots = sorted(keep, key=lambda c: (cl[b, c], -cs[b, c], c))
        for i, c in enumerate(slots[1:], 1):
            prod, node = 1.0, c
            while cp[b, node] >= 0:
                par = int(cp[b, node])
                prod *= _softmax(rows[(b, par)], T)[ct[b, node]]
                node = par
            assert np.isclose(score[b, i], prod, rtol=1e-6)


@pytest.mark.parametrize("seed", [5, 6, 7])
def test_kept_tree_has_the_largest_total_score(seed):
    """Brute force on tiny builds: over every ancestor-closed set of T nodes
    holding the root, none has a larger total path score than the tree the
    builder keeps.  Scores never grow along a path (each factor is a
    probability), which is why keeping the T best candidates is optimal."""
    import itertools
    rng = np.random.default_rng(seed)
    B, V, K, depth, Tn = 3, 6, 2, 3, 5
    (cp, ct, cs, cl), rows, (parent, token, score) = _build_tree(rng, B, V, K, depth, Tn)
    for b in range(B):
        valid = [c for c in range(1, cp.shape[1]) if ct[b, c] >= 0]
        best = -1.0
        for sub in itertools.combinations(valid, Tn - 1):
            s = set(sub) | {0}
            if all(int(cp[b, c]) in s for c in sub):
                best = max(best, sum(float(cs[b, c]) for c in s))
        got = sum(float(v) for v in score[b])
        assert np.isclose(got, best, rtol=1e-12, atol=0), (b, got, best)
        # a plausible wrong rule, keeping breadth-first (level, then score),
        # is ancestor-closed too but falls short: the pin tells them apart
        bfs = sorted([0] + valid, key=lambda c: (cl[b, c], -cs[b, c], c))[:Tn]
        assert sum(float(cs[b, c]) for c in bfs) < best - 1e-9
        # and the kept nodes form a tree with parents before children
        assert parent[b, 0] == -1 and all(0 <= parent[b, i] < i for i in range(1, Tn))
