"""The numbers the pages print (stored with their citations in
tests/golden/pages_numbers.txt) against the oracle's speedup model, tree mask
and chain walk.

The model is the lesson's: E[tokens per verifier pass] = (1 - a^(N+1)) /
(1 - a) and wall time per token (N c + 1) / E, so speedup = E / (N c + 1).
Where a printed number and the formula disagree beyond the page's rounding,
the test records the disagreement instead of bending the formula: the lesson's
own numbers are looser than its equation in places.
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "pages_numbers.txt")


def _load():
    vals = {}
    with open(GOLDEN, encoding="utf-8") as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, rhs = (s.strip() for s in line.split("=", 1))
            vals[key] = [float(t) for t in rhs.split()]
    return vals


P = _load()


def _one(key):
    (v,) = P[key]
    return v


def _best(a, c, Nmax=60):
    s = [oracle.speedup(a, N, c) for N in range(1, Nmax + 1)]
    return int(np.argmax(s)) + 1, max(s), s


def test_fixture_is_complete():
    for k in ("regime1.alpha", "regime1.c", "regime1.N", "regime1.speedup", "regime2.alpha",
              "regime2.c", "regime2.N", "regime2.speedup", "lever.N", "lever.alpha",
              "lever.tokens", "step6.alpha", "step6.tokens", "ex2.alpha", "ex2.c", "ex2.N",
              "ex3.shape", "ex3.paths", "breakeven.alpha", "breakeven.c", "example.drafts",
              "example.accepted", "example.tokens"):
        assert k in P, k


def test_regime1_agrees_within_the_pages_rounding():
    a, c = _one("regime1.alpha"), _one("regime1.c")
    lo, hi = (int(v) for v in P["regime1.N"])
    N_opt, s_opt, s = _best(a, c)
    assert N_opt == 8 and abs(s_opt - 3.09208) < 1e-4
    # every N the page names is within 5% of the optimum, and 3.2x within 4%
    assert all(s[N - 1] >= 0.95 * s_opt for N in range(lo, hi + 1))
    assert abs(_one("regime1.speedup") - s_opt) / s_opt < 0.04


def test_regime2_is_not_reproduced_by_the_formula():
    a, c = _one("regime2.alpha"), _one("regime2.c")
    lo, hi = (int(v) for v in P["regime2.N"])
    N_opt, s_opt, s = _best(a, c)
    assert N_opt == 31 and abs(s_opt - 9.95) < 0.01
    # at the page's N range the formula gives 6.4-7.2x, not about 5x
    assert all(s[N - 1] > _one("regime2.speedup") + 1.3 for N in range(lo, hi + 1))


def test_alpha_lever_is_not_reproduced_by_the_formula():
    N = int(_one("lever.N"))
    (a0, a1), (t0, t1) = P["lever.alpha"], P["lever.tokens"]
    e0, e1 = oracle.expected_tokens(a0, N), oracle.expected_tokens(a1, N)
    assert abs(e0 - 2.38336) < 1e-12 and abs(e1 - 4.68559) < 1e-12
    assert abs(e0 - t0) > 0.15 and abs(e1 - t1) > 0.5
    # the page's conclusion (about 2x the throughput from the same verifier) holds
    assert 1.9 < e1 / e0 < 2.0


def test_step6_tokens_per_call_at_eagle3_quality():
    a = _one("step6.alpha")
    lo, hi = P["step6.tokens"]
    inside = [N for N in range(1, 21) if lo <= oracle.expected_tokens(a, N) <= hi]
    assert inside == [4, 5]
    # the supremum over all N is 1 / (1 - a) = 10: 4-5 tokens is a choice of N, not a limit
    assert abs(oracle.expected_tokens(a, 400) - 1 / (1 - a)) < 1e-9


def test_exercise2_time_per_token_keeps_falling_to_n10():
    a, c = _one("ex2.alpha"), _one("ex2.c")
    lo, hi = (int(v) for v in P["ex2.N"])
    t = [(N * c + 1) / oracle.expected_tokens(a, N) for N in range(lo, hi + 1)]
    assert int(np.argmin(t)) + lo == hi
    assert all(t[i + 1] < t[i] for i in range(len(t) - 1))
    # beyond the sweep the curve turns: the minimum over all N is at N = 15
    t2 = [(N * c + 1) / oracle.expected_tokens(a, N) for N in range(1, 60)]
    assert int(np.argmin(t2)) + 1 == 15


def test_exercise3_tree_shape():
    shape = [int(v) for v in P["ex3.shape"]]
    parent, level = [-1], [0]
    frontier = [0]
    for width in shape:
        nxt = []
        for f in frontier:
            for _ in range(width):
                parent.append(f)
                level.append(level[f] + 1)
                nxt.append(len(parent) - 1)
        frontier = nxt
    parent = np.array(parent, np.int32)
    mask, depth = oracle.tree_mask(parent)
    mask, depth = mask[0], depth[0]
    leaves = [n for n in range(len(parent)) if n not in set(parent.tolist())]
    assert len(leaves) == int(_one("ex3.paths"))
    assert depth.tolist() == level
    bits = np.unpackbits(mask.view(np.uint8), axis=-1, bitorder="little").reshape(len(parent), -1)
    for n in leaves:
        assert bits[n].sum() == len(shape) + 1          # a leaf sees its whole path


@pytest.mark.parametrize("a", P["breakeven.alpha"])
def test_speculation_pays_iff_alpha_exceeds_c(a):
    """Blog section 2: some draft length N >= 1 beats plain decoding (N = 0,
    speedup 1) exactly when alpha > c.  N = 1 gives (1 + a) / (1 + c); for
    a <= c every N has E <= 1 + N a <= 1 + N c."""
    for c in P["breakeven.c"]:
        gain = max(oracle.speedup(a, N, c) for N in range(1, 40))
        assert oracle.speedup(a, 0, c) == 1.0
        if a > c:
            assert gain > 1.0 and oracle.speedup(a, 1, c) > 1.0, (a, c)
        else:
            assert gain <= 1.0 + 1e-12, (a, c)


def test_worked_example_counts():
    """Blog section 2: four drafts, the first two accepted, the third rejected
    and replaced from the residual: three tokens from one verifier pass."""
    n, acc, tok = (int(_one(k)) for k in ("example.drafts", "example.accepted", "example.tokens"))
    V = 8
    xq = np.zeros((1, n + 1, V), np.float32)
    xp = np.zeros((1, n, V), np.float32)
    d = np.array([[3, 1, 6, 2]], np.int32)[:, :n]
    xq[0, acc, :] = -np.inf
    xq[0, acc, 5] = 0.0                 # the verifier puts no mass on draft acc
    for seed in range(10):
        r = oracle.verify_chain(xq, xp, d, seed=seed, step=seed)
        assert r["accept_len"][0] == acc
        assert int((r["tokens"][0] >= 0).sum()) == tok
