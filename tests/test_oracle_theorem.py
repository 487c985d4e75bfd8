"""Pins for the oracle's verify walk against what the pages fix:

* the Leviathan theorem (the emitted token's law is exactly q, whatever p is)
  by enumeration on a vocabulary of 4 with the uniforms on dense grids;
* E[tokens per verifier pass] = (1 - a^(N+1)) / (1 - a) on constructed pairs
  with sum_v min(p_v, q_v) = a exactly, over 10^6 rounds, within 3 sigma;
* the lesson's Step 5: a chi-square of 50,000 speculative steps against
  50,000 direct samples of q, below the 95% critical value;
* the worked example "2 accepted + 1 correction = 3 tokens from one pass".
"""
import math

import numpy as np
import pytest
from scipy.stats import chi2

import oracle


def _grid(G):
    return ((np.arange(G) + 0.5) / G * 2**24).astype(np.uint32)


def test_enumeration_single_position_law_is_q():
    V, G = 4, 512
    xq = np.log(np.array([[0.55, 0.25, 0.15, 0.05], [0.1, 0.2, 0.3, 0.4]])).astype(np.float32)
    xp = np.log(np.array([[0.10, 0.20, 0.30, 0.40]])).astype(np.float32)
    q1, q2, p1 = oracle.softmax(xq[0]), oracle.softmax(xq[1]), oracle.softmax(xp[0])
    d, ga, gs = np.meshgrid(np.arange(V), _grid(G), _grid(G), indexing="ij")
    d, ga, gs = d.ravel(), ga.ravel(), gs.ravel()
    r = oracle.verify_chain(xq, xp, d[:, None], u_acc=ga[:, None], u_samp=gs, shared_rows=True)
    w = p1[d] / (G * G)                       # weight of each enumerated case
    law0 = np.bincount(r["tokens"][:, 0], weights=w, minlength=V)
    assert np.abs(law0 - q1).max() < 2.0 / G
    acc = r["accept_len"] == 1
    law1 = np.bincount(r["tokens"][acc, 1], weights=w[acc], minlength=V) / w[acc].sum()
    assert np.abs(law1 - q2).max() < 2.0 / G
    # a plausible mistake, planted in a copy of the inputs, is caught:
    # using the draft row as the verifier gives p1, far from q1
    r_bad = oracle.verify_chain(np.stack([xp[0], xq[1]]), xp, d[:, None], u_acc=ga[:, None],
                                u_samp=gs, shared_rows=True)
    bad = np.bincount(r_bad["tokens"][:, 0], weights=w, minlength=V)
    assert np.abs(bad - q1).max() > 0.2


def test_enumeration_two_positions_each_law_is_its_q():
    V, G = 4, 40
    q = np.array([[0.7, 0.1, 0.1, 0.1], [0.1, 0.1, 0.1, 0.7], [0.25, 0.05, 0.6, 0.1]])
    p = np.array([[0.1, 0.6, 0.2, 0.1], [0.4, 0.3, 0.2, 0.1]])
    xq, xp = np.log(q).astype(np.float32), np.log(p).astype(np.float32)
    qs = [oracle.softmax(x) for x in xq]
    ps = [oracle.softmax(x) for x in xp]
    d0, d1, a0, a1, s = np.meshgrid(np.arange(V), np.arange(V), _grid(G), _grid(G), _grid(G), indexing="ij")
    toks = np.stack([d0.ravel(), d1.ravel()], 1)
    ua = np.stack([a0.ravel(), a1.ravel()], 1)
    r = oracle.verify_chain(xq, xp, toks, u_acc=ua, u_samp=s.ravel(), shared_rows=True)
    w = ps[0][toks[:, 0]] * ps[1][toks[:, 1]] / G**3
    for pos in range(3):
        em = r["accept_len"] >= pos
        law = np.bincount(r["tokens"][em, pos], weights=w[em], minlength=V) / w[em].sum()
        assert np.abs(law - qs[pos]).max() < 3.0 / G, (pos, law, qs[pos])


def _constructed_pair(alpha, V=16):
    r = np.zeros(V); r[:8] = 1 / 8
    s1 = np.zeros(V); s1[8:12] = 1 / 4
    s2 = np.zeros(V); s2[12:] = 1 / 4
    q = alpha * r + (1 - alpha) * s1
    p = alpha * r + (1 - alpha) * s2
    with np.errstate(divide="ignore"):
        return np.log(q).astype(np.float32), np.log(p).astype(np.float32), p


@pytest.mark.parametrize("alpha,N", [(0.8, 4), (0.6, 5), (0.9, 7)])
def test_constructed_alpha_mean_tokens_per_pass(alpha, N):
    xq1, xp1, p = _constructed_pair(alpha)
    xq = np.tile(xq1, (N + 1, 1)); xp = np.tile(xp1, (N, 1))
    B, steps = 20000, 50
    rng = np.random.default_rng(int(alpha * 100) + N)
    emitted = []
    for step in range(steps):
        toks = rng.choice(16, size=(B, N), p=p)
        r = oracle.verify_chain(xq, xp, toks, seed=99, step=step, shared_rows=True)
        a = r["accept_len"]
        # every correction token lies where q > p (the residual's support)
        rej = a < N
        assert np.all((r["tokens"][rej, a[rej]] >= 8) & (r["tokens"][rej, a[rej]] < 12))
        emitted.append(a + 1)
    e = np.concatenate(emitted).astype(np.float64)
    # exact law of the accepted count: P(A=k) = a^k (1-a) for k < N, a^N at N
    k = np.arange(N + 1)
    pk = np.where(k < N, alpha ** k * (1 - alpha), alpha ** N)
    mean = (pk * (k + 1)).sum()
    var = (pk * (k + 1) ** 2).sum() - mean ** 2
    assert abs(mean - (1 - alpha ** (N + 1)) / (1 - alpha)) < 1e-12
    assert abs(oracle.expected_tokens(alpha, N) - mean) < 1e-12
    assert abs(e.mean() - mean) < 3 * math.sqrt(var / e.size), (e.mean(), mean)
    # the empirical law of A matches too
    hist = np.bincount(e.astype(int) - 1, minlength=N + 1) / e.size
    assert np.abs(hist - pk).max() < 4 * math.sqrt(0.25 / e.size)


def test_step5_chi_square_against_direct_sampling():
    V, N, n = 8, 3, 50000
    rng = np.random.default_rng(12)
    xq = (rng.standard_normal((N + 1, V)) * 1.2).astype(np.float32)
    xp = (xq[:N] + rng.standard_normal((N, V)) * 0.9).astype(np.float32)
    ps = [oracle.softmax(x) for x in xp]
    q1 = oracle.softmax(xq[0])
    toks = np.stack([rng.choice(V, size=n, p=ps[i]) for i in range(N)], 1)
    r = oracle.verify_chain(xq, xp, toks, seed=5, step=1, shared_rows=True)
    spec = np.bincount(r["tokens"][:, 0], minlength=V)
    # the direct samples come from their own stream
    direct = np.bincount(np.random.default_rng(2024).choice(V, size=n, p=q1), minlength=V)
    # two-sample chi-square, df = V - 1
    tot = spec + direct
    keep = tot > 0
    e1 = tot[keep] * 0.5
    stat = (((spec[keep] - e1) ** 2) / e1).sum() + (((direct[keep] - e1) ** 2) / e1).sum()
    assert stat < chi2.ppf(0.95, keep.sum() - 1), stat
    # goodness of fit of every emitted position against its own q_i
    for pos in range(N + 1):
        em = r["accept_len"] >= pos
        obs = np.bincount(r["tokens"][em, pos], minlength=V)
        exp_ = oracle.softmax(xq[pos]) * em.sum()
        assert ((obs - exp_) ** 2 / exp_).sum() < chi2.ppf(0.999, V - 1)


def test_worked_example_two_accepted_one_correction():
    # "北京 / 是 / 中国 / 的": the first two drafts pass, the third fails, and
    # the correction comes from the residual -- 3 tokens from one pass.
    V, N = 8, 4
    xq = np.zeros((N + 1, V), np.float32)
    xp = np.zeros((N, V), np.float32)
    drafts = np.array([[3, 1, 6, 2]])
    xq[2, :] = -np.inf
    xq[2, 5] = 0.0                    # q_3 is a point mass on token 5; q_3(6) = 0
    for seed in range(25):
        r = oracle.verify_chain(xq[None], xp[None], drafts, seed=seed, step=seed)
        assert r["accept_len"][0] == 2
        assert r["tokens"][0, :3].tolist() == [3, 1, 5]
        assert r["tokens"][0, 3:].tolist() == [-1, -1]
        assert r["status"][0] == 0


def test_data_faults_set_status_and_stop():
    V, N = 6, 2
    xq = np.zeros((1, N + 1, V), np.float32); xp = np.zeros((1, N, V), np.float32)
    bad = xq.copy(); bad[0, 1, 2] = np.nan
    r = oracle.verify_chain(bad, xp, np.array([[0, 1]]))
    assert r["status"][0] & oracle.ROW_NAN and r["accept_len"][0] == 0
    assert np.all(r["tokens"] == -1)
    r = oracle.verify_chain(xq, xp, np.array([[0, V]]))
    assert r["status"][0] & oracle.ROW_BAD_TOKEN and np.all(r["tokens"] == -1)
    inf = xq.copy(); inf[0, 0, 0] = np.inf
    assert oracle.verify_chain(inf, xp, np.array([[0, 1]]))["status"][0] & oracle.ROW_NAN
    allm = xp.copy(); allm[0, 1, :] = -np.inf
    assert oracle.verify_chain(xq, allm, np.array([[0, 1]]))["status"][0] & oracle.ROW_NAN
    # a -inf draft logit at the draft token: p(d) = 0, accepted outright
    pz = xp.copy(); pz[0, 0, 4] = -np.inf
    r = oracle.verify_chain(xq, pz, np.array([[4, 1]]), seed=3)
    assert r["status"][0] & oracle.ROW_P_ZERO and r["accept_len"][0] >= 1


# ---------------------------------------------------------------- greedy (T = 0)
def _bf16_rows(rng, shape, sigma=3.0):
    x = (rng.standard_normal(shape) * sigma).astype(np.float32)
    return (x.view(np.uint32) & 0xFFFF0000).view(np.float32)  # exact bf16 values


def test_greedy_matches_argmax_walk():
    """Greedy verification = accept while the draft token is the verifier
    row's arg max (numpy's first-occurrence arg max), then emit the arg max
    of the row where the walk stopped."""
    rng = np.random.default_rng(5)
    B, N, V = 64, 5, 37
    vq = _bf16_rows(rng, (B, N + 1, V))
    dp = _bf16_rows(rng, (B, N, V))
    am = vq.argmax(axis=-1)
    # half of the drafts copy the verifier's arg max, so walks run long
    d = np.where(rng.random((B, N)) < 0.7, am[:, :N], rng.integers(0, V, (B, N)))
    o = oracle.verify_chain(vq, dp, d, T=0.0, seed=1, step=2)
    for b in range(B):
        a = next((i for i in range(N) if d[b, i] != am[b, i]), N)
        assert o["accept_len"][b] == a
        assert list(o["tokens"][b, :a]) == list(d[b, :a])
        assert o["tokens"][b, a] == am[b, a]
        assert np.all(o["tokens"][b, a + 1:] == -1)
        assert np.array_equal(o["q_prob"][b], (d[b] == am[b, :N]).astype(float))
        assert o["status"][b] == 0


def test_greedy_is_the_low_temperature_limit():
    """Drafts drawn at T -> 0 are the draft rows' arg maxes.  At T = 1e-3 with
    a top-2 logit gap >= 1, every softmax is a point mass (exp(-1000)
    underflows): p(d) = 1, so min(1, q(d)/p(d)) is 1 iff d is the verifier's
    arg max, and the residual and the bonus are the verifier's arg max — the
    stochastic rule reduces exactly to the greedy walk."""
    rng = np.random.default_rng(6)
    B, N, V = 48, 4, 29
    vq = _bf16_rows(rng, (B, N + 1, V))
    dp = _bf16_rows(rng, (B, N, V))
    am = vq.argmax(axis=-1)
    # 60% of the draft rows share the verifier's arg max
    share = rng.random((B, N)) < 0.6
    top = np.where(share, am[:, :N], dp.argmax(axis=-1))
    np.put_along_axis(dp, top[..., None], dp.max(axis=-1, keepdims=True) + 2.0, -1)
    k = vq.argmax(axis=-1)
    np.put_along_axis(vq, k[..., None], vq.max(axis=-1, keepdims=True) + 2.0, -1)
    d = dp.argmax(axis=-1).astype(np.int32)
    g = oracle.verify_chain(vq, dp, d, T=0.0)
    s = oracle.verify_chain(vq, dp, d, T=1e-3, seed=3, step=9)
    assert np.array_equal(g["accept_len"], s["accept_len"])
    assert np.array_equal(g["tokens"], s["tokens"])


def test_greedy_ties_and_faults():
    V = 8
    vq = np.zeros((3, 2, V), np.float32)
    vq[:, :, 5] = 1.0
    vq[:, :, 2] = 1.0  # tie: the lowest token id wins
    vq[1, 0, 3] = np.nan
    d = np.array([[2], [2], [V]], np.int32)
    o = oracle.verify_chain(vq, np.zeros((3, 1, V), np.float32), d, T=0.0)
    assert o["accept_len"][0] == 1 and list(o["tokens"][0]) == [2, 2]
    assert o["status"][1] == 1 and o["accept_len"][1] == 0  # NaN row
    assert o["status"][2] == 2 and o["accept_len"][2] == 0  # token out of range
    assert oracle.argmax(vq[0, 0]) == 2


def test_greedy_tree_follows_best_path():
    """Tree mode at T = 0: the walk along the best-scored path accepts while
    each node's token is the arg max of its parent's verifier row."""
    rng = np.random.default_rng(7)
    T, V = 7, 19
    parent = np.array([-1, 0, 0, 1, 1, 2, 3], np.int32)
    score = np.array([1.0, 0.6, 0.3, 0.5, 0.1, 0.2, 0.4], np.float32)
    path = [0, 1, 3, 6]
    vq = _bf16_rows(rng, (1, T, V))
    dp = _bf16_rows(rng, (1, T, V))
    token = rng.integers(0, V, (1, T)).astype(np.int32)
    token[0, 1] = vq[0, 0].argmax()  # node 1 accepted
    token[0, 3] = vq[0, 1].argmax()  # node 3 accepted
    token[0, 6] = (vq[0, 3].argmax() + 1) % V  # node 6 rejected
    o = oracle.verify_tree(vq, dp, parent[None], token, score[None], 3, T=0.0)
    assert list(o["path"][0]) == [0, 1, 3, -1]
    assert o["accept_len"][0] == 2
    assert list(o["tokens"][0]) == [token[0, 1], token[0, 3], vq[0, 3].argmax(), -1]
