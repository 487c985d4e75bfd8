"""Pins for the oracle's early-exit reading of the chain walk (CPU only).

The pages' walk stops at the first rejection ([Lesson] Passo 3; [Blog]
section 4 spec_decode breaks out of its loop there), so the rows after it are
never needed.  Early exit reads, checks and reports only the rows the walk
reaches.  These tests tie that reading to the full reading (itself pinned by
the theorem tests) and to hand-built cases whose answer is fixed by the rule:

* on clean rows every emitted token, the accept length, the sampling gap and
  the status agree with the full reading; q(d), p(d) and the margin agree up
  to the rejecting position and are NaN after it;
* a NaN row or a bad token after the first rejection faults the full reading
  but not the early one; at or before it, both fault;
* the bonus row is checked only when every position passes.
"""
import numpy as np
import pytest

import oracle
from speculative_decoding_verification_vocab_gb300 import synth


def _inputs(seed, B=24, N=6, V=300):
    cfg = synth.CONFIGS[2]
    vq, dp, d = synth.chain_inputs(cfg, seed=seed, B=B, V=V, N=N)
    return vq.float().numpy(), dp.float().numpy(), d.numpy()


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_clean_rows_agree_with_full_reading(seed):
    vq, dp, d = _inputs(seed)
    B, N = d.shape
    full = oracle.verify_chain(vq, dp, d, seed=seed, step=7)
    ee = oracle.verify_chain(vq, dp, d, seed=seed, step=7, early_exit=True)
    for k in ("tokens", "accept_len", "status"):
        assert np.array_equal(full[k], ee[k]), k
    assert np.array_equal(full["gap"], ee["gap"])
    a = full["accept_len"]
    assert a.min() < N and a.max() == N          # both stopping kinds occur
    for b in range(B):
        last = min(int(a[b]), N - 1)             # the rejecting position, if any
        for k in ("q_prob", "p_prob"):
            assert np.array_equal(full[k][b, :last + 1], ee[k][b, :last + 1])
            assert np.all(np.isnan(ee[k][b, last + 1:]))
        assert np.array_equal(full["margin"][b, :last + 1], ee["margin"][b, :last + 1])
        assert np.all(np.isnan(ee["margin"][b, last + 1:N]))
        assert full["margin"][b, N] == ee["margin"][b, N] or np.isnan(full["margin"][b, N])


def _one_rejecting_sequence(N=5, V=16, reject_at=2):
    """Rows built so the walk accepts positions < reject_at and rejects there:
    the draft token is a point mass of p everywhere; q puts all its mass on it
    before reject_at (ratio 1) and none on it at reject_at (ratio 0)."""
    xq = np.zeros((1, N + 1, V), np.float32)
    xp = np.full((1, N, V), -np.inf, np.float32)
    d = np.arange(N, dtype=np.int32)[None] + 3
    for i in range(N):
        xp[0, i, d[0, i]] = 0.0
        if i < reject_at:
            xq[0, i, :] = -np.inf
            xq[0, i, d[0, i]] = 0.0
        elif i == reject_at:
            xq[0, i, d[0, i]] = -np.inf
    return xq, xp, d


def test_rejection_position_is_forced():
    xq, xp, d = _one_rejecting_sequence()
    for seed in range(10):
        for ee in (False, True):
            r = oracle.verify_chain(xq, xp, d, seed=seed, early_exit=ee)
            assert r["accept_len"][0] == 2 and r["status"][0] == 0
            assert r["tokens"][0, :2].tolist() == [3, 4]


@pytest.mark.parametrize("where", ["vrow", "drow", "token"])
def test_fault_after_rejection_only_faults_full_reading(where):
    xq, xp, d = _one_rejecting_sequence(reject_at=2)
    if where == "vrow":
        xq[0, 4, 7] = np.nan
    elif where == "drow":
        xp[0, 3, :] = -np.inf          # an all -inf row has no softmax
    else:
        d[0, 4] = 16                   # out of the vocabulary
    full = oracle.verify_chain(xq, xp, d, seed=1)
    ee = oracle.verify_chain(xq, xp, d, seed=1, early_exit=True)
    assert full["status"][0] & (oracle.ROW_NAN | oracle.ROW_BAD_TOKEN)
    assert full["accept_len"][0] == 0 and np.all(full["tokens"] == -1)
    assert ee["status"][0] == 0 and ee["accept_len"][0] == 2
    assert ee["tokens"][0, 2] >= 0     # the correction is drawn


@pytest.mark.parametrize("pos", [0, 1, 2])
def test_fault_at_or_before_rejection_faults_both(pos):
    xq, xp, d = _one_rejecting_sequence(reject_at=2)
    xq[0, pos, 0] = np.nan
    for ee in (False, True):
        r = oracle.verify_chain(xq, xp, d, seed=2, early_exit=ee)
        assert r["status"][0] == oracle.ROW_NAN
        assert r["accept_len"][0] == 0 and np.all(r["tokens"] == -1)
        assert np.all(np.isnan(r["q_prob"])) and np.all(np.isnan(r["margin"]))
    xq, xp, d = _one_rejecting_sequence(reject_at=2)
    d[0, pos] = -1
    r = oracle.verify_chain(xq, xp, d, seed=2, early_exit=True)
    assert r["status"][0] == oracle.ROW_BAD_TOKEN and r["accept_len"][0] == 0


def test_bonus_row_checked_only_when_reached():
    N = 5
    xq, xp, d = _one_rejecting_sequence(N=N, reject_at=N)   # every position passes
    xq[0, N, 1] = np.nan
    r = oracle.verify_chain(xq, xp, d, seed=0, early_exit=True)
    assert r["status"][0] == oracle.ROW_NAN and r["accept_len"][0] == 0
    xq2, xp2, d2 = _one_rejecting_sequence(N=N, reject_at=1)
    xq2[0, N, 1] = np.nan
    r = oracle.verify_chain(xq2, xp2, d2, seed=0, early_exit=True)
    assert r["status"][0] == 0 and r["accept_len"][0] == 1
    assert oracle.verify_chain(xq2, xp2, d2, seed=0)["status"][0] == oracle.ROW_NAN


def test_p_zero_flag_only_from_walked_positions():
    xq, xp, d = _one_rejecting_sequence(reject_at=2)
    # p(d) = 0 at position 1 (accepted outright) and at position 4 (never reached)
    for i in (1, 4):
        xp[0, i, :] = 0.0
        xp[0, i, d[0, i]] = -np.inf
    r = oracle.verify_chain(xq, xp, d, seed=5, early_exit=True)
    assert r["status"][0] == oracle.ROW_P_ZERO and r["accept_len"][0] == 2
    xp[0, 1, :] = -np.inf
    xp[0, 1, d[0, 1]] = 0.0
    r = oracle.verify_chain(xq, xp, d, seed=5, early_exit=True)
    assert r["status"][0] == 0


def test_greedy_has_no_early_exit_reading():
    xq, xp, d = _one_rejecting_sequence()
    with pytest.raises(ValueError):
        oracle.verify_chain(xq, xp, d, T=0.0, early_exit=True)
