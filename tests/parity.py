"""Comparison helpers for the GPU-vs-oracle parity tests.

Rules (the verify step's contract):
  * accept lengths, tokens, path nodes, status words and KV bytes are compared
    exactly;
  * the only allowed disagreement is a sequence whose accept decision is a
    near tie: the oracle's |min(1, q/p) - u| < 1e-5 at a position both sides
    tested.  Such sequences are counted and must stay under 0.01% of the
    verifier rows of the batch;
  * q(d), p(d) agree within 1e-6 absolute (fp32 against double); the accept
    margins within 2e-6; the sampled token's CDF gap within 1e-6 relative.
"""
import numpy as np

NEAR_TIE = 1e-5
PROB_TOL = 1e-6
MARGIN_TOL = 2e-6


def to_np(t):
    return None if t is None else t.detach().cpu().numpy()


def compare_verify(g, o, rows_per_seq, npos=None, label=""):
    """g: dict of GPU tensors, o: oracle dict.  Returns the near-tie count."""
    acc_g, acc_o = to_np(g["accept_len"]), o["accept_len"]
    tok_g, tok_o = to_np(g["tokens"]), o["tokens"]
    st_g, st_o = to_np(g["status"]).astype(np.uint32), o["status"]
    B = acc_o.shape[0]
    maxpos = tok_o.shape[1] - 1
    ties = []
    for b in range(B):
        same = acc_g[b] == acc_o[b] and np.array_equal(tok_g[b], tok_o[b]) and st_g[b] == st_o[b]
        if "path" in o:
            same = same and np.array_equal(to_np(g["path"])[b], o["path"][b])
        if same:
            continue
        a = min(int(acc_g[b]), int(acc_o[b]))
        n = maxpos if npos is None else int(npos[b])
        tested = [i for i in range(a + 1) if i < n]
        m = o["margin"][b, tested] if tested else np.array([])
        assert len(m) and np.nanmin(np.abs(m)) < NEAR_TIE, (
            f"{label} seq {b}: gpu a={acc_g[b]} tokens={tok_g[b].tolist()} status={st_g[b]} | "
            f"oracle a={acc_o[b]} tokens={tok_o[b].tolist()} status={st_o[b]} margins={m}")
        ties.append(b)
    assert len(ties) <= 1e-4 * B * rows_per_seq + 1e-9, f"{label}: {len(ties)} near ties"
    keep = np.ones(B, bool)
    keep[ties] = False
    if g.get("q_prob") is not None and maxpos > 0:
        for k in ("q_prob", "p_prob"):
            gv, ov = to_np(g[k])[keep, :maxpos], o[k][keep]
            fin = np.isfinite(ov)
            assert np.array_equal(fin, np.isfinite(gv)), f"{label} {k} NaN pattern"
            if fin.any():
                err = np.abs(gv[fin] - ov[fin]).max()
                assert err <= PROB_TOL, f"{label} {k} max err {err}"
        gm, om = to_np(g["margin"])[keep], o["margin"][keep]
        fin = np.isfinite(om[:, :maxpos])
        assert np.array_equal(fin, np.isfinite(gm[:, :maxpos])), f"{label} margin NaN pattern"
        if fin.any():
            err = np.abs(gm[:, :maxpos][fin] - om[:, :maxpos][fin]).max()
            assert err <= MARGIN_TOL, f"{label} margin max err {err}"
        gg, og = gm[:, maxpos], om[:, maxpos]
        fin = np.isfinite(og)
        assert np.array_equal(fin, np.isfinite(gg)), f"{label} gap NaN pattern"
        if fin.any():
            assert np.allclose(gg[fin], og[fin], rtol=1e-6, atol=1e-12), f"{label} gap"
    return len(ties)
