"""GPU parity of the dynamic draft-tree builder (sv_tree_expand,
sv_tree_select, sv_tree_finalize, and sv_tree_level, which runs a level's
expansion and selection through one candidate table) through the C ABI
against the oracle.
Tokens, picks and trees are compared exactly; child scores (fp32 softmax
against double) within 2e-6 relative."""
import numpy as np
import pytest
import torch

import oracle
from parity import to_np

pytestmark = pytest.mark.gpu

sv = pytest.importorskip("speculative_decoding_verification_vocab_gb300")

DEV = torch.device("cuda:0")
SCORE_RTOL = 2e-6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.load_library()


def _rows(g, shape, dtype, sigma=3.0):
    return (torch.randn(shape, generator=g) * sigma).to(dtype)


@pytest.mark.parametrize("dtype,V,K,T", [
    (torch.bfloat16, 128256, 10, 1.0),
    (torch.bfloat16, 1001, 16, 0.7),    # ragged rows, the largest K
    (torch.float32, 20481, 10, 1.0),
    (torch.bfloat16, 32000, 1, 1.0),
    (torch.bfloat16, 5000, 10, 0.0),    # greedy: probability 1 for the arg max
])
def test_expand_parity(dtype, V, K, T):
    g = torch.Generator().manual_seed(V + K)
    B, F = 6, 10
    x = _rows(g, (B, F, V), dtype, sigma=1.0)  # sigma 1 in bf16: many equal logits
    fs = torch.rand((B, F), generator=g) * 0.9 + 0.05
    x[0, 1, 17] = float("nan")
    x[1, 2, 5] = float("inf")
    x[2, 3] = -float("inf")
    fs[3, 4] = float("nan")
    tok, sc = sv.tree_expand(x.to(DEV), fs.to(DEV), K, temperature=T)
    torch.cuda.synchronize()
    otok, osc = oracle.tree_expand(x.float().numpy(), fs.numpy(), K, T=T)
    assert np.array_equal(to_np(tok), otok)
    gs = to_np(sc).astype(np.float64)
    assert np.array_equal(np.isneginf(gs), np.isneginf(osc))
    fin = np.isfinite(osc)
    assert np.allclose(gs[fin], osc[fin], rtol=SCORE_RTOL, atol=0.0)
    assert np.all(otok[0, 1] == -1) and np.all(otok[3, 4] == -1)


def test_select_and_finalize_exact():
    g = torch.Generator().manual_seed(3)
    B, C, K, Tn = 9, 511, 10, 60
    score = torch.randint(1, 40, (B, C), generator=g).float() / 64.0  # many ties
    score[:, 0] = 1.0
    token = torch.randint(-1, 1000, (B, C), generator=g, dtype=torch.int32)
    level = torch.randint(1, 7, (B, C), generator=g, dtype=torch.int32)
    level[:, 0] = 0
    parent = torch.zeros(B, C, dtype=torch.int32)
    parent[:, 0] = -1
    for c in range(1, C):
        parent[:, c] = torch.randint(0, c, (B,), generator=g, dtype=torch.int32)
    sel = sv.tree_select(score.to(DEV), token.to(DEV), K)
    p, t, s = sv.tree_finalize(parent.to(DEV), token.to(DEV), score.to(DEV), level.to(DEV), Tn)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(sel), oracle.tree_select(score.numpy(), token.numpy(), K))
    op, ot, os_ = oracle.tree_finalize(parent.numpy(), token.numpy(), score.numpy(),
                                       level.numpy(), Tn)
    assert np.array_equal(to_np(p), op) and np.array_equal(to_np(t), ot)
    assert np.array_equal(to_np(s), os_)


def test_build_config5_shaped_tree_and_verify_it():
    """A full EAGLE-2 build with config 5's shapes (B=128, depth 6, top-k 10,
    budget 60, V=128256): every level's expansion matches the oracle on the
    same rows, the pruning matches the oracle on the same candidates, the
    tree is valid, and sv_verify_tree accepts it."""
    B, V, K, depth, Tn = 128, 128256, 10, 6, 60
    levels = {}

    def level_rows(lvl, frontier):
        if lvl > depth:
            return None
        F = 1 if frontier is None else frontier.shape[1]
        g = torch.Generator(device=DEV).manual_seed(100 + lvl)
        x = (torch.randn((B, F, V), generator=g, device=DEV) * 3.0).to(torch.bfloat16)
        levels[lvl] = x
        return x

    (parent, token, score), (cp, ct, cs, cl) = sv.build_tree(level_rows, K, Tn,
                                                             return_candidates=True)
    torch.cuda.synchronize()
    # expansion of each level, on the rows and frontier scores the GPU used
    off = 1
    for lvl in range(1, depth + 1):
        x = levels[lvl]
        F = x.shape[1]
        n = F * K
        par = to_np(cp)[:, off:off + n].reshape(B, F, K)[:, :, 0]
        fs = np.take_along_axis(to_np(cs), par.astype(np.int64), 1)
        ids = np.random.default_rng(lvl).choice(B, 4, replace=False)
        otok, osc = oracle.tree_expand(x[ids].float().cpu().numpy(), fs[ids], K)
        assert np.array_equal(to_np(ct)[ids, off:off + n].reshape(4, F, K), otok)
        assert np.allclose(to_np(cs)[ids, off:off + n].reshape(4, F, K), osc, rtol=SCORE_RTOL)
        off += n
    op, ot, os_ = oracle.tree_finalize(to_np(cp), to_np(ct), to_np(cs), to_np(cl), Tn)
    assert np.array_equal(to_np(parent), op) and np.array_equal(to_np(token), ot)
    assert np.array_equal(to_np(score), os_)
    for b in range(0, B, 16):
        assert oracle.tree_valid(op[b], os_[b])
    # the built tree feeds the verify step
    g = torch.Generator(device=DEV).manual_seed(7)
    vq = (torch.randn((B, Tn, V), generator=g, device=DEV) * 3.0).to(torch.bfloat16)
    dp = (vq.float() + 0.3 * torch.randn((B, Tn, V), generator=g, device=DEV)).to(torch.bfloat16)
    out = sv.verify_tree(vq, dp, parent, token, score, depth)
    torch.cuda.synchronize()
    assert np.all(to_np(out["status"]) == 0)


def _plain_build(level_rows, K, Tn, T=1.0):
    """The same build from the plain primitives, with the bookkeeping between
    levels done here in torch: the reference for the candidate-table mode."""
    frontier, valid = None, None
    cp, ct, cs, cl = [], [], [], []
    depth = 0
    while True:
        rows = level_rows(depth + 1, frontier)
        if rows is None:
            break
        B, F, _ = rows.shape
        if frontier is None:
            frontier = torch.zeros(B, 1, dtype=torch.int64, device=DEV)
            cp.append(torch.full((B, 1), -1, dtype=torch.int32, device=DEV))
            ct.append(torch.zeros(B, 1, dtype=torch.int32, device=DEV))
            cs.append(torch.ones(B, 1, dtype=torch.float32, device=DEV))
            cl.append(torch.zeros(B, 1, dtype=torch.int32, device=DEV))
        depth += 1
        n0 = sum(c.shape[1] for c in ct)
        fs = torch.gather(torch.cat(cs, 1), 1, frontier)
        if valid is not None:
            fs = fs.masked_fill(~valid, float("nan"))
        tok, sc = sv.tree_expand(rows, fs.contiguous(), K, temperature=T)
        par = frontier.to(torch.int32)
        if valid is not None:
            par = torch.where(valid, par, torch.full_like(par, -1))
        cp.append(par.repeat_interleave(K, dim=1))
        ct.append(tok.reshape(B, F * K))
        cs.append(sc.reshape(B, F * K))
        cl.append(torch.full((B, F * K), depth, dtype=torch.int32, device=DEV))
        sel = sv.tree_select(cs[-1].contiguous(), ct[-1].contiguous(), K).to(torch.int64)
        valid = sel >= 0
        frontier = torch.where(valid, sel + n0, torch.zeros_like(sel))
    cands = tuple(torch.cat(a, 1).contiguous() for a in (cp, ct, cs, cl))
    return sv.tree_finalize(*cands, Tn), cands


@pytest.mark.parametrize("dtype,V,K,depth,Tn,T", [
    (torch.bfloat16, 3001, 4, 4, 20, 1.0),     # ragged rows
    (torch.float32, 4096, 10, 3, 60, 0.8),
    (torch.bfloat16, 5000, 16, 3, 100, 0.0),   # greedy, the largest K
])
def test_level_table_equals_plain_build(dtype, V, K, depth, Tn, T):
    """sv_tree_level (every step in the kernels) gives the candidate table
    and the tree of the plain primitives with host bookkeeping, bit for bit;
    a faulty level-1 row leaves its sequence with the root alone."""
    B = 6
    rows = {}

    def level_rows(lvl, frontier):
        if lvl > depth:
            return None
        F = 1 if lvl == 1 else K
        if lvl not in rows:
            g = torch.Generator(device=DEV).manual_seed(31 * lvl + V)
            x = (torch.randn((B, F, V), generator=g, device=DEV) * 2.0).to(dtype)
            if lvl == 1:
                x[2, 0, 7] = float("nan")     # sequence 2 proposes nothing
            rows[lvl] = x
        return rows[lvl]

    (p1, t1, s1), c1 = sv.build_tree(level_rows, K, Tn, temperature=T, return_candidates=True)
    (p0, t0, s0), c0 = _plain_build(level_rows, K, Tn, T=T)
    torch.cuda.synchronize()
    for a, b in zip(c1[1:], c0[1:]):            # tokens, scores, levels
        assert torch.equal(a, b)
    tok = c0[1]
    assert torch.equal(torch.where(tok >= 0, c1[0], 0), torch.where(tok >= 0, c0[0], 0))
    assert torch.equal(p1, p0) and torch.equal(t1, t0) and torch.equal(s1, s0)
    assert int((to_np(t1)[2] >= 0).sum()) == 1 and to_np(p1)[2, 0] == -1
    assert np.all(to_np(c1[1])[2, 1:] == -1) and np.all(to_np(c1[0])[2, 1 + K:] == -1)
