"""GPU parity over a seeded sweep of random shapes: chains (full and
early-exit readings, fp32 / bf16, ragged vocabularies, several temperatures,
N from 0 to 12) and trees (random level shapes, depth caps), each against the
oracle on the same inputs."""
import numpy as np
import pytest
import torch

import oracle
from parity import compare_verify

pytestmark = pytest.mark.gpu

sv = pytest.importorskip("speculative_decoding_verification_vocab_gb300")
from speculative_decoding_verification_vocab_gb300 import synth  # noqa: E402

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.load_library()


def _np32(t):
    return t.detach().float().cpu().numpy()


def _chain_case(seed):
    rng = np.random.default_rng(seed)
    dtype = torch.bfloat16 if rng.random() < 0.6 else torch.float32
    B = int(rng.integers(1, 40))
    N = int(rng.integers(0, 13))
    V = int(rng.choice([17, 100, 999, 2048, 3001, 9000, 16385, 40001]))
    T = float(rng.choice([0.5, 1.0, 1.7]))
    sn = float(rng.choice([0.05, 0.3, 1.0]))
    cfg = synth.Config(99, "sweep", "chain", B=B, V=V, dtype=dtype, sigma_q=3.0,
                       sigma_noise=sn, spike_frac=0.05, spike=8.0, temperature=T)
    return cfg, B, N, V, T


@pytest.mark.parametrize("seed", range(48))
def test_chain_sweep(seed):
    cfg, B, N, V, T = _chain_case(seed)
    vq, dp, d = synth.chain_inputs(cfg, seed=seed, B=B, V=V, N=N)
    for early in (False, True):
        g = sv.verify_chain(vq.to(DEV), dp.to(DEV), d.to(DEV), temperature=T, seed=seed,
                            step=3, early_exit=early)
        torch.cuda.synchronize()
        o = oracle.verify_chain(_np32(vq), _np32(dp), d.numpy(), T=T, seed=seed, step=3,
                                early_exit=early)
        compare_verify(g, o, rows_per_seq=N + 1,
                       label=f"sweep {seed} early={early} B{B} N{N} V{V} T{T} {cfg.dtype}")


@pytest.mark.parametrize("seed", range(24))
def test_tree_sweep(seed):
    rng = np.random.default_rng(100 + seed)
    B = int(rng.integers(1, 24))
    T = int(rng.integers(2, 64))
    depth = int(rng.integers(1, 8))
    V = int(rng.choice([50, 1001, 4096, 20000]))
    max_depth = int(rng.integers(0, depth + 2))
    dtype = torch.bfloat16 if rng.random() < 0.5 else torch.float32
    parent = synth.level_tree_parents(B, T, depth, seed=seed).to(torch.int32)
    g0 = torch.Generator().manual_seed(seed)
    vq = (torch.randn((B, T, V), generator=g0) * 3.0).to(dtype)
    dp = (vq.float() + 0.4 * torch.randn((B, T, V), generator=g0)).to(dtype)
    token = torch.randint(0, V, (B, T), generator=g0, dtype=torch.int32)
    score = torch.rand((B, T), generator=g0)
    # child scores never above the parent's (path products)
    for c in range(1, T):
        score[:, c] = torch.minimum(score[:, c], score.gather(1, parent[:, c:c + 1].long())[:, 0])
    g = sv.verify_tree(vq.to(DEV), dp.to(DEV), parent.to(DEV), token.to(DEV), score.to(DEV),
                       max_depth, seed=seed, step=5)
    torch.cuda.synchronize()
    par, sc = parent.numpy(), score.numpy()
    o = oracle.verify_tree(_np32(vq), _np32(dp), par, token.numpy(), sc, max_depth, seed=seed,
                           step=5)
    npos = np.array([len(oracle.tree_best_path(par[b], sc[b], max_depth)) - 1 for b in range(B)])
    compare_verify(g, o, rows_per_seq=T, npos=npos,
                   label=f"tree sweep {seed} B{B} T{T} depth{depth} cap{max_depth} V{V}")


@pytest.mark.parametrize("seed", range(24))
def test_greedy_sweep(seed):
    from test_gpu_greedy import _greedy_drafts, _same
    cfg, B, N, V, _ = _chain_case(1000 + seed)
    vq, dp, _ = synth.chain_inputs(cfg, seed=seed, B=B, V=V, N=N)
    d = _greedy_drafts(vq, N, 0.85, seed=seed)
    g = sv.verify_chain(vq.to(DEV), dp.to(DEV), d.to(DEV), temperature=0.0)
    torch.cuda.synchronize()
    o = oracle.verify_chain(_np32(vq), _np32(dp), d.numpy(), T=0.0)
    _same(g, o, f"greedy sweep {seed} B{B} N{N} V{V} {cfg.dtype}")


def _bytes(t):
    return t.detach().cpu().contiguous().view(torch.uint8).numpy().copy()


@pytest.mark.parametrize("seed", range(24))
def test_kv_compact_sweep(seed):
    """Random cache shapes and accepted paths, in place and as a commit from
    a separate buffer, byte for byte against the oracle."""
    rng = np.random.default_rng(500 + seed)
    L, B, H = int(rng.integers(1, 5)), int(rng.integers(1, 13)), int(rng.integers(1, 9))
    D = int(rng.choice([1, 3, 5, 16, 64, 128]))
    dtype = torch.bfloat16 if rng.random() < 0.6 else torch.float32
    esz = torch.tensor([], dtype=dtype).element_size()
    P = int(rng.integers(1, 12))
    span = P + int(rng.integers(0, 20))           # tree slots a path can use
    base = rng.integers(0, 16, B).astype(np.int32)
    S = int(base.max()) + span + 1
    rows = np.zeros((B, P), np.int32)
    for b in range(B):                            # root, then strictly increasing slots
        rows[b, 1:] = np.sort(rng.choice(np.arange(1, span), P - 1, replace=False))
    n = rng.integers(0, P + 1, B).astype(np.int32)  # rows kept (root included)
    kv = synth.kv_cache(L, B, S, H, D, device=DEV, seed=seed, dtype=dtype)
    ref = _bytes(kv)
    tb = torch.from_numpy(base).to(DEV)
    kl = sv.kv_compact(kv, kv, tb, tb, torch.from_numpy(rows).to(DEV),
                       torch.from_numpy(np.maximum(n - 1, 0)).to(DEV), 1)
    torch.cuda.synchronize()
    okl = oracle.kv_compact(ref, ref, L, B, S, S, H, D, esz, base, base, rows,
                            np.maximum(n, 1))
    assert np.array_equal(kl.cpu().numpy(), okl), seed
    assert np.array_equal(_bytes(kv), ref), seed
    # commit from a separate buffer of P rows to the cache at base
    src = synth.kv_cache(L, B, P, H, D, device=DEV, seed=seed + 50, dtype=dtype)
    dst = synth.kv_cache(L, B, S + P, H, D, device=DEV, seed=seed + 60, dtype=dtype)
    sref, dref = _bytes(src), _bytes(dst)
    zeros = torch.zeros(B, dtype=torch.int32, device=DEV)
    kl = sv.kv_compact(src, dst, zeros, tb, None, torch.from_numpy(n).to(DEV), 0)
    torch.cuda.synchronize()
    okl = oracle.kv_compact(sref, dref, L, B, P, S + P, H, D, esz, np.zeros(B, np.int32), base,
                            np.tile(np.arange(P, dtype=np.int32), (B, 1)), n)
    assert np.array_equal(kl.cpu().numpy(), okl), seed
    assert np.array_equal(_bytes(dst), dref), seed


@pytest.mark.parametrize("seed", range(16))
def test_tree_expand_sweep(seed):
    """Top-K expansion on random shapes: tokens exact, child scores within the
    builder's tolerance (bf16 rows with many equal logits included)."""
    from test_gpu_tree_build import SCORE_RTOL
    rng = np.random.default_rng(900 + seed)
    B, F = int(rng.integers(1, 9)), int(rng.integers(1, 11))
    V = int(rng.choice([16, 33, 1000, 1001, 4096, 20481, 70000]))
    K = int(rng.integers(1, min(16, V) + 1))
    T = float(rng.choice([0.0, 0.6, 1.0]))
    dtype = torch.bfloat16 if rng.random() < 0.6 else torch.float32
    sigma = float(rng.choice([0.3, 1.0, 3.0]))     # small sigma in bf16: many ties
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn((B, F, V), generator=g) * sigma).to(dtype)
    fs = torch.rand((B, F), generator=g) * 0.9 + 0.05
    tok, sc = sv.tree_expand(x.to(DEV), fs.to(DEV), K, temperature=T)
    torch.cuda.synchronize()
    otok, osc = oracle.tree_expand(x.float().numpy(), fs.numpy(), K, T=T)
    assert np.array_equal(tok.cpu().numpy(), otok), seed
    gs = sc.cpu().numpy().astype(np.float64)
    assert np.array_equal(np.isneginf(gs), np.isneginf(osc)), seed
    fin = np.isfinite(osc)
    assert np.allclose(gs[fin], osc[fin], rtol=SCORE_RTOL, atol=0.0), seed
