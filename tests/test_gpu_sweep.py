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
