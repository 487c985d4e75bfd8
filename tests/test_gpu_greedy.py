"""GPU parity of greedy verification (temperature 0) through the C ABI
against the CPU oracle: accept while the draft token is the verifier row's
arg max (ties to the lowest id), then emit the arg max where the walk stops.
Everything is integer-exact, so everything is compared exactly."""
import numpy as np
import pytest
import torch

import oracle
from parity import to_np

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


def _greedy_drafts(vq, N, frac, seed):
    """Draft tokens: the verifier's arg max with probability `frac`, else a
    random token (so walks of every length occur)."""
    g = torch.Generator().manual_seed(seed)
    am = vq[:, :N].float().argmax(dim=-1).to(torch.int32)
    rnd = torch.randint(0, vq.shape[-1], am.shape, generator=g, dtype=torch.int32)
    keep = torch.rand(am.shape, generator=g) < frac
    return torch.where(keep, am, rnd)


def _same(g, o, label):
    for k in ("accept_len", "tokens", "status"):
        assert np.array_equal(to_np(g[k]).astype(np.int64), o[k].astype(np.int64)), (label, k)
    if "path" in o:
        assert np.array_equal(to_np(g["path"]), o["path"]), (label, "path")
    N = o["q_prob"].shape[1]
    if N:
        gq, oq = to_np(g["q_prob"])[:, :N], o["q_prob"]
        assert np.array_equal(np.isnan(gq), np.isnan(oq)), (label, "q NaN pattern")
        assert np.array_equal(gq[~np.isnan(gq)], oq[~np.isnan(oq)]), (label, "q")
        assert np.all(np.isnan(to_np(g["p_prob"])[:, :N])), (label, "p")
    assert np.all(np.isnan(to_np(g["margin"]))), (label, "margin")


CASES = [
    # dtype, B, N, V
    (torch.bfloat16, 33, 5, 32000),
    (torch.bfloat16, 7, 3, 1001),      # ragged rows (not 16-byte aligned)
    (torch.float32, 9, 6, 20481),      # fp32, several segments, ragged
    (torch.bfloat16, 5, 0, 777),       # bonus only
    (torch.bfloat16, 3, 40, 3000),     # more positions than a warp
    (torch.bfloat16, 16, 7, 128256),   # large vocabulary, 4 segments
]


@pytest.mark.parametrize("dtype,B,N,V", CASES)
def test_greedy_chain_parity(dtype, B, N, V):
    cfg = synth.Config(99, "case", "chain", B=1, V=1, dtype=dtype, sigma_q=3.0,
                       sigma_noise=0.3)
    vq, dp, _ = synth.chain_inputs(cfg, seed=B + N, B=B, V=V, N=N)
    d = _greedy_drafts(vq, N, 0.8, seed=N)
    g = sv.verify_chain(vq.to(DEV), dp.to(DEV), d.to(DEV), temperature=0.0)
    torch.cuda.synchronize()
    o = oracle.verify_chain(_np32(vq), _np32(dp), d.numpy(), T=0.0)
    _same(g, o, f"greedy chain {dtype} B{B} N{N} V{V}")


def test_greedy_ties_and_faults():
    B, N, V = 8, 2, 40000  # rows span two segments
    vq = torch.zeros(B, N + 1, V, dtype=torch.bfloat16)
    vq[:, :, 100] = 3.0
    vq[:, :, 39000] = 3.0          # a tie across segments: 100 wins
    vq[1, 0, 5] = 3.0              # an earlier tie inside the first segment
    vq[2, 1, V - 1] = 4.0          # the maximum in the ragged last word
    vq[3, 0, 7] = float("nan")
    vq[4, 2, 9] = float("inf")     # +inf in the bonus row
    vq[5, 1, :] = -float("inf")    # all -inf
    d = torch.full((B, N), 100, dtype=torch.int32)
    d[6, 1] = V                    # token out of range
    d[7, 0] = 39000                # the tie's higher index: rejected
    dp = torch.zeros(B, N, V, dtype=torch.bfloat16)
    g = sv.verify_chain(vq.to(DEV), dp.to(DEV), d.to(DEV), temperature=0.0)
    torch.cuda.synchronize()
    o = oracle.verify_chain(_np32(vq), _np32(dp), d.numpy(), T=0.0)
    _same(g, o, "ties/faults")
    st, acc, tok = to_np(g["status"]), to_np(g["accept_len"]), to_np(g["tokens"])
    assert acc[0] == 2 and list(tok[0]) == [100, 100, 100]
    assert acc[1] == 0 and tok[1, 0] == 5
    assert acc[2] == 1 and tok[2, 1] == V - 1
    assert st[3] == sv.SV_ROW_NAN and st[4] == sv.SV_ROW_NAN and st[5] == sv.SV_ROW_NAN
    assert st[6] == sv.SV_ROW_BAD_TOKEN
    assert acc[7] == 0 and tok[7, 0] == 100


@pytest.mark.parametrize("index", [4, 5])
def test_greedy_tree_parity(index):
    cfg = synth.CONFIGS[index]
    vq, dp, parent, token, score = synth.tree_inputs(cfg, seed=31, B=24, V=5003)
    # about half the nodes carry their parent's verifier arg max
    am = vq.float().argmax(dim=-1).to(torch.int32)
    par = parent.clamp(min=0).long()
    g0 = torch.Generator().manual_seed(index)
    keep = torch.rand(token.shape, generator=g0) < 0.5
    token = torch.where(keep, torch.gather(am, 1, par), token)
    g = sv.verify_tree(*(x.to(DEV) for x in (vq, dp, parent, token, score)), cfg.depth,
                       temperature=0.0)
    torch.cuda.synchronize()
    o = oracle.verify_tree(_np32(vq), _np32(dp), parent.numpy(), token.numpy(), score.numpy(),
                           cfg.depth, T=0.0)
    _same(g, o, f"greedy tree config {index}")
    assert to_np(g["accept_len"]).max() >= 2


def test_greedy_full_size_dynamic_tree_sample():
    """Config 5 at full size in one call; 8 sequences replayed by the oracle."""
    cfg = synth.CONFIGS[5]
    vq, dp, parent, token, score = synth.tree_inputs(cfg, seed=77, device=DEV)
    g = sv.verify_tree(vq, dp, parent, token, score, cfg.depth, temperature=0.0)
    torch.cuda.synchronize()
    ids = np.random.default_rng(1).choice(cfg.B, 8, replace=False)
    tid = torch.as_tensor(ids, device=DEV)
    o = oracle.verify_tree(_np32(vq[tid]), _np32(dp[tid]), parent[tid].cpu().numpy(),
                           token[tid].cpu().numpy(), score[tid].cpu().numpy(), cfg.depth, T=0.0)
    sub = {k: v[tid] for k, v in g.items() if v is not None}
    _same(sub, o, "greedy config 5 sample")


def test_greedy_host_resident_matches_device():
    cfg = synth.CONFIGS[5]
    vq, dp, parent, token, score = synth.tree_inputs(cfg, seed=5, B=12, V=5003)
    gd = sv.verify_tree(*(x.to(DEV) for x in (vq, dp, parent, token, score)), cfg.depth,
                        temperature=0.0)
    gh = sv.verify_tree(*(x.pin_memory() for x in (vq, dp, parent, token, score)), cfg.depth,
                        temperature=0.0)
    torch.cuda.synchronize()
    for k in ("accept_len", "tokens", "path", "status"):
        assert torch.equal(gd[k].cpu(), gh[k].cpu()), k
