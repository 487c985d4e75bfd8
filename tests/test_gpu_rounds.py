"""GPU parity over many rounds of the small and medium configurations, full
batches, through the C ABI ([Lesson] Passo 5: the rule is checked over many
speculative steps, not one):

  * the tiny chain (B=1, N=4, V=1000, fp32): every one of its 100 rounds;
  * the batched chain (B=64, N=5, V=32000, bf16, 5% spiked rows) and the
    static EAGLE tree (B=32, 25 nodes, V=32000): every sequence of 100 rounds;
  * the dynamic tree (B=128, V=128256, 80-layer KV window): the in-place KV
    compaction of every sequence of a round ([Lesson] exercise 4, the batched
    rollback), byte for byte against the oracle.

Each configuration prints how many sequences were judged by the near-tie rule
and their rate per verifier row; the rate must stay below 1e-4."""
import numpy as np
import pytest
import torch

import oracle
from parity import compare_verify, to_np

pytestmark = pytest.mark.gpu

sv = pytest.importorskip("speculative_decoding_verification_vocab_gb300")
from speculative_decoding_verification_vocab_gb300 import synth  # noqa: E402

DEV = torch.device("cuda:0")
ROUNDS = 100


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.load_library()


def _np32(t):
    return t.detach().float().cpu().numpy()


def _report(label, ties, rows):
    rate = ties / rows
    print(f"{label}: {ties} near-tie sequences over {rows} verifier rows (rate {rate:.2e})")
    assert rate < 1e-4, (label, ties, rows)


@pytest.mark.parametrize("idx", [1, 2])
def test_chain_configs_every_round(idx):
    cfg = synth.CONFIGS[idx]
    ties, rows = 0, 0
    for rnd in range(ROUNDS):
        vq, dp, d = synth.chain_inputs(cfg, seed=rnd)  # drawn on the host, shared by both sides
        g = sv.verify_chain(vq.to(DEV), dp.to(DEV), d.to(DEV), temperature=cfg.temperature,
                            seed=idx, step=rnd)
        torch.cuda.synchronize()
        o = oracle.verify_chain(_np32(vq), _np32(dp), d.numpy(), T=cfg.temperature, seed=idx,
                                step=rnd)
        ties += compare_verify(g, o, rows_per_seq=cfg.N + 1, label=f"config {idx} round {rnd}")
        rows += cfg.B * (cfg.N + 1)
        assert np.all(to_np(g["status"]) == 0)
    _report(f"config {idx} ({ROUNDS} rounds)", ties, rows)


def test_static_tree_every_sequence_of_100_rounds():
    cfg = synth.CONFIGS[4]
    ties, rows = 0, 0
    for rnd in range(ROUNDS):
        vq, dp, parent, token, score = synth.tree_inputs(cfg, seed=rnd)
        par, sc = parent.numpy(), score.numpy()
        g = sv.verify_tree(vq.to(DEV), dp.to(DEV), parent.to(DEV), token.to(DEV), score.to(DEV),
                           cfg.depth, seed=4, step=rnd)
        torch.cuda.synchronize()
        o = oracle.verify_tree(_np32(vq), _np32(dp), par, token.numpy(), sc, cfg.depth, seed=4,
                               step=rnd)
        npos = np.array([len(oracle.tree_best_path(par[b], sc[b], cfg.depth)) - 1
                         for b in range(cfg.B)])
        ties += compare_verify(g, o, rows_per_seq=parent.shape[1], npos=npos,
                               label=f"config 4 round {rnd}")
        rows += cfg.B * parent.shape[1]
    _report(f"config 4 ({ROUNDS} rounds)", ties, rows)


def test_dynamic_tree_kv_compaction_every_sequence():
    """The accepted paths of a full config-5 round (B=128) gathered in place on
    the KV window of an 80-layer x 8-head x 128 cache (the root kept at its
    slot, accepted nodes moved to the slots after it), against the oracle's
    memmove-by-row."""
    cfg = synth.CONFIGS[5]
    vq, dp, parent, token, score = synth.tree_inputs(cfg, seed=3, device=DEV)
    g = sv.verify_tree(vq, dp, parent, token, score, cfg.depth, seed=5, step=3)
    torch.cuda.synchronize()
    del vq, dp
    L, H, D, B = cfg.kv.L, cfg.kv.H, cfg.kv.D, cfg.B
    S = parent.shape[1] + 4
    kv = synth.kv_cache(L, B, S, H, D, device=DEV, seed=5)
    ref = kv.detach().cpu().contiguous().view(torch.uint8).numpy().copy()
    base = torch.full((B,), 3, dtype=torch.int32, device=DEV)
    path, acc = g["path"].contiguous(), g["accept_len"].contiguous()
    kl = sv.kv_compact(kv, kv, base, base, path, acc, 1)
    torch.cuda.synchronize()
    okl = oracle.kv_compact(ref, ref, L, B, S, S, H, D, 2, to_np(base), to_np(base), to_np(path),
                            to_np(acc) + 1)
    assert np.array_equal(to_np(kl), okl)
    assert np.all(okl == 3 + to_np(acc) + 1)
    moved = int(sum(int(p != j) for b in range(B) for j, p in
                    enumerate(to_np(path)[b, 1:to_np(acc)[b] + 1], start=1)))
    assert moved > 0  # the round really moves rows
    assert np.array_equal(kv.detach().cpu().contiguous().view(torch.uint8).numpy(), ref)
