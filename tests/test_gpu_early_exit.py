"""GPU parity: sv_verify_chain_early_exit through the C ABI against the
oracle's early-exit reading on the same seeded inputs, and against the full
GPU path (same statistics, so the same decisions bit for bit)."""
import numpy as np
import pytest
import torch

import oracle
from parity import compare_verify, to_np

pytestmark = pytest.mark.gpu

sv = pytest.importorskip("speculative_decoding_verification_vocab_gb300")
from speculative_decoding_verification_vocab_gb300 import synth  # noqa: E402

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.load_library()


def _cfg(dtype, sigma_noise=0.3, spike_frac=0.0, temperature=1.0):
    return synth.Config(99, "case", "chain", B=1, V=1, dtype=dtype, sigma_q=3.0,
                        sigma_noise=sigma_noise, spike_frac=spike_frac, spike=8.0,
                        temperature=temperature)


def _np32(t):
    return t.detach().float().cpu().numpy()


CASES = [
    # dtype, B, N, V, T, sigma_noise, spike
    (torch.float32, 1, 4, 1000, 1.0, 0.5, 0.0),
    (torch.bfloat16, 7, 5, 1001, 1.0, 0.5, 0.05),     # rows not 16-byte aligned
    (torch.bfloat16, 33, 3, 4099, 0.7, 0.4, 0.0),     # temperature, ragged tail
    (torch.float32, 5, 0, 777, 1.0, 0.3, 0.0),        # no drafts: bonus only
    (torch.bfloat16, 3, 40, 3000, 1.0, 0.15, 0.0),    # more positions than a warp
    (torch.bfloat16, 16, 7, 40000, 1.0, 0.3, 0.0),    # several row segments
    (torch.float32, 9, 6, 20481, 1.3, 0.6, 0.05),     # fp32, segments, ragged
    (torch.bfloat16, 200, 7, 33000, 1.0, 0.3, 0.0),   # several position waves
]


@pytest.mark.parametrize("dtype,B,N,V,T,sn,spike", CASES)
def test_early_exit_parity(dtype, B, N, V, T, sn, spike):
    cfg = _cfg(dtype, sigma_noise=sn, spike_frac=spike, temperature=T)
    for rep in range(2):
        vq, dp, d = synth.chain_inputs(cfg, seed=rep + 10 * B, B=B, V=V, N=N)
        g = sv.verify_chain(vq.to(DEV), dp.to(DEV), d.to(DEV), temperature=T, seed=77 + rep,
                            step=rep, early_exit=True)
        full = sv.verify_chain(vq.to(DEV), dp.to(DEV), d.to(DEV), temperature=T, seed=77 + rep,
                               step=rep)
        torch.cuda.synchronize()
        o = oracle.verify_chain(_np32(vq), _np32(dp), d.numpy(), T=T, seed=77 + rep, step=rep,
                                early_exit=True)
        compare_verify(g, o, rows_per_seq=N + 1, label=f"early {dtype} B{B} N{N} V{V}")
        # against the full GPU path: identical decisions and draws
        for k in ("tokens", "accept_len", "status"):
            assert torch.equal(g[k], full[k]), k
        acc = to_np(g["accept_len"])
        gm, fm = to_np(g["margin"]), to_np(full["margin"])
        assert np.array_equal(gm[:, N], fm[:, N])           # the sampling gap
        for b in range(B):
            last = min(int(acc[b]), N - 1)
            for k in ("q_prob", "p_prob"):
                gv, fv = to_np(g[k])[b, :N], to_np(full[k])[b, :N]
                assert np.array_equal(gv[:last + 1], fv[:last + 1])
                assert np.all(np.isnan(gv[last + 1:]))
            assert np.array_equal(gm[b, :last + 1], fm[b, :last + 1])
            assert np.all(np.isnan(gm[b, last + 1:N]))


def _forced(B=6, N=5, V=700):
    """Sequence b rejects at position r = b % (N + 1): the drafts before r
    pass with ratio 1 (q and p both a point mass on the token) and q(d) = 0
    at r; r == N passes everywhere."""
    vq = torch.zeros(B, N + 1, V)
    dp = torch.full((B, N, V), -float("inf"))
    d = torch.arange(N, dtype=torch.int32)[None].repeat(B, 1) + 11
    rej = []
    for b in range(B):
        r = b % (N + 1)
        rej.append(r)
        for i in range(N):
            dp[b, i, d[b, i]] = 0.0
            if i < r:
                vq[b, i, :] = -float("inf")
                vq[b, i, d[b, i]] = 0.0
            elif i == r:
                vq[b, i, d[b, i]] = -float("inf")
    return vq, dp, d, rej


def test_faults_follow_the_walk():
    vq, dp, d, rej = _forced(B=12)
    N, V = 5, 700
    vq, dp, d = vq.clone(), dp.clone(), d.clone()
    # after the rejection: not seen by early exit
    vq[1, 3, 5] = float("nan")        # rejects at 1
    dp[2, 4, :] = -float("inf")       # rejects at 2
    d[3, 4] = V                       # rejects at 3
    vq[4, N, 0] = float("nan")        # rejects at 4: bonus row never reached
    # at or before the rejection: faults
    vq[7, 0, 9] = float("nan")        # rejects at 1, NaN at 0
    dp[8, 2, 3] = float("inf")        # rejects at 2, bad draft row at 2
    d[9, 1] = -5                      # rejects at 3, bad token at 1
    vq[11, N, 2] = float("inf")       # passes everywhere: bonus row bad
    g = sv.verify_chain(vq.to(DEV), dp.to(DEV), d.to(DEV), seed=4, step=1, early_exit=True)
    full = sv.verify_chain(vq.to(DEV), dp.to(DEV), d.to(DEV), seed=4, step=1)
    torch.cuda.synchronize()
    o = oracle.verify_chain(vq.numpy(), dp.numpy(), d.numpy(), seed=4, step=1,
                            early_exit=True)
    compare_verify(g, o, rows_per_seq=N + 1, label="early faults")
    st, acc = to_np(g["status"]), to_np(g["accept_len"])
    for b in (1, 2, 3, 4):
        assert st[b] == 0 and acc[b] == rej[b], b
        assert to_np(full["status"])[b] != 0
    assert st[7] == sv.SV_ROW_NAN and st[8] == sv.SV_ROW_NAN
    assert st[9] == sv.SV_ROW_BAD_TOKEN and st[11] == sv.SV_ROW_NAN
    assert np.all(to_np(g["tokens"])[[7, 8, 9, 11]] == -1)
    assert acc[5] == N and st[5] == 0  # b = 5 passes everywhere


def test_large_batch_parity_and_skipped_rows_never_used():
    """Many position waves (rows are skipped): every sequence's walk is the
    full path's, and rows poisoned after each rejection change nothing."""
    cfg = _cfg(torch.bfloat16, sigma_noise=0.3)
    B, N, V = 512, 7, 32000
    vq, dp, d = synth.chain_inputs(cfg, seed=21, B=B, V=V, N=N)
    vq, dp, d = vq.to(DEV), dp.to(DEV), d.to(DEV)
    full = sv.verify_chain(vq, dp, d, seed=5, step=3)
    torch.cuda.synchronize()
    acc = full["accept_len"]
    # poison every row after each sequence's rejection position
    pos = torch.arange(N + 1, device=DEV)[None]
    after = pos > acc[:, None]                                # [B][N+1]
    vq2 = vq.clone()
    vq2[after] = float("nan")
    dp2 = dp.clone()
    dp2[after[:, :N]] = float("nan")
    g = sv.verify_chain(vq2, dp2, d, seed=5, step=3, early_exit=True)
    torch.cuda.synchronize()
    for k in ("tokens", "accept_len", "status"):
        assert torch.equal(g[k], full[k]), k
    ids = np.sort(np.random.default_rng(2).choice(B, 12, replace=False))
    t = torch.from_numpy(ids).to(DEV)
    o = oracle.verify_chain(_np32(vq2[t]), _np32(dp2[t]), d[t].cpu().numpy(), seed=5, step=3,
                            seq_ids=ids, early_exit=True)
    compare_verify({k: (v[t] if v is not None else None) for k, v in g.items()}, o,
                   rows_per_seq=N + 1, label="poisoned tails")


def test_full_size_large_vocab_chain():
    cfg = synth.CONFIGS[3]
    vq, dp, d = synth.chain_inputs(cfg, seed=0, device=DEV)
    g = sv.verify_chain(vq, dp, d, seed=3, step=0, early_exit=True)
    full = sv.verify_chain(vq, dp, d, seed=3, step=0)
    torch.cuda.synchronize()
    for k in ("tokens", "accept_len", "status"):
        assert torch.equal(g[k], full[k]), k
    ids = np.sort(np.random.default_rng(3).choice(cfg.B, 8, replace=False))
    t = torch.from_numpy(ids).to(DEV)
    o = oracle.verify_chain(_np32(vq[t]), _np32(dp[t]), d[t].cpu().numpy(), seed=3, step=0,
                            seq_ids=ids, early_exit=True)
    compare_verify({k: (v[t] if v is not None else None) for k, v in g.items()}, o,
                   rows_per_seq=cfg.N + 1, label="config 3 early exit")


def test_host_resident_inputs():
    cfg = _cfg(torch.bfloat16, sigma_noise=0.4)
    B, N, V = 40, 5, 4097
    vq, dp, d = synth.chain_inputs(cfg, seed=8, B=B, V=V, N=N)
    gd = sv.verify_chain(vq.to(DEV), dp.to(DEV), d.to(DEV), seed=3, step=1, early_exit=True)
    hv, hd, ht = vq.pin_memory(), dp.pin_memory(), d.pin_memory()
    for ws_bytes in (sv.sv_verify_chain_workspace(B, N, V),
                     sv.sv_verify_chain_workspace_host(B, N, V, vq.dtype)):
        out = {k: torch.empty(v.shape, dtype=v.dtype, device=DEV) for k, v in gd.items()}
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV)
        sv.sv_verify_chain_early_exit(hv, hd, ht, 1.0, 3, 1, out["tokens"], out["accept_len"],
                                      out["q_prob"], out["p_prob"], out["margin"],
                                      out["status"], ws)
        torch.cuda.synchronize()
        for k, v in gd.items():
            assert torch.equal(torch.nan_to_num(v, nan=-7.0), torch.nan_to_num(out[k], nan=-7.0)), k


def test_repeated_calls_reset_their_counts():
    cfg = _cfg(torch.bfloat16)
    vq, dp, d = synth.chain_inputs(cfg, seed=3, B=300, V=5000, N=5)
    vq, dp, d = vq.to(DEV), dp.to(DEV), d.to(DEV)
    ws = torch.empty(sv.sv_verify_chain_workspace(300, 5, 5000), dtype=torch.uint8, device=DEV)
    outs = [sv.verify_chain(vq, dp, d, seed=1, step=s, workspace=ws, early_exit=True)
            for s in (4, 4, 5)]
    full = sv.verify_chain(vq, dp, d, seed=1, step=5)
    torch.cuda.synchronize()
    for k in ("tokens", "accept_len", "status"):
        assert torch.equal(outs[0][k], outs[1][k]), k
        assert torch.equal(outs[2][k], full[k]), k


def test_greedy_is_refused():
    x = torch.zeros(1, 3, 10, device=DEV)
    with pytest.raises(sv.SvError):
        sv.verify_chain(x, torch.zeros(1, 2, 10, device=DEV),
                        torch.zeros(1, 2, dtype=torch.int32, device=DEV), temperature=0.0,
                        early_exit=True)
