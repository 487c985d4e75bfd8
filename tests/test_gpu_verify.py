"""GPU parity: sv_verify_chain / sv_verify_tree / sv_tree_build_mask /
sv_kv_compact through the C ABI against the CPU oracle on the same seeded
inputs.  Small cases span several row segments, several 2048-token sampling
chunks and ragged tails; the full-size cases run the benchmark's launch
configuration and check a seeded sample of sequences one by one."""
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


def _cfg(dtype, sigma_q=3.0, sigma_noise=0.3, spike_frac=0.0, temperature=1.0):
    return synth.Config(99, "case", "chain", B=1, V=1, dtype=dtype, sigma_q=sigma_q,
                        sigma_noise=sigma_noise, spike_frac=spike_frac, spike=8.0,
                        temperature=temperature)


def _np32(t):
    return t.detach().float().cpu().numpy()


def run_chain(vq, dp, d, T=1.0, seed=0, step=0, seq_ids=None):
    g = sv.verify_chain(vq.to(DEV), dp.to(DEV), d.to(DEV), temperature=T, seed=seed, step=step)
    torch.cuda.synchronize()
    o = oracle.verify_chain(_np32(vq), _np32(dp), d.cpu().numpy(), T=T, seed=seed, step=step,
                            seq_ids=seq_ids)
    return g, o


CHAIN_CASES = [
    # dtype, B, N, V, T, sigma_noise, spike
    (torch.float32, 1, 4, 1000, 1.0, 0.5, 0.0),
    (torch.bfloat16, 7, 5, 1001, 1.0, 0.5, 0.05),     # ragged V: rows not 16-byte aligned
    (torch.bfloat16, 33, 3, 4099, 0.7, 0.4, 0.0),     # temperature, ragged tail chunk
    (torch.float32, 5, 0, 777, 1.0, 0.3, 0.0),        # no drafts: bonus only
    (torch.bfloat16, 3, 40, 3000, 1.0, 0.15, 0.0),    # more positions than a warp
    (torch.bfloat16, 16, 7, 40000, 1.0, 0.3, 0.0),    # several row segments and chunks
    (torch.float32, 9, 6, 20481, 1.3, 0.6, 0.05),     # fp32, segments, ragged
]


@pytest.mark.parametrize("dtype,B,N,V,T,sn,spike", CHAIN_CASES)
def test_chain_parity(dtype, B, N, V, T, sn, spike):
    cfg = _cfg(dtype, sigma_noise=sn, spike_frac=spike, temperature=T)
    for rep in range(2):
        vq, dp, d = synth.chain_inputs(cfg, seed=rep + 10 * B, B=B, V=V, N=N)
        g, o = run_chain(vq, dp, d, T=T, seed=1234 + rep, step=rep)
        compare_verify(g, o, rows_per_seq=N + 1, label=f"chain {dtype} B{B} N{N} V{V}")


def test_chain_data_faults():
    B, N, V = 8, 3, 517
    cfg = _cfg(torch.float32)
    vq, dp, d = synth.chain_inputs(cfg, seed=5, B=B, V=V, N=N)
    vq, dp, d = vq.clone(), dp.clone(), d.clone()
    vq[0, 1, 7] = float("nan")                 # NaN in a verifier row
    vq[1, 3, 0] = float("inf")                 # +inf in the bonus row
    dp[2, 0, :] = -float("inf")                # all -inf draft row
    d[3, 2] = V                                # token out of range
    d[4, 1] = -1
    dp[5, 0, d[5, 0]] = -float("inf")          # p(d) = 0: accepted outright
    vq[6, :, : V // 2] = -float("inf")         # masked half-vocabulary
    dp[6, :, : V // 2] = -float("inf")
    d[6] = torch.randint(V // 2, V, (N,))
    vq[7, 0, d[7, 0]] = -float("inf")          # q(d) = 0: always rejected
    g, o = run_chain(vq, dp, d, seed=9, step=2)
    compare_verify(g, o, rows_per_seq=N + 1, label="faults")
    st = to_np(g["status"])
    assert st[0] & sv.SV_ROW_NAN and st[1] & sv.SV_ROW_NAN and st[2] & sv.SV_ROW_NAN
    assert st[3] & sv.SV_ROW_BAD_TOKEN and st[4] & sv.SV_ROW_BAD_TOKEN
    assert st[5] & sv.SV_ROW_P_ZERO
    assert to_np(g["accept_len"])[7] == 0
    assert np.all(to_np(g["tokens"])[:5] == -1)


def test_chain_batch_zero_and_errors():
    x = torch.zeros(0, 3, 10, device=DEV)
    out = sv.verify_chain(x, torch.zeros(0, 2, 10, device=DEV),
                          torch.zeros(0, 2, dtype=torch.int32, device=DEV))
    assert out["tokens"].shape == (0, 3)
    with pytest.raises(sv.SvError):
        sv.verify_chain(torch.zeros(1, 3, 10, device=DEV), torch.zeros(1, 2, 10, device=DEV),
                        torch.zeros(1, 2, dtype=torch.int32, device=DEV), temperature=-1.0)


def test_chain_deterministic_and_step_dependent():
    cfg = _cfg(torch.bfloat16)
    vq, dp, d = synth.chain_inputs(cfg, seed=3, B=64, V=5000, N=5)
    vq, dp, d = vq.to(DEV), dp.to(DEV), d.to(DEV)
    a = sv.verify_chain(vq, dp, d, seed=1, step=4)
    b = sv.verify_chain(vq, dp, d, seed=1, step=4)
    c = sv.verify_chain(vq, dp, d, seed=1, step=5)
    torch.cuda.synchronize()
    for k in ("tokens", "accept_len", "status", "q_prob", "margin"):
        assert torch.equal(a[k], b[k]), k
    assert not torch.equal(a["tokens"], c["tokens"])


def test_gpu_law_chi_square_step5():
    """The lesson's Step 5 on the GPU path: 50,000 speculative steps, first
    emitted token against 50,000 direct samples of q, chi-square below the 95%
    critical value; and every emitted position against its own q_i."""
    from scipy.stats import chi2
    V, N, n = 8, 3, 50000
    rng = np.random.default_rng(12)
    xq = (rng.standard_normal((N + 1, V)) * 1.2).astype(np.float32)
    xp = (xq[:N] + rng.standard_normal((N, V)) * 0.9).astype(np.float32)
    ps = [oracle.softmax(x) for x in xp]
    toks = np.stack([rng.choice(V, size=n, p=ps[i]) for i in range(N)], 1).astype(np.int32)
    vq = torch.from_numpy(np.broadcast_to(xq, (n, N + 1, V)).copy()).to(DEV)
    dp = torch.from_numpy(np.broadcast_to(xp, (n, N, V)).copy()).to(DEV)
    g = sv.verify_chain(vq, dp, torch.from_numpy(toks).to(DEV), seed=77, step=3)
    tok, acc = to_np(g["tokens"]), to_np(g["accept_len"])
    spec = np.bincount(tok[:, 0], minlength=V)
    direct = np.bincount(np.random.default_rng(2024).choice(V, size=n, p=oracle.softmax(xq[0])),
                         minlength=V)
    tot = spec + direct
    e1 = tot * 0.5
    stat = (((spec - e1) ** 2) / e1).sum() + (((direct - e1) ** 2) / e1).sum()
    assert stat < chi2.ppf(0.95, V - 1), stat
    for pos in range(N + 1):
        em = acc >= pos
        obs = np.bincount(tok[em, pos], minlength=V)
        exp_ = oracle.softmax(xq[pos]) * em.sum()
        assert ((obs - exp_) ** 2 / exp_).sum() < chi2.ppf(0.999, V - 1)


# ------------------------------------------------------------------ trees
def run_tree(vq, dp, parent, token, score, max_depth, T=1.0, seed=0, step=0, seq_ids=None):
    g = sv.verify_tree(vq.to(DEV), dp.to(DEV), parent.to(DEV), token.to(DEV), score.to(DEV),
                       max_depth, temperature=T, seed=seed, step=step)
    torch.cuda.synchronize()
    o = oracle.verify_tree(_np32(vq), _np32(dp), parent.cpu().numpy(), token.cpu().numpy(),
                           score.cpu().numpy(), max_depth, T=T, seed=seed, step=step,
                           seq_ids=seq_ids)
    return g, o


def _npos_of(o, parent, score, max_depth):
    return np.array([len(oracle.tree_best_path(parent[b], score[b], max_depth)) - 1
                     for b in range(parent.shape[0])])


@pytest.mark.parametrize("V", [4099, 32000])
def test_static_tree_parity(V):
    c4 = synth.CONFIGS[4]
    for rep in range(2):
        vq, dp, parent, token, score = synth.static_tree_inputs(c4, seed=rep, B=12, V=V)
        for md in (c4.depth, 2):
            g, o = run_tree(vq, dp, parent, token, score, md, seed=rep, step=md)
            npos = _npos_of(o, parent.numpy(), score.numpy(), md)
            compare_verify(g, o, rows_per_seq=parent.shape[1], npos=npos, label=f"static V{V}")


def test_dynamic_tree_parity():
    c5 = synth.CONFIGS[5]
    vq, dp, parent, token, score = synth.dynamic_tree_inputs(c5, seed=4, B=16, V=6007)
    g, o = run_tree(vq, dp, parent, token, score, c5.depth, seed=8, step=1)
    npos = _npos_of(o, parent.numpy(), score.numpy(), c5.depth)
    compare_verify(g, o, rows_per_seq=parent.shape[1], npos=npos, label="dynamic")


def test_bad_trees_are_flagged():
    c4 = synth.CONFIGS[4]
    vq, dp, parent, token, score = synth.static_tree_inputs(c4, seed=2, B=4, V=999)
    parent, score = parent.clone(), score.clone()
    parent[0, 5] = 20            # parent after child
    parent[1, 0] = 0             # root with a parent
    score[2, 3] = float("nan")
    parent[3, 5] = -2            # a padded slot that still has children (13, 14, 15)
    g, o = run_tree(vq, dp, parent, token, score, c4.depth)
    assert np.all(to_np(g["status"]) == sv.SV_ROW_BAD_TREE)
    compare_verify(g, o, rows_per_seq=25, npos=np.zeros(4), label="bad trees")


def test_single_path_tree_equals_chain_bit_exactly():
    cfg = _cfg(torch.bfloat16)
    B, N, V = 24, 6, 9000
    vq, dp, d = synth.chain_inputs(cfg, seed=11, B=B, V=V, N=N)
    parent = torch.arange(-1, N, dtype=torch.int32).expand(B, N + 1).contiguous()
    token = torch.cat([torch.zeros(B, 1, dtype=torch.int32), d], 1)
    score = torch.rand(B, N + 1)
    dtree = torch.cat([dp, torch.zeros(B, 1, V, dtype=dp.dtype)], 1)
    ch = sv.verify_chain(vq.to(DEV), dp.to(DEV), d.to(DEV), temperature=0.9, seed=5, step=7)
    tr = sv.verify_tree(vq.to(DEV), dtree.to(DEV), parent.to(DEV), token.to(DEV), score.to(DEV),
                        N, temperature=0.9, seed=5, step=7)
    torch.cuda.synchronize()
    for k in ("tokens", "accept_len", "status", "q_prob", "p_prob"):
        assert torch.equal(ch[k], tr[k]), k
    assert torch.equal(torch.nan_to_num(ch["margin"], 9.0), torch.nan_to_num(tr["margin"], 9.0))


# ------------------------------------------------------------------ mask
def test_mask_parity():
    rng = np.random.default_rng(0)
    for T in (1, 15, 25, 64, 65, 130):
        B = 9
        parent = np.full((B, T), -2, np.int32)
        parent[:, 0] = -1
        for b in range(B):
            for c in range(1, T):
                if rng.random() < 0.9:
                    p = int(rng.integers(0, c))
                    while parent[b, p] == -2:
                        p = int(rng.integers(0, c))
                    parent[b, c] = p
        if T > 3:
            parent[0, 3] = 3          # invalid
        m, dpt = sv.tree_build_mask(torch.from_numpy(parent).to(DEV))
        torch.cuda.synchronize()
        om, od = oracle.tree_mask(parent)
        assert np.array_equal(to_np(m).view(np.uint64), om), T
        assert np.array_equal(to_np(dpt), od), T


# ------------------------------------------------------------------ KV
def _kv_case(L, B, S_src, S_dst, H, D, dtype, seed):
    src = synth.kv_cache(L, B, S_src, H, D, device=DEV, seed=seed, dtype=dtype)
    dst = synth.kv_cache(L, B, S_dst, H, D, device=DEV, seed=seed + 1, dtype=dtype)
    return src, dst


def _bytes(t):
    return t.detach().cpu().contiguous().view(torch.uint8).numpy().copy()


@pytest.mark.parametrize("L,B,H,D,dtype", [(3, 5, 8, 128, torch.bfloat16),
                                           (2, 4, 3, 5, torch.bfloat16),     # 30-byte rows
                                           (1, 7, 2, 16, torch.float32)])
def test_kv_compact_parity(L, B, H, D, dtype):
    rng = np.random.default_rng(L * 100 + D)
    S, P = 48, 10
    base = rng.integers(0, 20, B).astype(np.int32)
    rows = np.zeros((B, P), np.int32)
    n = rng.integers(0, P + 1, B).astype(np.int32)
    for b in range(B):                                # accepted-path-like rows
        r = np.sort(rng.choice(np.arange(1, 28 - 1), P - 1, replace=False))
        rows[b] = np.concatenate([[0], r])
    esz = torch.tensor([], dtype=dtype).element_size()
    # in place
    kv, _ = _kv_case(L, B, S, S, H, D, dtype, 1)
    ref = _bytes(kv)
    tb = torch.from_numpy(base).to(DEV)
    kl = sv.kv_compact(kv, kv, tb, tb, torch.from_numpy(rows).to(DEV),
                       torch.from_numpy(n - 1).to(DEV), 1)
    torch.cuda.synchronize()
    okl = oracle.kv_compact(ref, ref, L, B, S, S, H, D, esz, base, base, rows, n)
    assert np.array_equal(to_np(kl), okl)
    assert np.array_equal(_bytes(kv), ref)
    # scratch commit (separate buffers, identity rows)
    src, dst = _kv_case(L, B, 12, S, H, D, dtype, 2)
    sref, dref = _bytes(src), _bytes(dst)
    zeros = torch.zeros(B, dtype=torch.int32, device=DEV)
    nn = torch.from_numpy(np.minimum(n, 12)).to(DEV)
    kl = sv.kv_compact(src, dst, zeros, tb, None, nn, 0)
    torch.cuda.synchronize()
    okl = oracle.kv_compact(sref, dref, L, B, 12, S, H, D, esz, np.zeros(B, np.int32), base,
                            np.tile(np.arange(12, dtype=np.int32), (B, 1)), np.minimum(n, 12))
    assert np.array_equal(to_np(kl), okl)
    assert np.array_equal(_bytes(dst), dref)


def test_kv_invalid_requests_move_nothing():
    L, B, S, H, D = 2, 3, 16, 2, 8
    kv, _ = _kv_case(L, B, S, S, H, D, torch.bfloat16, 3)
    ref = _bytes(kv)
    rows = torch.tensor([[0, 3, 2], [0, 20, 0], [1, 0, 0]], dtype=torch.int32, device=DEV)
    base = torch.full((B,), 2, dtype=torch.int32, device=DEV)
    kl = sv.kv_compact(kv, kv, base, base, rows, torch.tensor([3, 2, 2], dtype=torch.int32,
                                                              device=DEV), 0)
    torch.cuda.synchronize()
    assert to_np(kl).tolist() == [-1, -1, -1]
    assert np.array_equal(_bytes(kv), ref)
    # The library moves at most 4096 rows of a sequence per call (its own
    # limit, stated in sv.h; the pages set none): sequence 0 asks for 4097 and
    # is refused with its destination untouched, sequence 1 asks for 4096 and
    # gets the oracle's bytes.
    big_src, big_dst = _kv_case(1, 2, 5000, 5000, 1, 8, torch.bfloat16, 4)
    sref, dref = _bytes(big_src), _bytes(big_dst)
    z = torch.zeros(2, dtype=torch.int32, device=DEV)
    nn = torch.tensor([4097, 4096], dtype=torch.int32, device=DEV)
    kl = sv.kv_compact(big_src, big_dst, z, z, None, nn, 0)
    torch.cuda.synchronize()
    assert to_np(kl).tolist() == [-1, 4096]
    okl = oracle.kv_compact(sref, dref, 1, 2, 5000, 5000, 1, 8, 2, np.zeros(2, np.int32),
                            np.zeros(2, np.int32), np.tile(np.arange(5000, dtype=np.int32), (2, 1)),
                            np.array([0, 4096], np.int32))
    assert okl.tolist() == [0, 4096]
    assert np.array_equal(_bytes(big_dst), dref)


# ------------------------------------------------------------------ full size
def _sample_ids(B, k, seed):
    return np.sort(np.random.default_rng(seed).choice(B, size=min(k, B), replace=False))


@pytest.mark.parametrize("idx", [1, 2, 3])
def test_full_size_chain_configs(idx):
    cfg = synth.CONFIGS[idx]
    vq, dp, d = synth.chain_inputs(cfg, seed=0, device=DEV)
    g = sv.verify_chain(vq, dp, d, temperature=cfg.temperature, seed=idx, step=0)
    torch.cuda.synchronize()
    ids = _sample_ids(cfg.B, 8, idx)
    o = oracle.verify_chain(_np32(vq[ids]), _np32(dp[ids]), d[ids].cpu().numpy(),
                            T=cfg.temperature, seed=idx, step=0, seq_ids=ids)
    sub = {k: (v[torch.from_numpy(ids).to(DEV)] if v is not None else None) for k, v in g.items()}
    compare_verify(sub, o, rows_per_seq=cfg.N + 1, label=f"config {idx}")
    # properties that hold for every sequence of the batch
    acc, tok = to_np(g["accept_len"]), to_np(g["tokens"])
    assert np.all((acc >= 0) & (acc <= cfg.N)) and np.all(to_np(g["status"]) == 0)
    for b in range(cfg.B):
        assert np.array_equal(tok[b, :acc[b]], to_np(d[b])[:acc[b]])
        assert 0 <= tok[b, acc[b]] < cfg.V and np.all(tok[b, acc[b] + 1:] == -1)


@pytest.mark.parametrize("idx", [4, 5])
def test_full_size_tree_configs(idx):
    cfg = synth.CONFIGS[idx]
    vq, dp, parent, token, score = synth.tree_inputs(cfg, seed=0, device=DEV)
    g = sv.verify_tree(vq, dp, parent, token, score, cfg.depth, seed=idx, step=0)
    mask, depth = sv.tree_build_mask(parent)
    torch.cuda.synchronize()
    ids = _sample_ids(cfg.B, 8, idx)
    tid = torch.from_numpy(ids).to(DEV)
    o = oracle.verify_tree(_np32(vq[tid]), _np32(dp[tid]), parent[tid].cpu().numpy(),
                           token[tid].cpu().numpy(), score[tid].cpu().numpy(), cfg.depth,
                           seed=idx, step=0, seq_ids=ids)
    sub = {k: (v[tid] if v is not None else None) for k, v in g.items()}
    npos = _npos_of(o, parent[tid].cpu().numpy(), score[tid].cpu().numpy(), cfg.depth)
    compare_verify(sub, o, rows_per_seq=parent.shape[1], npos=npos, label=f"config {idx}")
    om, od = oracle.tree_mask(parent.cpu().numpy())
    assert np.array_equal(to_np(mask).view(np.uint64), om)
    assert np.array_equal(to_np(depth), od)
    # compaction of the accepted paths, in place, on a window of the cache
    L, H, D = cfg.kv.L, cfg.kv.H, cfg.kv.D
    Bk = min(cfg.B, 16)
    S = parent.shape[1] + 4
    kv = synth.kv_cache(L, Bk, S, H, D, device=DEV, seed=idx)
    ref = _bytes(kv)
    base = torch.full((Bk,), 2, dtype=torch.int32, device=DEV)
    kl = sv.kv_compact(kv, kv, base, base, g["path"][:Bk].contiguous(),
                       g["accept_len"][:Bk].contiguous(), 1)
    torch.cuda.synchronize()
    okl = oracle.kv_compact(ref, ref, L, Bk, S, S, H, D, 2, to_np(base), to_np(base),
                            to_np(g["path"][:Bk]), to_np(g["accept_len"][:Bk]) + 1)
    assert np.array_equal(to_np(kl), okl)
    assert np.array_equal(_bytes(kv), ref)


def test_trace_and_launch_count():
    cfg = _cfg(torch.bfloat16)
    vq, dp, d = synth.chain_inputs(cfg, seed=1, B=4, V=3000, N=3)
    n0 = sv.sv_launch_count()
    sv.sv_trace_enable(True)
    sv.verify_chain(vq.to(DEV), dp.to(DEV), d.to(DEV))
    sv.sv_trace_enable(False)
    tr = sv.sv_trace_collect()
    assert sv.sv_launch_count() - n0 == 3
    assert set(tr) == {"row_stats", "decide", "sample"}
    assert all(v[0] == 1 and v[1] > 0 for v in tr.values())


# ------------------------------------------------------------ host-resident inputs
def _same(a, b):
    for k in a:
        if a[k] is None:
            continue
        x, y = a[k].cpu(), b[k].cpu()
        assert torch.equal(x.view(torch.int32) if x.dtype == torch.float32 else x,
                           y.view(torch.int32) if y.dtype == torch.float32 else y), k


def test_host_resident_tree_inputs():
    """Logits and tree arrays in page-locked host memory, read in place by the
    kernels: results bit-identical to the same call on device copies."""
    cfg = synth.CONFIGS[5]
    vq, dp, parent, token, score = synth.tree_inputs(cfg, seed=21, B=12, V=5003)
    dev_args = [x.to(DEV) for x in (vq, dp, parent, token, score)]
    host_args = [x.pin_memory() for x in (vq, dp, parent, token, score)]
    gd = sv.verify_tree(*dev_args, max_depth=cfg.depth, temperature=cfg.temperature, seed=5,
                        step=2)
    # with the host-size workspace (rows copied to the device once) ...
    gh = sv.verify_tree(*host_args, max_depth=cfg.depth, temperature=cfg.temperature, seed=5,
                        step=2)
    # ... and with the plain one (every step reads the host rows)
    B, T, V = vq.shape
    ws = torch.empty(sv.sv_verify_tree_workspace(B, T, cfg.depth, V), dtype=torch.uint8,
                     device=DEV)
    gp = sv.verify_tree(*host_args, max_depth=cfg.depth, temperature=cfg.temperature, seed=5,
                        step=2, workspace=ws)
    torch.cuda.synchronize()
    assert sv.sv_verify_tree_workspace_host(B, T, cfg.depth, V, vq.dtype) > ws.numel()
    _same(gd, gh)
    _same(gd, gp)
    md, dd = sv.tree_build_mask(dev_args[2])
    mh, dh = sv.tree_build_mask(host_args[2])
    torch.cuda.synchronize()
    assert torch.equal(md.cpu(), mh.cpu()) and torch.equal(dd.cpu(), dh.cpu())


def test_host_resident_chain_outputs():
    """Chain inputs and outputs both in page-locked host memory."""
    cfg = _cfg(torch.bfloat16, sigma_noise=0.4)
    vq, dp, d = synth.chain_inputs(cfg, seed=8, B=6, V=4097, N=5)
    gd = sv.verify_chain(vq.to(DEV), dp.to(DEV), d.to(DEV), seed=3, step=1)
    hv, hd, ht = vq.pin_memory(), dp.pin_memory(), d.pin_memory()
    B, N = 6, 5
    for ws_bytes in (sv.sv_verify_chain_workspace(B, N, 4097),
                     sv.sv_verify_chain_workspace_host(B, N, 4097, vq.dtype)):
        out = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in gd.items()}
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV)
        sv.sv_verify_chain(hv, hd, ht, 1.0, 3, 1, out["tokens"], out["accept_len"],
                           out["q_prob"], out["p_prob"], out["margin"], out["status"], ws)
        torch.cuda.synchronize()
        _same(gd, out)


def test_pageable_host_memory_refused():
    """A pageable host buffer is refused on the host before any launch."""
    import ctypes as C
    lib = sv.load_library()
    B, N, V = 2, 1, 64
    host = np.zeros((B, N + 1, V), np.float32)  # pageable
    dev = lambda shape, dt: torch.zeros(shape, dtype=dt, device=DEV)
    dl, dt_ = dev((B, N, V), torch.float32), dev((B, N), torch.int32)
    tok, acc, st = dev((B, N + 1), torch.int32), dev((B,), torch.int32), dev((B,), torch.int32)
    ws = dev((sv.sv_verify_chain_workspace(B, N, V),), torch.uint8)
    n0 = sv.sv_launch_count()
    p = lambda t: C.c_void_p(t.data_ptr())
    rc = lib.sv_verify_chain(C.c_void_p(host.ctypes.data), p(dl), 0, p(dt_), B, N, V, 1.0, 0, 0,
                             p(tok), p(acc), None, None, None, p(st), p(ws), ws.numel(), None,
                             None)
    assert rc == sv.SV_ERR_INVALID_ARG
    assert "pageable" in sv.sv_last_error()
    assert sv.sv_launch_count() == n0


def test_accept_event_marks_final_accept_outputs():
    """The accept event: once it has fired, accept lengths and paths are
    final, so a second stream can compact the KV cache while the sampling
    still runs; both streams' results match a plain single-stream call."""
    cfg = synth.CONFIGS[5]
    B, V = 16, 20000
    vq, dp, parent, token, score = (x.to(DEV) for x in synth.tree_inputs(cfg, seed=4, B=B, V=V))
    ref = sv.verify_tree(vq, dp, parent, token, score, cfg.depth, seed=9, step=3)
    torch.cuda.synchronize()
    main, side = torch.cuda.Stream(), torch.cuda.Stream()
    ev = torch.cuda.Event()
    L, S, H, D = 2, parent.shape[1] + 4, 2, 16
    kv = synth.kv_cache(L, B, S, H, D, device=DEV, seed=3)
    kv_ref = kv.clone()
    base = torch.zeros(B, dtype=torch.int32, device=DEV)
    main.wait_stream(torch.cuda.current_stream())
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(main):
        out = sv.verify_tree(vq, dp, parent, token, score, cfg.depth, seed=9, step=3,
                             stream=main, accept_event=ev)
    side.wait_event(ev)
    with torch.cuda.stream(side):
        acc_at_event = out["accept_len"].clone()
        path_at_event = out["path"].clone()
        kl = sv.kv_compact(kv, kv, base, base, out["path"], out["accept_len"], 1, stream=side)
    torch.cuda.synchronize()
    assert torch.equal(acc_at_event, ref["accept_len"])
    assert torch.equal(path_at_event, ref["path"])
    for k in ("tokens", "accept_len", "path", "status"):
        assert torch.equal(out[k], ref[k]), k
    kl_ref = sv.kv_compact(kv_ref, kv_ref, base, base, ref["path"], ref["accept_len"], 1)
    torch.cuda.synchronize()
    # random KV bytes hold NaN patterns: compare the bytes
    assert torch.equal(kl, kl_ref)
    assert torch.equal(kv.view(torch.int16), kv_ref.view(torch.int16))


def _path_rows_f32(x, parent, score, depth):
    """float32 copy of x [B][T][V] holding only each sequence's best-path rows
    (zeros elsewhere: the oracle reads only those rows), without a dense
    conversion of the whole tensor."""
    B, T, V = x.shape
    out = np.zeros((B, T, V), np.float32)
    for b in range(B):
        nodes = oracle.tree_best_path(parent[b], score[b], depth).astype(np.int64)
        out[b, nodes] = x[b, torch.from_numpy(nodes).to(x.device)].float().cpu().numpy()
    return out


@pytest.mark.parametrize("idx,early", [(3, False), (3, True), (5, False)])
def test_full_batch_parity_three_rounds(idx, early):
    """Every sequence of three rounds of the large configurations (not a
    sample): tokens, accept lengths, status and paths exact up to the near-tie
    rule, probabilities within tolerance."""
    cfg = synth.CONFIGS[idx]
    for rnd in range(3):
        if cfg.kind == "chain":
            vq, dp, d = synth.chain_inputs(cfg, seed=100 + rnd, device=DEV)
            g = sv.verify_chain(vq, dp, d, seed=idx, step=rnd, early_exit=early)
            torch.cuda.synchronize()
            o = oracle.verify_chain(_np32(vq), _np32(dp), d.cpu().numpy(), seed=idx, step=rnd,
                                    early_exit=early)
            compare_verify(g, o, rows_per_seq=cfg.N + 1, label=f"config {idx} round {rnd}")
        else:
            vq, dp, parent, token, score = synth.tree_inputs(cfg, seed=100 + rnd, device=DEV)
            g = sv.verify_tree(vq, dp, parent, token, score, cfg.depth, seed=idx, step=rnd)
            torch.cuda.synchronize()
            par, sc = parent.cpu().numpy(), score.cpu().numpy()
            o = oracle.verify_tree(_path_rows_f32(vq, par, sc, cfg.depth),
                                   _path_rows_f32(dp, par, sc, cfg.depth), par,
                                   token.cpu().numpy(), sc, cfg.depth, seed=idx, step=rnd)
            npos = _npos_of(o, par, sc, cfg.depth)
            compare_verify(g, o, rows_per_seq=parent.shape[1], npos=npos,
                           label=f"config {idx} round {rnd}")
