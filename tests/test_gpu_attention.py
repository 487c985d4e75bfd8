"""GPU parity of the tree-masked verifier attention (sv_tree_attention)
through the C ABI against the oracle (double precision).

Tolerance, derived from the kernel's arithmetic: scores are fp32 sums of
exact bf16 products; the softmax weights come from ex2.approx (relative error
about 2^-22), are rounded to bf16 (relative error <= 2^-9) before the P.V
product, and the output is rounded to bf16 (<= 2^-9 of |out|).  The two roundings are bounded by 2^-9
max|v| each over the visible value rows, so |out - ref| <= 2^-8 max|v| plus
terms below 1e-5 max|v| (covered by a 1% margin).  The lse bound is computed from the data: the fp32 score error
gamma_128 * scale * sum_d |q_d k_d|, plus the fp32 sum of n weights
(n * 2^-24) and the ex2 approximation (2^-21 relative).
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_vocab_gb300 import synth

pytestmark = pytest.mark.gpu

sv = pytest.importorskip("speculative_decoding_verification_vocab_gb300")

DEV = torch.device("cuda:0")
U32 = 2.0 ** -24


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.load_library()


def _np(t):
    return t.detach().float().cpu().numpy()


def _run(q, kv, base, parent, scale):
    """GPU result (mask from the library's own builder) and oracle result
    (mask from the oracle's builder)."""
    pd = parent.to(DEV)
    mask_d, _ = sv.tree_build_mask(pd)
    out, lse, st = sv.tree_attention(q.to(DEV), kv.to(DEV), base.to(DEV), mask_d, scale,
                                     return_lse=True)
    torch.cuda.synchronize()
    omask, _ = oracle.tree_mask(parent.numpy())
    ref, rlse = oracle.tree_attention(_np(q), _np(kv), base.numpy(), omask, scale)
    return out, lse, st, ref, rlse, omask


def _check(q, kv, base, out, lse, ref, rlse, scale, T):
    o = _np(out).astype(np.float64)
    l = _np(lse).astype(np.float64)
    qf, kf, vf = _np(q), _np(kv[0]), _np(kv[1])
    B, _, Hq, D = q.shape
    Hkv = kv.shape[3]
    G = Hq // Hkv
    for b in range(B):
        n_keys = int(base[b]) + T
        for kh in range(Hkv):
            vmax = np.abs(vf[b, :n_keys, kh]).max()
            hs = slice(kh * G, (kh + 1) * G)
            err = np.abs(o[b, :, hs] - ref[b, :, hs]).max()
            assert err <= 2.0 ** -8 * vmax * 1.01, (b, kh, err, vmax)
            # lse bound from the data
            qk = np.abs(qf[b, :, hs]) @ np.abs(kf[b, :n_keys, kh]).T   # [T][G][n]
            gamma = D * U32 / (1 - D * U32)
            bound = gamma * scale * qk.max() + (n_keys + 2) * U32 + 2.0 ** -21 + 1e-6
            lerr = np.abs(l[b, :, hs] - rlse[b, :, hs])
            fin = np.isfinite(rlse[b, :, hs])
            assert np.array_equal(np.isneginf(l[b, :, hs]), np.isneginf(rlse[b, :, hs]))
            assert lerr[fin].max(initial=0.0) <= bound, (b, kh, lerr[fin].max(), bound)


@pytest.mark.parametrize("B,T,Hq,Hkv,S,base,depth", [
    (3, 25, 8, 2, 400, [0, 131, 250], 5),        # G=4; base 0: tree keys dominate
    (2, 60, 16, 2, 4300, [4096, 3001], 6),       # G=8, the dynamic-tree shape
    (2, 130, 4, 4, 700, [5, 511], 7),            # G=1: 2 query tiles, 3 mask words
    (2, 33, 16, 1, 300, [127, 128], 4),          # G=16: 5 query tiles; key tile edges
    (1, 1, 8, 8, 64, [17], 0),                   # a root alone
])
def test_attention_parity(B, T, Hq, Hkv, S, base, depth):
    scale = 128 ** -0.5
    q, kv, bt = synth.attention_inputs(B, T, Hq, Hkv, 128, S, base, seed=T + Hq)
    parent = synth.level_tree_parents(B, T, depth, seed=T)
    out, lse, st, ref, rlse, _ = _run(q, kv, bt, parent, scale)
    assert torch.count_nonzero(st).item() == 0
    _check(q, kv, bt, out, lse, ref, rlse, scale, T)


def test_attention_sharp_scores_pin_the_mask():
    """Large scores make every output row close to one value row: a key
    admitted or dropped by mistake shows far above the tolerance."""
    B, T, Hq, Hkv, S = 2, 40, 8, 1, 200
    q, kv, bt = synth.attention_inputs(B, T, Hq, Hkv, 128, S, [0, 70], seed=9, sigma=1.0)
    parent = synth.level_tree_parents(B, T, 6, seed=9)
    scale = 2.0
    out, lse, st, ref, rlse, _ = _run(q, kv, bt, parent, scale)
    assert torch.count_nonzero(st).item() == 0
    _check(q, kv, bt, out, lse, ref, rlse, scale, T)


def test_attention_chain_tree_and_lazy_rescale():
    """A chain tree (causal over the tree rows) whose scores grow along the
    keys, so that the running max rises tile after tile and O is rescaled."""
    B, T, Hq, Hkv, S = 2, 12, 8, 2, 1100
    q, kv, bt = synth.attention_inputs(B, T, Hq, Hkv, 128, S, [1000, 700], seed=4)
    ramp = torch.linspace(0.0, 3.0, S)[None, :, None, None]
    kv[0] = (kv[0].float() * 0.2 + ramp * q[:, :1].float().mean(2, keepdim=True)).to(torch.bfloat16)
    parent = torch.tensor([[-1] + list(range(T - 1))] * B, dtype=torch.int32)
    out, lse, st, ref, rlse, _ = _run(q, kv, bt, parent, 0.5)
    assert torch.count_nonzero(st).item() == 0
    _check(q, kv, bt, out, lse, ref, rlse, 0.5, T)


def test_attention_degenerate_and_bad_base():
    B, T, Hq, Hkv, S = 3, 6, 8, 2, 40
    q, kv, bt = synth.attention_inputs(B, T, Hq, Hkv, 128, S, [0, 37, 10], seed=2)
    parent = torch.tensor([[-1, 0, 1, 2, 3, 4]] * B, dtype=torch.int32)
    parent[0, 3] = 7                     # not a tree: empty mask, and base 0
    out, lse, st, ref, rlse, _ = _run(q, kv, bt, parent, 0.3)
    stn = st.cpu().numpy()
    assert stn[0] == 0 and stn[2] == 0 and stn[1] == 32          # SV_ROW_BAD_BASE
    o = _np(out)
    assert np.all(o[0] == 0) and np.all(np.isneginf(_np(lse)[0]))
    assert np.all(np.isnan(o[1])) and np.all(np.isnan(_np(lse)[1]))
    assert np.all(np.isnan(ref[1]))
    _check(q[2:], kv[:, 2:], bt[2:], out[2:], lse[2:], ref[2:], rlse[2:], 0.3, T)


def test_attention_deterministic_and_tail_independent():
    """Two calls agree bit for bit, and the slots past base + T (NaN here,
    then random) never change a result."""
    B, T, Hq, Hkv, S = 2, 20, 8, 2, 600
    q, kv, bt = synth.attention_inputs(B, T, Hq, Hkv, 128, S, [300, 451], seed=5)
    parent = synth.level_tree_parents(B, T, 4, seed=5).to(DEV)
    mask, _ = sv.tree_build_mask(parent)
    qd, kvd, bd = q.to(DEV), kv.to(DEV), bt.to(DEV)
    o1 = sv.tree_attention(qd, kvd, bd, mask, 0.1)
    o2 = sv.tree_attention(qd, kvd, bd, mask, 0.1)
    kv2 = kvd.clone()
    kv2[:, 0, 320:] = 1.0
    kv2[:, 1, 471:] = -3.0
    o3 = sv.tree_attention(qd, kv2, bd, mask, 0.1)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(o1.view(torch.int16), o3.view(torch.int16))


def test_attention_invalid_arguments():
    q = torch.zeros(1, 4, 8, 128, dtype=torch.bfloat16, device=DEV)
    kv = torch.zeros(2, 1, 16, 2, 128, dtype=torch.bfloat16, device=DEV)
    base = torch.zeros(1, dtype=torch.int32, device=DEV)
    mask = torch.zeros(1, 4, 1, dtype=torch.int64, device=DEV)
    out = torch.empty_like(q)
    with pytest.raises(sv.SvError) as e:
        sv.sv_tree_attention(q, kv, base, mask, 0.0, out)
    assert e.value.status == sv.SV_ERR_INVALID_ARG
    q64 = torch.zeros(1, 4, 8, 64, dtype=torch.bfloat16, device=DEV)
    kv64 = torch.zeros(2, 1, 16, 2, 64, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(sv.SvError) as e:
        sv.sv_tree_attention(q64, kv64, base, mask, 1.0, torch.empty_like(q64))
    assert e.value.status == sv.SV_ERR_UNSUPPORTED
    kv3 = torch.zeros(2, 1, 16, 3, 128, dtype=torch.bfloat16, device=DEV)
    q9 = torch.zeros(1, 4, 9, 128, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(sv.SvError) as e:                     # G = 3 does not divide 128
        sv.sv_tree_attention(q9, kv3, base, mask, 1.0, torch.empty_like(q9))
    assert e.value.status == sv.SV_ERR_UNSUPPORTED
    with pytest.raises(sv.SvError) as e:                     # host memory for q
        sv.sv_tree_attention(q.cpu().pin_memory(), kv, base, mask, 1.0, out)
    assert e.value.status == sv.SV_ERR_INVALID_ARG


def test_attention_full_size_sampled_rows():
    """The dynamic-tree workload (B=128 trees of 60 nodes, 64 query heads on 8
    KV heads of 128, context 4096) in the launch the benchmark times; sampled
    rows against the oracle one by one."""
    B, T, Hq, Hkv, D = 128, 60, 64, 8, 128
    S = 4096 + 64
    g = torch.Generator().manual_seed(11)
    base = (4096 - torch.randint(0, 512, (B,), generator=g)).to(torch.int32)
    q, kv, bt = synth.attention_inputs(B, T, Hq, Hkv, D, S, base.tolist(), seed=11,
                                       device=DEV)
    parent = synth.level_tree_parents(B, T, 6, seed=11)
    mask, _ = sv.tree_build_mask(parent.to(DEV))
    out, lse, st = sv.tree_attention(q, kv, bt, mask, D ** -0.5, return_lse=True)
    torch.cuda.synchronize()
    assert torch.count_nonzero(st).item() == 0
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    seqs = sorted(set(torch.randint(0, B, (6,), generator=g).tolist()) | {0, B - 1})
    sub = torch.tensor(seqs, device=DEV)
    qs, kvs = q[sub].cpu(), kv[:, sub].cpu()
    omask, _ = oracle.tree_mask(parent[sub.cpu()].numpy())
    sel = []
    for i in range(len(seqs)):
        for _ in range(16):
            sel.append([i, int(torch.randint(0, T, (1,), generator=g)),
                        int(torch.randint(0, Hq, (1,), generator=g))])
    sel = np.array(sel, np.int32)
    bs = bt[sub].cpu().numpy()
    ref, rlse = oracle.tree_attention(_np(qs), _np(kvs), bs, omask, D ** -0.5, sel=sel)
    o = _np(out[sub])
    l = _np(lse[sub])
    qf, kf, vf = _np(qs), _np(kvs[0]), _np(kvs[1])
    gamma = D * U32 / (1 - D * U32)
    for k, (i, n, h) in enumerate(sel):
        nk = int(bs[i]) + T
        kh = h // (Hq // Hkv)
        vmax = np.abs(vf[i, :nk, kh]).max()
        assert np.abs(o[i, n, h] - ref[k]).max() <= 2.0 ** -8 * vmax * 1.01
        qk = (np.abs(kf[i, :nk, kh]) @ np.abs(qf[i, n, h])).max()
        bound = gamma * D ** -0.5 * qk + (nk + 2) * U32 + 2.0 ** -21 + 1e-6
        assert abs(l[i, n, h] - rlse[k]) <= bound


def test_attention_wait_limit_runs_out_and_the_context_survives():
    """The timeout path, reached in the allowed way: every pipeline wait is
    given a limit of 1 ns (sv_tree_attention_ex), so the first wait that is
    not already satisfied gives up.  The call returns, the sequence carries
    SV_ROW_TIMEOUT, the copies and products already issued still complete
    (the kernel's drains keep their 2 s bound), and a normal call straight
    after it on the same context matches the oracle."""
    B, T, Hq, Hkv, S = 1, 4, 8, 2, 256
    q, kv, base = synth.attention_inputs(B, T, Hq, Hkv, 128, S, [200], seed=11)
    parent = torch.tensor([[-1, 0, 0, 1]], dtype=torch.int32)
    mask, _ = sv.tree_build_mask(parent.to(DEV))
    out, lse, st = sv.tree_attention(q.to(DEV), kv.to(DEV), base.to(DEV), mask, 128 ** -0.5,
                                     return_lse=True, wait_ns=1)
    torch.cuda.synchronize()
    assert int(st[0]) & sv.SV_ROW_TIMEOUT
    # the context is usable: a normal call on the same inputs is exact
    out, lse, st, ref, rlse, _ = _run(q, kv, base, parent, 128 ** -0.5)
    assert int(st.count_nonzero()) == 0
    _check(q, kv, base, out, lse, ref, rlse, 128 ** -0.5, T)
