"""Pins for the oracle's tree-masked attention (CPU only).

The oracle computes, per query row, a softmax over the committed context
plus the node's own ancestors ([Blog] section 3: every flattened node sees
itself and its ancestors, never a sibling; [Lesson] "Reversão de KV cache":
the verifier's tree pass runs a non-causal mask that follows the tree).  These
tests tie it to things fixed independently of its code:

* a chain-shaped tree is ordinary causal attention, which torch's
  scaled_dot_product_attention computes (is_causal over the whole sequence);
* any tree equals unmasked attention over the rows gathered by walking the
  parent pointers (not the bitmask), one node at a time;
* zero queries give the mean of the visible value rows and lse = log(count);
* sibling rows never change a node's output, ancestor rows do;
* permuting the context rows (K and V together) changes nothing;
* the degenerate cases (no visible key, a base out of range).
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from speculative_decoding_verification_vocab_gb300 import synth


def _f(t):
    return t.float().numpy()


def _mask(parent):
    m, _ = oracle.tree_mask(np.asarray(parent, np.int32))
    return m


def _gqa(k, G):
    # [S][Hkv][D] -> [Hq][S][D]: query head h reads KV head h // G
    return k.permute(1, 0, 2).repeat_interleave(G, dim=0)


def test_chain_tree_is_causal_attention():
    B, T, Hq, Hkv, D, S = 2, 9, 4, 2, 16, 48
    base = [20, 31]
    q, kv, bt = synth.attention_inputs(B, T, Hq, Hkv, D, S, base, seed=1)
    parent = np.array([[-1] + list(range(T - 1))] * B, np.int32)
    out, lse = oracle.tree_attention(_f(q), _f(kv), bt.numpy(), _mask(parent), 0.25)
    G = Hq // Hkv
    for b in range(B):
        L = base[b] + T
        k = _gqa(kv[0, b, :L].double(), G)
        v = _gqa(kv[1, b, :L].double(), G)
        qf = torch.zeros((Hq, L, D), dtype=torch.float64)
        qf[:, base[b]:] = q[b].double().permute(1, 0, 2)
        ref = F.scaled_dot_product_attention(qf, k, v, is_causal=True, scale=0.25)
        got = torch.from_numpy(out[b]).permute(1, 0, 2)       # [Hq][T][D]
        assert torch.allclose(got, ref[:, base[b]:], rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tree_equals_gathered_ancestor_attention(seed):
    B, T, Hq, Hkv, D, S = 2, 25, 6, 3, 8, 64
    base = [0, 17] if seed == 0 else [5 + seed, 30]
    q, kv, bt = synth.attention_inputs(B, T, Hq, Hkv, D, S, base, seed=seed)
    parent = synth.level_tree_parents(B, T, 5, seed=seed).numpy()
    out, lse = oracle.tree_attention(_f(q), _f(kv), bt.numpy(), _mask(parent), 0.3)
    G = Hq // Hkv
    for b in range(B):
        for n in range(T):
            anc = []
            j = n
            while j >= 0:
                anc.append(j)
                j = int(parent[b, j])
            rows = list(range(base[b])) + [base[b] + a for a in sorted(anc)]
            k = _gqa(kv[0, b, rows].double(), G)
            v = _gqa(kv[1, b, rows].double(), G)
            qq = q[b, n].double()[:, None, :]                  # [Hq][1][D]
            ref = F.scaled_dot_product_attention(qq, k, v, scale=0.3)[:, 0]
            assert torch.allclose(torch.from_numpy(out[b, n]), ref, rtol=0, atol=1e-12)
            # lse against the log-sum-exp of the gathered scores
            sc = torch.einsum("hd,hsd->hs", q[b, n].double(), k) * 0.3
            assert np.allclose(lse[b, n], torch.logsumexp(sc, dim=1).numpy(), rtol=0, atol=1e-12)


def test_zero_queries_give_visible_mean_and_log_count():
    B, T, Hq, Hkv, D, S = 3, 12, 4, 4, 8, 40
    base = [0, 9, 28]
    q, kv, bt = synth.attention_inputs(B, T, Hq, Hkv, D, S, base, seed=4)
    q.zero_()
    parent = synth.level_tree_parents(B, T, 3, seed=4).numpy()
    mask, depth = oracle.tree_mask(parent)
    out, lse = oracle.tree_attention(_f(q), _f(kv), bt.numpy(), mask, 1.0)
    V = kv[1].double().numpy()
    for b in range(B):
        for n in range(T):
            cnt = base[b] + depth[b, n] + 1
            assert lse[b, n, 0] == pytest.approx(math.log(cnt), abs=1e-13)
            anc = [j for j in range(T) if (int(mask[b, n, 0]) >> j) & 1]
            rows = list(range(base[b])) + [base[b] + a for a in anc]
            for h in range(Hq):
                assert np.allclose(out[b, n, h], V[b, rows, h].mean(0), rtol=0, atol=1e-13)


def test_siblings_never_matter_ancestors_do():
    B, T, Hq, Hkv, D, S = 1, 7, 2, 1, 8, 20
    parent = np.array([[-1, 0, 0, 1, 1, 2, 2]], np.int32)     # 3 and 4 are siblings
    q, kv, bt = synth.attention_inputs(B, T, Hq, Hkv, D, S, [6], seed=5)
    m = _mask(parent)
    out0, _ = oracle.tree_attention(_f(q), _f(kv), bt.numpy(), m, 0.5)
    kv2 = kv.clone()
    kv2[:, 0, 6 + 4] = 3.0                                    # node 4: sibling of 3
    kv2[:, 0, 6 + 2] = -2.0                                   # node 2: other branch
    out1, _ = oracle.tree_attention(_f(q), _f(kv2), bt.numpy(), m, 0.5)
    assert np.array_equal(out0[0, 3], out1[0, 3])
    assert np.array_equal(out0[0, 1], out1[0, 1])
    assert not np.allclose(out0[0, 4], out1[0, 4])
    assert not np.allclose(out0[0, 5], out1[0, 5])            # child of node 2
    kv3 = kv.clone()
    kv3[:, 0, 6 + 1] = 1.5                                    # node 1: ancestor of 3
    out2, _ = oracle.tree_attention(_f(q), _f(kv3), bt.numpy(), m, 0.5)
    assert not np.allclose(out0[0, 3], out2[0, 3])


def test_context_permutation_invariance():
    B, T, Hq, Hkv, D, S = 1, 10, 4, 2, 16, 64
    q, kv, bt = synth.attention_inputs(B, T, Hq, Hkv, D, S, [40], seed=6)
    m = _mask(synth.level_tree_parents(B, T, 3, seed=6).numpy())
    out0, lse0 = oracle.tree_attention(_f(q), _f(kv), bt.numpy(), m, 0.2)
    perm = torch.randperm(40, generator=torch.Generator().manual_seed(3))
    kv2 = kv.clone()
    kv2[:, 0, :40] = kv[:, 0, perm]
    out1, lse1 = oracle.tree_attention(_f(q), _f(kv2), bt.numpy(), m, 0.2)
    assert np.allclose(out0, out1, rtol=0, atol=1e-12)
    assert np.allclose(lse0, lse1, rtol=0, atol=1e-12)


def test_degenerate_rows():
    B, T, Hq, Hkv, D, S = 3, 5, 2, 1, 4, 12
    q, kv, bt = synth.attention_inputs(B, T, Hq, Hkv, D, S, [0, 8, 3], seed=7)
    parent = np.array([[-1, 0, 1, 2, 3]] * B, np.int32)
    m = _mask(parent)
    m[0] = 0                                                  # invalid tree, no context
    out, lse = oracle.tree_attention(_f(q), _f(kv), bt.numpy(), m, 1.0)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isnan(out[1])) and np.all(np.isnan(lse[1]))   # 8 + 5 > 12
    assert np.all(np.isfinite(out[2])) and np.all(np.isfinite(lse[2]))


def test_selected_rows_match_full_call():
    B, T, Hq, Hkv, D, S = 2, 9, 8, 2, 16, 30
    q, kv, bt = synth.attention_inputs(B, T, Hq, Hkv, D, S, [11, 4], seed=8)
    m = _mask(synth.level_tree_parents(B, T, 4, seed=8).numpy())
    out, lse = oracle.tree_attention(_f(q), _f(kv), bt.numpy(), m, 0.7)
    sel = np.array([[1, 8, 7], [0, 0, 0], [1, 3, 2], [0, 5, 6]], np.int32)
    o2, l2 = oracle.tree_attention(_f(q), _f(kv), bt.numpy(), m, 0.7, sel=sel)
    for i, (b, n, h) in enumerate(sel):
        assert np.array_equal(o2[i], out[b, n, h]) and l2[i] == lse[b, n, h]
