"""Seeded synthetic workloads for the verify-and-accept step.

This module is the one piece that the tests, the oracle checks, the smoke run
and the benchmark share.  It draws inputs only: random logits, draft tokens
and draft trees.  It implements none of the verify path (no accept rule, no
residual, no inverse CDF).  The draft side -- which the pages leave to the
draft model -- is simulated with torch library routines: Gumbel-max draws for
d ~ p, ``torch.topk`` / ``torch.log_softmax`` for the EAGLE tree's top-k
children and path scores.

The five workloads follow the configurations the verify step is measured on:
  1 tiny chain    B=1,   N=4, V=1000,   fp32, q ~ N(0, 2^2), draft noise 0.5
  2 batched chain B=64,  N=5, V=32000,  bf16, q ~ N(0, 3^2), 5% rows spiked +8
  3 large vocab   B=256, N=7, V=128256, bf16, q ~ N(0, 3^2)
  4 static tree   B=32,  T=25 (levels 1|4|8|6|4|2, depth 5), V=32000, bf16
  5 dynamic tree  B=128, budget 60, depth 6, top-k 10, V=128256, bf16
Draft logits are verifier logits plus N(0, sigma^2), with sigma chosen so
that alpha = E[sum_v min(p_v, q_v)] is near 0.8 / 0.9 / 0.75 / 0.9
(``tests/golden/calibrate_sigma.py`` measures alpha with the oracle).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass
class KVShape:
    L: int
    H: int
    D: int
    base: int


@dataclass
class Config:
    index: int
    name: str
    kind: str               # "chain" | "tree_static" | "tree_dynamic"
    B: int
    V: int
    dtype: torch.dtype
    sigma_q: float
    sigma_noise: float
    N: int = 0              # chain drafts
    T: int = 0              # tree slots
    depth: int = 0          # tree depth
    topk: int = 0
    spike_frac: float = 0.0
    spike: float = 0.0
    temperature: float = 1.0
    rounds: int = 1
    kv: KVShape = field(default_factory=lambda: KVShape(2, 2, 64, 32))
    target_alpha: float = 0.0


CONFIGS = {
    1: Config(1, "tiny_chain", "chain", B=1, V=1000, dtype=torch.float32, sigma_q=2.0,
              sigma_noise=0.5, N=4, rounds=100, kv=KVShape(2, 2, 64, 32)),
    2: Config(2, "batched_chain", "chain", B=64, V=32000, dtype=torch.bfloat16, sigma_q=3.0,
              sigma_noise=0.51, N=5, spike_frac=0.05, spike=8.0, rounds=1000,
              kv=KVShape(32, 8, 128, 2048), target_alpha=0.8),
    3: Config(3, "large_vocab_chain", "chain", B=256, V=128256, dtype=torch.bfloat16,
              sigma_q=3.0, sigma_noise=0.255, N=7, rounds=200, kv=KVShape(32, 8, 128, 4096),
              target_alpha=0.9),
    4: Config(4, "static_eagle_tree", "tree_static", B=32, V=32000, dtype=torch.bfloat16,
              sigma_q=3.0, sigma_noise=0.65, T=25, depth=5, kv=KVShape(32, 8, 128, 2048),
              target_alpha=0.75),
    5: Config(5, "dynamic_eagle2_tree", "tree_dynamic", B=128, V=128256, dtype=torch.bfloat16,
              sigma_q=3.0, sigma_noise=0.26, T=60, depth=6, topk=10,
              kv=KVShape(80, 8, 128, 4096), target_alpha=0.9),
}

# Static EAGLE tree (config 4): number of children of each node, level by level,
# in slot order.  Levels 1|4|8|6|4|2 = 25 slots, depth 5.  Child r of a node
# carries the r-th most likely draft token at that node.
STATIC_TREE_CHILDREN = [
    [4],
    [4, 2, 1, 1],
    [3, 1, 0, 0, 1, 0, 1, 0],
    [2, 1, 0, 1, 0, 0],
    [1, 1, 0, 0],
    [0, 0],
]


def static_tree_parents():
    parent = [-1]
    level = [0]
    for counts in STATIC_TREE_CHILDREN:
        nxt = []
        assert len(counts) == len(level)
        for node, c in zip(level, counts):
            for _ in range(c):
                parent.append(node)
                nxt.append(len(parent) - 1)
        level = nxt
    return parent


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _gumbel_argmax(x, g):
    """One draw from softmax(x) per row (Gumbel-max), x float32 [..., V]."""
    u = torch.rand(x.shape, generator=g, device=x.device, dtype=torch.float32)
    u = u.clamp_(min=1e-20, max=1.0 - 1e-7)
    return torch.argmax(x - torch.log(-torch.log(u)), dim=-1).to(torch.int32)


def _rows(shape, sigma, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32) * sigma


def chain_inputs(cfg: Config, seed=None, device="cpu", B=None, V=None, N=None):
    """vlogits [B][N+1][V], dlogits [B][N][V] in cfg.dtype; draft tokens [B][N]
    drawn from the draft distributions the verifier will see."""
    B = cfg.B if B is None else B
    V = cfg.V if V is None else V
    N = cfg.N if N is None else N
    g = _gen(cfg.index * 1000003 + (0 if seed is None else seed), device)
    xq = _rows((B, N + 1, V), cfg.sigma_q, g, device)
    if cfg.spike_frac > 0:
        hit = torch.rand((B, N + 1), generator=g, device=device) < cfg.spike_frac
        tok = torch.randint(0, V, (B, N + 1), generator=g, device=device)
        bump = torch.zeros_like(xq)
        bump.scatter_(2, tok[..., None], cfg.spike)
        xq = xq + bump * hit[..., None]
    xp = xq[:, :N] + _rows((B, N, V), cfg.sigma_noise, g, device)
    vq = xq.to(cfg.dtype)
    dp = xp.to(cfg.dtype)
    d = _gumbel_argmax(dp.float() / cfg.temperature, g) if N > 0 else \
        torch.zeros((B, 0), dtype=torch.int32, device=device)
    return vq, dp, d.contiguous()


def _tree_from_levels(parents):
    T = len(parents)
    depth = [0] * T
    for c in range(1, T):
        depth[c] = depth[parents[c]] + 1
    return depth


def static_tree_inputs(cfg: Config, seed=None, device="cpu", B=None, V=None):
    """Config-4 style static tree: fixed shape, children = top-k draft tokens."""
    B = cfg.B if B is None else B
    V = cfg.V if V is None else V
    parents = static_tree_parents()
    T = len(parents)
    g = _gen(cfg.index * 1000003 + (0 if seed is None else seed), device)
    xq = _rows((B, T, V), cfg.sigma_q, g, device)
    xp = xq + _rows((B, T, V), cfg.sigma_noise, g, device)
    vq, dp = xq.to(cfg.dtype), xp.to(cfg.dtype)
    logp = torch.log_softmax(dp.float() / cfg.temperature, dim=-1)
    parent = torch.tensor(parents, dtype=torch.int32, device=device).expand(B, T).contiguous()
    token = torch.zeros((B, T), dtype=torch.int32, device=device)
    score = torch.zeros((B, T), dtype=torch.float32, device=device)
    score[:, 0] = 1.0
    token[:, 0] = torch.randint(0, V, (B,), generator=g, device=device).to(torch.int32)
    kids = {}
    for c in range(1, T):
        kids.setdefault(parents[c], []).append(c)
    for n, cs in kids.items():
        top = torch.topk(logp[:, n], len(cs), dim=-1)
        for r, c in enumerate(cs):
            token[:, c] = top.indices[:, r].to(torch.int32)
            score[:, c] = score[:, n] * torch.exp(top.values[:, r])
    return vq, dp, parent, token, score


def dynamic_tree_inputs(cfg: Config, seed=None, device="cpu", B=None, V=None, T=None,
                        depth=None, topk=None):
    """Config-5 style EAGLE-2 dynamic tree.  Per level, the top-k scored nodes
    of the previous level form the frontier; each frontier node proposes its
    top-k draft tokens with score = parent score * draft probability.  After
    `depth` levels the `T` best-scored nodes are kept (ancestor-closed, since a
    child never outscores its parent) and renumbered level by level."""
    B = cfg.B if B is None else B
    V = cfg.V if V is None else V
    T = cfg.T if T is None else T
    depth = cfg.depth if depth is None else depth
    K = cfg.topk if topk is None else topk
    g = _gen(cfg.index * 1000003 + (0 if seed is None else seed), device)
    # candidate store: per sequence lists of (parent_cand, token, score, level, frontier_row)
    root_q = _rows((B, V), cfg.sigma_q, g, device)
    root_p = root_q + _rows((B, V), cfg.sigma_noise, g, device)
    cand_parent = [torch.full((B, 1), -1, dtype=torch.int64, device=device)]
    cand_token = [torch.randint(0, V, (B, 1), generator=g, device=device)]
    cand_score = [torch.ones((B, 1), device=device)]
    cand_level = [torch.zeros((B, 1), dtype=torch.int64, device=device)]
    q_rows = {0: root_q}   # candidate id -> [B, V] rows, only for frontier nodes
    p_rows = {0: root_p}
    frontier = torch.zeros((B, 1), dtype=torch.int64, device=device)   # candidate ids
    f_q = root_q[:, None]
    f_p = root_p[:, None]
    n_cand = 1
    fq_store, fp_store, fid_store = [f_q], [f_p], [frontier]
    for lvl in range(1, depth + 1):
        F = frontier.shape[1]
        logp = torch.log_softmax(f_p.to(cfg.dtype).float() / cfg.temperature, dim=-1)
        top = torch.topk(logp, K, dim=-1)                      # [B, F, K]
        fscore = torch.gather(torch.cat(cand_score, 1), 1, frontier)
        sc = (fscore[..., None] * torch.exp(top.values)).reshape(B, F * K)
        par = frontier[..., None].expand(B, F, K).reshape(B, F * K)
        tok = top.indices.reshape(B, F * K)
        ids = torch.arange(n_cand, n_cand + F * K, device=device).expand(B, F * K)
        cand_parent.append(par)
        cand_token.append(tok)
        cand_score.append(sc)
        cand_level.append(torch.full((B, F * K), lvl, dtype=torch.int64, device=device))
        n_cand += F * K
        if lvl == depth:
            break
        sel = torch.topk(sc, K, dim=-1).indices                # next frontier
        frontier = torch.gather(ids, 1, sel)
        f_q = _rows((B, K, V), cfg.sigma_q, g, device)
        f_p = f_q + _rows((B, K, V), cfg.sigma_noise, g, device)
        fq_store.append(f_q)
        fp_store.append(f_p)
        fid_store.append(frontier)
    P_all = torch.cat(cand_parent, 1)
    Tok_all = torch.cat(cand_token, 1)
    S_all = torch.cat(cand_score, 1)
    Lv_all = torch.cat(cand_level, 1)
    # keep the T best (root first); order by (level, -score) so parents precede children
    # a child never outscores its parent; the level term breaks exact ties so
    # the kept set stays ancestor-closed
    key = S_all.double() - Lv_all.double() * 1e-9
    keep = torch.topk(key, T, dim=-1).indices
    kl = torch.gather(Lv_all, 1, keep)
    ks = torch.gather(S_all, 1, keep)
    order = torch.argsort(kl.double() * 4.0 - ks.double(), dim=-1)
    keep = torch.gather(keep, 1, order)                         # [B, T] candidate ids
    slot_of = torch.full((B, n_cand), -1, dtype=torch.int64, device=device)
    slot_of.scatter_(1, keep, torch.arange(T, device=device).expand(B, T))
    par_c = torch.gather(P_all, 1, keep)
    parent = torch.where(par_c < 0, torch.full_like(par_c, -1),
                         torch.gather(slot_of, 1, par_c.clamp(min=0)))
    token = torch.gather(Tok_all, 1, keep).to(torch.int32)
    score = torch.gather(S_all, 1, keep).float()
    # logit rows per kept slot: frontier nodes reuse their drafting rows
    xq = _rows((B, T, V), cfg.sigma_q, g, device)
    xp = xq + _rows((B, T, V), cfg.sigma_noise, g, device)
    for fid, fq, fp in zip(fid_store, fq_store, fp_store):
        for j in range(fid.shape[1]):
            s = torch.gather(slot_of, 1, fid[:, j:j + 1])[:, 0]
            m = s >= 0
            if m.any():
                bi = torch.nonzero(m)[:, 0]
                xq[bi, s[bi]] = fq[bi, j]
                xp[bi, s[bi]] = fp[bi, j]
    return (xq.to(cfg.dtype), xp.to(cfg.dtype), parent.to(torch.int32).contiguous(),
            token.contiguous(), score.contiguous())


def tree_inputs(cfg: Config, seed=None, device="cpu", **kw):
    if cfg.kind == "tree_static":
        return static_tree_inputs(cfg, seed, device, **{k: v for k, v in kw.items() if k in ("B", "V")})
    return dynamic_tree_inputs(cfg, seed, device, **kw)


def kv_cache(L, B, S, H, D, device="cpu", seed=0, dtype=torch.bfloat16):
    """Random KV cache [L][2][B][S][H][D] of `dtype` (random bytes)."""
    g = _gen(seed + 17, device)
    esize = torch.tensor([], dtype=dtype).element_size()
    raw = torch.randint(0, 256, (L, 2, B, S, H, D * esize), generator=g, device=device,
                        dtype=torch.uint8)
    return raw.view(dtype)


def level_tree_parents(B, T, depth, seed=0, device="cpu"):
    """Random draft trees shaped like the dynamic tree: T slots (root included)
    numbered level by level over `depth` levels of near-equal size; the parent
    of each node is drawn uniformly from the level above.  int32 [B][T]."""
    g = _gen(seed + 29, "cpu")
    n = T - 1
    sizes = [n // depth + (1 if lv < n % depth else 0) for lv in range(depth)] if depth else []
    parent = torch.full((B, T), -1, dtype=torch.int32)
    prev_lo, prev_hi, nxt = 0, 1, 1
    for sz in sizes:
        if sz == 0:
            break
        parent[:, nxt:nxt + sz] = torch.randint(prev_lo, prev_hi, (B, sz), generator=g,
                                                dtype=torch.int32)
        prev_lo, prev_hi, nxt = nxt, nxt + sz, nxt + sz
    return parent.to(device)


BF16_NAN = 0x7FC0


def attention_inputs(B, T, Hq, Hkv, D, S, base, seed=0, device="cpu", sigma=1.0,
                     poison_tail=True):
    """Tree-attention inputs: queries q [B][T][Hq][D] and one layer of the
    cache kv [2][B][S][Hkv][D] (K then V), bf16, iid N(0, sigma^2).  `base`
    (int or [B]) is each sequence's committed length; tree node n's K/V row is
    slot base + n.  With poison_tail the slots from base + T on hold NaN, which
    no output may depend on.  Returns (q, kv, base int32 [B])."""
    g = _gen(seed + 31, device)
    if isinstance(base, int):
        base = [base] * B
    base_t = torch.tensor(base, dtype=torch.int32)
    q = (torch.randn((B, T, Hq, D), generator=g, device=device) * sigma).to(torch.bfloat16)
    kv = (torch.randn((2, B, S, Hkv, D), generator=g, device=device) * sigma).to(torch.bfloat16)
    if poison_tail:
        nan = torch.tensor(BF16_NAN, dtype=torch.int16).view(torch.bfloat16).item()
        for b, bs in enumerate(base):
            if 0 <= bs and bs + T < S:
                kv[:, b, bs + T:] = nan
    return q, kv, base_t.to(device)
