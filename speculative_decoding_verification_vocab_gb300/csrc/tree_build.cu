// tree_build.cu -- the EAGLE-2 dynamic draft tree on sm_103a: per-row top-K
// expansion with path-product scores, per-level frontier selection, and the
// final pruning to the node budget with level-by-level numbering.
//
// Page: "投机解码发展" (blog), section 5 (三代之间的变化): the tree grows where
// the draft is confident; a node's score is the product of the draft
// probabilities along its path; the best-scored nodes are expanded and the
// tree is pruned to a budget.
#include "common.cuh"

namespace sv {
namespace {

constexpr int kExThreads = 256;
constexpr int kExWarps = kExThreads / 32;
constexpr int kExUnroll = 8;
constexpr int kMaxK = 16;
constexpr int kMaxCand = 4096;
constexpr int kSelWarps = 4;

// ---------------------------------------------------------------------------
// expand: one CTA per frontier row.  Each thread scans its 16-byte words in
// index order keeping (a) online softmax statistics in the log2 domain and
// (b) its own top-K list in shared memory (value descending, index
// ascending); a word whose packed maximum does not beat the thread's K-th
// value is skipped.  The CTA merges the lists with K rounds of a block-wide
// arg max and writes the K tokens and their child scores.
struct ExStat {
  float mx, mk, s;  // raw max, fl(mx * k), sum exp2(fma(x, k, -mk))
  uint32_t flags;   // 1: NaN or +inf seen, 2: a logit above -inf seen
};

__device__ __forceinline__ void ex_stat(ExStat &st, float x, float k) {
  if (x > st.mx) {
    const float nk = x * k;
    st.s = (st.mx == -INFINITY) ? 0.0f : st.s * ex2_approx(st.mk - nk);
    st.mx = x;
    st.mk = nk;
  }
  st.s += ex2_approx(fmaf(x, k, -(st.mx == -INFINITY ? 0.0f : st.mk)));
  if (x != x || x == INFINITY) st.flags |= 1u;
  if (x > -INFINITY) st.flags |= 2u;
}

// the thread's list: val/idx[j][tid], j < n, sorted (value desc, index asc);
// elements arrive in increasing index, so an equal value goes after
struct TopK {
  float (*val)[kExThreads];
  int (*idx)[kExThreads];
  int n, K;
  float thr;  // value of the K-th entry once full, else -inf
};

__device__ __forceinline__ void topk_offer(TopK &t, float x, int v) {
  const int tid = threadIdx.x;
  if (!(t.n < t.K ? x == x : x > t.thr)) return;
  int j = t.n < t.K ? t.n : t.K - 1;  // the slot freed (or the last one)
  while (j > 0 && t.val[j - 1][tid] < x) {
    t.val[j][tid] = t.val[j - 1][tid];
    t.idx[j][tid] = t.idx[j - 1][tid];
    --j;
  }
  t.val[j][tid] = x;
  t.idx[j][tid] = v;
  if (t.n < t.K) ++t.n;
  t.thr = t.n == t.K ? t.val[t.K - 1][tid] : -INFINITY;
}

template <typename E>
__device__ __forceinline__ void ex_word(ExStat &st, TopK &t, uint4 w, int v, float k);
template <>
__device__ __forceinline__ void ex_word<uint16_t>(ExStat &st, TopK &t, uint4 w, int v, float k) {
  const uint32_t q[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int j = 0; j < 8; ++j) ex_stat(st, (j & 1) ? bf16_hi(q[j >> 1]) : bf16_lo(q[j >> 1]), k);
  const uint32_t m = bf2_max(bf2_max(w.x, w.y), bf2_max(w.z, w.w));
  if (t.n < t.K || fmaxf(bf16_lo(m), bf16_hi(m)) > t.thr)
#pragma unroll
    for (int j = 0; j < 8; ++j)
      topk_offer(t, (j & 1) ? bf16_hi(q[j >> 1]) : bf16_lo(q[j >> 1]), v + j);
}
template <>
__device__ __forceinline__ void ex_word<float>(ExStat &st, TopK &t, uint4 w, int v, float k) {
  const float x[4] = {__uint_as_float(w.x), __uint_as_float(w.y), __uint_as_float(w.z),
                      __uint_as_float(w.w)};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    ex_stat(st, x[j], k);
    topk_offer(t, x[j], v + j);
  }
}

template <typename E>
__global__ void __launch_bounds__(kExThreads, 3)
tree_expand_kernel(const E *__restrict__ dlog, int V, float k, int greedy,
                   const float *__restrict__ fscore, int K, int32_t *__restrict__ out_tok,
                   float *__restrict__ out_score) {
  grid_dep_sync();
  const size_t rowi = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const E *row = dlog + rowi * (size_t)V;
  __shared__ float s_val[kMaxK][kExThreads];
  __shared__ int s_idx[kMaxK][kExThreads];
  TopK t{s_val, s_idx, 0, K, -INFINITY};
  ExStat st{-INFINITY, 0.0f, 0.0f, 0u};
  const uintptr_t pb = (uintptr_t)row, pe = (uintptr_t)(row + V);
  uintptr_t ab = (pb + 15) & ~(uintptr_t)15, ae = pe & ~(uintptr_t)15;
  if (ab > ae) ab = ae = pe;
  const int nhead = (int)((ab - pb) / sizeof(E));
  constexpr int kPer = 16 / (int)sizeof(E);
  const uint4 *body = (const uint4 *)ab;
  const int nv = (int)((ae - ab) / 16);
  // head elements first (lowest indices), then the body, then the tail
  if (tid == 0)
    for (int j = 0; j < nhead; ++j) {
      const float x = load_elem<E>(row + j);
      ex_stat(st, x, k);
      topk_offer(t, x, j);
    }
  int i = tid;
  for (; i + (kExUnroll - 1) * kExThreads < nv; i += kExUnroll * kExThreads) {
    uint4 buf[kExUnroll];
#pragma unroll
    for (int j = 0; j < kExUnroll; ++j) buf[j] = ld_stream_v4(body + i + j * kExThreads);
#pragma unroll
    for (int j = 0; j < kExUnroll; ++j)
      ex_word<E>(st, t, buf[j], nhead + (i + j * kExThreads) * kPer, k);
  }
  for (; i < nv; i += kExThreads) ex_word<E>(st, t, ld_stream_v4(body + i), nhead + i * kPer, k);
  if (tid == kExThreads - 1)
    for (int v = nhead + nv * kPer; v < V; ++v) {
      const float x = load_elem<E>(row + v);
      ex_stat(st, x, k);
      topk_offer(t, x, v);
    }
  // statistics: max of references, one rescale per thread, sums
  __shared__ float s_red[3][kExWarps];
  __shared__ uint32_t s_flags[kExWarps];
  {
    float a = (st.mx == -INFINITY) ? -INFINITY : st.mk, M = a, mx = st.mx;
    uint32_t fl = st.flags;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      fl |= __shfl_xor_sync(0xffffffffu, fl, o);
    }
    if (lane == 0) {
      s_red[0][warp] = M;
      s_red[1][warp] = mx;
      s_flags[warp] = fl;
    }
    __syncthreads();
    float MM = -INFINITY;
    uint32_t FF = 0u;
    for (int w = 0; w < kExWarps; ++w) {
      MM = fmaxf(MM, s_red[0][w]);
      FF |= s_flags[w];
    }
    float s = (MM == -INFINITY || a == -INFINITY) ? 0.0f : st.s * ex2_approx(a - MM);
#pragma unroll
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    __syncthreads();
    if (lane == 0) s_red[2][warp] = s;
    __syncthreads();
    st.mk = MM;
    st.flags = FF;
    st.s = 0.0f;
    for (int w = 0; w < kExWarps; ++w) st.s += s_red[2][w];
    st.mx = 0.0f;
    for (int w = 0; w < kExWarps; ++w) st.mx = fmaxf(st.mx, s_red[1][w]);
  }
  // a faulty row, or a frontier entry with a NaN score (no node), proposes nothing
  const bool bad = (st.flags & 1u) || !(st.flags & 2u) || fscore[rowi] != fscore[rowi];
  // K rounds of a block-wide arg max over the heads of the thread lists
  __shared__ float s_hv[kExWarps];
  __shared__ int s_hi[kExWarps];
  int head = 0;
  for (int r = 0; r < K; ++r) {
    float hv = head < t.n ? s_val[head][tid] : -INFINITY;
    int hi = head < t.n ? s_idx[head][tid] : 0x7fffffff;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, hv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, hi, o);
      if (ov > hv || (ov == hv && oi < hi)) {
        hv = ov;
        hi = oi;
      }
    }
    if (lane == 0) {
      s_hv[warp] = hv;
      s_hi[warp] = hi;
    }
    __syncthreads();
    float bv = s_hv[0];
    int bi = s_hi[0];
    for (int w = 1; w < kExWarps; ++w)
      if (s_hv[w] > bv || (s_hv[w] == bv && s_hi[w] < bi)) {
        bv = s_hv[w];
        bi = s_hi[w];
      }
    __syncthreads();
    if (head < t.n && s_idx[head][tid] == bi) ++head;  // indices are unique
    if (tid == 0) {
      const size_t o = rowi * (size_t)K + r;
      if (bad || bi == 0x7fffffff) {
        out_tok[o] = -1;
        out_score[o] = -INFINITY;
      } else {
        float p;
        if (greedy)
          p = (r == 0) ? 1.0f : 0.0f;
        else
          p = ex2_approx(fmaf(bv, k, -st.mk)) / st.s;
        out_tok[o] = bi;
        out_score[o] = fscore[rowi] * p;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// select: one warp per sequence, K rounds of a warp arg max (score
// descending, index ascending) over the not-yet-taken candidates with a
// token; a shared-memory bitmap marks the taken ones.
__global__ void __launch_bounds__(kSelWarps * 32)
tree_select_kernel(const float *__restrict__ score, const int32_t *__restrict__ token, int B,
                   int C, int K, int32_t *__restrict__ out) {
  grid_dep_sync();
  const int wi = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * kSelWarps + wi;
  __shared__ uint32_t taken[kSelWarps][kMaxCand / 32];
  for (int j = lane; j < (C + 31) / 32; j += 32) taken[wi][j] = 0u;
  __syncwarp();
  if (b >= B) return;
  const float *s = score + (size_t)b * C;
  const int32_t *tk = token + (size_t)b * C;
  for (int r = 0; r < K; ++r) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int c = lane; c < C; c += 32) {
      if ((taken[wi][c >> 5] >> (c & 31)) & 1u) continue;
      if (tk[c] < 0) continue;
      const float v = s[c];
      if (bi == 0x7fffffff || v > bv) {  // lane-local candidates in index order
        bv = v;
        bi = c;
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (oi != 0x7fffffff && (bi == 0x7fffffff || ov > bv || (ov == bv && oi < bi))) {
        bv = ov;
        bi = oi;
      }
    }
    if (lane == 0) {
      out[(size_t)b * K + r] = bi == 0x7fffffff ? -1 : bi;
      if (bi != 0x7fffffff) taken[wi][bi >> 5] |= 1u << (bi & 31);
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------------------
// finalize: one CTA per sequence.  T rounds of a block-wide pick in keep
// order (score descending, level ascending, index ascending) build the kept
// set; each kept node's slot is its rank in (level ascending, score
// descending, index ascending); parents map through the candidate -> slot
// table.
__device__ __forceinline__ bool keep_before(float sa, int la, int a, float sb, int lb, int b) {
  if (sa != sb) return sa > sb;
  if (la != lb) return la < lb;
  return a < b;
}

__global__ void __launch_bounds__(kExThreads)
tree_finalize_kernel(const int32_t *__restrict__ cparent, const int32_t *__restrict__ ctoken,
                     const float *__restrict__ cscore, const int32_t *__restrict__ clevel, int C,
                     int Tn, int32_t *__restrict__ parent, int32_t *__restrict__ token,
                     float *__restrict__ score) {
  grid_dep_sync();
  const int b = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int32_t *cp = cparent + (size_t)b * C, *ct = ctoken + (size_t)b * C;
  const int32_t *cl = clevel + (size_t)b * C;
  const float *cs = cscore + (size_t)b * C;
  __shared__ int slot_of[kMaxCand];
  __shared__ int keep[SV_MAX_TREE_NODES];
  __shared__ float w_v[kExWarps];
  __shared__ int w_l[kExWarps], w_i[kExWarps];
  __shared__ int s_n;
  for (int c = tid; c < C; c += kExThreads) slot_of[c] = -1;  // -1: not kept (yet)
  __syncthreads();
  int n = 0;
  for (; n < Tn; ++n) {
    float bv = 0.0f;
    int bl = 0, bi = 0x7fffffff;
    for (int c = tid; c < C; c += kExThreads) {
      if (slot_of[c] != -1) continue;
      if (c != 0 && ct[c] < 0) continue;
      const float v = cs[c];
      const int l = cl[c];
      if (bi == 0x7fffffff || keep_before(v, l, c, bv, bl, bi)) {
        bv = v;
        bl = l;
        bi = c;
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int ol = __shfl_xor_sync(0xffffffffu, bl, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (oi != 0x7fffffff && (bi == 0x7fffffff || keep_before(ov, ol, oi, bv, bl, bi))) {
        bv = ov;
        bl = ol;
        bi = oi;
      }
    }
    if (lane == 0) {
      w_v[warp] = bv;
      w_l[warp] = bl;
      w_i[warp] = bi;
    }
    __syncthreads();
    if (tid == 0) {
      float v = w_v[0];
      int l = w_l[0], i = w_i[0];
      for (int w = 1; w < kExWarps; ++w)
        if (w_i[w] != 0x7fffffff && (i == 0x7fffffff || keep_before(w_v[w], w_l[w], w_i[w], v, l, i))) {
          v = w_v[w];
          l = w_l[w];
          i = w_i[w];
        }
      s_n = i;
      if (i != 0x7fffffff) {
        keep[n] = i;
        slot_of[i] = -3;  // kept; its slot is set below
      }
    }
    __syncthreads();
    if (s_n == 0x7fffffff) break;
  }
  // slots: rank in (level asc, score desc, index asc) among the kept
  for (int i = tid; i < n; i += kExThreads) {
    const int c = keep[i];
    const int l = cl[c];
    const float v = cs[c];
    int rank = 0;
    for (int j = 0; j < n; ++j) {
      const int d = keep[j];
      const int ld = cl[d];
      const float vd = cs[d];
      rank += (ld < l) || (ld == l && (vd > v || (vd == v && d < c)));
    }
    slot_of[c] = rank;
  }
  __syncthreads();
  for (int i = tid; i < n; i += kExThreads) {
    const int c = keep[i], sl = slot_of[c];
    const int pc = cp[c];
    parent[(size_t)b * Tn + sl] = pc < 0 ? -1 : (slot_of[pc] >= 0 ? slot_of[pc] : -2);
    token[(size_t)b * Tn + sl] = ct[c];
    score[(size_t)b * Tn + sl] = cs[c];
  }
  for (int i = n + tid; i < Tn; i += kExThreads) {
    parent[(size_t)b * Tn + i] = -2;
    token[(size_t)b * Tn + i] = -1;
    score[(size_t)b * Tn + i] = 0.0f;
  }
}

constexpr float kLog2eB = 1.4426950408889634f;

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" sv_status sv_tree_expand(const void *dlogits, sv_dtype dt, int B, int F, int V,
                                    float temperature, const float *frontier_score, int K,
                                    int32_t *out_token, float *out_score, void *stream) {
  if (B < 0 || F < 1 || V < 1) return set_error(SV_ERR_INVALID_ARG, "need B >= 0, F >= 1, V >= 1");
  if (K < 1 || K > V) return set_error(SV_ERR_INVALID_ARG, "need 1 <= K <= V");
  if (K > kMaxK) return set_error(SV_ERR_UNSUPPORTED, "K > %d", kMaxK);
  if (V > SV_MAX_VOCAB) return set_error(SV_ERR_UNSUPPORTED, "V > %d", SV_MAX_VOCAB);
  if (dt != SV_F32 && dt != SV_BF16) return set_error(SV_ERR_INVALID_ARG, "unknown dtype %d", (int)dt);
  if (!(temperature >= 0.0f) || !isfinite(temperature))
    return set_error(SV_ERR_INVALID_ARG, "temperature must be finite and >= 0");
  if ((long long)B * F > 0x7fffffffLL) return set_error(SV_ERR_UNSUPPORTED, "B * F too large");
  if (B == 0) return SV_OK;
  if (!dlogits || !frontier_score || !out_token || !out_score)
    return set_error(SV_ERR_INVALID_ARG, "null pointer argument");
  if ((uintptr_t)dlogits % (dt == SV_F32 ? 4 : 2)) return set_error(SV_ERR_INVALID_ARG, "dlogits misaligned");
  sv_status s;
  if ((s = map_arg(dlogits, "dlogits")) != SV_OK ||
      (s = map_arg(frontier_score, "frontier_score")) != SV_OK ||
      (s = map_arg(out_token, "out_token")) != SV_OK || (s = map_arg(out_score, "out_score")) != SV_OK)
    return s;
  const int greedy = temperature == 0.0f;
  const float k = greedy ? kLog2eB : kLog2eB / temperature;
  cudaStream_t st = (cudaStream_t)stream;
  LaunchScope ls("tree_expand", st);
  const dim3 grid((unsigned)(B * F));
  return check_launch("tree_expand",
                      dt == SV_BF16
                          ? launch_pdl(tree_expand_kernel<uint16_t>, grid, dim3(kExThreads), 0, st,
                                       (const uint16_t *)dlogits, V, k, greedy, frontier_score, K,
                                       out_token, out_score)
                          : launch_pdl(tree_expand_kernel<float>, grid, dim3(kExThreads), 0, st,
                                       (const float *)dlogits, V, k, greedy, frontier_score, K,
                                       out_token, out_score));
}

extern "C" sv_status sv_tree_select(const float *cand_score, const int32_t *cand_token, int B,
                                    int C, int K, int32_t *out_index, void *stream) {
  if (B < 0 || C < 1 || K < 1) return set_error(SV_ERR_INVALID_ARG, "need B >= 0, C >= 1, K >= 1");
  if (C > kMaxCand) return set_error(SV_ERR_UNSUPPORTED, "C > %d", kMaxCand);
  if (B == 0) return SV_OK;
  if (!cand_score || !cand_token || !out_index) return set_error(SV_ERR_INVALID_ARG, "null pointer argument");
  sv_status s;
  if ((s = map_arg(cand_score, "cand_score")) != SV_OK ||
      (s = map_arg(cand_token, "cand_token")) != SV_OK || (s = map_arg(out_index, "out_index")) != SV_OK)
    return s;
  cudaStream_t st = (cudaStream_t)stream;
  LaunchScope ls("tree_select", st);
  return check_launch("tree_select",
                      launch_pdl(tree_select_kernel, dim3((B + kSelWarps - 1) / kSelWarps),
                                 dim3(kSelWarps * 32), 0, st, cand_score, cand_token, B, C, K,
                                 out_index));
}

extern "C" sv_status sv_tree_finalize(const int32_t *cand_parent, const int32_t *cand_token,
                                      const float *cand_score, const int32_t *cand_level, int B,
                                      int C, int T, int32_t *out_parent, int32_t *out_token,
                                      float *out_score, void *stream) {
  if (B < 0 || C < 1 || T < 1) return set_error(SV_ERR_INVALID_ARG, "need B >= 0, C >= 1, T >= 1");
  if (C > kMaxCand) return set_error(SV_ERR_UNSUPPORTED, "C > %d", kMaxCand);
  if (T > SV_MAX_TREE_NODES) return set_error(SV_ERR_UNSUPPORTED, "T > %d", SV_MAX_TREE_NODES);
  if (B == 0) return SV_OK;
  if (!cand_parent || !cand_token || !cand_score || !cand_level || !out_parent || !out_token ||
      !out_score)
    return set_error(SV_ERR_INVALID_ARG, "null pointer argument");
  sv_status s;
  if ((s = map_arg(cand_parent, "cand_parent")) != SV_OK ||
      (s = map_arg(cand_token, "cand_token")) != SV_OK ||
      (s = map_arg(cand_score, "cand_score")) != SV_OK ||
      (s = map_arg(cand_level, "cand_level")) != SV_OK ||
      (s = map_arg(out_parent, "out_parent")) != SV_OK ||
      (s = map_arg(out_token, "out_token")) != SV_OK || (s = map_arg(out_score, "out_score")) != SV_OK)
    return s;
  cudaStream_t st = (cudaStream_t)stream;
  LaunchScope ls("tree_finalize", st);
  return check_launch("tree_finalize",
                      launch_pdl(tree_finalize_kernel, dim3(B), dim3(kExThreads), 0, st,
                                 cand_parent, cand_token, cand_score, cand_level, C, T,
                                 out_parent, out_token, out_score));
}
