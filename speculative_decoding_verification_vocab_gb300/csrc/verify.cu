// verify.cu -- batched verify-and-accept for speculative decoding on sm_103a.
//
// Steps (one stream, no host synchronisation):
//   tree_path    (tree only) best-child walk per sequence
//   row_stats    single-pass online softmax statistics (max, sum of exp) of
//                every logit row the round can touch -- the one step that
//                streams the whole input; HBM-bound
//   decide       one warp per sequence: q(d)/p(d), Philox uniforms, the left-
//                to-right accept walk, outputs, and the sampling task
//   sample_sum   exact fixed-point normaliser of the 1-2 sampled rows
//   sample_chunk fixed-point residual / bonus masses per 2048-token chunk
//   sample_pick  inverse CDF: chunk search, then a warp scan in the chunk
//
// Pages: "Decodificação Especulativa e EAGLE-3" (lesson; "O invariante",
// Passo 1-3) and "投机解码发展" (blog; section 2 steps, section 4 spec_decode /
// eagle_round pseudocode).  p = draft, q = verifier.
#include <math.h>
#include <stdio.h>

#include "common.cuh"

namespace sv {
namespace {

constexpr int kStatsThreads = 512;
constexpr int kDecideWarps = 4;
constexpr int kSampleThreads = 256;
constexpr int kChunk = 2048;          // tokens per fixed-point chunk sum
constexpr int kChunksPerSeg = 8;      // chunks per sampler CTA
constexpr float kLog2e = 1.4426950408889634f;

struct Task {
  int active;  // 1: a correction / bonus token is to be drawn
  int a;       // accept length = output slot of the drawn token
  int vrow;    // absolute verifier row (rows of V elements)
  int drow;    // absolute draft row, -1 for a bonus draw
  float mq, mp;  // raw-logit maxima of those rows
  uint32_t u24;
  int pad;
};

struct Acc {  // exact fixed-point sums of one sampling task
  unsigned long long se_q, se_p;  // sum floor(e * 2^40)
  unsigned long long sw, sq;      // sum floor(w * 2^62), sum floor(q * 2^62)
};

struct Layout {
  int maxpos, P, G, seg_len, nchunk, G3;
  size_t partial, task, acc, chunks, path, npos, tok, tstat, total;
};

Layout plan(int B, int maxpos, int V, bool tree) {
  Layout L;
  L.maxpos = maxpos;
  L.P = 2 * maxpos + 1;
  const long nslots = (long)B * L.P;
  const long target = (long)num_sms() * 16;
  int g = (int)((target + nslots - 1) / (nslots > 0 ? nslots : 1));
  const int gmax = V / 4096 > 1 ? V / 4096 : 1;
  g = g < 1 ? 1 : (g > gmax ? gmax : g);
  int len = (V + g - 1) / g;
  len = (len + 63) / 64 * 64;
  L.seg_len = len;
  L.G = (V + len - 1) / len;
  L.nchunk = (V + kChunk - 1) / kChunk;
  L.G3 = (L.nchunk + kChunksPerSeg - 1) / kChunksPerSeg;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  L.partial = take(sizeof(float2) * (size_t)nslots * L.G);
  L.task = take(sizeof(Task) * (size_t)B);
  L.acc = take(sizeof(Acc) * (size_t)B);
  L.chunks = take(sizeof(ulonglong2) * (size_t)B * L.nchunk);
  if (tree) {
    L.path = take(sizeof(int32_t) * (size_t)B * (maxpos + 1));
    L.npos = take(sizeof(int32_t) * (size_t)B);
    L.tok = take(sizeof(int32_t) * (size_t)B * (maxpos > 0 ? maxpos : 1));
    L.tstat = take(sizeof(uint32_t) * (size_t)B);
  } else {
    L.path = L.npos = L.tok = L.tstat = 0;
  }
  L.total = off + 256;
  return L;
}

// ---------------------------------------------------------------------------
// Shared view of one round: how position i of sequence b maps to rows.
struct Round {
  const void *vlog, *dlog;
  int B, V, maxpos, P;
  int v_rows, d_rows;       // rows per sequence in vlogits / dlogits
  const int32_t *path;      // [B][maxpos+1] nodes, or null: identity (chain)
  const int32_t *npos;      // [B] or null: maxpos for all
  const int32_t *tok;       // [B][tok_stride] token tested at position i
  int tok_stride;
  const uint32_t *tstat;    // [B] tree status or null
  float invT, k;            // 1/T and log2(e)/T
};

__device__ __forceinline__ int round_npos(const Round &r, int b) {
  return r.npos ? r.npos[b] : r.maxpos;
}
__device__ __forceinline__ int round_node(const Round &r, int b, int i) {
  return r.path ? r.path[(size_t)b * (r.maxpos + 1) + i] : i;
}

// ---------------------------------------------------------------------------
// row_stats: work item = (slot, segment).  Slot j of a sequence is the
// verifier row of position j (j <= maxpos) or the draft row of position
// j - maxpos - 1.  Writes (max x, sum exp2((x - max) * k)) of its segment.
template <typename E>
__device__ __forceinline__ void accum8(uint4 v, float &m, float &s0, float &s1, float k);

template <>
__device__ __forceinline__ void accum8<uint16_t>(uint4 v, float &m, float &s0, float &s1,
                                                 float k) {
  const float x0 = bf16_lo(v.x), x1 = bf16_hi(v.x), x2 = bf16_lo(v.y), x3 = bf16_hi(v.y);
  const float x4 = bf16_lo(v.z), x5 = bf16_hi(v.z), x6 = bf16_lo(v.w), x7 = bf16_hi(v.w);
  const float cm = fmaxf(fmaxf(fmaxf(x0, x1), fmaxf(x2, x3)), fmaxf(fmaxf(x4, x5), fmaxf(x6, x7)));
  if (cm > m) {
    const float f = ex2_approx((m - cm) * k);
    s0 *= f;
    s1 *= f;
    m = cm;
  }
  const float mm = (m == -INFINITY) ? 0.0f : m;
  s0 += ex2_approx((x0 - mm) * k) + ex2_approx((x1 - mm) * k);
  s1 += ex2_approx((x2 - mm) * k) + ex2_approx((x3 - mm) * k);
  s0 += ex2_approx((x4 - mm) * k) + ex2_approx((x5 - mm) * k);
  s1 += ex2_approx((x6 - mm) * k) + ex2_approx((x7 - mm) * k);
}

template <>
__device__ __forceinline__ void accum8<float>(uint4 v, float &m, float &s0, float &s1, float k) {
  const float x0 = __uint_as_float(v.x), x1 = __uint_as_float(v.y);
  const float x2 = __uint_as_float(v.z), x3 = __uint_as_float(v.w);
  const float cm = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
  if (cm > m) {
    const float f = ex2_approx((m - cm) * k);
    s0 *= f;
    s1 *= f;
    m = cm;
  }
  const float mm = (m == -INFINITY) ? 0.0f : m;
  s0 += ex2_approx((x0 - mm) * k) + ex2_approx((x1 - mm) * k);
  s1 += ex2_approx((x2 - mm) * k) + ex2_approx((x3 - mm) * k);
}

// One scalar element (ragged head / tail of a segment).  Rescales both
// partial sums when the running max moves.
__device__ __forceinline__ void accum1(float x, float &m, float &s0, float &s1, bool to0,
                                       float k) {
  if (x > m) {
    const float f = ex2_approx((m - x) * k);
    s0 *= f;
    s1 *= f;
    m = x;
  }
  const float mm = (m == -INFINITY) ? 0.0f : m;
  const float e = ex2_approx((x - mm) * k);
  if (to0)
    s0 += e;
  else
    s1 += e;
}

template <typename E>
__global__ void __launch_bounds__(kStatsThreads)
row_stats_kernel(Round r, int G, int seg_len, float2 *__restrict__ partial) {
  const int w = blockIdx.x;
  const int slot = w / G, seg = w - slot * G;
  const int b = slot / r.P, j = slot - b * r.P;
  const int npos = round_npos(r, b);
  const bool is_v = j <= r.maxpos;
  const int i = is_v ? j : j - r.maxpos - 1;
  if (is_v ? (i > npos) : (i >= npos)) return;
  const int node = round_node(r, b, i);
  const E *row = (const E *)(is_v ? r.vlog : r.dlog) +
                 ((size_t)b * (is_v ? r.v_rows : r.d_rows) + node) * (size_t)r.V;
  const int v0 = seg * seg_len;
  const int v1 = min(r.V, v0 + seg_len);
  const float k = r.k;

  float m = -INFINITY, s0 = 0.0f, s1 = 0.0f;
  const uintptr_t pb = (uintptr_t)(row + v0), pe = (uintptr_t)(row + v1);
  uintptr_t ab = (pb + 15) & ~(uintptr_t)15, ae = pe & ~(uintptr_t)15;
  if (ab > ae) ab = ae = pe;
  const int nhead = (int)((ab - pb) / sizeof(E));
  const int ntail = (int)((pe - ae) / sizeof(E));
  const int tid = threadIdx.x;
  if (tid < nhead) accum1(load_elem<E>(row + v0 + tid), m, s0, s1, true, k);
  if (tid < ntail) accum1(load_elem<E>((const E *)ae + tid), m, s0, s1, false, k);
  const uint4 *body = (const uint4 *)ab;
  const long nvec = (long)((ae - ab) / 16);
  long vi = tid;
  for (; vi + 3L * kStatsThreads < nvec; vi += 4L * kStatsThreads) {
    const uint4 a0 = ld_stream_v4(body + vi);
    const uint4 a1 = ld_stream_v4(body + vi + kStatsThreads);
    const uint4 a2 = ld_stream_v4(body + vi + 2 * kStatsThreads);
    const uint4 a3 = ld_stream_v4(body + vi + 3 * kStatsThreads);
    accum8<E>(a0, m, s0, s1, k);
    accum8<E>(a1, m, s0, s1, k);
    accum8<E>(a2, m, s0, s1, k);
    accum8<E>(a3, m, s0, s1, k);
  }
  for (; vi < nvec; vi += kStatsThreads) accum8<E>(ld_stream_v4(body + vi), m, s0, s1, k);
  float s = s0 + s1;

  // warp, then block combine of (m, s)
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    ms_combine(m, s, m2, s2, k);
  }
  __shared__ float sm[kStatsThreads / 32], ss[kStatsThreads / 32];
  const int wid = tid >> 5, lane = tid & 31;
  if (lane == 0) {
    sm[wid] = m;
    ss[wid] = s;
  }
  __syncthreads();
  if (wid == 0) {
    m = lane < kStatsThreads / 32 ? sm[lane] : -INFINITY;
    s = lane < kStatsThreads / 32 ? ss[lane] : 0.0f;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
      ms_combine(m, s, m2, s2, k);
    }
    if (lane == 0) partial[w] = make_float2(m, s);
  }
}

// ---------------------------------------------------------------------------
// decide: one warp per sequence.
struct DecideOut {
  int32_t *tokens;       // [B][maxpos+1]
  int32_t *accept_len;   // [B]
  float *q_prob, *p_prob;  // [B][maxpos] or null
  float *margin;         // [B][maxpos+1] or null
  uint32_t *status;      // [B]
  int32_t *path_out;     // [B][maxpos+1] or null (tree)
};

template <typename E>
__device__ __forceinline__ void merge_slot(const float2 *part, int G, float k, float &m,
                                           float &s) {
  m = -INFINITY;
  s = 0.0f;
  for (int g = 0; g < G; ++g) {
    const float2 v = part[g];
    ms_combine(m, s, v.x, v.y, k);
  }
}

template <typename E>
__global__ void __launch_bounds__(kDecideWarps * 32)
decide_kernel(Round r, int G, const float2 *__restrict__ partial, uint64_t seed,
              uint64_t step, DecideOut o, Task *__restrict__ tasks, Acc *__restrict__ acc) {
  const int b = blockIdx.x * kDecideWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= r.B) return;
  const unsigned FULL = 0xffffffffu;
  const int npos = round_npos(r, b);
  const uint32_t tree_bad = r.tstat ? r.tstat[b] : 0u;
  const float2 *pb = partial + (size_t)b * r.P * G;
  const float k = r.k, invT = r.invT;

  uint32_t bad = 0, pzero_bits = 0, acc_bits = 0;
  // bonus row (verifier row of position npos) is checked by lane 0
  if (lane == 0 && !tree_bad) {
    float m, s;
    merge_slot<E>(pb + (size_t)npos * G, G, k, m, s);
    if (!(s > 0.0f)) bad |= SV_ROW_NAN;
  }
  const int nchunks = (npos + 31) / 32;
  for (int c = 0; c < nchunks && !tree_bad; ++c) {
    const int i = c * 32 + lane;
    if (i >= npos) break;
    float mq, sq, mp, sp;
    merge_slot<E>(pb + (size_t)i * G, G, k, mq, sq);
    merge_slot<E>(pb + (size_t)(r.maxpos + 1 + i) * G, G, k, mp, sp);
    if (!(sq > 0.0f) || !(sp > 0.0f)) bad |= SV_ROW_NAN;
    const int d = r.tok[(size_t)b * r.tok_stride + i];
    if (d < 0 || d >= r.V) {
      bad |= SV_ROW_BAD_TOKEN;
      continue;
    }
    const int node = round_node(r, b, i);
    const E *vrow = (const E *)r.vlog + ((size_t)b * r.v_rows + node) * (size_t)r.V;
    const E *drow = (const E *)r.dlog + ((size_t)b * r.d_rows + node) * (size_t)r.V;
    const float xq = load_elem<E>(vrow + d), xp = load_elem<E>(drow + d);
    const float lq = (xq - mq) * invT, lp = (xp - mp) * invT;  // log q(d) + log sq, ...
    const float qd = expf(lq) / sq, pd = expf(lp) / sp;
    const bool p_zero = (xp == -INFINITY);
    float ratio;
    if (p_zero)
      ratio = INFINITY;
    else if (xq == -INFINITY)
      ratio = 0.0f;
    else
      ratio = exp2f((lq - lp) * kLog2e + (log2f(sp) - log2f(sq)));
    const float rc = fminf(ratio, 1.0f);
    const uint32_t u24 = uniform_u24(seed, step, (uint32_t)b, (uint32_t)i, kDrawAccept);
    const float u = (float)u24 * 0x1p-24f;
    const bool accept = p_zero || (u < rc);
    if (accept) acc_bits |= 1u << c;
    if (p_zero) pzero_bits |= 1u << c;
    if (o.q_prob) o.q_prob[(size_t)b * r.maxpos + i] = qd;
    if (o.p_prob) o.p_prob[(size_t)b * r.maxpos + i] = pd;
    if (o.margin) o.margin[(size_t)b * (r.maxpos + 1) + i] = rc - u;
  }
  bad = __reduce_or_sync(FULL, bad);
  if (tree_bad) bad = SV_ROW_BAD_TREE;

  // first rejection
  int a = npos;
  uint32_t pz = 0;
  for (int c = 0; c < nchunks; ++c) {
    const int i = c * 32 + lane;
    const unsigned rej = __ballot_sync(FULL, i < npos && !((acc_bits >> c) & 1u));
    const unsigned pzc = __ballot_sync(FULL, i < npos && ((pzero_bits >> c) & 1u));
    if (rej) {
      a = c * 32 + __ffs(rej) - 1;
      const unsigned below = (a - c * 32) >= 32 ? FULL : ((1u << (a - c * 32)) - 1u);
      pz |= pzc & below;
      break;
    }
    pz |= pzc;
  }
  if (bad) a = 0;

  // outputs
  const int W = r.maxpos + 1;
  for (int i = lane; i < W; i += 32) {
    int32_t t = -1;
    if (!bad && i < a) t = r.tok[(size_t)b * r.tok_stride + i];
    o.tokens[(size_t)b * W + i] = t;
    if (o.path_out) o.path_out[(size_t)b * W + i] = (i == 0) ? 0 : ((!bad && i <= a) ? round_node(r, b, i) : -1);
    if (i >= npos || bad) {
      if (i < r.maxpos) {
        if (o.q_prob) o.q_prob[(size_t)b * r.maxpos + i] = NAN;
        if (o.p_prob) o.p_prob[(size_t)b * r.maxpos + i] = NAN;
      }
      if (o.margin) o.margin[(size_t)b * W + i] = NAN;
    }
  }
  if (lane == 0) {
    o.accept_len[b] = a;
    o.status[b] = bad ? bad : (pz ? SV_ROW_P_ZERO : 0u);
    Task t;
    t.active = bad ? 0 : 1;
    t.a = a;
    t.pad = 0;
    const int vi = a < npos ? a : npos;
    t.vrow = b * r.v_rows + round_node(r, b, vi);
    t.drow = a < npos ? b * r.d_rows + round_node(r, b, a) : -1;
    float m, s;
    merge_slot<E>(pb + (size_t)vi * G, G, k, m, s);
    t.mq = m;
    t.mp = 0.0f;
    if (a < npos) {
      merge_slot<E>(pb + (size_t)(r.maxpos + 1 + a) * G, G, k, m, s);
      t.mp = m;
    }
    t.u24 = uniform_u24(seed, step, (uint32_t)b, (uint32_t)a, kDrawSample);
    tasks[b] = t;
    acc[b] = Acc{0ull, 0ull, 0ull, 0ull};
  }
}

// ---------------------------------------------------------------------------
// The sampling arithmetic (fixed sequence of IEEE fp32 operations + exact
// 64-bit fixed point):
//   z = fl(x * invT); e = exp32_repro(fl(z - max z)); S_e = sum floor(e 2^40)
//   inv_s = fl32(2^40 / fl64(S_e)); q = fl(e * inv_s)
//   w = max(0, fl(q - p)) (residual) or q (bonus); W = floor(w 2^62)
//   t = floor(u24 * sum W / 2^24); token = min{k : sum_{v<=k} W_v > t}
template <typename E>
__device__ __forceinline__ float e_of(const E *row, int v, float invT, float mz) {
  return exp32_repro(__fsub_rn(__fmul_rn(load_elem<E>(row + v), invT), mz));
}

__device__ __forceinline__ float inv_sum(unsigned long long se) {
  return __double2float_rn(__ddiv_rn(0x1p40, __ull2double_rn(se)));
}

__device__ __forceinline__ unsigned long long fix40(float e) {
  return __float2ull_rz(__fmul_rn(e, 0x1p40f));
}
__device__ __forceinline__ unsigned long long fix62(float w) {
  return __float2ull_rz(__fmul_rn(w, 0x1p62f));
}

template <typename T>
__device__ __forceinline__ T block_sum(T v, T *red) {
  v = (T)warp_sum_u64((unsigned long long)v);
  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  T tot = 0;
  if (threadIdx.x == 0)
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) tot += red[i];
  return tot;  // valid on thread 0
}

template <typename E>
__global__ void __launch_bounds__(kSampleThreads)
sample_sum_kernel(Round r, const Task *__restrict__ tasks, Acc *__restrict__ acc) {
  const int b = blockIdx.x, g = blockIdx.y;
  const Task t = tasks[b];
  if (!t.active) return;
  const int v0 = g * kChunk * kChunksPerSeg;
  const int v1 = min(r.V, v0 + kChunk * kChunksPerSeg);
  const E *rq = (const E *)r.vlog + (size_t)t.vrow * r.V;
  const float mzq = __fmul_rn(t.mq, r.invT);
  unsigned long long sq = 0, sp = 0;
  for (int v = v0 + threadIdx.x; v < v1; v += kSampleThreads) sq += fix40(e_of(rq, v, r.invT, mzq));
  if (t.drow >= 0) {
    const E *rp = (const E *)r.dlog + (size_t)t.drow * r.V;
    const float mzp = __fmul_rn(t.mp, r.invT);
    for (int v = v0 + threadIdx.x; v < v1; v += kSampleThreads) sp += fix40(e_of(rp, v, r.invT, mzp));
  }
  __shared__ unsigned long long red[kSampleThreads / 32];
  sq = block_sum(sq, red);
  if (threadIdx.x == 0) atomicAdd(&acc[b].se_q, sq);
  if (t.drow >= 0) {
    sp = block_sum(sp, red);
    if (threadIdx.x == 0) atomicAdd(&acc[b].se_p, sp);
  }
}

template <typename E>
__device__ __forceinline__ void wmass(const Round &r, const E *rq, const E *rp, int v, float mzq,
                                      float iq, float mzp, float ip, unsigned long long &W,
                                      unsigned long long &Wq) {
  const float q = __fmul_rn(e_of(rq, v, r.invT, mzq), iq);
  Wq = fix62(q);
  if (rp) {
    const float p = __fmul_rn(e_of(rp, v, r.invT, mzp), ip);
    const float d = __fsub_rn(q, p);
    W = fix62(d > 0.0f ? d : 0.0f);
  } else {
    W = Wq;
  }
}

template <typename E>
__global__ void __launch_bounds__(kSampleThreads)
sample_chunk_kernel(Round r, const Task *__restrict__ tasks, Acc *__restrict__ acc,
                    ulonglong2 *__restrict__ chunks, int nchunk) {
  const int b = blockIdx.x, g = blockIdx.y;
  const Task t = tasks[b];
  if (!t.active) return;
  const E *rq = (const E *)r.vlog + (size_t)t.vrow * r.V;
  const E *rp = t.drow >= 0 ? (const E *)r.dlog + (size_t)t.drow * r.V : nullptr;
  const float mzq = __fmul_rn(t.mq, r.invT), iq = inv_sum(acc[b].se_q);
  const float mzp = rp ? __fmul_rn(t.mp, r.invT) : 0.0f;
  const float ip = rp ? inv_sum(acc[b].se_p) : 0.0f;
  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned long long tw = 0, tq = 0;
  for (int c = g * kChunksPerSeg + wid; c < min(nchunk, (g + 1) * kChunksPerSeg);
       c += kSampleThreads / 32) {
    const int v0 = c * kChunk, v1 = min(r.V, v0 + kChunk);
    unsigned long long sw = 0, sq = 0;
    for (int v = v0 + lane; v < v1; v += 32) {
      unsigned long long W, Wq;
      wmass(r, rq, rp, v, mzq, iq, mzp, ip, W, Wq);
      sw += W;
      sq += Wq;
    }
    sw = warp_sum_u64(sw);
    sq = warp_sum_u64(sq);
    if (lane == 0) {
      chunks[(size_t)b * nchunk + c] = make_ulonglong2(sw, sq);
      tw += sw;
      tq += sq;
    }
  }
  if (lane == 0) {
    atomicAdd(&acc[b].sw, tw);
    atomicAdd(&acc[b].sq, tq);
  }
}

__device__ __forceinline__ unsigned long long warp_incl_scan_u64(unsigned long long v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

template <typename E>
__global__ void __launch_bounds__(32)
sample_pick_kernel(Round r, const Task *__restrict__ tasks, const Acc *__restrict__ acc,
                   const ulonglong2 *__restrict__ chunks, int nchunk, DecideOut o) {
  const int b = blockIdx.x, lane = threadIdx.x;
  const Task t = tasks[b];
  if (!t.active) return;
  const Acc A = acc[b];
  const bool resid = t.drow >= 0;
  bool use_q = !resid;
  unsigned long long S = resid ? A.sw : A.sq;
  bool rz = false;
  if (resid && S == 0ull) {
    S = A.sq;
    use_q = true;
    rz = true;
  }
  const unsigned long long hi = __umul64hi((unsigned long long)t.u24, S);
  const unsigned long long lo = (unsigned long long)t.u24 * S;
  const unsigned long long thr = (hi << 40) | (lo >> 24);

  // chunk search
  unsigned long long base = 0;
  int cfound = -1;
  for (int c0 = 0; c0 < nchunk && cfound < 0; c0 += 32) {
    const int c = c0 + lane;
    unsigned long long v = 0;
    if (c < nchunk) {
      const ulonglong2 cv = chunks[(size_t)b * nchunk + c];
      v = use_q ? cv.y : cv.x;
    }
    const unsigned long long inc = warp_incl_scan_u64(v) + base;
    const unsigned hit = __ballot_sync(0xffffffffu, c < nchunk && inc > thr);
    if (hit) {
      const int l = __ffs(hit) - 1;
      cfound = c0 + l;
      base = __shfl_sync(0xffffffffu, inc - v, l);
    } else {
      base = __shfl_sync(0xffffffffu, inc, 31);
    }
  }
  if (cfound < 0) cfound = nchunk - 1;  // unreachable: thr < S
  // token search inside the chunk
  const E *rq = (const E *)r.vlog + (size_t)t.vrow * r.V;
  const E *rp = resid ? (const E *)r.dlog + (size_t)t.drow * r.V : nullptr;
  const float mzq = __fmul_rn(t.mq, r.invT), iq = inv_sum(A.se_q);
  const float mzp = rp ? __fmul_rn(t.mp, r.invT) : 0.0f;
  const float ip = rp ? inv_sum(A.se_p) : 0.0f;
  const int v0 = cfound * kChunk, v1 = min(r.V, v0 + kChunk);
  int token = -1;
  unsigned long long below = 0, above = 0;
  for (int vb = v0; vb < v1; vb += 32) {
    const int v = vb + lane;
    unsigned long long W = 0, Wq = 0;
    if (v < v1) wmass(r, rq, rp, v, mzq, iq, mzp, ip, W, Wq);
    const unsigned long long w = use_q ? Wq : W;
    const unsigned long long inc = warp_incl_scan_u64(w) + base;
    const unsigned hit = __ballot_sync(0xffffffffu, v < v1 && inc > thr);
    if (hit) {
      const int l = __ffs(hit) - 1;
      token = vb + l;
      const unsigned long long c_hi = __shfl_sync(0xffffffffu, inc, l);
      const unsigned long long c_lo = __shfl_sync(0xffffffffu, inc - w, l);
      below = thr - c_lo;
      above = c_hi - 1ull - thr;
      break;
    }
    base = __shfl_sync(0xffffffffu, inc, 31);
  }
  if (lane == 0) {
    const int W = r.maxpos + 1;
    o.tokens[(size_t)b * W + t.a] = token;
    if (o.margin)
      o.margin[(size_t)b * W + r.maxpos] =
          (float)((double)(below < above ? below : above) / (double)S);
    if (rz) o.status[b] |= SV_ROW_RESID_ZERO;
  }
}

// ---------------------------------------------------------------------------
// tree_path: one warp per sequence.  Validates the tree, walks best children
// (highest score; ties to the lower slot) at most max_depth steps.
__global__ void __launch_bounds__(32)
tree_path_kernel(const int32_t *__restrict__ parent, const int32_t *__restrict__ token,
                 const float *__restrict__ score, int B, int T, int max_depth,
                 int32_t *__restrict__ path, int32_t *__restrict__ npos,
                 int32_t *__restrict__ tok, int tok_stride, uint32_t *__restrict__ tstat) {
  const int b = blockIdx.x, lane = threadIdx.x;
  const int32_t *pa = parent + (size_t)b * T;
  const float *sc = score + (size_t)b * T;
  bool ok = true;
  for (int c = lane; c < T; c += 32) {
    const int p = pa[c];
    if (c == 0) {
      ok &= (p == -1);
    } else if (p != -2) {
      ok &= (p >= 0 && p < c);
      if (p >= 0 && p < c) ok &= (pa[p] != -2);
      ok &= !isnan(sc[c]);
    }
  }
  const bool bad = __any_sync(0xffffffffu, !ok);
  int32_t *pth = path + (size_t)b * (max_depth + 1);
  if (bad) {
    if (lane == 0) {
      pth[0] = 0;
      npos[b] = 0;
      tstat[b] = SV_ROW_BAD_TREE;
    }
    return;
  }
  int cur = 0, D = 0;
  if (lane == 0) pth[0] = 0;
  while (D < max_depth) {
    bool have = false;
    float bs = 0.0f;
    int bi = 0x7fffffff;
    for (int c = 1 + lane; c < T; c += 32) {
      if (pa[c] != cur) continue;
      const float s = sc[c];
      if (!have || s > bs || (s == bs && c < bi)) {
        have = true;
        bs = s;
        bi = c;
      }
    }
#pragma unroll
    for (int o2 = 16; o2; o2 >>= 1) {
      const int oh = __shfl_xor_sync(0xffffffffu, (int)have, o2);
      const float os = __shfl_xor_sync(0xffffffffu, bs, o2);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o2);
      if (oh && (!have || os > bs || (os == bs && oi < bi))) {
        have = true;
        bs = os;
        bi = oi;
      }
    }
    if (!have) break;
    ++D;
    cur = bi;
    if (lane == 0) {
      pth[D] = bi;
      tok[(size_t)b * tok_stride + D - 1] = token[(size_t)b * T + bi];
    }
  }
  if (lane == 0) {
    npos[b] = D;
    tstat[b] = 0u;
  }
}

// ---------------------------------------------------------------------------
template <typename E>
sv_status run_verify(const Round &r, const Layout &L, char *ws, uint64_t seed, uint64_t step,
                     const DecideOut &o, cudaStream_t st) {
  float2 *partial = (float2 *)(ws + L.partial);
  Task *tasks = (Task *)(ws + L.task);
  Acc *acc = (Acc *)(ws + L.acc);
  ulonglong2 *chunks = (ulonglong2 *)(ws + L.chunks);
  sv_status s;
  {
    const long nitems = (long)r.B * r.P * L.G;
    LaunchScope ls("row_stats", st);
    row_stats_kernel<E><<<(unsigned)nitems, kStatsThreads, 0, st>>>(r, L.G, L.seg_len, partial);
    if ((s = check_launch("row_stats")) != SV_OK) return s;
  }
  {
    LaunchScope ls("decide", st);
    decide_kernel<E><<<(r.B + kDecideWarps - 1) / kDecideWarps, kDecideWarps * 32, 0, st>>>(
        r, L.G, partial, seed, step, o, tasks, acc);
    if ((s = check_launch("decide")) != SV_OK) return s;
  }
  {
    LaunchScope ls("sample_sum", st);
    sample_sum_kernel<E><<<dim3(r.B, L.G3), kSampleThreads, 0, st>>>(r, tasks, acc);
    if ((s = check_launch("sample_sum")) != SV_OK) return s;
  }
  {
    LaunchScope ls("sample_chunk", st);
    sample_chunk_kernel<E><<<dim3(r.B, L.G3), kSampleThreads, 0, st>>>(r, tasks, acc, chunks,
                                                                        L.nchunk);
    if ((s = check_launch("sample_chunk")) != SV_OK) return s;
  }
  {
    LaunchScope ls("sample_pick", st);
    sample_pick_kernel<E><<<r.B, 32, 0, st>>>(r, tasks, acc, chunks, L.nchunk, o);
    if ((s = check_launch("sample_pick")) != SV_OK) return s;
  }
  return SV_OK;
}

sv_status check_common(const void *vlogits, sv_dtype dt, int B, int V, float temperature,
                       const void *out_tokens, const void *out_accept, const void *out_status,
                       const void *workspace) {
  if (B < 0) return set_error(SV_ERR_INVALID_ARG, "B must be >= 0 (got %d)", B);
  if (V < 1) return set_error(SV_ERR_INVALID_ARG, "V must be >= 1 (got %d)", V);
  if (V > SV_MAX_VOCAB) return set_error(SV_ERR_UNSUPPORTED, "V > %d", SV_MAX_VOCAB);
  if (dt != SV_F32 && dt != SV_BF16) return set_error(SV_ERR_INVALID_ARG, "unknown dtype %d", (int)dt);
  if (!(temperature > 0.0f) || !isfinite(temperature))
    return set_error(SV_ERR_INVALID_ARG, "temperature must be finite and > 0");
  if (B == 0) return SV_OK;
  if (!vlogits || !out_tokens || !out_accept || !out_status || !workspace)
    return set_error(SV_ERR_INVALID_ARG, "null pointer argument");
  const size_t es = dt == SV_F32 ? 4 : 2;
  if ((uintptr_t)vlogits % es) return set_error(SV_ERR_INVALID_ARG, "vlogits misaligned");
  return SV_OK;
}

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" size_t sv_verify_chain_workspace(int B, int N, int V) {
  if (B < 0 || N < 0 || V < 1) return 0;
  return plan(B, N, V, false).total;
}

extern "C" sv_status sv_verify_chain(const void *vlogits, const void *dlogits, sv_dtype dt,
                                     const int32_t *draft_tokens, int B, int N, int V,
                                     float temperature, uint64_t seed, uint64_t step,
                                     int32_t *out_tokens, int32_t *out_accept_len,
                                     float *out_q_prob, float *out_p_prob, float *out_margin,
                                     uint32_t *out_status, void *workspace,
                                     size_t workspace_bytes, void *stream) {
  sv_status s = check_common(vlogits, dt, B, V, temperature, out_tokens, out_accept_len,
                             out_status, workspace);
  if (s != SV_OK || B == 0) return s;
  if (N < 0) return set_error(SV_ERR_INVALID_ARG, "N must be >= 0 (got %d)", N);
  if (N > SV_MAX_POSITIONS) return set_error(SV_ERR_UNSUPPORTED, "N > %d", SV_MAX_POSITIONS);
  if (N > 0 && (!dlogits || !draft_tokens))
    return set_error(SV_ERR_INVALID_ARG, "dlogits and draft_tokens are required when N > 0");
  const Layout L = plan(B, N, V, false);
  if (workspace_bytes < L.total)
    return set_error(SV_ERR_INVALID_ARG, "workspace too small: %zu < %zu", workspace_bytes,
                     L.total);
  char *ws = (char *)align_up((uintptr_t)workspace, 256);
  Round r;
  r.vlog = vlogits;
  r.dlog = N > 0 ? dlogits : vlogits;
  r.B = B;
  r.V = V;
  r.maxpos = N;
  r.P = L.P;
  r.v_rows = N + 1;
  r.d_rows = N;
  r.path = nullptr;
  r.npos = nullptr;
  r.tok = draft_tokens;
  r.tok_stride = N;
  r.tstat = nullptr;
  r.invT = 1.0f / temperature;
  r.k = r.invT * kLog2e;
  DecideOut o{out_tokens, out_accept_len, out_q_prob, out_p_prob, out_margin, out_status, nullptr};
  cudaStream_t st = (cudaStream_t)stream;
  return dt == SV_BF16 ? run_verify<uint16_t>(r, L, ws, seed, step, o, st)
                       : run_verify<float>(r, L, ws, seed, step, o, st);
}

extern "C" size_t sv_verify_tree_workspace(int B, int T, int max_depth, int V) {
  if (B < 0 || T < 1 || max_depth < 0 || V < 1) return 0;
  return plan(B, max_depth, V, true).total;
}

extern "C" sv_status sv_verify_tree(const void *vlogits, const void *dlogits, sv_dtype dt,
                                    const int32_t *parent, const int32_t *token,
                                    const float *score, int B, int T, int max_depth, int V,
                                    float temperature, uint64_t seed, uint64_t step,
                                    int32_t *out_path_nodes, int32_t *out_tokens,
                                    int32_t *out_accept_len, float *out_q_prob,
                                    float *out_p_prob, float *out_margin, uint32_t *out_status,
                                    void *workspace, size_t workspace_bytes, void *stream) {
  sv_status s = check_common(vlogits, dt, B, V, temperature, out_tokens, out_accept_len,
                             out_status, workspace);
  if (s != SV_OK || B == 0) return s;
  if (T < 1) return set_error(SV_ERR_INVALID_ARG, "T must be >= 1 (got %d)", T);
  if (T > SV_MAX_TREE_NODES) return set_error(SV_ERR_UNSUPPORTED, "T > %d", SV_MAX_TREE_NODES);
  if (max_depth < 0) return set_error(SV_ERR_INVALID_ARG, "max_depth must be >= 0");
  if (max_depth > SV_MAX_POSITIONS) return set_error(SV_ERR_UNSUPPORTED, "max_depth > %d", SV_MAX_POSITIONS);
  if (!dlogits || !parent || !token || !score || !out_path_nodes)
    return set_error(SV_ERR_INVALID_ARG, "null pointer argument");
  const Layout L = plan(B, max_depth, V, true);
  if (workspace_bytes < L.total)
    return set_error(SV_ERR_INVALID_ARG, "workspace too small: %zu < %zu", workspace_bytes,
                     L.total);
  char *ws = (char *)align_up((uintptr_t)workspace, 256);
  int32_t *path = (int32_t *)(ws + L.path);
  int32_t *npos = (int32_t *)(ws + L.npos);
  int32_t *tok = (int32_t *)(ws + L.tok);
  uint32_t *tstat = (uint32_t *)(ws + L.tstat);
  cudaStream_t st = (cudaStream_t)stream;
  {
    LaunchScope ls("tree_path", st);
    tree_path_kernel<<<B, 32, 0, st>>>(parent, token, score, B, T, max_depth, path, npos, tok,
                                       max_depth > 0 ? max_depth : 1, tstat);
    if ((s = check_launch("tree_path")) != SV_OK) return s;
  }
  Round r;
  r.vlog = vlogits;
  r.dlog = dlogits;
  r.B = B;
  r.V = V;
  r.maxpos = max_depth;
  r.P = L.P;
  r.v_rows = T;
  r.d_rows = T;
  r.path = path;
  r.npos = npos;
  r.tok = tok;
  r.tok_stride = max_depth > 0 ? max_depth : 1;
  r.tstat = tstat;
  r.invT = 1.0f / temperature;
  r.k = r.invT * kLog2e;
  DecideOut o{out_tokens, out_accept_len, out_q_prob, out_p_prob, out_margin, out_status,
              out_path_nodes};
  return dt == SV_BF16 ? run_verify<uint16_t>(r, L, ws, seed, step, o, st)
                       : run_verify<float>(r, L, ws, seed, step, o, st);
}

// ---------------------------------------------------------------------------
// Allocation-free chain verify.  Its scratch is a file-scope device array of
// kStaticScratchBytes that every GPU loading this library holds until exit.
// Host code cannot hand the array's name to a kernel (on the host it names a
// stand-in, not device memory), so the device address is looked up once per
// device with cudaGetSymbolAddress, with that device current, on the first
// call made on it.
#include <mutex>

namespace sv {
namespace {
constexpr size_t kStaticScratchBytes = size_t(4) << 20;  // 4 MiB
constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void *g_static_ptr[kMaxDevices] = {};
}  // namespace
}  // namespace sv

static __device__ __align__(256) unsigned char g_static_scratch[sv::kStaticScratchBytes];

namespace sv {
namespace {
sv_status static_scratch_address(void **out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_error(SV_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return set_error(SV_ERR_UNSUPPORTED, "device ordinal %d >= %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (!g_static_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || !p)
      return set_error(SV_ERR_CUDA, "cudaGetSymbolAddress(static scratch): %s",
                       cudaGetErrorString(e));
    g_static_ptr[dev] = p;
  }
  *out = g_static_ptr[dev];
  return SV_OK;
}
}  // namespace
}  // namespace sv

extern "C" size_t sv_verify_chain_noalloc_max_bytes(void) { return kStaticScratchBytes; }

extern "C" sv_status sv_verify_chain_noalloc(const void *vlogits, const void *dlogits,
                                             sv_dtype dt, const int32_t *draft_tokens, int B,
                                             int N, int V, float temperature, uint64_t seed,
                                             uint64_t step, int32_t *out_tokens,
                                             int32_t *out_accept_len, float *out_q_prob,
                                             float *out_p_prob, float *out_margin,
                                             uint32_t *out_status, void *stream) {
  if (B < 0 || N < 0 || V < 1)
    return set_error(SV_ERR_INVALID_ARG, "need B >= 0, N >= 0, V >= 1");
  if (B == 0) return SV_OK;
  const size_t need = sv_verify_chain_workspace(B, N, V);
  if (need > kStaticScratchBytes)
    return set_error(SV_ERR_UNSUPPORTED,
                     "sv_verify_chain_noalloc: B=%d N=%d V=%d needs %zu bytes of scratch, "
                     "more than the %zu-byte static scratch; use sv_verify_chain with a "
                     "caller-owned workspace",
                     B, N, V, need, kStaticScratchBytes);
  void *ws = nullptr;
  sv_status s = static_scratch_address(&ws);
  if (s != SV_OK) return s;
  return sv_verify_chain(vlogits, dlogits, dt, draft_tokens, B, N, V, temperature, seed, step,
                         out_tokens, out_accept_len, out_q_prob, out_p_prob, out_margin,
                         out_status, ws, kStaticScratchBytes, stream);
}
