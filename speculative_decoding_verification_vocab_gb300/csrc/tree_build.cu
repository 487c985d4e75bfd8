// tree_build.cu -- the EAGLE-2 dynamic draft tree on sm_103a: per-row top-K
// expansion with path-product scores, per-level frontier selection, and the
// final pruning to the node budget with level-by-level numbering.
//
// Page: "投机解码发展" (blog), section 5 (三代之间的变化): the tree grows where
// the draft is confident; a node's score is the product of the draft
// probabilities along its path; the best-scored nodes are expanded and the
// tree is pruned to a budget.
#include "common.cuh"
#include "rowstat.cuh"

namespace sv {
namespace {

constexpr int kExThreads = 256;
constexpr int kExWarps = kExThreads / 32;
constexpr int kMaxK = 16;
constexpr int kMaxCand = 2048;

// ---------------------------------------------------------------------------
// expand: one CTA per frontier row.  Each thread streams its 16-byte words
// (online softmax statistics in the log2 domain, as the verify step's row
// pass), and each warp keeps a top-K list spread over its lanes (lane j
// holds entry j; value descending, index ascending).  A word is looked at
// only when its packed maximum reaches the list's K-th value; its elements
// are then offered one at a time to the whole warp, which inserts an element
// that precedes the K-th entry by shifting the lanes after its rank.  The
// CTA merges the eight warp lists and writes the K tokens and their child
// scores.
struct WarpTopK {
  float v;  // this lane's entry (lane < K), -inf when empty
  int i;    // its token id, INT_MAX when empty
  float tv; // the K-th entry, uniform over the warp
  int ti;
};

// (va, ia) precedes (vb, ib): larger value, or equal value and lower id
__device__ __forceinline__ bool tk_before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

__device__ __forceinline__ void warp_offer(WarpTopK &w, float x, int idx, int K) {
  // uniform: every lane holds the same (x, idx)
  if (!tk_before(x, idx, w.tv, w.ti)) return;
  const unsigned FULL = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const int pos = __popc(__ballot_sync(FULL, lane < K && tk_before(w.v, w.i, x, idx)));
  const float pv = __shfl_up_sync(FULL, w.v, 1);
  const int pi = __shfl_up_sync(FULL, w.i, 1);
  if (lane > pos && lane < K) {
    w.v = pv;
    w.i = pi;
  }
  if (lane == pos) {
    w.v = x;
    w.i = idx;
  }
  w.tv = __shfl_sync(FULL, w.v, K - 1);
  w.ti = __shfl_sync(FULL, w.i, K - 1);
}

template <typename E>
__device__ __forceinline__ float word_max(uint4 w);
template <>
__device__ __forceinline__ float word_max<uint16_t>(uint4 w) {
  const uint32_t m = bf2_max(bf2_max(w.x, w.y), bf2_max(w.z, w.w));
  return fmaxf(bf16_lo(m), bf16_hi(m));
}
template <>
__device__ __forceinline__ float word_max<float>(uint4 w) {
  return fmaxf(fmaxf(__uint_as_float(w.x), __uint_as_float(w.y)),
               fmaxf(__uint_as_float(w.z), __uint_as_float(w.w)));
}
template <typename E>
__device__ __forceinline__ float word_elem(uint4 w, int j) {
  if (sizeof(E) == 2) {
    const uint32_t c = (j >> 1) == 0 ? w.x : (j >> 1) == 1 ? w.y : (j >> 1) == 2 ? w.z : w.w;
    return (j & 1) ? bf16_hi(c) : bf16_lo(c);
  }
  return __uint_as_float(j == 0 ? w.x : j == 1 ? w.y : j == 2 ? w.z : w.w);
}

// every lane's word (element ids v, v+1, ...): the lanes whose word can
// reach the list offer their elements, lane by lane; `skip` is an element id
// of the lane already in the list (-1: none)
template <typename E>
__device__ __forceinline__ void warp_offer_words(WarpTopK &w, uint4 word, int v, bool in, int K,
                                                 int skip, float floor_v) {
  constexpr int kPer = 16 / (int)sizeof(E);
  const unsigned FULL = 0xffffffffu;
  const float m = in ? word_max<E>(word) : -INFINITY;
  // the lane marks the elements of its word that can reach the list
  unsigned emask = 0u;
  const float gate = fmaxf(w.tv, floor_v);
  if (in && m >= gate) {
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const float x = word_elem<E>(word, j);
      if (x >= gate && v + j != skip) emask |= 1u << j;  // NaN fails the compare
    }
  }
  unsigned cand = __ballot_sync(FULL, emask != 0u);
  while (cand) {
    const int src = __ffs(cand) - 1;
    cand &= cand - 1;
    const uint4 q = make_uint4(__shfl_sync(FULL, word.x, src), __shfl_sync(FULL, word.y, src),
                               __shfl_sync(FULL, word.z, src), __shfl_sync(FULL, word.w, src));
    const int v0 = __shfl_sync(FULL, v, src);
    unsigned em = __shfl_sync(FULL, emask, src);
    while (em) {
      const int j = __ffs(em) - 1;
      em &= em - 1;
      warp_offer(w, word_elem<E>(q, j), v0 + j, K);
    }
  }
}

// Seed an empty warp list from a full batch: every lane's best element of
// its batch (value desc, id asc) is sorted across the warp (bitonic, by
// shuffles) and the first K become the list, so the gate is tight from the
// start.  Returns the id the lane contributed, or -1 if it was not kept.
template <typename E>
__device__ __forceinline__ int warp_seed(WarpTopK &w, const uint4 (&buf)[kRsUnroll], int v0,
                                         int stride_elems, int K) {
  constexpr int kPer = 16 / (int)sizeof(E);
  const unsigned FULL = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  float bv = -INFINITY;
  int bi = 0x7fffffff;
#pragma unroll
  for (int j = 0; j < kRsUnroll; ++j) {
    const float m = word_max<E>(buf[j]);
    int first = 0;  // the word's first element equal to its maximum
#pragma unroll
    for (int e = kPer - 1; e >= 0; --e)
      if (word_elem<E>(buf[j], e) == m) first = e;
    if (m > bv) {  // words come in increasing id: strict keeps the lowest id
      bv = m;
      bi = v0 + j * stride_elems + first;
    }
  }
  float sv = bv;
  int si = bi;
  // bitonic sort, descending in (value, then ascending id)
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const float ov = __shfl_xor_sync(FULL, sv, stride);
      const int oi = __shfl_xor_sync(FULL, si, stride);
      const bool up = ((lane & size) == 0);       // this block sorts descending
      const bool lower = (lane & stride) == 0;    // the lane keeps the "first" of the pair
      const bool other_first = tk_before(ov, oi, sv, si);
      if ((up == lower) == other_first) {
        sv = ov;
        si = oi;
      }
    }
  const bool ok = sv == sv && si != 0x7fffffff;
  w.v = (lane < K && ok) ? sv : -INFINITY;
  w.i = (lane < K && ok) ? si : 0x7fffffff;
  w.tv = __shfl_sync(FULL, w.v, K - 1);
  w.ti = __shfl_sync(FULL, w.i, K - 1);
  // did my own best element land in the list?
  const unsigned kept = __ballot_sync(FULL, lane < K && ok);
  int mine = -1;
  for (int j = 0; j < K; ++j) {
    const int id = __shfl_sync(FULL, w.i, j);
    if (((kept >> j) & 1u) && id == bi) mine = bi;
  }
  return mine;
}

// The candidate table of a whole build ([B][ldc] parent / token / score /
// level, candidate 0 = the root): with it, a level's expansion reads its
// frontier scores from the table and appends its children at n0, and the
// selection writes the next frontier's candidate ids -- no step between
// levels runs outside these kernels.  token == null: the plain arrays.
struct Table {
  const int32_t *frontier;  // [B][K] candidate ids of the rows (-1: empty); null: the root
  int32_t *parent, *token, *level;
  float *score;
  int ldc, n0, lvl, F;
};

template <typename E>
__global__ void __launch_bounds__(kExThreads, 4)
tree_expand_kernel(const E *__restrict__ dlog, int V, float k, int greedy,
                   const float *__restrict__ fscore_in, int K, int32_t *__restrict__ out_tok,
                   float *__restrict__ out_score, Table tb) {
  grid_dep_sync();
  const size_t rowi = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const E *row = dlog + rowi * (size_t)V;
  WarpTopK w{-INFINITY, 0x7fffffff, -INFINITY, 0x7fffffff};
  StatState st{-INFINITY, 0.0f, 0ull, 0ull};
  const uintptr_t pb = (uintptr_t)row, pe = (uintptr_t)(row + V);
  uintptr_t ab = (pb + 15) & ~(uintptr_t)15, ae = pe & ~(uintptr_t)15;
  if (ab > ae) ab = ae = pe;
  const int nhead = (int)((ab - pb) / sizeof(E));
  constexpr int kPer = 16 / (int)sizeof(E);
  const uint4 *body = (const uint4 *)ab;
  const int nv = (int)((ae - ab) / 16);
  const int ntail = (int)((pe - ae) / sizeof(E));
  // The largest K-th value of any warp's list bounds the row's final K-th
  // value from below, so every warp may drop elements under it: kept in
  // shared memory as an order-preserving integer key, raised by each warp's
  // lane 0 whenever its full list's K-th value rises.
  __shared__ unsigned s_floor;
  if (tid == 0) s_floor = 0u;  // below every float's key
  __syncthreads();
  auto fkey = [](float x) {
    const unsigned u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  };
  auto raise_floor = [&]() {
    if (lane == 0 && w.ti != 0x7fffffff) atomicMax(&s_floor, fkey(w.tv));
  };
  auto floor_v = [&]() {
    const unsigned kk = *(volatile unsigned *)&s_floor;
    if (kk == 0u) return -INFINITY;
    return __uint_as_float((kk & 0x80000000u) ? (kk & 0x7fffffffu) : ~kk);
  };
  int i = tid;
  constexpr int kStep = kRsUnroll * kExThreads;
  // warp-uniform trip count (the warp's offers are warp-wide collectives):
  // i - lane is the warp's first word of the batch.  The warp's last batch
  // may run past the row's body: those words read as -inf (nothing added to
  // the sums, never offered)
  const uint32_t ninf = sizeof(E) == 2 ? 0xFF80FF80u : 0xFF800000u;
  auto load = [&](uint4 (&buf)[kRsUnroll], unsigned &inb) {
    inb = 0xffu;  // words of the batch inside the body
    if ((i - lane) + 31 + (kRsUnroll - 1) * kExThreads < nv) {
#pragma unroll
      for (int j = 0; j < kRsUnroll; ++j) buf[j] = ld_stream_v4(body + i + j * kExThreads);
    } else {
#pragma unroll
      for (int j = 0; j < kRsUnroll; ++j) {
        const bool in = i + j * kExThreads < nv;
        buf[j] = in ? ld_stream_v4(body + i + j * kExThreads) : make_uint4(ninf, ninf, ninf, ninf);
        if (!in) inb &= ~(1u << j);
      }
    }
  };
  // one gate per batch: the words are looked at only when some lane's batch
  // maximum reaches the list's K-th value
  auto offer = [&](const uint4 (&buf)[kRsUnroll], unsigned inb, float bm, int skip) {
    const float fl = __shfl_sync(0xffffffffu, floor_v(), 0);  // one read per warp and batch
    if (__any_sync(0xffffffffu, bm >= fmaxf(w.tv, fl))) {
      const float tv0 = w.tv;
#pragma unroll
      for (int j = 0; j < kRsUnroll; ++j)
        warp_offer_words<E>(w, buf[j], nhead + (i + j * kExThreads) * kPer, (inb >> j) & 1u, K,
                            skip, fl);
      if (w.tv != tv0) raise_floor();
    }
  };
  // After the seeding round the CTA ranks the union of the warps' lists (the
  // entries are distinct elements of the row, so their K-th is a lower bound
  // on the row's final K-th value) and raises the floor to it: a much
  // tighter bound than any one warp's K-th.  Every thread takes part, so the
  // rounds are counted for the whole CTA (a warp past the row's body reads
  // -inf words).  Once is enough: ranking again after later rounds costs
  // more (two barriers each) than the tighter floor saves.
  __shared__ float s_lv[kExWarps * kMaxK];
  __shared__ int s_li[kExWarps * kMaxK];
  auto cta_floor = [&]() {
    if (lane < K) {
      s_lv[warp * K + lane] = w.v;
      s_li[warp * K + lane] = w.i;
    }
    __syncthreads();
    if (tid < kExWarps * K && s_li[tid] != 0x7fffffff) {
      const float x = s_lv[tid];
      const int id = s_li[tid];
      int rank = 0;
      for (int e = 0; e < kExWarps * K; ++e)
        rank += (s_li[e] != 0x7fffffff && tk_before(s_lv[e], s_li[e], x, id));
      if (rank == K - 1) atomicMax(&s_floor, fkey(x));
    }
    __syncthreads();  // the lists are rewritten only after every rank is taken
  };
  const int rounds = (nv + kStep - 1) / kStep;  // batch rounds of the whole CTA
  // the first batch seeds the empty list (peeled off, so that the seeding
  // code stays out of the streaming loop)
  if (rounds > 0) {
    uint4 buf[kRsUnroll];
    unsigned inb;
    load(buf, inb);
    const float bm = stat_batch<E>(buf, st, k);  // the batch maximum
    const int skip = warp_seed<E>(w, buf, nhead + i * kPer, kExThreads * kPer, K);
    raise_floor();
    offer(buf, inb, bm, skip);
    if (rounds > 1) cta_floor();
    i += kStep;
  }
  for (int r = 1; r < rounds; ++r, i += kStep) {
    uint4 buf[kRsUnroll];
    unsigned inb;
    load(buf, inb);
    offer(buf, inb, stat_batch<E>(buf, st, k), -1);
  }
  // ragged head and tail elements (fewer than 8 each), by warp 0, offered
  // after the body so that seeding (which replaces an empty list) cannot
  // drop them
  if (warp == 0) {
    for (int j = 0; j < nhead + ntail; ++j) {
      const int v = j < nhead ? j : nhead + nv * kPer + (j - nhead);
      const float x = load_elem<E>(row + v);
      if (lane == 0) stat1(x, st, k);
      if (x == x) warp_offer(w, x, v, K);
    }
  }
  // the row's statistics, as the verify step's row pass combines them
  float a0, a1, a2, a3;
  f2_unpack(st.s01, a0, a1);
  f2_unpack(st.s23, a2, a3);
  float mx = st.mx, mk = st.mk, ssum = (a0 + a1) + (a2 + a3);
  warp_stat_combine(mx, mk, ssum);
  __shared__ float4 s_red[kExWarps];
  __shared__ float s_tv[kExWarps * kMaxK];
  __shared__ int s_ti[kExWarps * kMaxK];
  __shared__ int s_pick[kMaxK];
  if (lane == 0) s_red[warp] = make_float4(mx, mk, ssum, 0.0f);
  if (lane < K) {
    s_tv[warp * K + lane] = w.v;
    s_ti[warp * K + lane] = w.i;
  }
  if (tid < K) s_pick[tid] = -1;
  __syncthreads();
  // merge: every listed entry's rank among the eight warp lists' entries
  // (value descending, token ascending; the warps cover disjoint tokens);
  // rank r < K is pick r
  if (tid < kExWarps * K) {
    const float x = s_tv[tid];
    const int id = s_ti[tid];
    if (x == x && id != 0x7fffffff) {
      int rank = 0;
      for (int e = 0; e < kExWarps * K; ++e) {
        const float y = s_tv[e];
        const int iy = s_ti[e];
        rank += (y == y && iy != 0x7fffffff && tk_before(y, iy, x, id));
      }
      if (rank < K) s_pick[rank] = tid;
    }
  }
  __syncthreads();
  if (warp != 0) return;
  float4 rs = lane < kExWarps ? s_red[lane] : make_float4(-INFINITY, 0.0f, 0.0f, 0.0f);
  warp_stat_combine(rs.x, rs.y, rs.z);
  const float MK = rs.y, S = rs.z;
  // the row's node and its path score: from the arrays, or from the table
  // (an id outside [0, n0) is an empty entry)
  int node = 0;
  float fs;
  const int tb_b = tb.token ? (int)(rowi / tb.F) : 0, tb_f = tb.token ? (int)(rowi % tb.F) : 0;
  if (!tb.token) {
    fs = fscore_in[rowi];
  } else if (!tb.frontier) {
    fs = 1.0f;  // the root
  } else {
    node = tb.frontier[(size_t)tb_b * K + tb_f];
    fs = (node >= 0 && node < tb.n0) ? tb.score[(size_t)tb_b * tb.ldc + node] : NAN;
    if (!(node >= 0 && node < tb.n0)) node = -1;
  }
  // a faulty row (NaN or +inf: the sum is NaN; all -inf: the sum is 0), or a
  // frontier entry with a NaN score (no node), proposes nothing
  const bool bad = !(S > 0.0f) || fs != fs;
  if (lane < K) {
    const int e = s_pick[lane];
    int32_t tok_o = -1;
    float sc_o = -INFINITY;
    if (!bad && e >= 0) {
      const float p =
          greedy ? (lane == 0 ? 1.0f : 0.0f) : ex2_approx(fmaf(s_tv[e], k, -MK)) / S;
      tok_o = s_ti[e];
      sc_o = fs * p;
    }
    if (!tb.token) {
      out_tok[rowi * (size_t)K + lane] = tok_o;
      out_score[rowi * (size_t)K + lane] = sc_o;
    } else {
      const size_t c = (size_t)tb_b * tb.ldc + tb.n0 + (size_t)tb_f * K + lane;
      tb.token[c] = tok_o;
      tb.score[c] = sc_o;
      tb.parent[c] = node;
      tb.level[c] = tb.lvl;
      if (!tb.frontier && lane == 0) {  // level 1 also writes the root, candidate 0
        const size_t r = (size_t)tb_b * tb.ldc;
        tb.token[r] = 0;
        tb.score[r] = 1.0f;
        tb.parent[r] = -1;
        tb.level[r] = 0;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// select: one CTA per sequence.  A candidate's pick order is its rank among
// the candidates with a token (score descending, index ascending); every
// thread ranks its candidates against all others staged in shared memory,
// and a candidate of rank r < K is pick r.
__global__ void __launch_bounds__(kExThreads)
tree_select_kernel(const float *__restrict__ score_base, const int32_t *__restrict__ token_base,
                   int C, int ld, int off, int K, int32_t *__restrict__ out) {
  grid_dep_sync();
  const int b = blockIdx.x, tid = threadIdx.x;
  // the C candidates of this sequence start at row b, column off (row stride
  // ld); picks are written as off + their index
  const float *score = score_base + (size_t)b * ld + off;
  const int32_t *token = token_base + (size_t)b * ld + off;
  __shared__ float sv_[kMaxCand];
  __shared__ int ok_[kMaxCand];
  __shared__ int s_nvalid;
  if (tid == 0) s_nvalid = 0;
  __syncthreads();
  int nv = 0;
  for (int c = tid; c < C; c += kExThreads) {
    sv_[c] = score[c];
    ok_[c] = token[c] >= 0;
    nv += ok_[c];
  }
  atomicAdd(&s_nvalid, nv);
  __syncthreads();
  for (int c = tid; c < C; c += kExThreads) {
    if (!ok_[c]) continue;
    const float v = sv_[c];
    int rank = 0;
    for (int d = 0; d < C; ++d)
      rank += ok_[d] && (sv_[d] > v || (sv_[d] == v && d < c));
    if (rank < K) out[(size_t)b * K + rank] = off + c;
  }
  for (int r = s_nvalid + tid; r < K; r += kExThreads) out[(size_t)b * K + r] = -1;
}

// ---------------------------------------------------------------------------
// finalize: one CTA per sequence.  A candidate (the root, or one with a
// token) is kept when its rank in keep order (score descending, level
// ascending, index ascending) is below T; a kept node's slot is its rank
// among the kept in (level ascending, score descending, index ascending);
// parents map through the candidate -> slot table.
__device__ __forceinline__ bool keep_before(float sa, int la, int a, float sb, int lb, int b) {
  if (sa != sb) return sa > sb;
  if (la != lb) return la < lb;
  return a < b;
}

__global__ void __launch_bounds__(kExThreads)
tree_finalize_kernel(const int32_t *__restrict__ cparent, const int32_t *__restrict__ ctoken,
                     const float *__restrict__ cscore, const int32_t *__restrict__ clevel, int C,
                     int ld, int Tn, int32_t *__restrict__ parent, int32_t *__restrict__ token,
                     float *__restrict__ score) {
  grid_dep_sync();
  const int b = blockIdx.x, tid = threadIdx.x;
  const int32_t *cp = cparent + (size_t)b * ld, *ct = ctoken + (size_t)b * ld;
  __shared__ float sc_[kMaxCand];
  __shared__ int lv_[kMaxCand];  // level, or -1: not a node
  __shared__ int slot_of[kMaxCand];
  __shared__ int keep[kMaxCand];  // candidates in keep order, non-nodes (-1) last
  __shared__ int s_nodes;
  int P = 1;
  while (P < C) P <<= 1;
  if (tid == 0) s_nodes = 0;
  for (int c = tid; c < P; c += kExThreads) {
    const bool in = c < C;
    if (in) {
      sc_[c] = cscore[(size_t)b * ld + c];
      lv_[c] = (c == 0 || ct[c] >= 0) ? clevel[(size_t)b * ld + c] : -1;
      slot_of[c] = -1;
    }
    keep[c] = (in && lv_[c] >= 0) ? c : -1;
  }
  __syncthreads();
  // keep order: a bitonic sort of the candidate ids in shared memory (the
  // order is total: ids are unique), the first Tn nodes are kept
  auto before = [&](int x, int y) {
    return x >= 0 && (y < 0 || keep_before(sc_[x], lv_[x], x, sc_[y], lv_[y], y));
  };
  for (int size = 2; size <= P; size <<= 1)
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int q = tid; q < P / 2; q += kExThreads) {
        const int lo = 2 * q - (q & (stride - 1)), hi = lo + stride;
        const int x = keep[lo], y = keep[hi];
        if (((lo & size) == 0) ? before(y, x) : before(x, y)) {
          keep[lo] = y;
          keep[hi] = x;
        }
      }
      __syncthreads();
    }
  for (int i = tid; i < P; i += kExThreads)
    if (keep[i] >= 0 && (i + 1 == P || keep[i + 1] < 0)) s_nodes = i + 1;
  __syncthreads();
  const int n = min(s_nodes, Tn);
  for (int i = tid; i < n; i += kExThreads) {
    const int c = keep[i];
    const int l = lv_[c];
    const float v = sc_[c];
    int rank = 0;
    for (int j = 0; j < n; ++j) {
      const int d = keep[j];
      rank += (lv_[d] < l) || (lv_[d] == l && (sc_[d] > v || (sc_[d] == v && d < c)));
    }
    slot_of[c] = rank;
  }
  __syncthreads();
  for (int i = tid; i < n; i += kExThreads) {
    const int c = keep[i], sl = slot_of[c];
    const int pc = cp[c];
    parent[(size_t)b * Tn + sl] =
        pc < 0 ? -1 : (pc < C && slot_of[pc] >= 0 ? slot_of[pc] : -2);
    token[(size_t)b * Tn + sl] = ct[c];
    score[(size_t)b * Tn + sl] = sc_[c];
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
                                       out_token, out_score, Table{})
                          : launch_pdl(tree_expand_kernel<float>, grid, dim3(kExThreads), 0, st,
                                       (const float *)dlogits, V, k, greedy, frontier_score, K,
                                       out_token, out_score, Table{}));
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
                      launch_pdl(tree_select_kernel, dim3(B), dim3(kExThreads), 0, st,
                                 cand_score, cand_token, C, C, 0, K, out_index));
}

extern "C" sv_status sv_tree_finalize(const int32_t *cand_parent, const int32_t *cand_token,
                                      const float *cand_score, const int32_t *cand_level, int B,
                                      int C, int ldc, int T, int32_t *out_parent,
                                      int32_t *out_token, float *out_score, void *stream) {
  if (B < 0 || C < 1 || T < 1) return set_error(SV_ERR_INVALID_ARG, "need B >= 0, C >= 1, T >= 1");
  if (ldc < C) return set_error(SV_ERR_INVALID_ARG, "need ldc >= C (got ldc %d, C %d)", ldc, C);
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
                                 cand_parent, cand_token, cand_score, cand_level, C, ldc, T,
                                 out_parent, out_token, out_score));
}

extern "C" sv_status sv_tree_level(const void *dlogits, sv_dtype dt, int B, int F, int V,
                                   float temperature, int K, int level, int n0, int ldc,
                                   int32_t *frontier, int32_t *cand_parent, int32_t *cand_token,
                                   float *cand_score, int32_t *cand_level, void *stream) {
  if (B < 0 || F < 1 || V < 1) return set_error(SV_ERR_INVALID_ARG, "need B >= 0, F >= 1, V >= 1");
  if (K < 1 || K > V) return set_error(SV_ERR_INVALID_ARG, "need 1 <= K <= V");
  if (K > kMaxK) return set_error(SV_ERR_UNSUPPORTED, "K > %d", kMaxK);
  if (V > SV_MAX_VOCAB) return set_error(SV_ERR_UNSUPPORTED, "V > %d", SV_MAX_VOCAB);
  if (dt != SV_F32 && dt != SV_BF16) return set_error(SV_ERR_INVALID_ARG, "unknown dtype %d", (int)dt);
  if (!(temperature >= 0.0f) || !isfinite(temperature))
    return set_error(SV_ERR_INVALID_ARG, "temperature must be finite and >= 0");
  if (level < 1) return set_error(SV_ERR_INVALID_ARG, "level must be >= 1");
  if (level == 1 && (F != 1 || n0 != 1))
    return set_error(SV_ERR_INVALID_ARG, "level 1 expands the root: F = 1, n0 = 1");
  if (level > 1 && (F > K || n0 < 2))
    return set_error(SV_ERR_INVALID_ARG, "level > 1: F <= K (the frontier) and n0 >= 2");
  if ((long long)n0 + (long long)F * K > ldc)
    return set_error(SV_ERR_INVALID_ARG, "candidate table full: n0 + F*K > ldc");
  if (ldc > kMaxCand) return set_error(SV_ERR_UNSUPPORTED, "ldc > %d", kMaxCand);
  if ((long long)B * F > 0x7fffffffLL) return set_error(SV_ERR_UNSUPPORTED, "B * F too large");
  if (B == 0) return SV_OK;
  if (!dlogits || !frontier || !cand_parent || !cand_token || !cand_score || !cand_level)
    return set_error(SV_ERR_INVALID_ARG, "null pointer argument");
  if ((uintptr_t)dlogits % (dt == SV_F32 ? 4 : 2)) return set_error(SV_ERR_INVALID_ARG, "dlogits misaligned");
  sv_status s;
  if ((s = map_arg(dlogits, "dlogits")) != SV_OK || (s = map_arg(frontier, "frontier")) != SV_OK ||
      (s = map_arg(cand_parent, "cand_parent")) != SV_OK ||
      (s = map_arg(cand_token, "cand_token")) != SV_OK ||
      (s = map_arg(cand_score, "cand_score")) != SV_OK ||
      (s = map_arg(cand_level, "cand_level")) != SV_OK)
    return s;
  const int greedy = temperature == 0.0f;
  const float k = greedy ? kLog2eB : kLog2eB / temperature;
  cudaStream_t st = (cudaStream_t)stream;
  Table tb{level == 1 ? nullptr : frontier, cand_parent, cand_token, cand_level, cand_score,
           ldc, n0, level, F};
  {
    LaunchScope ls("tree_expand", st);
    const dim3 grid((unsigned)(B * F));
    s = check_launch("tree_expand",
                     dt == SV_BF16
                         ? launch_pdl(tree_expand_kernel<uint16_t>, grid, dim3(kExThreads), 0, st,
                                      (const uint16_t *)dlogits, V, k, greedy, nullptr, K, nullptr,
                                      nullptr, tb)
                         : launch_pdl(tree_expand_kernel<float>, grid, dim3(kExThreads), 0, st,
                                      (const float *)dlogits, V, k, greedy, nullptr, K, nullptr,
                                      nullptr, tb));
    if (s != SV_OK) return s;
  }
  // the next frontier: the K best of this level's F*K children, as ids
  LaunchScope ls("tree_select", st);
  return check_launch("tree_select",
                      launch_pdl(tree_select_kernel, dim3(B), dim3(kExThreads), 0, st,
                                 (const float *)cand_score, (const int32_t *)cand_token, F * K, ldc,
                                 n0, K, frontier));
}
