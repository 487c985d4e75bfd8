// verify.cu -- batched verify-and-accept for speculative decoding on sm_103a.
//
// Steps (one stream, no host synchronisation):
//   tree_path    (tree only) best-child walk per sequence
//   row_stats    single-pass online softmax statistics (max, sum of exp) of
//                every logit row the round can touch -- the one step that
//                streams the whole input; HBM-bound
//   decide       one warp per sequence: q(d)/p(d), Philox uniforms, the left-
//                to-right accept walk, outputs, and the sampling task
//   sample_norm  exact fixed-point normaliser partials of the 1-2 sampled rows;
//                the last slice CTA of a sequence turns them into 1/S_e
//   sample_mass  fixed-point residual / bonus masses per slice and per run;
//                the last slice CTA of a sequence does the inverse-CDF pick
//
// Pages: "Decodificação Especulativa e EAGLE-3" (lesson; "O invariante",
// Passo 1-3) and "投机解码发展" (blog; section 2 steps, section 4 spec_decode /
// eagle_round pseudocode).  p = draft, q = verifier.
#include <math.h>
#include <stdio.h>

#include "common.cuh"
#include "rowstat.cuh"


namespace sv {
namespace {

constexpr int kDecideWarps = 4;
// sampler geometry: a CTA owns a 4096-element slice of a row; each of its
// threads owns kSpRun consecutive elements of the slice
constexpr int kSpThreads = 128;
constexpr int kSpWarps = kSpThreads / 32;
constexpr int kSpRun = 32;
constexpr int kSpSlice = kSpThreads * kSpRun;  // 4096 elements per CTA
constexpr float kLog2e = 1.4426950408889634f;

struct Task {
  const void *rq;  // the verifier row to sample from (its device copy for host logits)
  const void *rp;  // the draft row of a residual draw, null for a bonus draw
  int active;      // 1: a correction / bonus token is to be drawn
  int a;           // accept length = output slot of the drawn token
  float mq, mp;    // raw-logit maxima of those rows
  uint32_t u24;
  int pad;
};

struct Layout {
  int maxpos, P, G, CS;
  size_t ctr, rowlist, partial, task, norm, mass, run, done, inv, path, npos, tok, tstat;
  size_t ee;     // early exit (chain): [B][maxpos] position counts, then [B] stop
  size_t end;    // end of the regions (256-aligned); an optional row copy follows
  size_t total;  // bytes to request: the regions plus base-pointer alignment
};

Layout plan(int B, int maxpos, int V, bool tree);

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
  int stage;                // logits in device memory: row_stats may stage through
                            // shared memory with asynchronous copies
  char *copy;               // host-resident logits: device copy of every row slot
  size_t pitch;             // that row_stats reads (bytes per slot), or null
};

__device__ __forceinline__ int round_npos(const Round &r, int b) {
  return r.npos ? r.npos[b] : r.maxpos;
}
__device__ __forceinline__ int round_node(const Round &r, int b, int i) {
  return r.path ? r.path[(size_t)b * (r.maxpos + 1) + i] : i;
}

// Row slot j of sequence b: the verifier row of position j (j <= maxpos) or
// the draft row of position j - maxpos - 1, in the caller's logits ...
template <typename E>
__device__ __forceinline__ const E *src_row(const Round &r, int b, int j) {
  const bool is_v = j <= r.maxpos;
  const int node = round_node(r, b, is_v ? j : j - r.maxpos - 1);
  return (const E *)(is_v ? r.vlog : r.dlog) +
         ((size_t)b * (is_v ? r.v_rows : r.d_rows) + node) * (size_t)r.V;
}
// ... and where the steps after row_stats read it: the device copy when the
// logits are host-resident (same offset within 16 bytes as the source row,
// so the vector paths line up), else the source row itself
template <typename E>
__device__ __forceinline__ const E *used_row(const Round &r, int b, int j, const E *src) {
  if (!r.copy) return src;
  return (const E *)(r.copy + ((size_t)b * r.P + j) * r.pitch + ((uintptr_t)src & 15));
}

// ---------------------------------------------------------------------------
// row_stats: online softmax statistics of every used logit row.
// One CTA per (row, kSegElems-element segment); grid x = row (tree: the rows
// on the best paths, listed by tree_path), y = segment.  Each thread loads
// kRsUnroll 16-byte words at once, takes the batch maximum on packed pairs,
// moves its log2-domain reference only when that maximum exceeds the running
// one, and folds the batch into a sum of exp2(fma(x, k, -ref)) with packed
// fp32 pair arithmetic (one ex2 per element).  The CTA combines the
// per-thread triples and writes (max x, mk, sum exp2(fma(x, k, -mk))) for the
// segment.  Ragged head / tail elements (outside the 16-byte-aligned body)
// are read one by one.  Row slot j of a sequence is the verifier row of
// position j (j <= maxpos) or the draft row of position j - maxpos - 1.
constexpr int kSegElems = 8192;  // smallest segment (fp32); sizes the workspace
constexpr int kRsThreads = 128;
// A thread owns 2 * kRsUnroll 16-byte words of a segment: the first
// kRsUnroll go to registers, the second are staged into shared memory by
// asynchronous copies issued first, so a CTA keeps 32 KB of loads in flight
// while holding only 32 words of registers per thread.  Segments of 32 KB
// (128 threads, 10 CTAs/SM) rather than 64 KB: twice the CTAs of half the
// work even out the end of a launch (row pass 0.86 -> 0.95 of the copy
// bandwidth on the large-vocabulary chain).
template <typename E>
__host__ __device__ constexpr int seg_elems() {
  return kRsThreads * 2 * kRsUnroll * 16 / (int)sizeof(E);
}

// Row slot of active row `a` of sequence b (tree: a <= npos verifier, then draft)
__device__ __forceinline__ int slot_of_active(int a, int npos, int maxpos) {
  return a <= npos ? a : maxpos + 1 + (a - npos - 1);
}

struct SegInfo {
  const char *row;   // row base
  char *copy;        // its device copy (host-resident logits), or null
  int v0, v1;        // element range of the segment
  uintptr_t ab, ae;  // 16-byte-aligned body [ab, ae)
  size_t out;        // partial index
};

template <typename E>
__device__ __forceinline__ SegInfo seg_info(const Round &r, int G, const int32_t *rowlist,
                                            int row_i, int seg) {
  int b, j;
  if (rowlist) {
    const int e = rowlist[row_i];
    b = e >> 12;
    j = slot_of_active(e & 0xfff, round_npos(r, b), r.maxpos);
  } else {
    b = row_i / r.P;
    j = row_i - b * r.P;
  }
  SegInfo si;
  const E *row = src_row<E>(r, b, j);
  si.row = (const char *)row;
  si.copy = r.copy ? (char *)used_row<E>(r, b, j, row) : nullptr;
  si.v0 = seg * seg_elems<E>();
  si.v1 = min(r.V, si.v0 + seg_elems<E>());
  const uintptr_t pb = (uintptr_t)(row + si.v0), pe = (uintptr_t)(row + si.v1);
  si.ab = (pb + 15) & ~(uintptr_t)15;
  si.ae = pe & ~(uintptr_t)15;
  if (si.ab > si.ae) si.ab = si.ae = pe;
  si.out = ((size_t)b * r.P + j) * G + seg;
  return si;
}

// statistics of segment seg of listed row row_i, by the whole CTA
template <typename E, bool kCopy>
__device__ __forceinline__ void stat_segment(const Round &r, int G, const int32_t *rowlist,
                                             int row_i, int seg, float4 *partial) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const SegInfo si = seg_info<E>(r, G, rowlist, row_i, seg);
  const E *row = (const E *)si.row;
  const float k = r.k;
  StatState st{-INFINITY, 0.0f, 0ull, 0ull};
  const int nhead = (int)((si.ab - (uintptr_t)(row + si.v0)) / sizeof(E));
  const int ntail = (int)(((uintptr_t)(row + si.v1) - si.ae) / sizeof(E));
  // host-resident logits: every element read is also written to the row's
  // device copy, which the accept walk and the sampler read instead
  E *crow = kCopy ? (E *)si.copy : nullptr;
  uint4 *cbody = kCopy ? (uint4 *)(si.copy + (si.ab - (uintptr_t)si.row)) : nullptr;
  if (tid < nhead) {
    const E x = __ldg(row + si.v0 + tid);
    if (kCopy) crow[si.v0 + tid] = x;
    stat1(elem_to_f32(x), st, k);
  }
  if (tid < ntail) {
    const int v = (int)((si.ae - (uintptr_t)row) / sizeof(E)) + tid;
    const E x = __ldg(row + v);
    if (kCopy) crow[v] = x;
    stat1(elem_to_f32(x), st, k);
  }
  const uint4 *body = (const uint4 *)si.ab;
  const int nv = (int)((si.ae - si.ab) / 16);
  int i = tid;
  if (!kCopy && r.stage && i + (2 * kRsUnroll - 1) * kRsThreads < nv) {
    // full pattern: the second half through shared memory (each thread reads
    // back only the slots it copied, so its own wait is the only sync needed)
    __shared__ uint4 sbuf[kRsUnroll][kRsThreads];
#pragma unroll
    for (int j = 0; j < kRsUnroll; ++j)
      cp_async16(&sbuf[j][tid], body + i + (kRsUnroll + j) * kRsThreads);
    cp_async_commit();
    uint4 buf[kRsUnroll];
#pragma unroll
    for (int j = 0; j < kRsUnroll; ++j) buf[j] = ld_stream_v4(body + i + j * kRsThreads);
    stat_batch<E>(buf, st, k);
    cp_async_wait_all();
#pragma unroll
    for (int j = 0; j < kRsUnroll; ++j) buf[j] = sbuf[j][tid];
    stat_batch<E>(buf, st, k);
    i += 2 * kRsUnroll * kRsThreads;
  }
  for (; i + (kRsUnroll - 1) * kRsThreads < nv; i += kRsUnroll * kRsThreads) {
    uint4 buf[kRsUnroll];
#pragma unroll
    for (int j = 0; j < kRsUnroll; ++j) buf[j] = ld_stream_v4(body + i + j * kRsThreads);
    if (kCopy)
#pragma unroll
      for (int j = 0; j < kRsUnroll; ++j) cbody[i + j * kRsThreads] = buf[j];
    stat_batch<E>(buf, st, k);
  }
  for (; i < nv; i += kRsThreads) {
    const uint4 w = ld_stream_v4(body + i);
    if (kCopy) cbody[i] = w;
    stat_word<E>(w, st, k);
  }

  float a0, a1, a2, a3;
  f2_unpack(st.s01, a0, a1);
  f2_unpack(st.s23, a2, a3);
  float mx = st.mx, mk = st.mk, s = (a0 + a1) + (a2 + a3);
  warp_stat_combine(mx, mk, s);
  __shared__ float4 red[kRsThreads / 32];
  if (lane == 0) red[warp] = make_float4(mx, mk, s, 0.0f);
  __syncthreads();
  if (warp == 0) {
    float4 v = lane < kRsThreads / 32 ? red[lane] : make_float4(-INFINITY, 0.0f, 0.0f, 0.0f);
    warp_stat_combine(v.x, v.y, v.z);
    if (lane == 0) partial[si.out] = v;
  }
  __syncthreads();  // red[] is reused by the CTA's next row
}

template <typename E, bool kCopy>
__global__ void __launch_bounds__(kRsThreads, sizeof(E) == 2 ? 10 : 8)
row_stats_kernel(Round r, int G, const int32_t *__restrict__ rowlist,
                 const int32_t *__restrict__ rowcount, float4 *__restrict__ partial) {
  grid_dep_sync();
  // chain: one row per CTA (exact grid); tree: the grid covers half the row
  // slots and a CTA takes a second listed row when the paths are deep
  const int nrows = rowlist ? *rowcount : (int)gridDim.x;
  for (int row_i = blockIdx.x; row_i < nrows; row_i += gridDim.x)
    stat_segment<E, kCopy>(r, G, rowlist, row_i, blockIdx.y, partial);
}

Layout plan(int B, int maxpos, int V, bool tree) {
  Layout L;
  L.maxpos = maxpos;
  L.P = 2 * maxpos + 1;
  L.G = (V + kSegElems - 1) / kSegElems;
  const size_t nslots = (size_t)B * L.P;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  L.ctr = take(sizeof(int));  // active row count (tree)
  L.rowlist = tree ? take(sizeof(int32_t) * nslots) : 0;
  L.partial = take(sizeof(float4) * nslots * L.G);
  L.task = take(sizeof(Task) * (size_t)B);
  L.CS = (V + kSpSlice - 1) / kSpSlice;
  L.norm = take(sizeof(ulonglong2) * (size_t)B * L.CS);
  L.mass = take(sizeof(unsigned long long) * (size_t)B * L.CS);
  L.run = take(sizeof(unsigned long long) * (size_t)B * L.CS * kSpThreads);
  L.done = take(sizeof(unsigned) * 2 * (size_t)B);
  L.inv = take(sizeof(float2) * (size_t)B);
  L.ee = take(sizeof(int) * (size_t)B * (maxpos + 1));
  if (tree) {
    L.path = take(sizeof(int32_t) * (size_t)B * (maxpos + 1));
    L.npos = take(sizeof(int32_t) * (size_t)B);
    L.tok = take(sizeof(int32_t) * (size_t)B * (maxpos > 0 ? maxpos : 1));
    L.tstat = take(sizeof(uint32_t) * (size_t)B);
  } else {
    L.path = L.npos = L.tok = L.tstat = 0;
  }
  L.end = off;
  L.total = off + 256;
  return L;
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

// Merge the G segment partials of one row: raw max mx, log2 reference mk and
// the sum s = sum_v exp2(fma(x_v, k, -mk)).  kCg: the partials were written by
// other CTAs of the running kernel (read through L2).
// The loads of a group of 8 partials are issued together, then merged in
// segment order (the same order for every G, so the result does not depend on
// how the loads were grouped).
template <bool kCg = false>
__device__ __forceinline__ void merge_slot(const float4 *part, int G, float &mx, float &mk,
                                           float &s) {
  mx = -INFINITY;
  mk = 0.0f;
  s = 0.0f;
  for (int g0 = 0; g0 < G; g0 += 8) {
    float4 v[8];
#pragma unroll
    for (int g = 0; g < 8; ++g)
      if (g0 + g < G) v[g] = kCg ? __ldcg(part + g0 + g) : part[g0 + g];
#pragma unroll
    for (int g = 0; g < 8; ++g)
      if (g0 + g < G) st_combine(mx, mk, s, v[g].x, v[g].y, v[g].z);
  }
}

// One position of the walk from the merged statistics of its verifier and
// draft rows ([Lesson] Passo 1: accept iff u < min(1, q(d)/p(d)), p(d) = 0
// accepted outright): q(d), p(d), the clipped ratio, the uniform, and the
// position's faults (a row without a finite positive sum, a token outside the
// vocabulary).  The accept walk and the early-exit hint both call it on the
// same partials, so they take the same decision.
struct Judged {
  float mxq, mxp;    // raw maxima of the verifier / draft row
  float qd, pd, rc;  // q(d), p(d), min(1, q(d)/p(d))
  uint32_t u24;      // the accept uniform
  uint32_t bad;      // SV_ROW_NAN / SV_ROW_BAD_TOKEN found at this position
  bool accept, p_zero;
};
template <typename E, bool kCg>
__device__ __forceinline__ Judged judge_position(const Round &r, int G, const float4 *pb, int b,
                                                 int i, int d, const E *vrow, const E *drow,
                                                 uint64_t seed, uint64_t step) {
  Judged J;
  // the two logits at the token first: their loads overlap the merges
  const bool tok_ok = d >= 0 && d < r.V;
  const float xq = tok_ok ? load_elem<E>(vrow + d) : 0.0f;
  const float xp = tok_ok ? load_elem<E>(drow + d) : 0.0f;
  float mkq, sq, mkp, sp;
  merge_slot<kCg>(pb + (size_t)i * G, G, J.mxq, mkq, sq);
  merge_slot<kCg>(pb + (size_t)(r.maxpos + 1 + i) * G, G, J.mxp, mkp, sp);
  J.bad = (!(sq > 0.0f) || !(sp > 0.0f)) ? SV_ROW_NAN : 0u;
  J.qd = J.pd = J.rc = NAN;
  J.u24 = 0u;
  J.accept = J.p_zero = false;
  if (!tok_ok) {
    J.bad |= SV_ROW_BAD_TOKEN;
    return J;
  }
  const float k = r.k;
  // log2 q(d) + log2 sq and log2 p(d) + log2 sp, against the row references
  const float lq = fmaf(xq, k, -mkq), lp = fmaf(xp, k, -mkp);
  J.qd = exp2f(lq) / sq;
  J.pd = exp2f(lp) / sp;
  J.p_zero = (xp == -INFINITY);
  float ratio;
  if (J.p_zero)
    ratio = INFINITY;
  else if (xq == -INFINITY)
    ratio = 0.0f;
  else
    ratio = exp2f((lq - lp) + (log2f(sp) - log2f(sq)));
  J.rc = fminf(ratio, 1.0f);
  J.u24 = uniform_u24(seed, step, (uint32_t)b, (uint32_t)i, kDrawAccept);
  const float u = (float)J.u24 * 0x1p-24f;
  J.accept = J.p_zero || (u < J.rc);
  return J;
}

// kEarly: the early-exit reading -- only the rows the walk reaches count: a
// position's faults stop the walk there (and fault the sequence), the bonus
// row faults only when every position passes, and q(d), p(d) and the margin
// after the first rejection are NaN (those rows may never have been read).
template <typename E, bool kEarly>
__global__ void __launch_bounds__(kDecideWarps * 32)
decide_kernel(Round r, int G, const float4 *__restrict__ partial, uint64_t seed,
              uint64_t step, DecideOut o, Task *__restrict__ tasks,
              unsigned *__restrict__ done) {
  grid_dep_sync();
  const int b = blockIdx.x * kDecideWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= r.B) return;
  const unsigned FULL = 0xffffffffu;
  const int npos = round_npos(r, b);
  const uint32_t tree_bad = r.tstat ? r.tstat[b] : 0u;
  const float4 *pb = partial + (size_t)b * r.P * G;
  // per position: raw max of the verifier / draft row and the sample uniform,
  // kept for the task so that lane 0 needs no further global reads
  extern __shared__ float dsm[];
  float *mxv = dsm + (threadIdx.x >> 5) * 3 * (r.maxpos + 1);
  float *mxd = mxv + (r.maxpos + 1);
  uint32_t *usm = (uint32_t *)(mxd + (r.maxpos + 1));

  uint32_t bad = 0, pzero_bits = 0, acc_bits = 0;
  // early exit: per chunk, this lane's position faults (row / token)
  uint32_t nan_bits = 0, tokbad_bits = 0;
  // bonus row (verifier row of position npos) is checked by lane 0
  if (lane == 0 && !tree_bad) {
    float mx, mk, s;
    merge_slot(pb + (size_t)npos * G, G, mx, mk, s);
    if (!(s > 0.0f)) bad |= SV_ROW_NAN;
    mxv[npos] = mx;
    usm[npos] = uniform_u24(seed, step, (uint32_t)b, (uint32_t)npos, kDrawSample);
  }
  const uint32_t bonus_bad = kEarly ? __shfl_sync(FULL, bad, 0) : 0u;
  if (kEarly) bad = 0;
  const int nchunks = (npos + 31) / 32;
  for (int c = 0; c < nchunks && !tree_bad; ++c) {
    const int i = c * 32 + lane;
    if (i >= npos) break;
    const int d = r.tok[(size_t)b * r.tok_stride + i];  // issued first: x_d depends on it
    const E *vrow = used_row<E>(r, b, i, src_row<E>(r, b, i));
    const E *drow = used_row<E>(r, b, r.maxpos + 1 + i, src_row<E>(r, b, r.maxpos + 1 + i));
    const Judged J = judge_position<E, false>(r, G, pb, b, i, d, vrow, drow, seed, step);
    mxv[i] = J.mxq;
    mxd[i] = J.mxp;
    usm[i] = uniform_u24(seed, step, (uint32_t)b, (uint32_t)i, kDrawSample);
    if (kEarly) {
      if (J.bad & SV_ROW_NAN) nan_bits |= 1u << c;
      if (J.bad & SV_ROW_BAD_TOKEN) tokbad_bits |= 1u << c;
    } else {
      bad |= J.bad;
    }
    if (J.bad & SV_ROW_BAD_TOKEN) continue;
    if (J.accept && !(kEarly && J.bad)) acc_bits |= 1u << c;
    if (J.p_zero) pzero_bits |= 1u << c;
    if (o.q_prob) o.q_prob[(size_t)b * r.maxpos + i] = J.qd;
    if (o.p_prob) o.p_prob[(size_t)b * r.maxpos + i] = J.pd;
    if (o.margin) o.margin[(size_t)b * (r.maxpos + 1) + i] = J.rc - (float)J.u24 * 0x1p-24f;
  }
  bad = __reduce_or_sync(FULL, bad);
  if (tree_bad) bad = SV_ROW_BAD_TREE;

  // first rejection (early exit: first rejection or fault)
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
      if (kEarly && !tree_bad) {
        const int la = a - c * 32;
        const uint32_t nb = __shfl_sync(FULL, nan_bits >> c, la) & 1u;
        const uint32_t tb = __shfl_sync(FULL, tokbad_bits >> c, la) & 1u;
        bad = (nb ? SV_ROW_NAN : 0u) | (tb ? SV_ROW_BAD_TOKEN : 0u);
      }
      break;
    }
    pz |= pzc;
  }
  if (kEarly && !tree_bad && a == npos) bad = bonus_bad;
  if (bad) a = 0;

  // outputs
  const int W = r.maxpos + 1;
  for (int i = lane; i < W; i += 32) {
    int32_t t = -1;
    if (!bad && i < a) t = r.tok[(size_t)b * r.tok_stride + i];
    o.tokens[(size_t)b * W + i] = t;
    if (o.path_out) o.path_out[(size_t)b * W + i] = (i == 0) ? 0 : ((!bad && i <= a) ? round_node(r, b, i) : -1);
    if (i >= npos || bad || (kEarly && i > a)) {
      if (i < r.maxpos) {
        if (o.q_prob) o.q_prob[(size_t)b * r.maxpos + i] = NAN;
        if (o.p_prob) o.p_prob[(size_t)b * r.maxpos + i] = NAN;
      }
      if (o.margin) o.margin[(size_t)b * W + i] = NAN;
    }
  }
  __syncwarp();
  if (lane == 0) {
    o.accept_len[b] = a;
    o.status[b] = bad ? bad : (pz ? SV_ROW_P_ZERO : 0u);
    Task t;
    t.active = bad ? 0 : 1;
    t.a = a;
    t.pad = 0;
    const int vi = a < npos ? a : npos;
    t.rq = used_row<E>(r, b, vi, src_row<E>(r, b, vi));
    t.rp = a < npos ? used_row<E>(r, b, r.maxpos + 1 + a, src_row<E>(r, b, r.maxpos + 1 + a))
                    : nullptr;
    t.mq = bad ? 0.0f : mxv[vi];
    t.mp = (!bad && a < npos) ? mxd[a] : 0.0f;
    t.u24 = bad ? 0u : usm[vi];
    tasks[b] = t;
    done[b] = 0u;        // the sampler's per-sequence completion counts:
    done[r.B + b] = 0u;  // slice CTAs of sample_mass, of sample_norm
  }
}

// ---------------------------------------------------------------------------
// row_stats in early-exit order (chain, T > 0): the walk ends at the first
// rejection ([Lesson] Passo 3; [Blog] section 4 spec_decode), so rows after it
// need not be read.  One CTA per (position i, sequence b, row, segment), in
// position-major order: the rows of position i of a sequence are scheduled a
// whole position-wave (2 B G CTAs) after those of position i - 1, by which
// time that position has usually been judged.  The CTA completing the 2G
// segments of position i (a per-position count; nothing waits on it) judges
// it with the accept walk's own function on the same partials and, on a
// rejection or a fault, lowers stop[b] to i.  A CTA that finds stop[b] < i
// reads nothing and writes a NaN partial, so a walk that ever reached such a
// row would fault instead of using stale statistics.  The bonus row
// (position N) is read unless the sequence stopped before it.
constexpr unsigned kEeInit = 0x7F7F7F7Fu;  // counts and stop[] start here (byte fill)

template <typename E, bool kCopy>
__global__ void __launch_bounds__(kRsThreads, sizeof(E) == 2 ? 10 : 8)
row_stats_ee_kernel(Round r, int G, float4 *__restrict__ partial, unsigned *__restrict__ count,
                    int *__restrict__ stop, uint64_t seed, uint64_t step) {
  grid_dep_sync();
  const int N = r.maxpos;
  const long long wave = 2LL * r.B * G;  // CTAs per drafted position
  const long long x = blockIdx.x;
  int i, b, j, seg;
  if (x < wave * N) {
    i = (int)(x / wave);
    const int rem = (int)(x - (long long)i * wave);
    b = rem / (2 * G);
    const int k = rem - b * 2 * G;
    seg = k < G ? k : k - G;
    j = k < G ? i : N + 1 + i;
  } else {
    i = N;
    const int rem = (int)(x - wave * N);
    b = rem / G;
    seg = rem - b * G;
    j = N;
  }
  __shared__ int skip;
  if (threadIdx.x == 0) skip = *(volatile int *)(stop + b) < i;
  __syncthreads();
  if (skip) {
    if (threadIdx.x == 0)
      partial[((size_t)b * r.P + j) * G + seg] = make_float4(NAN, NAN, NAN, NAN);
    return;
  }
  stat_segment<E, kCopy>(r, G, nullptr, b * r.P + j, seg, partial);
  // thread 0 wrote this segment's partial; the position's last CTA judges it
  if (i == N || threadIdx.x != 0) return;
  __threadfence();
  if (atomicAdd(count + (size_t)b * N + i, 1u) != kEeInit + 2u * (unsigned)G - 1u) return;
  __threadfence();
  const int d = r.tok[(size_t)b * r.tok_stride + i];
  // x_d from the source rows: a host-resident row's device copy is being
  // written by this kernel and is not read through the read-only path here
  const Judged J = judge_position<E, true>(r, G, partial + (size_t)b * r.P * G, b, i, d,
                                           src_row<E>(r, b, i), src_row<E>(r, b, N + 1 + i),
                                           seed, step);
  if (J.bad || !J.accept) atomicMin(stop + b, i);
}

// ---------------------------------------------------------------------------
// Greedy verification (temperature 0): the T -> 0 limit of the accept rule.
// row_argmax: per (verifier row, segment) the maximum, its lowest index and
// fault flags; decide_greedy: one warp per sequence accepts while the draft
// token is the row's arg max and emits the arg max where the walk stops.
// Only verifier rows are read; nothing is sampled.
constexpr uint32_t kArgNan = 1u;   // a NaN or +inf logit
constexpr uint32_t kArgSeen = 2u;  // a logit above -inf

struct ArgState {
  float best;  // running maximum (NaN ignored)
  int idx;     // lowest index holding it
  uint32_t flags;
};

__device__ __forceinline__ void arg1(ArgState &a, float x, int v) {
  if (x > a.best) {
    a.best = x;
    a.idx = v;
  }
  if (x != x || x == INFINITY) a.flags |= kArgNan;
  if (x > -INFINITY) a.flags |= kArgSeen;
}
// (best, idx) pairs: larger value wins, equal values go to the lower index
__device__ __forceinline__ void arg_merge(ArgState &a, float best, int idx, uint32_t flags) {
  if (best > a.best || (best == a.best && idx < a.idx)) {
    a.best = best;
    a.idx = idx;
  }
  a.flags |= flags;
}

// one 16-byte word of logits starting at element v; the word's maximum is
// taken on packed pairs first and the elements are scanned only when it
// beats the running maximum (in index order, so the lowest index is kept)
template <typename E>
__device__ __forceinline__ void arg_word(ArgState &a, uint4 w, int v);
template <>
__device__ __forceinline__ void arg_word<uint16_t>(ArgState &a, uint4 w, int v) {
  const uint32_t m = bf2_max(bf2_max(w.x, w.y), bf2_max(w.z, w.w));
  const uint32_t mn = bf2_max_nan(bf2_max_nan(w.x, w.y), bf2_max_nan(w.z, w.w));
  const float wm = fmaxf(bf16_lo(m), bf16_hi(m));
  const float n0 = bf16_lo(mn), n1 = bf16_hi(mn);  // NaN in either half: a NaN element
  if (n0 != n0 || n1 != n1 || wm == INFINITY) a.flags |= kArgNan;
  if (wm > -INFINITY) a.flags |= kArgSeen;
  if (wm > a.best) {
    const uint32_t q[4] = {w.x, w.y, w.z, w.w};
    int k = 7;
#pragma unroll
    for (int j = 7; j >= 0; --j) {
      const float x = (j & 1) ? bf16_hi(q[j >> 1]) : bf16_lo(q[j >> 1]);
      if (x == wm) k = j;
    }
    a.best = wm;
    a.idx = v + k;
  }
}
template <>
__device__ __forceinline__ void arg_word<float>(ArgState &a, uint4 w, int v) {
  const float x[4] = {__uint_as_float(w.x), __uint_as_float(w.y), __uint_as_float(w.z),
                      __uint_as_float(w.w)};
#pragma unroll
  for (int j = 0; j < 4; ++j) arg1(a, x[j], v + j);
}

template <typename E>
__device__ __forceinline__ void argmax_segment(const Round &r, int G, const int32_t *rowlist,
                                               int row_i, float4 *partial) {
  const int seg = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const SegInfo si = seg_info<E>(r, G, rowlist, row_i, seg);
  const E *row = (const E *)si.row;
  ArgState a{-INFINITY, 0x7fffffff, 0u};
  const int nhead = (int)((si.ab - (uintptr_t)(row + si.v0)) / sizeof(E));
  const int ntail = (int)(((uintptr_t)(row + si.v1) - si.ae) / sizeof(E));
  const int vbody = si.v0 + nhead;  // element index of the body's first word
  if (tid < nhead) arg1(a, load_elem<E>(row + si.v0 + tid), si.v0 + tid);
  const uint4 *body = (const uint4 *)si.ab;
  const int nv = (int)((si.ae - si.ab) / 16);
  constexpr int kPer = 16 / (int)sizeof(E);
  int i = tid;
  if (r.stage && i + (2 * kRsUnroll - 1) * kRsThreads < nv) {
    // as row_stats: the second half of the thread's words through shared
    // memory; words are still taken in increasing index order
    __shared__ uint4 sbuf[kRsUnroll][kRsThreads];
#pragma unroll
    for (int j = 0; j < kRsUnroll; ++j)
      cp_async16(&sbuf[j][tid], body + i + (kRsUnroll + j) * kRsThreads);
    cp_async_commit();
    uint4 buf[kRsUnroll];
#pragma unroll
    for (int j = 0; j < kRsUnroll; ++j) buf[j] = ld_stream_v4(body + i + j * kRsThreads);
#pragma unroll
    for (int j = 0; j < kRsUnroll; ++j) arg_word<E>(a, buf[j], vbody + (i + j * kRsThreads) * kPer);
    cp_async_wait_all();
#pragma unroll
    for (int j = 0; j < kRsUnroll; ++j)
      arg_word<E>(a, sbuf[j][tid], vbody + (i + (kRsUnroll + j) * kRsThreads) * kPer);
    i += 2 * kRsUnroll * kRsThreads;
  }
  for (; i + (kRsUnroll - 1) * kRsThreads < nv; i += kRsUnroll * kRsThreads) {
    uint4 buf[kRsUnroll];
#pragma unroll
    for (int j = 0; j < kRsUnroll; ++j) buf[j] = ld_stream_v4(body + i + j * kRsThreads);
#pragma unroll
    for (int j = 0; j < kRsUnroll; ++j) arg_word<E>(a, buf[j], vbody + (i + j * kRsThreads) * kPer);
  }
  for (; i < nv; i += kRsThreads) arg_word<E>(a, ld_stream_v4(body + i), vbody + i * kPer);
  if (tid < ntail) arg1(a, load_elem<E>((const E *)si.ae + tid), vbody + nv * kPer + tid);
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, a.best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, a.idx, o);
    const uint32_t of = __shfl_xor_sync(0xffffffffu, a.flags, o);
    arg_merge(a, ob, oi, of);
  }
  __shared__ float4 red[kRsThreads / 32];
  if (lane == 0) red[warp] = make_float4(a.best, __int_as_float(a.idx), __uint_as_float(a.flags), 0.f);
  __syncthreads();
  if (warp == 0) {
    const float4 v = lane < kRsThreads / 32 ? red[lane]
                                            : make_float4(-INFINITY, __int_as_float(0x7fffffff),
                                                          0.0f, 0.0f);
    ArgState c{v.x, __float_as_int(v.y), __float_as_uint(v.z)};
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, c.best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, c.idx, o);
      const uint32_t of = __shfl_xor_sync(0xffffffffu, c.flags, o);
      arg_merge(c, ob, oi, of);
    }
    if (lane == 0)
      partial[si.out] = make_float4(c.best, __int_as_float(c.idx), __uint_as_float(c.flags), 0.f);
  }
  __syncthreads();  // red[] is reused by the CTA's next row
}

template <typename E>
__global__ void __launch_bounds__(kRsThreads, sizeof(E) == 2 ? 10 : 8)
row_argmax_kernel(Round r, int G, const int32_t *__restrict__ rowlist,
                  const int32_t *__restrict__ rowcount, float4 *__restrict__ partial) {
  grid_dep_sync();
  const int nrows = rowlist ? *rowcount : (int)gridDim.x;
  for (int row_i = blockIdx.x; row_i < nrows; row_i += gridDim.x)
    argmax_segment<E>(r, G, rowlist, row_i, partial);
}

// arg max of verifier row slot j of sequence b from its G segment partials
__device__ __forceinline__ ArgState merge_arg(const float4 *part, int G) {
  ArgState a{-INFINITY, 0x7fffffff, 0u};
  for (int g = 0; g < G; ++g) {
    const float4 v = part[g];
    arg_merge(a, v.x, __float_as_int(v.y), __float_as_uint(v.z));
  }
  return a;
}
__device__ __forceinline__ bool arg_bad(const ArgState &a) {
  return (a.flags & kArgNan) || !(a.flags & kArgSeen);
}

__global__ void __launch_bounds__(kDecideWarps * 32)
decide_greedy_kernel(Round r, int G, const float4 *__restrict__ partial, DecideOut o) {
  grid_dep_sync();
  const int b = blockIdx.x * kDecideWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= r.B) return;
  const unsigned FULL = 0xffffffffu;
  const int npos = round_npos(r, b);
  const uint32_t tree_bad = r.tstat ? r.tstat[b] : 0u;
  const float4 *pb = partial + (size_t)b * r.P * G;
  extern __shared__ int am_sm[];  // per warp: arg max of row slot j, j <= maxpos
  int *am = am_sm + (threadIdx.x >> 5) * (r.maxpos + 1);
  uint32_t bad = 0, rej_bits = 0;
  if (lane == 0 && !tree_bad) {
    const ArgState a = merge_arg(pb + (size_t)npos * G, G);
    if (arg_bad(a)) bad |= SV_ROW_NAN;
    am[npos] = a.idx;
  }
  const int nchunks = (npos + 31) / 32;
  for (int c = 0; c < nchunks && !tree_bad; ++c) {
    const int i = c * 32 + lane;
    if (i >= npos) break;
    const int d = r.tok[(size_t)b * r.tok_stride + i];
    const ArgState a = merge_arg(pb + (size_t)i * G, G);
    am[i] = a.idx;
    if (arg_bad(a)) bad |= SV_ROW_NAN;
    if (d < 0 || d >= r.V) bad |= SV_ROW_BAD_TOKEN;
    if (d != a.idx) rej_bits |= 1u << c;
    if (o.q_prob) o.q_prob[(size_t)b * r.maxpos + i] = (d == a.idx) ? 1.0f : 0.0f;
  }
  bad = __reduce_or_sync(FULL, bad);
  if (tree_bad) bad = SV_ROW_BAD_TREE;
  int a = npos;
  for (int c = 0; c < nchunks; ++c) {
    const int i = c * 32 + lane;
    const unsigned rej = __ballot_sync(FULL, i < npos && ((rej_bits >> c) & 1u));
    if (rej) {
      a = c * 32 + __ffs(rej) - 1;
      break;
    }
  }
  if (bad) a = 0;
  __syncwarp();
  const int W = r.maxpos + 1;
  for (int i = lane; i < W; i += 32) {
    int32_t t = -1;
    if (!bad && i < a) t = r.tok[(size_t)b * r.tok_stride + i];
    if (!bad && i == a) t = am[a];
    o.tokens[(size_t)b * W + i] = t;
    if (o.path_out)
      o.path_out[(size_t)b * W + i] = (i == 0) ? 0 : ((!bad && i <= a) ? round_node(r, b, i) : -1);
    if (i < r.maxpos) {
      if (o.p_prob) o.p_prob[(size_t)b * r.maxpos + i] = NAN;
      if (o.q_prob && (i >= npos || bad)) o.q_prob[(size_t)b * r.maxpos + i] = NAN;
    }
    if (o.margin) o.margin[(size_t)b * W + i] = NAN;
  }
  if (lane == 0) {
    o.accept_len[b] = a;
    o.status[b] = bad;
  }
}

// ---------------------------------------------------------------------------
// The sampling arithmetic (fixed sequence of IEEE fp32 operations + exact
// 64-bit fixed point), shared by specification with the CPU oracle:
//   z = fl(x * invT); e = exp32_repro(fl(z - max z)); S_e = sum floor(e 2^40)
//   inv_s = fl32(2^40 / fl64(S_e)); q = fl(e * inv_s)
//   w = max(0, fl(q - p)) (residual) or q (bonus); W = floor(w 2^62)
//   t = floor(u24 * sum W / 2^24); token = min{k : sum_{v<=k} W_v > t}
// Only scalar _rn intrinsics are used where a product feeds a sum, so no
// multiply can be fused into a later add.
//
// Exact sums without 64-bit conversions (slow on this GPU): a value v in
// [0, 1] splits exactly into parts on fixed grids -- a = v truncated to a
// multiple of 2^-16 (an add rounding toward zero onto 2^7, minus 2^7), then
// the remainder truncated to 2^-32, and so on.  Parts of up to 128 values sum
// exactly in fp32 (each part fits 17 bits, 7 more bits of headroom); the
// per-thread part sums become integers once and meet in uint64.  The result is
// sum floor(v 2^40) (three parts) or sum floor(v 2^62) (four parts) exactly.
//
// Two kernels per round.  A CTA owns one kSpSlice-element slice of one
// sequence's q row (and p row for a residual); thread t owns the kSpRun
// consecutive elements [t * kSpRun, (t + 1) * kSpRun) of the slice:
//   sample_norm  partial sums of floor(e 2^40) of the slice; the CTA that
//                completes a sequence's slices last (a per-sequence count)
//                computes 1/S_e of the q and p rows once
//   sample_mass  W of every element; the sum of each thread's run is stored
//                (the prefix search's blocks)
// Both evaluate the exponentials and the splits on packed fp32 pairs: the q
// and p element of one position (residual), or two neighbouring q elements
// (bonus), one per lane.
//   (pick)       in the CTA that finishes a sequence's masses last, one warp:
//                the threshold, the slice, the run, then a warp scan of the
//                run's 32 elements

struct Parts40 {
  float a, b, c;  // multiples of 2^-16, 2^-32, 2^-40
};
struct Parts62 {
  float a, b, c, d;  // multiples of 2^-16, 2^-32, 2^-48, 2^-62
};
__device__ __forceinline__ unsigned long long fix_of(const Parts40 &P) {
  return (unsigned long long)__float2uint_rn(__fmul_rn(P.a, 0x1p16f)) * (1ull << 24) +
         (unsigned long long)__float2uint_rn(__fmul_rn(P.b, 0x1p32f)) * (1ull << 8) +
         (unsigned long long)__float2uint_rn(__fmul_rn(P.c, 0x1p40f));
}
__device__ __forceinline__ unsigned long long fix_of(const Parts62 &P) {
  return (unsigned long long)__float2uint_rn(__fmul_rn(P.a, 0x1p16f)) * (1ull << 46) +
         (unsigned long long)__float2uint_rn(__fmul_rn(P.b, 0x1p32f)) * (1ull << 30) +
         (unsigned long long)__float2uint_rn(__fmul_rn(P.c, 0x1p48f)) * (1ull << 14) +
         (unsigned long long)__float2uint_rn(__fmul_rn(P.d, 0x1p62f));
}
// single values (the final scan only)
__device__ __forceinline__ unsigned long long fix62(float w) {
  return __float2ull_rz(__fmul_rn(w, 0x1p62f));
}
__device__ __forceinline__ float inv_sum(unsigned long long se) {
  return __double2float_rn(__ddiv_rn(0x1p40, __ull2double_rn(se)));
}

// A thread's run of kSpRun consecutive logits of one row, kept as the raw
// 16-byte words (bf16 pairs or fp32) and converted element by element when
// used.  Elements past the row's end read as -inf, whose exponential is 0.
template <typename E>
struct Run;
template <>
struct Run<uint16_t> {
  uint4 w[kSpRun / 8];
  __device__ __forceinline__ float operator[](int j) const {
    const uint4 &q = w[j >> 3];
    const int c = (j >> 1) & 3;
    const uint32_t x = c == 0 ? q.x : c == 1 ? q.y : c == 2 ? q.z : q.w;
    return (j & 1) ? bf16_hi(x) : bf16_lo(x);
  }
};
template <>
struct Run<float> {
  uint4 w[kSpRun / 4];
  __device__ __forceinline__ float operator[](int j) const {
    const uint4 &q = w[j >> 2];
    const int c = j & 3;
    return __uint_as_float(c == 0 ? q.x : c == 1 ? q.y : c == 2 ? q.z : q.w);
  }
};

template <typename E>
__device__ __forceinline__ void load_run(Run<E> &run, const E *row, int v, int V, bool vec) {
  constexpr int kPer = 16 / sizeof(E);  // elements per word
  if (vec && v + kSpRun <= V) {
    const uint4 *p = (const uint4 *)(row + v);
#pragma unroll
    for (int k = 0; k < kSpRun / kPer; ++k) run.w[k] = __ldg(p + k);
    return;
  }
  // ragged or unaligned run: element by element
  uint32_t bits[kSpRun];
#pragma unroll
  for (int j = 0; j < kSpRun; ++j) {
    const bool in = v + j < V;
    if (sizeof(E) == 2)
      bits[j] = in ? (uint32_t)__ldg((const unsigned short *)row + v + j) : 0xff80u;
    else
      bits[j] = in ? __float_as_uint(__ldg((const float *)row + v + j)) : 0xff800000u;
  }
#pragma unroll
  for (int k = 0; k < kSpRun / kPer; ++k) {
    uint32_t q[4];
#pragma unroll
    for (int c = 0; c < 4; ++c)
      q[c] = sizeof(E) == 2 ? (bits[8 * k + 2 * c] | (bits[8 * k + 2 * c + 1] << 16))
                            : bits[4 * k + c];
    run.w[k] = make_uint4(q[0], q[1], q[2], q[3]);
  }
}

// packed exponent arguments fl(fl(x * invT) - mz) of two elements (the
// multiply is skipped at T = 1; scalar where a multiply is involved)
__device__ __forceinline__ unsigned long long arg2(float x0, float x1, float m0, float m1,
                                                   float invT, bool unit_t) {
  if (unit_t) return f2_sub(f2_pack(x0, x1), f2_pack(m0, m1));
  return f2_pack(__fsub_rn(__fmul_rn(x0, invT), m0), __fsub_rn(__fmul_rn(x1, invT), m1));
}

// split-part accumulation of a packed pair (each lane as add40 / add62)
struct Parts40x2 {
  unsigned long long a, b, c;
};
struct Parts62x2 {
  unsigned long long a, b, c, d;
};
__device__ __forceinline__ unsigned long long trunc2(unsigned long long v, float grid_top) {
  const unsigned long long g = f2_splat(grid_top);
  return f2_sub(f2_add_rz(v, g), g);
}
__device__ __forceinline__ void add40x2(Parts40x2 &P, unsigned long long e) {
  const unsigned long long a = trunc2(e, 0x1p7f);
  const unsigned long long r1 = f2_sub(e, a);
  const unsigned long long b = trunc2(r1, 0x1p-9f);
  const unsigned long long r2 = f2_sub(r1, b);
  const unsigned long long c = trunc2(r2, 0x1p-17f);
  P.a = f2_add(P.a, a);
  P.b = f2_add(P.b, b);
  P.c = f2_add(P.c, c);
}
__device__ __forceinline__ void add62x2(Parts62x2 &P, unsigned long long w) {
  const unsigned long long a = trunc2(w, 0x1p7f);
  const unsigned long long r1 = f2_sub(w, a);
  const unsigned long long b = trunc2(r1, 0x1p-9f);
  const unsigned long long r2 = f2_sub(r1, b);
  const unsigned long long c = trunc2(r2, 0x1p-25f);
  const unsigned long long r3 = f2_sub(r2, c);
  const unsigned long long d = trunc2(r3, 0x1p-39f);
  P.a = f2_add(P.a, a);
  P.b = f2_add(P.b, b);
  P.c = f2_add(P.c, c);
  P.d = f2_add(P.d, d);
}
// the two lanes' exact sums
__device__ __forceinline__ void fix_lanes(const Parts40x2 &P, unsigned long long &s0,
                                          unsigned long long &s1) {
  Parts40 l0, l1;
  f2_unpack(P.a, l0.a, l1.a);
  f2_unpack(P.b, l0.b, l1.b);
  f2_unpack(P.c, l0.c, l1.c);
  s0 = fix_of(l0);
  s1 = fix_of(l1);
}
__device__ __forceinline__ unsigned long long fix_sum(const Parts62x2 &P) {
  Parts62 l0, l1;
  f2_unpack(P.a, l0.a, l1.a);
  f2_unpack(P.b, l0.b, l1.b);
  f2_unpack(P.c, l0.c, l1.c);
  f2_unpack(P.d, l0.d, l1.d);
  return fix_of(l0) + fix_of(l1);
}

__device__ __forceinline__ float e1(float x, float invT, float mz, bool unit_t) {
  const float z = unit_t ? x : __fmul_rn(x, invT);
  return exp32_repro(__fsub_rn(z, mz));
}

struct SampleWs {
  ulonglong2 *norm;          // [B][CS] partial (sum floor(e_q 2^40), sum floor(e_p 2^40))
  unsigned long long *mass;  // [B][CS] slice sum W
  unsigned long long *run;   // [B][CS][kSpThreads] run sums of W
  unsigned *done;            // [2][B] slice CTAs of sample_mass / sample_norm finished
                             // (zeroed by decide)
  float2 *inv;               // [B] (1/S_e of q, of p) from the last sample_norm CTA
  int CS;                    // slices per row
  int B;
};

struct RowPair {
  const void *rq, *rp;
  float mzq, mzp;
  bool resid, vec, unit_t;
};

template <typename E>
__device__ __forceinline__ RowPair row_pair(const Round &r, const Task &t) {
  RowPair p;
  p.resid = t.rp != nullptr;
  const E *rq = (const E *)t.rq;
  const E *rp = p.resid ? (const E *)t.rp : rq;
  p.rq = rq;
  p.rp = rp;
  p.mzq = __fmul_rn(t.mq, r.invT);
  p.mzp = __fmul_rn(t.mp, r.invT);
  p.vec = ((((uintptr_t)rq) | ((uintptr_t)rp)) & 15) == 0;
  p.unit_t = r.invT == 1.0f;
  return p;
}

__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long v,
                                                            unsigned long long *red) {
  v = warp_sum_u64(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  unsigned long long tot = 0;
  if (threadIdx.x == 0)
    for (int i = 0; i < kSpWarps; ++i) tot += red[i];
  __syncthreads();
  return tot;  // valid on thread 0
}

// S_e of the q and p rows of sequence b -> 1 / sum, by one thread
__device__ __forceinline__ void inv_sums(const SampleWs &sw, int b, bool resid, float &iq,
                                         float &ip) {
  unsigned long long Sq = 0, Sp = 0;
  for (int c = 0; c < sw.CS; ++c) {
    const ulonglong2 n = __ldcg(sw.norm + (size_t)b * sw.CS + c);  // other CTAs' sums
    Sq += n.x;
    Sp += n.y;
  }
  iq = inv_sum(Sq);
  ip = resid ? inv_sum(Sp) : 0.0f;
}

template <typename E>
__global__ void __launch_bounds__(kSpThreads, sizeof(E) == 2 ? 8 : 4)
sample_norm_kernel(Round r, const Task *__restrict__ tasks, SampleWs sw) {
  grid_dep_sync();
  const int b = blockIdx.x / sw.CS, cs = blockIdx.x - b * sw.CS;
  const Task t = tasks[b];
  if (!t.active) return;
  const RowPair p = row_pair<E>(r, t);
  const int v = cs * kSpSlice + kSpRun * threadIdx.x;
  Run<E> rq;
  load_run<E>(rq, (const E *)p.rq, v, r.V, p.vec);
  Parts40x2 P{0ull, 0ull, 0ull};
  unsigned long long fq, fp;
  if (p.resid) {  // lanes (q row, p row) of the same element
    Run<E> rp;
    load_run<E>(rp, (const E *)p.rp, v, r.V, p.vec);
#pragma unroll
    for (int j = 0; j < kSpRun; ++j)
      add40x2(P, exp32x2(arg2(rq[j], rp[j], p.mzq, p.mzp, r.invT, p.unit_t)));
    fix_lanes(P, fq, fp);
  } else {  // lanes (element j, element j + 1) of the q row
#pragma unroll
    for (int j = 0; j < kSpRun; j += 2)
      add40x2(P, exp32x2(arg2(rq[j], rq[j + 1], p.mzq, p.mzq, r.invT, p.unit_t)));
    unsigned long long f1;
    fix_lanes(P, fq, f1);
    fq += f1;
    fp = 0ull;
  }
  __shared__ unsigned long long red[kSpWarps];
  const unsigned long long sq = block_sum_u64(fq, red);
  const unsigned long long sp = block_sum_u64(fp, red);
  if (threadIdx.x == 0) {
    // the last slice CTA of the sequence turns the slice sums into 1/S_e
    sw.norm[blockIdx.x] = make_ulonglong2(sq, sp);
    __threadfence();
    if (atomicAdd(sw.done + sw.B + b, 1u) == (unsigned)(sw.CS - 1)) {
      __threadfence();
      float iq, ip;
      inv_sums(sw, b, p.resid, iq, ip);
      sw.inv[b] = make_float2(iq, ip);
    }
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

// first index i in [0, n) where the running sum of get(i) exceeds thr;
// `base` gets the sum before it.  One warp, uniform result.
template <typename F>
__device__ __forceinline__ int warp_find(int n, unsigned long long thr, F get,
                                         unsigned long long &base) {
  base = 0;
  for (int c0 = 0; c0 < n; c0 += 32) {
    const int c = c0 + (threadIdx.x & 31);
    const unsigned long long v = c < n ? get(c) : 0ull;
    const unsigned long long inc = warp_incl_scan_u64(v) + base;
    const unsigned hit = __ballot_sync(0xffffffffu, c < n && inc > thr);
    if (hit) {
      const int l = __ffs(hit) - 1;
      base = __shfl_sync(0xffffffffu, inc - v, l);
      return c0 + l;
    }
    base = __shfl_sync(0xffffffffu, inc, 31);
  }
  return n - 1;  // not reached when thr < total
}

// W (or the q mass) of one element
template <typename E>
__device__ __forceinline__ unsigned long long w_elem(const Round &r, const RowPair &p, int v,
                                                     float iq, float ip, bool use_q) {
  if (v >= r.V) return 0ull;
  const float q = __fmul_rn(e1(load_elem<E>((const E *)p.rq + v), r.invT, p.mzq, p.unit_t), iq);
  if (use_q) return fix62(q);
  const float d = __fsub_rn(
      q, __fmul_rn(e1(load_elem<E>((const E *)p.rp + v), r.invT, p.mzp, p.unit_t), ip));
  return fix62(d > 0.0f ? d : 0.0f);
}


// The inverse-CDF pick of sequence b, by one warp (the last sample_mass CTA
// of the sequence; the other CTAs' masses are read through L2).
template <typename E>
__device__ __forceinline__ void pick_sequence(const Round &r, const Task &t, const RowPair &p,
                                              const SampleWs &sw, const DecideOut &o, int b) {
  const int lane = threadIdx.x & 31;
  const float2 iv = sw.inv[b];
  const float iq = iv.x, ip = iv.y;
  const unsigned long long *mass = sw.mass + (size_t)b * sw.CS;
  unsigned long long Sw = 0;
  for (int c0 = 0; c0 < sw.CS; c0 += 32)  // one load per lane, then a warp sum
    Sw += warp_sum_u64(c0 + lane < sw.CS ? __ldcg(mass + c0 + lane) : 0ull);
  // residual mass 0 (q == p to the last bit): fall back to q; its masses are
  // recomputed here (a warp per slice / run), which only this case needs
  const bool use_q = !p.resid || Sw == 0ull;
  const bool fallback = p.resid && use_q;
  auto run_mass = [&](int c, int th) -> unsigned long long {  // one lane, one run
    unsigned long long m = 0;
    const int v0 = c * kSpSlice + kSpRun * th;
    for (int j = 0; j < kSpRun; ++j) m += w_elem<E>(r, p, v0 + j, iq, ip, true);
    return m;
  };
  auto slice_mass = [&](int c) -> unsigned long long {  // one lane, one slice
    unsigned long long m = 0;
    for (int th = 0; th < kSpThreads; ++th) m += run_mass(c, th);
    return m;
  };
  unsigned long long S = Sw;
  if (fallback) {
    S = 0;
    for (int c0 = 0; c0 < sw.CS; c0 += 32) {
      const unsigned long long m = (c0 + lane < sw.CS) ? slice_mass(c0 + lane) : 0ull;
      S += warp_sum_u64(m);
    }
  }
  const unsigned long long thr =
      (__umul64hi((unsigned long long)t.u24, S) << 40) | (((unsigned long long)t.u24 * S) >> 24);
  unsigned long long base_s, base_r;
  const int cs = warp_find(sw.CS, thr,
                           [&](int c) { return fallback ? slice_mass(c) : __ldcg(mass + c); },
                           base_s);
  const unsigned long long *run = sw.run + ((size_t)b * sw.CS + cs) * kSpThreads;
  const unsigned long long tl = thr - base_s;
  int ri;
  if (fallback) {
    ri = warp_find(kSpThreads, tl, [&](int th) { return run_mass(cs, th); }, base_r);
  } else {
    // the slice's run sums: lane l loads runs [8l, 8l + 8) at once, the warp
    // finds the lane whose group crosses the threshold, that lane the run
    constexpr int kPer = kSpThreads / 32;
    unsigned long long rs[kPer], own = 0;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      rs[k] = __ldcg(run + lane * kPer + k);
      own += rs[k];
    }
    const unsigned long long inc = warp_incl_scan_u64(own);
    const unsigned hit = __ballot_sync(0xffffffffu, inc > tl);
    const int lh = hit ? __ffs(hit) - 1 : 31;  // tl < slice mass: some lane crosses
    // this lane's group: the first run whose running sum crosses tl
    unsigned long long run_acc = inc - own, base_k = run_acc;
    int k_hit = kPer - 1;
    bool found = false;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      if (!found && run_acc + rs[k] > tl) {
        found = true;
        k_hit = k;
        base_k = run_acc;
      }
      run_acc += rs[k];
    }
    ri = __shfl_sync(0xffffffffu, lane * kPer + k_hit, lh);
    base_r = __shfl_sync(0xffffffffu, base_k, lh);
  }
  // the run's 32 elements, one per lane
  const int v = cs * kSpSlice + kSpRun * ri + lane;
  const unsigned long long w = w_elem<E>(r, p, v, iq, ip, use_q);
  const unsigned long long tb = tl - base_r;
  const unsigned long long inc = warp_incl_scan_u64(w);
  const unsigned hit = __ballot_sync(0xffffffffu, inc > tb);
  const int l = __ffs(hit) - 1;
  if (lane == l) {
    const unsigned long long c = inc - w;
    const unsigned long long b_lo = tb - c, b_hi = c + w - 1ull - tb;
    const int Wd = r.maxpos + 1;
    o.tokens[(size_t)b * Wd + t.a] = v;
    if (o.margin)
      o.margin[(size_t)b * Wd + r.maxpos] =
          (float)((double)(b_lo < b_hi ? b_lo : b_hi) / (double)S);
    if (fallback) o.status[b] |= SV_ROW_RESID_ZERO;
  }
}

template <typename E>
__global__ void __launch_bounds__(kSpThreads, sizeof(E) == 2 ? 8 : 4)
sample_mass_kernel(Round r, const Task *__restrict__ tasks, SampleWs sw, DecideOut o) {
  grid_dep_sync();
  const int b = blockIdx.x / sw.CS, cs = blockIdx.x - b * sw.CS;
  const Task t = tasks[b];
  if (!t.active) return;
  const RowPair p = row_pair<E>(r, t);
  const int v = cs * kSpSlice + kSpRun * threadIdx.x;
  Run<E> rq, rp;
  load_run<E>(rq, (const E *)p.rq, v, r.V, p.vec);
  if (p.resid) load_run<E>(rp, (const E *)p.rp, v, r.V, p.vec);
  const float2 iv = sw.inv[b];  // written by sample_norm
  const float iq = iv.x, ip = iv.y;
  Parts62x2 P{0ull, 0ull, 0ull, 0ull};
  if (p.resid) {
#pragma unroll
    for (int j = 0; j < kSpRun; j += 2) {
      float q0, p0, q1, p1;
      f2_unpack(exp32x2(arg2(rq[j], rp[j], p.mzq, p.mzp, r.invT, p.unit_t)), q0, p0);
      f2_unpack(exp32x2(arg2(rq[j + 1], rp[j + 1], p.mzq, p.mzp, r.invT, p.unit_t)), q1, p1);
      const float d0 = __fsub_rn(__fmul_rn(q0, iq), __fmul_rn(p0, ip));
      const float d1 = __fsub_rn(__fmul_rn(q1, iq), __fmul_rn(p1, ip));
      add62x2(P, f2_pack(fmaxf(d0, 0.0f), fmaxf(d1, 0.0f)));
    }
  } else {
#pragma unroll
    for (int j = 0; j < kSpRun; j += 2) {
      float e0, e1;
      f2_unpack(exp32x2(arg2(rq[j], rq[j + 1], p.mzq, p.mzq, r.invT, p.unit_t)), e0, e1);
      // q >= 0; the max keeps the product out of the split's addition
      add62x2(P, f2_pack(fmaxf(__fmul_rn(e0, iq), 0.0f), fmaxf(__fmul_rn(e1, iq), 0.0f)));
    }
  }
  const unsigned long long mine = fix_sum(P);
  sw.run[(size_t)blockIdx.x * kSpThreads + threadIdx.x] = mine;
  __shared__ unsigned long long red[kSpWarps];
  const unsigned long long tot = block_sum_u64(mine, red);  // also a CTA barrier
  __shared__ int s_last;
  if (threadIdx.x == 0) {
    // the barrier above orders every thread's run store before this
    // thread's device-scope fence, which orders them (cumulatively) before
    // the count that the last CTA of the sequence observes
    sw.mass[blockIdx.x] = tot;
    __threadfence();
    s_last = atomicAdd(sw.done + b, 1u) == (unsigned)(sw.CS - 1);
  }
  __syncthreads();
  // the last slice CTA of the sequence picks the token
  if (s_last && threadIdx.x < 32) pick_sequence<E>(r, t, p, sw, o, b);
}

// ---------------------------------------------------------------------------
// tree_path: one warp per sequence.  Validates the tree, walks best children
// (highest score; ties to the lower slot) at most max_depth steps.
__global__ void __launch_bounds__(32)
tree_path_kernel(const int32_t *__restrict__ parent, const int32_t *__restrict__ token,
                 const float *__restrict__ score, int B, int T, int max_depth,
                 int32_t *__restrict__ path, int32_t *__restrict__ npos,
                 int32_t *__restrict__ tok, int tok_stride, uint32_t *__restrict__ tstat,
                 int32_t *__restrict__ rowlist, int *__restrict__ rowcount, int greedy) {
  grid_dep_sync();
  const int b = blockIdx.x, lane = threadIdx.x;
  __shared__ int32_t pa[SV_MAX_TREE_NODES];
  __shared__ float sc[SV_MAX_TREE_NODES];
  __shared__ int32_t tk[SV_MAX_TREE_NODES];
  __shared__ int32_t pn[SV_MAX_POSITIONS + 1];  // the path, written out at the end
  for (int c = lane; c < T; c += 32) {  // one coalesced pass over the tree
    pa[c] = parent[(size_t)b * T + c];
    sc[c] = score[(size_t)b * T + c];
    tk[c] = token[(size_t)b * T + c];
  }
  __syncwarp();
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
      rowlist[atomicAdd(rowcount, 1)] = b << 12;  // the root row only
    }
    return;
  }
  int cur = 0, D = 0;
  if (lane == 0) pn[0] = 0;
  while (D < max_depth) {
    bool have = false;
    float bs = 0.0f;
    int bi = 0x7fffffff;
    for (int c = 1 + lane; c < T; c += 32) {
      if (pa[c] != cur) continue;
      const float sv = sc[c];
      if (!have || sv > bs || (sv == bs && c < bi)) {
        have = true;
        bs = sv;
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
    if (lane == 0) pn[D] = bi;
  }
  __syncwarp();
  // the path and its tested tokens token[n_1..n_D], written in parallel
  for (int i = lane; i <= D; i += 32) pth[i] = pn[i];
  for (int i = lane; i < D; i += 32) tok[(size_t)b * tok_stride + i] = tk[pn[i + 1]];
  int base = 0;
  if (lane == 0) {
    npos[b] = D;
    tstat[b] = 0u;
    base = atomicAdd(rowcount, greedy ? D + 1 : 2 * D + 1);
  }
  base = __shfl_sync(0xffffffffu, base, 0);
  // the verifier rows n_0..n_D, then (stochastic rule) the draft rows
  const int nrow = greedy ? D + 1 : 2 * D + 1;
  for (int a = lane; a < nrow; a += 32) rowlist[base + a] = (b << 12) | a;
}

// ---------------------------------------------------------------------------
template <typename E>
sv_status run_verify(const Round &r, const Layout &L, char *ws, uint64_t seed, uint64_t step,
                     const DecideOut &o, cudaStream_t st, cudaEvent_t accept_event,
                     bool early = false) {
  float4 *partial = (float4 *)(ws + L.partial);
  Task *tasks = (Task *)(ws + L.task);
  sv_status s;
  // segments per row for this element type (the workspace holds L.G >= G)
  const int G = (r.V + seg_elems<E>() - 1) / seg_elems<E>();
  if (early) {
    // per-position counts [B][N] and stop [B], byte-filled to kEeInit
    unsigned *count = (unsigned *)(ws + L.ee);
    int *stop = (int *)(count + (size_t)r.B * r.maxpos);
    if (cudaMemsetAsync(count, 0x7F, sizeof(int) * (size_t)r.B * (r.maxpos + 1), st) !=
        cudaSuccess)
      return set_error(SV_ERR_CUDA, "row_stats_ee: count reset");
    const long long nblk = (long long)r.B * G * r.P;
    LaunchScope ls("row_stats_ee", st);
    s = check_launch("row_stats_ee", launch_pdl(r.copy ? row_stats_ee_kernel<E, true>
                                                       : row_stats_ee_kernel<E, false>,
                                                dim3((unsigned)nblk), dim3(kRsThreads), 0, st,
                                                r, G, partial, count, stop, seed, step));
    if (s != SV_OK) return s;
  } else {
    // tree: B * P row slots bound the listed rows; half as many CTAs per
    // segment, each taking a second row when the paths are deep
    const int32_t *rowlist = r.path ? (const int32_t *)(ws + L.rowlist) : nullptr;
    const unsigned gx = rowlist ? (unsigned)((r.B * r.P + 1) / 2) : (unsigned)(r.B * r.P);
    LaunchScope ls("row_stats", st);
    s = check_launch("row_stats", launch_pdl(r.copy ? row_stats_kernel<E, true>
                                                    : row_stats_kernel<E, false>,
                                             dim3(gx, (unsigned)G),
                                             dim3(kRsThreads), 0, st, r, G, rowlist,
                                             (const int *)(ws + L.ctr), partial));
    if (s != SV_OK) return s;
  }
  {
    // per warp: raw maxima of both rows and the sample uniform per position
    const size_t dsm = (size_t)kDecideWarps * 3 * (r.maxpos + 1) * sizeof(float);
    auto kern = early ? decide_kernel<E, true> : decide_kernel<E, false>;
    if (dsm > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dsm) !=
            cudaSuccess)
      return set_error(SV_ERR_CUDA, "decide: shared memory attribute");
    LaunchScope ls("decide", st);
    s = check_launch("decide", launch_pdl(kern,
                                          dim3((r.B + kDecideWarps - 1) / kDecideWarps),
                                          dim3(kDecideWarps * 32), dsm, st, r, G, partial, seed,
                                          step, o, tasks, (unsigned *)(ws + L.done)));
    if (s != SV_OK) return s;
  }
  if (accept_event) {
    const cudaError_t e = cudaEventRecord(accept_event, st);
    if (e != cudaSuccess) return set_error(SV_ERR_CUDA, "accept_event: %s", cudaGetErrorString(e));
  }
  SampleWs sw;
  sw.norm = (ulonglong2 *)(ws + L.norm);
  sw.mass = (unsigned long long *)(ws + L.mass);
  sw.run = (unsigned long long *)(ws + L.run);
  sw.done = (unsigned *)(ws + L.done);
  sw.inv = (float2 *)(ws + L.inv);
  sw.CS = L.CS;
  sw.B = r.B;
  const unsigned grid = (unsigned)((long)r.B * L.CS);
  {
    LaunchScope ls("sample_norm", st);
    s = check_launch("sample_norm", launch_pdl(sample_norm_kernel<E>, dim3(grid),
                                               dim3(kSpThreads), 0, st, r, tasks, sw));
    if (s != SV_OK) return s;
  }
  {
    LaunchScope ls("sample_mass", st);
    s = check_launch("sample_mass", launch_pdl(sample_mass_kernel<E>, dim3(grid),
                                               dim3(kSpThreads), 0, st, r, tasks, sw, o));
    if (s != SV_OK) return s;
  }
  return SV_OK;
}

template <typename E>
sv_status run_verify_greedy(const Round &r, const Layout &L, char *ws, const DecideOut &o,
                            cudaStream_t st, cudaEvent_t accept_event) {
  float4 *partial = (float4 *)(ws + L.partial);
  const int G = (r.V + seg_elems<E>() - 1) / seg_elems<E>();
  sv_status s;
  {
    const int32_t *rowlist = r.path ? (const int32_t *)(ws + L.rowlist) : nullptr;
    const unsigned gx = rowlist ? (unsigned)((r.B * r.P + 1) / 2) : (unsigned)(r.B * r.P);
    LaunchScope ls("row_argmax", st);
    s = check_launch("row_argmax", launch_pdl(row_argmax_kernel<E>, dim3(gx, (unsigned)G),
                                              dim3(kRsThreads), 0, st, r, G, rowlist,
                                              (const int *)(ws + L.ctr), partial));
    if (s != SV_OK) return s;
  }
  {
    const size_t dsm = (size_t)kDecideWarps * (r.maxpos + 1) * sizeof(int);
    LaunchScope ls("decide_greedy", st);
    s = check_launch("decide_greedy",
                     launch_pdl(decide_greedy_kernel, dim3((r.B + kDecideWarps - 1) / kDecideWarps),
                                dim3(kDecideWarps * 32), dsm, st, r, G, partial, o));
    if (s != SV_OK) return s;
  }
  if (accept_event) {
    const cudaError_t e = cudaEventRecord(accept_event, st);
    if (e != cudaSuccess) return set_error(SV_ERR_CUDA, "accept_event: %s", cudaGetErrorString(e));
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
  if (!(temperature >= 0.0f) || !isfinite(temperature))
    return set_error(SV_ERR_INVALID_ARG, "temperature must be finite and >= 0 (0 = greedy)");
  if (B == 0) return SV_OK;
  if (!vlogits || !out_tokens || !out_accept || !out_status || !workspace)
    return set_error(SV_ERR_INVALID_ARG, "null pointer argument");
  const size_t es = dt == SV_F32 ? 4 : 2;
  if ((uintptr_t)vlogits % es) return set_error(SV_ERR_INVALID_ARG, "vlogits misaligned");
  return SV_OK;
}

// grid sizes of the round's kernels must fit a 32-bit grid dimension
sv_status check_grid(int B, const Layout &L) {
  if ((long long)B * L.P > 0x7fffffffLL || (long long)B * L.CS > 0x7fffffffLL)
    return set_error(SV_ERR_UNSUPPORTED, "batch too large: B=%d", B);
  return SV_OK;
}

// Host-resident logits and a workspace with room for it: row_stats copies
// every row slot it reads into the workspace (one slot per (sequence, slot),
// pitch = the row rounded up to 16 bytes plus 16 for the source's offset
// within 16 bytes), and the accept walk and the sampler read the copies, so
// each row crosses the host link once.
size_t row_copy_pitch(int V, sv_dtype dt) {
  return align_up((size_t)V * (dt == SV_F32 ? 4 : 2), 16) + 16;
}
size_t row_copy_bytes(int B, const Layout &L, int V, sv_dtype dt) {
  return (size_t)B * L.P * row_copy_pitch(V, dt);
}
void set_row_copy(Round &r, const Layout &L, char *ws, size_t workspace_bytes, int B,
                  sv_dtype dt) {
  r.copy = nullptr;
  r.pitch = 0;
  if (!r.stage && workspace_bytes >= L.total + row_copy_bytes(B, L, r.V, dt)) {
    r.copy = ws + L.end;
    r.pitch = row_copy_pitch(r.V, dt);
  }
}

sv_status map_chain_args(const void *&vlogits, const void *&dlogits, const int32_t *&tokens,
                         int32_t *&out_tokens, int32_t *&out_accept_len, float *&out_q_prob,
                         float *&out_p_prob, float *&out_margin, uint32_t *&out_status) {
  sv_status s;
  if ((s = map_arg(vlogits, "vlogits")) != SV_OK || (s = map_arg(dlogits, "dlogits")) != SV_OK ||
      (s = map_arg(tokens, "tokens")) != SV_OK || (s = map_arg(out_tokens, "out_tokens")) != SV_OK ||
      (s = map_arg(out_accept_len, "out_accept_len")) != SV_OK ||
      (s = map_arg(out_q_prob, "out_q_prob")) != SV_OK ||
      (s = map_arg(out_p_prob, "out_p_prob")) != SV_OK ||
      (s = map_arg(out_margin, "out_margin")) != SV_OK ||
      (s = map_arg(out_status, "out_status")) != SV_OK)
    return s;
  return SV_OK;
}

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" size_t sv_verify_chain_workspace(int B, int N, int V) {
  if (B < 0 || N < 0 || V < 1) return 0;
  return plan(B, N, V, false).total;
}

extern "C" size_t sv_verify_chain_workspace_host(int B, int N, int V, sv_dtype dt) {
  if (B < 0 || N < 0 || V < 1 || (dt != SV_F32 && dt != SV_BF16)) return 0;
  const Layout L = plan(B, N, V, false);
  return L.total + row_copy_bytes(B, L, V, dt);
}

namespace sv {
namespace {
sv_status verify_chain(const void *vlogits, const void *dlogits, sv_dtype dt,
                       const int32_t *draft_tokens, int B, int N, int V, float temperature,
                       uint64_t seed, uint64_t step, int32_t *out_tokens,
                       int32_t *out_accept_len, float *out_q_prob, float *out_p_prob,
                       float *out_margin, uint32_t *out_status, void *workspace,
                       size_t workspace_bytes, void *stream, void *accept_event, bool early) {
  sv_status s = check_common(vlogits, dt, B, V, temperature, out_tokens, out_accept_len,
                             out_status, workspace);
  if (s != SV_OK) return s;
  if (early && temperature == 0.0f)
    return set_error(SV_ERR_UNSUPPORTED,
                     "early exit needs temperature > 0 (greedy reads only verifier rows)");
  if (B == 0) return s;
  if (N < 0) return set_error(SV_ERR_INVALID_ARG, "N must be >= 0 (got %d)", N);
  if (N > SV_MAX_POSITIONS) return set_error(SV_ERR_UNSUPPORTED, "N > %d", SV_MAX_POSITIONS);
  if (N > 0 && (!dlogits || !draft_tokens))
    return set_error(SV_ERR_INVALID_ARG, "dlogits and draft_tokens are required when N > 0");
  const Layout L = plan(B, N, V, false);
  if ((s = check_grid(B, L)) != SV_OK) return s;
  if (early && (long long)B * L.P * ((V + seg_elems<float>() - 1) / seg_elems<float>()) >
                   0x7fffffffLL)
    return set_error(SV_ERR_UNSUPPORTED, "batch too large for early exit: B=%d", B);
  if (workspace_bytes < L.total)
    return set_error(SV_ERR_INVALID_ARG, "workspace too small: %zu < %zu", workspace_bytes,
                     L.total);
  if ((s = map_chain_args(vlogits, dlogits, draft_tokens, out_tokens, out_accept_len, out_q_prob,
                          out_p_prob, out_margin, out_status)) != SV_OK ||
      (s = map_arg(workspace, "workspace")) != SV_OK)
    return s;
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
  r.invT = temperature > 0.0f ? 1.0f / temperature : 0.0f;
  r.k = r.invT * kLog2e;
  r.stage = is_device_memory(r.vlog) && is_device_memory(r.dlog);
  set_row_copy(r, L, ws, workspace_bytes, B, dt);
  DecideOut o{out_tokens, out_accept_len, out_q_prob, out_p_prob, out_margin, out_status, nullptr};
  cudaStream_t st = (cudaStream_t)stream;
  if (temperature == 0.0f) {  // greedy: verifier rows only, nothing sampled
    r.P = N + 1;
    r.copy = nullptr;
    return dt == SV_BF16 ? run_verify_greedy<uint16_t>(r, L, ws, o, st, (cudaEvent_t)accept_event)
                         : run_verify_greedy<float>(r, L, ws, o, st, (cudaEvent_t)accept_event);
  }
  return dt == SV_BF16
             ? run_verify<uint16_t>(r, L, ws, seed, step, o, st, (cudaEvent_t)accept_event, early)
             : run_verify<float>(r, L, ws, seed, step, o, st, (cudaEvent_t)accept_event, early);
}
}  // namespace
}  // namespace sv

extern "C" sv_status sv_verify_chain(const void *vlogits, const void *dlogits, sv_dtype dt,
                                     const int32_t *draft_tokens, int B, int N, int V,
                                     float temperature, uint64_t seed, uint64_t step,
                                     int32_t *out_tokens, int32_t *out_accept_len,
                                     float *out_q_prob, float *out_p_prob, float *out_margin,
                                     uint32_t *out_status, void *workspace,
                                     size_t workspace_bytes, void *stream,
                                     void *accept_event) {
  return sv::verify_chain(vlogits, dlogits, dt, draft_tokens, B, N, V, temperature, seed, step,
                          out_tokens, out_accept_len, out_q_prob, out_p_prob, out_margin,
                          out_status, workspace, workspace_bytes, stream, accept_event, false);
}

extern "C" sv_status sv_verify_chain_early_exit(
    const void *vlogits, const void *dlogits, sv_dtype dt, const int32_t *draft_tokens, int B,
    int N, int V, float temperature, uint64_t seed, uint64_t step, int32_t *out_tokens,
    int32_t *out_accept_len, float *out_q_prob, float *out_p_prob, float *out_margin,
    uint32_t *out_status, void *workspace, size_t workspace_bytes, void *stream,
    void *accept_event) {
  return sv::verify_chain(vlogits, dlogits, dt, draft_tokens, B, N, V, temperature, seed, step,
                          out_tokens, out_accept_len, out_q_prob, out_p_prob, out_margin,
                          out_status, workspace, workspace_bytes, stream, accept_event, true);
}

extern "C" size_t sv_verify_tree_workspace(int B, int T, int max_depth, int V) {
  if (B < 0 || T < 1 || max_depth < 0 || V < 1) return 0;
  return plan(B, max_depth, V, true).total;
}

extern "C" size_t sv_verify_tree_workspace_host(int B, int T, int max_depth, int V,
                                                sv_dtype dt) {
  if (B < 0 || T < 1 || max_depth < 0 || V < 1 || (dt != SV_F32 && dt != SV_BF16)) return 0;
  const Layout L = plan(B, max_depth, V, true);
  return L.total + row_copy_bytes(B, L, V, dt);
}

extern "C" sv_status sv_verify_tree(const void *vlogits, const void *dlogits, sv_dtype dt,
                                    const int32_t *parent, const int32_t *token,
                                    const float *score, int B, int T, int max_depth, int V,
                                    float temperature, uint64_t seed, uint64_t step,
                                    int32_t *out_path_nodes, int32_t *out_tokens,
                                    int32_t *out_accept_len, float *out_q_prob,
                                    float *out_p_prob, float *out_margin, uint32_t *out_status,
                                    void *workspace, size_t workspace_bytes, void *stream,
                                    void *accept_event) {
  sv_status s = check_common(vlogits, dt, B, V, temperature, out_tokens, out_accept_len,
                             out_status, workspace);
  if (s != SV_OK || B == 0) return s;
  if (T < 1) return set_error(SV_ERR_INVALID_ARG, "T must be >= 1 (got %d)", T);
  if (T > SV_MAX_TREE_NODES) return set_error(SV_ERR_UNSUPPORTED, "T > %d", SV_MAX_TREE_NODES);
  if (max_depth < 0) return set_error(SV_ERR_INVALID_ARG, "max_depth must be >= 0");
  if (max_depth > SV_MAX_POSITIONS) return set_error(SV_ERR_UNSUPPORTED, "max_depth > %d", SV_MAX_POSITIONS);
  if (B > (1 << 19)) return set_error(SV_ERR_UNSUPPORTED, "B > %d for trees", 1 << 19);
  if (!dlogits || !parent || !token || !score || !out_path_nodes)
    return set_error(SV_ERR_INVALID_ARG, "null pointer argument");
  const Layout L = plan(B, max_depth, V, true);
  if ((s = check_grid(B, L)) != SV_OK) return s;
  if (workspace_bytes < L.total)
    return set_error(SV_ERR_INVALID_ARG, "workspace too small: %zu < %zu", workspace_bytes,
                     L.total);
  if ((s = map_chain_args(vlogits, dlogits, token, out_tokens, out_accept_len, out_q_prob,
                          out_p_prob, out_margin, out_status)) != SV_OK ||
      (s = map_arg(parent, "parent")) != SV_OK || (s = map_arg(score, "score")) != SV_OK ||
      (s = map_arg(out_path_nodes, "out_path_nodes")) != SV_OK ||
      (s = map_arg(workspace, "workspace")) != SV_OK)
    return s;
  char *ws = (char *)align_up((uintptr_t)workspace, 256);
  int32_t *path = (int32_t *)(ws + L.path);
  int32_t *npos = (int32_t *)(ws + L.npos);
  int32_t *tok = (int32_t *)(ws + L.tok);
  uint32_t *tstat = (uint32_t *)(ws + L.tstat);
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(ws + L.ctr, 0, sizeof(int), st) != cudaSuccess)
    return check_launch("row counter reset");
  {
    LaunchScope ls("tree_path", st);
    s = check_launch("tree_path",
                     launch_pdl(tree_path_kernel, dim3(B), dim3(32), 0, st, parent, token, score,
                                B, T, max_depth, path, npos, tok, max_depth > 0 ? max_depth : 1,
                                tstat, (int32_t *)(ws + L.rowlist), (int *)(ws + L.ctr),
                                temperature == 0.0f ? 1 : 0));
    if (s != SV_OK) return s;
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
  r.invT = temperature > 0.0f ? 1.0f / temperature : 0.0f;
  r.k = r.invT * kLog2e;
  r.stage = is_device_memory(r.vlog) && is_device_memory(r.dlog);
  set_row_copy(r, L, ws, workspace_bytes, B, dt);
  DecideOut o{out_tokens, out_accept_len, out_q_prob, out_p_prob, out_margin, out_status,
              out_path_nodes};
  if (temperature == 0.0f) {  // greedy: the path's verifier rows only, nothing sampled
    r.P = max_depth + 1;
    r.copy = nullptr;
    return dt == SV_BF16 ? run_verify_greedy<uint16_t>(r, L, ws, o, st, (cudaEvent_t)accept_event)
                         : run_verify_greedy<float>(r, L, ws, o, st, (cudaEvent_t)accept_event);
  }
  return dt == SV_BF16 ? run_verify<uint16_t>(r, L, ws, seed, step, o, st, (cudaEvent_t)accept_event)
                       : run_verify<float>(r, L, ws, seed, step, o, st, (cudaEvent_t)accept_event);
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
                                             uint32_t *out_status, void *stream,
                                             void *accept_event) {
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
                         out_status, ws, kStaticScratchBytes, stream, accept_event);
}
