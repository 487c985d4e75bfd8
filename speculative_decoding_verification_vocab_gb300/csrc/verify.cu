// verify.cu -- batched verify-and-accept for speculative decoding on sm_103a.
//
// Steps (one stream, no host synchronisation):
//   tree_path    (tree only) best-child walk per sequence
//   row_stats    single-pass online softmax statistics (max, sum of exp) of
//                every logit row the round can touch -- the one step that
//                streams the whole input; HBM-bound
//   decide       one warp per sequence: q(d)/p(d), Philox uniforms, the left-
//                to-right accept walk, outputs, and the sampling task
//   sample       the correction / bonus draws: exact fixed-point weights of
//                the sampled row(s) of every sequence and the inverse-CDF
//                pick, one persistent kernel over (sequence, slice) items
//
// Pages: "Decodificação Especulativa e EAGLE-3" (lesson; "O invariante",
// Passo 1-3) and "投机解码发展" (blog; section 2 steps, section 4 spec_decode /
// eagle_round pseudocode).  p = draft, q = verifier.
#include <math.h>
#include <stdio.h>

#include <mutex>

#include "common.cuh"
#include "rowstat.cuh"


namespace sv {
namespace {

constexpr int kDecideWarps = 4;
constexpr int kSpSlice = 4096;   // sampler: elements of a row per work item
constexpr int kSpThreads = 128;  // sampler: consumer threads (the producer warp is extra)
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
  int maxpos, P, G, NS;
  size_t ctr, rowlist, partial, task, slice, runs, done, rlist, qc, path, npos, tok, tstat;
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
// row_stats: online softmax statistics of every used logit row, per
// (row, segment) unit.  Logits in device memory go through the persistent
// bulk-ring kernel further below; host-resident logits (read in place over
// the host link) through one CTA per unit: grid x = row (tree: the rows on
// the best paths, listed by tree_path), y = segment.  Each thread loads
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
// A segment is 32 KB: 2 * kRsUnroll 16-byte words for each of 128 threads.
// (The early-exit pass, and every pass over host-resident logits, take one
// segment per CTA with plain 16-byte loads.)
template <typename E>
__host__ __device__ constexpr int seg_elems() {
  return kRsThreads * 2 * kRsUnroll * 16 / (int)sizeof(E);
}

struct SegInfo {
  const char *row;   // row base
  char *copy;        // its device copy (host-resident logits), or null
  int v0, v1;        // element range of the segment
  uintptr_t ab, ae;  // 16-byte-aligned body [ab, ae)
  size_t out;        // partial index
};

// Tree rows known before the best path is: each sequence's root rows (the
// verifier row of node 0, and its draft row when a path can go deeper), which
// are row slots 0 and maxpos + 1 of every path.
__device__ __forceinline__ int root_rows(const Round &r, bool greedy) {
  return (greedy || r.maxpos == 0) ? 1 : 2;
}

// Row index space of a row pass: a chain's rows b * P + j; a tree's root rows
// first (R0 per sequence, row_i < R0 B), then the rows tree_path listed.
template <typename E>
__device__ __forceinline__ SegInfo seg_info(const Round &r, int G, const uint64_t *rowlist,
                                            int row_i, int seg, int R0 = 0) {
  int b, j;
  const E *row;
  if (rowlist && row_i < R0 * r.B) {
    b = row_i / R0;
    const bool is_v = row_i - b * R0 == 0;
    j = is_v ? 0 : r.maxpos + 1;
    row = (const E *)(is_v ? r.vlog : r.dlog) + (size_t)b * (is_v ? r.v_rows : r.d_rows) * r.V;
  } else if (rowlist) {
    // one load: tree_path stored the row slot and the row itself
    const uint64_t e = rowlist[row_i - R0 * r.B];
    b = (int)(e >> 44);
    j = (int)((e >> 32) & 0xfffu);
    row = (const E *)((e >> 30) & 1u ? r.dlog : r.vlog) + (size_t)(e & 0x3fffffffu) * r.V;
  } else {
    b = row_i / r.P;
    j = row_i - b * r.P;
    row = src_row<E>(r, b, j);
  }
  SegInfo si;
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
__device__ __forceinline__ void stat_segment(const Round &r, int G, const uint64_t *rowlist,
                                             int row_i, int seg, float4 *partial, int R0 = 0) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const SegInfo si = seg_info<E>(r, G, rowlist, row_i, seg, R0);
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
row_stats_kernel(Round r, int G, const uint64_t *__restrict__ rowlist,
                 const int32_t *__restrict__ rowcount, float4 *__restrict__ partial,
                 unsigned *__restrict__ qc, int nroot) {
  // Tree: the root-row CTAs need nothing from tree_path, the grid before this
  // one, so they start streaming without waiting for it (this grid can only
  // launch once tree_path's CTAs have passed their own wait for the grids
  // before it, so the workspace is free).  The listed-row CTAs wait.
  if (!rowlist) {
    // chain: one CTA per (row = x, segment = y)
    grid_dep_sync();
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x < 3) qc[threadIdx.x] = 0u;
    stat_segment<E, kCopy>(r, G, nullptr, blockIdx.x, blockIdx.y, partial);
    return;
  }
  // tree: segment = x, row CTA = y, so that CTAs are dispatched root rows
  // first (x runs fastest); gridDim.y = nroot root CTAs + the listed-row CTAs
  const int R0 = root_rows(r, false), nroot_rows = R0 * r.B;
  if ((int)blockIdx.y < nroot) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // the sampler's lists and item counter are rebuilt by the accept walk
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x < 3) qc[threadIdx.x] = 0u;
    for (int row_i = blockIdx.y; row_i < nroot_rows; row_i += nroot)
      stat_segment<E, kCopy>(r, G, rowlist, row_i, blockIdx.x, partial, R0);
    return;
  }
  grid_dep_sync();
  // the listed rows, a CTA taking further rows when the paths are deep
  const int ncta = (int)gridDim.y - nroot, nrows = *rowcount;
  for (int li = (int)blockIdx.y - nroot; li < nrows; li += ncta)
    stat_segment<E, kCopy>(r, G, rowlist, nroot_rows + li, blockIdx.x, partial, R0);
}

// ---------------------------------------------------------------------------
// row_stats over logits in device memory: a persistent grid, one TMA bulk
// ring per CTA.  The units are the same (row, segment) pairs as above, in the
// same index space (tree: root rows, then the rows tree_path listed), claimed
// one at a time from a counter shared by the grid, so that SMs that stream
// faster take more of them; a segment's 16-byte-aligned body is staged as
// kRbChunk-byte chunks, one per ring stage.
//   producer (one thread of warp 4)  claims the CTA's next unit, waits until
//              a stage is released, writes the chunk's description and starts
//              a bulk copy of it into the stage (arrival with the byte count
//              on the stage's "full" barrier)
//   consumers (warps 0-3)  wait for a full stage, fold its words into their
//              statistics (thread t takes words t + 128 j of the segment),
//              release the stage, read any ragged head / tail elements
//              directly, and after a segment's last chunk combine the CTA's
//              triples into the segment's partial
// Tree: the root units need nothing from tree_path; the producer waits for
// it (griddepcontrol.wait) only when it first claims a listed unit.  A wait
// that runs out (kRingWaitNs) stops the CTA; the partials of the units it may
// not have finished are written as NaN sums with .w = 1, which the accept
// walk reports as SV_ROW_TIMEOUT.
constexpr int kRbStages = 3;
constexpr int kRbChunk = 16384;  // bytes per stage: half a 32 KB segment
constexpr int kRbConsumers = 128;              // 4 consumer warps
constexpr int kRbThreads = kRbConsumers + 32;  // + the producer warp
static_assert(kRbChunk % (16 * kRbConsumers) == 0, "a chunk is whole words of every consumer");

struct RbMeta {
  const char *row;   // row base
  int v0, v1;        // element range of the segment
  int nhead, ntail;  // ragged elements before / after the staged body
  int w0, w1;        // the body words of this chunk (segment-relative)
  int first, last;   // the chunk opens / closes its segment
  int end;           // 1: no further unit (consumers stop)
  size_t out;        // partial index
};
struct RbSmem {
  unsigned long long full[kRbStages], empty[kRbStages], reduced[kRbStages];
  RbMeta meta[kRbStages];
  long long unit[kRbStages];  // the unit each stage was last filled for
  float4 red[kRbStages][kRbConsumers / 32];
  int abort;
};

// unit u of a row pass: its row / segment and where its partial goes
template <typename E>
__device__ __forceinline__ SegInfo rb_unit(const Round &r, int G, const uint64_t *rowlist, int R0,
                                           long long u) {
  const int row_i = (int)(u / G), seg = (int)(u - (long long)row_i * G);
  return rowlist ? seg_info<E>(r, G, rowlist, row_i, seg, R0)
                 : seg_info<E>(r, G, nullptr, row_i, seg);
}

// Arg-max primitives (the greedy row pass): per thread the largest logit and
// its lowest index, with fault flags.
constexpr uint32_t kArgNan = 1u;   // a NaN or +inf logit
constexpr uint32_t kArgSeen = 2u;  // a logit above -inf
constexpr uint32_t kArgLost = 4u;  // the row pass gave up on a bounded wait

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

// The consumers' per-thread state: online statistics, or (kArg) the arg max.
template <bool kArg>
struct RbState;
template <>
struct RbState<false> {
  StatState st;
  __device__ __forceinline__ void reset() { st = StatState{-INFINITY, 0.0f, 0ull, 0ull}; }
};
template <>
struct RbState<true> {
  ArgState a;
  __device__ __forceinline__ void reset() { a = ArgState{-INFINITY, 0x7fffffff, 0u}; }
};

// A segment's partial that the row pass never computed (a wait ran out):
// statistics: NaN sums with .w = 1; arg max: the fault and "lost" flags.
template <bool kArg>
__device__ __forceinline__ float4 rb_lost() {
  return kArg ? make_float4(-INFINITY, __int_as_float(0x7fffffff),
                            __uint_as_float(kArgNan | kArgLost), 0.0f)
              : make_float4(NAN, NAN, NAN, 1.0f);
}

template <typename E, bool kArg>
__global__ void __launch_bounds__(kRbThreads)
row_pass_bulk_kernel(Round r, int G, const uint64_t *__restrict__ rowlist,
                     const int32_t *__restrict__ rowcount,
                     unsigned long long *__restrict__ next_unit, float4 *__restrict__ partial,
                     unsigned *__restrict__ qc) {
  extern __shared__ __align__(128) uint4 rb_stage[];  // [kRbStages][kRbChunk]
  __shared__ RbSmem sm;
  constexpr int kCW = kRbChunk / 16;  // words per stage
  constexpr int kPer = 16 / (int)sizeof(E);
  const int tid = threadIdx.x;
  const bool tree = rowlist != nullptr;
  const int R0 = tree ? root_rows(r, kArg) : 0;
  if (!tree)
    grid_dep_sync();  // chain: the workspace is free once the previous step's grids are done
  else
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (qc && blockIdx.x == 0 && tid < 3) qc[tid] = 0u;  // the sampler's counters, rebuilt by the walk
  if (tid == 0) {
    for (int i = 0; i < kRbStages; ++i) {
      ring_init(ring_addr(&sm.full[i]), 1);
      ring_init(ring_addr(&sm.empty[i]), kRbConsumers);
      ring_init(ring_addr(&sm.reduced[i]), kRbConsumers / 32);
    }
    sm.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  volatile int *abort = &sm.abort;
  long long n_units = tree ? (long long)R0 * r.B * G : (long long)r.B * r.P * G;
  bool waited = !tree;
  if (tid >= kRbConsumers) {
    // ---------------------------------------------------------------- producer
    if (tid != kRbConsumers) return;
    long long k = 0;  // stages filled so far
    bool lost = false;
    // A unit's description: its chunks' metadata, body and chunk count.
    struct Prep {
      RbMeta m;
      const uint4 *ab;
      int nw, nc;
    };
    auto prepare = [&](long long v, Prep &p) {
      if (v >= n_units && !waited) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        waited = true;
        n_units += (long long)__ldcg(rowcount) * G;
      }
      p.m.end = v >= n_units;
      p.nc = 1;
      p.nw = 0;
      p.ab = nullptr;
      if (p.m.end) return;
      const SegInfo si = rb_unit<E>(r, G, rowlist, R0, v);
      const E *row = (const E *)si.row;
      p.m.row = si.row;
      p.m.v0 = si.v0;
      p.m.v1 = si.v1;
      p.m.nhead = (int)((si.ab - (uintptr_t)(row + si.v0)) / sizeof(E));
      p.m.ntail = (int)(((uintptr_t)(row + si.v1) - si.ae) / sizeof(E));
      p.m.out = si.out;
      p.ab = (const uint4 *)si.ab;
      p.nw = (int)((si.ae - si.ab) / 16);
      p.nc = p.nw > kCW ? (p.nw + kCW - 1) / kCW : 1;
    };
    // Units are claimed from a counter shared by the grid (zeroed before the
    // launch), so SMs that stream faster take more of them.  The next claim
    // is kept one unit ahead, and a unit is described (for a listed tree row
    // that takes a load of its list entry) while the previous unit's copies
    // are in flight, so a released stage is refilled at once.
    long long cu = (long long)atomicAdd(next_unit, 1ull);
    long long na = (long long)atomicAdd(next_unit, 1ull);
    Prep p;
    prepare(cu, p);
    for (;;) {
      for (int c = 0; c < p.nc; ++c, ++k) {
        const int stage = (int)(k % kRbStages);
        const long long use = k / kRbStages;
        if (use > 0 &&
            !ring_wait(ring_addr(&sm.empty[stage]), (uint32_t)((use - 1) & 1), abort)) {
          lost = true;
          break;
        }
        sm.unit[stage] = p.m.end ? -1 : cu;
        const uint32_t full = ring_addr(&sm.full[stage]);
        RbMeta m = p.m;
        if (m.end) {
          sm.meta[stage] = m;
          ring_arrive(full);
          continue;
        }
        m.w0 = c * kCW;
        m.w1 = min(p.nw, m.w0 + kCW);
        m.first = c == 0;
        m.last = c == p.nc - 1;
        sm.meta[stage] = m;
        const uint32_t bytes = (uint32_t)(m.w1 - m.w0) * 16u;
        if (bytes) {
          ring_expect_tx(full, bytes);
          ring_bulk(ring_addr(rb_stage + (size_t)stage * kCW), p.ab + m.w0, bytes, full);
        } else {
          ring_arrive(full);
        }
      }
      if (lost || p.m.end) break;
      cu = na;
      prepare(cu, p);
      na = p.m.end ? -1 : (long long)atomicAdd(next_unit, 1ull);
    }
    // copies issued for the last kRbStages stages land before the CTA's
    // shared memory is released (at once unless a wait ran out)
    for (long long kk = k - 1; kk >= 0 && kk >= k - kRbStages; --kk) {
      const uint32_t bar = ring_addr(&sm.full[kk % kRbStages]);
      const unsigned long long t0 = ring_ns();
      while (!ring_try(bar, (uint32_t)((kk / kRbStages) & 1)) && ring_ns() - t0 < kRingWaitNs) {
      }
    }
    if (lost || *abort) {
      // a wait ran out: the units this CTA may not have finished -- those of
      // the stages in use, the one being filled and the one claimed ahead --
      // get partials marked as never computed (a finished one among them
      // only widens the report)
      if (!waited) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        n_units += (long long)__ldcg(rowcount) * G;
      }
      auto mark = [&](long long v) {
        if (v >= 0 && v < n_units)
          partial[rb_unit<E>(r, G, rowlist, R0, v).out] = rb_lost<kArg>();
      };
      for (int i = 0; i < kRbStages && i < k; ++i) mark(sm.unit[i]);
      mark(cu);
      mark(na);
    }
    return;
  }
  // ------------------------------------------------------------------ consumers
  const int warp = tid >> 5, lane = tid & 31;
  const float k2 = r.k;
  // a stage's reduction barrier completes once per unit that ends in it, not
  // once per use: bit s is the parity of stage s's next reduction
  unsigned rpar = 0u;
  RbState<kArg> ps;
  ps.reset();
  for (long long k = 0;; ++k) {
    const int stage = (int)(k % kRbStages);
    const uint32_t ph = (uint32_t)((k / kRbStages) & 1);
    if (!ring_wait(ring_addr(&sm.full[stage]), ph, abort)) break;
    const RbMeta m = sm.meta[stage];
    if (m.end) break;
    const E *row = (const E *)m.row;
    // ragged elements.  Arg max: the head before the first chunk's words,
    // the tail after the last chunk's (increasing index order within a
    // thread keeps the lowest index).  Statistics: head and tail first, the
    // order of every other row-statistics kernel, so that all of them round
    // a segment's sum alike.
    if (m.first) {
      ps.reset();
      if (tid < m.nhead) {
        if constexpr (kArg)
          arg1(ps.a, load_elem<E>(row + m.v0 + tid), m.v0 + tid);
        else
          stat1(elem_to_f32(__ldg(row + m.v0 + tid)), ps.st, k2);
      }
      if constexpr (!kArg) {
        if (tid < m.ntail) stat1(elem_to_f32(__ldg(row + m.v1 - m.ntail + tid)), ps.st, k2);
      }
    }
    // thread t takes words t + 128 i of the segment, kRsUnroll at a time
    const uint4 *sb = rb_stage + (size_t)stage * kCW;
    const int nw = m.w1 - m.w0;
    const int vw = m.v0 + m.nhead + m.w0 * kPer;  // element index of the chunk's first word
    int i = tid;
    for (; i + (kRsUnroll - 1) * kRbConsumers < nw; i += kRsUnroll * kRbConsumers) {
      uint4 buf[kRsUnroll];
#pragma unroll
      for (int q = 0; q < kRsUnroll; ++q) buf[q] = sb[i + q * kRbConsumers];
      if constexpr (kArg) {
#pragma unroll
        for (int q = 0; q < kRsUnroll; ++q)
          arg_word<E>(ps.a, buf[q], vw + (i + q * kRbConsumers) * kPer);
      } else {
        stat_batch<E>(buf, ps.st, k2);
      }
    }
    for (; i < nw; i += kRbConsumers) {
      if constexpr (kArg)
        arg_word<E>(ps.a, sb[i], vw + i * kPer);
      else
        stat_word<E>(sb[i], ps.st, k2);
    }
    if (!m.last) {
      ring_arrive(ring_addr(&sm.empty[stage]));
      continue;
    }
    if constexpr (kArg) {
      if (tid < m.ntail) arg1(ps.a, load_elem<E>(row + m.v1 - m.ntail + tid), m.v1 - m.ntail + tid);
    }
    // last chunk: warps 1-3 release the stage now; warp 0 once it has read
    // the stage's reduction slots, so that no warp writes them for a later
    // unit first
    if (warp) ring_arrive(ring_addr(&sm.empty[stage]));
    float4 mine;
    if constexpr (kArg) {
      ArgState c = ps.a;
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const float ob = __shfl_xor_sync(0xffffffffu, c.best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, c.idx, o);
        const uint32_t of = __shfl_xor_sync(0xffffffffu, c.flags, o);
        arg_merge(c, ob, oi, of);
      }
      mine = make_float4(c.best, __int_as_float(c.idx), __uint_as_float(c.flags), 0.0f);
    } else {
      float a0, a1, a2, a3;
      f2_unpack(ps.st.s01, a0, a1);
      f2_unpack(ps.st.s23, a2, a3);
      float mx = ps.st.mx, mk = ps.st.mk, sum = (a0 + a1) + (a2 + a3);
      warp_stat_combine(mx, mk, sum);
      mine = make_float4(mx, mk, sum, 0.0f);
    }
    if (lane == 0) {
      sm.red[stage][warp] = mine;
      ring_arrive(ring_addr(&sm.reduced[stage]));
    }
    const uint32_t rph = (rpar >> stage) & 1u;
    rpar ^= 1u << stage;
    if (warp == 0) {
      if (!ring_wait(ring_addr(&sm.reduced[stage]), rph, abort)) break;
      const float4 none = kArg ? make_float4(-INFINITY, __int_as_float(0x7fffffff), 0.0f, 0.0f)
                               : make_float4(-INFINITY, 0.0f, 0.0f, 0.0f);
      float4 v = lane < kRbConsumers / 32 ? sm.red[stage][lane] : none;
      ring_arrive(ring_addr(&sm.empty[stage]));
      if constexpr (kArg) {
        ArgState c{v.x, __float_as_int(v.y), __float_as_uint(v.z)};
#pragma unroll
        for (int o = 16; o; o >>= 1) {
          const float ob = __shfl_xor_sync(0xffffffffu, c.best, o);
          const int oi = __shfl_xor_sync(0xffffffffu, c.idx, o);
          const uint32_t of = __shfl_xor_sync(0xffffffffu, c.flags, o);
          arg_merge(c, ob, oi, of);
        }
        v = make_float4(c.best, __int_as_float(c.idx), __uint_as_float(c.flags), 0.0f);
      } else {
        warp_stat_combine(v.x, v.y, v.z);
      }
      if (lane == 0) partial[m.out] = v;
    }
  }
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
  L.ctr = take(16);  // [0] active row count (tree); [8] the row pass's next unit (u64)
  L.rowlist = tree ? take(sizeof(uint64_t) * nslots) : 0;
  L.partial = take(sizeof(float4) * nslots * L.G);
  L.task = take(sizeof(Task) * (size_t)B);
  L.NS = (V + kSpSlice - 1) / kSpSlice;
  L.slice = take(sizeof(unsigned long long) * 3 * (size_t)B * L.NS);
  L.runs = take(sizeof(unsigned long long) * (size_t)B * L.NS * kSpThreads);
  L.done = take(sizeof(unsigned) * 2 * (size_t)B);
  L.rlist = take(sizeof(int) * 2 * (size_t)B);
  L.qc = take(sizeof(unsigned) * 4);
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
// Returns true when a segment's partial is marked as never computed (.w != 0:
// the row pass gave up on a bounded wait).
template <bool kCg = false>
__device__ __forceinline__ bool merge_slot(const float4 *part, int G, float &mx, float &mk,
                                           float &s) {
  mx = -INFINITY;
  mk = 0.0f;
  s = 0.0f;
  bool lost = false;
  for (int g0 = 0; g0 < G; g0 += 8) {
    float4 v[8];
#pragma unroll
    for (int g = 0; g < 8; ++g)
      if (g0 + g < G) v[g] = kCg ? __ldcg(part + g0 + g) : part[g0 + g];
#pragma unroll
    for (int g = 0; g < 8; ++g)
      if (g0 + g < G) {
        st_combine(mx, mk, s, v[g].x, v[g].y, v[g].z);
        lost |= v[g].w != 0.0f;
      }
  }
  return lost;
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
  const bool lq_ = merge_slot<kCg>(pb + (size_t)i * G, G, J.mxq, mkq, sq);
  const bool lp_ = merge_slot<kCg>(pb + (size_t)(r.maxpos + 1 + i) * G, G, J.mxp, mkp, sp);
  J.bad = (!(sq > 0.0f) || !(sp > 0.0f)) ? SV_ROW_NAN : 0u;
  if (lq_ || lp_) J.bad |= SV_ROW_TIMEOUT;
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
              uint64_t step, DecideOut o, Task *__restrict__ tasks, int *__restrict__ lists,
              unsigned *__restrict__ qc, unsigned *__restrict__ done) {
  grid_dep_sync();
  const int b = blockIdx.x * kDecideWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= r.B) return;
  const unsigned FULL = 0xffffffffu;
  // the first chunk's draft token and path node, loaded beside the path
  // length instead of after it (in bounds whatever the length)
  int d_pf = 0, n_pf = lane;
  if (lane < r.maxpos) {
    d_pf = r.tok[(size_t)b * r.tok_stride + lane];
    if (r.path) n_pf = r.path[(size_t)b * (r.maxpos + 1) + lane];
  }
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
  const int nchunks = (npos + 31) / 32;
  for (int c = 0; c < nchunks && !tree_bad; ++c) {
    const int i = c * 32 + lane;
    if (i >= npos) break;
    // issued first: x_d depends on them
    const int d = c == 0 ? d_pf : r.tok[(size_t)b * r.tok_stride + i];
    const int node = c == 0 ? n_pf : round_node(r, b, i);
    const E *vrow = used_row<E>(r, b, i, (const E *)r.vlog + ((size_t)b * r.v_rows + node) * r.V);
    const E *drow = used_row<E>(r, b, r.maxpos + 1 + i,
                                (const E *)r.dlog + ((size_t)b * r.d_rows + node) * r.V);
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
  // bonus row (verifier row of position npos), checked by lane 0 after the
  // positions (its results are needed only from here on)
  uint32_t bonus_bits = 0;
  if (lane == 0 && !tree_bad) {
    float mx, mk, s;
    if (merge_slot(pb + (size_t)npos * G, G, mx, mk, s)) bonus_bits |= SV_ROW_TIMEOUT;
    if (!(s > 0.0f)) bonus_bits |= SV_ROW_NAN;
    mxv[npos] = mx;
    usm[npos] = uniform_u24(seed, step, (uint32_t)b, (uint32_t)npos, kDrawSample);
  }
  const uint32_t bonus_bad = kEarly ? __shfl_sync(FULL, bonus_bits, 0) : 0u;
  if (!kEarly) bad |= bonus_bits;
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
    // the sampler's lists: residual draws, then bonus draws; its counts
    if (t.active) {
      if (a < npos)
        lists[atomicAdd(qc, 1u)] = b;
      else
        lists[r.B + atomicAdd(qc + 1, 1u)] = b;
    }
    done[b] = 0u;
    done[r.B + b] = 0u;
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
                    int *__restrict__ stop, uint64_t seed, uint64_t step,
                    unsigned *__restrict__ qc) {
  grid_dep_sync();
  // the sampler's lists and item counter are rebuilt by the accept walk
  if (blockIdx.x == 0 && threadIdx.x < 3) qc[threadIdx.x] = 0u;
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
template <typename E>
__device__ __forceinline__ void argmax_segment(const Round &r, int G, const uint64_t *rowlist,
                                               int row_i, int seg, float4 *partial, int R0 = 0) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const SegInfo si = seg_info<E>(r, G, rowlist, row_i, seg, R0);
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
row_argmax_kernel(Round r, int G, const uint64_t *__restrict__ rowlist,
                  const int32_t *__restrict__ rowcount, float4 *__restrict__ partial,
                  int nroot) {
  if (!rowlist) {  // chain: one CTA per (row = x, segment = y)
    grid_dep_sync();
    argmax_segment<E>(r, G, nullptr, blockIdx.x, blockIdx.y, partial);
    return;
  }
  // tree, as row_stats: segment = x, row CTA = y, the root rows (which need
  // nothing from tree_path) first
  const int nroot_rows = root_rows(r, true) * r.B;
  if ((int)blockIdx.y < nroot) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (int row_i = blockIdx.y; row_i < nroot_rows; row_i += nroot)
      argmax_segment<E>(r, G, rowlist, row_i, blockIdx.x, partial, 1);
    return;
  }
  grid_dep_sync();
  const int ncta = (int)gridDim.y - nroot, nrows = *rowcount;
  for (int li = (int)blockIdx.y - nroot; li < nrows; li += ncta)
    argmax_segment<E>(r, G, rowlist, nroot_rows + li, blockIdx.x, partial, 1);
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
    if (a.flags & kArgLost) bad |= SV_ROW_TIMEOUT;
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
    if (a.flags & kArgLost) bad |= SV_ROW_TIMEOUT;
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
//   z = fl(x * invT); e = exp32_repro(fl(z - max z)); E = floor(e 2^40)
//   a draw from q (bonus; zero residual): weights E, S = sum E
//   a residual draw: inv_s = fl32(2^40 / fl64(sum E)) per row, q = fl(e inv_s),
//     p likewise, w = max(0, fl(q - p)), weights W = floor(w 2^62), S = sum W
//   t = floor(u24 * S / 2^24); token = min{k : sum_{v<=k} weight_v > t}
// Only scalar or packed _rn operations are used where a product feeds a sum,
// so no multiply can be fused into a later add.
//
// Exact sums without 64-bit conversions: a value v in [0, 1] splits exactly
// into parts on fixed grids, each part truncated by one add rounding toward
// zero onto a power of two and one subtraction of it:
//   E (2^-40 grid): a on 2^-20 (21 bits), then the remainder on 2^-40
//                   (20 bits); up to 16 values per part sum exactly in fp32;
//   W (2^-62 grid): parts on 2^-21, 2^-42 and 2^-62; up to 8 values per part.
// The part sums become integers once per 16 (8) values and meet in uint64, so
// sum floor(v 2^40) and sum floor(v 2^62) are exact whatever the order.  The
// sums stay below 2^63: sum E <= V 2^40 with V <= 2^22, and sum W <= 2^62
// (1 + 2^-20) because the normalised q row sums to 1 up to rounding.
//
// One persistent kernel.  Its work items are (sequence, slice) pairs, a slice
// being kSpSlice consecutive elements of the sampled row(s); consumer thread t
// owns the run of 32 consecutive elements [32 t, 32 t + 32) of a slice.  A CTA
// is one producer warp and four consumer warps around a two-stage ring in
// shared memory:
//   producer   counts the item a released stage held for its sequence (and,
//              if that completed the sequence's pass, picks the token),
//              claims the next item from a grid-wide counter, reads its
//              sequence's task and starts TMA bulk copies of the slice of
//              each row into the stage ("full" barrier, with the byte count)
//   consumers  wait for a full stage, compute the item, store the run sums,
//              combine the warps' slice sums (a bounded "reduced" barrier;
//              thread 0 stores them) and release the stage ("empty" barrier)
// Items are claimed in this order:
//   pass 1, residual draws  exact sums of E over the slice of the q and the p
//                           row (the accept walk lists these sequences)
//   pass 1, bonus draws     the run sums of E of the q row, stored
//   pass 2, residual draws  the run sums of W, stored, with both rows' 1/S
//                           formed by the producer from the pass-1 sums
// Each item ends with its slice sums and a per-sequence completion count; the
// CTA that completes a sequence's last pass picks its token: the slice holding
// the threshold (slice sums), the run (stored run sums), then one lane per
// element of the run.  A pass-2 item needs its sequence's pass 1 complete;
// every pass-1 item is claimed before any pass-2 item and pass-1 items never
// wait, so that wait always ends.  Every wait (barriers, the pass-1 count) is
// bounded by a wall-clock limit; one that runs out sets SV_ROW_TIMEOUT for
// the sequence concerned and the CTA stops taking items.

constexpr int kSpWarps = kSpThreads / 32;
template <typename E>
__host__ __device__ constexpr int sp_per() { return 16 / (int)sizeof(E); }  // elements per word
template <typename E>
__host__ __device__ constexpr int sp_words() { return kSpSlice / sp_per<E>(); }  // words per slice
template <typename E>
__host__ __device__ constexpr int sp_wpt() { return sp_words<E>() / kSpThreads; }  // words per thread
// shared memory of one stage: q and p words of the slice
template <typename E>
__host__ __device__ constexpr size_t sp_stage_bytes() { return 2 * (size_t)sp_words<E>() * 16; }

__device__ __forceinline__ float inv_sum(unsigned long long se) {
  return __double2float_rn(__ddiv_rn(0x1p40, __ull2double_rn(se)));
}
__device__ __forceinline__ unsigned long long fix62(float w) {
  return __float2ull_rz(__fmul_rn(w, 0x1p62f));
}
__device__ __forceinline__ unsigned long long fix40(float e) {
  return __float2ull_rz(__fmul_rn(e, 0x1p40f));
}

__device__ __forceinline__ unsigned long long trunc2(unsigned long long v, float grid_top) {
  const unsigned long long g = f2_splat(grid_top);
  return f2_sub(f2_add_rz(v, g), g);
}
// E parts of a packed pair (<= 16 values per lane between conversions)
struct Acc40 {
  unsigned long long a, b;
};
__device__ __forceinline__ void acc40(Acc40 &P, unsigned long long e) {
  const unsigned long long a = trunc2(e, 0x1p3f);     // 2^-20 grid
  const unsigned long long b = trunc2(f2_sub(e, a), 0x1p-17f);  // 2^-40 grid
  P.a = f2_add(P.a, a);
  P.b = f2_add(P.b, b);
}
// adds both lanes' exact sums to s0 / s1 and clears the parts
__device__ __forceinline__ void drain40(Acc40 &P, unsigned long long &s0, unsigned long long &s1) {
  float a0, a1, b0, b1;
  f2_unpack(P.a, a0, a1);
  f2_unpack(P.b, b0, b1);
  s0 += ((unsigned long long)__float2uint_rn(__fmul_rn(a0, 0x1p20f)) << 20) +
        __float2uint_rn(__fmul_rn(b0, 0x1p40f));
  s1 += ((unsigned long long)__float2uint_rn(__fmul_rn(a1, 0x1p20f)) << 20) +
        __float2uint_rn(__fmul_rn(b1, 0x1p40f));
  P.a = P.b = 0ull;
}
// W parts of a packed pair (<= 8 values per lane between conversions)
struct Acc62 {
  unsigned long long a, b, c;
};
__device__ __forceinline__ void acc62(Acc62 &P, unsigned long long w) {
  const unsigned long long a = trunc2(w, 0x1p2f);     // 2^-21 grid
  const unsigned long long r1 = f2_sub(w, a);
  const unsigned long long b = trunc2(r1, 0x1p-19f);  // 2^-42 grid
  const unsigned long long c = trunc2(f2_sub(r1, b), 0x1p-39f);  // 2^-62 grid
  P.a = f2_add(P.a, a);
  P.b = f2_add(P.b, b);
  P.c = f2_add(P.c, c);
}
__device__ __forceinline__ unsigned long long drain62(Acc62 &P) {
  float a[2], b[2], c[2];
  f2_unpack(P.a, a[0], a[1]);
  f2_unpack(P.b, b[0], b[1]);
  f2_unpack(P.c, c[0], c[1]);
  unsigned long long s = 0;
#pragma unroll
  for (int l = 0; l < 2; ++l)
    s += ((unsigned long long)__float2uint_rn(__fmul_rn(a[l], 0x1p21f)) << 41) +
         ((unsigned long long)__float2uint_rn(__fmul_rn(b[l], 0x1p42f)) << 20) +
         __float2uint_rn(__fmul_rn(c[l], 0x1p62f));
  P.a = P.b = P.c = 0ull;
  return s;
}

// packed exponent arguments fl(fl(x * invT) - mz) of two elements (the
// multiply is skipped at T = 1; scalar where a multiply is involved)
__device__ __forceinline__ unsigned long long arg2(float x0, float x1, float m0, float m1,
                                                   float invT, bool unit_t) {
  if (unit_t) return f2_sub(f2_pack(x0, x1), f2_pack(m0, m1));
  return f2_pack(__fsub_rn(__fmul_rn(x0, invT), m0), __fsub_rn(__fmul_rn(x1, invT), m1));
}
__device__ __forceinline__ float e1(float x, float invT, float mz, bool unit_t) {
  const float z = unit_t ? x : __fmul_rn(x, invT);
  return exp32_repro(__fsub_rn(z, mz));
}

// element j of a 16-byte word of logits
template <typename E>
__device__ __forceinline__ float word_elem(const uint4 &q, int j);
template <>
__device__ __forceinline__ float word_elem<uint16_t>(const uint4 &q, int j) {
  const int c = j >> 1;
  const uint32_t x = c == 0 ? q.x : c == 1 ? q.y : c == 2 ? q.z : q.w;
  return (j & 1) ? bf16_hi(x) : bf16_lo(x);
}
template <>
__device__ __forceinline__ float word_elem<float>(const uint4 &q, int j) {
  return __uint_as_float(j == 0 ? q.x : j == 1 ? q.y : j == 2 ? q.z : q.w);
}

// The residual weights of two elements from their exponentials (q and p
// lanes packed): max(0, fl(fl(e_q iq) - fl(e_p ip))).  Scalar _rn intrinsics:
// the packed multiply and subtract were observed to be contracted into a
// fused multiply-add by the compiler, which changes the last bit of q - p.
__device__ __forceinline__ unsigned long long resid_pair(unsigned long long eq,
                                                         unsigned long long ep, float iq,
                                                         float ip) {
  float q0, q1, p0, p1;
  f2_unpack(eq, q0, q1);
  f2_unpack(ep, p0, p1);
  const float d0 = __fsub_rn(__fmul_rn(q0, iq), __fmul_rn(p0, ip));
  const float d1 = __fsub_rn(__fmul_rn(q1, iq), __fmul_rn(p1, ip));
  return f2_pack(fmaxf(d0, 0.0f), fmaxf(d1, 0.0f));
}

// A word of a row read element by element (ragged or unaligned rows);
// elements at or past V read as -inf, whose exponential is 0.
template <typename E>
__device__ __forceinline__ uint4 load_word_slow(const E *row, int v0, int V) {
  uint32_t q[4];
  if (sizeof(E) == 2) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t lo = v0 + 2 * c < V ? (uint32_t)__ldg((const unsigned short *)row + v0 + 2 * c) : 0xff80u;
      const uint32_t hi = v0 + 2 * c + 1 < V ? (uint32_t)__ldg((const unsigned short *)row + v0 + 2 * c + 1) : 0xff80u;
      q[c] = lo | (hi << 16);
    }
  } else {
#pragma unroll
    for (int c = 0; c < 4; ++c)
      q[c] = v0 + c < V ? __float_as_uint(__ldg((const float *)row + v0 + c)) : 0xff800000u;
  }
  return make_uint4(q[0], q[1], q[2], q[3]);
}
template <typename E>
__device__ __forceinline__ uint4 load_word(const E *row, int v0, int V, bool vec) {
  if (vec && v0 + sp_per<E>() <= V) return __ldg((const uint4 *)(row + v0));
  return load_word_slow<E>(row, v0, V);
}

struct RowPair {
  const void *rq, *rp;
  float mzq, mzp;
  bool resid, vec, unit_t;
};
template <typename E, typename TaskLike>
__device__ __forceinline__ RowPair row_pair(const Round &r, const TaskLike &t) {
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

// the weight of one element: E (a draw from q) or W (residual)
template <typename E>
__device__ __forceinline__ unsigned long long weight_elem(const Round &r, const RowPair &p, int v,
                                                          float iq, float ip, bool use_q) {
  if (v >= r.V) return 0ull;
  const float eq = e1(load_elem<E>((const E *)p.rq + v), r.invT, p.mzq, p.unit_t);
  if (use_q) return fix40(eq);
  const float d = __fsub_rn(
      __fmul_rn(eq, iq),
      __fmul_rn(e1(load_elem<E>((const E *)p.rp + v), r.invT, p.mzp, p.unit_t), ip));
  return fix62(d > 0.0f ? d : 0.0f);
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

// First index i in [0, n) whose running sum of vals exceeds thr, by one warp
// (uniform result); base gets the sum before it.
template <typename F>
__device__ __forceinline__ int warp_find(int n, unsigned long long thr, F get,
                                         unsigned long long &base) {
  base = 0;
  for (int c0 = 0; c0 < n; c0 += 32) {
    const int c = c0 + (int)(threadIdx.x & 31);
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
  return n - 1;  // not reached when thr < the total
}



// A consumer thread's 32 elements of one row's slice: words
// [t wpt, (t + 1) wpt) of the slice.  The bulk copy staged the slice's first
// nbulk words in order; the rest (a ragged row end, or every word of a row
// that is not 16-byte aligned) is read from global memory, -inf past V.  The
// words are fetched in an order rotated by the thread index, which keeps the
// 16-byte shared-memory reads of a quarter warp on distinct banks; the sums
// below do not depend on the order.
template <typename E>
__device__ __forceinline__ void fetch_run(uint4 (&w)[sp_wpt<E>()], const uint4 *stage,
                                          const E *row, int V, int s, int nbulk) {
  constexpr int kWpt = sp_wpt<E>();
  constexpr int kSh = kWpt == 4 ? 1 : 0;  // threads per 128-byte line: 2 (bf16), 1 (fp32)
  const int t = threadIdx.x;
#pragma unroll
  for (int k = 0; k < kWpt; ++k) {
    const int wi = t * kWpt + ((k + (t >> kSh)) & (kWpt - 1));
    w[k] = wi < nbulk ? stage[wi]
                      : load_word_slow<E>(row, s * kSpSlice + wi * sp_per<E>(), V);
  }
}

// The run sums of a thread.
// E of the q row; lanes (element j, element j + 1), 16 values per lane.
template <typename E>
__device__ __forceinline__ unsigned long long run_e40(const Round &r, const RowPair &p,
                                                      const uint4 (&wq)[sp_wpt<E>()]) {
  Acc40 P{0ull, 0ull};
#pragma unroll
  for (int k = 0; k < sp_wpt<E>(); ++k)
#pragma unroll
    for (int j = 0; j < sp_per<E>(); j += 2)
      acc40(P, exp32x2(arg2(word_elem<E>(wq[k], j), word_elem<E>(wq[k], j + 1), p.mzq, p.mzq,
                            r.invT, p.unit_t)));
  unsigned long long s0 = 0, s1 = 0;
  drain40(P, s0, s1);
  return s0 + s1;
}
// E of the q row and of the p row; lanes (q element, p element), drained
// every 16 values.
template <typename E>
__device__ __forceinline__ void run_e40_pair(const Round &r, const RowPair &p,
                                             const uint4 (&wq)[sp_wpt<E>()],
                                             const uint4 (&wp)[sp_wpt<E>()],
                                             unsigned long long &fq, unsigned long long &fp) {
  Acc40 P{0ull, 0ull};
  fq = fp = 0;
#pragma unroll
  for (int k = 0; k < sp_wpt<E>(); ++k)
#pragma unroll
    for (int j = 0; j < sp_per<E>(); ++j) {
      acc40(P, exp32x2(arg2(word_elem<E>(wq[k], j), word_elem<E>(wp[k], j), p.mzq, p.mzp, r.invT,
                            p.unit_t)));
      if ((k * sp_per<E>() + j) % 16 == 15) drain40(P, fq, fp);
    }
}
// W; lanes (element j, element j + 1), drained every 8 values.
template <typename E>
__device__ __forceinline__ unsigned long long run_w62(const Round &r, const RowPair &p,
                                                      const uint4 (&wq)[sp_wpt<E>()],
                                                      const uint4 (&wp)[sp_wpt<E>()], float iq,
                                                      float ip) {
  Acc62 P{0ull, 0ull, 0ull};
  unsigned long long fw = 0;
#pragma unroll
  for (int k = 0; k < sp_wpt<E>(); ++k)
#pragma unroll
    for (int j = 0; j < sp_per<E>(); j += 2) {
      const unsigned long long eq = exp32x2(arg2(word_elem<E>(wq[k], j), word_elem<E>(wq[k], j + 1),
                                                 p.mzq, p.mzq, r.invT, p.unit_t));
      const unsigned long long ep = exp32x2(arg2(word_elem<E>(wp[k], j), word_elem<E>(wp[k], j + 1),
                                                 p.mzp, p.mzp, r.invT, p.unit_t));
      acc62(P, resid_pair(eq, ep, iq, ip));
      if (((k * sp_per<E>() + j) / 2) % 8 == 7) fw += drain62(P);
    }
  return fw;
}

struct SampleWs {
  unsigned long long *slice;  // [3][B][NS] slice sums: E of q, E of p, W
  unsigned long long *runs;   // [B][NS][kSpThreads] run sums in use (E or W)
  unsigned *done;             // [2][B] completed slices of pass 1 / 2 (zeroed by decide)
  const int *rlist, *blist;   // residual / bonus draws, listed by the accept walk
  unsigned *qc;               // [0] residual count, [1] bonus count, [2] next item
                              // (zeroed by the row pass)
  int NS, B;
};

// 1 / S of the q and p rows of residual draw b from its pass-1 slice sums,
// by one warp (uniform result)
__device__ __forceinline__ float2 resid_inv(const SampleWs &sw, int b) {
  const unsigned long long *slq = sw.slice + (size_t)b * sw.NS;
  const unsigned long long *slp = sw.slice + ((size_t)sw.B + b) * sw.NS;
  unsigned long long Sq = 0, Sp = 0;
  for (int c = (int)(threadIdx.x & 31); c < sw.NS; c += 32) {
    Sq += __ldcg(slq + c);
    Sp += __ldcg(slp + c);
  }
  Sq = warp_sum_u64(Sq);
  Sp = warp_sum_u64(Sp);
  return make_float2(inv_sum(Sq), inv_sum(Sp));
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}


// What the producer tells the consumers about the item in a stage
struct ItemMeta {
  const void *rq, *rp;  // the sampled rows (rp null for a bonus draw)
  float mq, mp;         // their raw maxima
  float iq, ip;         // 1/S of both rows (pass 2)
  uint32_t u24;
  int a, b, s, kind;    // kind: 0 pass 1 residual, 1 pass 1 bonus, 2 pass 2, -1 none left
  int ok;               // pass 2: the sequence's pass 1 was complete
  int nbulk;            // leading words of the slice staged by the bulk copy
};

struct SampleSmem {
  unsigned long long full[2], empty[2];  // the ring's barriers
  unsigned long long reduced[2];         // the consumer warps' slice sums are in
  ItemMeta meta[2];
  unsigned long long red[2][2][kSpWarps];  // per stage, per sum: the warps' partial sums
  int abort;
};

// The inverse-CDF pick of sequence b by one warp (the producer warp of the
// CTA that completed the sequence): the slice (slice sums), the run (stored
// run sums, or the q row's run sums recomputed for the zero-residual
// fallback), then one lane per element of the run.
template <typename E>
__device__ __forceinline__ void pick_token_warp(const Round &r, const ItemMeta &t, int b,
                                                const SampleWs &sw,
                                                const unsigned long long *slices, bool use_q,
                                                bool recompute, const DecideOut &o) {
  const int lane = threadIdx.x & 31;
  const int NS = sw.NS;
  const RowPair p = row_pair<E>(r, t);
  unsigned long long S = 0;
  for (int c = lane; c < NS; c += 32) S += __ldcg(slices + c);
  S = warp_sum_u64(S);
  const unsigned long long thr =
      (__umul64hi((unsigned long long)t.u24, S) << 40) | (((unsigned long long)t.u24 * S) >> 24);
  unsigned long long base;
  const int s = warp_find(NS, thr, [&](int c) { return __ldcg(slices + c); }, base);
  const unsigned long long tl = thr - base;
  // the run: lane l holds runs [4l, 4l + 4)
  constexpr int kPer = kSpThreads / 32;
  const unsigned long long *runs = sw.runs + ((size_t)b * NS + s) * kSpThreads;
  unsigned long long rs[kPer], own = 0;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int ri = lane * kPer + k;
    if (recompute) {  // E of the q row over run ri of slice s
      Acc40 P{0ull, 0ull};
#pragma unroll
      for (int w = 0; w < sp_wpt<E>(); ++w) {
        const uint4 q = load_word<E>((const E *)p.rq,
                                     s * kSpSlice + (ri * sp_wpt<E>() + w) * sp_per<E>(), r.V,
                                     p.vec);
#pragma unroll
        for (int j = 0; j < sp_per<E>(); j += 2)
          acc40(P, exp32x2(arg2(word_elem<E>(q, j), word_elem<E>(q, j + 1), p.mzq, p.mzq, r.invT,
                                p.unit_t)));
      }
      unsigned long long s0 = 0, s1 = 0;
      drain40(P, s0, s1);
      rs[k] = s0 + s1;
    } else {
      rs[k] = __ldcg(runs + ri);
    }
    own += rs[k];
  }
  const unsigned long long inc = warp_incl_scan_u64(own);
  const unsigned hit_g = __ballot_sync(0xffffffffu, inc > tl);
  const int lh = hit_g ? __ffs(hit_g) - 1 : 31;  // tl < the slice sum: some lane crosses
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
  const int ri = __shfl_sync(0xffffffffu, lane * kPer + k_hit, lh);
  const unsigned long long tb = tl - __shfl_sync(0xffffffffu, base_k, lh);
  // the run's 32 elements, one per lane
  const int v = s * kSpSlice + 32 * ri + lane;
  const unsigned long long wt = weight_elem<E>(r, p, v, t.iq, t.ip, use_q);
  const unsigned long long incw = warp_incl_scan_u64(wt);
  const unsigned hit = __ballot_sync(0xffffffffu, incw > tb);
  const int l = __ffs(hit) - 1;
  if (lane == l) {
    const unsigned long long c = incw - wt;
    const unsigned long long b_lo = tb - c, b_hi = c + wt - 1ull - tb;
    const int Wd = r.maxpos + 1;
    o.tokens[(size_t)b * Wd + t.a] = v;
    if (o.margin)
      o.margin[(size_t)b * Wd + r.maxpos] =
          (float)((double)(b_lo < b_hi ? b_lo : b_hi) / (double)S);
    if (p.resid && use_q) o.status[b] |= SV_ROW_RESID_ZERO;
  }
}

// The producer warp finishes an item whose results the consumers have stored
// (their arrivals on the stage's "empty" barrier precede this): the item is
// counted for its sequence, and the warp that completes a sequence's bonus
// pass or residual pass 2 picks its token.
template <typename E>
__device__ __forceinline__ void finish_item(const Round &r, const ItemMeta &m, const SampleWs &sw,
                                            const DecideOut &o) {
  if (m.kind < 0 || (m.kind == 2 && !m.ok)) return;
  const int lane = threadIdx.x & 31;
  unsigned old = 0;
  if (lane == 0) {
    __threadfence();  // the consumers' sums (seen through the barrier) before the count
    old = atomicAdd(sw.done + (m.kind == 2 ? sw.B + m.b : m.b), 1u);
  }
  old = __shfl_sync(0xffffffffu, old, 0);
  if (old != (unsigned)(sw.NS - 1) || m.kind == 0) return;
  __threadfence();  // the other CTAs' sums of this sequence, after the count
  if (m.kind == 1) {
    pick_token_warp<E>(r, m, m.b, sw, sw.slice + (size_t)m.b * sw.NS, true, false, o);
    return;
  }
  const unsigned long long *slw = sw.slice + ((size_t)2 * sw.B + m.b) * sw.NS;
  unsigned long long Sw = 0;
  for (int c = lane; c < sw.NS; c += 32) Sw += __ldcg(slw + c);
  if (warp_sum_u64(Sw) != 0ull)
    pick_token_warp<E>(r, m, m.b, sw, slw, false, false, o);
  else  // residual mass 0 (q == p to the last bit): the draw from q
    pick_token_warp<E>(r, m, m.b, sw, sw.slice + (size_t)m.b * sw.NS, true, true, o);
}

// bf16: five CTAs per SM (at most 72 registers, no spills) keep more
// consumer warps resident than four; fp32 would spill at that cap
template <typename E>
__global__ void __launch_bounds__(kSpThreads + 32, sizeof(E) == 2 ? 5 : 4)
sample_kernel(Round r, const Task *__restrict__ tasks, SampleWs sw, DecideOut o) {
  grid_dep_sync();
  extern __shared__ __align__(128) uint4 stage_sm[];  // [2 stages][q, p][words]
  __shared__ SampleSmem sm;
  constexpr int kW = sp_words<E>();
  const int tid = threadIdx.x, NS = sw.NS;
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      ring_init(ring_addr(&sm.full[i]), 1);            // the producer's arrival (+ bytes)
      ring_init(ring_addr(&sm.empty[i]), kSpThreads);  // every consumer, results stored
      ring_init(ring_addr(&sm.reduced[i]), kSpWarps);   // lane 0 of every consumer warp
      sm.meta[i].kind = -1;
    }
    sm.abort = 0;
  }
  __syncthreads();
  volatile int *abort = &sm.abort;
  if (tid >= kSpThreads) {
    // ------------------------------------------------------ producer / finisher
    const int lane = tid - kSpThreads;
    const int R = (int)__ldcg(sw.qc), Bn = (int)__ldcg(sw.qc + 1);
    const int n1r = R * NS, n1 = n1r + Bn * NS, total = n1 + R * NS;
    ItemMeta held[2];  // the item each stage holds, finished once it is released
    held[0].kind = held[1].kind = -1;
    int n = 0;
    for (;; ++n) {
      const int slot = n & 1;
      if (n >= 2) {
        if (!ring_wait(ring_addr(&sm.empty[slot]), ((n >> 1) - 1) & 1, abort)) break;
        finish_item<E>(r, held[slot], sw, o);
        held[slot].kind = -1;
      }
      int i = 0;
      if (lane == 0) i = *abort ? total : (int)atomicAdd(sw.qc + 2, 1u);
      i = __shfl_sync(0xffffffffu, i, 0);
      ItemMeta m;
      m.kind = -1;
      m.nbulk = 0;
      if (i < total) {
        int b, s;
        if (i < n1r) {
          m.kind = 0;
          b = sw.rlist[i / NS];
          s = i % NS;
        } else if (i < n1) {
          m.kind = 1;
          b = sw.blist[(i - n1r) / NS];
          s = (i - n1r) % NS;
        } else {
          m.kind = 2;
          b = sw.rlist[(i - n1) / NS];
          s = (i - n1) % NS;
        }
        const Task t = tasks[b];
        m.rq = t.rq;
        m.rp = t.rp;
        m.mq = t.mq;
        m.mp = t.mp;
        m.u24 = t.u24;
        m.a = t.a;
        m.b = b;
        m.s = s;
        m.ok = 1;
        m.iq = m.ip = 0.0f;
        if (m.kind == 2) {
          // The sequence's pass 1 must be complete (bounded wait).  The item
          // in flight in the other stage may be one of those pass-1 items: it
          // is counted here as soon as its consumers are done, or this wait
          // could never end.
          const int other = (n + 1) & 1;
          const unsigned long long t0 = ring_ns();
          for (;;) {
            unsigned done = 0;
            if (lane == 0) done = ld_acquire(sw.done + b);
            done = __shfl_sync(0xffffffffu, done, 0);
            if (done >= (unsigned)NS) break;
            if (held[other].kind >= 0 && n >= 1 &&
                ring_try(ring_addr(&sm.empty[other]), ((n - 1) >> 1) & 1)) {
              finish_item<E>(r, held[other], sw, o);
              held[other].kind = -1;
              continue;
            }
            if (ring_ns() - t0 > kRingWaitNs) {
              m.ok = 0;
              break;
            }
            __nanosleep(64);
          }
          const float2 iv = resid_inv(sw, b);
          m.iq = iv.x;
          m.ip = iv.y;
          if (!m.ok && lane == 0) atomicOr(o.status + b, SV_ROW_TIMEOUT);
        }
        // the words of the slice that lie inside an aligned row: one bulk copy
        // per row (the consumers read the rest themselves)
        const RowPair p = row_pair<E>(r, t);
        const int left = r.V - s * kSpSlice;
        m.nbulk = p.vec ? (left < kSpSlice ? left : kSpSlice) / sp_per<E>() : 0;
      }
      const uint32_t bytes = (uint32_t)m.nbulk * 16u * (m.kind == 1 ? 1u : 2u);
      if (lane == 0) {
        sm.meta[slot] = m;
        ring_expect_tx(ring_addr(&sm.full[slot]), bytes);  // arrival (release) + expected bytes
        if (bytes) {
          const uint32_t dst = ring_addr(stage_sm + (size_t)(2 * slot) * kW);
          const size_t off = (size_t)m.s * kSpSlice * sizeof(E);
          ring_bulk(dst, (const char *)m.rq + off, (uint32_t)m.nbulk * 16u,
                       ring_addr(&sm.full[slot]));
          if (m.kind != 1)
            ring_bulk(dst + (uint32_t)kW * 16u, (const char *)m.rp + off,
                         (uint32_t)m.nbulk * 16u, ring_addr(&sm.full[slot]));
        }
      }
      __syncwarp();
      held[slot] = m;
      if (m.kind < 0) break;
    }
    // the item still held by the other stage: released once the consumers are done
    const int other = (n + 1) & 1;
    if (!*abort && held[other].kind >= 0 && n >= 1 &&
        ring_wait(ring_addr(&sm.empty[other]), ((n - 1) >> 1) & 1, abort))
      finish_item<E>(r, held[other], sw, o);
    // after an abort, let this CTA's bulk copies in flight land before it exits
    if (*abort && lane == 0) {
      for (int k = n - 1; k <= n; ++k) {
        if (k < 0) continue;
        const unsigned long long t0 = ring_ns();
        while (!ring_try(ring_addr(&sm.full[k & 1]), (k >> 1) & 1) && ring_ns() - t0 < kRingWaitNs) {
        }
      }
    }
    return;
  }
  // ---------------------------------------------------------------- consumers
  for (int n = 0;; ++n) {
    const int slot = n & 1;
    if (!ring_wait(ring_addr(&sm.full[slot]), (n >> 1) & 1, abort)) {
      if (tid == 0 && sm.meta[slot].kind >= 0) atomicOr(o.status + sm.meta[slot].b, SV_ROW_TIMEOUT);
      break;
    }
    const ItemMeta m = sm.meta[slot];
    if (m.kind < 0) break;
    const int b = m.b, s = m.s;
    if (m.kind == 2 && !m.ok) {
      // nothing computed; both barriers still complete their phase for it
      if ((tid & 31) == 0) ring_arrive(ring_addr(&sm.reduced[slot]));
      ring_arrive(ring_addr(&sm.empty[slot]));
      continue;
    }
    const RowPair p = row_pair<E>(r, m);
    const uint4 *sq = stage_sm + (size_t)(2 * slot) * kW;
    uint4 wq[sp_wpt<E>()], wp[sp_wpt<E>()];
    fetch_run<E>(wq, sq, (const E *)p.rq, r.V, s, m.nbulk);
    if (m.kind != 1) fetch_run<E>(wp, sq + kW, (const E *)p.rp, r.V, s, m.nbulk);
    unsigned long long f0, f1 = 0;
    if (m.kind == 0) {
      run_e40_pair<E>(r, p, wq, wp, f0, f1);
    } else if (m.kind == 1) {
      f0 = run_e40<E>(r, p, wq);
    } else {
      f0 = run_w62<E>(r, p, wq, wp, m.iq, m.ip);
    }
    // run sums (bonus E, residual W) and the slice sums
    if (m.kind != 0) sw.runs[((size_t)b * NS + s) * kSpThreads + tid] = f0;
    // (per-stage buffers: a warp can be one item ahead of thread 0's reads,
    // never two, since the stage is refilled only after thread 0 releases it)
    f0 = warp_sum_u64(f0);
    f1 = warp_sum_u64(f1);
    if ((tid & 31) == 0) {
      sm.red[slot][0][tid >> 5] = f0;
      sm.red[slot][1][tid >> 5] = f1;
      ring_arrive(ring_addr(&sm.reduced[slot]));
    }
    // warps 1-3 release the stage now (their stores precede the arrival);
    // warp 0 once thread 0 has combined the warps' sums (a bounded wait on
    // the stage's "reduced" barrier), so that no warp writes them for a
    // later item first
    if (tid >= 32) {
      ring_arrive(ring_addr(&sm.empty[slot]));
      continue;
    }
    if (!ring_wait(ring_addr(&sm.reduced[slot]), (n >> 1) & 1, abort)) {
      if (tid == 0) atomicOr(o.status + b, SV_ROW_TIMEOUT);
      break;
    }
    if (tid == 0) {
      unsigned long long a0 = 0, a1 = 0;
      for (int w = 0; w < kSpWarps; ++w) {
        a0 += sm.red[slot][0][w];
        a1 += sm.red[slot][1][w];
      }
      const int which = m.kind == 2 ? 2 : 0;
      sw.slice[((size_t)which * sw.B + b) * NS + s] = a0;
      if (m.kind == 0) sw.slice[((size_t)sw.B + b) * NS + s] = a1;
    }
    // every consumer's stores precede its arrival: the producer then counts
    // the item (and may pick) and reuses the stage
    ring_arrive(ring_addr(&sm.empty[slot]));
  }
}

// ---------------------------------------------------------------------------
// tree_path: one warp per sequence.  Validates the tree, walks best children
// (highest score; ties to the lower slot) at most max_depth steps.  Every
// node's best child comes from one parallel pass (a 64-bit shared-memory
// maximum per parent of the key (score in a monotone integer order, ~slot)),
// so the walk itself is a chain of max_depth shared-memory loads.
// A listed row: bits 0-29 its row in the verifier / draft logits
// (b T + node), bit 30 draft, bits 32-43 its row slot, bits 44-63 b.
__device__ __forceinline__ uint64_t list_entry(int b, int slot, bool draft, long long row) {
  return (uint64_t)row | ((uint64_t)draft << 30) | ((uint64_t)slot << 32) | ((uint64_t)b << 44);
}

__device__ __forceinline__ unsigned long long child_key(float s, int c) {
  const unsigned u = __float_as_uint(__fadd_rn(s, 0.0f));  // -0 joins +0: they compare equal
  const unsigned o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)o << 32) | (0xffffffffu - (unsigned)c);
}

__global__ void __launch_bounds__(32)
tree_path_kernel(const int32_t *__restrict__ parent, const int32_t *__restrict__ token,
                 const float *__restrict__ score, int B, int T, int max_depth,
                 int32_t *__restrict__ path, int32_t *__restrict__ npos,
                 int32_t *__restrict__ tok, int tok_stride, uint32_t *__restrict__ tstat,
                 uint64_t *__restrict__ rowlist, int *__restrict__ rowcount, int greedy) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int b = blockIdx.x, lane = threadIdx.x;
  __shared__ int32_t pa[SV_MAX_TREE_NODES];
  __shared__ float sc[SV_MAX_TREE_NODES];
  __shared__ int32_t tk[SV_MAX_TREE_NODES];
  __shared__ unsigned long long best[SV_MAX_TREE_NODES];  // 0: no child
  __shared__ int32_t pn[SV_MAX_POSITIONS + 1];  // the path, written out at the end
  for (int c = lane; c < T; c += 32) {  // one coalesced pass over the tree
    pa[c] = parent[(size_t)b * T + c];
    sc[c] = score[(size_t)b * T + c];
    tk[c] = token[(size_t)b * T + c];
    best[c] = 0ull;
  }
  // the next grid (the row pass) starts streaming its root rows once this
  // grid's few loads have returned, not while they are in flight
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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
      tstat[b] = SV_ROW_BAD_TREE;  // (its root rows are read by their own CTAs)
    }
    return;
  }
  // valid tree: every live node c > 0 has a live parent p < c and a score
  // that is not NaN, so the keys order exactly as the scores do
  for (int c = 1 + lane; c < T; c += 32) {
    const int p = pa[c];
    if (p >= 0) atomicMax(&best[p], child_key(sc[c], c));
  }
  __syncwarp();
  int D = 0;
  if (lane == 0) {
    int cur = 0;
    pn[0] = 0;
    while (D < max_depth) {
      const unsigned long long k = best[cur];
      if (k == 0ull) break;
      cur = (int)(0xffffffffu - (unsigned)k);
      pn[++D] = cur;
    }
  }
  D = __shfl_sync(0xffffffffu, D, 0);
  __syncwarp();
  // the path and its tested tokens token[n_1..n_D], written in parallel
  for (int i = lane; i <= D; i += 32) pth[i] = pn[i];
  for (int i = lane; i < D; i += 32) tok[(size_t)b * tok_stride + i] = tk[pn[i + 1]];
  // the path's rows other than the root's (the row pass reads those without
  // waiting for this grid): the verifier rows n_1..n_D, then (stochastic
  // rule) the draft rows n_1..n_{D-1}
  const int nrow = D == 0 ? 0 : (greedy ? D : 2 * D - 1);
  int base = 0;
  if (lane == 0) {
    npos[b] = D;
    tstat[b] = 0u;
    if (nrow) base = atomicAdd(rowcount, nrow);
  }
  base = __shfl_sync(0xffffffffu, base, 0);
  for (int k = lane; k < nrow; k += 32) {
    // verifier row of path position k + 1, or draft row of position k - D + 1
    const bool draft = k >= D;
    const int i = draft ? k - D + 1 : k + 1;
    rowlist[base + k] =
        list_entry(b, draft ? max_depth + 1 + i : i, draft, (long long)b * T + pn[i]);
  }
}

// ---------------------------------------------------------------------------
// Tree row-pass grids: gridDim.y holds the root-row CTAs then the listed-row
// CTAs (at most 65535 in all); either kind loops when there are more rows.
int tree_root_ctas(int root_rows) { return root_rows < 32768 ? root_rows : 32768; }
int tree_list_ctas(int list_slots, int nroot) {
  // half as many CTAs as listed-row slots: one takes a second row when the
  // paths are deep
  const int want = (list_slots + 1) / 2 > 0 ? (list_slots + 1) / 2 : 1;
  return want < 65535 - nroot ? want : 65535 - nroot;
}

// ---------------------------------------------------------------------------
// Persistent grids (the row passes' bulk rings, the sampler): every SM filled
// with as many CTAs as fit, looked up once per device and kernel (`which`
// tells apart kernels of one signature: 0 sampler, 1 statistics, 2 arg max).
template <typename E, typename K>
int persistent_grid(K k, int which, size_t smem, int threads) {
  static std::mutex mu;
  static int cache[64][3] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lk(mu);
  if (!cache[dev][which]) {
    // (dynamic plus static shared memory may pass 48 KB below 48 KB dynamic)
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return 0;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, threads, smem) !=
            cudaSuccess ||
        per_sm < 1)
      return 0;
    cache[dev][which] = per_sm * num_sms();
  }
  return cache[dev][which];
}

template <typename E>
sv_status launch_sampler(const Round &r, const Layout &L, char *ws, const Task *tasks,
                         const DecideOut &o, cudaStream_t st) {
  SampleWs sw;
  sw.slice = (unsigned long long *)(ws + L.slice);
  sw.runs = (unsigned long long *)(ws + L.runs);
  sw.done = (unsigned *)(ws + L.done);
  sw.rlist = (const int *)(ws + L.rlist);
  sw.blist = sw.rlist + r.B;
  sw.qc = (unsigned *)(ws + L.qc);
  sw.NS = L.NS;
  sw.B = r.B;
  const size_t smem = 2 * sp_stage_bytes<E>();
  // at most 2 B NS items: never more CTAs than that
  const long long items = 2LL * r.B * L.NS;
  const int g = persistent_grid<E>(sample_kernel<E>, 0, smem, kSpThreads + 32);
  if (!g) return set_error(SV_ERR_CUDA, "sample: occupancy query");
  LaunchScope ls("sample", st);
  return check_launch("sample",
                      launch_pdl(sample_kernel<E>, dim3((unsigned)(items < g ? items : g)),
                                 dim3(kSpThreads + 32), smem, st, r, tasks, sw, o));
}

// A row pass over device-resident logits: the persistent bulk-ring grid,
// never more CTAs than units (tree: root units and every listed-row slot).
// qc: the sampler's counters to zero (statistics pass), or null.
template <typename E, bool kArg>
sv_status launch_row_pass_bulk(const char *name, const Round &r, int G, const uint64_t *rowlist,
                               const int *rowcount, float4 *partial, unsigned *qc,
                               cudaStream_t st) {
  const size_t smem = (size_t)kRbStages * kRbChunk;
  const int g = persistent_grid<E>(row_pass_bulk_kernel<E, kArg>, kArg ? 2 : 1, smem, kRbThreads);
  if (!g) return set_error(SV_ERR_CUDA, "%s: occupancy query", name);
  const long long units = (long long)r.B * r.P * G;
  // the unit counter sits after the row count; a tree call zeroed both before
  // its path walk, a chain zeroes it here
  unsigned long long *next_unit = (unsigned long long *)((char *)rowcount + 8);
  if (!rowlist && cudaMemsetAsync(next_unit, 0, 8, st) != cudaSuccess)
    return set_error(SV_ERR_CUDA, "%s: unit counter reset", name);
  LaunchScope ls(name, st);
  return check_launch(name, launch_pdl(row_pass_bulk_kernel<E, kArg>,
                                       dim3((unsigned)(units < g ? units : g)), dim3(kRbThreads),
                                       smem, st, r, G, rowlist, rowcount, next_unit, partial, qc));
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
                                                r, G, partial, count, stop, seed, step,
                                                (unsigned *)(ws + L.qc)));
    if (s != SV_OK) return s;
  } else {
    const uint64_t *rowlist = r.path ? (const uint64_t *)(ws + L.rowlist) : nullptr;
    if (r.stage && !r.copy) {
      s = launch_row_pass_bulk<E, false>("row_stats", r, G, rowlist, (const int *)(ws + L.ctr),
                                         partial, (unsigned *)(ws + L.qc), st);
    } else {
      // host-resident logits: one CTA per (row, segment); tree: B * P row
      // slots bound the listed rows, half as many CTAs per segment, each
      // taking a second row when the paths are deep
      dim3 grid((unsigned)(r.B * r.P), (unsigned)G);
      int nroot = 0;
      if (rowlist) {  // tree: (segment, root CTAs + listed-row CTAs)
        const int R0 = r.maxpos == 0 ? 1 : 2;  // root rows per sequence (root_rows)
        nroot = tree_root_ctas(R0 * r.B);
        grid = dim3((unsigned)G, (unsigned)(nroot + tree_list_ctas(r.B * (r.P - R0), nroot)));
      }
      LaunchScope ls("row_stats", st);
      s = check_launch("row_stats", launch_pdl(r.copy ? row_stats_kernel<E, true>
                                                      : row_stats_kernel<E, false>,
                                               grid, dim3(kRsThreads), 0, st, r, G, rowlist,
                                               (const int *)(ws + L.ctr), partial,
                                               (unsigned *)(ws + L.qc), nroot));
    }
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
                                          step, o, tasks, (int *)(ws + L.rlist),
                                          (unsigned *)(ws + L.qc), (unsigned *)(ws + L.done)));
    if (s != SV_OK) return s;
  }
  if (accept_event) {
    const cudaError_t e = cudaEventRecord(accept_event, st);
    if (e != cudaSuccess) return set_error(SV_ERR_CUDA, "accept_event: %s", cudaGetErrorString(e));
  }
  if ((s = launch_sampler<E>(r, L, ws, tasks, o, st)) != SV_OK) return s;
  return SV_OK;
}

template <typename E>
sv_status run_verify_greedy(const Round &r, const Layout &L, char *ws, const DecideOut &o,
                            cudaStream_t st, cudaEvent_t accept_event) {
  float4 *partial = (float4 *)(ws + L.partial);
  const int G = (r.V + seg_elems<E>() - 1) / seg_elems<E>();
  sv_status s;
  {
    const uint64_t *rowlist = r.path ? (const uint64_t *)(ws + L.rowlist) : nullptr;
    if (r.stage) {
      s = launch_row_pass_bulk<E, true>("row_argmax", r, G, rowlist, (const int *)(ws + L.ctr),
                                        partial, nullptr, st);
    } else {
      // host-resident logits: one CTA per (row, segment)
      dim3 grid((unsigned)(r.B * r.P), (unsigned)G);
      int nroot = 0;
      if (rowlist) {  // tree: (segment, root CTAs + listed-row CTAs)
        nroot = tree_root_ctas(r.B);
        grid = dim3((unsigned)G, (unsigned)(nroot + tree_list_ctas(r.B * (r.P - 1), nroot)));
      }
      LaunchScope ls("row_argmax", st);
      s = check_launch("row_argmax", launch_pdl(row_argmax_kernel<E>, grid, dim3(kRsThreads), 0,
                                                st, r, G, rowlist, (const int *)(ws + L.ctr),
                                                partial, nroot));
    }
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
  if ((long long)B * L.P > 0x7fffffffLL || (long long)B * L.NS > 0x7fffffffLL)
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
  if (cudaMemsetAsync(ws + L.ctr, 0, 16, st) != cudaSuccess)
    return check_launch("row counter reset");
  {
    LaunchScope ls("tree_path", st);
    s = check_launch("tree_path",
                     launch_pdl(tree_path_kernel, dim3(B), dim3(32), 0, st, parent, token, score,
                                B, T, max_depth, path, npos, tok, max_depth > 0 ? max_depth : 1,
                                tstat, (uint64_t *)(ws + L.rowlist), (int *)(ws + L.ctr),
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
namespace sv {
namespace {
constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB
constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void *g_static_ptr[kMaxDevices] = {};
}  // namespace
}  // namespace sv

static __device__ __align__(256) unsigned char g_static_scratch[sv::kStaticScratchBytes];

namespace sv {
namespace {
// a non-null stand-in for the argument checks, which want a workspace pointer;
// the host-side name of the array is never dereferenced or passed to a kernel
const void *g_static_scratch_host_name() { return (const void *)&g_static_scratch; }

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
  // the argument checks of sv_verify_chain, in its order, before the
  // capacity check (the scratch itself is never null)
  sv_status s = check_common(vlogits, dt, B, V, temperature, out_tokens, out_accept_len,
                             out_status, g_static_scratch_host_name());
  if (s != SV_OK || B == 0) return s;
  if (N < 0) return set_error(SV_ERR_INVALID_ARG, "N must be >= 0 (got %d)", N);
  if (N > SV_MAX_POSITIONS) return set_error(SV_ERR_UNSUPPORTED, "N > %d", SV_MAX_POSITIONS);
  if (N > 0 && (!dlogits || !draft_tokens))
    return set_error(SV_ERR_INVALID_ARG, "dlogits and draft_tokens are required when N > 0");
  const size_t need = sv_verify_chain_workspace(B, N, V);
  if (need > kStaticScratchBytes)
    return set_error(SV_ERR_UNSUPPORTED,
                     "sv_verify_chain_noalloc: B=%d N=%d V=%d needs %zu bytes of scratch, "
                     "more than the %zu-byte static scratch; use sv_verify_chain with a "
                     "caller-owned workspace",
                     B, N, V, need, kStaticScratchBytes);
  void *ws = nullptr;
  s = static_scratch_address(&ws);
  if (s != SV_OK) return s;
  return sv_verify_chain(vlogits, dlogits, dt, draft_tokens, B, N, V, temperature, seed, step,
                         out_tokens, out_accept_len, out_q_prob, out_p_prob, out_margin,
                         out_status, ws, kStaticScratchBytes, stream, accept_event);
}
