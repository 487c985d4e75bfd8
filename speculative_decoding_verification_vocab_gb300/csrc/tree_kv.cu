// tree_kv.cu -- the tree attention mask and KV rollback / compaction (sm_103a).
//
// Pages: "投机解码发展" (blog; section 3: flattened tree, each node sees only
// itself and its ancestors; the accepted path's KV rows are copied together
// and the other branches dropped; compact_kv in the section 4 listing) and
// "Decodificação Especulativa e EAGLE-3" (lesson; "Reversão de KV cache",
// Passo 4: logical length truncated on rejection, or scratch committed on
// acceptance).
#include "common.cuh"

namespace sv {
namespace {

constexpr int kMaskThreads = 256;
constexpr int kKvThreads = 256;

// ---------------------------------------------------------------------------
// ancestor mask: one CTA per sequence; node n walks its parent chain and sets
// bit j (j on the chain) in word j/64.  Validation mirrors sv_verify_tree.
__global__ void __launch_bounds__(kMaskThreads)
tree_mask_kernel(const int32_t *__restrict__ parent, int T, int W, uint64_t *__restrict__ mask,
                 int32_t *__restrict__ depth) {
  grid_dep_sync();
  const int b = blockIdx.x;
  __shared__ int32_t pa[SV_MAX_TREE_NODES];
  for (int c = threadIdx.x; c < T; c += kMaskThreads) pa[c] = parent[(size_t)b * T + c];
  __syncthreads();
  int ok = 1;
  for (int c = threadIdx.x; c < T; c += kMaskThreads) {
    const int p = pa[c];
    if (c == 0)
      ok &= (p == -1);
    else if (p != -2)
      ok &= (p >= 0 && p < c) && (pa[p] != -2);
  }
  ok = __syncthreads_and(ok);
  for (int n = threadIdx.x; n < T; n += kMaskThreads) {
    uint64_t *mk = mask + ((size_t)b * T + n) * W;
    const bool used = ok && pa[n] != -2;
    if (W == 1) {  // one word: a single walk up the chain
      uint64_t bits = 0;
      int d = -1;
      if (used)
        for (int j = n; j >= 0; j = pa[j]) {
          bits |= 1ull << j;
          ++d;
        }
      mk[0] = bits;
      depth[(size_t)b * T + n] = used ? d : -1;
      continue;
    }
    int d = -1;
    for (int w = 0; w < W; ++w) {
      uint64_t bits = 0;
      if (used) {
        int cnt = -1;
        for (int j = n; j >= 0; j = pa[j]) {
          if ((j >> 6) == w) bits |= 1ull << (j & 63);
          ++cnt;
        }
        d = cnt;
      }
      mk[w] = bits;
    }
    depth[(size_t)b * T + n] = used ? d : -1;
  }
}

// ---------------------------------------------------------------------------
// KV compaction: one CTA per (sequence, group of kKvSlabs (layer, K/V) slabs).
// Warp 0 validates the request (lanes read 32 row indices at a time and vote)
// and lists the rows that actually move (in place, rows[k] == k stays) in
// shared memory, in increasing k.  Each thread then owns kUnits (slab, 16-byte
// column) units and walks its (unit, move) pairs unit by unit, in batches of
// kKvBatch: all loads of a batch, then its stores.  In place, rows[k] >= k and
// strictly increasing mean a later batch never reads a slot an earlier one
// wrote (a unit's moves go in increasing k), and a batch's reads precede its
// writes; different threads touch different columns or slabs.
constexpr int kKvSlabs = 16;
constexpr int kKvMaxRows = 4096;
constexpr int kKvBatch = 8;

struct KvArgs {
  const char *src;
  char *dst;
  int L, B, S_src, S_dst;
  size_t row_bytes;
  const int32_t *src_base, *dst_base, *rows, *n_rows;
  int n_add, P;
  int32_t *kv_len;
  int inplace, vec, copy;
  int ncol;             // units per row: 16-byte words (vec) or bytes
  int step_sl, step_c;  // kKvThreads units = step_sl rows + step_c units
  int mcap;             // room for moves in shared memory: min(P, kKvMaxRows), >= 1
};

struct KvCursor {
  int sl, c;  // slab (relative to the CTA's first) and column of the unit
  int mv;     // move index
};
// next (unit, move) pair: the next move, or the first move of the next unit
__device__ __forceinline__ void kv_step(KvCursor &q, int nm, int step_sl, int step_c, int ncol) {
  if (++q.mv == nm) {
    q.mv = 0;
    q.c += step_c;
    q.sl += step_sl;
    if (q.c >= ncol) {
      q.c -= ncol;
      ++q.sl;
    }
  }
}

__global__ void __launch_bounds__(kKvThreads) kv_compact_kernel(KvArgs a) {
  grid_dep_sync();
  const int b = blockIdx.x;
  const int lane = threadIdx.x & 31;
  const unsigned FULL = 0xffffffffu;
  __shared__ int s_ok, s_nm;
  // the moves (at most min(P, kKvMaxRows) per sequence): sources, then targets
  extern __shared__ int s_moves[];
  int *s_src = s_moves, *s_dst = s_moves + a.mcap;
  if (threadIdx.x < 32) {
    const int n = a.n_rows[b] + a.n_add;
    const int sb = a.src_base[b], db = a.dst_base[b];
    bool ok = n >= 0 && n <= a.P && n <= kKvMaxRows && sb >= 0 && db >= 0 &&
              (long)db + n <= a.S_dst && !(a.inplace && sb != db);
    const int32_t *rows = a.rows ? a.rows + (size_t)b * a.P : nullptr;
    int nm = 0, prev_last = -1;
    for (int k0 = 0; ok && k0 < n; k0 += 32) {
      const int k = k0 + lane;
      const bool in = k < n;
      const int r = in ? (rows ? rows[k] : k) : 0;
      int prev = __shfl_up_sync(FULL, r, 1);
      if (lane == 0) prev = prev_last;
      bool bad = in && (r < 0 || (long)sb + r >= a.S_src);
      if (a.inplace) bad = bad || (in && (r < k || r <= prev));
      if (__any_sync(FULL, bad)) ok = false;
      const bool moves = in && !(a.inplace && r == k);
      const unsigned mm = __ballot_sync(FULL, moves);
      if (moves) {
        const int pos = nm + __popc(mm & ((1u << lane) - 1u));
        s_src[pos] = r;
        s_dst[pos] = k;
      }
      nm += __popc(mm);
      prev_last = __shfl_sync(FULL, r, 31);
    }
    if (lane == 0) {
      s_ok = ok;
      s_nm = nm;
      if (blockIdx.y == 0) a.kv_len[b] = ok ? db + n : -1;
    }
  }
  __syncthreads();
  if (!s_ok || !a.copy) return;
  const int nm = s_nm;
  if (nm == 0) return;
  const int slab0 = blockIdx.y * kKvSlabs;
  const int nslab = min(kKvSlabs, 2 * a.L - slab0);
  const size_t rb = a.row_bytes;
  // row 0 of this sequence's window in slab 0: [L][2][B][S][row_bytes]
  const char *src0 = a.src + ((size_t)b * a.S_src + a.src_base[b]) * rb;
  char *dst0 = a.dst + ((size_t)b * a.S_dst + a.dst_base[b]) * rb;
  const size_t src_slab = (size_t)a.B * a.S_src * rb, dst_slab = (size_t)a.B * a.S_dst * rb;
  const int ncol = a.ncol;  // units per row: 16-byte words, or bytes
  const long units = (long)nslab * ncol;
  const long my_units = units > threadIdx.x ? (units - 1 - threadIdx.x) / kKvThreads + 1 : 0;
  const long items = my_units * nm;
  // (unit, move) cursor, unit-major: unit = threadIdx.x + uu * kKvThreads
  // sits in slab slab0 + sl at column c; stepping a unit adds kKvThreads
  KvCursor cur{(int)(threadIdx.x / ncol), (int)(threadIdx.x % ncol), 0};
  const size_t colw = a.vec ? 16 : 1;
  for (long i0 = 0; i0 < items; i0 += kKvBatch) {
    const int cnt = (int)min((long)kKvBatch, items - i0);
    const KvCursor start = cur;
    auto src_of = [&](const KvCursor &q) {
      return src0 + (size_t)(slab0 + q.sl) * src_slab + (size_t)s_src[q.mv] * rb + q.c * colw;
    };
    auto dst_of = [&](const KvCursor &q) {
      return dst0 + (size_t)(slab0 + q.sl) * dst_slab + (size_t)s_dst[q.mv] * rb + q.c * colw;
    };
    if (a.vec) {
      uint4 v[kKvBatch];
#pragma unroll
      for (int j = 0; j < kKvBatch; ++j)
        if (j < cnt) {
          v[j] = ld_stream_v4(src_of(cur));
          kv_step(cur, nm, a.step_sl, a.step_c, ncol);
        }
      cur = start;
#pragma unroll
      for (int j = 0; j < kKvBatch; ++j)
        if (j < cnt) {
          *(uint4 *)dst_of(cur) = v[j];
          kv_step(cur, nm, a.step_sl, a.step_c, ncol);
        }
    } else {
      char v[kKvBatch];
#pragma unroll
      for (int j = 0; j < kKvBatch; ++j)
        if (j < cnt) {
          v[j] = *src_of(cur);
          kv_step(cur, nm, a.step_sl, a.step_c, ncol);
        }
      cur = start;
#pragma unroll
      for (int j = 0; j < kKvBatch; ++j)
        if (j < cnt) {
          *dst_of(cur) = v[j];
          kv_step(cur, nm, a.step_sl, a.step_c, ncol);
        }
    }
  }
}

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" sv_status sv_tree_build_mask(const int32_t *parent, int B, int T, uint64_t *out_mask,
                                        int32_t *out_depth, void *stream) {
  if (B < 0 || T < 1) return set_error(SV_ERR_INVALID_ARG, "need B >= 0 and T >= 1");
  if (T > SV_MAX_TREE_NODES) return set_error(SV_ERR_UNSUPPORTED, "T > %d", SV_MAX_TREE_NODES);
  if (B == 0) return SV_OK;
  if (!parent || !out_mask || !out_depth) return set_error(SV_ERR_INVALID_ARG, "null pointer");
  if ((uintptr_t)out_mask % 8) return set_error(SV_ERR_INVALID_ARG, "out_mask misaligned");
  sv_status s;
  if ((s = map_arg(parent, "parent")) != SV_OK || (s = map_arg(out_mask, "out_mask")) != SV_OK ||
      (s = map_arg(out_depth, "out_depth")) != SV_OK)
    return s;
  cudaStream_t st = (cudaStream_t)stream;
  LaunchScope ls("tree_mask", st);
  return check_launch("tree_mask", launch_pdl(tree_mask_kernel, dim3(B), dim3(kMaskThreads), 0, st,
                                              parent, T, (T + 63) / 64, out_mask, out_depth));
}

extern "C" sv_status sv_kv_compact(const void *src_kv, void *dst_kv, int L, int B, int S_src,
                                   int S_dst, int H, int D, int elem_bytes,
                                   const int32_t *src_base, const int32_t *dst_base,
                                   const int32_t *rows, const int32_t *n_rows, int n_rows_add,
                                   int P, int32_t *out_kv_len, void *stream) {
  if (L < 1 || B < 0 || S_src < 1 || S_dst < 1 || H < 1 || D < 1 || elem_bytes < 1 || P < 0)
    return set_error(SV_ERR_INVALID_ARG, "bad KV shape");
  if ((2L * L + kKvSlabs - 1) / kKvSlabs > 65535) return set_error(SV_ERR_UNSUPPORTED, "L too large");
  if (B == 0) return SV_OK;
  if (!src_kv || !dst_kv || !src_base || !dst_base || !n_rows || !out_kv_len)
    return set_error(SV_ERR_INVALID_ARG, "null pointer");
  sv_status s;
  if ((s = map_arg(src_kv, "src_kv")) != SV_OK || (s = map_arg(dst_kv, "dst_kv")) != SV_OK ||
      (s = map_arg(src_base, "src_base")) != SV_OK ||
      (s = map_arg(dst_base, "dst_base")) != SV_OK || (s = map_arg(rows, "rows")) != SV_OK ||
      (s = map_arg(n_rows, "n_rows")) != SV_OK || (s = map_arg(out_kv_len, "out_kv_len")) != SV_OK)
    return s;
  KvArgs a;
  a.src = (const char *)src_kv;
  a.dst = (char *)dst_kv;
  a.L = L;
  a.B = B;
  a.S_src = S_src;
  a.S_dst = S_dst;
  a.row_bytes = (size_t)H * D * elem_bytes;
  a.src_base = src_base;
  a.dst_base = dst_base;
  a.rows = rows;
  a.n_rows = n_rows;
  a.n_add = n_rows_add;
  a.P = P;
  a.kv_len = out_kv_len;
  a.inplace = (src_kv == dst_kv);
  a.vec = (a.row_bytes % 16 == 0) && ((uintptr_t)src_kv % 16 == 0) && ((uintptr_t)dst_kv % 16 == 0);
  // rows == NULL in place moves no byte (every row stays): validate and set
  // the lengths with one CTA per sequence
  a.copy = !(rows == nullptr && a.inplace);
  if (a.row_bytes / (a.vec ? 16 : 1) > 0x7fffffff)
    return set_error(SV_ERR_UNSUPPORTED, "KV row too long");
  a.ncol = (int)(a.row_bytes / (a.vec ? 16 : 1));
  a.step_sl = kKvThreads / a.ncol;
  a.step_c = kKvThreads % a.ncol;
  const unsigned gy = a.copy ? (unsigned)((2 * L + kKvSlabs - 1) / kKvSlabs) : 1u;
  // shared memory for the move lists sized by P (a few rows for a tree path),
  // so that the copy CTAs fit beside other kernels' CTAs on an SM
  a.mcap = P < kKvMaxRows ? (P > 0 ? P : 1) : kKvMaxRows;
  cudaStream_t st = (cudaStream_t)stream;
  LaunchScope ls("kv_compact", st);
  return check_launch("kv_compact", launch_pdl(kv_compact_kernel, dim3(B, gy), dim3(kKvThreads),
                                               2 * (size_t)a.mcap * sizeof(int), st, a));
}
