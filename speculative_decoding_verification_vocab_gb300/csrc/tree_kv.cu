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
constexpr int kKvGroup = 8;  // rows loaded before any is stored

// ---------------------------------------------------------------------------
// ancestor mask: one CTA per sequence; node n walks its parent chain and sets
// bit j (j on the chain) in word j/64.  Validation mirrors sv_verify_tree.
__global__ void __launch_bounds__(kMaskThreads)
tree_mask_kernel(const int32_t *__restrict__ parent, int T, int W, uint64_t *__restrict__ mask,
                 int32_t *__restrict__ depth) {
  const int b = blockIdx.x;
  const int32_t *pa = parent + (size_t)b * T;
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
// Every warp validates the request on its own (no block barrier): lanes read
// 32 row indices at a time and vote.  Then each thread owns (slab, 16-byte
// column) units and moves the rows in groups of kKvGroup: all loads of a
// group, then its stores, groups in increasing k.  In place, rows[k] >= k and
// strictly increasing mean a later group never reads a slot an earlier group
// wrote, and a group's reads precede its writes; rows[k] == k are skipped.
constexpr int kKvSlabs = 8;
constexpr int kKvMaxRows = 4096;

struct KvArgs {
  const char *src;
  char *dst;
  int L, B, S_src, S_dst;
  size_t row_bytes;
  const int32_t *src_base, *dst_base, *rows, *n_rows;
  int n_add, P;
  int32_t *kv_len;
  int inplace, vec;
};

__global__ void __launch_bounds__(kKvThreads) kv_compact_kernel(KvArgs a) {
  const int b = blockIdx.x;
  const int lane = threadIdx.x & 31;
  const unsigned FULL = 0xffffffffu;
  const int n = a.n_rows[b] + a.n_add;
  const int sb = a.src_base[b], db = a.dst_base[b];
  bool ok = n >= 0 && n <= a.P && n <= kKvMaxRows && sb >= 0 && db >= 0 &&
            (long)db + n <= a.S_dst && !(a.inplace && sb != db);
  const int32_t *rows = a.rows ? a.rows + (size_t)b * a.P : nullptr;
  int prev_last = -1;
  for (int k0 = 0; ok && k0 < n; k0 += 32) {
    const int k = k0 + lane;
    const bool in = k < n;
    const int r = in ? (rows ? rows[k] : k) : 0;
    int prev = __shfl_up_sync(FULL, r, 1);
    if (lane == 0) prev = prev_last;
    bool bad = in && (r < 0 || (long)sb + r >= a.S_src);
    if (a.inplace) bad = bad || (in && (r < k || r <= prev));
    if (__any_sync(FULL, bad)) ok = false;
    prev_last = __shfl_sync(FULL, r, 31);
  }
  if (blockIdx.y == 0 && threadIdx.x == 0) a.kv_len[b] = ok ? db + n : -1;
  if (!ok || n == 0) return;
  const int slab0 = blockIdx.y * kKvSlabs;
  const int nslab = min(kKvSlabs, 2 * a.L - slab0);
  const size_t ncol = a.vec ? a.row_bytes / 16 : a.row_bytes;
  const size_t units = (size_t)nslab * ncol;
  const size_t sbase_off = (size_t)sb * a.row_bytes, dbase_off = (size_t)db * a.row_bytes;
  for (int k0 = 0; k0 < n; k0 += 32) {
    // this chunk's moves: lane j holds row k0 + j
    const int kn = min(32, n - k0);
    const int my_r = lane < kn ? (rows ? rows[k0 + lane] : k0 + lane) : 0;
    for (int g0 = 0; g0 < kn; g0 += kKvGroup) {
      int rr[kKvGroup];  // warp-uniform: broadcast before the divergent unit loop
#pragma unroll
      for (int j = 0; j < kKvGroup; ++j) rr[j] = __shfl_sync(FULL, my_r, (g0 + j) & 31);
      for (size_t u = threadIdx.x; u < units; u += kKvThreads) {
        const int sl = (int)(u / ncol);
        const size_t c = u - (size_t)sl * ncol;
        const size_t slab = (size_t)(slab0 + sl) * a.B + b;
        const char *sp = a.src + slab * a.S_src * a.row_bytes + sbase_off;
        char *dp = a.dst + slab * a.S_dst * a.row_bytes + dbase_off;
        if (a.vec) {
          uint4 v[kKvGroup];
#pragma unroll
          for (int j = 0; j < kKvGroup; ++j) {
            const int k = k0 + g0 + j;
            if (g0 + j < kn && !(a.inplace && rr[j] == k))
              v[j] = ld_stream_v4(sp + (size_t)rr[j] * a.row_bytes + c * 16);
          }
#pragma unroll
          for (int j = 0; j < kKvGroup; ++j) {
            const int k = k0 + g0 + j;
            if (g0 + j < kn && !(a.inplace && rr[j] == k))
              *(uint4 *)(dp + (size_t)k * a.row_bytes + c * 16) = v[j];
          }
        } else {
          char v[kKvGroup];
#pragma unroll
          for (int j = 0; j < kKvGroup; ++j)
            if (g0 + j < kn) v[j] = sp[(size_t)rr[j] * a.row_bytes + c];
#pragma unroll
          for (int j = 0; j < kKvGroup; ++j)
            if (g0 + j < kn) dp[(size_t)(k0 + g0 + j) * a.row_bytes + c] = v[j];
        }
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
  cudaStream_t st = (cudaStream_t)stream;
  LaunchScope ls("tree_mask", st);
  tree_mask_kernel<<<B, kMaskThreads, 0, st>>>(parent, T, (T + 63) / 64, out_mask, out_depth);
  return check_launch("tree_mask");
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
  cudaStream_t st = (cudaStream_t)stream;
  LaunchScope ls("kv_compact", st);
  kv_compact_kernel<<<dim3(B, (2 * L + kKvSlabs - 1) / kKvSlabs), kKvThreads, 0, st>>>(a);
  return check_launch("kv_compact");
}
