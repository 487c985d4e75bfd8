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
constexpr int kKvThreads = 128;
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
// KV compaction: one CTA per (sequence, layer, K/V).  Each thread owns a
// column of 16-byte words (or bytes on the unaligned path) across the kept
// rows; rows are moved in groups of kKvGroup: all loads of a group, then its
// stores.  In place, rows[k] >= k and strictly increasing guarantee that a
// later group never reads a slot an earlier group wrote, and a group's own
// reads precede its writes.
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

__device__ __forceinline__ int kv_rows_ok(const KvArgs &a, int b, int &n) {
  n = a.n_rows[b] + a.n_add;
  const int sb = a.src_base[b], db = a.dst_base[b];
  if (n < 0 || n > a.P || sb < 0 || db < 0 || (long)db + n > a.S_dst) return 0;
  if (a.inplace && sb != db) return 0;
  int prev = -1;
  for (int k = 0; k < n; ++k) {
    const int r = a.rows ? a.rows[(size_t)b * a.P + k] : k;
    if (r < 0 || (long)sb + r >= a.S_src) return 0;
    if (a.inplace && (r < k || r <= prev)) return 0;
    prev = r;
  }
  return 1;
}

__global__ void __launch_bounds__(kKvThreads) kv_compact_kernel(KvArgs a) {
  const int b = blockIdx.x;
  const int slab_i = blockIdx.y;  // l * 2 + kv
  __shared__ int s_ok, s_n;
  if (threadIdx.x == 0) {
    int n;
    const int ok = kv_rows_ok(a, b, n);
    s_ok = ok;
    s_n = n;
    if (slab_i == 0) a.kv_len[b] = ok ? a.dst_base[b] + n : -1;
  }
  __syncthreads();
  if (!s_ok) return;
  const int n = s_n;
  const size_t slab = (size_t)slab_i * a.B + b;
  const char *sbase = a.src + (slab * a.S_src + a.src_base[b]) * a.row_bytes;
  char *dbase = a.dst + (slab * a.S_dst + a.dst_base[b]) * a.row_bytes;
  const int32_t *rows = a.rows ? a.rows + (size_t)b * a.P : nullptr;
  for (int k0 = 0; k0 < n; k0 += kKvGroup) {
    const int kn = min(kKvGroup, n - k0);
    int rr[kKvGroup];
#pragma unroll
    for (int j = 0; j < kKvGroup; ++j) rr[j] = (j < kn) ? (rows ? rows[k0 + j] : k0 + j) : 0;
    if (a.vec) {
      const size_t nw = a.row_bytes / 16;
      for (size_t c = threadIdx.x; c < nw; c += kKvThreads) {
        uint4 v[kKvGroup];
#pragma unroll
        for (int j = 0; j < kKvGroup; ++j)
          if (j < kn && !(a.inplace && rr[j] == k0 + j))
            v[j] = ld_stream_v4(sbase + (size_t)rr[j] * a.row_bytes + c * 16);
#pragma unroll
        for (int j = 0; j < kKvGroup; ++j)
          if (j < kn && !(a.inplace && rr[j] == k0 + j))
            *(uint4 *)(dbase + (size_t)(k0 + j) * a.row_bytes + c * 16) = v[j];
      }
    } else {
      for (size_t c = threadIdx.x; c < a.row_bytes; c += kKvThreads) {
        char v[kKvGroup];
#pragma unroll
        for (int j = 0; j < kKvGroup; ++j)
          if (j < kn) v[j] = sbase[(size_t)rr[j] * a.row_bytes + c];
#pragma unroll
        for (int j = 0; j < kKvGroup; ++j)
          if (j < kn) dbase[(size_t)(k0 + j) * a.row_bytes + c] = v[j];
      }
    }
    // in place, the next group reads slots >= k0 + kKvGroup, which this
    // group never writes; other threads touch other columns.
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
  if (2L * L > 65535) return set_error(SV_ERR_UNSUPPORTED, "L > 32767");
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
  kv_compact_kernel<<<dim3(B, 2 * L), kKvThreads, 0, st>>>(a);
  return check_launch("kv_compact");
}
