// tree_attn.cu -- tree-masked verifier attention on the 5th-generation tensor
// cores (sm_103a): TMA tile loads, tcgen05.mma with accumulators in tensor
// memory, online softmax in registers.
//
// [Blog] "投机解码发展", section 3: the verifier scores the flattened draft tree
// in one forward pass in which each node attends to the committed context and
// to itself and its ancestors only (never to a sibling or another branch);
// [Lesson] "Decodificação Especulativa e EAGLE-3", "Reversão de KV cache": the
// tree pass runs a non-causal mask that follows the tree.  This is the
// attention of that pass for one layer, with grouped-query heads.
//
// Work item: 128 query rows of one (sequence, KV head) -- the G = Hq / Hkv
// query heads sharing that KV head times 128 / G consecutive tree nodes, row
// r = node_local * G + head_local.  The kernel is persistent: one CTA per SM
// walks items c, c + gridDim.x, ... and, per item, the sequence's keys
// (context, then the T tree rows) in tiles of 128:
//   warp 0      TMA producer: each item's query tile into shared memory, K
//               and V tiles into three-stage rings (128B-swizzled boxes of 64
//               columns), each load issued as soon as its stage is free;
//   warp 1      MMA issuer (converged warp, elect.sync): S_j = Q K_j^T into
//               the S buffer of tensor memory as soon as the softmax warps
//               have read S_{j-1} out of it, O += P_j V_j once P_j is ready;
//               both with the A operand (Q, P) in tensor memory;
//   warps 2..9  softmax: query tile from shared memory to tensor memory;
//               per tile S_j to registers (16-lane shapes: a row over a quad
//               of threads), ancestor mask, running max with a lazy rescale
//               of O (only when the max grows by more than 2^8), P_j =
//               exp2(...) as bf16 into one of two P buffers in tensor memory;
//               at the end of the item O / l to global memory.
// Every wait on an mbarrier is bounded by a wall-clock limit; a wait that runs
// out sets SV_ROW_TIMEOUT for the sequences left and the CTA drains and exits.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"

namespace sv {
namespace {

constexpr int kHd = 128;               // head dimension
constexpr int kRows = 128;             // query rows per CTA = tensor-memory lanes
constexpr int kKeys = 128;             // keys per tile
constexpr int kAttnThreads = 320;      // 10 warps
constexpr uint32_t kTile = 32768;      // one 128 x 128 bf16 operand tile
constexpr uint32_t kHalfTile = 16384;  // one 128-byte-wide swizzled box of it
constexpr int kStages = 3;             // K and V ring depth
constexpr uint32_t kOffK = 0;                        // kStages K tiles
constexpr uint32_t kOffV = kOffK + kStages * kTile;  // kStages V tiles
constexpr uint32_t kOffQ = kOffV + kStages * kTile;  // the next item's query tile
constexpr uint32_t kOffBar = kOffQ + kTile;
constexpr uint32_t kOffMisc = kOffBar + 32 * 8;
constexpr size_t kAttnSmem = kOffMisc + 64 + 1024;  // + alignment slack
// barrier indices: query in tensor memory (kBarQ), K/V landed and stage free
// (per stage), S ready / read out, P ready and PV retired (per parity), query
// tile landed in / read out of shared memory (kBarQS / kBarQF)
constexpr int kBarQ = 0, kBarK = 1, kBarV = kBarK + kStages, kBarKF = kBarV + kStages,
              kBarVF = kBarKF + kStages, kBarS = kBarVF + kStages, kBarSF = kBarS + 2,
              kBarP = kBarSF + 2, kBarPV = kBarP + 2, kBarQS = kBarPV + 2, kBarQF = kBarQS + 1;
// tensor-memory columns: S at 0, O at 128, Q (bf16 pairs) at 256, two P
// buffers (bf16 pairs) at 320 and 384
constexpr uint32_t kColS = 0, kColO = 128, kColQ = 256, kColP = 320;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;   // lazy rescale threshold (log2 units)
constexpr unsigned long long kWaitNs = 2000000000ull;  // 2 s: default wait limit, and every drain's

struct AttnArgs {
  const uint16_t *q;
  const int32_t *base;
  const uint64_t *mask;
  uint16_t *out;
  float *lse;
  uint32_t *status;
  int B, T, Hq, Hkv, S, G, W, npt;  // npt = tree nodes per item = 128 / G
  int mtiles, n_items;              // query tiles per (sequence, KV head); items
  float scale_log2;                 // softmax scale * log2(e)
  unsigned long long wait_ns;       // limit of each wait of the pipeline (drains: kWaitNs)
};

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase of `parity` to complete.  Gives up after
// `limit` ns or as soon as another role of the CTA has given up (*abort != 0).
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile int *abort,
                                            unsigned long long limit) {
  const unsigned long long t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try(bar, parity)) return true;
    if ((it & 63) == 0) {
      if (*abort) return false;
      if (global_ns() - t0 > limit) {
        *abort = 1;
        return false;
      }
    }
  }
}

// Short limits (below 1 ms) poll with the non-blocking test and read the
// clock every time: a blocking try_wait may itself suspend the thread longer
// than such a limit.
constexpr unsigned long long kShortWaitNs = 1000000ull;
__device__ __noinline__ bool mbar_wait_short(uint32_t bar, uint32_t parity, volatile int *abort,
                                             unsigned long long limit);
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                          unsigned long long limit = kWaitNs) {
  if (limit < kShortWaitNs) return mbar_wait_short(bar, parity, abort, limit);
  return mbar_try(bar, parity) || mbar_wait_slow(bar, parity, abort, limit);
}

// Non-blocking test of the phase of `parity`.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __noinline__ bool mbar_wait_short(uint32_t bar, uint32_t parity, volatile int *abort,
                                             unsigned long long limit) {
  const unsigned long long t0 = global_ns();
  for (;;) {
    if (mbar_test(bar, parity)) return true;
    if (*abort) return false;
    if (global_ns() - t0 > limit) {
      *abort = 1;
      return false;
    }
  }
}

// One lane of the (converged) warp: true there, false elsewhere.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(pred));
  return pred != 0;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// 4-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load4(uint32_t dst, const CUtensorMap *map, int x, int y,
                                          int z, int w, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
      : "memory");
}

// Shared-memory matrix descriptor of tcgen05: start, leading and stride byte
// offsets (16-byte units), the fixed 0b001 at bits 46-48, swizzle mode at
// bits 61-63 (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator (bits 4-5 = 1), bf16 A
// and B (bits 7-9, 10-12 = 1), N >> 3 at bit 17, M >> 4 at bit 24; bit 16 =
// B is MN-major (the V tile: keys x head dim, head dim contiguous).
constexpr uint32_t kIdescS = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kKeys >> 3) << 17) |
                             ((uint32_t)(kRows >> 4) << 24);
constexpr uint32_t kIdescO = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) |
                             ((uint32_t)(kHd >> 3) << 17) | ((uint32_t)(kRows >> 4) << 24);

// D (+)= A * B with the A operand in tensor memory (rows on lanes, K as bf16
// pairs, the even element in the low half: one K16 slice = 8 columns) and B
// in shared memory.
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                       uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive 32-bit columns of this thread's tensor-memory lane (32x32b).
__device__ __forceinline__ void tm_st32(uint32_t taddr, const float *v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

// 16x256b shape, 8 repetitions (64 columns): thread t gets rows t/4 and
// t/4 + 8 of the 16-lane window, columns 8c + 2 (t % 4) + {0, 1}:
// v[4c + 0, 1] = first row, v[4c + 2, 3] = second row.
__device__ __forceinline__ void tm_ld16x256_x8(uint32_t taddr, float *v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

__device__ __forceinline__ void tm_st16x256_x8(uint32_t taddr, const float *v) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x256b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

// 16x128b shape, 16 repetitions (64 columns): thread t writes column
// 4c + t % 4 of rows t/4 (v[2c]) and t/4 + 8 (v[2c + 1]).
__device__ __forceinline__ void tm_st16x128_x16(uint32_t taddr, const uint32_t *v) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x128b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
      "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
      "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

__device__ __forceinline__ void tm_st32u(uint32_t taddr, const uint32_t *v) {
  tm_st32(taddr, reinterpret_cast<const float *>(v));
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ex2 of a packed pair on the MUFU (ex2.approx.ftz: -inf gives +0).
__device__ __forceinline__ unsigned long long ex2_2(unsigned long long x) {
  float a, b;
  f2_unpack(x, a, b);
  return f2_pack(ex2(a), ex2(b));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Word w of a node's ancestor mask: words 0 and 1 prefetched (m01), later
// ones from memory, words past W zero.
__device__ __forceinline__ uint64_t mask_word(const uint64_t *mrow, int W, uint64_t m0,
                                              uint64_t m1, int w) {
  return w == 0 ? m0 : (w == 1 ? m1 : (w < W ? __ldg(mrow + w) : 0ull));
}

// Bits [pos, pos + 32) of a node's ancestor mask (pos >= 0).
__device__ __forceinline__ uint32_t mask_bits32(const uint64_t *mrow, int W, uint64_t m0,
                                                uint64_t m1, int pos) {
  const int w = pos >> 6, sh = pos & 63;
  const uint64_t lo = mask_word(mrow, W, m0, m1, w);
  const uint64_t hi = sh ? mask_word(mrow, W, m0, m1, w + 1) : 0ull;
  return (uint32_t)(sh ? (lo >> sh) | (hi << (64 - sh)) : lo);
}

// Visibility of keys base + rel + i, i = 0..31: context keys (rel + i < 0)
// are visible, tree key m = rel + i < T iff bit m of the node's mask, keys at
// or past base + T never.  mrow == nullptr (a padding row): context only.
__device__ __forceinline__ uint32_t visible32(const uint64_t *mrow, int W, uint64_t m0,
                                              uint64_t m1, int T, int rel) {
  const uint32_t pre = rel >= 0 ? 0u : (rel <= -32 ? 0xFFFFFFFFu : ((1u << (-rel)) - 1u));
  if (rel <= -32 || rel >= T || mrow == nullptr) return pre;
  uint32_t tree;
  int nvalid;
  if (rel >= 0) {
    tree = mask_bits32(mrow, W, m0, m1, rel);
    nvalid = T - rel;
  } else {
    tree = mask_bits32(mrow, W, m0, m1, 0) << (-rel);
    nvalid = T - rel;
  }
  if (nvalid < 32) tree &= (1u << nvalid) - 1u;
  return pre | tree;
}

// One work item: 128 query rows (query tile mt) of one (sequence, KV head).
struct Item {
  int mt, kvh, b, bs, n_keys, n_tiles;
  bool bad;
};

__device__ __forceinline__ Item decode_item(const AttnArgs &a, int it) {
  Item x;
  x.mt = it % a.mtiles;
  const int rest = it / a.mtiles;
  x.kvh = rest % a.Hkv;
  x.b = rest / a.Hkv;
  x.bs = a.base[x.b];
  x.bad = x.bs < 0 || (long long)x.bs + a.T > a.S;
  x.n_keys = x.bs + a.T;
  x.n_tiles = x.bad ? 0 : (x.n_keys + kKeys - 1) / kKeys;
  return x;
}

// Persistent: CTA c takes items c, c + gridDim.x, ...  Every role walks the
// same item sequence; ring stages, S buffers and barrier phases follow
// CTA-wide tile counters, so the producer runs ahead into the next item while
// the current one drains and the per-CTA setup happens once.
__global__ void __launch_bounds__(kAttnThreads, 1)
    tree_attn_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tkv,
                     AttnArgs a) {
  grid_dep_sync();
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;

  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kOffBar);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + kOffMisc);
  volatile int *abort = reinterpret_cast<volatile int *>(sm + kOffMisc + 4);
  volatile int *abort_item = reinterpret_cast<volatile int *>(sm + kOffMisc + 8);
  const uint32_t bar0 = smem_addr(bars);
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  const uint32_t sK = smem_addr(sm + kOffK), sV = smem_addr(sm + kOffV), sQ = smem_addr(sm + kOffQ);

  if (threadIdx.x == 0) {
    mbar_init(bar(kBarQ), 8);
    mbar_init(bar(kBarQS), 1);
    mbar_init(bar(kBarQF), 8);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarK + s), 1);
      mbar_init(bar(kBarV + s), 1);
      mbar_init(bar(kBarKF + s), 1);
      mbar_init(bar(kBarVF + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kBarS + s), 1);
      mbar_init(bar(kBarSF + s), 8);
      mbar_init(bar(kBarP + s), 8);
      mbar_init(bar(kBarPV + s), 1);
    }
    *abort = 0;
    *abort_item = a.n_items;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      // K tile g (CTA-wide count) goes to stage g % kStages once S_{g-kStages}
      // has read that stage (kBarKF), V tile g once PV_{g-kStages} has
      // (kBarVF).  Each condition is a phase of a barrier whose earlier
      // phases this thread has already seen and whose next phase needs the
      // tile about to be loaded, so the parity test cannot alias.  The two
      // rings are polled; V never runs ahead of K.
      int gk = 0, gv = 0, nq = 0;
      unsigned long long t_last = global_ns();
      bool stop = false;
      for (int it = blockIdx.x; it < a.n_items && !stop; it += gridDim.x) {
        const Item x = decode_item(a, it);
        if (x.n_tiles > 0) {
          // the item's query tile, once the softmax warps have read the last
          // one (the previous phase of kBarQF, already seen by this thread)
          if (nq > 0 && !mbar_wait(bar(kBarQF), (nq - 1) & 1, abort, a.wait_ns)) {
            atomicMin(const_cast<int *>(abort_item), it);
            break;
          }
          mbar_expect_tx(bar(kBarQS), kTile);
          tma_load4(sQ, &tq, 0, x.kvh * a.G, x.mt * a.npt, x.b, bar(kBarQS));
          tma_load4(sQ + kHalfTile, &tq, 64, x.kvh * a.G, x.mt * a.npt, x.b, bar(kBarQS));
          ++nq;
          t_last = global_ns();
        }
        int kn = 0, vn = 0;
        while (kn < x.n_tiles || vn < x.n_tiles) {
          bool did = false;
          if (kn < x.n_tiles &&
              (gk < kStages ||
               mbar_test(bar(kBarKF + gk % kStages), ((gk - kStages) / kStages) & 1))) {
            const int st = gk % kStages;
            mbar_expect_tx(bar(kBarK + st), kTile);
            tma_load4(sK + st * kTile, &tkv, 0, x.kvh, kn * kKeys, x.b, bar(kBarK + st));
            tma_load4(sK + st * kTile + kHalfTile, &tkv, 64, x.kvh, kn * kKeys, x.b,
                      bar(kBarK + st));
            ++kn;
            ++gk;
            did = true;
          }
          if (vn < kn &&
              (gv < kStages ||
               mbar_test(bar(kBarVF + gv % kStages), ((gv - kStages) / kStages) & 1))) {
            const int st = gv % kStages;
            mbar_expect_tx(bar(kBarV + st), kTile);
            tma_load4(sV + st * kTile, &tkv, 0, x.kvh, vn * kKeys, a.B + x.b, bar(kBarV + st));
            tma_load4(sV + st * kTile + kHalfTile, &tkv, 64, x.kvh, vn * kKeys, a.B + x.b,
                      bar(kBarV + st));
            ++vn;
            ++gv;
            did = true;
          }
          if (did) {
            t_last = global_ns();
            continue;
          }
          if (*abort || global_ns() - t_last > a.wait_ns) {
            *abort = 1;
            atomicMin(const_cast<int *>(abort_item), it);
            stop = true;
            break;
          }
          __nanosleep(64);
        }
      }
      // every copy issued has landed before the CTA exits (immediate unless a
      // consumer gave up early): the newest phase of each stage barrier
      volatile int no_abort = 0;
      for (int g = gk > kStages ? gk - kStages : 0; g < gk; ++g)
        mbar_wait(bar(kBarK + g % kStages), (g / kStages) & 1, &no_abort);
      for (int g = gv > kStages ? gv - kStages : 0; g < gv; ++g)
        mbar_wait(bar(kBarV + g % kStages), (g / kStages) & 1, &no_abort);
      if (nq > 0) mbar_wait(bar(kBarQS), (nq - 1) & 1, &no_abort);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    // Both products take their A operand from tensor memory (Q, then P) and
    // only K or V from shared memory.  One S buffer: S_{i+1} is issued as soon
    // as the softmax warps have read S_i out of it (early in their tile i),
    // so it is ready when they finish tile i; PV_i follows once P_i is ready,
    // reading P buffer i % 2 (the softmax writes P_{i+1} into the other one
    // meanwhile).  The whole warp runs the loop
    // converged and elect.sync picks the issuing lane: a lone diverged lane
    // issues far more slowly while the softmax warps keep the sub-partition
    // busy.  Descriptors are a stage base plus a constant step (the start
    // address is the low 14 bits).  gS / gP count S and PV tiles CTA-wide.
    int gS = 0, gP = 0, nq = 0;
    bool ok = true;
    const uint64_t dK0 = sdesc(sK, 16, 1024), dV0 = sdesc(sV, kHalfTile, 1024);
    constexpr uint64_t kStageStep = kTile >> 4;
    auto issue_s = [&](int g) {
      const uint64_t dk = dK0 + (g % kStages) * kStageStep;
#pragma unroll
      for (int ks = 0; ks < kHd / 16; ++ks)
        mma_ts(tmem + kColS, tmem + kColQ + ks * 8,
               dk + (uint64_t)(((ks >> 2) * kHalfTile + (ks & 3) * 32) >> 4), kIdescS, ks > 0);
      mma_commit(bar(kBarS));
      mma_commit(bar(kBarKF + g % kStages));
    };
    auto wait_s_ready = [&](int g) -> bool {  // K_g landed, S_{g-1} read out
      return (g < 1 || mbar_wait(bar(kBarSF), (g - 1) & 1, abort, a.wait_ns)) &&
             mbar_wait(bar(kBarK + g % kStages), (g / kStages) & 1, abort, a.wait_ns);
    };
    int it = blockIdx.x;
    for (; ok && it < a.n_items; it += gridDim.x) {
      const Item x = decode_item(a, it);
      if (x.n_tiles == 0) continue;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarQ), nq & 1, abort, a.wait_ns));  // this item's Q
      ++nq;
      if (!ok) break;
      tc_fence_after();
      ok = __all_sync(0xffffffffu, wait_s_ready(gS));
      if (!ok) break;
      tc_fence_after();
      if (elect_one()) issue_s(gS);
      __syncwarp();
      ++gS;
      for (int i = 0; ok && i < x.n_tiles; ++i) {
        if (i + 1 < x.n_tiles) {
          ok = __all_sync(0xffffffffu, wait_s_ready(gS));
          if (!ok) break;
          tc_fence_after();
          if (elect_one()) issue_s(gS);
          __syncwarp();
          ++gS;
        }
        ok = __all_sync(0xffffffffu,
                        mbar_wait(bar(kBarP + (gP & 1)), (gP >> 1) & 1, abort, a.wait_ns) &&
                            mbar_wait(bar(kBarV + gP % kStages), (gP / kStages) & 1, abort, a.wait_ns));
        if (!ok) break;
        // the last tile's PV runs only the K16 steps holding keys below
        // n_keys; value rows past the last key inside the last step may hold
        // anything (NaN included) and are zeroed, so that P = 0 there adds 0
        const int sv = gP % kStages;
        const int rem = x.n_keys - i * kKeys;
        const int pv_steps = (i == x.n_tiles - 1) ? (rem + 15) >> 4 : 8;
        if (i == x.n_tiles - 1 && (rem & 15)) {
          uint8_t *vt = sm + kOffV + sv * kTile;
          const int nrow = 16 * pv_steps - rem;  // < 16 rows, 16 chunks each
          for (int c = lane; c < nrow * 16; c += 32) {
            const int row = rem + (c >> 4), ch = c & 15;
            *reinterpret_cast<uint4 *>(vt + (ch >> 3) * kHalfTile + row * 128 + (ch & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
        }
        tc_fence_after();
        if (elect_one()) {
          const uint64_t dv = dV0 + sv * kStageStep;
          const uint32_t pa = tmem + kColP + (gP & 1) * 64;
          for (int ks = 0; ks < pv_steps; ++ks)
            mma_ts(tmem + kColO, pa + ks * 8, dv + (uint64_t)(ks * 128), kIdescO,
                   (i > 0 || ks > 0) ? 1u : 0u);
          mma_commit(bar(kBarPV + (gP & 1)));
          mma_commit(bar(kBarVF + sv));
        }
        __syncwarp();
        ++gP;
      }
    }
    if (!ok) {
      if (lane == 0) atomicMin(const_cast<int *>(abort_item), it);
      // retire the MMAs in flight before tensor memory is released: the last
      // S and the last PV commit are the newest phases of their barriers
      volatile int no_abort = 0;
      if (gS > 0) mbar_wait(bar(kBarS), (gS - 1) & 1, &no_abort);
      if (gP > 0) mbar_wait(bar(kBarPV + ((gP - 1) & 1)), ((gP - 1) >> 1) & 1, &no_abort);
    }
  } else {
    // ---------------------------------------------------------------- softmax
    // Warp w reads tensor-memory lanes of quarter w % 4; the pair (w, w + 4)
    // splits them into two 16-lane halves.  With the 16x256b / 16x128b
    // shapes thread t holds rows h16 + t/4 and h16 + t/4 + 8 of its half and,
    // in every 8-column chunk, columns 2 (t % 4) and 2 (t % 4) + 1: a row is
    // spread over the four threads of a quad, so row maxima and sums are two
    // shuffles and no warp waits for another.  The P store (16x128b) writes
    // bf16 pair column 4 c + t % 4, exactly the two keys the thread holds.
    // gT counts tiles CTA-wide (S buffers, P and PV barriers follow it).
    const int half = (warp - 2) >> 2;
    const int q4 = lane & 3;
    const uint32_t lane16 = (uint32_t)(quarter * 32 + half * 16) << 16;
    const int rowA = quarter * 32 + half * 16 + (lane >> 2);  // and rowA + 8
    const float NEG_INF = -INFINITY;
    int gT = 0, it = blockIdx.x, nq = 0;
    bool ok = true;
    for (; ok && it < a.n_items; it += gridDim.x) {
      const Item x = decode_item(a, it);
      const int node0 = x.mt * a.npt;
      // the 32x32b row of this thread (query copy, rows of a bad sequence)
      const int r32 = quarter * 32 + lane;
      const int node32 = node0 + r32 / a.G;
      const bool ok32 = node32 < a.T;
      const size_t orow32 = ((size_t)x.b * a.T + node32) * a.Hq + x.kvh * a.G + r32 % a.G;
      if (x.bad) {
        // base out of range: NaN rows, nothing read
        if (half == 0 && ok32) {
          const uint4 nan4 = make_uint4(0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u);
          uint4 *o = reinterpret_cast<uint4 *>(a.out + orow32 * kHd);
          for (int c = 0; c < kHd / 8; ++c) o[c] = nan4;
          if (a.lse) a.lse[orow32] = __int_as_float(0x7FC00000);
        }
        if (threadIdx.x == 64 && a.status && x.mt == 0 && x.kvh == 0)
          atomicOr(a.status + x.b, SV_ROW_BAD_BASE);
        continue;
      }
      {
        // this warp's query columns (head-dim half) for all 32 lanes of the
        // quarter, from the tile the producer staged in shared memory (128-byte
        // swizzled: row r32, chunk c at (c ^ (r32 & 7)) * 16; rows past T are
        // the copy's zero fill), into tensor memory as bf16 pairs (32x32b:
        // lane = row); the item's S products wait for all eight warps
        ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarQS), nq & 1, abort, a.wait_ns));
        ++nq;
        if (!ok) break;
        uint32_t qv[32];
        const uint8_t *qrow = sm + kOffQ + half * kHalfTile + r32 * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 w = *reinterpret_cast<const uint4 *>(qrow + ((c ^ (r32 & 7)) << 4));
          qv[4 * c] = w.x;
          qv[4 * c + 1] = w.y;
          qv[4 * c + 2] = w.z;
          qv[4 * c + 3] = w.w;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarQF));  // this warp is done with the tile
        tm_st32u(tmem + ((uint32_t)(quarter * 32) << 16) + kColQ + 32 * half, qv);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarQ));
      }
      // the two rows of this thread
      int rnode[2];
      size_t rrow[2];
      bool rok[2];
      const uint64_t *rmask[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int rr = rowA + 8 * e;
        rnode[e] = node0 + rr / a.G;
        rok[e] = rnode[e] < a.T;
        rrow[e] = ((size_t)x.b * a.T + rnode[e]) * a.Hq + x.kvh * a.G + rr % a.G;
        rmask[e] = rok[e] ? a.mask + ((size_t)x.b * a.T + rnode[e]) * a.W : nullptr;
      }
      // the first two mask words of both rows, fetched now for the tiles that
      // reach the tree (the last one or two of the item)
      uint64_t mw[2][2];
#pragma unroll
      for (int e = 0; e < 2; ++e)
#pragma unroll
        for (int w = 0; w < 2; ++w) mw[e][w] = (rmask[e] && w < a.W) ? __ldg(rmask[e] + w) : 0ull;
      float m_ref[2] = {NEG_INF, NEG_INF};  // reference max (log2 domain, scaled)
      float l[2] = {0.0f, 0.0f};            // partial sums over this thread's columns
      for (int j = 0; j < x.n_tiles; ++j) {
        const int g = gT + j, pb = g & 1;
        ok = mbar_wait(bar(kBarS), g & 1, abort, a.wait_ns);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        // s[4c + 0, 1]: row A, keys 8c + 2 q4 + {0, 1}; s[4c + 2, 3]: row B
        float s[64];
        tm_ld16x256_x8(tmem + lane16 + kColS, s);
        tm_ld16x256_x8(tmem + lane16 + kColS + 64, s + 32);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarSF));  // the S buffer is free for S_{g+1}
        const int key0 = j * kKeys;
        if (key0 + kKeys > x.bs) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
#pragma unroll
            for (int gg = 0; gg < 4; ++gg) {
              // keys key0 + 32 gg .. +31: chunks c = 4 gg .. 4 gg + 3
              const uint32_t vis = visible32(rmask[e], a.W, mw[e][0], mw[e][1], a.T, key0 + 32 * gg - x.bs);
#pragma unroll
              for (int cc = 0; cc < 4; ++cc) {
                const int c = 4 * gg + cc, bit = 8 * cc + 2 * q4;
                if (!((vis >> bit) & 1u)) s[4 * c + 2 * e] = NEG_INF;
                if (!((vis >> (bit + 1)) & 1u)) s[4 * c + 2 * e + 1] = NEG_INF;
              }
            }
          }
        }
        float factor[2], mneg[2];
        bool any_grow = false;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          // four independent chains over the 32 values of row e (chunks 0..15)
          float pm[4] = {s[2 * e], s[2 * e + 1], s[4 + 2 * e], s[4 + 2 * e + 1]};
#pragma unroll
          for (int c = 2; c < 16; c += 2) {
            pm[0] = fmaxf(pm[0], s[4 * c + 2 * e]);
            pm[1] = fmaxf(pm[1], s[4 * c + 2 * e + 1]);
            pm[2] = fmaxf(pm[2], s[4 * c + 4 + 2 * e]);
            pm[3] = fmaxf(pm[3], s[4 * c + 4 + 2 * e + 1]);
          }
          float mx = fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3]));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
          mx *= a.scale_log2;  // scale > 0: max commutes with it
          const bool grow = mx > m_ref[e] + kRescaleLog2;
          const float m_new = grow ? mx : m_ref[e];
          factor[e] = (grow && m_ref[e] != NEG_INF) ? ex2(m_ref[e] - m_new) : 1.0f;
          any_grow |= factor[e] != 1.0f;
          l[e] *= factor[e];
          m_ref[e] = m_new;
          mneg[e] = m_new == NEG_INF ? 0.0f : -m_new;
        }
        // p = 2^(scale*log2e*s - m): scaling and sums on packed fp32 pairs,
        // the exponentials on the MUFU (moving a share of them to a polynomial
        // on the FMA pipe measured slower: the warps are bound by issue slots)
        uint32_t pk[32];
        unsigned long long la2 = 0ull, lb2 = 0ull;
        const unsigned long long sc2 = f2_splat(a.scale_log2);
        const unsigned long long ma2 = f2_splat(mneg[0]), mb2 = f2_splat(mneg[1]);
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const unsigned long long xa = f2_fma(f2_pack(s[4 * c], s[4 * c + 1]), sc2, ma2);
          const unsigned long long xb = f2_fma(f2_pack(s[4 * c + 2], s[4 * c + 3]), sc2, mb2);
          const unsigned long long pa = ex2_2(xa);
          const unsigned long long pb = ex2_2(xb);
          la2 = f2_add(la2, pa);
          lb2 = f2_add(lb2, pb);
          float p0, p1, p2, p3;
          f2_unpack(pa, p0, p1);
          f2_unpack(pb, p2, p3);
          pk[2 * c] = pack_bf16(p0, p1);      // row A, pair column 4c + q4
          pk[2 * c + 1] = pack_bf16(p2, p3);  // row B
        }
        {
          float u0, u1, v0, v1;
          f2_unpack(la2, u0, u1);
          f2_unpack(lb2, v0, v1);
          l[0] += u0 + u1;
          l[1] += v0 + v1;
        }
        if (g >= 2) {
          // PV_{g-2} has retired: P buffer pb is free (this warp has seen
          // every earlier phase of its barrier)
          const int i = g - 2;
          ok = mbar_wait(bar(kBarPV + (i & 1)), (i >> 1) & 1, abort, a.wait_ns);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
        }
        if (__any_sync(0xffffffffu, any_grow)) {
          // the max grew: once O covers tiles < j (PV_{g-1} retired), bring
          // these rows of it to the new reference
          if (j >= 1) {
            const int i = g - 1;
            ok = mbar_wait(bar(kBarPV + (i & 1)), (i >> 1) & 1, abort, a.wait_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
          }
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < kHd; c += 64) {
            float o[32];
            tm_ld16x256_x8(tmem + lane16 + kColO + c, o);
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] *= factor[(k >> 1) & 1];
            tm_st16x256_x8(tmem + lane16 + kColO + c, o);
          }
        }
        tm_st16x128_x16(tmem + lane16 + kColP + pb * 64, pk);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarP + pb));
      }
      if (ok) {
        const int i = gT + x.n_tiles - 1;
        ok = mbar_wait(bar(kBarPV + (i & 1)), (i >> 1) & 1, abort, a.wait_ns);
        ok = __all_sync(0xffffffffu, ok);
      }
      if (ok) {
        tc_fence_after();
        float inv[2], lt[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float v = l[e];
          v += __shfl_xor_sync(0xffffffffu, v, 1);
          v += __shfl_xor_sync(0xffffffffu, v, 2);
          lt[e] = v;
          inv[e] = v > 0.0f ? 1.0f / v : 0.0f;
        }
#pragma unroll
        for (int c = 0; c < kHd; c += 64) {
          float o[32];
          tm_ld16x256_x8(tmem + lane16 + kColO + c, o);
          asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
          // o[4k + 0, 1]: row A, columns c + 8k + 2 q4 + {0, 1}; o[4k + 2, 3]: row B
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            if (!rok[e]) continue;
            uint32_t *orow32 = reinterpret_cast<uint32_t *>(a.out + rrow[e] * kHd + c + 2 * q4);
#pragma unroll
            for (int k = 0; k < 8; ++k)
              orow32[4 * k] = pack_bf16(o[4 * k + 2 * e] * inv[e], o[4 * k + 2 * e + 1] * inv[e]);
          }
        }
        if (q4 == 0 && a.lse) {
#pragma unroll
          for (int e = 0; e < 2; ++e)
            if (rok[e])
              a.lse[rrow[e]] =
                  lt[e] > 0.0f ? (m_ref[e] + __log2f(lt[e])) * 0.69314718055994531f : NEG_INF;
        }
      }
      gT += x.n_tiles;
    }
    if (!ok) atomicMin(const_cast<int *>(abort_item), it);
  }
  tc_fence_before();
  __syncthreads();
  if (*abort && threadIdx.x == 0 && a.status)
    for (int it = *abort_item; it < a.n_items; it += gridDim.x)
      if (it % (int)gridDim.x == (int)blockIdx.x) atomicOr(a.status + decode_item(a, it).b, SV_ROW_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// cuTensorMapEncodeTiled, fetched from the driver at run time (the library
// does not link libcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)p;
  }
  return fn;
}

// 4-D bf16 map with 128-byte swizzle; dims innermost first, strides in bytes
// for dims 1..3, box {64, b1, b2, 1}.
sv_status encode4(CUtensorMap *m, const void *base, const cuuint64_t dims[4],
                  const cuuint64_t strides[3], cuuint32_t b1, cuuint32_t b2, const char *what) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return set_error(SV_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  const cuuint32_t box[4] = {64, b1, b2, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(SV_ERR_CUDA, "tensor map for %s: error %d", what, (int)r);
  return SV_OK;
}

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" sv_status sv_tree_attention_ex(const void *q, const void *kv, const int32_t *base,
                                          const uint64_t *mask, int B, int T, int Hq, int Hkv,
                                          int D, int S, float scale, void *out, float *out_lse,
                                          uint32_t *out_status, uint64_t wait_ns, void *stream) {
  if (B < 0 || T < 1 || Hq < 1 || Hkv < 1 || S < 1)
    return set_error(SV_ERR_INVALID_ARG, "need B >= 0, T >= 1, Hq >= 1, Hkv >= 1, S >= 1");
  if (T > SV_MAX_TREE_NODES) return set_error(SV_ERR_UNSUPPORTED, "T > %d", SV_MAX_TREE_NODES);
  if (D != kHd) return set_error(SV_ERR_UNSUPPORTED, "head dimension %d (only 128)", D);
  if (Hq % Hkv) return set_error(SV_ERR_INVALID_ARG, "Hq must be a multiple of Hkv");
  const int G = Hq / Hkv;
  if (G > kRows || (kRows % G)) return set_error(SV_ERR_UNSUPPORTED, "Hq / Hkv must divide 128");
  if (!(scale > 0.0f) || !isfinite(scale)) return set_error(SV_ERR_INVALID_ARG, "scale must be > 0");
  if (Hkv > 65535 || B > 65535) return set_error(SV_ERR_UNSUPPORTED, "Hkv or B above 65535");
  if (B == 0) return SV_OK;
  if (!q || !kv || !base || !mask || !out) return set_error(SV_ERR_INVALID_ARG, "null pointer");
  if (!is_device_memory(q) || !is_device_memory(kv))
    return set_error(SV_ERR_INVALID_ARG, "q and kv must be device memory (tensor-map loads)");
  if ((uintptr_t)q % 16 || (uintptr_t)kv % 16 || (uintptr_t)out % 16 || (uintptr_t)mask % 8)
    return set_error(SV_ERR_INVALID_ARG, "q, kv, out need 16-byte and mask 8-byte alignment");
  sv_status s;
  if ((s = map_arg(base, "base")) != SV_OK || (s = map_arg(mask, "mask")) != SV_OK ||
      (s = map_arg(out, "out")) != SV_OK || (s = map_arg(out_lse, "out_lse")) != SV_OK ||
      (s = map_arg(out_status, "out_status")) != SV_OK)
    return s;
  const int npt = kRows / G;
  CUtensorMap tq, tkv;
  {
    const cuuint64_t dims[4] = {(cuuint64_t)kHd, (cuuint64_t)Hq, (cuuint64_t)T, (cuuint64_t)B};
    const cuuint64_t str[3] = {(cuuint64_t)kHd * 2, (cuuint64_t)Hq * kHd * 2,
                               (cuuint64_t)T * Hq * kHd * 2};
    if ((s = encode4(&tq, q, dims, str, (cuuint32_t)G, (cuuint32_t)(kRows / G), "q")) != SV_OK)
      return s;
  }
  {
    const cuuint64_t dims[4] = {(cuuint64_t)kHd, (cuuint64_t)Hkv, (cuuint64_t)S,
                                (cuuint64_t)2 * B};
    const cuuint64_t str[3] = {(cuuint64_t)kHd * 2, (cuuint64_t)Hkv * kHd * 2,
                               (cuuint64_t)S * Hkv * kHd * 2};
    if ((s = encode4(&tkv, kv, dims, str, 1, (cuuint32_t)kKeys, "kv")) != SV_OK) return s;
  }
  static int smem_set_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (smem_set_dev != dev) {
    const cudaError_t e = cudaFuncSetAttribute(tree_attn_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)kAttnSmem);
    if (e != cudaSuccess) return check_launch("tree_attention", e);
    smem_set_dev = dev;
  }
  AttnArgs a;
  a.q = (const uint16_t *)q;
  a.base = base;
  a.mask = mask;
  a.out = (uint16_t *)out;
  a.lse = out_lse;
  a.status = out_status;
  a.B = B;
  a.T = T;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.S = S;
  a.G = G;
  a.W = (T + 63) / 64;
  a.npt = npt;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.wait_ns = wait_ns ? wait_ns : kWaitNs;
  const int mtiles = (T + npt - 1) / npt;
  const long long n_items = (long long)mtiles * Hkv * B;
  if (n_items > 0x7fffffffLL) return set_error(SV_ERR_UNSUPPORTED, "too many query tiles");
  a.mtiles = mtiles;
  a.n_items = (int)n_items;
  const int grid = (int)(n_items < num_sms() ? n_items : num_sms());
  cudaStream_t st = (cudaStream_t)stream;
  LaunchScope ls("tree_attention", st);
  return check_launch("tree_attention",
                      launch_pdl(tree_attn_kernel, dim3(grid), dim3(kAttnThreads),
                                 kAttnSmem, st, tq, tkv, a));
}

extern "C" sv_status sv_tree_attention(const void *q, const void *kv, const int32_t *base,
                                       const uint64_t *mask, int B, int T, int Hq, int Hkv, int D,
                                       int S, float scale, void *out, float *out_lse,
                                       uint32_t *out_status, void *stream) {
  return sv_tree_attention_ex(q, kv, base, mask, B, T, Hq, Hkv, D, S, scale, out, out_lse,
                              out_status, 0, stream);
}
