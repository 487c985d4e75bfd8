// common.cuh -- device helpers and the host runtime hooks shared by the
// library's translation units (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sv.h"

namespace sv {

// ----------------------------------------------------------------- host side
// Error reporting (thread-local message) and launch bookkeeping.
sv_status set_error(sv_status st, const char *fmt, ...);
sv_status check_launch(const char *what);
sv_status check_launch(const char *what, cudaError_t launched);
int num_sms();

// Pointer arguments: device or managed memory of the current device is used
// as is; page-locked host memory (cudaHostAlloc, cudaHostRegister) through its
// device mapping, so the kernels read or write it in place over the host link;
// pageable host memory and other devices' memory are refused with
// SV_ERR_INVALID_ARG (a kernel would fault on them).  NULL stays NULL.
sv_status map_ptr(const void **p, const char *what);
// 1 when p is memory of the current device (not host memory mapped into it)
int is_device_memory(const void *p);
template <typename T>
sv_status map_arg(T *&p, const char *what) {
  const void *q = p;
  const sv_status s = map_ptr(&q, what);
  p = (T *)q;
  return s;
}

// Every kernel of the library is launched with programmatic stream
// serialisation allowed: the next kernel of the stream may be launched while
// this one drains.  Each kernel therefore waits for the grids before it
// (griddepcontrol.wait, below) before it touches global memory, so results
// are ordered as on a plain stream while launch latency and CTA rasterisation
// overlap the previous kernel's tail.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Wraps every kernel launch: counts it and, while tracing is on, records an
// event pair around it on the launching stream.
struct LaunchScope {
  int slot;
  cudaStream_t stream;
  LaunchScope(const char *name, cudaStream_t s);
  ~LaunchScope();
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ----------------------------------------------------------------- device side
// Start of every kernel: wait until the grids this one depends on have
// completed and their writes are visible, then allow the stream's next grid
// to begin launching (its CTAs wait in turn at their own start).
__device__ __forceinline__ void grid_dep_sync() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
constexpr uint32_t kDrawAccept = 0u;
constexpr uint32_t kDrawSample = 1u;

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of two
// 32x32->64 products with multipliers 0xD2511F53 / 0xCD9E8D57, a word
// permutation XOR-ing the high halves into the other words and the round key,
// and a Weyl key bump (0x9E3779B9, 0xBB67AE85) between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k.x += 0x9E3779B9u;
      k.y += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
  }
  return c;
}

// Top 24 bits of the first Philox word for counter (pos, draw, seq, step).
__device__ __forceinline__ uint32_t uniform_u24(uint64_t seed, uint64_t step,
                                                uint32_t seq, uint32_t pos,
                                                uint32_t draw) {
  const uint4 o = philox4x32_10(make_uint4(pos, draw, seq, (uint32_t)step),
                                make_uint2((uint32_t)seed, (uint32_t)(seed >> 32)));
  return o.x >> 8;
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float elem_to_f32(float x) { return x; }
__device__ __forceinline__ float elem_to_f32(uint16_t x) {
  return __uint_as_float((uint32_t)x << 16);
}

template <typename T> __device__ __forceinline__ float load_elem(const T *p);
template <> __device__ __forceinline__ float load_elem<float>(const float *p) { return __ldg(p); }
template <> __device__ __forceinline__ float load_elem<uint16_t>(const uint16_t *p) {
  return __uint_as_float((uint32_t)__ldg(p) << 16);
}

__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Packed fp32 pairs (sm_100+ f32x2 arithmetic): two IEEE round-to-nearest
// operations per instruction, bit-identical to the scalar ones.  A packed
// multiply feeding a packed add or subtract has been seen contracted into a
// fused multiply-add despite the explicit rounding modifier; where each
// rounding is part of a specification, the products go through the scalar
// __fmul_rn intrinsic instead.
__device__ __forceinline__ unsigned long long f2_pack(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(unsigned long long r, float &a, float &b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long f2_sub(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
// max of two bf16 pairs (a NaN operand yields the other operand)
__device__ __forceinline__ uint32_t bf2_max(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// max of two bf16 pairs, NaN-propagating
__device__ __forceinline__ uint32_t bf2_max_nan(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ----------------------------------------------------------------------------
// The sampling arithmetic: an fp32 exponential from basic IEEE operations
// only (explicit _rn intrinsics, so no contraction or fast-math can change a
// bit): 0 below -80; n = nearest integer to a*log2(e) by the 1.5*2^23 shift;
// Cody-Waite two-constant reduction r = a - n*ln2; e^r by the Taylor series to
// degree 7 (coefficients 1/k! rounded to fp32) in Horner form with fused
// multiply-adds; scaled by 2^n.  Max error about 2 ulp over [-80, 0].
// ----------------------------------------------------------------------------
__device__ __forceinline__ float exp32_repro(float a) {
  const float t = __fmaf_rn(a, 0x1.715476p+0f, 0x1.8p+23f);
  const float n = __fsub_rn(t, 0x1.8p+23f);
  float r = __fmaf_rn(-n, 0x1.62e4p-1f, a);
  r = __fmaf_rn(-n, 0x1.7f7d1cp-20f, r);
  float p = 1.0f / 5040.0f;
  p = __fmaf_rn(p, r, 1.0f / 720.0f);
  p = __fmaf_rn(p, r, 1.0f / 120.0f);
  p = __fmaf_rn(p, r, 1.0f / 24.0f);
  p = __fmaf_rn(p, r, 1.0f / 6.0f);
  p = __fmaf_rn(p, r, 0.5f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  // t is 1.5*2^23 + n exactly (|n| < 2^22), so the integer n sits in its bits;
  // p * 2^n is exact for a >= -80 (p in [0.7, 1.5], the product is a normal
  // number), so adding n to p's exponent field gives its bits without a
  // multiply
  const int ni = __float_as_int(t) - 0x4B400000;
  const float e = __int_as_float(__float_as_int(p) + (ni << 23));
  return (a >= -80.0f) ? e : 0.0f;
}

// exp32_repro of both lanes of a packed pair: the same fp32 operations as
// packed pair instructions (fused multiply-adds and one subtraction; no
// multiply feeds an addition, so none can be contracted), bit for bit equal
// to exp32_repro for a >= -80.  Below -80 the argument is clamped to -80, so
// the result is exp32_repro(-80) (about 1.8e-35) instead of 0: both are 0
// once floored onto the 2^-40 or 2^-62 grid of the sampling weights, and a
// product or difference with a value of at least 2^-62 rounds the same way.
__device__ __forceinline__ unsigned long long f2_add_rz(unsigned long long a,
                                                        unsigned long long b) {
  unsigned long long r;
  asm("add.rz.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long f2_splat(float a) { return f2_pack(a, a); }
__device__ __forceinline__ unsigned long long exp32x2(unsigned long long a2) {
  float a0, a1;
  f2_unpack(a2, a0, a1);
  a2 = f2_pack(fmaxf(a0, -80.0f), fmaxf(a1, -80.0f));
  const unsigned long long t2 = f2_fma(a2, f2_splat(0x1.715476p+0f), f2_splat(0x1.8p+23f));
  const unsigned long long n2 = f2_sub(t2, f2_splat(0x1.8p+23f));
  unsigned long long r2 = f2_fma(n2, f2_splat(-0x1.62e4p-1f), a2);
  r2 = f2_fma(n2, f2_splat(-0x1.7f7d1cp-20f), r2);
  unsigned long long p2 = f2_fma(f2_splat(1.0f / 5040.0f), r2, f2_splat(1.0f / 720.0f));
  p2 = f2_fma(p2, r2, f2_splat(1.0f / 120.0f));
  p2 = f2_fma(p2, r2, f2_splat(1.0f / 24.0f));
  p2 = f2_fma(p2, r2, f2_splat(1.0f / 6.0f));
  p2 = f2_fma(p2, r2, f2_splat(0.5f));
  p2 = f2_fma(p2, r2, f2_splat(1.0f));
  p2 = f2_fma(p2, r2, f2_splat(1.0f));
  float t0, t1, q0, q1;
  f2_unpack(t2, t0, t1);
  f2_unpack(p2, q0, q1);
  // t = 1.5 2^23 + n, whose bits are 0x4B400000 + n; shifted left by 23 the
  // constant leaves the 32-bit word, so (t bits << 23) adds n to p's exponent
  const float e0 = __int_as_float(__float_as_int(q0) + (__float_as_int(t0) << 23));
  const float e1 = __int_as_float(__float_as_int(q1) + (__float_as_int(t1) << 23));
  return f2_pack(e0, e1);
}

// ---------------------------------------------------------------- bulk ring
// mbarrier primitives of a shared-memory ring filled by TMA bulk copies, every
// wait bounded by kRingWaitNs
constexpr unsigned long long kRingWaitNs = 2000000000ull;  // 2 s
__device__ __forceinline__ unsigned long long ring_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ uint32_t ring_addr(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void ring_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void ring_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// an arrival that also expects `bytes` of bulk copies to complete on the barrier
__device__ __forceinline__ void ring_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
// TMA bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from global into this CTA's shared memory, completing on `bar`
__device__ __forceinline__ void ring_bulk(uint32_t dst, const void *src, uint32_t bytes,
                                             uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ bool ring_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase of `parity`; false (and *abort set) when it runs
// out or another warp of the CTA has given up.
static __device__ __noinline__ bool ring_wait_slow(uint32_t bar, uint32_t parity,
                                               volatile int *abort) {
  const unsigned long long t0 = ring_ns();
  for (uint32_t it = 1;; ++it) {
    if (ring_try(bar, parity)) return true;
    if ((it & 63) == 0) {
      if (*abort) return false;
      if (ring_ns() - t0 > kRingWaitNs) {
        *abort = 1;
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool ring_wait(uint32_t bar, uint32_t parity, volatile int *abort) {
  return ring_try(bar, parity) || ring_wait_slow(bar, parity, abort);
}

}  // namespace sv
