// rowstat.cuh -- online softmax statistics of logit rows in the log2
// domain, shared by the kernels that stream vocabulary rows (row statistics
// of the verify step, top-K expansion of the draft tree), sm_103a.
#pragma once

#include "common.cuh"

namespace sv {

constexpr int kRsUnroll = 8;  // 16-byte words per thread and batch

// Per-thread online statistics.  mx = running max of raw logits (exact);
// mk = fl(mx * k), the log2-domain reference of the sum; s = sum of
// exp2(fma(x, k, -mk)) over the elements seen, kept as two packed pairs.
// Each exponent is one fused multiply-add, rounded once, and the output pair
// (mk, s) states the reference the sum was taken against, so no rounding of
// mk enters q.
struct StatState {
  float mx, mk;
  unsigned long long s01, s23;  // packed partial sums
};

// the reference used inside the exponent (a row that so far holds only -inf
// or NaN uses 0, so -inf contributes 0 and NaN stays NaN)
__device__ __forceinline__ float stat_ref(const StatState &st) {
  return st.mx == -INFINITY ? 0.0f : st.mk;
}

__device__ __forceinline__ void stat_raise(StatState &st, float cm, float k) {
  // cm > st.mx: move the reference up and rescale the sums
  const float nk = __fmul_rn(cm, k);
  const float f = (st.mx == -INFINITY) ? 0.0f : ex2_approx(__fsub_rn(st.mk, nk));
  const unsigned long long f2 = f2_pack(f, f);
  st.s01 = f2_mul(st.s01, f2);
  st.s23 = f2_mul(st.s23, f2);
  st.mx = cm;
  st.mk = nk;
}

// exp2 of a packed pair, accumulated
__device__ __forceinline__ unsigned long long ex2_acc(unsigned long long acc,
                                                      unsigned long long y2) {
  float y0, y1;
  f2_unpack(y2, y0, y1);
  return f2_add(acc, f2_pack(ex2_approx(y0), ex2_approx(y1)));
}

// Returns the batch's maximum logit (NaN elements are skipped by the maxima),
// which the tree expansion reuses as its top-K gate.
template <typename E>
__device__ __forceinline__ float stat_batch(const uint4 (&w)[kRsUnroll], StatState &st, float k);

// kRsUnroll words of 8 bf16 logits
template <>
__device__ __forceinline__ float stat_batch<uint16_t>(const uint4 (&w)[kRsUnroll], StatState &st,
                                                      float k) {
  uint32_t m[kRsUnroll];
#pragma unroll
  for (int j = 0; j < kRsUnroll; ++j) m[j] = bf2_max(bf2_max(w[j].x, w[j].y), bf2_max(w[j].z, w[j].w));
#pragma unroll
  for (int h = kRsUnroll / 2; h; h >>= 1)
#pragma unroll
    for (int j = 0; j < h; ++j) m[j] = bf2_max(m[j], m[j + h]);
  const float cm = fmaxf(bf16_lo(m[0]), bf16_hi(m[0]));
  if (cm > st.mx) stat_raise(st, cm, k);
  const float r = stat_ref(st);
  const unsigned long long k2 = f2_pack(k, k), nr2 = f2_pack(-r, -r);
#pragma unroll
  for (int j = 0; j < kRsUnroll; ++j) {
    const uint32_t q[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const unsigned long long y2 = f2_fma(f2_pack(bf16_lo(q[h]), bf16_hi(q[h])), k2, nr2);
      if (h & 1)
        st.s23 = ex2_acc(st.s23, y2);
      else
        st.s01 = ex2_acc(st.s01, y2);
    }
  }
  return cm;
}

// kRsUnroll words of 4 fp32 logits
template <>
__device__ __forceinline__ float stat_batch<float>(const uint4 (&w)[kRsUnroll], StatState &st,
                                                   float k) {
  float m[kRsUnroll];
#pragma unroll
  for (int j = 0; j < kRsUnroll; ++j)
    m[j] = fmaxf(fmaxf(__uint_as_float(w[j].x), __uint_as_float(w[j].y)),
                 fmaxf(__uint_as_float(w[j].z), __uint_as_float(w[j].w)));
#pragma unroll
  for (int h = kRsUnroll / 2; h; h >>= 1)
#pragma unroll
    for (int j = 0; j < h; ++j) m[j] = fmaxf(m[j], m[j + h]);
  if (m[0] > st.mx) stat_raise(st, m[0], k);
  const float r = stat_ref(st);
  const unsigned long long k2 = f2_pack(k, k), nr2 = f2_pack(-r, -r);
#pragma unroll
  for (int j = 0; j < kRsUnroll; ++j) {
    st.s01 = ex2_acc(st.s01, f2_fma(f2_pack(__uint_as_float(w[j].x), __uint_as_float(w[j].y)),
                                    k2, nr2));
    st.s23 = ex2_acc(st.s23, f2_fma(f2_pack(__uint_as_float(w[j].z), __uint_as_float(w[j].w)),
                                    k2, nr2));
  }
  return m[0];
}

// one logit (ragged head / tail, and the short remainder of a segment)
__device__ __forceinline__ void stat1(float x, StatState &st, float k) {
  if (x > st.mx) stat_raise(st, x, k);
  st.s01 = f2_add(st.s01, f2_pack(ex2_approx(fmaf(x, k, -stat_ref(st))), 0.0f));
}
template <typename E>
__device__ __forceinline__ void stat_word(uint4 v, StatState &st, float k);
template <>
__device__ __forceinline__ void stat_word<uint16_t>(uint4 v, StatState &st, float k) {
  const uint32_t q[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    stat1(bf16_lo(q[h]), st, k);
    stat1(bf16_hi(q[h]), st, k);
  }
}
template <>
__device__ __forceinline__ void stat_word<float>(uint4 v, StatState &st, float k) {
  stat1(__uint_as_float(v.x), st, k);
  stat1(__uint_as_float(v.y), st, k);
  stat1(__uint_as_float(v.z), st, k);
  stat1(__uint_as_float(v.w), st, k);
}

// Merge (mx2, mk2, s2) into (mx, mk, s): log2-domain references, -inf refs
// contribute nothing, NaN sums stay NaN.  The rescaled sum is one explicit
// multiply and one fused multiply-add, so every kernel that inlines this
// merge rounds it the same way (no contraction choice left to the compiler).
__device__ __forceinline__ void st_combine(float &mx, float &mk, float &s, float mx2, float mk2,
                                           float s2) {
  const float a = (mx == -INFINITY) ? -INFINITY : mk;
  const float b = (mx2 == -INFINITY) ? -INFINITY : mk2;
  const float M = fmaxf(a, b);
  if (M == -INFINITY) {
    s = s + s2;
  } else {
    s = __fmaf_rn(s, ex2_approx(a - M), __fmul_rn(s2, ex2_approx(b - M)));
  }
  mx = fmaxf(mx, mx2);
  mk = M;
}

// Combine the triples of the lanes of a warp: the largest reference wins,
// every lane rescales its sum to it once, then max and sum reductions.
__device__ __forceinline__ void warp_stat_combine(float &mx, float &mk, float &s) {
  const float a = (mx == -INFINITY) ? -INFINITY : mk;
  float M = a;
#pragma unroll
  for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (M != -INFINITY) s = __fmul_rn(s, ex2_approx(a - M));
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  mk = M;
}


}  // namespace sv
