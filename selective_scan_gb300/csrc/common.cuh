// Internal helpers shared by the libmamba2 kernels (product path only).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mamba2.h"
#include "kernels.h"

namespace mamba2 {

__device__ __forceinline__ int32_t seq_slot(const SeqTable& t, int i) {
  return (int32_t)(t.slot_fresh[i] & 0x7fffffffu);
}
__device__ __forceinline__ bool seq_fresh(const SeqTable& t, int i) {
  return (t.slot_fresh[i] >> 31) != 0u;
}

// Largest i in [0, n) with tile[i] <= w (tile is non-decreasing).
__device__ __forceinline__ int find_tile_seq(const SeqTable& t, int w) {
  int lo = 0, hi = t.n - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (t.tile[mid] <= w) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// ---------------------------------------------------------------------------
// Activation access
// ---------------------------------------------------------------------------
template <typename T> struct Act;
template <> struct Act<float> {
  static constexpr mamba2_dtype code = MAMBA2_F32;
  static constexpr int kVec = 4;  // elements per 16-byte vector
  __device__ __forceinline__ static float to_f(float v) { return v; }
  __device__ __forceinline__ static float from_f(float v) { return v; }
};
template <> struct Act<__nv_bfloat16> {
  static constexpr mamba2_dtype code = MAMBA2_BF16;
  static constexpr int kVec = 8;
  __device__ __forceinline__ static float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
  __device__ __forceinline__ static __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

// Round-trip of an fp32 value through the activation type (a rounding point).
template <typename T>
__device__ __forceinline__ float round_act(float v) {
  return Act<T>::to_f(Act<T>::from_f(v));
}

// 16-byte vector of activations, unpacked to fp32.
template <typename T> struct Vec16;
template <> struct Vec16<float> {
  static constexpr int n = 4;
  __device__ __forceinline__ static void load(const float* p, float* o) {
    float4 v = *reinterpret_cast<const float4*>(p);
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  }
  __device__ __forceinline__ static void load_stream(const float* p, float* o) {
    float4 v = __ldcs(reinterpret_cast<const float4*>(p));
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  }
  __device__ __forceinline__ static void store(float* p, const float* o) {
    *reinterpret_cast<float4*>(p) = make_float4(o[0], o[1], o[2], o[3]);
  }
  __device__ __forceinline__ static void store_stream(float* p, const float* o) {
    __stcs(reinterpret_cast<float4*>(p), make_float4(o[0], o[1], o[2], o[3]));
  }
};
template <> struct Vec16<__nv_bfloat16> {
  static constexpr int n = 8;
  __device__ __forceinline__ static void unpack(uint4 v, float* o) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = __uint_as_float(w[i] << 16);
      o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ __forceinline__ static uint4 pack(const float* o) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 h = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
  __device__ __forceinline__ static void load(const __nv_bfloat16* p, float* o) {
    unpack(*reinterpret_cast<const uint4*>(p), o);
  }
  __device__ __forceinline__ static void load_stream(const __nv_bfloat16* p, float* o) {
    unpack(__ldcs(reinterpret_cast<const uint4*>(p)), o);
  }
  __device__ __forceinline__ static void store(__nv_bfloat16* p, const float* o) {
    *reinterpret_cast<uint4*>(p) = pack(o);
  }
  __device__ __forceinline__ static void store_stream(__nv_bfloat16* p, const float* o) {
    __stcs(reinterpret_cast<uint4*>(p), pack(o));
  }
};

// silu(v) = v * sigmoid(v) with the fast exponential and reciprocal (a few ulp).
__device__ __forceinline__ float silu_f(float v) { return __fdividef(v, 1.0f + __expf(-v)); }

// softplus(v) = max(v, 0) + log1p(exp(-|v|)), no clamp.
__device__ __forceinline__ float softplus_f(float v) {
  return fmaxf(v, 0.0f) + log1pf(__expf(-fabsf(v)));
}

// fp64 evaluation of silu(bias + sum_k w_k u_k) with separately rounded
// multiplies and adds in tap order, rounded double -> fp32 -> bf16.
template <int K>
__device__ __forceinline__ float conv_silu_bf16_fp64(float bias, const float* w, const float* u) {
  double pd = (double)bias;
#pragma unroll
  for (int k = 0; k < K; ++k) pd = __dadd_rn(pd, __dmul_rn((double)w[k], (double)u[k]));
  const double vd = __ddiv_rn(pd, __dadd_rn(1.0, exp(-pd)));
  return __bfloat162float(__float2bfloat16_rn(__double2float_rn(vd)));
}

// Fast half of the rounding test: the fp32 value rounded to bf16, with
// `retry` set when the value lies within its error bound of the bf16 rounding
// boundary (then only the fp64 evaluation decides the rounding). For a value
// v >= 0 whose bf16 truncation is t, round-to-nearest-even goes up exactly
// when v passes the midpoint m = t + half a bf16 step, whose fp32 bit
// pattern is (bits(v) & 0xffff0000) | 0x8000 (likewise for v < 0 by
// symmetry); that is the only boundary within half a bf16 step of v.
template <int K>
__device__ __forceinline__ float conv_silu_bf16_fast(float bias, const float (&w)[K], const float (&u)[K],
                                                     bool& retry) {
  float pre = bias;
  float psum = 0.0f;  // sum of |partial sums|: each fma rounds once, by <= 2^-24 of its result
#pragma unroll
  for (int k = 0; k < K; ++k) {
    pre = fmaf(w[k], u[k], pre);
    psum += fabsf(pre);
  }
  const float v = __fdividef(pre, 1.0f + __expf(-pre));
  // |v - silu_exact| <= 1.1 * 2^-24 * psum            (pre's error; |silu'| < 1.1)
  //   + (14 + 0.75 |pre|) * 2^-24 * |v|   (ex2 8, argument scaling 0.7|pre|, add 1,
  //                                        reciprocal 2, multiply 1, fp32 rounding of
  //                                        the exact value 2, all in units of 2^-24 |v|)
  // Any violation of this bound would show as a conv output differing from
  // the double-precision definition, which the GPU parity tests compare bit
  // for bit.
  const float err = fmaf(1.1f * 0x1p-24f, psum, fmaf(0.75f, fabsf(pre), 14.0f) * 0x1p-24f * fabsf(v)) +
                    0x1p-126f;
  const float mid = __uint_as_float((__float_as_uint(v) & 0xffff0000u) | 0x8000u);
  retry = !(fabsf(v - mid) > err);  // also true for NaN / inf
  return __bfloat162float(__float2bfloat16_rn(v));
}

// ---- double-float (pair of fp32) arithmetic: Dekker's and Knuth's error-free
// transformations (two-sum, two-product with a fused multiply-add), about 46
// significant bits
struct DF {
  float hi, lo;
};
__device__ __forceinline__ DF df_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  return {s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}
__device__ __forceinline__ DF df_fast_two_sum(float a, float b) {  // |a| >= |b|
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ DF df_add(DF x, DF y) {
  const DF s = df_two_sum(x.hi, y.hi);
  return df_fast_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(x.lo, y.lo)));
}
__device__ __forceinline__ DF df_mul(DF x, DF y) {
  const float p = __fmul_rn(x.hi, y.hi);
  const float e = __fmaf_rn(x.hi, y.hi, -p);
  return df_fast_two_sum(p, __fmaf_rn(x.hi, y.lo, __fmaf_rn(x.lo, y.hi, e)));
}
__device__ __forceinline__ DF df_div(DF x, DF y) {
  const float q1 = __fdiv_rn(x.hi, y.hi);
  const DF r = df_add(x, df_mul(y, DF{-q1, 0.0f}));
  return df_fast_two_sum(q1, __fdiv_rn(r.hi, y.hi));
}
// 1/k! as a double-float constant
__host__ __device__ constexpr DF df_inv_fact(int k) {
  double f = 1.0;
  for (int i = 2; i <= k; ++i) f *= (double)i;
  const double v = 1.0 / f;
  const float hi = (float)v;
  return {hi, (float)(v - (double)hi)};
}

// Middle tier of the rounding test: silu(bias + sum_k w_k u_k) in double-float
// (exact products and sums; e^-p by range reduction to |r| <= ln2/2 and its
// Taylor series to degree 12, then 2^n), rounded as the double-precision
// definition rounds it: to fp32, then to bf16. Undecided (left to fp64) when the
// value lies within its error bound of the edge of the fp32 rounding interval of
// the bf16 midpoint, or outside the range handled here.
template <int K>
__device__ __forceinline__ float conv_silu_bf16_df(float bias, const float* w, const float* u, bool& undecided) {
  DF p = {bias, 0.0f};
  float psum = fabsf(bias);
#pragma unroll
  for (int k = 0; k < K; ++k) {
    const float m = __fmul_rn(w[k], u[k]);
    p = df_add(p, DF{m, __fmaf_rn(w[k], u[k], -m)});
    psum += fabsf(p.hi);
  }
  undecided = true;
  if (!(fabsf(p.hi) <= 80.0f) || !(fabsf(p.hi) >= 0x1p-60f)) return 0.0f;
  // e^-p = 2^n e^r, r = -p - n ln 2 (ln 2 as 0.693145751953125 + its remainder, so
  // that n times the first part is exact for |n| <= 128)
  const float n = rintf(__fmul_rn(-p.hi, 1.4426950408889634f));
  const float ln2a = 0.693145751953125f, ln2b = (float)(0.69314718055994530942 - 0.693145751953125);
  DF r = df_add(DF{-p.hi, -p.lo}, DF{__fmul_rn(-n, ln2a), 0.0f});
  const float nb = __fmul_rn(-n, ln2b);
  r = df_add(r, DF{nb, __fmaf_rn(-n, ln2b, -nb)});
  // sum_{k<=12} r^k / k! by Estrin's scheme (four dependent levels instead of twelve)
  auto ma = [](DF a, DF x, DF b) { return df_add(df_mul(a, x), b); };  // a x + b
  const DF r2 = df_mul(r, r), r4 = df_mul(r2, r2), r8 = df_mul(r4, r4);
  const DF q0 = ma(df_inv_fact(1), r, df_inv_fact(0)), q1 = ma(df_inv_fact(3), r, df_inv_fact(2));
  const DF q2 = ma(df_inv_fact(5), r, df_inv_fact(4)), q3 = ma(df_inv_fact(7), r, df_inv_fact(6));
  const DF q4 = ma(df_inv_fact(9), r, df_inv_fact(8)), q5 = ma(df_inv_fact(11), r, df_inv_fact(10));
  const DF s0 = ma(q1, r2, q0), s1 = ma(q3, r2, q2), s2 = ma(q5, r2, q4);
  const DF t0 = ma(s1, r4, s0), t1 = ma(df_inv_fact(12), r4, s2);
  DF e = ma(t1, r8, t0);
  const float sc = __int_as_float((127 + (int)n) << 23);  // 2^n, |n| <= 116 here
  e = DF{__fmul_rn(e.hi, sc), __fmul_rn(e.lo, sc)};
  const DF v = df_div(p, df_add(DF{1.0f, 0.0f}, e));
  // the bf16 midpoint m nearest v, and the half-width h of m's fp32 rounding interval
  const float m = __uint_as_float((__float_as_uint(v.hi) & 0xffff0000u) | 0x8000u);
  const uint32_t ex = (__float_as_uint(m) >> 23) & 0xffu;
  if (ex <= 30u) return 0.0f;  // near the subnormal range: fp64 decides
  const float h = __uint_as_float((ex - 24u) << 23);
  // |v - (the definition's double value)| <= E: 2^-38 |v| covers this tier's
  // arithmetic and the definition's own rounding, 2^-44 psum the cancellation
  // of the sum's partial values in either evaluation
  const float E = fmaf(0x1p-38f, fabsf(v.hi), 0x1p-44f * psum);
  const float d = fabsf(__fadd_rn(__fsub_rn(v.hi, m), v.lo));
  if (d < h - E) {  // the value rounds to m in fp32: a tie, to even in bf16
    undecided = false;
    return __bfloat162float(__float2bfloat16_rn(m));
  }
  if (d > h + E) {  // strictly on one side of m's interval
    undecided = false;
    const float x = __fadd_rn(v.hi, v.lo);
    return __bfloat162float(__float2bfloat16_rn(x));
  }
  return 0.0f;
}

// Conv output rounded to bf16 as the double-precision definition rounds it.
//
// The value silu(bias + sum_k w_k u_k) is computed in fp32 together with a
// bound on its error; when the fp32 value lies farther than that bound from
// the bf16 rounding boundary nearest to it, its bf16 rounding equals that of
// the exact value rounded first to fp32 and then to bf16. Otherwise (about
// one element in two thousand) the value is recomputed in double-float, and in
// fp64 when that is still too close to call (which no workload here has shown).
// This is Ziv's rounding test; it keeps the conv output, and so the state it
// feeds, independent of fp32 rounding noise.
template <int K>
__device__ __forceinline__ float conv_silu_bf16_exact(float bias, const float (&w)[K], const float (&u)[K]) {
  bool retry;
  const float v = conv_silu_bf16_fast<K>(bias, w, u, retry);
  if (!retry) return v;
  bool undecided;
  const float v2 = conv_silu_bf16_df<K>(bias, w, u, undecided);
  return undecided ? conv_silu_bf16_fp64<K>(bias, w, u) : v2;
}

// Conv output for one channel at the activation type: bf16 through the exact
// rounding test, fp32 as computed.
template <typename T, int K>
__device__ __forceinline__ float conv_silu_act(float bias, const float (&w)[K], const float (&u)[K]) {
  if constexpr (Act<T>::code == MAMBA2_BF16) {
    return conv_silu_bf16_exact<K>(bias, w, u);
  } else {
    float acc = bias;
#pragma unroll
    for (int k = 0; k < K; ++k) acc = fmaf(w[k], u[k], acc);
    return silu_f(acc);
  }
}

}  // namespace mamba2
