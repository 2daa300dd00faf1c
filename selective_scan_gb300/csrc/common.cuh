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

// Conv output rounded to bf16 as the double-precision definition rounds it.
//
// The value silu(bias + sum_k w_k u_k) is computed in fp32 together with a
// bound on its error; when the fp32 value lies farther than that bound from
// the bf16 rounding boundary nearest to it, its bf16 rounding equals that of
// the exact value rounded first to fp32 and then to bf16. Otherwise (about
// one element in a thousand) the value is recomputed in fp64. This is Ziv's
// rounding test; it keeps the conv output, and so the state it feeds,
// independent of fp32 rounding noise.
template <int K>
__device__ __forceinline__ float conv_silu_bf16_exact(float bias, const float (&w)[K], const float (&u)[K]) {
  bool retry;
  const float v = conv_silu_bf16_fast<K>(bias, w, u, retry);
  return retry ? conv_silu_bf16_fp64<K>(bias, w, u) : v;
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
