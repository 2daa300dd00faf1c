// Gated RMSNorm: out = rmsnorm(x * silu(z)) * weight, RMS per channel group.
//
// Semantics: gllm PR #85 "feat(backend): Mamba2 ops, with CPU reference
// implementations", section "Ops" (GatedRMSNorm, the gate applied before the
// norm, the RMS taken per group).
//
// One CTA of kNormThreads per (row, group). Each thread holds up to kVPT
// 16-byte vectors of the group in registers (x * silu(z) in fp32), so x and z
// are read from HBM exactly once and the output written once:
// 3 * dim * sizeof(act) bytes per row, HBM-bound. The sum of squares is
// reduced warp by warp and then across the CTA's warps in a fixed order
// (deterministic). Groups wider than kNormThreads * kVPT vectors stream the
// remainder twice (the second pass mostly hits L2).
#include "common.cuh"

namespace mamba2 {

constexpr int kNormThreads = 128;
constexpr int kVPT = 4;  // 16-byte vectors per thread kept in registers

template <typename T>
__global__ void __launch_bounds__(kNormThreads)
gated_rmsnorm_kernel(const NormArgs a) {
  constexpr int V = Vec16<T>::n;
  __shared__ float wsum[kNormThreads / 32];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t item = blockIdx.x;  // (row, group)
  const int gs = a.dim / a.groups;
  const int nv = gs / V;
  const int64_t row = item / a.groups;
  const int grp = (int)(item - row * a.groups);
  const int64_t base = row * a.dim + (int64_t)grp * gs;
  const T* x = static_cast<const T*>(a.x) + base;
  const T* z = static_cast<const T*>(a.z) + base;
  T* out = static_cast<T*>(a.dst) + base;
  const float* w = a.weight + (int64_t)grp * gs;

  uint4 xr[kVPT], zr[kVPT];
#pragma unroll
  for (int i = 0; i < kVPT; ++i) {
    const int vi = tid + kNormThreads * i;
    if (vi < nv) {
      xr[i] = __ldcs(reinterpret_cast<const uint4*>(x + vi * V));
      zr[i] = __ldcs(reinterpret_cast<const uint4*>(z + vi * V));
    }
  }
  float v[kVPT][V];
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < kVPT; ++i) {
    const int vi = tid + kNormThreads * i;
    if (vi < nv) {
      float xv[V], zv[V];
      Vec16<T>::load(reinterpret_cast<const T*>(&xr[i]), xv);
      Vec16<T>::load(reinterpret_cast<const T*>(&zr[i]), zv);
#pragma unroll
      for (int j = 0; j < V; ++j) {
        v[i][j] = xv[j] * silu_f(zv[j]);
        ss = fmaf(v[i][j], v[i][j], ss);
      }
    }
  }
  for (int vi = tid + kNormThreads * kVPT; vi < nv; vi += kNormThreads) {  // wide groups
    float xv[V], zv[V];
    Vec16<T>::load(x + vi * V, xv);
    Vec16<T>::load(z + vi * V, zv);
#pragma unroll
    for (int j = 0; j < V; ++j) {
      const float g = xv[j] * silu_f(zv[j]);
      ss = fmaf(g, g, ss);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) wsum[warp] = ss;
  __syncthreads();
  float tot = 0.0f;
#pragma unroll
  for (int i = 0; i < kNormThreads / 32; ++i) tot += wsum[i];
  const float inv = rsqrtf(tot / (float)gs + a.eps);

#pragma unroll
  for (int i = 0; i < kVPT; ++i) {
    const int vi = tid + kNormThreads * i;
    if (vi < nv) {
      float o[V];
      const float4* wp = reinterpret_cast<const float4*>(w + vi * V);
#pragma unroll
      for (int q = 0; q < V / 4; ++q) {
        const float4 wq = __ldg(wp + q);
        o[4 * q + 0] = v[i][4 * q + 0] * inv * wq.x;
        o[4 * q + 1] = v[i][4 * q + 1] * inv * wq.y;
        o[4 * q + 2] = v[i][4 * q + 2] * inv * wq.z;
        o[4 * q + 3] = v[i][4 * q + 3] * inv * wq.w;
      }
      Vec16<T>::store_stream(out + vi * V, o);
    }
  }
  for (int vi = tid + kNormThreads * kVPT; vi < nv; vi += kNormThreads) {
    float xv[V], zv[V], o[V];
    Vec16<T>::load(x + vi * V, xv);
    Vec16<T>::load(z + vi * V, zv);
#pragma unroll
    for (int j = 0; j < V; ++j) o[j] = xv[j] * silu_f(zv[j]) * inv * w[vi * V + j];
    Vec16<T>::store(out + vi * V, o);
  }
}

cudaError_t launch_gated_rmsnorm(const NormArgs& a, mamba2_dtype act, cudaStream_t st) {
  const int64_t items = (int64_t)a.rows * a.groups;
  if (items == 0) return cudaSuccess;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (act == MAMBA2_BF16)
    gated_rmsnorm_kernel<__nv_bfloat16><<<(unsigned)items, kNormThreads, 0, st>>>(a);
  else
    gated_rmsnorm_kernel<float><<<(unsigned)items, kNormThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace mamba2
