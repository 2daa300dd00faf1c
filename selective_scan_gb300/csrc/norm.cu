// Gated RMSNorm: out = rmsnorm(x * silu(z)) * weight, RMS per channel group.
//
// Semantics: gllm PR #85 "feat(backend): Mamba2 ops, with CPU reference
// implementations", section "Ops" (GatedRMSNorm, the gate applied before the
// norm, the RMS taken per group).
//
// One warp per (row, group). Each lane holds up to kMaxVec 16-byte vectors of
// the group in registers (x * silu(z) in fp32), so x and z are read from HBM
// exactly once and the output written once: 3 * dim * sizeof(act) bytes per
// row, HBM-bound. Groups wider than 32 * kMaxVec vectors are streamed twice
// (the second pass mostly hits L2).
#include "common.cuh"

namespace mamba2 {

constexpr int kNormWarps = 8;
constexpr int kMaxVec = 12;

template <typename T>
__global__ void __launch_bounds__(kNormWarps * 32)
gated_rmsnorm_kernel(const NormArgs a) {
  constexpr int V = Vec16<T>::n;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t item = (int64_t)blockIdx.x * kNormWarps + warp;
  if (item >= (int64_t)a.rows * a.groups) return;
  const int gs = a.dim / a.groups;
  const int nv = gs / V;  // vectors in the group
  const int64_t row = item / a.groups;
  const int grp = (int)(item - row * a.groups);
  const int64_t base = row * a.dim + (int64_t)grp * gs;
  const T* x = static_cast<const T*>(a.x) + base;
  const T* z = static_cast<const T*>(a.z) + base;
  T* out = static_cast<T*>(a.dst) + base;
  const float* w = a.weight + (int64_t)grp * gs;

  float v[kMaxVec][V];
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < kMaxVec; ++i) {
    const int vi = lane + 32 * i;
    if (vi < nv) {
      float xv[V], zv[V];
      Vec16<T>::load_stream(x + vi * V, xv);
      Vec16<T>::load_stream(z + vi * V, zv);
#pragma unroll
      for (int j = 0; j < V; ++j) {
        v[i][j] = xv[j] * silu_f(zv[j]);
        ss = fmaf(v[i][j], v[i][j], ss);
      }
    }
  }
  for (int vi = lane + 32 * kMaxVec; vi < nv; vi += 32) {  // wide groups
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
  const float inv = rsqrtf(ss / (float)gs + a.eps);

#pragma unroll
  for (int i = 0; i < kMaxVec; ++i) {
    const int vi = lane + 32 * i;
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
  for (int vi = lane + 32 * kMaxVec; vi < nv; vi += 32) {
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
  const int64_t blocks = (items + kNormWarps - 1) / kNormWarps;
  if (act == MAMBA2_BF16)
    gated_rmsnorm_kernel<__nv_bfloat16><<<(unsigned)blocks, kNormWarps * 32, 0, st>>>(a);
  else
    gated_rmsnorm_kernel<float><<<(unsigned)blocks, kNormWarps * 32, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace mamba2
