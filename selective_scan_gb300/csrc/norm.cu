// Gated RMSNorm: out = rmsnorm(x * silu(z)) * weight, RMS per channel group.
//
// Semantics: gllm PR #85 "feat(backend): Mamba2 ops, with CPU reference
// implementations", section "Ops" (GatedRMSNorm, the gate applied before the
// norm, the RMS taken per group).
//
// One CTA per (kNormRows rows, group): kNormThreads threads (two warps) take
// each row. Each thread holds up to kVPT 16-byte vectors of its row's group in
// registers (x * silu(z) in fp32), so x and z are read from HBM exactly once
// and the output written once: 3 * dim * sizeof(act) bytes per row,
// HBM-bound. The group's fp32 weights are copied once per CTA into shared
// memory while x and z are in flight (from global memory directly when the
// group is wider than kNormSmemW channels): a quarter of their L2 traffic
// against one row per CTA. (Measured at 65 536 x 3 072: 0.188 ms with two
// warps a row and four rows a CTA, against 0.207 with four warps a row and
// two rows, 0.222 with four and four, 0.198 with one warp and eight rows.) The sum of squares is reduced warp by warp and then across
// the half's warps in a fixed order (deterministic). Groups wider than
// kNormThreads * kVPT vectors stream the remainder twice (the second pass
// mostly hits L2).
#include "common.cuh"

namespace mamba2 {

constexpr int kNormThreads = 64;   // threads per row
constexpr int kNormRows = 4;       // rows per CTA
constexpr int kVPT = 6;            // 16-byte vectors per thread kept in registers
constexpr int kNormSmemW = 12288;  // widest group whose weights are staged in shared memory (48 KB)

template <typename T>
__global__ void __launch_bounds__(kNormThreads * kNormRows)
gated_rmsnorm_kernel(const NormArgs a, const int w_smem) {
  constexpr int V = Vec16<T>::n;
  extern __shared__ __align__(16) float wsm[];  // [group width] when w_smem
  __shared__ float wsum[kNormRows][kNormThreads / 32];
  const int r = threadIdx.x / kNormThreads;
  const int tid = threadIdx.x - r * kNormThreads, warp = tid >> 5, lane = tid & 31;
  const int gs = a.dim / a.groups;
  const int nv = gs / V;
  const int64_t rp = blockIdx.x / a.groups;
  const int grp = (int)(blockIdx.x - rp * a.groups);
  const int64_t row = rp * kNormRows + r;
  const bool live = row < a.rows;  // the last CTA may hold fewer rows
  const float* wg = a.weight + (int64_t)grp * gs;
  if (w_smem) {
    for (int i = threadIdx.x; i < gs / 4; i += kNormThreads * kNormRows)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"((uint32_t)__cvta_generic_to_shared(wsm + 4 * i)),
                   "l"(wg + 4 * i));
  }
  asm volatile("cp.async.commit_group;\n" ::: "memory");
  // launched as a programmatic dependent of the kernel before it (the scan that
  // writes x): the weights above are a parameter; x and z come after this wait
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const float* w = w_smem ? wsm : wg;
  const int64_t base = row * a.dim + (int64_t)grp * gs;
  const T* x = static_cast<const T*>(a.x) + base;
  const T* z = static_cast<const T*>(a.z) + base;
  T* out = static_cast<T*>(a.dst) + base;

  uint4 xr[kVPT], zr[kVPT];
#pragma unroll
  for (int i = 0; i < kVPT; ++i) {
    const int vi = tid + kNormThreads * i;
    if (live && vi < nv) {
      xr[i] = __ldcs(reinterpret_cast<const uint4*>(x + vi * V));
      zr[i] = __ldcs(reinterpret_cast<const uint4*>(z + vi * V));
    }
  }
  float v[kVPT][V];
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < kVPT; ++i) {
    const int vi = tid + kNormThreads * i;
    if (live && vi < nv) {
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
  for (int vi = tid + kNormThreads * kVPT; live && vi < nv; vi += kNormThreads) {  // wide groups
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
  if (lane == 0) wsum[r][warp] = ss;
  asm volatile("cp.async.wait_group 0;\n" ::: "memory");
  __syncthreads();  // partial sums and the staged weights
  if (!live) return;
  float tot = 0.0f;
#pragma unroll
  for (int i = 0; i < kNormThreads / 32; ++i) tot += wsum[r][i];
  const float inv = rsqrtf(tot / (float)gs + a.eps);

#pragma unroll
  for (int i = 0; i < kVPT; ++i) {
    const int vi = tid + kNormThreads * i;
    if (vi < nv) {
      float o[V];
#pragma unroll
      for (int q = 0; q < V / 4; ++q) {
        const float4 wq = *reinterpret_cast<const float4*>(w + vi * V + 4 * q);
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
  const int64_t items = (int64_t)((a.rows + kNormRows - 1) / kNormRows) * a.groups;
  if (items == 0) return cudaSuccess;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int gs = a.dim / a.groups;
  const int w_smem = gs <= kNormSmemW ? 1 : 0;
  const size_t smem = w_smem ? (size_t)gs * sizeof(float) : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)items, 1, 1);
  cfg.blockDim = dim3(kNormThreads * kNormRows, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (act == MAMBA2_BF16) return cudaLaunchKernelEx(&cfg, gated_rmsnorm_kernel<__nv_bfloat16>, a, w_smem);
  return cudaLaunchKernelEx(&cfg, gated_rmsnorm_kernel<float>, a, w_smem);
}

}  // namespace mamba2
