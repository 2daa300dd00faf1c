// Depthwise causal conv1d + SiLU over packed variable-length runs, with the
// conv-state slot read and rewritten in the same kernel.
//
// Semantics: gllm PR #85 "feat(backend): Mamba2 ops, with CPU reference
// implementations", section "Ops" (CausalConv1D): row t of a run is
// silu(bias + sum_k w[:, k] * u[t + k]) with u = slot history (zeros when
// fresh) followed by the run's inputs; the slot then holds u's last kernel-1
// rows.
//
// Layout and work split: every thread owns one 16-byte channel vector (8 bf16
// or 4 fp32 channels) over a tile of kRows consecutive rows of ONE sequence.
// Tiles never straddle sequences (the host numbers tiles per sequence). The
// tile's rows and the kernel-1 rows before it are copied asynchronously into
// the thread's own shared-memory slots, so four CTAs per SM keep enough loads
// in flight to stream at HBM speed.
// Only tile 0 of a sequence reads the slot (kRows >= kernel-1), and that same
// thread writes the new history for its channels at the end: no other thread
// touches those slot bytes, so no ordering between CTAs is needed. A
// zero-length sequence still gets one (empty) tile for its slot update.
//
// Memory: each input row is read once by its tile plus kernel-1 window rows
// read again by the next tile (L2 hits); each output row written once. The
// kernel is HBM-bound: 2 * conv_dim * sizeof(act) bytes per row.
//
// Rounding: outputs are computed in fp32 (taps in order, fast exponential and
// reciprocal for SiLU) and rounded once to the activation type, so a value
// within a few fp32 ulps of a bf16 rounding boundary may land one bf16 step
// from the double-precision definition. (The fused decode kernel rounds
// exactly instead: there the conv output feeds a state whose tolerance is
// tighter than one such step; for the 16x more outputs of a prefill the fp64
// retries of that test cost more than the whole conv.)
#include "common.cuh"
#include "kernels.h"

namespace mamba2 {

template <typename T, int K>
__global__ void __launch_bounds__(kConvThreads, 4)
conv1d_silu_kernel(const __grid_constant__ ConvArgs a) {
  constexpr int V = Vec16<T>::n;
  constexpr int H = K - 1;  // history rows
  constexpr int R = H + kConvRows;
  // raw conv inputs of this thread, u[q0 - H .. q0 + kConvRows - 1], one 16-byte
  // vector per row: [row][thread], so a warp's reads of one row are 512
  // contiguous bytes. Copied asynchronously: the thread holds no registers for
  // them while they are in flight (four CTAs per SM keep the loads deep).
  __shared__ __align__(16) uint4 sm_rows[R][kConvThreads];
  const int nvec = a.conv_dim / V;
  const int64_t item = (int64_t)blockIdx.x * kConvThreads + threadIdx.x;
  const int64_t total = (int64_t)a.tab.tile[a.tab.n] * nvec;
  if (item >= total) return;
  const int tile = (int)(item / nvec);
  const int cv = (int)(item - (int64_t)tile * nvec);
  const int s = find_tile_seq(a.tab, tile);
  const int local_tile = tile - a.tab.tile[s];
  const int row0 = a.tab.cu[s];
  const int T_len = a.tab.cu[s + 1] - row0;
  const int q0 = local_tile * kConvRows;
  const int nrows = min(kConvRows, T_len - q0);
  const bool fresh = seq_fresh(a.tab, s);
  const int64_t slot_base = (int64_t)seq_slot(a.tab, s) * H * a.conv_dim;
  const int c0 = cv * V;
  const T* x = static_cast<const T*>(a.x);
  T* dst = static_cast<T*>(a.dst);
  T* cst = static_cast<T*>(a.conv_state);
  const int t = threadIdx.x;

  // the H window rows before the tile (zeros for a fresh slot), then the tile's rows
#pragma unroll
  for (int i = 0; i < H; ++i) {
    const int pos = q0 - H + i;
    const T* src = pos >= 0 ? x + (int64_t)(row0 + pos) * a.conv_dim + c0
                            : cst + slot_base + (int64_t)(H + pos) * a.conv_dim + c0;
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(&sm_rows[i][t]);
    // a fresh slot's history is zeros: a zero-byte copy (source in the slot row, never read)
    const bool real = pos >= 0 || !fresh;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(d), "l"(real ? src : cst + slot_base + c0),
                 "r"(real ? 16 : 0));
  }
#pragma unroll
  for (int r = 0; r < kConvRows; ++r) {
    if (r < nrows) {
      const uint32_t d = (uint32_t)__cvta_generic_to_shared(&sm_rows[H + r][t]);
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(x + (int64_t)(row0 + q0 + r) * a.conv_dim + c0));
    }
  }
  asm volatile("cp.async.commit_group;\n" ::: "memory");

  // taps and bias for this thread's channels, while the rows are in flight
  // (16-byte loads: V*K floats are contiguous and 16-byte aligned since V*4 bytes is)
  float w[K][V], b[V];
  {
    const float4* wp = reinterpret_cast<const float4*>(a.weight + (int64_t)c0 * K);
#pragma unroll
    for (int q = 0; q < V * K / 4; ++q) {
      const float4 f = __ldg(wp + q);
      const float e[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) w[(4 * q + i) % K][(4 * q + i) / K] = e[i];
    }
    const float4* bp = reinterpret_cast<const float4*>(a.bias + c0);
#pragma unroll
    for (int q = 0; q < V / 4; ++q) {
      const float4 f = __ldg(bp + q);
      b[4 * q] = f.x; b[4 * q + 1] = f.y; b[4 * q + 2] = f.z; b[4 * q + 3] = f.w;
    }
  }
  asm volatile("cp.async.wait_group 0;\n" ::: "memory");  // this thread's own rows (it reads no other's)

  // tile row r: silu(bias + sum_k w[:, k] u[r + k]), each tap unpacked from smem
#pragma unroll
  for (int r = 0; r < kConvRows; ++r) {
    if (r < nrows) {
      float acc[V];
#pragma unroll
      for (int j = 0; j < V; ++j) acc[j] = b[j];
#pragma unroll
      for (int k = 0; k < K; ++k) {
        float u[V];
        Vec16<T>::load(reinterpret_cast<const T*>(&sm_rows[r + k][t]), u);
#pragma unroll
        for (int j = 0; j < V; ++j) acc[j] = fmaf(w[k][j], u[j], acc[j]);
      }
#pragma unroll
      for (int j = 0; j < V; ++j) acc[j] = silu_f(acc[j]);
      Vec16<T>::store(dst + (int64_t)(row0 + q0 + r) * a.conv_dim + c0, acc);
    }
  }

  // slot update by tile 0: new history = u[T .. T + H - 1] (bit copies)
  if (local_tile == 0) {
#pragma unroll
    for (int j = 0; j < H; ++j) {
      const int upos = T_len + j;  // index into u
      uint4 r = make_uint4(0u, 0u, 0u, 0u);
      if (upos >= H) {
        r = *reinterpret_cast<const uint4*>(x + (int64_t)(row0 + upos - H) * a.conv_dim + c0);
      } else if (!fresh) {
        // old history row upos (only when the run is shorter than H); rows
        // below j are already rewritten, but upos > j, so row upos is not
        r = *reinterpret_cast<const uint4*>(cst + slot_base + (int64_t)upos * a.conv_dim + c0);
      }
      *reinterpret_cast<uint4*>(cst + slot_base + (int64_t)j * a.conv_dim + c0) = r;
    }
  }
}

template <typename T, int K>
static cudaError_t launch_conv_t(const ConvArgs& a, cudaStream_t st) {
  const int nvec = a.conv_dim / Vec16<T>::n;
  const int64_t total = (int64_t)a.tab.tile[a.tab.n] * nvec;
  if (total == 0) return cudaSuccess;
  const int64_t blocks = (total + kConvThreads - 1) / kConvThreads;
  // four CTAs of 40-44 KB static shared memory per SM
  cudaError_t e = cudaFuncSetAttribute(conv1d_silu_kernel<T, K>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                       (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  conv1d_silu_kernel<T, K><<<(unsigned)blocks, kConvThreads, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_conv1d(const ConvArgs& a, mamba2_dtype act, int kernel, cudaStream_t st) {
  if (act == MAMBA2_BF16) {
    switch (kernel) {
      case 1: return launch_conv_t<__nv_bfloat16, 1>(a, st);
      case 2: return launch_conv_t<__nv_bfloat16, 2>(a, st);
      case 3: return launch_conv_t<__nv_bfloat16, 3>(a, st);
      case 4: return launch_conv_t<__nv_bfloat16, 4>(a, st);
    }
  } else {
    switch (kernel) {
      case 1: return launch_conv_t<float, 1>(a, st);
      case 2: return launch_conv_t<float, 2>(a, st);
      case 3: return launch_conv_t<float, 3>(a, st);
      case 4: return launch_conv_t<float, 4>(a, st);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace mamba2
