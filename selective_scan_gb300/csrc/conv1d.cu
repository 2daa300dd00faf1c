// Depthwise causal conv1d + SiLU over packed variable-length runs, with the
// conv-state slot read and rewritten in the same kernel.
//
// Semantics: gllm PR #85 "feat(backend): Mamba2 ops, with CPU reference
// implementations", section "Ops" (CausalConv1D): row t of a run is
// silu(bias + sum_k w[:, k] * u[t + k]) with u = slot history (zeros when
// fresh) followed by the run's inputs; the slot then holds u's last kernel-1
// rows.
//
// Layout and work split: a CTA covers 32 consecutive 16-byte channel vectors
// (8 bf16 or 4 fp32 channels each) over kConvThreads / 32 consecutive tiles of
// kConvRows rows; lane l of warp w owns channel vector l of tile w. Tiles never
// straddle sequences (the host numbers tiles per sequence). A warp copies its
// tile's rows and the kernel-1 window rows before them (from the input, or from
// the slot at a sequence start) asynchronously into its own shared-memory
// slots (a row of the warp's 32 vectors is 512 contiguous bytes), and starts
// on them as soon as its own copies land: the one CTA-wide barrier waits only
// for the taps and bias of the CTA's channels, copied once into shared memory
// beside the rows. (Window rows are read twice, the second time from L2.)
// Only tile 0 of a sequence reads the slot (kRows >= kernel-1), and that same
// thread writes the new history for its channels at the end: no other thread
// touches those slot bytes, so no ordering between CTAs is needed. A
// zero-length sequence still gets one (empty) tile for its slot update.
//
// Memory: each input row is read once (plus kernel-1 window rows at the first
// tile of a CTA or of a sequence, L2 hits); each output row written once. The
// kernel is HBM-bound: 2 * conv_dim * sizeof(act) bytes per row.
//
// Rounding: outputs are computed in fp32 (taps in order, hardware exponential
// and reciprocal for SiLU; channel pairs in packed f32x2 instructions, each
// lane rounding as the scalar instruction does) and rounded once to the
// activation type, so a value
// within a few fp32 ulps of a bf16 rounding boundary may land one bf16 step
// from the double-precision definition. (The fused decode kernel rounds
// exactly instead: there the conv output feeds a state whose tolerance is
// tighter than one such step; for the 16x more outputs of a prefill the fp64
// retries of that test cost more than the whole conv.)
#include "common.cuh"
#include "kernels.h"

namespace mamba2 {

constexpr int kConvTilesPerCta = kConvThreads / 32;  // one tile per warp

// packed fp32 pairs: one instruction does a pair's multiply-add (the kernel is
// bound by instruction issue, not by HBM, when every element costs its own)
struct P2 {
  uint64_t v;
};
__device__ __forceinline__ P2 p2(float lo, float hi) {
  P2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void p2split(P2 a, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a.v));
}
__device__ __forceinline__ P2 p2fma(P2 a, P2 b, P2 c) {
  P2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r.v) : "l"(a.v), "l"(b.v), "l"(c.v));
  return r;
}
__device__ __forceinline__ P2 p2mul(P2 a, P2 b) {
  P2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}
__device__ __forceinline__ P2 p2add(P2 a, P2 b) {
  P2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// silu(v) = v / (1 + 2^(-v log2 e)) of a pair (hardware exponential and
// reciprocal; a denominator beyond the fp32 range gives 0, the limit)
__device__ __forceinline__ P2 silu2(P2 v) {
  float t0, t1;
  p2split(p2mul(v, p2(-1.4426950408889634f, -1.4426950408889634f)), t0, t1);
  float d0, d1;
  p2split(p2add(p2(ex2_approx(t0), ex2_approx(t1)), p2(1.0f, 1.0f)), d0, d1);
  return p2mul(v, p2(rcp_approx(d0), rcp_approx(d1)));
}

template <typename T, int K>
__global__ void __launch_bounds__(kConvThreads, 3)
conv1d_silu_kernel(const __grid_constant__ ConvArgs a) {
  constexpr int V = Vec16<T>::n;
  constexpr int H = K - 1;  // history rows
  constexpr int R = H + kConvRows;
  constexpr int kWq = V * K / 4 + V / 4;  // float4s of taps and bias per channel vector
  static_assert(H <= kConvRows, "the window rows must fit in one tile");
  // raw conv inputs of this thread, u[q0 - H .. q0 + kConvRows - 1], one 16-byte
  // vector per row: [row][thread]; then the taps (V*K floats) and bias (V floats)
  // of the CTA's 32 channel vectors, [float4 q][vector] (a warp's reads of one q
  // are 512 contiguous bytes)
  __shared__ __align__(16) uint4 sm_rows[R][kConvThreads];
  __shared__ __align__(16) float4 sm_w[kWq][32];
  const int nvec = a.conv_dim / V;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int ntiles = a.tab.tile[a.tab.n];
  // CTAs in order of channel block first: neighbouring CTAs read the same rows
  const int ncb = (nvec + 31) / 32;
  const int cb = (int)(blockIdx.x % (unsigned)ncb), tg = (int)(blockIdx.x / (unsigned)ncb);
  const int tile = tg * kConvTilesPerCta + warp;
  const int cv = cb * 32 + lane;
  const bool active = tile < ntiles && cv < nvec;  // (no early return: the CTA synchronises below)
  const int s = active ? find_tile_seq(a.tab, tile) : 0;
  const int local_tile = tile - a.tab.tile[s];
  const int row0 = a.tab.cu[s];
  const int T_len = a.tab.cu[s + 1] - row0;
  const int q0 = local_tile * kConvRows;
  const int nrows = min(kConvRows, T_len - q0);
  const int c0 = cv * V;
  const T* x = static_cast<const T*>(a.x);
  T* dst = static_cast<T*>(a.dst);
  T* cst = static_cast<T*>(a.conv_state);

  // taps and bias of the CTA's channel vectors (vectors past nvec are not copied)
  for (int i = t; i < 32 * kWq; i += kConvThreads) {
    const int v = i / kWq, q = i - v * kWq;
    const int cvv = cb * 32 + v;
    if (cvv < nvec) {
      const float* src = q < V * K / 4 ? a.weight + (int64_t)cvv * V * K + 4 * q : a.bias + (int64_t)cvv * V + 4 * (q - V * K / 4);
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"((uint32_t)__cvta_generic_to_shared(&sm_w[q][v])), "l"(src));
    }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");  // the taps: group 1
  if (active) {
    {
      const bool fresh = seq_fresh(a.tab, s);
      const int64_t slot_base = (int64_t)seq_slot(a.tab, s) * H * a.conv_dim;
      // the H window rows before the tile (zeros for a fresh slot)
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
    }
#pragma unroll
    for (int r = 0; r < kConvRows; ++r) {
      if (r < nrows) {
        const uint32_t d = (uint32_t)__cvta_generic_to_shared(&sm_rows[H + r][t]);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(x + (int64_t)(row0 + q0 + r) * a.conv_dim + c0));
      }
    }
  }
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 1;\n" ::: "memory");
  __syncthreads();  // every thread's tap copies are in shared memory
  if (!active) return;
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  __syncwarp();  // this warp's rows are in shared memory

  float w[K][V], b[V];
#pragma unroll
  for (int q = 0; q < V * K / 4; ++q) {
    const float4 f = sm_w[q][lane];
    const float e[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) w[(4 * q + i) % K][(4 * q + i) / K] = e[i];
  }
#pragma unroll
  for (int q = 0; q < V / 4; ++q) {
    const float4 f = sm_w[V * K / 4 + q][lane];
    b[4 * q] = f.x; b[4 * q + 1] = f.y; b[4 * q + 2] = f.z; b[4 * q + 3] = f.w;
  }
  // taps and bias as channel pairs
  P2 w2[K][V / 2], b2[V / 2];
#pragma unroll
  for (int j = 0; j < V / 2; ++j) {
    b2[j] = p2(b[2 * j], b[2 * j + 1]);
#pragma unroll
    for (int k = 0; k < K; ++k) w2[k][j] = p2(w[k][2 * j], w[k][2 * j + 1]);
  }

  // window row i < H of this tile: win[i * kConvThreads]
  const uint4* win = &sm_rows[0][t];
  // tile row r: silu(bias + sum_k w[:, k] u[r + k]), each tap unpacked from smem
#pragma unroll
  for (int r = 0; r < kConvRows; ++r) {
    if (r < nrows) {
      P2 acc2[V / 2];
#pragma unroll
      for (int j = 0; j < V / 2; ++j) acc2[j] = b2[j];
#pragma unroll
      for (int k = 0; k < K; ++k) {  // taps in order, one rounding each (fma of each lane)
        float u[V];
        const uint4* src = r + k < H ? win + (r + k) * kConvThreads : &sm_rows[r + k][t];
        Vec16<T>::load(reinterpret_cast<const T*>(src), u);
#pragma unroll
        for (int j = 0; j < V / 2; ++j) acc2[j] = p2fma(w2[k][j], p2(u[2 * j], u[2 * j + 1]), acc2[j]);
      }
      float acc[V];
#pragma unroll
      for (int j = 0; j < V / 2; ++j) p2split(silu2(acc2[j]), acc[2 * j], acc[2 * j + 1]);
      Vec16<T>::store(dst + (int64_t)(row0 + q0 + r) * a.conv_dim + c0, acc);
    }
  }

  // slot update by tile 0: new history = u[T .. T + H - 1] (bit copies)
  if (local_tile == 0) {
    const bool fresh = seq_fresh(a.tab, s);
    const int64_t slot_base = (int64_t)seq_slot(a.tab, s) * H * a.conv_dim;
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
  const int ntiles = a.tab.tile[a.tab.n];
  if (ntiles == 0 || nvec == 0) return cudaSuccess;
  const int64_t nblocks = (int64_t)((ntiles + kConvTilesPerCta - 1) / kConvTilesPerCta) * ((nvec + 31) / 32);
  if (nblocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)nblocks);
  // three CTAs of up to 74 KB static shared memory per SM (14-row tiles)
  cudaError_t e = cudaFuncSetAttribute(conv1d_silu_kernel<T, K>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                       (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  conv1d_silu_kernel<T, K><<<grid, kConvThreads, 0, st>>>(a);
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
