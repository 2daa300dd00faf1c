// The projections around the recurrent path, as tcgen05 GEMMs:
//   in_proj   [rows, d_model] x W_in[d_in_proj, d_model]^T, the output columns split
//             into z [rows, d_inner], xBC [rows, conv_dim] and dt [rows, heads] by the
//             epilogue (gllm PR #85 "feat(backend): Mamba2 ops, with CPU reference
//             implementations", "Ops": the model splits in_proj into z, xBC and dt, so
//             no split op is needed; here the split is the GEMM's store)
//   out_proj  [rows, d_inner] x W_out[d_model, d_inner]^T -> [rows, d_model]
// bf16 operands, fp32 accumulation in tensor memory, bf16 output rounded once.
//
// One persistent CTA per SM walks 128 x 256 output tiles, N fastest, so the CTAs
// working at one time share the same rows of the activations in L2. Each CTA loads
// its own A and B blocks from global memory (no load is shared between CTAs).
// Roles:
//   warp 0      TMA loads of the A (128 x 64) and B (256 x 64) k-blocks, 4 stages
//   warp 1      tcgen05.mma issue (one thread), M=128 N=256 K=16, into one of two
//               256-column accumulators, so the epilogue of a tile overlaps the
//               next tile's products
//   warps 2-5   epilogue: tensor memory -> registers -> bf16 -> global, each
//               thread one output row, 16-byte stores, rows and columns past the
//               matrix skipped
// A stage is refilled once the products have read it (the MMA commit arrives on the
// stage's barrier). Every mbarrier wait is bounded; a timeout stops every role,
// drains what was issued, frees tensor memory and counts the CTA in
// g_gemm_timeouts.
#include <cuda.h>

#include <algorithm>
#include <cstring>

#include "common.cuh"

namespace mamba2 {

__device__ unsigned int g_gemm_timeouts = 0;

namespace {

#include "tc.cuh"

constexpr int GBM = 128, GBN = 256, GBK = 64, kGStages = 4;
constexpr int kGThreads = 6 * 32;
constexpr uint32_t kGTileA = GBM * GBK * 2;  // 16 KB
constexpr uint32_t kGTileB = GBN * GBK * 2;  // 32 KB
constexpr uint32_t kGStage = kGTileA + kGTileB;
constexpr uint32_t kGOffBar = kGStages * kGStage;
enum GemmBar : int { kGFull = 0, kGEmpty = kGStages, kGAccFull = 2 * kGStages, kGAccEmpty = 2 * kGStages + 2,
                     kGDone = 2 * kGStages + 4, kGNumBars = 2 * kGStages + 5 };
constexpr uint32_t kGOffMisc = kGOffBar + 8 * kGNumBars;  // TMEM base, abort flag
constexpr uint32_t kGemmSmem = kGOffMisc + 16 + 1024;
static_assert(kGemmSmem <= 232448, "GEMM shared memory plan exceeds 227 KB");

// 32 consecutive fp32 columns of this thread's lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t bf16x2(uint32_t lo, uint32_t hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
  return *reinterpret_cast<uint32_t*>(&v);
}

__global__ void __launch_bounds__(kGThreads, 1)
gemm_tc_kernel(const __grid_constant__ GemmArgs g, const __grid_constant__ CUtensorMap tma,
               const __grid_constant__ CUtensorMap tmb) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw_base = su32(smem_raw);
  unsigned char* smem = smem_raw + (((raw_base + 1023u) & ~1023u) - raw_base);
  const uint32_t sbase = su32(smem);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kGOffMisc);
  volatile uint32_t* s_abort = reinterpret_cast<volatile uint32_t*>(smem + kGOffMisc + 4);
  auto bar = [&](int id) { return sbase + kGOffBar + 8u * (uint32_t)id; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int tiles_m = (g.M + GBM - 1) / GBM, tiles_n = (g.N + GBN - 1) / GBN;
  const int tiles = tiles_m * tiles_n;
  const int kblocks = (g.K + GBK - 1) / GBK;
  const int cta = (int)blockIdx.x, ncta = (int)gridDim.x;
  // this CTA's tiles: cta, + ncta, ... (N fastest)
  const int my_tiles = cta < tiles ? (tiles - 1 - cta) / ncta + 1 : 0;
  auto tile_m0 = [&](int t) { return ((cta + t * ncta) / tiles_n) * GBM; };
  auto tile_n0 = [&](int t) { return ((cta + t * ncta) % tiles_n) * GBN; };

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" :: "r"(su32(s_tmem)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (threadIdx.x == 32) {
    for (int s = 0; s < kGStages; ++s) {
      mbar_init(bar(kGFull + s), 1);
      mbar_init(bar(kGEmpty + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(kGAccFull + b), 1);
      mbar_init(bar(kGAccEmpty + b), 4);  // one arrival per epilogue warp
    }
    mbar_init(bar(kGDone), 1);
    *s_abort = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (warp == 0) {
    // =================== TMA producer
    int it = 0, issued = 0;
    bool ok = true;
    for (int t = 0; t < my_tiles && ok; ++t) {
      const int m0 = tile_m0(t), n0 = tile_n0(t);
      for (int kb = 0; kb < kblocks; ++kb, ++it) {
        const int s = it % kGStages;
        if (it >= kGStages && !warp_wait(bar(kGEmpty + s), (uint32_t)(((it / kGStages) - 1) & 1), s_abort)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t dst = sbase + (uint32_t)s * kGStage;
          mbar_expect_tx(bar(kGFull + s), kGStage);  // A + B
          tma_load_2d(dst, &tma, kb * GBK, m0, bar(kGFull + s));
          tma_load_2d(dst + kGTileA, &tmb, kb * GBK, n0, bar(kGFull + s));
        }
        __syncwarp();
        issued = it + 1;
      }
    }
    // on an abort, let the loads in flight land before the CTA exits
    if (lane == 0 && *s_abort)
      for (int i = max(0, issued - kGStages); i < issued; ++i)
        drain_bar(bar(kGFull + i % kGStages), (uint32_t)((i / kGStages) & 1));
  } else if (warp == 1) {
    // =================== MMA issuer
    if (lane == 0) {
      const uint32_t id = idesc128(GBN, 0, 0);
      int it = 0;
      bool ok = true;
      for (int t = 0; t < my_tiles && ok; ++t) {
        const int buf = t & 1;
        if (t >= 2 && !wait_bar(bar(kGAccEmpty + buf), (uint32_t)(((t >> 1) - 1) & 1), s_abort)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * GBN);
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const int s = it % kGStages;
          if (!wait_bar(bar(kGFull + s), (uint32_t)((it / kGStages) & 1), s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = sbase + (uint32_t)s * kGStage;
          const uint64_t ad = sdesc(a0, 16, 1024), bd = sdesc(a0 + kGTileA, 16, 1024);
#pragma unroll
          for (int k = 0; k < GBK / 16; ++k)  // 16 bf16 = 32 bytes along the 128-byte swizzled row
            mma_ss(d, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), id, (kb > 0 || k > 0) ? 1u : 0u);
          mma_commit(bar(kGEmpty + s));  // stage s may be refilled once read
        }
        if (!ok) break;
        mma_commit(bar(kGAccFull + buf));
      }
      // every product issued (a whole tile's or, after an abort, part of one) completes
      // before the teardown frees tensor memory
      mma_commit(bar(kGDone));
      drain_bar(bar(kGDone), 0u);
    }
    __syncwarp();
  } else {
    // =================== epilogue: warp w reads lanes 32 (w % 4) .. + 31
    const int q = warp & 3;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    for (int t = 0; t < my_tiles; ++t) {
      const int buf = t & 1;
      if (!warp_wait(bar(kGAccFull + buf), (uint32_t)((t >> 1) & 1), s_abort)) break;
      tc_fence_after();
      const int m0 = tile_m0(t), n0 = tile_n0(t);
      const int64_t row = (int64_t)m0 + q * 32 + lane;
#pragma unroll 1
      for (int c = 0; c < GBN; c += 32) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + (uint32_t)(buf * GBN + c), r);
        if (row >= g.M) continue;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int col = n0 + c + 8 * v;  // 8 output columns, all in one destination
          if (col >= g.N) break;
          int seg = 0;
          while (seg + 1 < g.nseg && col >= g.seg_end[seg]) ++seg;
          const int c0 = col - (seg > 0 ? g.seg_end[seg - 1] : 0);
          uint4 o;
          o.x = bf16x2(r[8 * v + 0], r[8 * v + 1]);
          o.y = bf16x2(r[8 * v + 2], r[8 * v + 3]);
          o.z = bf16x2(r[8 * v + 4], r[8 * v + 5]);
          o.w = bf16x2(r[8 * v + 6], r[8 * v + 7]);
          __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(g.dst[seg]) + row * g.ld[seg] + c0;
          *reinterpret_cast<uint4*>(dst) = o;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kGAccEmpty + buf));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *s_abort) atomicAdd(&g_gemm_timeouts, 1u);
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" :: "r"(tmem));
}

using Encode = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*, const cuuint64_t*,
                            const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                            CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

Encode encode_fn() {
  static Encode fn = []() -> Encode {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<Encode>(p);
  }();
  return fn;
}

// [rows][K] bf16, K contiguous: boxes of 64 (K) x box_rows, 128-byte swizzle, zeros past the edges
bool make_kmajor_map(CUtensorMap* tm, const void* base, int64_t rows, int64_t K, int box_rows) {
  const Encode enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)GBK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

unsigned int read_gemm_timeouts() {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_gemm_timeouts, sizeof v) != cudaSuccess) return 0xffffffffu;
  return v;
}

cudaError_t launch_gemm_tc(const GemmArgs& g, const void* A, const void* B, cudaStream_t st) {
  if (g.M == 0 || g.N == 0) return cudaSuccess;
  CUtensorMap tma, tmb;
  std::memset(&tma, 0, sizeof tma);
  std::memset(&tmb, 0, sizeof tmb);
  if (!make_kmajor_map(&tma, A, g.M, g.K, GBM) || !make_kmajor_map(&tmb, B, g.N, g.K, GBN))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGemmSmem);
  if (e != cudaSuccess) return e;
  const int tiles = ((g.M + GBM - 1) / GBM) * ((g.N + GBN - 1) / GBN);
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // one CTA per SM (the shared-memory plan admits one), at most one per tile
  const int grid = std::max(1, std::min(tiles, sms));
  gemm_tc_kernel<<<grid, kGThreads, kGemmSmem, st>>>(g, tma, tmb);
  return cudaGetLastError();
}

}  // namespace mamba2
