// Mamba-3 SISO varlen forward on the tcgen05 tensor cores, head dim 64 x
// state 128 (the frozen shapes of the page "Mamba-3 SISO Long-Ragged
// Multi-Chunk Joint States Full VJP": one Q/K head of width 128 serving every
// value head of width 64, up to 64 rotary pairs).
//
// Semantics (that page, "What You Have", steps 1-7), per sequence and head,
// token by token:
//   phi_t = (sum_{s<=t} tanh(angles_s) pi dt_s) mod 2 pi          (per rotary pair)
//   q^_t, k^_t = pairs (2i, 2i+1), i < R, of q_t + q_bias, k_t + k_bias rotated by phi_t[i]
//   p = sigmoid(trap), sg_t = dt_{t+1} (1 - p_{t+1}) (0 at the last token),
//   scale_t = dt_t p_t + sg_t
//   h_t = exp(adt_t) h_{t-1} + scale_t v_t (x) k^_t
//   y_t = h_t q^_t + d v_t - (q^_t . k^_t) sg_t v_t,   out_t = y_t z_t sigmoid(z_t)
// and the final angle, state, rotated k and v of the sequence's last token.
//
// Chunked form (Q = 128 tokens, S_t = adt_0 + ... + adt_t within the chunk):
//   y_t = exp(S_t) q^_t . H_in + sum_{s<=t} M[t][s] v_s + d v_t
//   M[t][s] = (q^_t . k^_s) exp(S_t - S_s) scale_s    (s < t)
//   M[t][t] = (q^_t . k^_t) dt_t p_t                   (the correction removes sg_t)
//   H_out   = exp(S_end) H_in + sum_s exp(S_end - S_s) scale_s v_s (x) k^_s
// The diagonal's q^ . k^ comes from the fp32 rotated values (the largest
// entries of y are there), the rest from the tensor cores.
//
// One CTA of 16 warps per (sequence, head), chunk after chunk:
//   1. per-token scalars (S in log2 units, scale, dt p), the cumulative angles
//      (one thread per rotary pair and block of 8 tokens), q^ and k^ as fp16
//      [token][n] tiles (128-byte swizzle) and the exact diagonal q^ . k^;
//      v as fp16 and v o w (w_s = exp(S_end - S_s) scale_s) as fp16 tiles;
//   2. CB = Q^ K^T (N = 128), Yoff = Q^ H^T (N = 64), dH^T = K^T (v o w)
//      (N = 64, lane = state row n), K = 128 each;
//   3. M written to TMEM as fp16 (the A operand of the next product), and the
//      state H^T = exp(S_end) H^T + dH^T in fp32 registers (lane n, 16 columns
//      per thread), its fp16 copy to shared memory for the next chunk's Yoff;
//   4. Yd = M V (A from TMEM), then out = (Yd + exp(S_t) Yoff + d v) silu(z).
// Global memory reaches the CTA only through asynchronous copies, issued by one
// thread: the next chunk's raw q and k rows and angles (bulk copies) and, when the
// head count makes its rows 16-byte multiples, its per-token dt, adt and trap (TMA
// boxes of the 16-byte column group holding the head, 129 rows for the next-token
// terms) land while the current chunk runs; v and z pass through one 16 KB TMA
// staging tile (v of the next chunk during the output, z during the products).
// Strided per-thread loads of [rows, heads] columns, 32 lines a warp instruction,
// held the load pipe for thousands of cycles a chunk, and every warp behind them.
// fp16 operands (11 significant bits) keep the worst y error about a tenth of
// the bf16 output's own rounding. fp16 holds magnitudes up to 65 504: a larger
// operand converts to inf, which reaches the y it feeds or the state (inf, or
// NaN through inf * 0). Each thread sums the y it stores and its final state
// entries; a CTA whose sums are not finite recomputes that (sequence, head) token
// by token in fp32 (correct, slow; no workload here comes near it). An operand
// that overflows where no product uses it (q^ of a chunk's first token before any
// state exists) changes nothing and is not caught, which is also correct.
// Every wait is bounded: on a timeout the CTA records it in a device counter
// (mamba2_device_timeouts), drains what it issued, frees its TMEM and returns.
#include <cuda.h>

#include <cstring>

#include <type_traits>

#include "common.cuh"

namespace mamba2 {

__device__ unsigned int g_m3_timeouts = 0;

namespace {

#include "tc.cuh"

constexpr int kQ = 128;  // tokens per chunk
constexpr int kP = 64;   // value head width
constexpr int kN = 128;  // Q/K width (state columns)
constexpr int kThreads = 512;
constexpr float kTwoPi = 6.283185307179586f;
constexpr float kPiF = 3.14159265358979f;
constexpr float kLog2e = 1.4426950408889634f;

// ---- shared memory (operand tiles 1024-byte aligned)
constexpr uint32_t kTileQK = kQ * kN * 2;  // 32 KB [token][n] fp16
constexpr uint32_t kTileV = kQ * kP * 2;   // 16 KB [token][p] fp16
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kTileQK;
constexpr uint32_t kOffV = kOffK + kTileQK;
constexpr uint32_t kOffVW = kOffV + kTileV;
constexpr uint32_t kOffHT = kOffVW + kTileV;  // H^T fp16 [n][p]
// the chunk's raw inputs, row-major as in memory (copied one chunk ahead)
constexpr uint32_t kOffRawQ = kOffHT + kN * kP * 2;  // [128][128] bf16
constexpr uint32_t kOffRawK = kOffRawQ + kQ * kN * 2;
constexpr uint32_t kOffRawA = kOffRawK + kQ * kN * 2;  // [128][rot_dim] bf16, rot_dim <= 64
// v, then z, of the chunk's rows for this head ([128][64] bf16, 128-byte swizzle,
// by TMA): v lands while the previous chunk finishes, z while the products run
constexpr uint32_t kOffVZ = kOffRawA + kQ * 64 * 2;
// the chunk's per-token scalars of this head and the next token's (rows rb ..
// rb + 128) by TMA with the raw rows: dt and adt as [129][4] f32, trap as [129][8]
// bf16 (the 16-byte column group holding head h)
constexpr uint32_t kScBox = (kQ + 1) * 16;               // bytes of one scalar box
constexpr uint32_t kScSlot = (kScBox + 127) / 128 * 128;  // its 128-byte aligned slot
constexpr uint32_t kOffSc = kOffVZ + kQ * kP * 2;
constexpr uint32_t kOffF = kOffSc + 3 * kScSlot;
// float offsets inside the scalar block
constexpr int kFS = 0;          // [128] cumulative log2 decay S
constexpr int kFW = 128;        // [128] scale
constexpr int kFDD = 256;       // [128] dt p
constexpr int kFDG = 384;       // [128] q^ . k^ of each token (fp32)
constexpr int kFWS = 512;       // [8] warp sums of the decay scan (warps 0-3)
constexpr int kFAP = 520;       // [16][64] angle sums per block of 8 tokens
constexpr int kFCar = 1544;     // [2][64] angle carried into chunk c (buffer c % 2)
constexpr int kFDT = 1672;      // [128] dt of the head
constexpr int kNumF = 1800;
constexpr uint32_t kOffBar = kOffF + kNumF * 4;  // mbarriers: products, Yd, raw q/k copy, v/z copy
constexpr uint32_t kOffMisc = kOffBar + 32;      // TMEM base, abort flag, fp16 range flag
constexpr uint32_t kSmemUsed = kOffMisc + 16;
constexpr uint32_t kSmem = kSmemUsed + 1024;     // + alignment slack
static_assert(kSmem <= 232448, "shared memory plan exceeds 227 KB");
static_assert(kOffBar % 8 == 0, "mbarrier alignment");
static_assert(kOffVZ % 1024 == 0, "the swizzled v/z staging tile needs a 1024-byte aligned offset");

// ---- TMEM columns (128 lanes)
constexpr uint32_t kColCB = 0;    // [0,128)  CB = Q^ K^T, column = token s
constexpr uint32_t kColYo = 128;  // [128,192) Q^ H^T, column = p
constexpr uint32_t kColDH = 192;  // [192,256) K^T (v o w), lane = n, column = p
constexpr uint32_t kColM = 256;   // [256,320) M as fp16 pairs, k-step s at 8 s
constexpr uint32_t kColYd = 320;  // [320,384) M V, column = p

// byte offset of element (r, c) in a [128][cols] 16-bit tile, 128-byte
// swizzle, 64-column blocks of 128 rows each
__device__ __forceinline__ uint32_t toff(int r, int c) {
  return (uint32_t)((c >> 6) * kQ * 128 + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) + (c & 7) * 2);
}

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// fp16 pair (lo in the low half); a value beyond the fp16 range becomes inf, and
// inf (or inf * 0) reaches y or the state it feeds: caught there
__device__ __forceinline__ uint32_t h2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + __expf(-x)); }
__device__ __forceinline__ float bf(const __nv_bfloat16* p, int64_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ float f16lo(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w & 0xffffu))); }
__device__ __forceinline__ float f16hi(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w >> 16))); }

__device__ __forceinline__ float wrap2pi(float x) { return x - kTwoPi * floorf(x * (1.0f / kTwoPi)); }
// tanh(x) = 1 - 2 / (exp(2x) + 1), branch-free (absolute error a few 1e-7; |x|
// clamped at 15, where tanh is 1 in fp32)
__device__ __forceinline__ float tanh_fast(float x) {
  x = fminf(fmaxf(x, -15.0f), 15.0f);
  return 1.0f - __fdividef(2.0f, 1.0f + __expf(2.0f * x));
}
// (sin, cos) of phi in [0, 2 pi), taken at phi - 2 pi above pi so the hardware
// approximation works in [-pi, pi] (absolute error about 1e-6)
__device__ __forceinline__ void sincos_wrapped(float phi, float& sn, float& cs) {
  __sincosf(phi > kPiF ? phi - kTwoPi : phi, &sn, &cs);
}

// one contiguous global -> shared copy (16-byte aligned ends), completing on `bar`
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(valid ? 4 : 0));
}

__device__ __forceinline__ float warp_incl(float v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  return v;
}

struct Item {
  int s, h, row0, T;
};
__device__ __forceinline__ Item item_at(const Mamba3Args& a, int i) {
  Item it;
  it.s = a.order[i / a.heads];
  it.h = i - (i / a.heads) * a.heads;
  it.row0 = a.cu[it.s];
  it.T = a.cu[it.s + 1] - it.row0;
  return it;
}

// One (sequence, head) token by token in fp32 (512 threads; thread tid owns
// state row p = tid / 8, columns n = 16 (tid % 8) .. + 15). Shared scratch:
// q^, k^ [128], v [64], cos/sin [64 each], scalars.
__device__ __noinline__ void serial_item(const Mamba3Args& a, const Item& it, float* scratch) {
  const int tid = threadIdx.x, H = a.heads, R = a.rot_dim;
  float* qh = scratch;
  float* kh = scratch + 128;
  float* vv = scratch + 256;
  float* cs = scratch + 320;
  float* sn = scratch + 384;
  float* sc = scratch + 448;  // decay, scale, sg
  const int p = tid >> 3, n0 = (tid & 7) * 16;
  float hreg[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) hreg[e] = 0.0f;
  float cum = 0.0f;
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
  const __nv_bfloat16* k = static_cast<const __nv_bfloat16*>(a.k);
  const __nv_bfloat16* v = static_cast<const __nv_bfloat16*>(a.v);
  const __nv_bfloat16* z = static_cast<const __nv_bfloat16*>(a.z);
  const __nv_bfloat16* trap = static_cast<const __nv_bfloat16*>(a.trap);
  const __nv_bfloat16* ang = static_cast<const __nv_bfloat16*>(a.angles);
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
  const float dh = a.d[it.h];
  for (int t = 0; t < it.T; ++t) {
    const int64_t r = it.row0 + t;
    if (tid < R) {
      cum = wrap2pi(cum + tanhf(bf(ang, r * R + tid)) * kPiF * a.dt[r * H + it.h]);
      float s_, c_;
      sincosf(cum, &s_, &c_);
      cs[tid] = c_;
      sn[tid] = s_;
    }
    if (tid >= 64 && tid < 128) vv[tid - 64] = bf(v, (r * H + it.h) * kP + tid - 64);
    if (tid == 128) {
      const float dtv = a.dt[r * H + it.h];
      const float pp = sigmoidf_(bf(trap, r * H + it.h));
      float sg = 0.0f;
      if (t + 1 < it.T) sg = a.dt[(r + 1) * H + it.h] * (1.0f - sigmoidf_(bf(trap, (r + 1) * H + it.h)));
      sc[0] = expf(a.adt[r * H + it.h]);
      sc[1] = dtv * pp + sg;
      sc[2] = sg;
    }
    __syncthreads();
    if (tid < 64) {
      const int c0 = 2 * tid;
      const float q0 = bf(q, r * kN + c0) + a.q_bias[it.h * kN + c0], q1 = bf(q, r * kN + c0 + 1) + a.q_bias[it.h * kN + c0 + 1];
      const float k0 = bf(k, r * kN + c0) + a.k_bias[it.h * kN + c0], k1 = bf(k, r * kN + c0 + 1) + a.k_bias[it.h * kN + c0 + 1];
      const float c_ = tid < R ? cs[tid] : 1.0f, s_ = tid < R ? sn[tid] : 0.0f;
      qh[c0] = c_ * q0 - s_ * q1;
      qh[c0 + 1] = s_ * q0 + c_ * q1;
      kh[c0] = c_ * k0 - s_ * k1;
      kh[c0 + 1] = s_ * k0 + c_ * k1;
    }
    __syncthreads();
    const float dec = sc[0], scl = sc[1], sg = sc[2], vp = vv[p];
    float acc = 0.0f;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float kv = kh[n0 + e] * vp;
      hreg[e] = fmaf(dec, hreg[e], scl * kv);
      acc = fmaf(hreg[e] - sg * kv, qh[n0 + e], acc);
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    acc += __shfl_xor_sync(0xffffffffu, acc, 4);
    if ((tid & 7) == 0) {
      const float zz = bf(z, (r * H + it.h) * kP + p);
      out[(r * H + it.h) * kP + p] = __float2bfloat16_rn(fmaf(dh, vp, acc) * silu_f(zz));
    }
    __syncthreads();
  }
  // final states (zeros for an empty sequence)
  const int64_t sh = (int64_t)it.s * H + it.h;
#pragma unroll
  for (int e = 0; e < 16; ++e) a.final_ssm[(sh * kP + p) * kN + n0 + e] = hreg[e];
  if (tid < 128) a.final_k[sh * kN + tid] = it.T > 0 ? kh[tid] : 0.0f;
  if (tid >= 128 && tid < 128 + kP)
    static_cast<__nv_bfloat16*>(a.final_v)[sh * kP + tid - 128] = __float2bfloat16_rn(it.T > 0 ? vv[tid - 128] : 0.0f);
  if (tid < R) static_cast<__nv_bfloat16*>(a.final_angle)[sh * R + tid] = __float2bfloat16_rn(cum);
}

__global__ void __launch_bounds__(kThreads, 1)
m3_fwd_kernel(const __grid_constant__ Mamba3Args a, const __grid_constant__ CUtensorMap tmv,
              const __grid_constant__ CUtensorMap tmz, const __grid_constant__ CUtensorMap tmdt,
              const __grid_constant__ CUtensorMap tmadt, const __grid_constant__ CUtensorMap tmtr, const int sc_tma) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = su32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  unsigned char* smem = smem_raw + (sb - raw);
  float* F = reinterpret_cast<float*>(smem + kOffF);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile uint32_t* s_abort = reinterpret_cast<volatile uint32_t*>(smem + kOffMisc + 4);
  volatile uint32_t* s_range = reinterpret_cast<volatile uint32_t*>(smem + kOffMisc + 8);
  const uint32_t bar0 = sb + kOffBar, bar1 = sb + kOffBar + 8, bar2 = sb + kOffBar + 16, bar3 = sb + kOffBar + 24;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.heads, R = a.rot_dim;

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" :: "r"(su32(s_tmem)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 32) {
    mbar_init(bar0, 1);
    mbar_init(bar1, 1);
    mbar_init(bar2, 1);
    mbar_init(bar3, 1);
    *s_abort = 0u;
    *s_range = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
  const __nv_bfloat16* k = static_cast<const __nv_bfloat16*>(a.k);
  const __nv_bfloat16* trap = static_cast<const __nv_bfloat16*>(a.trap);
  const __nv_bfloat16* ang = static_cast<const __nv_bfloat16*>(a.angles);
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);

  // TMEM lane quarter and column quarter of this thread's row (row = TMEM lane)
  const int row = 32 * (warp & 3) + lane, cq = warp >> 2;
  const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
  // rotation role: pairs lane and lane + 32 (columns 2 pair, 2 pair + 1) of tokens
  // 8 warp .. 8 warp + 7 (one rotated and one plain pair each when rot_dim = 32)
  const int pA = lane, pB = lane + 32;
  uint32_t n_bar0 = 0, n_bar1 = 0, n_bar2 = 0, n_bar3 = 0;  // phases waited on
  uint32_t n_pref = 0, n_vz = 0;                             // raw and v/z copies issued
  // the asynchronous copies are issued by the last warp's lane 0, which waits the
  // least at the barriers those copies sit before (thread 0 issues the products)
  const bool copier = tid == kThreads - 32;
  // v or z rows [rb, rb + 128) of head h into the staging tile (rows past the
  // tensor read as zero, rows of the next sequence are masked where used)
  auto copy_vz = [&](const CUtensorMap* tm, int64_t rb, int h) {
    ++n_vz;
    if (copier) {
      fence_async_smem();  // the staging tile's previous reads come first
      mbar_expect_tx(bar3, kQ * kP * 2);
      tma_load_2d(sb + kOffVZ, tm, h * kP, (int)rb, bar3);
    }
  };
  bool aborted = false;

  const int items = a.nseq * H;
  for (int round = 0;; ++round) {
    const int i0 = round * (int)gridDim.x;
    if (i0 >= items) break;
    const int item = i0 + ((round & 1) ? (int)gridDim.x - 1 - (int)blockIdx.x : (int)blockIdx.x);
    if (item >= items) continue;
    const Item it = item_at(a, item);
    const int64_t sh = (int64_t)it.s * H + it.h;
    const int nch = (it.T + kQ - 1) / kQ;
    float hs[16];  // H^T[row][16 cq + e]
#pragma unroll
    for (int e = 0; e < 16; ++e) hs[e] = 0.0f;
    if (tid < 64) F[kFCar + tid] = 0.0f;
    const float2 qbA = *reinterpret_cast<const float2*>(a.q_bias + (int64_t)it.h * kN + 2 * pA);
    const float2 qbB = *reinterpret_cast<const float2*>(a.q_bias + (int64_t)it.h * kN + 2 * pB);
    const float2 kbA = *reinterpret_cast<const float2*>(a.k_bias + (int64_t)it.h * kN + 2 * pA);
    const float2 kbB = *reinterpret_cast<const float2*>(a.k_bias + (int64_t)it.h * kN + 2 * pB);
    const float dh = a.d[it.h];
    // sum of every stored y and of the final state: not finite iff an fp16 operand
    // of the products overflowed (or an input was not finite)
    float fsum = 0.f;

    // raw q and k rows of the chunk starting at row rb: one bulk copy each (rows
    // past the run keep stale values, masked where they are read);
    // angles likewise, or as 4-byte cp.async pieces (rows past the run zero-filled)
    // when rot_dim is even but not a multiple of 8
    // (rows of rot_dim a multiple of 8 are 16-byte multiples: the angles then come
    // as one bulk copy too)
    const bool ang_bulk = R > 0 && (R & 7) == 0;
    auto prefetch = [&](int64_t rb, int len) {
      ++n_pref;
      if (copier) {
        fence_async_smem();  // the previous chunk's reads of the staging rows come first
        const uint32_t bytes = (uint32_t)len * kN * 2, abytes = ang_bulk ? (uint32_t)(len * R * 2) : 0u;
        mbar_expect_tx(bar2, 2 * bytes + abytes + (sc_tma ? 3 * kScBox : 0u));
        bulk_g2s(sb + kOffRawQ, q + rb * kN, bytes, bar2);
        bulk_g2s(sb + kOffRawK, k + rb * kN, bytes, bar2);
        if (ang_bulk) bulk_g2s(sb + kOffRawA, ang + rb * R, abytes, bar2);
        if (sc_tma) {
          tma_load_2d(sb + kOffSc, &tmdt, it.h & ~3, (int)rb, bar2);
          tma_load_2d(sb + kOffSc + kScSlot, &tmadt, it.h & ~3, (int)rb, bar2);
          tma_load_2d(sb + kOffSc + 2 * kScSlot, &tmtr, it.h & ~7, (int)rb, bar2);
        }
      }
      if (!ang_bulk && R > 0 && (R & 1) == 0) {
        const int pieces = R >> 1;
        for (int i = tid; i < kQ * pieces; i += kThreads) {
          const int t = i / pieces, pc = i - t * pieces;
          const bool ok = t < len;
          cp_async4(sb + kOffRawA + (uint32_t)(t * 2 * R + 4 * pc), ang + (ok ? rb + t : rb) * R + 2 * pc, ok);
        }
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    };
    if (nch > 0) {
      prefetch(it.row0, min(kQ, it.T));
      copy_vz(&tmv, it.row0, it.h);
    }
    // raw per-token scalars of the chunk at row rb (thread tid < 128: token tid and
    // the next one), loaded a chunk ahead, when they do not come by TMA (a head count
    // whose rows are not 16-byte multiples). Each load reads a row of the sequence
    // (past its end, the last one) and is masked where it is used.
    const int64_t seq_end = it.row0 + it.T;
    float r_dt = 0.f, r_tr = 0.f, r_adt = 0.f, r_dtn = 0.f, r_trn = 0.f;
    auto load_scalars = [&](int64_t rb, int len) {
      if (tid < kQ) {
        const int64_t r = rb + min(tid, len - 1), rn = min(r + 1, seq_end - 1);
        r_dt = a.dt[r * H + it.h];
        r_tr = bf(trap, r * H + it.h);
        r_adt = a.adt[r * H + it.h];
        r_dtn = a.dt[rn * H + it.h];
        r_trn = bf(trap, rn * H + it.h);
      }
    };
    if (nch > 0 && !sc_tma) load_scalars(it.row0, min(kQ, it.T));

    for (int c = 0; c < nch; ++c) {
      const int len = min(kQ, it.T - c * kQ);
      const int64_t rb = it.row0 + (int64_t)c * kQ;  // first row of the chunk
      const bool last_chunk = c == nch - 1;

      const bool in_run = row < len;
      const int64_t off = ((rb + row) * H + it.h) * kP + 16 * cq;
      if ((R & 1) != 0) {  // odd rot_dim: angles element by element
        __nv_bfloat16* ra = reinterpret_cast<__nv_bfloat16*>(smem + kOffRawA);
        for (int i = tid; i < kQ * R; i += kThreads) {
          const int t = i / R;
          ra[i] = t < len ? ang[(rb + t) * R + (i - t * R)] : __float2bfloat16_rn(0.f);
        }
      }
      asm volatile("cp.async.wait_group 0;" ::: "memory");
      if (wait_bar(bar2, n_bar2 & 1u, s_abort))
        ++n_bar2;
      else
        *s_abort = 1u;
      // ---- per-token scalars (warps 0-3: token tid)
      float a2 = 0.f, incl = 0.f;
      if (tid < kQ) {
        if (sc_tma) {
          const int cf = it.h & 3, cb = it.h & 7;
          const float* sdt = reinterpret_cast<const float*>(smem + kOffSc);
          const float* sadt = reinterpret_cast<const float*>(smem + kOffSc + kScSlot);
          const __nv_bfloat16* str = reinterpret_cast<const __nv_bfloat16*>(smem + kOffSc + 2 * kScSlot);
          r_dt = sdt[4 * tid + cf];
          r_dtn = sdt[4 * (tid + 1) + cf];
          r_adt = sadt[4 * tid + cf];
          r_tr = __bfloat162float(str[8 * tid + cb]);
          r_trn = __bfloat162float(str[8 * (tid + 1) + cb]);
        }
        float scl = 0.f, dtp = 0.f, dtv = 0.f;
        if (tid < len) {
          const float sg = rb + tid + 1 < seq_end ? r_dtn * (1.0f - sigmoidf_(r_trn)) : 0.f;
          a2 = r_adt * kLog2e;
          dtp = r_dt * sigmoidf_(r_tr);
          scl = dtp + sg;
          dtv = r_dt;
        }
        F[kFW + tid] = scl;
        F[kFDD + tid] = dtp;
        F[kFDT + tid] = dtv;
        incl = warp_incl(a2, lane);
        if (lane == 31) F[kFWS + warp] = incl;
      }
      __syncthreads();  // (A) raw chunk, scalars, warp sums
      if (*s_abort) {
        aborted = true;
        break;
      }
      if (tid < kQ) {
        float before = 0.f;  // decay of the warps' earlier tokens
        for (int w = 0; w < warp; ++w) before += F[kFWS + w];
        F[kFS + tid] = incl + before;
      }
      // ---- angle increments of this thread's rotated pairs over its 8 tokens
      const bool rotA = pA < R, rotB = pB < R;
      float incA[8], incB[8];
      {
        const __nv_bfloat16* ra = reinterpret_cast<const __nv_bfloat16*>(smem + kOffRawA);
        float partA = 0.f, partB = 0.f;
        const int iA = rotA ? pA : 0, iB = rotB ? pB : 0;  // in-range columns (R may be 0: rows are then empty)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int t = 8 * warp + e;
          const float pd = kPiF * F[kFDT + t];  // 0 past the run
          const float xa = tanh_fast(__bfloat162float(ra[t * R + iA])) * pd;
          incA[e] = rotA ? xa : 0.f;
          partA += incA[e];
          incB[e] = 0.f;
          if (R > 32) {  // (uniform) some second pairs rotate
            const float xb = tanh_fast(__bfloat162float(ra[t * R + iB])) * pd;
            incB[e] = rotB ? xb : 0.f;
            partB += incB[e];
          }
        }
        F[kFAP + 64 * warp + pA] = partA;
        F[kFAP + 64 * warp + pB] = partB;
      }
      __syncthreads();  // (A2) angle block sums
      {
        float runA = F[kFCar + 64 * (c & 1) + pA], runB = F[kFCar + 64 * (c & 1) + pB];
        for (int j = 0; j < warp; ++j) {
          runA += F[kFAP + 64 * j + pA];
          runB += F[kFAP + 64 * j + pB];
        }
        float dv[8];
        auto rotate_rows = [&](auto b_rotates) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int t = 8 * warp + e;
          const bool live = t < len;
          runA += incA[e];  // increments are 0 past the run
          runB += incB[e];
          const float phA = wrap2pi(runA), phB = wrap2pi(runB);
          const uint32_t* rq = reinterpret_cast<const uint32_t*>(smem + kOffRawQ + t * 256);
          const uint32_t* rk = reinterpret_cast<const uint32_t*>(smem + kOffRawK + t * 256);
          // staging rows past the run hold stale bytes: read as zero
          const uint32_t qA = live ? rq[pA] : 0u, qB = live ? rq[pB] : 0u;
          const uint32_t kA = live ? rk[pA] : 0u, kB = live ? rk[pB] : 0u;
          float snA, csA, snB = 0.f, csB = 1.f;
          sincos_wrapped(phA, snA, csA);
          if (!rotA) { snA = 0.f; csA = 1.f; }
          if constexpr (decltype(b_rotates)::value) {
            sincos_wrapped(phB, snB, csB);
            if (!rotB) { snB = 0.f; csB = 1.f; }
          }
          const float qa0 = __uint_as_float(qA << 16) + qbA.x, qa1 = __uint_as_float(qA & 0xffff0000u) + qbA.y;
          const float ka0 = __uint_as_float(kA << 16) + kbA.x, ka1 = __uint_as_float(kA & 0xffff0000u) + kbA.y;
          const float qb0 = __uint_as_float(qB << 16) + qbB.x, qb1 = __uint_as_float(qB & 0xffff0000u) + qbB.y;
          const float kb0 = __uint_as_float(kB << 16) + kbB.x, kb1 = __uint_as_float(kB & 0xffff0000u) + kbB.y;
          const float rqa0 = csA * qa0 - snA * qa1, rqa1 = snA * qa0 + csA * qa1;
          const float rka0 = csA * ka0 - snA * ka1, rka1 = snA * ka0 + csA * ka1;
          float rqb0 = qb0, rqb1 = qb1, rkb0 = kb0, rkb1 = kb1;
          if constexpr (decltype(b_rotates)::value) {
            rqb0 = csB * qb0 - snB * qb1;
            rqb1 = snB * qb0 + csB * qb1;
            rkb0 = csB * kb0 - snB * kb1;
            rkb1 = snB * kb0 + csB * kb1;
          }
          const uint32_t qa = h2(rqa0, rqa1), ka = h2(rka0, rka1);
          const uint32_t qb = h2(rqb0, rqb1), kb = h2(rkb0, rkb1);
          if (t == len - 1) {
            if (rotA) F[kFCar + 64 * ((c + 1) & 1) + pA] = phA;
            if (rotB) F[kFCar + 64 * ((c + 1) & 1) + pB] = phB;
            if (last_chunk) {
              *reinterpret_cast<float2*>(a.final_k + sh * kN + 2 * pA) = make_float2(rka0, rka1);
              *reinterpret_cast<float2*>(a.final_k + sh * kN + 2 * pB) = make_float2(rkb0, rkb1);
              __nv_bfloat16* fa = static_cast<__nv_bfloat16*>(a.final_angle) + sh * R;
              if (rotA) fa[pA] = __float2bfloat16_rn(phA);
              if (rotB) fa[pB] = __float2bfloat16_rn(phB);
            }
          }
          *reinterpret_cast<uint32_t*>(smem + kOffQ + toff(t, 2 * pA)) = live ? qa : 0u;
          *reinterpret_cast<uint32_t*>(smem + kOffK + toff(t, 2 * pA)) = live ? ka : 0u;
          *reinterpret_cast<uint32_t*>(smem + kOffQ + toff(t, 2 * pB)) = live ? qb : 0u;
          *reinterpret_cast<uint32_t*>(smem + kOffK + toff(t, 2 * pB)) = live ? kb : 0u;
          dv[e] = live ? (rqa0 * rka0 + rqa1 * rka1) + (rqb0 * rkb0 + rqb1 * rkb1) : 0.f;
        }
        };
        if (R > 32)
          rotate_rows(std::true_type{});
        else
          rotate_rows(std::false_type{});
        // q^ . k^ of each token: the four lane octets summed first, then a
        // transpose-reduce over the 8 tokens (lane l ends with token 8 warp + l % 8)
#pragma unroll
        for (int e = 0; e < 8; ++e) dv[e] += __shfl_xor_sync(0xffffffffu, dv[e], 16);
#pragma unroll
        for (int e = 0; e < 8; ++e) dv[e] += __shfl_xor_sync(0xffffffffu, dv[e], 8);
#pragma unroll
        for (int o = 4; o >= 1; o >>= 1) {
          const bool up = (lane & o) != 0;
#pragma unroll
          for (int e = 0; e < o; ++e) {
            const float send = up ? dv[e] : dv[e + o];
            const float keep = up ? dv[e + o] : dv[e];
            dv[e] = keep + __shfl_xor_sync(0xffffffffu, send, o);
          }
        }
        if (lane < 8) F[kFDG + 8 * warp + lane] = dv[0];
      }
      __syncthreads();  // (B) S, diagonal partials; the raw chunk is spent
      if (c + 1 < nch) {
        prefetch(rb + kQ, min(kQ, it.T - (c + 1) * kQ));
        if (!sc_tma) load_scalars(rb + kQ, min(kQ, it.T - (c + 1) * kQ));
      }
      // ---- v (fp16) and v o w tiles; the last token's v is the final V state
      if (wait_bar(bar3, n_bar3 & 1u, s_abort))
        ++n_bar3;
      else
        *s_abort = 1u;
      {
        const float s_end = F[kFS + kQ - 1];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int idx = tid + kThreads * e, t = idx >> 3, c8 = idx & 7;
          const float w = ex2f(s_end - F[kFS + t]) * F[kFW + t];
          const uint4 vs = *reinterpret_cast<const uint4*>(smem + kOffVZ + toff(t, 8 * c8));
          const uint4 vr = t < len ? vs : make_uint4(0u, 0u, 0u, 0u);  // past the run: zero
          const uint32_t vw4[4] = {vr.x, vr.y, vr.z, vr.w};
          uint32_t f[4], g[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float x0 = __uint_as_float(vw4[u] << 16), x1 = __uint_as_float(vw4[u] & 0xffff0000u);
            f[u] = h2(x0, x1);
            g[u] = h2(x0 * w, x1 * w);
          }
          *reinterpret_cast<uint4*>(smem + kOffV + toff(t, 8 * c8)) = make_uint4(f[0], f[1], f[2], f[3]);
          *reinterpret_cast<uint4*>(smem + kOffVW + toff(t, 8 * c8)) = make_uint4(g[0], g[1], g[2], g[3]);
          if (last_chunk && t == len - 1)
            *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.final_v) + sh * kP + 8 * c8) = vs;
        }
      }
      fence_async_smem();
      tc_fence_before();
      __syncthreads();  // (C) operand tiles complete; the staging tile's v is spent
      if (*s_abort) {
        aborted = true;
        break;
      }
      if (tid == 0) {
        tc_fence_after();
        const uint64_t q0 = sdesc(sb + kOffQ, 16, 1024), k0 = sdesc(sb + kOffK, 16, 1024);
#pragma unroll
        for (int s2 = 0; s2 < kN / 16; ++s2) {
          const uint32_t ko = ((s2 >> 2) * kQ * 128 + (s2 & 3) * 32) >> 4;
          mma_ss(tmem + kColCB, q0 + ko, k0 + ko, idesc128(kQ, 0, 0, 0), s2 > 0);
        }
        if (c > 0) {
          const uint64_t h0 = sdesc(sb + kOffHT, kN * 128, 1024);
#pragma unroll
          for (int s2 = 0; s2 < kN / 16; ++s2) {
            const uint32_t ko = ((s2 >> 2) * kQ * 128 + (s2 & 3) * 32) >> 4;
            mma_ss(tmem + kColYo, q0 + ko, h0 + ((s2 * 2048) >> 4), idesc128(kP, 0, 1, 0), s2 > 0);
          }
        }
        const uint64_t kt0 = sdesc(sb + kOffK, kQ * 128, 1024), vw0 = sdesc(sb + kOffVW, kQ * 128, 1024);
#pragma unroll
        for (int s2 = 0; s2 < kQ / 16; ++s2)
          mma_ss(tmem + kColDH, kt0 + ((s2 * 2048) >> 4), vw0 + ((s2 * 2048) >> 4), idesc128(kP, 1, 1, 0), s2 > 0);
        mma_commit(bar0);
      }
      copy_vz(&tmz, rb, it.h);  // z of this chunk, for the output
      if (!wait_bar(bar0, n_bar0 & 1u, s_abort)) *s_abort = 1u;
      ++n_bar0;
      __syncthreads();
      if (*s_abort) {
        aborted = true;
        break;
      }
      tc_fence_after();
      // ---- M (fp16, to TMEM) and the state through this chunk
      {
        const float St = F[kFS + row];
        const float diag = F[kFDD + row] * F[kFDG + row];
#pragma unroll 1
        for (int kk = 0; kk < 2; ++kk) {
          const int s2 = 2 * cq + kk, j0 = 16 * s2;
          uint32_t m[8];
          if (j0 > 32 * (warp & 3) + 31) {  // above every row of this warp (warp-uniform: the TMEM load is .aligned)
#pragma unroll
            for (int e = 0; e < 8; ++e) m[e] = 0u;
          } else {
            float cb[16];
            tmem_ld16(tmem + lane_off + kColCB + (uint32_t)j0, cb);
            float mv[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int j = j0 + e;
              mv[e] = j < row ? cb[e] * ex2f(St - F[kFS + j]) * F[kFW + j] : (j == row ? diag : 0.f);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) m[e] = h2(mv[2 * e], mv[2 * e + 1]);
          }
          asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                       :: "r"(tmem + lane_off + kColM + 8u * (uint32_t)s2), "r"(m[0]), "r"(m[1]), "r"(m[2]),
                          "r"(m[3]), "r"(m[4]), "r"(m[5]), "r"(m[6]), "r"(m[7]) : "memory");
        }
        const float dec = ex2f(F[kFS + kQ - 1]);
        float d0[16];
        tmem_ld16(tmem + lane_off + kColDH + 16u * (uint32_t)cq, d0);
#pragma unroll
        for (int e = 0; e < 16; ++e) hs[e] = fmaf(dec, hs[e], d0[e]);
        if (!last_chunk) {
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) w[e] = h2(hs[8 * u + 2 * e], hs[8 * u + 2 * e + 1]);
            *reinterpret_cast<uint4*>(smem + kOffHT + toff(row, 16 * cq + 8 * u)) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      }
      fence_async_smem();
      tc_fence_before();
      __syncthreads();  // (D) M in TMEM, next H^T in shared memory
      if (tid == 0) {
        tc_fence_after();
        const uint64_t v0 = sdesc(sb + kOffV, kQ * 128, 1024);
#pragma unroll
        for (int s2 = 0; s2 < kQ / 16; ++s2)
          mma_ts(tmem + kColYd, tmem + kColM + 8u * (uint32_t)s2, v0 + ((s2 * 2048) >> 4), idesc128(kP, 0, 1, 0), s2 > 0);
        mma_commit(bar1);
      }
      if (!wait_bar(bar1, n_bar1 & 1u, s_abort)) *s_abort = 1u;
      ++n_bar1;
      if (wait_bar(bar3, n_bar3 & 1u, s_abort))
        ++n_bar3;
      else
        *s_abort = 1u;
      __syncthreads();
      if (*s_abort) {
        aborted = true;
        break;
      }
      tc_fence_after();
      // ---- output
      {
        const float et = ex2f(F[kFS + row]);
        float yd[16], yo[16];
        if (c > 0) {
          tmem_ld16x2(tmem + lane_off + kColYd + 16u * (uint32_t)cq, tmem + lane_off + kColYo + 16u * (uint32_t)cq, yd, yo);
        } else {
          tmem_ld16(tmem + lane_off + kColYd + 16u * (uint32_t)cq, yd);
#pragma unroll
          for (int e = 0; e < 16; ++e) yo[e] = 0.f;
        }
        uint32_t o[8];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const uint4 vv = *reinterpret_cast<const uint4*>(smem + kOffV + toff(row, 16 * cq + 8 * u));
          const uint32_t vw[4] = {vv.x, vv.y, vv.z, vv.w};
          const uint4 zz = *reinterpret_cast<const uint4*>(smem + kOffVZ + toff(row, 16 * cq + 8 * u));
          const uint32_t zw[4] = {zz.x, zz.y, zz.z, zz.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i0 = 8 * u + 2 * e;
            const float y0 = fmaf(et, yo[i0], yd[i0]) + dh * f16lo(vw[e]);
            const float y1 = fmaf(et, yo[i0 + 1], yd[i0 + 1]) + dh * f16hi(vw[e]);
            if (in_run) fsum += y0 + y1;
            const float z0 = __uint_as_float(zw[e] << 16), z1 = __uint_as_float(zw[e] & 0xffff0000u);
            const __nv_bfloat162 ob = __floats2bfloat162_rn(y0 * silu_f(z0), y1 * silu_f(z1));
            o[4 * u + e] = *reinterpret_cast<const uint32_t*>(&ob);
          }
        }
        if (in_run) {
          *reinterpret_cast<uint4*>(out + off) = make_uint4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<uint4*>(out + off + 8) = make_uint4(o[4], o[5], o[6], o[7]);
        }
      }
      tc_fence_before();
      __syncthreads();  // (E) tiles and TMEM free for the next chunk; z spent
      if (c + 1 < nch) copy_vz(&tmv, rb + kQ, it.h);
    }
    if (aborted) break;
    // ---- final state (an empty sequence has zero final states)
    if (nch == 0) {
      if (tid < kN) a.final_k[sh * kN + tid] = 0.f;
      if (tid < kP) static_cast<__nv_bfloat16*>(a.final_v)[sh * kP + tid] = __float2bfloat16_rn(0.f);
      if (tid < R) static_cast<__nv_bfloat16*>(a.final_angle)[sh * R + tid] = __float2bfloat16_rn(0.f);
    }
#pragma unroll
    for (int e = 0; e < 16; ++e) a.final_ssm[(sh * kP + 16 * cq + e) * kN + row] = hs[e];
#pragma unroll
    for (int e = 0; e < 16; ++e) fsum += hs[e];
    if (!isfinite(fsum)) *s_range = 1u;
    __syncthreads();
    if (*s_range) {
      // an fp16 operand overflowed: this (sequence, head) again, token by token
      serial_item(a, it, reinterpret_cast<float*>(smem));
      __syncthreads();
      if (tid == 0) *s_range = 0u;
      __syncthreads();
    }
  }
  // ---- teardown
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  if (aborted && tid == 0) {
    atomicAdd(&g_m3_timeouts, 1u);
    // what was issued last completes before its TMEM is released
    if (n_bar0 > 0) drain_bar(bar0, (n_bar0 - 1) & 1u);
    if (n_bar1 > 0) drain_bar(bar1, (n_bar1 - 1) & 1u);
    if (n_bar2 < n_pref) drain_bar(bar2, n_bar2 & 1u);  // a raw copy in flight
    if (n_bar3 < n_vz) drain_bar(bar3, n_bar3 & 1u);    // a v/z copy in flight
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" :: "r"(tmem));
}

}  // namespace

unsigned int read_m3_timeouts() {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_m3_timeouts, sizeof v) != cudaSuccess) return 0xffffffffu;
  return v;
}

namespace {
using Encode = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
Encode encoder() {
  static Encode encode = []() -> Encode {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<Encode>(fn);
  }();
  return encode;
}
// [rows][cols] of 2- or 4-byte elements as boxes of box_cols x box_rows (rows past
// the tensor read as zero)
bool make_map(CUtensorMap* tm, const void* base, int64_t rows, int64_t cols, int elem, int box_cols, int box_rows,
              bool swizzle) {
  const Encode encode = encoder();
  if (!encode || rows <= 0 || (reinterpret_cast<uintptr_t>(base) & 15u) != 0 || (cols * elem) % 16 != 0) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)(cols * elem)};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return encode(tm, elem == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

cudaError_t launch_m3_forward(const Mamba3Args& a, int num_sms, cudaStream_t st) {
  const int items = a.nseq * a.heads;
  if (items == 0) return cudaSuccess;
  const int64_t rows = a.cu[a.nseq];
  CUtensorMap tmv, tmz, tmdt, tmadt, tmtr;
  std::memset(&tmv, 0, sizeof tmv);  // maps that are not built are never read
  std::memset(&tmz, 0, sizeof tmz);
  std::memset(&tmdt, 0, sizeof tmdt);
  std::memset(&tmadt, 0, sizeof tmadt);
  std::memset(&tmtr, 0, sizeof tmtr);
  // v and z ([rows][heads * 64] bf16) as 64-column x 128-row boxes, 128-byte swizzle
  if (rows > 0 && !(make_map(&tmv, a.v, rows, (int64_t)a.heads * kP, 2, kP, kQ, true) &&
                    make_map(&tmz, a.z, rows, (int64_t)a.heads * kP, 2, kP, kQ, true)))
    return cudaErrorNotSupported;  // no tensor-map encoder: the kernel has no other way to load v and z
  // dt, adt ([rows][heads] f32) as 4 x 129 boxes and trap (bf16) as 8 x 129: when every
  // row is a 16-byte multiple (heads a multiple of 8), else strided loads
  const int sc_tma = rows > 0 && a.heads % 8 == 0 && make_map(&tmdt, a.dt, rows, a.heads, 4, 4, kQ + 1, false) &&
                     make_map(&tmadt, a.adt, rows, a.heads, 4, 4, kQ + 1, false) &&
                     make_map(&tmtr, a.trap, rows, a.heads, 2, 8, kQ + 1, false);
  cudaError_t e = cudaFuncSetAttribute(m3_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
  if (e != cudaSuccess) return e;
  const int grid = items < num_sms ? items : num_sms;
  m3_fwd_kernel<<<grid, kThreads, kSmem, st>>>(a, tmv, tmz, tmdt, tmadt, tmtr, sc_tma);
  return cudaGetLastError();
}

}  // namespace mamba2
