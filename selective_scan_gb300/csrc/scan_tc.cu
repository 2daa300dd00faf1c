// Chunked selective scan on the 5th-generation tensor cores (tcgen05 MMAs with
// TMEM accumulators, TMA tile loads) for headdim 64 x d_state 128, bf16.
//
// Semantics: gllm PR #85 "feat(backend): Mamba2 ops, with CPU reference
// implementations", section "Ops" (SSMScan): per token
//   dt' = softplus(dt + dt_bias),  h = h*exp(-exp(A_log)*dt') + dt'*B (x) x,
//   y = h.C + D*x,
// state seeded from / written back to the sequence's slot; the same page's
// section "CPU reference" names the chunked scan as the GPU technique checked
// against the token loop, and the page "Granite Mamba2 Inference
// Optimization" describes long prefill as a chunked parallel scan.
//
// Chunk of Q = 128 tokens, a_t = -exp(A_log) dt'_t, s_t = a_0 + ... + a_t:
//   y_t   = exp(s_t) C_t . h_in + sum_{j<=t} M[t][j] x_j,
//           M[t][j] = (C_t . B_j) exp(s_t - s_j) dt'_j  (+ D when j = t)
//   h_out = exp(s_{Q-1}) h_in + sum_j exp(s_{Q-1} - s_j) dt'_j x_j (x) B_j
// (every exponent a difference taken in the <= 0 direction).
//
// Full pass: one CTA per (sequence segment, head), 20 warps in fixed roles
// that hand work to each other through mbarriers (no CTA-wide barrier in the
// chunk loop):
//   warps 0-3   M(i) = CB o decay (+ D on the diagonal) in fp16, written over
//               the first 64 columns of chunk i's CB buffer in TMEM (one thread
//               per token row t = TMEM lane)
//   warps 4-7   X o w of chunk i (bf16 hi + lo) for the state product, and x
//               converted to fp16 in place for Y = M . X
//   warps 8-15  per chunk i: the state through chunk i (H = exp(total) H + dH,
//               fp32 in registers; TMEM lane n = state row n), the output y = Y
//               + exp(s_t) C . H^T(i-1) stored from registers, then H(i) as bf16
//               hi + lo to smem (two warps per TMEM lane quarter, 32 columns p each)
//   warp 16     the chunk's dt' = softplus(dt + dt_bias), cumulative log-decay
//               and block factors; CB = C . B^T   M=128 N=128 K=128
//   warp 17     Yoff = C . [H hi | H lo]^T       M=128 N=128 K=128 (H^T MN-major);
//               also loads the C and B tiles of chunk i+2
//   warp 18     dH^T = B^T . [X o w hi | lo]     M=128 N=128 K=128
//   warp 19     Y = M . X (fp16, A from TMEM)    M=128 N=64  K=128, into the
//               other 64 columns of the CB buffer (so Y is double-buffered by
//               chunk parity); also loads the X tile of chunk i+2
// An MMA-issuing thread spends about 200 cycles on each tcgen05.mma it issues,
// whatever its N (64 to 256): the time of a product is its instruction count,
// so the four products run as four concurrent streams from four warps, and
// the hi + lo splits that precision needs sit on the N side (one instruction
// covers both halves), never on the K side. A [rows][cols] tile stored with the
// 128-byte swizzle in 64-column blocks (the TMA box layout) is both the K-major
// and the MN-major tcgen05 operand, so every tile is used in its load layout.
// Precision (measured against the token loop on the 65 536-token workload):
// H carried as a single bf16 puts the worst y error at 1.03x its tolerance,
// as bf16 hi + lo at 5e-5 absolute; M and x in fp16 (11 significant bits) keep
// the worst y error within 0.86 of the tolerance (most of it the output's own
// bf16 rounding); X o w as a single bf16 gives a state error of 1.7e-3 against
// a 1e-3 tolerance, so it stays hi + lo. fp16 holds magnitudes up to 65 504: a
// CTA that meets a larger M entry or x recomputes its segment's y token by
// token in fp32 (correct, slow; no workload here comes near it).
//
// Long runs are cut into segments. The state pass computes, per segment but
// the last, the end state from zero (the first segment from the slot's state)
// and the total log-decay, walking the chunks from last to first so that every
// token's weight exp(s_end - s_j) dt'_j is known when its chunk is read: the
// products B^T . (X o w) of all chunks then accumulate in TMEM with no per-chunk
// state update. The full pass seeds segment k by folding the earlier segments'
// entries. Every wait is bounded: on a timeout the CTA records it in a device
// counter (mamba2_device_timeouts), drains what it issued, frees its TMEM and
// returns.
#include <cuda.h>

#include "common.cuh"

namespace mamba2 {

__device__ unsigned int g_tc_timeouts = 0;

namespace {

#include "tc.cuh"

constexpr int TQ = 128;  // tokens per chunk
constexpr int TP = 64;   // headdim
constexpr int TN = 128;  // d_state
constexpr int kMathWarps = 16;  // element-wise warps of either pass
constexpr int kMathThreads = 32 * kMathWarps;
constexpr int kFullThreads = kMathThreads + 4 * 32;   // + CB (and dt), Yoff (and C/B loads), dH, Y (and X loads) issuers
constexpr int kStateThreads = kMathThreads + 5 * 32;  // + X loader, B loader, hi issuer, weight producer, lo issuer
// full pass: the element-wise warps by role
constexpr int kMWarps = 8;   // warps 0-7: X o w (bf16 hi + lo) and the fp16 copy of x, then M
constexpr int kSWarps = 8;   // warps 8-15: state, output, H hi + lo
static_assert(kMWarps + kSWarps == kMathWarps, "full-pass roles");

// ---- full pass: TMEM columns (128 lanes each)
// [0,256): chunk parity b at 128 b: CB = C . B^T (fp32, 128 columns), then M (fp16,
// columns [0,64), k-step s at m_col(s)) written over it and Y = M . X (columns [64,128))
constexpr uint32_t kColM = 0, kColY = 64;
// TMEM column of M's k-step s (tokens [16 s, 16 s + 16)). The thread of half h =
// s % 2 of a row computes steps h, h + 2, h + 4, h + 6 in that order and reads CB
// columns [16 s, 16 s + 16) for each; step k of them (s = 2 k + h) goes to
// 32 (k / 2) + 16 h + 8 (k % 2), inside CB columns that the same thread read at
// its step k / 2 <= k. So no thread overwrites CB another thread has yet to read,
// and M fills columns [0, 64) whole, leaving [64, 128) to Y.
__host__ __device__ constexpr uint32_t m_col(int s) {
  return (uint32_t)(32 * ((s >> 1) >> 1) + 16 * (s & 1) + 8 * ((s >> 1) & 1));
}
constexpr uint32_t kColYo = 256;   // [256,384): C . [H hi | H lo]^T, column = p (hi) or 64 + p (lo)
constexpr uint32_t kColDH = 384;   // [384,512): B^T . [X o w hi | lo], lane = n

// ---- full pass: shared memory (operand tiles 1024-byte aligned; the base is)
constexpr uint32_t kTileC = TQ * TN * 2;  // 32 KB [t][n]
constexpr uint32_t kTileB = TQ * TN * 2;  // 32 KB [j][n]
constexpr uint32_t kTileX = TQ * TP * 2;  // 16 KB [j][p] (bf16 as loaded, then fp16 in place)
constexpr uint32_t kStage = kTileC + kTileB + kTileX;  // chunk parity b at b * kStage
constexpr uint32_t kOffXWhi = 2 * kStage;
constexpr uint32_t kOffXWlo = kOffXWhi + kTileX;
constexpr uint32_t kOffHT = kOffXWlo + kTileX;         // H^T bf16 [n][p hi | p lo] (two 64-column blocks)
constexpr uint32_t kTileHT = TN * 2 * TP * 2;          // 32 KB
constexpr int kDtRing = 2;                              // dt buffers (chunk i in i % 2)
constexpr int kDtS = 0, kDtP = TQ, kDtV = 2 * TQ;       // float offsets: S (log2), dt', v (tokens 0..95)
constexpr uint32_t kDtBuf = (2 * TQ + 96) * 4;
constexpr uint32_t kOffDt = kOffHT + kTileHT;
constexpr uint32_t kOffBar = kOffDt + kDtRing * kDtBuf;
enum FullBar : int {  // + chunk % 2
  kFullCB = 0, kFullX = 2, kDtReady = 4, kDtFree = 6, kCBDone = 8, kMReady = 10, kXWReady = 12, kYdDone = 14,
  kYoDone = 16, kDHDone = 18, kDHFree = 20, kHReady = 22, kEpiDone = 24, kYoIssued = 26, kYIssued = 28,
  kNumFullBars = 30
};
constexpr uint32_t kOffMisc = kOffBar + 8 * kNumFullBars;  // TMEM base, abort flag, fp16 range flag
constexpr uint32_t kFullSmem = kOffMisc + 16;
static_assert(kFullSmem <= 232448, "full-pass shared memory plan exceeds 227 KB");

// ---- state pass: two heads of one group per CTA (they share the B tile). The
// product is D = (X o w)^T . B with X o w (bf16 hi and lo) written to TMEM by the
// element-wise warps as the A operand (lane = column p of head 0, then head 1), so
// shared memory holds only the loaded X and B tiles, three chunks deep: an X stage
// is free once X o w of its chunk is formed, a B stage once its chunk's products
// are done.
constexpr int kStStages = 3;                            // X and B rings: chunk i in stage i % 3
constexpr uint32_t kStXStage = 2 * kTileX;              // the X tiles of both heads
constexpr uint32_t kStOffB = kStStages * kStXStage;     // B stages
constexpr uint32_t kStOffW = kStOffB + kStStages * kTileB;  // [2 buffers][2 heads][TQ] token weights
constexpr uint32_t kStOffR = kStOffW + 2 * 2 * TQ * 4;  // [2 heads] total log2 decay of the piece
constexpr uint32_t kStOffBar = kStOffR + 16;
enum StateBar : int {  // + chunk % 3 on the rings of three, + chunk % 2 on the rings of two
  kStFullX = 0, kStFullB = 3, kStXFree = 6, kStBFree = 9, kStXWReady = 12, kStDHDone = 14, kStWReady = 16,
  kNumStateBars = 18
};
constexpr uint32_t kStOffMisc = kStOffBar + 8 * kNumStateBars;
constexpr uint32_t kStateSmem = kStOffMisc + 16;  // the base is 1024-byte aligned (checked)
// TMEM: D = (X o w)^T . B as hi and lo accumulators (lane = p of head 0 then head 1,
// column = n), and X o w itself, the products' A operand, in two stages (lane = p,
// column j / 2 holds tokens j and j + 1 as a bf16 pair): hi, then lo
constexpr uint32_t kStColDHi = 0, kStColDLo = 128, kStColXW = 256;
static_assert(kStateSmem <= 232448, "state-pass shared memory plan exceeds 227 KB");


// byte offset of element (r, c) in a [R][cols] bf16 tile, 128-byte swizzle,
// 64-column blocks of R rows each (the layout a TMA box of 64 x R lands in)
__device__ __forceinline__ uint32_t tile_off(int r, int c, int R) {
  return (uint32_t)((c >> 6) * R * 128 + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) + (c & 7) * 2);
}




// 2^x with the hardware approximation (flushes subnormal results to zero)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
// fp32 pair -> (hi, lo) bf16 pairs with hi + lo ~ v to ~2^-17
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = pack2(a, b);
  lo = pack2(a - __uint_as_float(hi << 16), b - __uint_as_float(hi & 0xffff0000u));
}
// ---- packed fp32 pairs (one instruction for two lanes of arithmetic)
struct F2 {
  uint64_t v;
};
__device__ __forceinline__ F2 f2(float lo, float hi) {
  F2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float f2lo(F2 a) {
  float lo;
  asm("{\n .reg .f32 t;\n mov.b64 {%0, t}, %1;\n}" : "=f"(lo) : "l"(a.v));
  return lo;
}
__device__ __forceinline__ float f2hi(F2 a) {
  float hi;
  asm("{\n .reg .f32 t;\n mov.b64 {t, %0}, %1;\n}" : "=f"(hi) : "l"(a.v));
  return hi;
}
__device__ __forceinline__ F2 add2(F2 a, F2 b) {
  F2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}
__device__ __forceinline__ F2 mul2(F2 a, F2 b) {
  F2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}
__device__ __forceinline__ F2 fma2(F2 a, F2 b, F2 c) {
  F2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r.v) : "l"(a.v), "l"(b.v), "l"(c.v));
  return r;
}
// bf16 pair of a packed pair (round to nearest even), lo in the low half
__device__ __forceinline__ uint32_t pack2(F2 a) { return pack2(f2lo(a), f2hi(a)); }

// ---- tile loads

// Where one chunk's tiles come from: xbc rows [rb, rb + len), 1 <= len <= TQ.
struct ChunkSrc {
  const __nv_bfloat16* xbc;
  int64_t ld;  // row stride (conv_dim)
  int64_t rb;
  int len;
};

// One [TQ][ncols] tile (64-column blocks, 128-byte swizzle) of columns
// [col0, col0 + ncols), by the whole calling warp: a TMA box per 64 columns
// when the chunk is whole, else 16-byte cp.async pieces with the rows past the
// run zero-filled. Arms `bar` with the bytes (TMA) or arrives on it once the
// copies are visible to the tensor cores (cp.async): one arrival per call, so
// a barrier shared by two tiles is initialised with count 2.
__device__ __forceinline__ void load_tile(uint32_t dst, const ChunkSrc& s, const CUtensorMap* tm, bool use_tma,
                                          int col0, int ncols, uint32_t bar, int lane) {
  if (use_tma && s.len == TQ) {
    if (lane == 0) {
      mbar_expect_tx(bar, (uint32_t)(TQ * ncols * 2));
      for (int b = 0; b < ncols / 64; ++b) tma_load_2d(dst + b * TQ * 128, tm, col0 + 64 * b, (int)s.rb, bar);
    }
  } else {
    const int pieces = ncols / 8;
    for (int i = lane; i < TQ * pieces; i += 32) {
      const int t = i / pieces, pc = i - t * pieces;
      const bool ok = t < s.len;
      const int64_t grow = ok ? s.rb + t : s.rb;
      cp_async16(dst + tile_off(t, pc * 8, TQ), s.xbc + grow * s.ld + col0 + pc * 8, ok);
    }
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;\n" ::: "memory");
    fence_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
  }
}

// What one CTA works on: head h of segment k of sequence sq, chunks [c_begin, c_end).
struct Cta {
  int sq, seg0, k, nseg, h, row0, T, c_begin, c_end, n;
  bool fresh;
  int x_col, b_col, c_col;
  float A2, Dh;  // decay rate in log2 units, skip weight
};
__device__ __forceinline__ Cta cta_info(const ScanArgs& a, int seg) {
  Cta c;
  c.h = blockIdx.y;
  c.sq = find_tile_seq(a.tab, seg);
  c.seg0 = a.tab.tile[c.sq];
  c.k = seg - c.seg0;
  c.nseg = a.tab.tile[c.sq + 1] - c.seg0;
  const int H = a.heads, G = a.ngroups;
  const int g = c.h / (H / G);
  c.row0 = a.tab.cu[c.sq];
  c.T = a.tab.cu[c.sq + 1] - c.row0;
  const int nchunks = (c.T + TQ - 1) / TQ;
  c.c_begin = c.k * a.seg_chunks;
  c.c_end = min(nchunks, c.c_begin + a.seg_chunks);
  c.n = max(0, c.c_end - c.c_begin);
  c.fresh = seq_fresh(a.tab, c.sq);
  c.x_col = c.h * TP;
  c.b_col = H * TP + g * TN;
  c.c_col = H * TP + G * TN + g * TN;
  c.A2 = expf(a.A_log[c.h]) * 1.4426950408889634f;
  c.Dh = a.D[c.h];
  return c;
}

// dt' of this lane's four tokens (4l .. 4l+3) of one chunk, 0 past the run.
struct DtQuad {
  float v[4];
};
// dt' = softplus(dt + dt_bias) of every (row, head), transposed to [head][row]
// so that a chunk's 128 values of one head are contiguous. 32 x 32 tiles.
__global__ void __launch_bounds__(256) dt_prime_kernel(const __nv_bfloat16* __restrict__ dt, const float* __restrict__ dt_bias,
                                                      float* __restrict__ dtp, int rows, int heads) {
  __shared__ float tile[32][33];
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // the state pass may be scheduled
  const int r0 = blockIdx.x * 32, h0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  for (int k = ty; k < 32; k += 8) {
    const int r = r0 + k, h = h0 + tx;
    if (r < rows && h < heads) tile[k][tx] = softplus_f(__bfloat162float(dt[(int64_t)r * heads + h]) + dt_bias[h]);
  }
  __syncthreads();
  for (int k = ty; k < 32; k += 8) {
    const int h = h0 + k, r = r0 + tx;
    if (r < rows && h < heads) dtp[(int64_t)h * rows + r] = tile[tx][k];
  }
}
// The same, 64 rows x every head per CTA: the rows' dt are one contiguous run
// (read with coalesced loads), and each head's 64 dt' one contiguous 256-byte
// run (written with coalesced stores); [head][row] staging in shared memory.
constexpr int kDtRows = 64;
__global__ void __launch_bounds__(256) dt_prime_rows_kernel(const __nv_bfloat16* __restrict__ dt,
                                                           const float* __restrict__ dt_bias, float* __restrict__ dtp,
                                                           int rows, int heads) {
  extern __shared__ float dts[];  // [heads][kDtRows + 1]
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // the state pass may be scheduled
  const int r0 = blockIdx.x * kDtRows;
  const int nr = min(kDtRows, rows - r0);
  const __nv_bfloat16* src = dt + (int64_t)r0 * heads;
  // thread t: head t % heads of rows t / heads, + rpp, + 2 rpp, ... (rpp rows a pass)
  const int rpp = max(1, 256 / heads);
  if (threadIdx.x < rpp * heads) {
    const int h = (int)threadIdx.x % heads;
    const float bias = dt_bias[h];
    for (int r = (int)threadIdx.x / heads; r < nr; r += rpp) {
      // softplus(v) = max(v, 0) + log(1 + e^-|v|), with the hardware base-2
      // exponential and logarithm (absolute error about 1e-7)
      const float v = __bfloat162float(src[(int64_t)r * heads + h]) + bias;
      float e, l;
      asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(-fabsf(v) * 1.4426950408889634f));
      asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(l) : "f"(1.0f + e));
      dts[h * (kDtRows + 1) + r] = fmaxf(v, 0.0f) + l * 0.6931471805599453f;
    }
  }
  // (heads above 256: the remaining heads, one per thread and row)
  for (int h = 256; h < heads; h += 256) {
    const int hh = h + (int)threadIdx.x;
    if (hh < heads)
      for (int r = 0; r < nr; ++r) dts[hh * (kDtRows + 1) + r] = softplus_f(__bfloat162float(src[(int64_t)r * heads + hh]) + dt_bias[hh]);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < heads * kDtRows; e += 256) {
    const int h = e / kDtRows, r = e - h * kDtRows;
    if (r < nr) dtp[(int64_t)h * rows + r0 + r] = dts[h * (kDtRows + 1) + r];
  }
}
constexpr int kDtRowsMaxHeads = 768;  // shared memory [heads][65] floats within 200 KB

// inclusive warp scan
__device__ __forceinline__ float warp_incl_sum(float v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  return v;
}

// fp16 pair (lo in the low half), the TMEM A-operand packing of a k-step
__device__ __forceinline__ uint32_t f16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ uint32_t f16x2(F2 a) { return f16x2(f2lo(a), f2hi(a)); }
// bf16 hi + lo of a packed pair
__device__ __forceinline__ void split2(F2 a, uint32_t& hi, uint32_t& lo) {
  hi = pack2(a);
  lo = pack2(add2(a, f2(-__uint_as_float(hi << 16), -__uint_as_float(hi & 0xffff0000u))));
}

// Seed of segment k of a sequence for state rows [p0, p0 + np) x column n: the
// slot (zero when fresh; the state pass's copy when the last segment of the same
// launch overwrites the slot), or the in-order fold of every piece's entry of
// the earlier segments.
__device__ __forceinline__ float seed_at(const ScanArgs& a, const Cta& ci, int p, int n) {
  const int H = a.heads;
  const int P = a.state_pieces > 0 ? a.state_pieces : 1;
  const int64_t head_off = (int64_t)ci.h * TP * TN + (int64_t)p * TN + n;
  auto entry = [&](int e) { return a.ws_state + (int64_t)e * H * TP * TN + head_off; };
  if (ci.k == 0) {
    if (ci.fresh) return 0.0f;
    if (ci.nseg > 1) return *entry((ci.seg0 + ci.nseg - 1) * P);
    return a.ssm_state[(int64_t)seq_slot(a.tab, ci.sq) * H * TP * TN + head_off];
  }
  float h = *entry(ci.seg0 * P);
  for (int e = ci.seg0 * P + 1; e < (ci.seg0 + ci.k) * P; ++e)
    h = fmaf(__expf(a.ws_decay[(int64_t)e * H + ci.h]), h, *entry(e));
  return h;
}

// Token-by-token recomputation of y for this CTA's (segment, head), used when
// a chunk's fp16 operands of Y = M . X would overflow. State in fp32 in shared
// memory; thread (p, n-sixteenth) of 512 keeps 16 state entries in registers.
__device__ __noinline__ void full_pass_serial_y(const ScanArgs& a, const Cta& ci, int tid) {
  if (tid >= 512) return;
  const int p = tid >> 3, n0 = (tid & 7) * 16;
  const int H = a.heads;
  float h[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) h[e] = seed_at(a, ci, p, n0 + e);
  const __nv_bfloat16* xbc = static_cast<const __nv_bfloat16*>(a.xbc);
  __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.dst);
  const int64_t rows_all = a.tab.cu[a.tab.n];
  const int t0 = ci.c_begin * TQ, t1 = min(ci.c_end * TQ, ci.T);
  for (int t = t0; t < t1; ++t) {
    const int64_t r = ci.row0 + t;
    const float dp = a.dtp[(int64_t)ci.h * rows_all + r];
    const float decay = ex2(-ci.A2 * dp);
    const __nv_bfloat16* row = xbc + r * a.conv_dim;
    const float x = __bfloat162float(row[ci.x_col + p]);
    const float dx = dp * x;
    float acc = 0.0f;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float B = __bfloat162float(row[ci.b_col + n0 + e]);
      const float C = __bfloat162float(row[ci.c_col + n0 + e]);
      h[e] = fmaf(h[e], decay, dx * B);
      acc = fmaf(h[e], C, acc);
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    acc += __shfl_xor_sync(0xffffffffu, acc, 4);
    if ((tid & 7) == 0) dst[r * (int64_t)(H * TP) + ci.x_col + p] = __float2bfloat16_rn(fmaf(ci.Dh, x, acc));
  }
}

__global__ void __launch_bounds__(kFullThreads, 1)
ssd_tc_full(const __grid_constant__ ScanArgs a, const __grid_constant__ CUtensorMap tm, const int use_tma) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const uint32_t sbase = su32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if ((sbase & 1023u) != 0) {  // the swizzled operand tiles need a 1024-byte aligned base
    if (tid == 0) atomicAdd(&g_tc_timeouts, 1u);
    return;
  }
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile uint32_t* s_abort = reinterpret_cast<volatile uint32_t*>(smem + kOffMisc + 4);
  volatile uint32_t* s_range = reinterpret_cast<volatile uint32_t*>(smem + kOffMisc + 8);
  auto bar = [&](int id) { return sbase + kOffBar + 8u * (uint32_t)id; };
  auto par = [](int i) { return (uint32_t)((i >> 1) & 1); };  // phase parity of chunk i on a [2] barrier
  auto stage = [&](int i) { return sbase + (uint32_t)(i & 1) * kStage; };
  auto dtbuf = [&](int i) { return reinterpret_cast<const float*>(smem + kOffDt + (uint32_t)(i & 1) * kDtBuf); };

  const Cta ci = cta_info(a, blockIdx.x);
  const int n = ci.n;
  const int H = a.heads;
  const __nv_bfloat16* xbc = static_cast<const __nv_bfloat16*>(a.xbc);

  // ---- TMEM (warp 0) and barriers
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" :: "r"(su32(s_tmem)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == kMathThreads) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(kFullCB + b), 2);  // C tile, B tile
      mbar_init(bar(kFullX + b), 1);
      mbar_init(bar(kDtReady + b), 1);
      mbar_init(bar(kDtFree + b), kMathWarps);
      mbar_init(bar(kCBDone + b), 1);
      mbar_init(bar(kMReady + b), kMWarps);
      mbar_init(bar(kXWReady + b), kMWarps);
      mbar_init(bar(kYdDone + b), 1);
      mbar_init(bar(kYoDone + b), 1);
      mbar_init(bar(kDHDone + b), 1);
      mbar_init(bar(kDHFree + b), kSWarps);
      mbar_init(bar(kHReady + b), kSWarps);
      mbar_init(bar(kEpiDone + b), kSWarps);
      mbar_init(bar(kYoIssued + b), 1);
      mbar_init(bar(kYIssued + b), 1);
    }
    *s_abort = 0u;
    *s_range = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  // Launched as a programmatic dependent of the state pass (or of the dt'
  // pre-pass): the tile loaders (warps 17 and 19) read only the conv's output
  // and start at once; every other role reads dt', the state entries or the
  // slot, or writes dst, after this wait.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // the norm may be scheduled
  if (warp != kMathWarps + 1 && warp != kMathWarps + 3) asm volatile("griddepcontrol.wait;" ::: "memory");

  auto chunk_src = [&](int i) {
    ChunkSrc s;
    const int c = ci.c_begin + i;
    s.xbc = xbc;
    s.ld = a.conv_dim;
    s.rb = ci.row0 + (int64_t)c * TQ;
    s.len = min(TQ, ci.T - c * TQ);
    return s;
  };

  // the running state of the S warps (H^T: state row n = TMEM lane, 32 columns p),
  // kept to the end for the slot write
  F2 hs[16];  // pair e: columns pc0 + 2 e, pc0 + 2 e + 1
  bool live = true;
  const int sw = warp - kMWarps;  // S warp index when >= 0
  const int s_half = (sw >> 2) & 1;
  const int s_row = (warp & 3) * 32 + lane;
  const int pc0 = 32 * s_half;

  if (warp < kMWarps) {
    // =================== per chunk i, (a) X o w (bf16 hi + lo, w_j = exp(s_end -
    // s_j) dt'_j) for the state product and x converted to fp16 in place for Y = M .
    // X, by the warps of TMEM lane quarters 0-2 (quarter 3 has the largest share of
    // M); (b) M(i) = CB o exp(s_t - s_j) dt'_j (j <= t), + D on the diagonal, in fp16
    // over the chunk's CB buffer, two threads per token row t (TMEM lane), four
    // k-steps each (see m_col). Below the diagonal block exp(s_t - s_j) = exp(s_t -
    // s_e) exp(s_e - s_j) with e the 32-block's last token (the second factor times
    // dt'_j being v_j); the diagonal block exponentiates each pair; above it, zero.
    const int qrt = warp & 3;
    const int half = warp >> 2;
    const int row = qrt * 32 + lane;
    const uint32_t lane_off = (uint32_t)(qrt * 32) << 16;
    const int xu = qrt < 3 ? half * 96 + qrt * 32 + lane : -1;  // X o w thread index (192 of them)
    for (int i = 0; i < n; ++i) {
      // (a) X o w and fp16 x of chunk i
      bool ok = warp_wait(bar(kDtReady + (i & 1)), par(i), s_abort);
      if (ok && qrt < 3) {
        ok = warp_wait(bar(kFullX + (i & 1)), par(i), s_abort);
        if (ok && i > 0) ok = warp_wait(bar(kDHDone + ((i - 1) & 1)), par(i - 1), s_abort);  // X o w buffer read
      }
      if (!ok) break;
      const float* D0 = dtbuf(i);
      if (qrt < 3) {
        unsigned char* xt = smem + (uint32_t)(i & 1) * kStage + kTileC + kTileB;
        const float Send = D0[kDtS + TQ - 1];
#pragma unroll 1
        for (int v = xu; v < TQ * TP / 8; v += 192) {  // 16-byte vector v: row v / 8, columns 8 (v % 8) ..
          const int j = v >> 3;
          const uint32_t o = tile_off(j, 8 * (v & 7), TQ);
          const float w = ex2(Send - D0[kDtS + j]) * D0[kDtP + j];
          const F2 w2 = f2(w, w);
          const uint4 xv = *reinterpret_cast<const uint4*>(xt + o);
          const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
          uint32_t hi[4], lo[4], f[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const F2 x2 = f2(__uint_as_float(xw[e] << 16), __uint_as_float(xw[e] & 0xffff0000u));
            split2(mul2(x2, w2), hi[e], lo[e]);
            f[e] = f16x2(x2);  // an x beyond the fp16 range makes y non-finite: caught at the output
          }
          *reinterpret_cast<uint4*>(smem + kOffXWhi + o) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(smem + kOffXWlo + o) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          *reinterpret_cast<uint4*>(xt + o) = make_uint4(f[0], f[1], f[2], f[3]);
        }
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kXWReady + (i & 1)));

      // (b) M(i)
      if (!warp_wait(bar(kCBDone + (i & 1)), par(i), s_abort)) break;
      tc_fence_after();
      const float St = D0[kDtS + row];
      const uint32_t buf = tmem + lane_off + 128u * (uint32_t)(i & 1);
#pragma unroll 1
      for (int k = 0; k < 4; ++k) {
        const int s = 2 * k + half, bb = s >> 1, j0 = 16 * s;
        uint32_t m[8];
        if (bb > qrt) {
#pragma unroll
          for (int e = 0; e < 8; ++e) m[e] = 0u;
        } else {
          float cb[16];
          tmem_ld16(buf + (uint32_t)j0, cb);
          if (bb < qrt) {
            const float u = ex2(St - D0[kDtS + 32 * bb + 31]);
            const F2 u2 = f2(u, u);
            float v[16];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              *reinterpret_cast<float4*>(v + 4 * e) = *reinterpret_cast<const float4*>(D0 + kDtV + j0 + 4 * e);
#pragma unroll
            for (int e = 0; e < 8; ++e)  // an entry beyond the fp16 range makes y non-finite: caught at the output
              m[e] = f16x2(mul2(f2(cb[2 * e], cb[2 * e + 1]), mul2(u2, f2(v[2 * e], v[2 * e + 1]))));
          } else {
            float sj[16], dj[16];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              *reinterpret_cast<float4*>(sj + 4 * e) = *reinterpret_cast<const float4*>(D0 + kDtS + j0 + 4 * e);
              *reinterpret_cast<float4*>(dj + 4 * e) = *reinterpret_cast<const float4*>(D0 + kDtP + j0 + 4 * e);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int ja = j0 + 2 * e, jb = ja + 1;
              float ma = ja <= row ? cb[2 * e] * ex2(St - sj[2 * e]) * dj[2 * e] : 0.f;
              float mb = jb <= row ? cb[2 * e + 1] * ex2(St - sj[2 * e + 1]) * dj[2 * e + 1] : 0.f;
              if (ja == row) ma += ci.Dh;
              if (jb == row) mb += ci.Dh;
              m[e] = f16x2(ma, mb);
            }
          }
        }
        asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                     :: "r"(buf + kColM + m_col(s)), "r"(m[0]), "r"(m[1]), "r"(m[2]), "r"(m[3]), "r"(m[4]),
                        "r"(m[5]), "r"(m[6]), "r"(m[7]) : "memory");
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(kMReady + (i & 1)));
        mbar_arrive(bar(kDtFree + (i & 1)));
      }
    }
  } else if (warp < kMathWarps) {
    // =================== S warps: per chunk i, (a) the state through chunk i (H =
    // exp(total) H + dH, dH = hi part + lo part; TMEM lane = state row n), (b) once
    // C . H^T(i-1) is done, its value read and H(i) written to shared memory as bf16
    // hi + lo, (c) the output y = M . X + exp(s_t) C . H^T, straight to HBM. Two
    // warps per TMEM lane quarter, 32 columns p each.
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int row = s_row;
    {
      // the seed (seed_at's rule), entry by entry, each entry's 32 loads independent
      const int P = a.state_pieces > 0 ? a.state_pieces : 1;
      const int64_t col = (int64_t)pc0 * TN + row, head_off = (int64_t)ci.h * TP * TN;
      auto entry = [&](int e) { return a.ws_state + (int64_t)e * H * TP * TN + head_off + col; };
      auto load = [&](const float* src) {
#pragma unroll
        for (int e = 0; e < 16; ++e) hs[e] = f2(src[(int64_t)(2 * e) * TN], src[(int64_t)(2 * e + 1) * TN]);
      };
      if (ci.k == 0) {
        if (ci.fresh) {
#pragma unroll
          for (int e = 0; e < 16; ++e) hs[e] = f2(0.0f, 0.0f);
        } else {
          load(ci.nseg > 1 ? entry((ci.seg0 + ci.nseg - 1) * P)
                           : a.ssm_state + (int64_t)seq_slot(a.tab, ci.sq) * H * TP * TN + head_off + col);
        }
      } else {
        load(entry(ci.seg0 * P));
#pragma unroll 1
        for (int e = ci.seg0 * P + 1; e < (ci.seg0 + ci.k) * P; ++e) {
          const float d = __expf(a.ws_decay[(int64_t)e * H + ci.h]);
          const F2 d2 = f2(d, d);
          const float* src = entry(e);
#pragma unroll
          for (int q = 0; q < 16; ++q) hs[q] = fma2(d2, hs[q], f2(src[(int64_t)(2 * q) * TN], src[(int64_t)(2 * q + 1) * TN]));
        }
      }
    }
    auto write_h = [&]() {  // bf16 hi + lo of H^T: row n, columns [pc0, +32) of each block
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) split2(hs[4 * q + e], hw[e], lw[e]);
        *reinterpret_cast<uint4*>(smem + kOffHT + tile_off(row, pc0 + 8 * q, TN)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4*>(smem + kOffHT + tile_off(row, TP + pc0 + 8 * q, TN)) =
            make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
    };
    write_h();
    fence_async_smem();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(bar(kHReady));
      mbar_arrive(bar(kDHFree));
    }
    // sum of every output: not finite iff an fp16 operand of Y = M . X overflowed
    // (an M entry or x beyond 65 504 becomes inf, and inf or inf * 0 reaches y)
    F2 ysum = f2(0.0f, 0.0f);
    for (int i = 0; i < n; ++i) {
      // (a) state through chunk i; releases the dH accumulator and the dt buffer
      if (!(warp_wait(bar(kDtReady + (i & 1)), par(i), s_abort) && warp_wait(bar(kDHDone + (i & 1)), par(i), s_abort))) {
        live = false;
        break;
      }
      tc_fence_after();
      const float* D0 = dtbuf(i);
      const float decay = ex2(D0[kDtS + TQ - 1]);
      const float et = ex2(D0[kDtS + row]);
      const F2 dec2 = f2(decay, decay), et2 = f2(et, et);
#pragma unroll
      for (int q = 0; q < 2; ++q) {  // unrolled: the state must stay in registers
        float dh[16], dl[16];
        tmem_ld16x2(tmem + lane_off + kColDH + pc0 + 16 * q, tmem + lane_off + kColDH + TP + pc0 + 16 * q, dh, dl);
#pragma unroll
        for (int e = 0; e < 8; ++e)
          hs[8 * q + e] = fma2(dec2, hs[8 * q + e], add2(f2(dh[2 * e], dh[2 * e + 1]), f2(dl[2 * e], dl[2 * e + 1])));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(kDHFree + ((i + 1) & 1)));
        mbar_arrive(bar(kDtFree + (i & 1)));
      }
      // (b) the output of chunk i, y = M . X + exp(s_t) C . H^T(i-1), straight to HBM;
      // then H(i) for C . H^T(i+1) (C . H^T(i-1) has read the previous one)
      if (!(warp_wait(bar(kYoDone + (i & 1)), par(i), s_abort) && warp_wait(bar(kYdDone + (i & 1)), par(i), s_abort))) {
        live = false;
        break;
      }
      tc_fence_after();
      {
        const int c = ci.c_begin + i;
        const bool in_run = row < min(TQ, ci.T - c * TQ);
        __nv_bfloat16* ydst = static_cast<__nv_bfloat16*>(a.dst) +
                              (ci.row0 + (int64_t)c * TQ + row) * (int64_t)(H * TP) + ci.x_col + pc0;
        const uint32_t ybuf = tmem + lane_off + 128u * (uint32_t)(i & 1) + kColY + pc0;
        const uint32_t obuf = tmem + lane_off + kColYo + pc0;
#pragma unroll 1
        for (int q = 0; q < 2; ++q) {  // 16 columns at a time
          float yd[16], oh[16], ol[16];
          tmem_ld16x2(obuf + 16 * q, obuf + TP + 16 * q, oh, ol);
          tmem_ld16(ybuf + 16 * q, yd);
          uint32_t o[8];
#pragma unroll
          for (int f = 0; f < 8; ++f) {
            const F2 yv = fma2(et2, add2(f2(oh[2 * f], oh[2 * f + 1]), f2(ol[2 * f], ol[2 * f + 1])),
                               f2(yd[2 * f], yd[2 * f + 1]));
            ysum = add2(ysum, yv);
            o[f] = pack2(yv);
          }
          // one full 32-byte sector (y rows and the 16-column groups are 32-byte aligned)
          if (in_run)
            asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(ydst + 16 * q), "r"(o[0]), "r"(o[1]),
                         "r"(o[2]), "r"(o[3]), "r"(o[4]), "r"(o[5]), "r"(o[6]), "r"(o[7]) : "memory");
        }
      }
      write_h();
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(kHReady + ((i + 1) & 1)));
        mbar_arrive(bar(kEpiDone + (i & 1)));
      }
    }
    if (!isfinite(f2lo(ysum) + f2hi(ysum))) *s_range = 1u;
  } else if (warp == kMathWarps) {
    // =================== per chunk i: dt' (loaded four chunks ahead), log2-scaled
    // cumulative decay S and block factors v into dt buffer i % 2 (lane l: tokens
    // 4l .. 4l+3; the buffer last served chunk i-2, whose readers are done); then
    // CB = C . B^T (lane 0) into buffer i % 2 once chunk i-2's output has left it
    const int64_t rows_all = a.tab.cu[a.tab.n];
    auto load_dtp = [&](int i) {
      DtQuad r = {{0.f, 0.f, 0.f, 0.f}};
      if (i < n) {
        const int c = ci.c_begin + i, len = min(TQ, ci.T - c * TQ);
        const float* src = a.dtp + (int64_t)ci.h * rows_all + ci.row0 + (int64_t)c * TQ;
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (4 * lane + e < len) r.v[e] = src[4 * lane + e];
      }
      return r;
    };
    DtQuad r0 = load_dtp(0), r1 = load_dtp(1), r2 = load_dtp(2), r3 = load_dtp(3);
    int last = -1;
    for (int i = 0; i < n; ++i) {
      if (i >= 2 && !warp_wait(bar(kDtFree + (i & 1)), par(i - 2), s_abort)) break;
      {
        float dp[4], S[4], run = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          dp[e] = r0.v[e];
          run -= ci.A2 * dp[e];
          S[e] = run;
        }
        r0 = r1;
        r1 = r2;
        r2 = r3;
        r3 = load_dtp(i + 4);
        const float excl = warp_incl_sum(run, lane) - run;
#pragma unroll
        for (int e = 0; e < 4; ++e) S[e] += excl;
        const float Se = __shfl_sync(0xffffffffu, S[3], (lane & ~7) | 7);  // S at the end of this 32-block
        float* D0 = reinterpret_cast<float*>(smem + kOffDt + (uint32_t)(i & 1) * kDtBuf);
        *reinterpret_cast<float4*>(D0 + kDtS + 4 * lane) = make_float4(S[0], S[1], S[2], S[3]);
        *reinterpret_cast<float4*>(D0 + kDtP + 4 * lane) = make_float4(dp[0], dp[1], dp[2], dp[3]);
        if (lane < 24)  // v of tokens 0..95 (the last block is never below a diagonal)
          *reinterpret_cast<float4*>(D0 + kDtV + 4 * lane) =
              make_float4(ex2(Se - S[0]) * dp[0], ex2(Se - S[1]) * dp[1], ex2(Se - S[2]) * dp[2], ex2(Se - S[3]) * dp[3]);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kDtReady + (i & 1)));
      }
      if (!warp_wait(bar(kFullCB + (i & 1)), par(i), s_abort)) break;
      if (i >= 2 && !warp_wait(bar(kEpiDone + (i & 1)), par(i - 2), s_abort)) break;  // buffer i % 2 free
      // behind C . H^T(i-1) and Y(i-1) in the tensor pipe: those two gate the output
      if (i >= 1 && !warp_wait(bar(kYIssued + ((i - 1) & 1)), par(i - 1), s_abort)) break;
      tc_fence_after();
      if (lane == 0) {
        const uint64_t a0 = sdesc(stage(i), 16, 1024), b0 = sdesc(stage(i) + kTileC, 16, 1024);
#pragma unroll
        for (int s2 = 0; s2 < TN / 16; ++s2) {
          const uint32_t ko = ((s2 >> 2) * TQ * 128 + (s2 & 3) * 32) >> 4;
          mma_ss(tmem + 128u * (uint32_t)(i & 1), a0 + ko, b0 + ko, idesc128(128, 0, 0), s2 > 0);
        }
        mma_commit(bar(kCBDone + (i & 1)));
      }
      __syncwarp();
      last = i;
    }
    if (lane == 0 && last >= 0) drain_bar(bar(kCBDone + (last & 1)), par(last));
  } else if (warp == kMathWarps + 1) {
    // =================== Yoff = C . [H hi | H lo]^T (N = 128); C and B tile loads
    auto load_cb = [&](int i) {
      const ChunkSrc s = chunk_src(i);
      load_tile(stage(i), s, &tm, use_tma != 0, ci.c_col, TN, bar(kFullCB + (i & 1)), lane);
      load_tile(stage(i) + kTileC, s, &tm, use_tma != 0, ci.b_col, TN, bar(kFullCB + (i & 1)), lane);
    };
    int loaded = min(n, 2), last = -1;
    for (int i = 0; i < loaded; ++i) load_cb(i);
    for (int i = 0; i < n; ++i) {
      if (!(warp_wait(bar(kFullCB + (i & 1)), par(i), s_abort) && warp_wait(bar(kHReady + (i & 1)), par(i), s_abort)))
        break;
      tc_fence_after();
      if (lane == 0) {
        const uint64_t a0 = sdesc(stage(i), 16, 1024), h0 = sdesc(sbase + kOffHT, TN * 128, 1024);
#pragma unroll
        for (int s2 = 0; s2 < TN / 16; ++s2) {
          const uint32_t ko = ((s2 >> 2) * TQ * 128 + (s2 & 3) * 32) >> 4;
          mma_ss(tmem + kColYo, a0 + ko, h0 + ((s2 * 2048) >> 4), idesc128(2 * TP, 0, 1), s2 > 0);
        }
        mma_commit(bar(kYoDone + (i & 1)));
        mbar_arrive(bar(kYoIssued + (i & 1)));
      }
      __syncwarp();
      last = i;
      if (i + 2 < n) {
        // chunk i's C and B tiles are spent once its three products are done
        if (!(warp_wait(bar(kYoDone + (i & 1)), par(i), s_abort) && warp_wait(bar(kCBDone + (i & 1)), par(i), s_abort) &&
              warp_wait(bar(kDHDone + (i & 1)), par(i), s_abort)))
          break;
        load_cb(i + 2);
        loaded = i + 3;
      }
    }
    if (lane == 0 && last >= 0) drain_bar(bar(kYoDone + (last & 1)), par(last));
    if (lane == 0 && *s_abort)
      for (int i = max(0, loaded - 2); i < loaded; ++i) drain_bar(bar(kFullCB + (i & 1)), par(i));
  } else if (warp == kMathWarps + 2) {
    // =================== dH^T = B^T . [X o w hi | lo] (N = 128)
    int last = -1;
    for (int i = 0; i < n; ++i) {
      if (!(warp_wait(bar(kFullCB + (i & 1)), par(i), s_abort) && warp_wait(bar(kXWReady + (i & 1)), par(i), s_abort) &&
            warp_wait(bar(kDHFree + (i & 1)), par(i), s_abort)))
        break;
      tc_fence_after();
      if (lane == 0) {
        // B operand [X o w hi | X o w lo]: two 64-column blocks 16 KB apart
        static_assert(kOffXWlo == kOffXWhi + kTileX, "X o w hi and lo must be adjacent");
        const uint64_t bt0 = sdesc(stage(i) + kTileC, TQ * 128, 1024);
        const uint64_t xw0 = sdesc(sbase + kOffXWhi, kTileX, 1024);
#pragma unroll
        for (int s2 = 0; s2 < TQ / 16; ++s2) {
          const uint32_t jk = (s2 * 2048) >> 4;  // 16 rows of the [j][*] tiles
          mma_ss(tmem + kColDH, bt0 + jk, xw0 + jk, idesc128(128, 1, 1), s2 > 0);
        }
        mma_commit(bar(kDHDone + (i & 1)));
      }
      __syncwarp();
      last = i;
    }
    if (lane == 0 && last >= 0) drain_bar(bar(kDHDone + (last & 1)), par(last));
  } else {
    // =================== Y = M . X (fp16; A = M from TMEM, 8 k-steps); X tile loads
    auto load_x = [&](int i) {
      load_tile(stage(i) + kTileC + kTileB, chunk_src(i), &tm, use_tma != 0, ci.x_col, TP, bar(kFullX + (i & 1)), lane);
    };
    int loaded = min(n, 2), last = -1;
    for (int i = 0; i < loaded; ++i) load_x(i);
    for (int i = 0; i < n; ++i) {
      // behind C . H^T(i) in the tensor pipe (the output needs both; C . H^T(i) is on the
      // state's critical loop)
      if (!(warp_wait(bar(kMReady + (i & 1)), par(i), s_abort) && warp_wait(bar(kXWReady + (i & 1)), par(i), s_abort) &&
            warp_wait(bar(kYoIssued + (i & 1)), par(i), s_abort)))
        break;
      tc_fence_after();
      if (lane == 0) {
        const uint64_t x0 = sdesc(stage(i) + kTileC + kTileB, TQ * 128, 1024);
        const uint32_t buf = tmem + 128u * (uint32_t)(i & 1);
#pragma unroll
        for (int s2 = 0; s2 < TQ / 16; ++s2)  // tokens [16 s2, 16 s2 + 16)
          mma_ts(buf + kColY, buf + kColM + m_col(s2), x0 + ((s2 * 2048) >> 4), idesc128(TP, 0, 1, 0), s2 > 0);
        mma_commit(bar(kYdDone + (i & 1)));
        mbar_arrive(bar(kYIssued + (i & 1)));
      }
      __syncwarp();
      last = i;
      if (i + 2 < n) {
        if (!warp_wait(bar(kYdDone + (i & 1)), par(i), s_abort)) break;  // chunk i's X tile spent
        load_x(i + 2);
        loaded = i + 3;
      }
    }
    if (lane == 0 && last >= 0) drain_bar(bar(kYdDone + (last & 1)), par(last));
    if (lane == 0 && *s_abort)
      for (int i = max(0, loaded - 2); i < loaded; ++i) drain_bar(bar(kFullX + (i & 1)), par(i));
  }

  // ---- teardown: every role has drained what it issued
  tc_fence_before();
  __syncthreads();
  const bool aborted = *s_abort != 0u;
  if (tid == 0 && aborted) atomicAdd(&g_tc_timeouts, 1u);
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" :: "r"(tmem));
  if (aborted) return;
  const bool s_warp = sw >= 0 && warp < kMathWarps;
  const bool write_slot = ci.k == ci.nseg - 1;
  float* slot_ptr = a.ssm_state + (int64_t)seq_slot(a.tab, ci.sq) * H * TP * TN + (int64_t)ci.h * TP * TN;
  if (*s_range == 0u) {
    // ---- state after the last chunk
    if (s_warp && live && write_slot) {
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        slot_ptr[(int64_t)(pc0 + 2 * e) * TN + s_row] = f2lo(hs[e]);
        slot_ptr[(int64_t)(pc0 + 2 * e + 1) * TN + s_row] = f2hi(hs[e]);
      }
    }
    return;
  }
  // A chunk whose fp16 operands would overflow: y of the whole segment again,
  // token by token. The final state waits in shared memory ([p][n] fp32 over the
  // H^T tiles), since the recomputation may read its seed from the slot.
  float* s_state = reinterpret_cast<float*>(smem + kOffHT);
  static_assert(TP * TN * 4 <= kTileHT, "final state fits over the H^T tiles");
  if (s_warp) {
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      s_state[(pc0 + 2 * e) * TN + s_row] = f2lo(hs[e]);
      s_state[(pc0 + 2 * e + 1) * TN + s_row] = f2hi(hs[e]);
    }
  }
  __syncthreads();
  full_pass_serial_y(a, ci, tid);
  __syncthreads();  // every seed has been read from the slot before it is overwritten
  if (write_slot)
    for (int e = tid; e < TP * TN; e += kFullThreads) slot_ptr[e] = s_state[e];
}

// State pass: end state (from zero; the first segment from the slot's state)
// and total log-decay of every segment but the last, for two heads of one
// group per CTA (heads 2 y and 2 y + 1; one head when the group has an odd
// number of heads). Chunks are read last to first; with R the log2 decay of
// the chunks already read, token j's weight is w_j = 2^(R + S_end - S_j) dt'_j
// (S the chunk's cumulative log2 decay, per head), so B^T . (X o w) of every
// chunk accumulates into the same TMEM columns.
//   warps 0-15  X o w (bf16 hi + lo) of both heads into TMEM (warp w: lanes of
//               quarter w % 4, tokens [32 (w / 4), +32)); at the end, the pieces' states
//   warp 16     X tile loads (two heads, three stages)
//   warp 17     B tile loads (three stages)
//   warp 18     D hi += (X o w hi)^T . B  (A from TMEM; M=128 N=128 K=128 per chunk)
//   warp 19     dt' and the token weights of both heads, up to two chunks ahead
//   warp 20     D lo += (X o w lo)^T . B  (the two accumulators are summed at the end;
//               one issuing thread per half, so the two halves' instructions overlap)
__global__ void __launch_bounds__(kStateThreads, 1)
ssd_tc_state(const __grid_constant__ ScanArgs a, const __grid_constant__ CUtensorMap tm, const int use_tma) {
  // CTA (b, y): piece q = b % P of segment b / P, an equal share of the segment's
  // chunks, for heads h0 = hpc y and h0 + 1; its entry (index b) is the piece's end
  // state from zero (the first piece of a sequence's first segment from the slot)
  // and total log-decay
  const int P = a.state_pieces > 0 ? a.state_pieces : 1;
  const int entry = blockIdx.x, q = entry % P;
  const int H = a.heads;
  const int hpc = ((H / a.ngroups) & 1) == 0 ? 2 : 1;  // heads per CTA (never across a group)
  const int h0 = hpc * (int)blockIdx.y;
  const int nh = hpc;                                   // heads this CTA writes
  Cta ci = cta_info(a, entry / P);
  ci.h = h0;
  ci.x_col = h0 * TP;
  ci.b_col = H * TP + (h0 / (H / a.ngroups)) * TN;  // both heads' group
  if (ci.k == ci.nseg - 1) return;  // the last segment has no entry (the full pass ends it)
  {
    // balanced shares: sizes differ by at most one chunk, none empty while P <= chunks
    const int nk = ci.c_end - ci.c_begin;
    const int pb = ci.c_begin + (int)((int64_t)q * nk / P), pe = ci.c_begin + (int)((int64_t)(q + 1) * nk / P);
    ci.c_begin = pb;
    ci.c_end = pe;
    ci.n = pe - pb;
  }
  const int x_col1 = (h0 + nh - 1) * TP;  // the second head's x columns (the first's again when one head)
  float A2h[2];
  A2h[0] = expf(a.A_log[h0]) * 1.4426950408889634f;
  A2h[1] = expf(a.A_log[h0 + nh - 1]) * 1.4426950408889634f;
  if (ci.n == 0) {  // an empty piece (only when a segment has fewer than P chunks): zero state, zero decay
    for (int hh = 0; hh < nh; ++hh) {
      float* dst = a.ws_state + ((int64_t)entry * H + h0 + hh) * TP * TN;
      for (int i = threadIdx.x; i < TP * TN; i += blockDim.x) dst[i] = 0.0f;
      if (threadIdx.x == 0) a.ws_decay[(int64_t)entry * H + h0 + hh] = 0.0f;
    }
    return;
  }
  extern __shared__ __align__(1024) unsigned char smem[];
  const uint32_t sbase = su32(smem);
  if ((sbase & 1023u) != 0) {  // the swizzled operand tiles need a 1024-byte aligned base
    if (threadIdx.x == 0) atomicAdd(&g_tc_timeouts, 1u);
    return;
  }
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kStOffMisc);
  volatile uint32_t* s_abort = reinterpret_cast<volatile uint32_t*>(smem + kStOffMisc + 4);
  float* s_w = reinterpret_cast<float*>(smem + kStOffW);
  float* s_R = reinterpret_cast<float*>(smem + kStOffR);
  auto bar = [&](int id) { return sbase + kStOffBar + 8u * (uint32_t)id; };
  auto stg_x = [&](int i) { return sbase + (uint32_t)(i % kStStages) * kStXStage; };
  auto stg_b = [&](int i) { return sbase + kStOffB + (uint32_t)(i % kStStages) * kTileB; };
  auto p2 = [](int i) { return (uint32_t)((i >> 1) & 1); };          // phase parity on a [2] barrier
  auto p3 = [](int i) { return (uint32_t)((i / kStStages) & 1); };   // phase parity on a [3] barrier

  const int n = ci.n;  // >= 1 here
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" :: "r"(su32(s_tmem)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == kMathThreads) {
    for (int b = 0; b < kStStages; ++b) {
      mbar_init(bar(kStFullX + b), 2);  // one tile per head
      mbar_init(bar(kStFullB + b), 1);
      mbar_init(bar(kStXFree + b), kMathWarps);
      mbar_init(bar(kStBFree + b), 2);  // one commit from each issuer
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(kStXWReady + b), kMathWarps);
      mbar_init(bar(kStDHDone + b), 2);
      mbar_init(bar(kStWReady + b), 1);
    }
    *s_abort = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  // Launched as a programmatic dependent of the dt' pre-pass: the tile loaders
  // (warps 16, 17) and the product issuer start at once; the weight producer
  // (dt') and the element-wise warps (the slot) wait.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // the full pass may be scheduled
  if (warp < kMathWarps || warp == kMathWarps + 3) asm volatile("griddepcontrol.wait;" ::: "memory");

  // local chunk i is chunk c_end - 1 - i
  auto chunk_src = [&](int i) {
    ChunkSrc s;
    const int c = ci.c_end - 1 - i;
    s.xbc = static_cast<const __nv_bfloat16*>(a.xbc);
    s.ld = a.conv_dim;
    s.rb = ci.row0 + (int64_t)c * TQ;
    s.len = min(TQ, ci.T - c * TQ);
    return s;
  };

  if (warp < kMathWarps) {
    // =================== X o w of every chunk into TMEM (lane = p: head 0's columns in
    // lane quarters 0-1, head 1's in 2-3; warp group tg takes tokens [32 tg, +32)),
    // then the pieces' states
    const int qrt = warp & 3, tg = warp >> 2;
    const int hq = qrt >> 1, p = 32 * (qrt & 1) + lane;
    const uint32_t lane_off = (uint32_t)(qrt * 32) << 16;
    bool live = true;
    for (int i = 0; i < n; ++i) {
      if (!(warp_wait(bar(kStFullX + i % kStStages), p3(i), s_abort) &&
            warp_wait(bar(kStWReady + (i & 1)), p2(i), s_abort) &&
            (i < 2 || warp_wait(bar(kStDHDone + (i & 1)), p2(i - 2), s_abort)))) {  // TMEM stage i % 2 read
        live = false;
        break;
      }
      const unsigned char* xt = smem + (uint32_t)(i % kStStages) * kStXStage + (uint32_t)hq * kTileX;
      const float* w = s_w + ((i & 1) * 2 + hq) * TQ;
      uint32_t hw[16], lw[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int j = 32 * tg + 2 * k;
        const float x0 = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(xt + tile_off(j, p, TQ)));
        const float x1 = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(xt + tile_off(j + 1, p, TQ)));
        split2(x0 * w[j], x1 * w[j + 1], hw[k], lw[k]);
      }
      fence_async_smem();  // the X tile's reads come before its refill
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kStXFree + i % kStStages));
      const uint32_t ta = tmem + lane_off + kStColXW + 128u * (uint32_t)(i & 1) + 16u * (uint32_t)tg;
      asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                   :: "r"(ta), "r"(hw[0]), "r"(hw[1]), "r"(hw[2]), "r"(hw[3]), "r"(hw[4]), "r"(hw[5]), "r"(hw[6]),
                      "r"(hw[7]), "r"(hw[8]), "r"(hw[9]), "r"(hw[10]), "r"(hw[11]), "r"(hw[12]), "r"(hw[13]),
                      "r"(hw[14]), "r"(hw[15]) : "memory");
      asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                   :: "r"(ta + 64u), "r"(lw[0]), "r"(lw[1]), "r"(lw[2]), "r"(lw[3]), "r"(lw[4]), "r"(lw[5]), "r"(lw[6]),
                      "r"(lw[7]), "r"(lw[8]), "r"(lw[9]), "r"(lw[10]), "r"(lw[11]), "r"(lw[12]), "r"(lw[13]),
                      "r"(lw[14]), "r"(lw[15]) : "memory");
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kStXWReady + (i & 1)));
    }
    if (live && warp_wait(bar(kStDHDone + ((n - 1) & 1)), p2(n - 1), s_abort)) {
      tc_fence_after();
      // D row p (this lane), columns n = [32 tg, +32): hi + lo
      float dsum[32];
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        float dhi[16], dlo[16];
        tmem_ld16x2(tmem + lane_off + kStColDHi + 32u * (uint32_t)tg + 16u * (uint32_t)g,
                    tmem + lane_off + kStColDLo + 32u * (uint32_t)tg + 16u * (uint32_t)g, dhi, dlo);
#pragma unroll
        for (int e = 0; e < 16; ++e) dsum[16 * g + e] = dhi[e] + dlo[e];
      }
      if (hq < nh) {
        const int h = h0 + hq;
        const float Rt = s_R[hq];  // written before the weights of the last chunk were published
        const int64_t head_off = (int64_t)h * TP * TN, row_off = (int64_t)p * TN + 32 * tg;
        float* dst = a.ws_state + (int64_t)entry * H * TP * TN + head_off + row_off;
        if (ci.k == 0 && q == 0 && !ci.fresh) {
          // the first piece starts from the slot's state: add its decayed share, and
          // leave a copy of it for the full pass (whose last segment overwrites the slot)
          // in the first entry of the last segment, which has no entries of its own
          const float d = ex2(Rt);
          const float* slot_ptr = a.ssm_state + (int64_t)seq_slot(a.tab, ci.sq) * H * TP * TN + head_off + row_off;
          float* copy = a.ws_state + (int64_t)((ci.seg0 + ci.nseg - 1) * P) * H * TP * TN + head_off + row_off;
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float4 hv = *reinterpret_cast<const float4*>(slot_ptr + e);
            *reinterpret_cast<float4*>(copy + e) = hv;
            *reinterpret_cast<float4*>(dst + e) = make_float4(fmaf(d, hv.x, dsum[e]), fmaf(d, hv.y, dsum[e + 1]),
                                                              fmaf(d, hv.z, dsum[e + 2]), fmaf(d, hv.w, dsum[e + 3]));
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(dst + e) = make_float4(dsum[e], dsum[e + 1], dsum[e + 2], dsum[e + 3]);
        }
      }
      if (tid == 0)
        for (int hh = 0; hh < nh; ++hh) a.ws_decay[(int64_t)entry * H + h0 + hh] = s_R[hh] * 0.6931471805599453f;
    }
  } else if (warp == kMathWarps) {
    // =================== X tile loads of both heads: stage i % 3 is free once X o w of chunk i - 3 is formed
    int loaded = 0;
    for (int i = 0; i < n; ++i) {
      if (i >= kStStages && !warp_wait(bar(kStXFree + i % kStStages), p3(i - kStStages), s_abort)) break;
      load_tile(stg_x(i), chunk_src(i), &tm, use_tma != 0, ci.x_col, TP, bar(kStFullX + i % kStStages), lane);
      load_tile(stg_x(i) + kTileX, chunk_src(i), &tm, use_tma != 0, x_col1, TP, bar(kStFullX + i % kStStages), lane);
      loaded = i + 1;
    }
    if (lane == 0 && *s_abort)
      for (int i = max(0, loaded - kStStages); i < loaded; ++i) drain_bar(bar(kStFullX + i % kStStages), p3(i));
  } else if (warp == kMathWarps + 1) {
    // =================== B tile loads: stage i % 3 is free once the products of chunk i - 3 are done
    int loaded = 0;
    for (int i = 0; i < n; ++i) {
      if (i >= kStStages && !warp_wait(bar(kStBFree + i % kStStages), p3(i - kStStages), s_abort)) break;
      load_tile(stg_b(i), chunk_src(i), &tm, use_tma != 0, ci.b_col, TN, bar(kStFullB + i % kStStages), lane);
      loaded = i + 1;
    }
    if (lane == 0 && *s_abort)
      for (int i = max(0, loaded - kStStages); i < loaded; ++i) drain_bar(bar(kStFullB + i % kStStages), p3(i));
  } else if (warp == kMathWarps + 2 || warp == kMathWarps + 4) {
    // =================== D += (X o w)^T . B, the hi part from one thread and the lo
    // part from another (two accumulators, summed at the end)
    if (lane == 0) {
      const bool lo = warp == kMathWarps + 4;
      const uint32_t dcol = lo ? kStColDLo : kStColDHi, acol = kStColXW + (lo ? 64u : 0u);
      int last = -1;
      for (int i = 0; i < n; ++i) {
        if (!wait_bar(bar(kStFullB + i % kStStages), p3(i), s_abort)) break;
        if (!wait_bar(bar(kStXWReady + (i & 1)), p2(i), s_abort)) break;
        tc_fence_after();
        const uint64_t b0 = sdesc(stg_b(i), TQ * 128, 1024);
        const uint32_t a0 = tmem + acol + 128u * (uint32_t)(i & 1);
#pragma unroll
        for (int s2 = 0; s2 < TQ / 16; ++s2)
          mma_ts(tmem + dcol, a0 + 8u * (uint32_t)s2, b0 + ((s2 * 2048) >> 4), idesc128(TN, 0, 1),
                 (i > 0 || s2 > 0) ? 1u : 0u);
        mma_commit(bar(kStDHDone + (i & 1)));
        mma_commit(bar(kStBFree + i % kStStages));
        last = i;
      }
      if (last >= 0) drain_bar(bar(kStDHDone + (last & 1)), p2(last));
    }
  } else {
    // =================== dt' and token weights of chunk i, both heads, into buffer
    // i % 2 (lane l: tokens 4l .. 4l+3); buffer i % 2 last served chunk i-2
    const int64_t rows_all = a.tab.cu[a.tab.n];
    auto load_dtp = [&](int i, int h) {
      DtQuad r = {{0.f, 0.f, 0.f, 0.f}};
      if (i < n) {
        const int c = ci.c_end - 1 - i, len = min(TQ, ci.T - c * TQ);
        const float* src = a.dtp + (int64_t)h * rows_all + ci.row0 + (int64_t)c * TQ;
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (4 * lane + e < len) r.v[e] = src[4 * lane + e];
      }
      return r;
    };
    const int hB = h0 + nh - 1;
    float R[2] = {0.f, 0.f};  // log2 decay from the end of the chunks already read to the piece's end
    DtQuad a0 = load_dtp(0, h0), a1 = load_dtp(1, h0), b0 = load_dtp(0, hB), b1 = load_dtp(1, hB);
    for (int i = 0; i < n; ++i) {
      if (i >= 2 && !warp_wait(bar(kStXWReady + (i & 1)), p2(i - 2), s_abort)) break;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const DtQuad& r = hh == 0 ? a0 : b0;
        float dp[4], S[4], run = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          dp[e] = r.v[e];
          run -= A2h[hh] * dp[e];
          S[e] = run;
        }
        const float incl = warp_incl_sum(run, lane);
        const float tot = __shfl_sync(0xffffffffu, incl, 31);
        const float base = R[hh] + (tot - (incl - run));  // R + S_end - (S before this lane's tokens)
        *reinterpret_cast<float4*>(s_w + ((i & 1) * 2 + hh) * TQ + 4 * lane) = make_float4(
            ex2(base - S[0]) * dp[0], ex2(base - S[1]) * dp[1], ex2(base - S[2]) * dp[2], ex2(base - S[3]) * dp[3]);
        R[hh] += tot;
      }
      a0 = a1;
      b0 = b1;
      a1 = load_dtp(i + 2, h0);
      b1 = load_dtp(i + 2, hB);
      if (i == n - 1 && lane == 0) {
        s_R[0] = R[0];
        s_R[1] = R[1];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kStWReady + (i & 1)));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *s_abort) atomicAdd(&g_tc_timeouts, 1u);
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" :: "r"(tmem));
}

// Tensor map over xbc [rows][conv_dim] bf16: boxes of 64 columns x TQ rows,
// 128-byte swizzle. False when TMA cannot address it (base not 16-byte
// aligned, row stride not a multiple of 16 bytes, or no driver entry point):
// the kernels then load every tile with cp.async.
bool make_xbc_map(CUtensorMap* tm, const ScanArgs& a) {
  using Encode = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static Encode encode = []() -> Encode {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<Encode>(fn);
  }();
  const uint64_t rows = (uint64_t)a.tab.cu[a.tab.n];
  if (!encode || rows == 0 || (reinterpret_cast<uintptr_t>(a.xbc) & 15u) != 0 || (a.conv_dim * 2) % 16 != 0) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)a.conv_dim, rows};
  const cuuint64_t strides[1] = {(cuuint64_t)a.conv_dim * 2};
  const cuuint32_t box[2] = {64, TQ};
  const cuuint32_t estr[2] = {1, 1};
  return encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.xbc), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

unsigned int read_device_timeouts() {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_tc_timeouts, sizeof v) != cudaSuccess) return 0xffffffffu;
  return v;
}

// A launch as a programmatic dependent of the previous kernel on the stream: it
// may be scheduled while that kernel runs, and waits (griddepcontrol.wait)
// before it touches what that kernel writes.
template <typename Kern>
cudaError_t launch_dependent(Kern kern, dim3 grid, int threads, size_t smem, cudaStream_t st, const ScanArgs& a,
                             const CUtensorMap& tm, int use_tma) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a, tm, use_tma);
}

cudaError_t launch_scan_tc(const ScanArgs& a, cudaStream_t st) {
  const int segs = a.tab.tile[a.tab.n];
  if (segs == 0) return cudaSuccess;
  CUtensorMap tm;
  memset(&tm, 0, sizeof tm);
  const int use_tma = make_xbc_map(&tm, a) ? 1 : 0;
  const int rows = a.tab.cu[a.tab.n];
  if (rows > 0) {
    if (a.heads <= kDtRowsMaxHeads) {
      const size_t dsm = sizeof(float) * (size_t)a.heads * (kDtRows + 1);
      if (dsm > 48 * 1024) {
        const cudaError_t ea = cudaFuncSetAttribute(dt_prime_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dsm);
        if (ea != cudaSuccess) return ea;
      }
      dt_prime_rows_kernel<<<(unsigned)((rows + kDtRows - 1) / kDtRows), 256, dsm, st>>>(
          static_cast<const __nv_bfloat16*>(a.dt), a.dt_bias, a.dtp, rows, a.heads);
    } else {
      const dim3 pg((unsigned)((rows + 31) / 32), (unsigned)((a.heads + 31) / 32));
      dt_prime_kernel<<<pg, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(a.dt), a.dt_bias, a.dtp, rows, a.heads);
    }
    const cudaError_t e0 = cudaGetLastError();
    if (e0 != cudaSuccess) return e0;
  }
  const dim3 grid((unsigned)segs, (unsigned)a.heads);
  bool segmented = false;
  for (int i = 0; i < a.tab.n; ++i) segmented |= (a.tab.tile[i + 1] - a.tab.tile[i]) > 1;
  if (segmented) {
    cudaError_t e = cudaFuncSetAttribute(ssd_tc_state, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kStateSmem);
    if (e != cudaSuccess) return e;
    // two heads of one group per CTA (one when a group has an odd number of heads)
    const int hpc = ((a.heads / a.ngroups) & 1) == 0 ? 2 : 1;
    const dim3 sgrid((unsigned)(segs * (a.state_pieces > 0 ? a.state_pieces : 1)), (unsigned)(a.heads / hpc));
    e = launch_dependent(ssd_tc_state, sgrid, kStateThreads, kStateSmem, st, a, tm, use_tma);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = cudaFuncSetAttribute(ssd_tc_full, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFullSmem);
  if (e != cudaSuccess) return e;
  return launch_dependent(ssd_tc_full, grid, kFullThreads, kFullSmem, st, a, tm, use_tma);
}

}  // namespace mamba2
