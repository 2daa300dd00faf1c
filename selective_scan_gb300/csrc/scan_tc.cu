// Chunked selective scan on the 5th-generation tensor cores (tcgen05, TMEM)
// for headdim 64 x d_state 128 with bf16 activations.
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
//   y_t   = exp(s_t) C_t . h_in + sum_{j<=t} (C_t . B_j) exp(s_t - s_j) dt'_j x_j + D x_t
//   h_out = exp(s_{Q-1}) h_in + sum_j exp(s_{Q-1} - s_j) dt'_j x_j (x) B_j
// (every exponent a difference taken in the <= 0 direction).
//
// One CTA of 8 warps per (sequence segment, head); TMEM lane t = token row t
// (or state row n). Per chunk, with every tile in its natural load layout
// (a [rows][cols] bf16 tile stored with the 128-byte swizzle in 64-column
// blocks is both the K-major and the MN-major tcgen05 operand):
//   MMA batch 1:
//     CB      = C . B^T                       M=128 N=128 K=128 (C, B K-major)
//     Yoff    = C . H^T                       M=128 N=64  K=128 (H^T MN-major)
//     dH^T    = B^T . (X o w)  (hi + lo)      M=128 N=64  K=128 (both MN-major)
//   threads: M = CB o exp(s_t - s_j) dt'_j (j <= t), split bf16 hi + lo into
//            TMEM (A operand); H^T = exp(s_{Q-1}) H^T + dH^T kept in fp32
//            registers, its bf16 copy written to smem for the next chunk
//   MMA batch 2:  Y = M . X  (A from TMEM)    M=128 N=64  K=128 (X MN-major)
//   threads: y = Y + exp(s_t) Yoff + D x  -> bf16 -> HBM
// M and X o w are carried as bf16 hi + lo (about 16 mantissa bits): with a
// single bf16 M the worst y error reaches 1.4x its tolerance, and a single
// bf16 X o w gives a state error of 1.7e-3 against a 1e-3 tolerance
// (measured on the 130m, varlen and 65 536-token workloads). A single bf16
// copy of H costs y less than 5 % of its tolerance, so H is not split.
//
// Long runs are cut into segments; a state pass (kFull = false: only the
// dH^T products) computes each segment's end state from zero and its total
// log-decay, and the full pass seeds segment k by folding the earlier
// segments' entries (see the scan entry point). Waits on the MMA-completion
// mbarriers are bounded: on a timeout the kernel records it in a device
// counter (mamba2_device_timeouts), stops issuing work, frees its TMEM and
// returns.
#include "common.cuh"

namespace mamba2 {

__device__ unsigned int g_tc_timeouts = 0;

namespace {

constexpr int TQ = 128;  // tokens per chunk
constexpr int TP = 64;   // headdim
constexpr int TN = 128;  // d_state
constexpr int kTcThreads = 512;  // 16 warps: 4 per TMEM lane quarter
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kWaitLimit = 1u << 22;  // try_wait rounds before giving up (far above a healthy MMA batch)

// TMEM column map (128 lanes each)
constexpr uint32_t kColCB = 0;     // [0,128)   C . B^T (fp32)
constexpr uint32_t kColMhi = 128;  // [128,192) M hi (bf16 pairs)
constexpr uint32_t kColMlo = 192;  // [192,256) M lo
constexpr uint32_t kColYo = 256;   // [256,384) C . H^T (fp32), two buffers of 64 (chunk parity)
constexpr uint32_t kColDH = 384;   // [384,448) B^T . (X o w) (fp32, lane = n)
constexpr uint32_t kColYd = 448;   // [448,512) M . X (fp32)

// Shared memory plan (bytes). Operand tiles are 1024-byte aligned.
constexpr uint32_t kTileC = TQ * TN * 2;  // 32 KB  [t][n]
constexpr uint32_t kTileB = TQ * TN * 2;  // 32 KB  [j][n]
constexpr uint32_t kTileX = TQ * TP * 2;  // 16 KB  [j][p]
constexpr uint32_t kStage = kTileC + kTileB + kTileX;  // 80 KB per input stage
constexpr uint32_t kOffIn = 0;                          // 2 stages; a spent C tile stages y
constexpr uint32_t kOffXWhi = 2 * kStage;               // (X o w) hi [j][p]
constexpr uint32_t kOffXWlo = kOffXWhi + kTileX;
constexpr uint32_t kOffHT = kOffXWlo + kTileX;          // H^T (bf16) [n][p]
constexpr uint32_t kOffS = kOffHT + TN * TP * 2;        // float s2[2][TQ]  (log2e * cumulative log-decay)
constexpr uint32_t kOffDtp = kOffS + 2 * TQ * 4;        // float dtp[2][TQ]
constexpr uint32_t kOffV = kOffDtp + 2 * TQ * 4;        // float v[2][TQ]
constexpr uint32_t kOffMisc = kOffV + 2 * TQ * 4;       // mbarriers, tmem base
constexpr uint32_t kSmemBytes = kOffMisc + 64 + 1024;  // + slack to align the base to 1024 bytes
static_assert(kSmemBytes <= 232448, "shared memory plan exceeds 227 KB");

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// byte offset of element (r, c) in a [R][cols] bf16 tile, 128-byte swizzle,
// 64-column blocks of R rows each
__device__ __forceinline__ uint32_t tile_off(int r, int c, int R) {
  return (uint32_t)((c >> 6) * R * 128 + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) + (c & 7) * 2);
}

__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// kind::f16 instruction descriptor: D f32, A/B bf16, M = 128
__host__ __device__ constexpr uint32_t idesc128(int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
               :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
               :: "r"(d), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void mma_commit(uint32_t mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" :: "r"(mbar) : "memory");
}
// Bounded wait for the mbarrier phase; false on timeout.
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t phase) {
  for (uint32_t it = 0; it < kWaitLimit; ++it) {
    uint32_t done;
    asm volatile("{\n.reg .pred P;\nmbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\nselp.u32 %0, 1, 0, P;\n}\n"
                 : "=r"(done) : "r"(mbar), "r"(phase) : "memory");
    if (done) return true;
  }
  return false;
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                 "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
               :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
                  "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
               : "memory");
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

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0));
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// two 16-column loads, one wait
__device__ __forceinline__ void tmem_ld16x2(uint32_t ta, uint32_t tb, float (&va)[16], float (&vb)[16]) {
  uint32_t r[32];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                 "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
               : "r"(ta));
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
               : "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
                 "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
                 "=r"(r[30]), "=r"(r[31])
               : "r"(tb));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    va[i] = __uint_as_float(r[i]);
    vb[i] = __uint_as_float(r[16 + i]);
  }
}

template <bool kFull>
__global__ void __launch_bounds__(kTcThreads, 1)
ssd_tc_kernel(const __grid_constant__ ScanArgs a) {
  extern __shared__ unsigned char smem_raw[];
  // operand tiles need a 1024-byte aligned base (the swizzle keys on address bits 7-9)
  const uint32_t raw_base = su32(smem_raw);
  unsigned char* smem = smem_raw + (((raw_base + 1023u) & ~1023u) - raw_base);
  const uint32_t sbase = su32(smem);
  float* s_s2 = reinterpret_cast<float*>(smem + kOffS);    // [2][TQ] log2e * cumulative log-decay
  float* s_dtp = reinterpret_cast<float*>(smem + kOffDtp); // [2][TQ] dt'
  float* s_v = reinterpret_cast<float*>(smem + kOffV);     // [2][TQ] exp(s_e - s_j) dt'_j, e = end of j's 32-block
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kOffMisc + 8);
  const uint32_t mbar1 = sbase + kOffMisc + 16, mbar2 = sbase + kOffMisc + 24;

  const int seg = blockIdx.x, h = blockIdx.y;
  const int sq = find_tile_seq(a.tab, seg);
  const int seg0 = a.tab.tile[sq];
  const int k = seg - seg0;
  const int nseg = a.tab.tile[sq + 1] - seg0;
  if (!kFull && k == nseg - 1) return;  // the state pass skips last segments

  const int H = a.heads, G = a.ngroups;
  const int g = h / (H / G);
  const int row0 = a.tab.cu[sq];
  const int T = a.tab.cu[sq + 1] - row0;
  const int nchunks = (T + TQ - 1) / TQ;
  const int c_begin = k * a.seg_chunks;
  const int c_end = min(nchunks, c_begin + a.seg_chunks);
  const bool fresh = seq_fresh(a.tab, sq);
  const int64_t ld = a.conv_dim;
  const __nv_bfloat16* xbc = static_cast<const __nv_bfloat16*>(a.xbc);
  const __nv_bfloat16* dtg = static_cast<const __nv_bfloat16*>(a.dt);
  const int x_col = h * TP, b_col = H * TP + g * TN, c_col = H * TP + G * TN + g * TN;
  const float A2 = expf(a.A_log[h]) * 1.4426950408889634f;  // decay rate in log2 units
  const float dtb = a.dt_bias[h];
  const float Dh = a.D[h];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = tid & 127;   // TMEM lane = tile row this thread works on
  const int cg = tid >> 7;     // column group 0..3 (warps 4 cg .. 4 cg + 3)
  const int qrt = warp & 3;    // TMEM lane quarter = 32-row block of `row`
  const uint32_t lane_off = (uint32_t)(qrt * 32) << 16;

  // ---- TMEM allocation (warp 0), barriers (thread 0)
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" :: "r"(su32(s_tmem)), "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(mbar1), "r"(kFull ? 2 : 1));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 2;" :: "r"(mbar2));
    asm volatile("fence.mbarrier_init.release.cluster;");
  }

  // ---- running state: this thread holds H^T[n = row][p], p in [16 cg, 16 cg + 16)
  const int64_t head_off = (int64_t)h * TP * TN;
  float* slot_ptr = a.ssm_state + (int64_t)seq_slot(a.tab, sq) * H * TP * TN + head_off;
  auto ws_entry = [&](int segidx) -> float* { return a.ws_state + (int64_t)segidx * H * TP * TN + head_off; };
  float hst[16];
  auto load_state = [&](const float* src) {
#pragma unroll
    for (int i = 0; i < 16; ++i) hst[i] = src ? src[(int64_t)(16 * cg + i) * TN + row] : 0.0f;
  };
  auto store_state = [&](float* dst) {
#pragma unroll
    for (int i = 0; i < 16; ++i) dst[(int64_t)(16 * cg + i) * TN + row] = hst[i];
  };
  if (k == 0) {
    const float* src = fresh ? nullptr : ((kFull && nseg > 1) ? ws_entry(seg0 + nseg - 1) : slot_ptr);
    load_state(src);
    if (!kFull && !fresh) store_state(ws_entry(seg0 + nseg - 1));  // seed copy for the full pass
  } else if (!kFull) {
    load_state(nullptr);
  } else {
    load_state(ws_entry(seg0));
    for (int j = 1; j < k; ++j) {
      const float d = __expf(a.ws_decay[(int64_t)(seg0 + j) * H + h]);
      const float* e = ws_entry(seg0 + j);
      float ev[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) ev[i] = e[(int64_t)(16 * cg + i) * TN + row];
#pragma unroll
      for (int i = 0; i < 16; ++i) hst[i] = fmaf(d, hst[i], ev[i]);
    }
  }
  // bf16 copy of H^T (B operand of C . H^T): row n, columns [16 cg, +16)
  auto state_to_smem = [&]() {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      uint32_t hw[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) hw[e] = pack2(hst[8 * q + 2 * e], hst[8 * q + 2 * e + 1]);
      *reinterpret_cast<uint4*>(smem + kOffHT + tile_off(row, 16 * cg + 8 * q, TN)) =
          make_uint4(hw[0], hw[1], hw[2], hw[3]);
    }
  };

  // ---- chunk loads: cp.async 16-byte pieces into the swizzled tiles (zero past the run)
  auto issue_chunk = [&](int c, int stage) {
    const int len = min(TQ, T - c * TQ);
    const int64_t rb = row0 + (int64_t)c * TQ;
    const uint32_t st = sbase + kOffIn + stage * kStage;
    for (int i = tid; i < TQ * (TN / 8); i += kTcThreads) {  // B and C: 16 pieces per row
      const int t = i >> 4, pc = i & 15;
      const bool ok = t < len;
      const int64_t grow = ok ? rb + t : row0;
      const uint32_t o = tile_off(t, pc * 8, TQ);
      cp_async16(st + kTileC + o, xbc + grow * ld + b_col + pc * 8, ok);
      if (kFull) cp_async16(st + o, xbc + grow * ld + c_col + pc * 8, ok);
    }
    for (int i = tid; i < TQ * (TP / 8); i += kTcThreads) {  // x: 8 pieces per row
      const int t = i >> 3, pc = i & 7;
      const bool ok = t < len;
      const int64_t grow = ok ? rb + t : row0;
      cp_async16(st + kTileC + kTileB + tile_off(t, pc * 8, TQ), xbc + grow * ld + x_col + pc * 8, ok);
    }
    asm volatile("cp.async.commit_group;\n" ::);
  };
  // ---- dt of a chunk: warps 0, 4, 8, 12 (TMEM lane quarter 0, the lightest M
  // share), warp 4k taking the 32-block k (lane l: token 32 k + l)
  const bool dt_warp = (warp & 3) == 0;
  const int dblk = warp >> 2;
  float* s_btot = reinterpret_cast<float*>(smem + kOffMisc + 32);  // [2][4] block totals of the log2 decay
  // raw bf16 bits: the load stays in flight until the next chunk's dt phase converts it
  unsigned short dt_raw = 0;
  auto load_dt = [&](int c) {
    const int t = 32 * dblk + lane;
    dt_raw = t < min(TQ, T - c * TQ) ? reinterpret_cast<const unsigned short*>(dtg)[(row0 + (int64_t)c * TQ + t) * H + h]
                                     : (unsigned short)0;
  };
  // dt', log2-scaled cumulative decay S and block-relative factors v of chunk c into buffer sb
  auto dt_phase = [&](int c, int sb) {
    const int t = 32 * dblk + lane;
    const float dp = t < min(TQ, T - c * TQ) ? softplus_f(__uint_as_float((uint32_t)dt_raw << 16) + dtb) : 0.f;
    float incl = -A2 * dp;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) s_btot[sb * 4 + dblk] = incl;
    asm volatile("bar.sync 1, 128;" ::: "memory");  // the four dt warps
    float pre = 0.f;
    for (int k2 = 0; k2 < dblk; ++k2) pre += s_btot[sb * 4 + k2];
    const float S = pre + incl;
    const float Se = __shfl_sync(0xffffffffu, S, 31);  // S at the end of this 32-block
    s_s2[sb * TQ + t] = S;
    s_dtp[sb * TQ + t] = dp;
    s_v[sb * TQ + t] = ex2(Se - S) * dp;
  };
  // (X o w) hi + lo of the chunk in `stage`, row j = row, columns [16 cg, +16)
  auto xw_phase = [&](int stage, int sb) {
    const float tot2 = s_s2[sb * TQ + TQ - 1];
    const float wj = ex2(tot2 - s_s2[sb * TQ + row]) * s_dtp[sb * TQ + row];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint32_t o = tile_off(row, 16 * cg + 8 * q, TQ);
      const uint4 xv = *reinterpret_cast<const uint4*>(smem + kOffIn + stage * kStage + kTileC + kTileB + o);
      const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        split2(__uint_as_float(xw[e] << 16) * wj, __uint_as_float(xw[e] & 0xffff0000u) * wj, hi[e], lo[e]);
      *reinterpret_cast<uint4*>(smem + kOffXWhi + o) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(smem + kOffXWlo + o) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
  };
  // ---- MMA issue. Four independent streams, each from lane 0 of a warp whose
  // M share is the lightest (TMEM lane quarter 0): an issuing thread waits out each
  // MMA, so separate issuers let the streams overlap on the tensor pipe.
  // Descriptors are precomputed bases plus constant offsets (a descriptor's address
  // field is the byte address / 16, and shared addresses stay below 2^18).
  uint32_t tmem = 0;  // TMEM base, read after the allocation barrier below
  constexpr int kIssYd = 0, kIssYo = 128, kIssCB = 256, kIssDH = 384;  // issuing threads
  auto stage_addr = [&](int stage) { return sbase + kOffIn + stage * kStage; };
  auto issue_cb = [&](int stage) {  // CB = C . B^T
    const uint64_t a0 = sdesc(stage_addr(stage), 16, 1024), b0 = sdesc(stage_addr(stage) + kTileC, 16, 1024);
#pragma unroll
    for (int s2 = 0; s2 < TN / 16; ++s2) {
      const uint32_t ko = ((s2 >> 2) * TQ * 128 + (s2 & 3) * 32) >> 4;
      mma_ss(tmem + kColCB, a0 + ko, b0 + ko, idesc128(128, 0, 0), s2 > 0);
    }
  };
  auto issue_dh = [&](int stage) {  // dH^T = B^T . (X o w), hi then lo
    const uint64_t bt0 = sdesc(stage_addr(stage) + kTileC, TQ * 128, 1024);
    const uint64_t hi0 = sdesc(sbase + kOffXWhi, TQ * 128, 1024), lo0 = sdesc(sbase + kOffXWlo, TQ * 128, 1024);
#pragma unroll
    for (int s2 = 0; s2 < TQ / 16; ++s2) {
      const uint32_t jk = (s2 * 2048) >> 4;  // 16 rows of the [j][*] tiles
      mma_ss(tmem + kColDH, bt0 + jk, hi0 + jk, idesc128(64, 1, 1), s2 > 0);
      mma_ss(tmem + kColDH, bt0 + jk, lo0 + jk, idesc128(64, 1, 1), 1);
    }
  };
  auto issue_yo = [&](int stage, int yb) {  // Yoff = C . H^T into Yo buffer yb
    const uint64_t a0 = sdesc(stage_addr(stage), 16, 1024), h0 = sdesc(sbase + kOffHT, TN * 128, 1024);
#pragma unroll
    for (int s2 = 0; s2 < TN / 16; ++s2) {
      const uint32_t ko = ((s2 >> 2) * TQ * 128 + (s2 & 3) * 32) >> 4;
      mma_ss(tmem + kColYo + 64 * yb, a0 + ko, h0 + ((s2 * 2048) >> 4), idesc128(64, 0, 1), s2 > 0);
    }
  };
  auto issue_yd = [&](int stage) {  // Y = M . X (A = M hi, lo from TMEM)
    const uint64_t x0 = sdesc(stage_addr(stage) + kTileC + kTileB, TQ * 128, 1024);
#pragma unroll
    for (int s2 = 0; s2 < TQ / 16; ++s2) {
      const uint64_t xd = x0 + ((s2 * 2048) >> 4);
      mma_ts(tmem + kColYd, tmem + kColMhi + s2 * 8, xd, idesc128(64, 0, 1), s2 > 0);
      mma_ts(tmem + kColYd, tmem + kColMlo + s2 * 8, xd, idesc128(64, 0, 1), 1);
    }
  };
  // block-wide barrier with the TMEM / async-proxy fences around it
  auto tc_sync = [&]() {
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  };

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  tmem = *s_tmem;

  float seg_logdecay = 0.f;
  uint32_t ph1 = 0, ph2 = 0;
  bool ok_run = true;

  // ---- prologue: chunk c_begin's loads, dt, (X o w), and its first MMAs
  if (c_begin < c_end) {
    issue_chunk(c_begin, 0);
    if (c_begin + 1 < c_end) issue_chunk(c_begin + 1, 1);
    if (dt_warp) {
      load_dt(c_begin);
      dt_phase(c_begin, 0);
      if (c_begin + 1 < c_end) load_dt(c_begin + 1);
    }
    if (kFull) state_to_smem();
    if (c_begin + 1 < c_end) asm volatile("cp.async.wait_group 1;\n" ::: "memory");
    else asm volatile("cp.async.wait_group 0;\n" ::: "memory");
    __syncthreads();
    xw_phase(0, 0);
    tc_sync();
    if (kFull && tid == kIssCB) {
      issue_cb(0);
      mma_commit(mbar1);
    }
    if (tid == kIssDH) {
      issue_dh(0);
      mma_commit(mbar1);
    }
    if (kFull && tid == kIssYo) issue_yo(0, 0);  // completion covered by this thread's next commit
  }

  for (int c = c_begin; c < c_end; ++c) {
    const int st = (c - c_begin) & 1;  // stage, decay-array buffer and Yo buffer of chunk c
    const int len = min(TQ, T - c * TQ);
    const bool more = c + 1 < c_end;
    // (1) CB(c), dH(c) (and Yoff(c)) complete
    if (!__syncthreads_and(mbar_wait(mbar1, ph1))) {
      if (tid == 0) atomicAdd(&g_tc_timeouts, 1u);
      ok_run = false;
      break;
    }
    ph1 ^= 1u;
    tc_fence_after();
    const float tot2 = s_s2[st * TQ + TQ - 1];

    // (2) M(c) into TMEM; H(c) = exp(total) H(c-1) + dH(c); the dt warps also prepare chunk c+1's decays
    if (kFull) {
      // M = CB o exp(s_t - s_j) dt'_j (j <= t) for row t = row. This thread takes
      // columns 32 bb + 8 cg .. +7 of each 32-column block bb, so every warp gets
      // the same mix of blocks: above the diagonal all zero; below it
      // exp(s_t - s_j) = exp(s_t - s_e) exp(s_e - s_j) with e the block's last
      // token (both factors <= 1, the second times dt'_j being v_j); the
      // diagonal block exponentiates each pair.
      const float* S2 = s_s2 + st * TQ;
      const float* DP = s_dtp + st * TQ;
      const float* VV = s_v + st * TQ;
      float cbv[4][8];
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) {
        if (bb <= qrt) {
          uint32_t r[8];
          asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                       : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                       : "r"(tmem + lane_off + kColCB + 32 * bb + 8 * cg));
#pragma unroll
          for (int i = 0; i < 8; ++i) cbv[bb][i] = __uint_as_float(r[i]);
        }
      }
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      const float St = S2[row];
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) {
        uint32_t hi[4], lo[4];
        const int j0 = 32 * bb + 8 * cg;
        if (bb > qrt) {
#pragma unroll
          for (int e = 0; e < 4; ++e) hi[e] = lo[e] = 0u;
        } else if (bb < qrt) {
          const float u = ex2(St - S2[32 * bb + 31]);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            split2(cbv[bb][2 * e] * u * VV[j0 + 2 * e], cbv[bb][2 * e + 1] * u * VV[j0 + 2 * e + 1], hi[e], lo[e]);
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int ja = j0 + 2 * e, jb = ja + 1;
            const float ma = ja <= row ? cbv[bb][2 * e] * ex2(St - S2[ja]) * DP[ja] : 0.f;
            const float mb = jb <= row ? cbv[bb][2 * e + 1] * ex2(St - S2[jb]) * DP[jb] : 0.f;
            split2(ma, mb, hi[e], lo[e]);
          }
        }
        const uint32_t pc = (uint32_t)(j0 >> 1);  // packed bf16-pair column
        asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};"
                     :: "r"(tmem + lane_off + kColMhi + pc), "r"(hi[0]), "r"(hi[1]), "r"(hi[2]), "r"(hi[3]) : "memory");
        asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};"
                     :: "r"(tmem + lane_off + kColMlo + pc), "r"(lo[0]), "r"(lo[1]), "r"(lo[2]), "r"(lo[3]) : "memory");
      }
    }
    {
      const float decay = ex2(tot2);
      float dv[16];
      {
        uint32_t r[16];
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                       "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                       "=r"(r[15])
                     : "r"(tmem + lane_off + kColDH + 16 * cg));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
        for (int i = 0; i < 16; ++i) dv[i] = __uint_as_float(r[i]);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) hst[i] = fmaf(decay, hst[i], dv[i]);
      if (kFull) state_to_smem();
      else seg_logdecay += tot2 * 0.6931471805599453f;
    }
    if (dt_warp && more) {
      dt_phase(c + 1, st ^ 1);
      if (c + 2 < c_end) load_dt(c + 2);
    }
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    if (more) asm volatile("cp.async.wait_group 0;\n" ::: "memory");  // chunk c+1's tiles
    tc_sync();

    // (3) MMAs: Y(c) = M(c) . X(c); Yoff(c+1) = C(c+1) . H(c)^T
    if (kFull && tid == kIssYd) {
      issue_yd(st);
      mma_commit(mbar2);
    }
    if (kFull && tid == kIssYo) {
      if (more) issue_yo(st ^ 1, st ^ 1);
      mma_commit(mbar2);
    }
    // (4) chunk c+1's (X o w), then its CB and dH MMAs
    if (more) {
      xw_phase(st ^ 1, st ^ 1);
      tc_sync();
      if (kFull && tid == kIssCB) {
        issue_cb(st ^ 1);
        mma_commit(mbar1);
      }
      if (tid == kIssDH) {
        issue_dh(st ^ 1);
        mma_commit(mbar1);
      }
    }
    if (kFull) {
      // (5) epilogue of chunk c: y = Y + exp(s_t) Yoff + D x, staged in the spent
      // C tile of this stage, then written as whole rows
      if (!__syncthreads_and(mbar_wait(mbar2, ph2))) {
        if (tid == 0) atomicAdd(&g_tc_timeouts, 1u);
        ok_run = false;
        break;
      }
      ph2 ^= 1u;
      tc_fence_after();
      unsigned char* stage_p = smem + kOffIn + st * kStage;
      {
        const float et = ex2(s_s2[st * TQ + row]);
        float yd[16], yo[16];
        tmem_ld16x2(tmem + lane_off + kColYd + 16 * cg, tmem + lane_off + kColYo + 64 * st + 16 * cg, yd, yo);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const uint32_t o = tile_off(row, 16 * cg + 8 * e, TQ);
          const uint4 xv = *reinterpret_cast<const uint4*>(stage_p + kTileC + kTileB + o);
          const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
          uint32_t outw[4];
#pragma unroll
          for (int f = 0; f < 4; ++f) {
            const int i = 8 * e + 2 * f;
            const float y0 = fmaf(Dh, __uint_as_float(xw[f] << 16), fmaf(et, yo[i], yd[i]));
            const float y1 = fmaf(Dh, __uint_as_float(xw[f] & 0xffff0000u), fmaf(et, yo[i + 1], yd[i + 1]));
            outw[f] = pack2(y0, y1);
          }
          *reinterpret_cast<uint4*>(stage_p + o) = make_uint4(outw[0], outw[1], outw[2], outw[3]);
        }
      }
      tc_fence_before();
      __syncthreads();
      {
        __nv_bfloat16* yout = static_cast<__nv_bfloat16*>(a.dst);
        for (int i = tid; i < TQ * (TP / 8); i += kTcThreads) {
          const int t = i >> 3, pc = i & 7;
          if (t < len) {
            const uint4 v = *reinterpret_cast<const uint4*>(stage_p + tile_off(t, pc * 8, TQ));
            *reinterpret_cast<uint4*>(yout + (row0 + (int64_t)c * TQ + t) * (int64_t)(H * TP) + x_col + pc * 8) = v;
          }
        }
      }
    }
    __syncthreads();  // this stage's tiles are spent
    if (c + 2 < c_end) issue_chunk(c + 2, st);
  }

  // ---- results
  if (ok_run) {
    if (kFull) {
      if (k == nseg - 1) store_state(slot_ptr);
    } else {
      store_state(ws_entry(seg));
      if (tid == 0) a.ws_decay[(int64_t)seg * H + h] = seg_logdecay;
    }
  }
  asm volatile("cp.async.wait_group 0;\n" ::: "memory");
  tc_fence_before();
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(kTmemCols));
}

}  // namespace

unsigned int read_device_timeouts() {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_tc_timeouts, sizeof v) != cudaSuccess) return 0xffffffffu;
  return v;
}

cudaError_t launch_scan_tc(const ScanArgs& a, cudaStream_t st) {
  const int segs = a.tab.tile[a.tab.n];
  if (segs == 0) return cudaSuccess;
  const dim3 grid((unsigned)segs, (unsigned)a.heads);
  bool segmented = false;
  for (int i = 0; i < a.tab.n; ++i) segmented |= (a.tab.tile[i + 1] - a.tab.tile[i]) > 1;
  if (segmented) {
    cudaError_t e = cudaFuncSetAttribute(ssd_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    ssd_tc_kernel<false><<<grid, kTcThreads, kSmemBytes, st>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = cudaFuncSetAttribute(ssd_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  ssd_tc_kernel<true><<<grid, kTcThreads, kSmemBytes, st>>>(a);
  return cudaGetLastError();
}

}  // namespace mamba2
