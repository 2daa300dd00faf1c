// Selective scan (SSMScan) for prefill: a chunked scan on the tensor cores,
// and a token-serial CUDA-core kernel for shapes the chunked one does not
// cover.
//
// Semantics: gllm PR #85 "feat(backend): Mamba2 ops, with CPU reference
// implementations", section "Ops" (SSMScan): per token
//   dt' = softplus(dt + dt_bias),  h = h*exp(-exp(A_log)*dt') + dt'*B (x) x,
//   y = h.C + D*x,
// head h reading group h/(heads/groups), state seeded from and written back
// to the sequence's slot. The same page (section "CPU reference") calls a
// chunked scan the GPU throughput technique, validated against the
// token-at-a-time loop; the page "Granite Mamba2 Inference Optimization"
// describes long prefill as a chunked parallel scan.
//
// Chunked form. For a chunk of Q = 64 tokens with a_t = -exp(A_log)*dt'_t and
// s_t = a_0 + ... + a_t (inclusive, s <= 0, non-increasing):
//   y_t   = exp(s_t) * C_t . h_in  +  sum_{j<=t} (C_t . B_j) exp(s_t - s_j) dt'_j x_j  +  D x_t
//   h_out = exp(s_{Q-1}) h_in  +  sum_j exp(s_{Q-1} - s_j) dt'_j x_j (x) B_j
// Every exponent is a difference of cumulative sums taken in the safe
// direction (<= 0), so nothing overflows for any decay.
//
// CTA = (sequence segment, head), 4 warps. Warp w owns token rows
// [16w, 16w+16) of the chunk for y, and state rows p in [16w, 16w+16) (all
// d_state columns, fp32 registers) for the state products. Per chunk
// (m16n8k16 bf16 MMAs, fp32 accumulate):
//   Yoff^T = H . C^T             (state-row warps; A = H straight from the
//                                 accumulator registers, scaled by exp(s_t),
//                                 staged in smem as fp32)
//   CB     = C . B^T             (token-row warps, causal column blocks only)
//   M      = CB o exp(s_t - s_j) dt'_j   (accumulator -> A operand in registers)
//   Y      = M . X ;  y = Y + Yoff + D x  -> bf16
//   H      = exp(s_{Q-1}) H + (X o w)^T . B,  w_j = exp(s_{Q-1} - s_j) dt'_j
// The running state H stays in fp32 registers across chunks (it never goes
// to HBM between chunks). Every fp32 operand (H, M, X o w) is split into bf16
// hi + lo parts (two MMAs), which keeps ~16 mantissa bits: the sums feeding y
// can cancel strongly, and plain bf16 operands then lose the output.
//
// Long runs are cut into segments of seg_chunks chunks so enough CTAs run.
// A state pass (kFull = false) computes each segment's end state from zero
// (segment 0 from the slot) and its total log-decay into the workspace; the
// full pass (kFull = true) seeds segment k with
//   h_in(k) = e(k-1) + exp(d(k-1)) * (e(k-2) + exp(d(k-2)) * (...))
// and writes y; only the sequence's last segment writes the slot. Segment 0
// of the full pass reads its seed from a workspace copy the state pass made,
// so no CTA reads a slot another CTA may be writing.
#include "common.cuh"

namespace mamba2 {
namespace {

constexpr int kQ = kChunk;
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}

// D += A(16x16, row) * B(16x8, col), bf16 in, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

template <int P, int N>
struct ScanSmem {
  static constexpr int XS = P + 8;  // padded row strides (conflict-free ldmatrix)
  static constexpr int BS = N + 8;
  __nv_bfloat16 x[2][kQ][XS];
  __nv_bfloat16 b[2][kQ][BS];
  __nv_bfloat16 c[2][kQ][BS];
  float yoff[kQ][P + 4];   // exp(s_t) * C_t . H (fp32), token-major
  float s[kQ];             // inclusive cumulative log-decay within the chunk
  float dtp[kQ];           // dt'
  float w[kQ];             // exp(s_{Q-1} - s_j) * dt'_j
  float total;             // s_{Q-1}
};

template <int P, int N, bool kFull>
__global__ void __launch_bounds__(kThreads, 2)
ssd_chunk_kernel(const __grid_constant__ ScanArgs a) {
  using Sm = ScanSmem<P, N>;
  constexpr int NT = N / 8;   // 8-wide state column tiles
  constexpr int PB = P / 16;  // 16-row state blocks, one per warp
  constexpr int TPW = NT;     // state tiles per owning warp (a full row block)
  static_assert(P % 16 == 0 && N % 16 == 0 && PB <= kWarps, "tile shape");

  extern __shared__ __align__(128) unsigned char smem_raw[];
  Sm& sm = *reinterpret_cast<Sm*>(smem_raw);

  const int seg = blockIdx.x, h = blockIdx.y;
  const int s = find_tile_seq(a.tab, seg);
  const int seg0 = a.tab.tile[s];
  const int k = seg - seg0;
  const int nseg = a.tab.tile[s + 1] - seg0;
  if (!kFull && k == nseg - 1) return;  // the state pass skips last segments

  const int H = a.heads, G = a.ngroups;
  const int g = h / (H / G);
  const int row0 = a.tab.cu[s];
  const int T = a.tab.cu[s + 1] - row0;
  const int nchunks = (T + kQ - 1) / kQ;
  const int c_begin = k * a.seg_chunks;
  const int c_end = min(nchunks, c_begin + a.seg_chunks);
  const bool fresh = seq_fresh(a.tab, s);
  const int64_t ld = a.conv_dim;
  const __nv_bfloat16* xbc = static_cast<const __nv_bfloat16*>(a.xbc);
  const __nv_bfloat16* dtg = static_cast<const __nv_bfloat16*>(a.dt);
  const int x_col = h * P, b_col = H * P + g * N, c_col = H * P + G * N + g * N;
  const float A = expf(a.A_log[h]);
  const float dtb = a.dt_bias[h];
  const float Dh = a.D[h];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;

  // ---- state rows owned by this warp: rows pb*16 + {gq, gq+8}, cols nt*8 + 2tq + {0,1}
  const int pb = warp;
  const int nt0 = 0;
  const bool owns = warp < PB;
  float hreg[TPW][4];

  const int64_t head_off = (int64_t)h * P * N;
  float* slot_ptr = a.ssm_state + (int64_t)seq_slot(a.tab, s) * H * P * N + head_off;
  auto ws_entry = [&](int segidx) -> float* { return a.ws_state + (int64_t)segidx * H * P * N + head_off; };
  auto load_state = [&](const float* src) {
#pragma unroll
    for (int i = 0; i < TPW; ++i) {
      const int r0 = pb * 16 + gq, cn = (nt0 + i) * 8 + 2 * tq;
      float2 v0 = make_float2(0.f, 0.f), v1 = v0;
      if (owns && src) {
        v0 = *reinterpret_cast<const float2*>(src + (int64_t)r0 * N + cn);
        v1 = *reinterpret_cast<const float2*>(src + (int64_t)(r0 + 8) * N + cn);
      }
      hreg[i][0] = v0.x; hreg[i][1] = v0.y; hreg[i][2] = v1.x; hreg[i][3] = v1.y;
    }
  };
  auto store_state = [&](float* dst) {
    if (!owns) return;
#pragma unroll
    for (int i = 0; i < TPW; ++i) {
      const int r0 = pb * 16 + gq, cn = (nt0 + i) * 8 + 2 * tq;
      *reinterpret_cast<float2*>(dst + (int64_t)r0 * N + cn) = make_float2(hreg[i][0], hreg[i][1]);
      *reinterpret_cast<float2*>(dst + (int64_t)(r0 + 8) * N + cn) = make_float2(hreg[i][2], hreg[i][3]);
    }
  };

  // ---- seed the running state
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
#pragma unroll
      for (int i = 0; i < TPW; ++i) {
        const int r0 = pb * 16 + gq, cn = (nt0 + i) * 8 + 2 * tq;
        if (owns) {
          const float2 v0 = *reinterpret_cast<const float2*>(e + (int64_t)r0 * N + cn);
          const float2 v1 = *reinterpret_cast<const float2*>(e + (int64_t)(r0 + 8) * N + cn);
          hreg[i][0] = fmaf(d, hreg[i][0], v0.x);
          hreg[i][1] = fmaf(d, hreg[i][1], v0.y);
          hreg[i][2] = fmaf(d, hreg[i][2], v1.x);
          hreg[i][3] = fmaf(d, hreg[i][3], v1.y);
        }
      }
    }
  }

  // ---- chunk loads (cp.async, zero-filled past the run's end)
  auto issue_chunk = [&](int c, int buf) {
    const int len = min(kQ, T - c * kQ);
    const int64_t r_base = row0 + (int64_t)c * kQ;
    constexpr int XV = P / 8, BV = N / 8;  // 16-byte vectors per row
    for (int i = tid; i < kQ * XV; i += kThreads) {
      const int t = i / XV, v = i % XV;
      const bool ok = t < len;
      const __nv_bfloat16* src = xbc + (ok ? (r_base + t) * ld : row0 * ld) + x_col + v * 8;
      cp_async16(smem_u32(&sm.x[buf][t][v * 8]), src, ok);
    }
    for (int i = tid; i < kQ * BV; i += kThreads) {
      const int t = i / BV, v = i % BV;
      const bool ok = t < len;
      const int64_t rb = (ok ? (r_base + t) * ld : row0 * ld);
      cp_async16(smem_u32(&sm.b[buf][t][v * 8]), xbc + rb + b_col + v * 8, ok);
      if (kFull) cp_async16(smem_u32(&sm.c[buf][t][v * 8]), xbc + rb + c_col + v * 8, ok);
    }
    cp_async_commit();
  };
  // dt for chunk c: warp 0, lane l holds tokens 2l and 2l+1 (raw, pre-softplus)
  float dt_raw[2] = {0.f, 0.f};
  auto load_dt = [&](int c) {
    if (warp != 0) return;
    const int len = min(kQ, T - c * kQ);
    const int64_t r_base = row0 + (int64_t)c * kQ;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int t = 2 * lane + e;
      dt_raw[e] = t < len ? __bfloat162float(dtg[(r_base + t) * H + h]) : 0.f;
    }
  };

  float seg_logdecay = 0.f;
  if (c_begin < c_end) {
    issue_chunk(c_begin, 0);
    load_dt(c_begin);
  }

  for (int c = c_begin; c < c_end; ++c) {
    const int buf = (c - c_begin) & 1;
    const int len = min(kQ, T - c * kQ);
    cp_async_wait_all();
    __syncthreads();  // chunk c staged; the previous chunk's readers of buf^1 and sm.yoff are done
    if (c + 1 < c_end) issue_chunk(c + 1, buf ^ 1);

    // dt', inclusive cumulative log-decay, and the state weights w
    if (warp == 0) {
      float dp[2], av[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int t = 2 * lane + e;
        dp[e] = t < len ? softplus_f(dt_raw[e] + dtb) : 0.f;
        av[e] = -A * dp[e];
      }
      float incl = av[0] + av[1];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const float s1 = incl, s0 = incl - av[1];
      const float tot = __shfl_sync(0xffffffffu, incl, 31);
      sm.s[2 * lane] = s0;
      sm.s[2 * lane + 1] = s1;
      sm.dtp[2 * lane] = dp[0];
      sm.dtp[2 * lane + 1] = dp[1];
      sm.w[2 * lane] = __expf(tot - s0) * dp[0];
      sm.w[2 * lane + 1] = __expf(tot - s1) * dp[1];
      if (lane == 0) sm.total = tot;
      if (c + 1 < c_end) load_dt(c + 1);
    }
    __syncthreads();

    if (kFull) {
      // ---------------- Yoff^T = H . C^T on the state-row warps --------------
      // A = H rows [16 pb, 16 pb + 16) x n, straight from the accumulator
      // registers (hi + lo bf16); B = C^T (n x t) from sm.c rows t.
      if (owns) {
        float yo[kQ / 8][4];
#pragma unroll
        for (int i = 0; i < kQ / 8; ++i) yo[i][0] = yo[i][1] = yo[i][2] = yo[i][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < N / 16; ++kk) {
          uint32_t ahi[4], alo[4];
          const float hv[4][2] = {{hreg[2 * kk][0], hreg[2 * kk][1]},
                                  {hreg[2 * kk][2], hreg[2 * kk][3]},
                                  {hreg[2 * kk + 1][0], hreg[2 * kk + 1][1]},
                                  {hreg[2 * kk + 1][2], hreg[2 * kk + 1][3]}};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            ahi[e] = pack_bf16(hv[e][0], hv[e][1]);
            alo[e] = pack_bf16(hv[e][0] - bf16_lo(ahi[e]), hv[e][1] - bf16_hi(ahi[e]));
          }
#pragma unroll
          for (int tp = 0; tp < kQ / 16; ++tp) {
            uint32_t bf[4];
            const int rr = tp * 16 + (lane & 7) + ((lane >> 4) << 3);
            const int cc = kk * 16 + ((lane >> 3) & 1) * 8;
            ldsm_x4(smem_u32(&sm.c[buf][rr][cc]), bf);
            mma_bf16(yo[2 * tp], ahi, bf[0], bf[1]);
            mma_bf16(yo[2 * tp], alo, bf[0], bf[1]);
            mma_bf16(yo[2 * tp + 1], ahi, bf[2], bf[3]);
            mma_bf16(yo[2 * tp + 1], alo, bf[2], bf[3]);
          }
        }
        // scale column t by exp(s_t) and stage token-major in smem
#pragma unroll
        for (int i = 0; i < kQ / 8; ++i) {
          const int t0 = i * 8 + 2 * tq;
          const float e0 = __expf(sm.s[t0]), e1 = __expf(sm.s[t0 + 1]);
          const int p0 = pb * 16 + gq;
          sm.yoff[t0][p0] = yo[i][0] * e0;
          sm.yoff[t0 + 1][p0] = yo[i][1] * e1;
          sm.yoff[t0][p0 + 8] = yo[i][2] * e0;
          sm.yoff[t0 + 1][p0 + 8] = yo[i][3] * e1;
        }
      }

      // ---------------- y for token rows [16 warp, 16 warp + 16) --------------
      constexpr int PT = P / 8;  // 8-wide column tiles of y
      float yacc[PT][4];
#pragma unroll
      for (int i = 0; i < PT; ++i) yacc[i][0] = yacc[i][1] = yacc[i][2] = yacc[i][3] = 0.f;
      const int m0 = warp * 16;
      const int lrow = lane & 15, lcol8 = (lane >> 4) * 8;  // A-operand ldmatrix lane address
      const int t_lo = m0 + gq, t_hi = t_lo + 8;
      const float st_lo = sm.s[t_lo], st_hi = sm.s[t_hi];
      // CB = C . B^T for causal column blocks j < 16*(warp+1)
      float cb[kQ / 8][4];
#pragma unroll
      for (int i = 0; i < kQ / 8; ++i) cb[i][0] = cb[i][1] = cb[i][2] = cb[i][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < N / 16; ++kk) {
        uint32_t af[4];
        ldsm_x4(smem_u32(&sm.c[buf][m0 + lrow][kk * 16 + lcol8]), af);
#pragma unroll
        for (int jp = 0; jp < kQ / 16; ++jp) {
          if (jp <= warp) {
            uint32_t bf[4];
            const int rr = jp * 16 + (lane & 7) + ((lane >> 4) << 3);
            const int cc = kk * 16 + ((lane >> 3) & 1) * 8;
            ldsm_x4(smem_u32(&sm.b[buf][rr][cc]), bf);
            mma_bf16(cb[2 * jp], af, bf[0], bf[1]);
            mma_bf16(cb[2 * jp + 1], af, bf[2], bf[3]);
          }
        }
      }
      // M = CB o exp(s_t - s_j) dt'_j (j <= t) as hi + lo A operands; Y = M . X
#pragma unroll
      for (int kk = 0; kk < kQ / 16; ++kk) {
        if (kk <= warp) {
          float mv[4][2];  // {row lo k 0-7, row hi k 0-7, row lo k 8-15, row hi k 8-15}
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int jt = 2 * kk + half;
            const int j0 = jt * 8 + 2 * tq;
            const float sj0 = sm.s[j0], sj1 = sm.s[j0 + 1];
            const float dj0 = sm.dtp[j0], dj1 = sm.dtp[j0 + 1];
            mv[2 * half][0] = j0 <= t_lo ? cb[jt][0] * __expf(st_lo - sj0) * dj0 : 0.f;
            mv[2 * half][1] = j0 + 1 <= t_lo ? cb[jt][1] * __expf(st_lo - sj1) * dj1 : 0.f;
            mv[2 * half + 1][0] = j0 <= t_hi ? cb[jt][2] * __expf(st_hi - sj0) * dj0 : 0.f;
            mv[2 * half + 1][1] = j0 + 1 <= t_hi ? cb[jt][3] * __expf(st_hi - sj1) * dj1 : 0.f;
          }
          uint32_t ahi[4], alo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            ahi[e] = pack_bf16(mv[e][0], mv[e][1]);
            alo[e] = pack_bf16(mv[e][0] - bf16_lo(ahi[e]), mv[e][1] - bf16_hi(ahi[e]));
          }
#pragma unroll
          for (int pt = 0; pt < PT; pt += 2) {
            uint32_t bf[4];
            const int rr = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
            const int cc = pt * 8 + (lane >> 4) * 8;
            ldsm_x4_t(smem_u32(&sm.x[buf][rr][cc]), bf);
            mma_bf16(yacc[pt], ahi, bf[0], bf[1]);
            mma_bf16(yacc[pt], alo, bf[0], bf[1]);
            mma_bf16(yacc[pt + 1], ahi, bf[2], bf[3]);
            mma_bf16(yacc[pt + 1], alo, bf[2], bf[3]);
          }
        }
      }
      __syncthreads();  // sm.yoff complete
      // y = Y + Yoff + D x, rounded to bf16
      __nv_bfloat16* yout = static_cast<__nv_bfloat16*>(a.dst);
      const int64_t ldy = (int64_t)H * P;
#pragma unroll
      for (int pt = 0; pt < PT; ++pt) {
        const int p = pt * 8 + 2 * tq;
        if (t_lo < len) {
          const __nv_bfloat162 xv = *reinterpret_cast<const __nv_bfloat162*>(&sm.x[buf][t_lo][p]);
          const float y0 = fmaf(Dh, __low2float(xv), yacc[pt][0] + sm.yoff[t_lo][p]);
          const float y1 = fmaf(Dh, __high2float(xv), yacc[pt][1] + sm.yoff[t_lo][p + 1]);
          *reinterpret_cast<uint32_t*>(yout + (row0 + (int64_t)c * kQ + t_lo) * ldy + x_col + p) = pack_bf16(y0, y1);
        }
        if (t_hi < len) {
          const __nv_bfloat162 xv = *reinterpret_cast<const __nv_bfloat162*>(&sm.x[buf][t_hi][p]);
          const float y0 = fmaf(Dh, __low2float(xv), yacc[pt][2] + sm.yoff[t_hi][p]);
          const float y1 = fmaf(Dh, __high2float(xv), yacc[pt][3] + sm.yoff[t_hi][p + 1]);
          *reinterpret_cast<uint32_t*>(yout + (row0 + (int64_t)c * kQ + t_hi) * ldy + x_col + p) = pack_bf16(y0, y1);
        }
      }
    }

    // ---------------- H = exp(total) H + (X o w)^T . B --------------------
    {
      const float tot = sm.total;
      const float decay = __expf(tot);
#pragma unroll
      for (int i = 0; i < TPW; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) hreg[i][e] *= decay;
      if (owns) {
#pragma unroll
        for (int kk = 0; kk < kQ / 16; ++kk) {
          // A = (X o w)^T rows p in [16 pb, 16 pb + 16), cols j in [16 kk, 16 kk + 16)
          uint32_t xr[4];
          {
            const int rr = kk * 16 + (lane & 7) + (lane >> 4) * 8;
            const int cc = pb * 16 + ((lane >> 3) & 1) * 8;
            ldsm_x4_t(smem_u32(&sm.x[buf][rr][cc]), xr);
          }
          const int j0 = kk * 16 + 2 * tq;
          const float w0 = sm.w[j0], w1 = sm.w[j0 + 1], w8 = sm.w[j0 + 8], w9 = sm.w[j0 + 9];
          uint32_t ahi[4], alo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float wa = (e < 2) ? w0 : w8, wb = (e < 2) ? w1 : w9;
            const float v0 = bf16_lo(xr[e]) * wa, v1 = bf16_hi(xr[e]) * wb;
            ahi[e] = pack_bf16(v0, v1);
            alo[e] = pack_bf16(v0 - bf16_lo(ahi[e]), v1 - bf16_hi(ahi[e]));
          }
          if constexpr (TPW >= 2) {
#pragma unroll
            for (int i = 0; i < TPW; i += 2) {
              uint32_t bf[4];
              const int rr = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
              const int cc = (nt0 + i) * 8 + (lane >> 4) * 8;
              ldsm_x4_t(smem_u32(&sm.b[buf][rr][cc]), bf);
              mma_bf16(hreg[i], ahi, bf[0], bf[1]);
              mma_bf16(hreg[i], alo, bf[0], bf[1]);
              mma_bf16(hreg[i + 1], ahi, bf[2], bf[3]);
              mma_bf16(hreg[i + 1], alo, bf[2], bf[3]);
            }
          } else {
            uint32_t bf[2];
            const int rr = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
            const int cc = nt0 * 8;
            ldsm_x2_t(smem_u32(&sm.b[buf][rr][cc]), bf);
            mma_bf16(hreg[0], ahi, bf[0], bf[1]);
            mma_bf16(hreg[0], alo, bf[0], bf[1]);
          }
        }
      }
      if (!kFull) seg_logdecay += tot;
    }
  }

  if (kFull) {
    if (k == nseg - 1) store_state(slot_ptr);
  } else {
    store_state(ws_entry(seg));
    if (tid == 0) a.ws_decay[(int64_t)seg * H + h] = seg_logdecay;
  }
}

template <int P, int N>
cudaError_t launch_chunked_pn(const ScanArgs& a, cudaStream_t st) {
  const int segs = a.tab.tile[a.tab.n];
  if (segs == 0) return cudaSuccess;
  const size_t smem = sizeof(ScanSmem<P, N>);
  const dim3 grid((unsigned)segs, (unsigned)a.heads);
  bool segmented = false;
  for (int i = 0; i < a.tab.n; ++i) segmented |= (a.tab.tile[i + 1] - a.tab.tile[i]) > 1;
  if (segmented) {
    auto kA = ssd_chunk_kernel<P, N, false>;
    cudaError_t e = cudaFuncSetAttribute(kA, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kA<<<grid, kThreads, smem, st>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  auto kB = ssd_chunk_kernel<P, N, true>;
  cudaError_t e = cudaFuncSetAttribute(kB, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kB<<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Token-serial kernel: one CTA per (sequence, head), one thread per state row
// p holding h[p, :] in registers/local memory; B, C of each token staged in
// shared memory. Used for fp32 activations and shapes the chunked kernel does
// not cover.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void ssd_serial_kernel(const __grid_constant__ ScanArgs a) {
  extern __shared__ float bcs[];  // [2 * N]
  const int s = blockIdx.x, h = blockIdx.y, p = threadIdx.x;
  const int H = a.heads, P = a.headdim, N = a.d_state, G = a.ngroups;
  const int g = h / (H / G);
  const int row0 = a.tab.cu[s], T_len = a.tab.cu[s + 1] - row0;
  const bool fresh = seq_fresh(a.tab, s);
  float* slot_ptr = a.ssm_state + ((int64_t)seq_slot(a.tab, s) * H + h) * P * N;
  const T* xbc = static_cast<const T*>(a.xbc);
  const T* dtg = static_cast<const T*>(a.dt);
  T* y = static_cast<T*>(a.dst);
  const int64_t ld = a.conv_dim;
  const int b_col = H * P + g * N, c_col = H * P + G * N + g * N;
  float hl[kSerialMaxN];
  for (int n = 0; n < N; ++n) hl[n] = (fresh || p >= P) ? 0.f : slot_ptr[(int64_t)p * N + n];
  const float A = expf(a.A_log[h]);
  const float Dh = a.D[h];
  for (int t = 0; t < T_len; ++t) {
    const int64_t r = row0 + t;
    __syncthreads();
    for (int i = threadIdx.x; i < 2 * N; i += blockDim.x)
      bcs[i] = Act<T>::to_f(xbc[r * ld + (i < N ? b_col + i : c_col + i - N)]);
    __syncthreads();
    const float dtp = softplus_f(Act<T>::to_f(dtg[r * H + h]) + a.dt_bias[h]);
    const float decay = expf(-A * dtp);
    if (p < P) {
      const float xv = Act<T>::to_f(xbc[r * ld + h * P + p]);
      float acc = 0.f;
      for (int n = 0; n < N; ++n) {
        hl[n] = fmaf(hl[n], decay, dtp * bcs[n] * xv);
        acc = fmaf(hl[n], bcs[N + n], acc);
      }
      y[r * (int64_t)H * P + h * P + p] = Act<T>::from_f(acc + Dh * xv);
    }
  }
  if (p < P)
    for (int n = 0; n < N; ++n) slot_ptr[(int64_t)p * N + n] = hl[n];
}

}  // namespace

bool scan_chunked_supported(mamba2_dtype act, int headdim, int d_state) {
  return act == MAMBA2_BF16 && ((headdim == 64 && d_state == 128) || (headdim == 16 && d_state == 16));
}

cudaError_t launch_scan_chunked(const ScanArgs& a, cudaStream_t st) {
  if (a.headdim == 64 && a.d_state == 128) return launch_scan_tc(a, st);
  if (a.headdim == 16 && a.d_state == 16) return launch_chunked_pn<16, 16>(a, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_scan_serial(const ScanArgs& a, mamba2_dtype act, cudaStream_t st) {
  if (a.tab.n == 0) return cudaSuccess;
  const dim3 grid((unsigned)a.tab.n, (unsigned)a.heads);
  const int threads = ((a.headdim + 31) / 32) * 32;
  const size_t smem = sizeof(float) * 2 * a.d_state;
  if (act == MAMBA2_BF16)
    ssd_serial_kernel<__nv_bfloat16><<<grid, threads, smem, st>>>(a);
  else
    ssd_serial_kernel<float><<<grid, threads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace mamba2
