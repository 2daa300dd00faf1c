// One decode step: conv (one token) -> selective scan (one token) -> gated
// RMSNorm, fused in one kernel for a batch of sequences.
//
// Semantics: the three ops of gllm PR #85 "feat(backend): Mamba2 ops, with
// CPU reference implementations", section "Ops", applied to a single token per
// sequence, with the conv output and y rounded to the activation type exactly
// where the unfused ops store them. The page "Granite Mamba2 Inference
// Optimization" describes decode as a per-token recurrence over conv and SSM
// cache state; InfiniLM PR #575 "feat(mamba2): integrate model loading and
// recurrent inference" (section "Summary") runs it as indexed recurrent decode
// over a state pool.
//
// Two kernels per step. decode_step_kernel: CTA r of a sequence owns heads
// [r*hpc, (r+1)*hpc) (hpc heads per CTA, chosen from the batch size so that the
// grid fills the GPU: one head per CTA for a single sequence, up to 8 for large
// batches). Each CTA
//   1. computes the conv for its heads' x channels and for all B/C channels
//      (B/C recomputed per CTA: 2*G*N channels, tiny), writes the new conv
//      history of its own x channels (no other CTA touches them);
//   2. streams its heads' fp32 SSM state once: 16-byte loads along d_state,
//      h = h*decay + dt'*x*B, y = h.C + D*x (warp-shuffle reduction), store;
//   3. writes y, rounded to the activation type (the unfused scan's output), to dst.
// decode_finish_kernel, one CTA per sequence, once every CTA of the first kernel
// is done (stream order): shifts the B/C conv history (every CTA has read the old
// one), then forms g = y*silu(z) and the gated RMSNorm over each group in a fixed
// order, writing the output over y in dst.
// HBM traffic per sequence: SSM state read + write (H*P*N*4 bytes each), conv
// history read + write, the token's inputs and outputs (y once more through the
// second kernel). The state stream is the roofline term.
#include "common.cuh"

namespace mamba2 {

constexpr int kDecodeWarps = kDecodeThreads / 32;
static_assert(kDecodeWarps % 4 == 0, "the finish kernel's norm-weight buffer follows the warp sums 16-byte aligned");
constexpr int kDecodeUnroll = 16;  // state rows in flight per lane (16-byte loads)
static_assert(kDecodeUnroll == 16, "the d_state = 128 path reduces 16 rows by recursive halving");

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

constexpr int kRingRows = 8;  // d_state = 128: state rows per ring stage (one float4 per lane per row)
// float offset of the state ring in the dynamic shared memory (16-byte aligned) and its bytes
__host__ __device__ constexpr int ring_offset(int hpc, int P, int G, int N) {
  return (2 * hpc * P + 2 * G * N + 3 * hpc + 3) & ~3;
}
constexpr int kRingBytes = kDecodeWarps * 2 * kRingRows * 32 * 16;

// kRing: d_state = 128, the state streamed through a per-warp ring in shared memory
// (no state rows held in registers, three CTAs per SM); otherwise rows in registers.
template <typename T, int K, bool kRing>
__global__ void __launch_bounds__(kDecodeThreads, kRing ? 3 : 2)
decode_step_kernel(const __grid_constant__ DecodeArgs a) {
  constexpr int V = Vec16<T>::n;
  constexpr int HIST = K - 1;
  extern __shared__ __align__(16) float dsm[];

  const int rank = blockIdx.x;  // CTA of the sequence
  const int s = blockIdx.y;
  const int H = a.heads, P = a.headdim, N = a.d_state, G = a.ngroups;
  const int d_inner = H * P;
  const int conv_dim = d_inner + 2 * G * N;
  const int h0 = rank * a.heads_per_cta;
  const int h1 = min(H, h0 + a.heads_per_cta);
  const int nh = max(0, h1 - h0);
  const int rows = nh * P;  // state rows owned by this CTA
  const bool dev = a.dev_slots != nullptr;
  // Launched as a programmatic dependent of whatever precedes it on the stream
  // (the previous step's finish kernel lets it be scheduled early): only the
  // model's parameters may be read before this wait; the batch, the token's
  // inputs, both pools and dst come after it.
  float A_h = 0.f, D_h = 0.f, bias_h = 0.f;
  if (threadIdx.x < nh) {
    A_h = a.A_log[h0 + threadIdx.x];
    D_h = a.D[h0 + threadIdx.x];
    bias_h = a.dt_bias[h0 + threadIdx.x];
  }
  {
    // the conv taps and bias of this thread's first conv vector into L1
    const int nxv0 = rows / V, i0 = threadIdx.x;
    if (i0 < nxv0 + 2 * G * N / V) {
      const int c0 = i0 < nxv0 ? h0 * P + i0 * V : d_inner + (i0 - nxv0) * V;
      asm volatile("prefetch.global.L1 [%0];" ::"l"(a.conv_w + (int64_t)c0 * K));
      asm volatile("prefetch.global.L1 [%0];" ::"l"(a.conv_b + c0));
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // a device batch: nothing is touched unless the batch check (the launch before) passed
  if (dev && (__ldg(a.dev_status) != 0 || s >= __ldg(a.dev_n))) return;
  const bool fresh = dev ? __ldg(a.dev_fresh + s) != 0 : seq_fresh(a.tab, s);
  const int64_t slot = dev ? (int64_t)__ldg(a.dev_slots + s) : (int64_t)seq_slot(a.tab, s);

  float* xs = dsm;                           // [heads_per_cta * P] conv output x
  float* ys = xs + a.heads_per_cta * P;      // [heads_per_cta * P] h . C
  float* bc = ys + a.heads_per_cta * P;      // [2 * G * N] conv output B, C
  float* hdt = bc + 2 * G * N;               // [heads_per_cta] dt'
  float* hdec = hdt + a.heads_per_cta;       // [heads_per_cta] decay
  float* hD = hdec + a.heads_per_cta;        // [heads_per_cta] D

  const T* xBC = static_cast<const T*>(a.xBC) + (int64_t)s * conv_dim;
  T* cst = static_cast<T*>(a.conv_state) + slot * HIST * conv_dim;
  // the finish kernel of this step may be scheduled once every CTA has started (it
  // waits for this grid's completion before it reads anything this grid writes)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // per-head constants, loaded before the conv so their latency overlaps it
  if (threadIdx.x < nh) {
    const int h = h0 + threadIdx.x;
    const float v = Act<T>::to_f(static_cast<const T*>(a.dt)[(int64_t)s * H + h]) + bias_h;
    const float dtp = softplus_f(v);
    hdt[threadIdx.x] = dtp;
    hdec[threadIdx.x] = expf(-expf(A_h) * dtp);
    hD[threadIdx.x] = D_h;
  }

  // ---- state-stream geometry; the first batch of state loads is issued now
  // so it is in flight while the conv phase below waits on its own inputs
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nq = N / 4;                  // float4 per state row
  const int lpr = nq < 32 ? nq : 32;     // lanes per row
  const int rpp = 32 / lpr;              // rows per warp pass
  const int qpl = (nq + lpr - 1) / lpr;  // float4 per lane per row
  const int q0 = lane % lpr, rs = lane / lpr;
  float4* st = reinterpret_cast<float4*>(a.ssm_state + (slot * H + h0) * (int64_t)P * N);
  const int base0 = warp * rpp * kDecodeUnroll;
  const int bstep = kDecodeWarps * rpp * kDecodeUnroll;
  float4 hv[kDecodeUnroll];
  auto load_rows = [&](int base, int qq) {
    const int q = q0 + qq * lpr;
#pragma unroll
    for (int u = 0; u < kDecodeUnroll; ++u) {
      const int r = base + u * rpp + rs;
      hv[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (!fresh && r < rows && q < nq) hv[u] = __ldcs(st + (int64_t)r * nq + q);
    }
  };
  // kRing: warp w streams its rows [128 j + 16 w, +16) as two 8-row stages each
  // (stage k: j = k / 2, half k % 2) through two ring slots filled by cp.async;
  // stages 0 and 1 are issued now, stage k + 2 once stage k is done
  float4* ring = reinterpret_cast<float4*>(dsm + ring_offset(a.heads_per_cta, P, G, N));
  auto stage_base = [&](int k) { return (k >> 1) * (kDecodeWarps * 16) + warp * 16 + (k & 1) * kRingRows; };
  auto issue = [&](int k) {
    asm volatile("" ::: "memory");  // the slot's earlier shared-memory reads stay before its refill
    const int base = stage_base(k);
    if (base < rows) {
      float4* slot = ring + (warp * 2 + (k & 1)) * kRingRows * 32 + lane;
#pragma unroll
      for (int u = 0; u < kRingRows; ++u) {
        const int r = base + u;
        const bool real = !fresh && r < rows;  // a fresh state is zeros: a zero-byte copy (source never read)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_addr(slot + u * 32)),
                     "l"(real ? st + (int64_t)r * 32 + lane : st), "r"(real ? 16 : 0));
      }
    }
    asm volatile("cp.async.commit_group;\n" ::: "memory");
  };
  if constexpr (kRing) {
    issue(0);
    issue(1);
  } else {
    load_rows(base0, 0);
  }

  // ---- 1. conv for own x channels and all B/C channels -------------------
  const int nxv = rows / V;
  const int nbcv = 2 * G * N / V;
  for (int i = threadIdx.x; i < nxv + nbcv; i += kDecodeThreads) {
    const bool is_x = i < nxv;
    const int c0 = is_x ? h0 * P + i * V : d_inner + (i - nxv) * V;
    uint4 hraw[HIST > 0 ? HIST : 1];
    float hist[HIST > 0 ? HIST : 1][V], cur[V], out[V];
#pragma unroll
    for (int j = 0; j < HIST; ++j) {
      hraw[j] = fresh ? make_uint4(0u, 0u, 0u, 0u)
                      : *reinterpret_cast<const uint4*>(cst + (int64_t)j * conv_dim + c0);
      Vec16<T>::load(reinterpret_cast<const T*>(&hraw[j]), hist[j]);
    }
    const uint4 craw = *reinterpret_cast<const uint4*>(xBC + c0);
    Vec16<T>::load(reinterpret_cast<const T*>(&craw), cur);
    float wv[V * K], bv[V];
    {
      const float4* wp = reinterpret_cast<const float4*>(a.conv_w + (int64_t)c0 * K);
#pragma unroll
      for (int q = 0; q < V * K / 4; ++q) {
        const float4 f = __ldg(wp + q);
        wv[4 * q] = f.x; wv[4 * q + 1] = f.y; wv[4 * q + 2] = f.z; wv[4 * q + 3] = f.w;
      }
      const float4* bp = reinterpret_cast<const float4*>(a.conv_b + c0);
#pragma unroll
      for (int q = 0; q < V / 4; ++q) {
        const float4 f = __ldg(bp + q);
        bv[4 * q] = f.x; bv[4 * q + 1] = f.y; bv[4 * q + 2] = f.z; bv[4 * q + 3] = f.w;
      }
    }
    uint32_t retry_mask = 0;
#pragma unroll
    for (int j = 0; j < V; ++j) {
      float wk[K], uk[K];
#pragma unroll
      for (int k = 0; k < K; ++k) {
        wk[k] = wv[j * K + k];
        uk[k] = k < HIST ? hist[k < HIST ? k : 0][j] : cur[j];
      }
      if constexpr (Act<T>::code == MAMBA2_BF16) {
        bool retry;
        out[j] = conv_silu_bf16_fast<K>(bv[j], wk, uk, retry);
        if (retry) retry_mask |= 1u << j;
      } else {
        out[j] = conv_silu_act<T, K>(bv[j], wk, uk);
      }
    }
    float* o = is_x ? xs + i * V : bc + (c0 - d_inner);
#pragma unroll
    for (int j = 0; j < V; ++j) o[j] = out[j];
    // retry of the outputs the fast rounding test could not decide
    // (inputs re-read; this thread has not yet rewritten its history rows)
    while (retry_mask) {
      const int j = __ffs(retry_mask) - 1;
      retry_mask &= retry_mask - 1;
      const int c = c0 + j;
      float wk[K], uk[K];
#pragma unroll
      for (int k = 0; k < K; ++k) {
        wk[k] = a.conv_w[(int64_t)c * K + k];
        uk[k] = k < HIST ? (fresh ? 0.f : Act<T>::to_f(cst[(int64_t)k * conv_dim + c])) : Act<T>::to_f(xBC[c]);
      }
      bool undecided;  // double-float first (fp64 is slow on this part), fp64 when that cannot decide
      const float v2 = conv_silu_bf16_df<K>(a.conv_b[c], wk, uk, undecided);
      o[j] = undecided ? conv_silu_bf16_fp64<K>(a.conv_b[c], wk, uk) : v2;
    }
    if (is_x) {  // own channels: shift the history now
#pragma unroll
      for (int j = 0; j + 1 < HIST; ++j)
        *reinterpret_cast<uint4*>(cst + (int64_t)j * conv_dim + c0) = hraw[j + 1];
      if (HIST > 0)
        *reinterpret_cast<uint4*>(cst + (int64_t)(HIST > 0 ? HIST - 1 : 0) * conv_dim + c0) = craw;
    }
  }
  __syncthreads();

  // ---- 2. state stream: h = h*decay + dt'*x*B; y = h.C + D*x -------------
  if constexpr (kRing) {
    const int hpg = H / G;
    for (int k = 0; stage_base(k) < rows; ++k) {
      asm volatile("cp.async.wait_group 1;\n" ::: "memory");  // stage k has landed (k + 1 may be in flight)
      const int base = stage_base(k);
      const int hl = base / P;  // a stage lies in one head (P % 8 == 0)
      const int g = (h0 + hl) / hpg;
      const float dtp = hdt[hl], dec = hdec[hl];
      const float4 b4 = *reinterpret_cast<const float4*>(bc + g * N + 4 * lane);
      const float4 c4 = *reinterpret_cast<const float4*>(bc + G * N + g * N + 4 * lane);
      const float4* slot = ring + (warp * 2 + (k & 1)) * kRingRows * 32 + lane;
      float acc[kRingRows];
#pragma unroll
      for (int u = 0; u < kRingRows; ++u) {
        const int r = base + u;
        acc[u] = 0.0f;
        if (r < rows) {
          const float xd = dtp * xs[r];
          float4 h = slot[u * 32];
          h.x = fmaf(h.x, dec, xd * b4.x);
          h.y = fmaf(h.y, dec, xd * b4.y);
          h.z = fmaf(h.z, dec, xd * b4.z);
          h.w = fmaf(h.w, dec, xd * b4.w);
          __stcs(st + (int64_t)r * nq + lane, h);
          float t = h.x * c4.x;
          t = fmaf(h.y, c4.y, t);
          t = fmaf(h.z, c4.z, t);
          acc[u] = fmaf(h.w, c4.w, t);
        }
      }
      // the 8 row sums across the warp by recursive halving, then the last two lane bits
#pragma unroll
      for (int d = 16, m = kRingRows; d >= 4; d >>= 1, m >>= 1) {
        const bool upper = (lane & d) != 0;
#pragma unroll
        for (int i = 0; i < m / 2; ++i) {
          const float send = upper ? acc[i] : acc[i + m / 2];
          const float keep = upper ? acc[i + m / 2] : acc[i];
          acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, d);
        }
      }
      acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], 2);
      acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], 1);
      const int rl = ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
      if ((lane & 3) == 0 && base + rl < rows) ys[base + rl] = acc[0];
      issue(k + 2);
    }
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
  } else if (lpr == 32 && qpl == 1) {
    // d_state = 128: one float4 per lane per row, rows of a 16-row batch all
    // in one head (P % 16 == 0), so B and C are loaded once per batch; the 16
    // row sums are reduced across the warp by recursive halving (16 shuffles
    // per lane instead of 5 per row).
    const int hpg = H / G;
    for (int base = base0; base < rows; base += bstep) {
      if (base != base0) load_rows(base, 0);
      const int hl = base / P;
      const int g = (h0 + hl) / hpg;
      const float dtp = hdt[hl], dec = hdec[hl];
      const float4 b4 = *reinterpret_cast<const float4*>(bc + g * N + 4 * lane);
      const float4 c4 = *reinterpret_cast<const float4*>(bc + G * N + g * N + 4 * lane);
      float acc[kDecodeUnroll];
#pragma unroll
      for (int u = 0; u < kDecodeUnroll; ++u) {
        const int r = base + u;
        acc[u] = 0.0f;
        if (r < rows) {
          const float xd = dtp * xs[r];
          float4 h = hv[u];
          h.x = fmaf(h.x, dec, xd * b4.x);
          h.y = fmaf(h.y, dec, xd * b4.y);
          h.z = fmaf(h.z, dec, xd * b4.z);
          h.w = fmaf(h.w, dec, xd * b4.w);
          __stcs(st + (int64_t)r * nq + lane, h);
          float t = h.x * c4.x;
          t = fmaf(h.y, c4.y, t);
          t = fmaf(h.z, c4.z, t);
          acc[u] = fmaf(h.w, c4.w, t);
        }
      }
#pragma unroll
      for (int d = 16, m = kDecodeUnroll; d >= 2; d >>= 1, m >>= 1) {
        const bool upper = (lane & d) != 0;
#pragma unroll
        for (int i = 0; i < m / 2; ++i) {
          const float send = upper ? acc[i] : acc[i + m / 2];
          const float keep = upper ? acc[i + m / 2] : acc[i];
          acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, d);
        }
      }
      acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], 1);
      const int rl = ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
      if ((lane & 1) == 0 && base + rl < rows) ys[base + rl] = acc[0];
    }
  } else {
    const int hpg = H / G;
    for (int base = base0; base < rows; base += bstep) {
      for (int qq = 0; qq < qpl; ++qq) {
        const int q = q0 + qq * lpr;
        if (base != base0 || qq != 0) load_rows(base, qq);
#pragma unroll
        for (int u = 0; u < kDecodeUnroll; ++u) {
          const int r = base + u * rpp + rs;
          float acc = 0.0f;
          if (r < rows && q < nq) {
            const int hl = r / P;
            const int g = (h0 + hl) / hpg;
            const float xv = xs[r], dtp = hdt[hl], dec = hdec[hl];
            const float4 b4 = *reinterpret_cast<const float4*>(bc + g * N + 4 * q);
            const float4 c4 = *reinterpret_cast<const float4*>(bc + G * N + g * N + 4 * q);
            float4 h = hv[u];
            h.x = fmaf(h.x, dec, dtp * b4.x * xv);
            h.y = fmaf(h.y, dec, dtp * b4.y * xv);
            h.z = fmaf(h.z, dec, dtp * b4.z * xv);
            h.w = fmaf(h.w, dec, dtp * b4.w * xv);
            __stcs(st + (int64_t)r * nq + q, h);
            acc = h.x * c4.x;
            acc = fmaf(h.y, c4.y, acc);
            acc = fmaf(h.z, c4.z, acc);
            acc = fmaf(h.w, c4.w, acc);
          }
          for (int o = lpr >> 1; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
          if (qq == 0) {
            if (q0 == 0 && r < rows) ys[r] = acc;
          } else if (q0 == 0 && r < rows) {
            ys[r] += acc;
          }
        }
      }
    }
  }
  __syncthreads();

  // ---- 3. y = h.C + D*x, rounded to the activation type, to dst ------------
  if (rows > 0) {
    T* orow = static_cast<T*>(a.dst) + (int64_t)s * d_inner + h0 * P;
    for (int i = threadIdx.x; i < rows / V; i += kDecodeThreads) {
      float o[V];
#pragma unroll
      for (int j = 0; j < V; ++j) {
        const int r = i * V + j;
        o[j] = ys[r] + hD[r / P] * xs[r];
      }
      Vec16<T>::store(orow + i * V, o);
    }
  }
}

// The rest of the step for sequence s = blockIdx.x, after every CTA of
// decode_step_kernel is done: the B/C conv history shifted by the token, then
// g = y * silu(z) and per norm group out = g / sqrt(mean(g^2) + eps) * weight,
// written over y in dst. Sums of squares in a fixed order (deterministic).
template <typename T, int K>
__global__ void __launch_bounds__(kDecodeThreads)
decode_finish_kernel(const __grid_constant__ DecodeArgs a) {
  constexpr int V = Vec16<T>::n;
  constexpr int HIST = K - 1;
  extern __shared__ __align__(16) float gbuf[];  // [d_inner] g, [kDecodeWarps] warp sums, [d_inner] norm weight
  const int s = blockIdx.x;
  const bool dev = a.dev_slots != nullptr;
  if (dev && (__ldg(a.dev_status) != 0 || s >= __ldg(a.dev_n))) return;
  const bool fresh = dev ? __ldg(a.dev_fresh + s) != 0 : seq_fresh(a.tab, s);
  const int64_t slot = dev ? (int64_t)__ldg(a.dev_slots + s) : (int64_t)seq_slot(a.tab, s);
  const int H = a.heads, P = a.headdim, N = a.d_state, G = a.ngroups;
  const int d_inner = H * P;
  const int conv_dim = d_inner + 2 * G * N;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // the next step's state kernel may be scheduled now (it waits for this grid's
  // completion before it reads anything this grid writes)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // the norm weight (a parameter) and silu(z) (this step's input, not written by
  // the state kernel) first ...
  float* wbuf = gbuf + d_inner + kDecodeWarps;  // [d_inner] norm weight
  for (int i = threadIdx.x; i < d_inner / 4; i += kDecodeThreads)
    reinterpret_cast<float4*>(wbuf)[i] = __ldg(reinterpret_cast<const float4*>(a.norm_w) + i);
  T* row = static_cast<T*>(a.dst) + (int64_t)s * d_inner;
  const T* zrow = static_cast<const T*>(a.z) + (int64_t)s * d_inner;
  for (int i = threadIdx.x; i < d_inner / V; i += kDecodeThreads) {
    float zv[V];
    Vec16<T>::load(zrow + i * V, zv);
#pragma unroll
    for (int j = 0; j < V; ++j) gbuf[i * V + j] = silu_f(zv[j]);
  }
  // ... then wait until the state kernel of this step has finished and its writes
  // (y in dst) are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // B/C conv history: older rows move up, the token's B/C becomes the newest row.
  // Each thread's history rows are loaded first and stored after its y vectors
  // are loaded, so the two round trips overlap.
  const T* xBC = static_cast<const T*>(a.xBC) + (int64_t)s * conv_dim;
  T* cst = static_cast<T*>(a.conv_state) + slot * HIST * conv_dim;
  const int nbcv = 2 * G * N / V;
  const int i_bc = threadIdx.x;  // this thread's first history vector
  uint4 hrow[HIST > 0 ? HIST : 1];
  if (HIST > 0 && i_bc < nbcv) {
    const int c0 = d_inner + i_bc * V;
#pragma unroll
    for (int j = 0; j + 1 < HIST; ++j)
      hrow[j] = fresh ? make_uint4(0u, 0u, 0u, 0u) : *reinterpret_cast<const uint4*>(cst + (int64_t)(j + 1) * conv_dim + c0);
    hrow[HIST > 0 ? HIST - 1 : 0] = *reinterpret_cast<const uint4*>(xBC + c0);
  }

  // g = y * silu(z) (each thread the same vectors it filled above)
  for (int i = threadIdx.x; i < d_inner / V; i += kDecodeThreads) {
    float y[V];
    Vec16<T>::load(row + i * V, y);
#pragma unroll
    for (int j = 0; j < V; ++j) gbuf[i * V + j] *= y[j];
  }
  if (HIST > 0 && i_bc < nbcv) {
    const int c0 = d_inner + i_bc * V;
#pragma unroll
    for (int j = 0; j < HIST; ++j) *reinterpret_cast<uint4*>(cst + (int64_t)j * conv_dim + c0) = hrow[j];
  }
  for (int i = i_bc + kDecodeThreads; i < nbcv && HIST > 0; i += kDecodeThreads) {  // wider B/C: the rest
    const int c0 = d_inner + i * V;
    const uint4 craw = *reinterpret_cast<const uint4*>(xBC + c0);
#pragma unroll
    for (int j = 0; j + 1 < HIST; ++j) {
      const uint4 nxt = fresh ? make_uint4(0u, 0u, 0u, 0u)
                              : *reinterpret_cast<const uint4*>(cst + (int64_t)(j + 1) * conv_dim + c0);
      *reinterpret_cast<uint4*>(cst + (int64_t)j * conv_dim + c0) = nxt;
    }
    *reinterpret_cast<uint4*>(cst + (int64_t)(HIST > 0 ? HIST - 1 : 0) * conv_dim + c0) = craw;
  }
  __syncthreads();
  float* wsum = gbuf + d_inner;
  const int gs = d_inner / a.norm_groups;
  for (int grp = 0; grp < a.norm_groups; ++grp) {
    float ss = 0.0f;
    for (int r = grp * gs + threadIdx.x; r < (grp + 1) * gs; r += kDecodeThreads) ss = fmaf(gbuf[r], gbuf[r], ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) wsum[warp] = ss;
    __syncthreads();
    float tot = 0.0f;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) tot += wsum[w];
    const float inv = rsqrtf(tot / (float)gs + a.eps);
    for (int i = grp * gs / V + threadIdx.x; i < (grp + 1) * gs / V; i += kDecodeThreads) {
      float o[V];
#pragma unroll
      for (int j = 0; j < V; ++j) o[j] = gbuf[i * V + j] * inv * wbuf[i * V + j];
      Vec16<T>::store(row + i * V, o);
    }
    __syncthreads();  // wsum is reused by the next group
  }
}

bool decode_supported(mamba2_dtype act, const mamba2_dims& d, int norm_groups) {
  const int V = act == MAMBA2_BF16 ? 8 : 4;
  const int nq = d.d_state / 4;
  if (d.d_state % 4 != 0 || nq == 0) return false;
  if (nq < 32 && (nq & (nq - 1)) != 0) return false;
  if (d.headdim % V != 0 || (2 * d.ngroups * d.d_state) % V != 0) return false;
  if (d.conv_kernel < 1 || d.conv_kernel > 4) return false;
  if (norm_groups < 1 || norm_groups > kDecodeMaxNormGroups) return false;
  const int d_inner = d.heads * d.headdim;
  if (d_inner % norm_groups != 0 || (d_inner / norm_groups) % V != 0) return false;
  return true;
}

// The batch check of a device batch, in the host check's order: the count, then every
// slot's range, then slots named twice (a bitmap in shared memory when the pool has at
// most kCheckBitmapWords * 32 slots, else pairwise). One CTA; writes only *status.
constexpr int kCheckThreads = 1024;
constexpr int kCheckBitmapWords = 8192;  // 32 KB
__global__ void __launch_bounds__(kCheckThreads) check_device_batch_kernel(const int32_t* __restrict__ slots,
                                                                          const int32_t* __restrict__ n_ptr,
                                                                          int32_t capacity, int32_t num_slots,
                                                                          int32_t* __restrict__ status) {
  extern __shared__ uint32_t seen[];
  const int n = *n_ptr;
  if (n < 0 || n > capacity) {  // the same n in every thread: the CTA leaves together
    if (threadIdx.x == 0) *status = MAMBA2_ERR_INVALID_ARGUMENT;
    return;
  }
  int bad = 0;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int32_t sl = slots[i];
    bad |= (sl < 0 || sl >= num_slots) ? 1 : 0;
  }
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0) *status = MAMBA2_ERR_SLOT_OUT_OF_RANGE;
    return;
  }
  int dup = 0;
  const int words = (num_slots + 31) / 32;
  if (words <= kCheckBitmapWords) {
    for (int w = threadIdx.x; w < words; w += blockDim.x) seen[w] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const int32_t sl = slots[i];  // in range here
      const uint32_t bit = 1u << (sl & 31);
      dup |= (atomicOr(&seen[sl >> 5], bit) & bit) ? 1 : 0;
    }
  } else {
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const int32_t sl = slots[i];
      for (int j = 0; j < i; ++j) dup |= (slots[j] == sl) ? 1 : 0;
    }
  }
  dup = __syncthreads_or(dup);
  if (threadIdx.x == 0) *status = dup ? MAMBA2_ERR_SLOT_SHARED : MAMBA2_OK;
}

template <typename T, int K, bool kRing>
static cudaError_t launch_decode_tk(const DecodeArgs& a, cudaStream_t st) {
  size_t smem = sizeof(float) * (2 * (size_t)a.heads_per_cta * a.headdim + 2 * (size_t)a.ngroups * a.d_state +
                                 3 * (size_t)a.heads_per_cta);
  if (kRing) smem = sizeof(float) * (size_t)ring_offset(a.heads_per_cta, a.headdim, a.ngroups, a.d_state) + kRingBytes;
  auto kern = decode_step_kernel<T, K, kRing>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  // programmatic dependent launch: scheduled while the kernel before it (the
  // previous step's finish kernel) runs; it waits (griddepcontrol.wait) before
  // reading anything but the parameters
  cudaLaunchConfig_t scfg = {};
  scfg.gridDim = dim3((unsigned)a.ctas_per_seq, (unsigned)a.tab.n, 1);
  scfg.blockDim = dim3(kDecodeThreads, 1, 1);
  scfg.dynamicSmemBytes = smem;
  scfg.stream = st;
  cudaLaunchAttribute sattr[1];
  sattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  sattr[0].val.programmaticStreamSerializationAllowed = 1;
  scfg.attrs = sattr;
  scfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&scfg, kern, a);
  if (e != cudaSuccess) return e;
  const size_t fsmem = sizeof(float) * (2 * (size_t)a.heads * a.headdim + kDecodeWarps);
  auto fin = decode_finish_kernel<T, K>;
  if (fsmem > 48 * 1024) {
    e = cudaFuncSetAttribute(fin, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fsmem);
    if (e != cudaSuccess) return e;
  }
  // programmatic dependent launch: the finish kernel is scheduled while the state
  // kernel runs and waits for it (griddepcontrol.wait) before reading its output
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.tab.n, 1, 1);
  cfg.blockDim = dim3(kDecodeThreads, 1, 1);
  cfg.dynamicSmemBytes = fsmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fin, a);
}

template <typename T, int K>
static cudaError_t launch_decode_t(const DecodeArgs& a, cudaStream_t st) {
  if (a.d_state == 128 && a.headdim % kRingRows == 0) return launch_decode_tk<T, K, true>(a, st);
  return launch_decode_tk<T, K, false>(a, st);
}

cudaError_t launch_check_device_batch(const int32_t* slots, const int32_t* n, int32_t capacity, int32_t num_slots,
                                      int32_t* status, cudaStream_t st) {
  const int words = (num_slots + 31) / 32;
  const size_t smem = words <= kCheckBitmapWords ? sizeof(uint32_t) * (size_t)(words > 0 ? words : 1) : 0;
  check_device_batch_kernel<<<1, kCheckThreads, smem, st>>>(slots, n, capacity, num_slots, status);
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeArgs& a, mamba2_dtype act, cudaStream_t st) {
  if (a.tab.n == 0) return cudaSuccess;
  if (act == MAMBA2_BF16) {
    switch (a.conv_kernel) {
      case 1: return launch_decode_t<__nv_bfloat16, 1>(a, st);
      case 2: return launch_decode_t<__nv_bfloat16, 2>(a, st);
      case 3: return launch_decode_t<__nv_bfloat16, 3>(a, st);
      case 4: return launch_decode_t<__nv_bfloat16, 4>(a, st);
    }
  } else {
    switch (a.conv_kernel) {
      case 1: return launch_decode_t<float, 1>(a, st);
      case 2: return launch_decode_t<float, 2>(a, st);
      case 3: return launch_decode_t<float, 3>(a, st);
      case 4: return launch_decode_t<float, 4>(a, st);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace mamba2
