/*
 * Plain CPU oracle for the Mamba2 recurrent path: TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, the smoke check and the benchmark's CPU-baseline leg load this
 * library; the CUDA product path neither links nor calls it, and the two share
 * no code. It is deliberately the slow, obvious definition:
 *
 *   - gllm PR #85 "feat(backend): Mamba2 ops, with CPU reference
 *     implementations", section "Ops": CausalConv1D, SSMScan, GatedRMSNorm and
 *     the RecurrentBatch rules (fresh slots never read; out-of-range slots,
 *     shared slots and runs that do not cover the rows are rejected).
 *   - same page, section "CPU reference": the recurrence runs one token at a
 *     time and the state is rounded to fp32 after every token.
 *
 * Arithmetic is double throughout. Readings where the pages leave a step open
 * are listed in the design notes; the ones that shape this file:
 *   - the conv tap w[:, kernel-1] multiplies the current token (section
 *     "Testing" pins this with the pre-activations 0.5+3*1, 0.5+2*1+3*2, ...);
 *   - the conv slot holds the raw conv inputs, oldest first;
 *   - y uses the state after the token's update (section "Testing": y = 7 on
 *     the first token of a fresh sequence needs the updated state);
 *   - softplus(v) = max(v, 0) + log1p(exp(-|v|)), no dt clamp (section "Ops");
 *   - A_log, dt_bias and D are per head;
 *   - interface tensors (conv output, scan output, norm output) are rounded to
 *     the activation type at the end of their op.
 * Parallel loops only split independent (sequence, channel), (sequence, head)
 * and row work; each result is computed by exactly the serial arithmetic.
 */
#include "mamba2_ref.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------------- */
/* Activation storage                                                      */
/* ---------------------------------------------------------------------- */

static double act_load(const void* base, size_t i, int32_t act) {
  if (act == MAMBA2_REF_F32) return (double)((const float*)base)[i];
  uint32_t bits = (uint32_t)((const uint16_t*)base)[i] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* fp32 -> bf16, round to nearest even; NaN stays a (quiet) NaN. */
static uint16_t bf16_from_f32(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static void act_store(void* base, size_t i, int32_t act, double v) {
  float f = (float)v; /* round to nearest even */
  if (act == MAMBA2_REF_F32) {
    ((float*)base)[i] = f;
  } else {
    ((uint16_t*)base)[i] = bf16_from_f32(f);
  }
}

static size_t act_size(int32_t act) { return act == MAMBA2_REF_F32 ? 4 : 2; }

static int act_ok(int32_t act) {
  return act == MAMBA2_REF_F32 || act == MAMBA2_REF_BF16;
}

static double silu(double v) { return v / (1.0 + exp(-v)); }

static double softplus(double v) {
  return (v > 0.0 ? v : 0.0) + log1p(exp(-fabs(v)));
}

/* ---------------------------------------------------------------------- */
/* RecurrentBatch validation (section "Ops": reject, never write)         */
/* ---------------------------------------------------------------------- */

int mamba2_ref_validate_batch(int32_t num_seqs, const int32_t* cu_seqlens,
                              const int32_t* slots, int32_t num_slots,
                              int32_t rows) {
  if (num_seqs < 0 || rows < 0 || num_slots < 0)
    return MAMBA2_REF_ERR_INVALID_ARGUMENT;
  if (num_seqs == 0)
    return rows == 0 ? MAMBA2_REF_OK : MAMBA2_REF_ERR_RUNS_DONT_COVER_ROWS;
  if (!cu_seqlens || !slots) return MAMBA2_REF_ERR_INVALID_ARGUMENT;
  for (int32_t i = 0; i < num_seqs; ++i)
    if (slots[i] < 0 || slots[i] >= num_slots)
      return MAMBA2_REF_ERR_SLOT_OUT_OF_RANGE;
  for (int32_t i = 0; i < num_seqs; ++i)
    for (int32_t j = i + 1; j < num_seqs; ++j)
      if (slots[i] == slots[j]) return MAMBA2_REF_ERR_SLOT_SHARED;
  if (cu_seqlens[0] != 0) return MAMBA2_REF_ERR_RUNS_DONT_COVER_ROWS;
  for (int32_t i = 0; i < num_seqs; ++i)
    if (cu_seqlens[i + 1] < cu_seqlens[i])
      return MAMBA2_REF_ERR_RUNS_DONT_COVER_ROWS;
  if (cu_seqlens[num_seqs] != rows) return MAMBA2_REF_ERR_RUNS_DONT_COVER_ROWS;
  return MAMBA2_REF_OK;
}

/* ---------------------------------------------------------------------- */
/* CausalConv1D (section "Ops")                                            */
/* ---------------------------------------------------------------------- */

/*
 * For one sequence the conv input is u = history ++ x, where history is the
 * slot's kernel-1 previous inputs (zeros when fresh). Output row t is
 *   silu(bias + sum_k w[:, k] * u[t + k]),   k = 0 .. kernel-1,
 * i.e. w[:, kernel-1] multiplies the current token x[t] = u[t + kernel-1].
 * Afterwards the slot holds u's last kernel-1 rows.
 */
int mamba2_ref_causal_conv1d(void* dst, const void* x, const float* weight,
                             const float* bias, void* conv_state,
                             int32_t num_slots, int32_t rows, int32_t conv_dim,
                             int32_t kernel, int32_t act, int32_t num_seqs,
                             const int32_t* cu_seqlens, const int32_t* slots,
                             const uint8_t* fresh, double* dst_f64) {
  if (!act_ok(act) || conv_dim <= 0 || kernel < 1)
    return MAMBA2_REF_ERR_INVALID_ARGUMENT;
  int st = mamba2_ref_validate_batch(num_seqs, cu_seqlens, slots, num_slots,
                                     rows);
  if (st != MAMBA2_REF_OK) return st;
  if (num_seqs > 0 && (!fresh || !weight || !bias || (kernel > 1 && !conv_state)))
    return MAMBA2_REF_ERR_INVALID_ARGUMENT;
  if (rows > 0 && (!dst || !x)) return MAMBA2_REF_ERR_INVALID_ARGUMENT;

  const int32_t hist = kernel - 1;
  for (int32_t s = 0; s < num_seqs; ++s) {
    const int32_t row0 = cu_seqlens[s];
    const int32_t T = cu_seqlens[s + 1] - row0;
    const size_t slot_base = (size_t)slots[s] * (size_t)hist * (size_t)conv_dim;
    const int is_fresh = fresh[s] != 0;
#pragma omp parallel for schedule(static)
    for (int32_t c = 0; c < conv_dim; ++c) {
      /* u(i) for i in [0, hist + T): the sequence's conv input. */
#define U(i)                                                                  \
  ((i) < hist ? (is_fresh ? 0.0                                               \
                          : act_load(conv_state,                              \
                                     slot_base + (size_t)(i) * conv_dim + c,  \
                                     act))                                    \
              : act_load(x, (size_t)(row0 + (i) - hist) * conv_dim + c, act))
      for (int32_t t = 0; t < T; ++t) {
        double pre = (double)bias[c];
        for (int32_t k = 0; k < kernel; ++k)
          pre += (double)weight[(size_t)c * kernel + k] * U(t + k);
        double out = silu(pre);
        size_t o = (size_t)(row0 + t) * conv_dim + c;
        act_store(dst, o, act, out);
        if (dst_f64) dst_f64[o] = out;
      }
      /* New history = u[T .. T + hist - 1]; read all before writing. */
      double next[64];
      double* nh = hist <= 64 ? next : (double*)malloc(sizeof(double) * hist);
      for (int32_t j = 0; j < hist; ++j) nh[j] = U(T + j);
      for (int32_t j = 0; j < hist; ++j)
        act_store(conv_state, slot_base + (size_t)j * conv_dim + c, act, nh[j]);
      if (nh != next) free(nh);
#undef U
    }
  }
  return MAMBA2_REF_OK;
}

/* ---------------------------------------------------------------------- */
/* SSMScan (sections "Ops" and "CPU reference")                            */
/* ---------------------------------------------------------------------- */

/*
 * Per sequence and head h (group g = h / (heads / ngroups)), per token t:
 *   dt'   = softplus(dt[t, h] + dt_bias[h])
 *   decay = exp(-exp(A_log[h]) * dt')
 *   h[p, n] = fp32( h[p, n] * decay + dt' * B[t, g, n] * x[t, h, p] )
 *   y[t, h, p] = sum_n h[p, n] * C[t, g, n] + D[h] * x[t, h, p]
 * x, B and C sit at fixed column offsets of xbc: x at h*P + p, B at
 * H*P + g*N + n, C at H*P + G*N + g*N + n. The state seeds from the slot
 * (zero when fresh) and is written back after the sequence's last token.
 */
int mamba2_ref_ssd_scan(void* dst, const void* xbc, const void* dt,
                        const float* A_log, const float* dt_bias,
                        const float* D, float* ssm_state, int32_t num_slots,
                        int32_t rows, int32_t heads, int32_t headdim,
                        int32_t d_state, int32_t ngroups, int32_t act,
                        int32_t num_seqs, const int32_t* cu_seqlens,
                        const int32_t* slots, const uint8_t* fresh,
                        double* dst_f64) {
  if (!act_ok(act) || heads <= 0 || headdim <= 0 || d_state <= 0 ||
      ngroups <= 0 || heads % ngroups != 0)
    return MAMBA2_REF_ERR_INVALID_ARGUMENT;
  int st = mamba2_ref_validate_batch(num_seqs, cu_seqlens, slots, num_slots,
                                     rows);
  if (st != MAMBA2_REF_OK) return st;
  if (num_seqs > 0 && (!fresh || !ssm_state || !A_log || !dt_bias || !D))
    return MAMBA2_REF_ERR_INVALID_ARGUMENT;
  if (rows > 0 && (!dst || !xbc || !dt)) return MAMBA2_REF_ERR_INVALID_ARGUMENT;

  const int32_t H = heads, P = headdim, N = d_state, G = ngroups;
  const size_t xbc_cols = (size_t)H * P + 2 * (size_t)G * N;
  const size_t head_state = (size_t)P * N;
  const int64_t work = (int64_t)num_seqs * H;

#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t w = 0; w < work; ++w) {
    const int32_t s = (int32_t)(w / H);
    const int32_t h = (int32_t)(w % H);
    const int32_t g = h / (H / G);
    const int32_t row0 = cu_seqlens[s];
    const int32_t T = cu_seqlens[s + 1] - row0;
    float* slot = ssm_state + ((size_t)slots[s] * H + h) * head_state;
    float* hs = (float*)malloc(sizeof(float) * head_state);
    if (fresh[s]) {
      memset(hs, 0, sizeof(float) * head_state);
    } else {
      memcpy(hs, slot, sizeof(float) * head_state);
    }
    const double A = exp((double)A_log[h]);
    for (int32_t t = 0; t < T; ++t) {
      const size_t r = (size_t)(row0 + t);
      const double dtp = softplus(act_load(dt, r * H + h, act) + (double)dt_bias[h]);
      const double decay = exp(-A * dtp);
      const size_t xo = r * xbc_cols + (size_t)h * P;
      const size_t bo = r * xbc_cols + (size_t)H * P + (size_t)g * N;
      const size_t co = bo + (size_t)G * N;
      for (int32_t p = 0; p < P; ++p) {
        const double xv = act_load(xbc, xo + p, act);
        float* hp = hs + (size_t)p * N;
        double y = 0.0;
        for (int32_t n = 0; n < N; ++n) {
          const double b = act_load(xbc, bo + n, act);
          hp[n] = (float)((double)hp[n] * decay + dtp * b * xv);
          y += (double)hp[n] * act_load(xbc, co + n, act);
        }
        y += (double)D[h] * xv;
        const size_t o = r * (size_t)H * P + (size_t)h * P + p;
        act_store(dst, o, act, y);
        if (dst_f64) dst_f64[o] = y;
      }
    }
    memcpy(slot, hs, sizeof(float) * head_state);
    free(hs);
  }
  return MAMBA2_REF_OK;
}

/* ---------------------------------------------------------------------- */
/* GatedRMSNorm (section "Ops")                                            */
/* ---------------------------------------------------------------------- */

/*
 * v = x * silu(z) (the gate comes before the norm); per row and per group of
 * dim/groups consecutive channels: out = v / sqrt(mean(v^2) + eps) * weight.
 */
int mamba2_ref_gated_rmsnorm(void* dst, const void* x, const void* z,
                             const float* weight, int32_t rows, int32_t dim,
                             int32_t groups, float eps, int32_t act,
                             double* dst_f64) {
  if (!act_ok(act) || rows < 0 || dim <= 0 || groups <= 0 || dim % groups != 0)
    return MAMBA2_REF_ERR_INVALID_ARGUMENT;
  if (rows > 0 && (!dst || !x || !z || !weight))
    return MAMBA2_REF_ERR_INVALID_ARGUMENT;
  const int32_t gs = dim / groups;
#pragma omp parallel for schedule(static)
  for (int32_t r = 0; r < rows; ++r) {
    double* v = (double*)malloc(sizeof(double) * gs);
    for (int32_t g = 0; g < groups; ++g) {
      const size_t base = (size_t)r * dim + (size_t)g * gs;
      double ss = 0.0;
      for (int32_t i = 0; i < gs; ++i) {
        v[i] = act_load(x, base + i, act) * silu(act_load(z, base + i, act));
        ss += v[i] * v[i];
      }
      const double inv = 1.0 / sqrt(ss / gs + (double)eps);
      for (int32_t i = 0; i < gs; ++i) {
        const double o = v[i] * inv * (double)weight[g * gs + i];
        act_store(dst, base + i, act, o);
        if (dst_f64) dst_f64[base + i] = o;
      }
    }
    free(v);
  }
  return MAMBA2_REF_OK;
}

/* ---------------------------------------------------------------------- */
/* Decode step: the three ops on one token per sequence                    */
/* ---------------------------------------------------------------------- */

int mamba2_ref_decode_step(void* dst, const void* xBC, const void* z,
                           const void* dt, const float* conv_w,
                           const float* conv_b, const float* A_log,
                           const float* dt_bias, const float* D,
                           const float* norm_w, int32_t norm_groups, float eps,
                           void* conv_state, float* ssm_state,
                           int32_t num_slots, int32_t heads, int32_t headdim,
                           int32_t d_state, int32_t ngroups,
                           int32_t conv_kernel, int32_t act, int32_t num_seqs,
                           const int32_t* slots, const uint8_t* fresh,
                           double* dst_f64) {
  if (!act_ok(act) || num_seqs < 0 || heads <= 0 || headdim <= 0 ||
      d_state <= 0 || ngroups <= 0 || heads % ngroups != 0 || conv_kernel < 1)
    return MAMBA2_REF_ERR_INVALID_ARGUMENT;
  int32_t* cu = (int32_t*)malloc(sizeof(int32_t) * ((size_t)num_seqs + 1));
  for (int32_t i = 0; i <= num_seqs; ++i) cu[i] = i;
  int st = mamba2_ref_validate_batch(num_seqs, cu, slots, num_slots, num_seqs);
  if (st != MAMBA2_REF_OK) {
    free(cu);
    return st;
  }
  const int32_t d_inner = heads * headdim;
  const int32_t conv_dim = d_inner + 2 * ngroups * d_state;
  void* xbc = malloc(act_size(act) * (size_t)num_seqs * conv_dim + 1);
  void* y = malloc(act_size(act) * (size_t)num_seqs * d_inner + 1);
  st = mamba2_ref_causal_conv1d(xbc, xBC, conv_w, conv_b, conv_state,
                                num_slots, num_seqs, conv_dim, conv_kernel, act,
                                num_seqs, cu, slots, fresh, NULL);
  if (st == MAMBA2_REF_OK)
    st = mamba2_ref_ssd_scan(y, xbc, dt, A_log, dt_bias, D, ssm_state,
                             num_slots, num_seqs, heads, headdim, d_state,
                             ngroups, act, num_seqs, cu, slots, fresh, NULL);
  if (st == MAMBA2_REF_OK)
    st = mamba2_ref_gated_rmsnorm(dst, y, z, norm_w, num_seqs, d_inner,
                                  norm_groups, eps, act, dst_f64);
  free(xbc);
  free(y);
  free(cu);
  return st;
}

/* ---------------------------------------------------------------------- */
/* State size (InfiniLM PR #575 "feat(mamba2): integrate model loading and */
/* recurrent inference", section "Motivation": conv plus fp32 SSM state    */
/* per request, independent of history length)                             */
/* ---------------------------------------------------------------------- */

int64_t mamba2_ref_state_bytes_per_layer(int32_t heads, int32_t headdim,
                                         int32_t d_state, int32_t ngroups,
                                         int32_t conv_kernel, int32_t conv_act) {
  const int64_t conv_dim = (int64_t)heads * headdim + 2LL * ngroups * d_state;
  const int64_t ssm = (int64_t)heads * headdim * d_state * 4;
  const int64_t conv = conv_dim * (conv_kernel - 1) * (int64_t)act_size(conv_act);
  return ssm + conv;
}

int mamba2_ref_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void mamba2_ref_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
