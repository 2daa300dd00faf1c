/*
 * Mamba-3 SISO forward, the plain definition in double: TEST INFRASTRUCTURE
 * ONLY (see mamba3_ref.h). Steps follow the page "Mamba-3 SISO Long-Ragged
 * Multi-Chunk Joint States Full VJP", list of the reference's forward steps:
 *   1. the single Q/K head serves all H value heads;
 *   2. theta = tanh(angles) * pi; per sequence and head the cumulative angle
 *      phi_t = (sum over s <= t of theta_s * dt_s) mod 2 pi;
 *   3. q_bias and k_bias added, then q and k rotated pair by pair:
 *      (x[2i], x[2i+1]) by phi_t[i] for i < R, the other columns unchanged;
 *   4. p = sigmoid(trap); dt_next and p_next the next token's (zero after the
 *      last token); sg = dt_next * (1 - p_next); scale = dt * p + sg;
 *   5. the causal decayed QK interaction, token by token:
 *      h_t = exp(adt_t) h_{t-1} + scale_t k^_t (x) v_t,   y_t = h_t . q^_t;
 *   6. + d * v_t, minus the shifted-QK correction (q^_t . k^_t) sg_t v_t (the
 *      part of k^_t's weight that belongs to the next token), then the gate
 *      z * sigmoid(z);
 *   7. final states per sequence: angle, SSM state, K (k^ of the last token)
 *      and V (v of the last token).
 */
#include "mamba3_ref.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_load(const void* base, size_t i) {
  uint32_t bits = (uint32_t)((const uint16_t*)base)[i] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* double -> fp32 (round to nearest even) -> bf16 (round to nearest even) */
static uint16_t bf16_round(double v) {
  float f = (float)v;
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static const double kPi = 3.14159265358979323846;

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

int mamba3_ref_siso_forward(void* out, void* final_angle, float* final_ssm, float* final_k, void* final_v,
                            const void* q, const void* k, const void* v, const float* adt, const float* dt,
                            const void* trap, const float* q_bias, const float* k_bias, const void* angles,
                            const float* d, const void* z, int32_t num_seqs, const int32_t* cu_seqlens,
                            int32_t heads, int32_t headdim, int32_t d_state, int32_t rot_dim, double* out_f64) {
  const int H = heads, P = headdim, N = d_state, R = rot_dim;
  if (num_seqs < 0 || H <= 0 || P <= 0 || N <= 0 || R < 0 || 2 * R > N || !cu_seqlens || cu_seqlens[0] != 0) return 1;
  for (int s = 0; s < num_seqs; ++s)
    if (cu_seqlens[s + 1] < cu_seqlens[s]) return 1;
  const double two_pi = 2.0 * kPi;

#ifdef _OPENMP
#pragma omp parallel for collapse(2) schedule(dynamic)
#endif
  for (int s = 0; s < num_seqs; ++s) {
    for (int h = 0; h < H; ++h) {
      const int r0 = cu_seqlens[s], L = cu_seqlens[s + 1] - r0;
      double* st = (double*)calloc((size_t)P * N, sizeof(double));
      double* cum = (double*)calloc((size_t)(R > 0 ? R : 1), sizeof(double));
      double* qr = (double*)malloc(sizeof(double) * N);
      double* kr = (double*)malloc(sizeof(double) * N);
      double* phi = (double*)calloc((size_t)(R > 0 ? R : 1), sizeof(double));
      for (int n = 0; n < N; ++n) kr[n] = 0.0;
      for (int tt = 0; tt < L; ++tt) {
        const int64_t t = r0 + tt;
        const double dtv = (double)dt[t * H + h];
        /* 2. cumulative angle, then mod 2 pi */
        for (int i = 0; i < R; ++i) {
          cum[i] += tanh(bf16_load(angles, (size_t)t * R + i)) * kPi * dtv;
          phi[i] = cum[i] - two_pi * floor(cum[i] / two_pi);
        }
        /* 3. biases, then rotation of the pairs (2i, 2i+1), i < R */
        for (int n = 0; n < N; ++n) {
          qr[n] = bf16_load(q, (size_t)t * N + n) + (double)q_bias[h * N + n];
          kr[n] = bf16_load(k, (size_t)t * N + n) + (double)k_bias[h * N + n];
        }
        for (int i = 0; i < R; ++i) {
          const double c = cos(phi[i]), sn = sin(phi[i]);
          const double q0 = qr[2 * i], q1 = qr[2 * i + 1], k0 = kr[2 * i], k1 = kr[2 * i + 1];
          qr[2 * i] = q0 * c - q1 * sn;
          qr[2 * i + 1] = q0 * sn + q1 * c;
          kr[2 * i] = k0 * c - k1 * sn;
          kr[2 * i + 1] = k0 * sn + k1 * c;
        }
        /* 4. trapezoid weights */
        const double p = sigmoid(bf16_load(trap, (size_t)t * H + h));
        double dt_next = 0.0, p_next = 0.0;
        if (tt + 1 < L) {
          dt_next = (double)dt[(t + 1) * H + h];
          p_next = sigmoid(bf16_load(trap, (size_t)(t + 1) * H + h));
        }
        const double sg = dt_next * (1.0 - p_next);
        const double scale = dtv * p + sg;
        const double decay = exp((double)adt[t * H + h]);
        double qk = 0.0;
        for (int n = 0; n < N; ++n) qk += qr[n] * kr[n];
        /* 5-6. state, output, skip, correction, gate */
        for (int pp = 0; pp < P; ++pp) {
          const size_t vi = ((size_t)t * H + h) * P + pp;
          const double vv = bf16_load(v, vi);
          double y = 0.0;
          for (int n = 0; n < N; ++n) {
            double* hp = st + (size_t)pp * N + n;
            *hp = decay * *hp + scale * kr[n] * vv;
            y += *hp * qr[n];
          }
          y += (double)d[h] * vv - qk * sg * vv;
          const double zz = bf16_load(z, vi);
          const double o = y * zz * sigmoid(zz);
          ((uint16_t*)out)[vi] = bf16_round(o);
          if (out_f64) out_f64[vi] = o;
        }
      }
      /* 7. final states */
      for (int i = 0; i < R; ++i) ((uint16_t*)final_angle)[((size_t)s * H + h) * R + i] = bf16_round(L > 0 ? phi[i] : 0.0);
      for (size_t e = 0; e < (size_t)P * N; ++e) final_ssm[((size_t)s * H + h) * P * N + e] = (float)st[e];
      for (int n = 0; n < N; ++n) final_k[((size_t)s * H + h) * N + n] = (float)(L > 0 ? kr[n] : 0.0);
      for (int pp = 0; pp < P; ++pp)
        ((uint16_t*)final_v)[((size_t)s * H + h) * P + pp] =
            L > 0 ? ((const uint16_t*)v)[((size_t)(r0 + L - 1) * H + h) * P + pp] : (uint16_t)0;
      free(st);
      free(cum);
      free(qr);
      free(kr);
      free(phi);
    }
  }
  return 0;
}
