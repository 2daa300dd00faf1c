/*
 * libmamba2 — Mamba-3 SISO varlen forward, the second workload of the same
 * library (same status codes and conventions as mamba2.h: caller-owned device
 * buffers, host batch metadata validated before anything is enqueued,
 * asynchronous on `stream`).
 *
 * The operator is the forward half of the page "Mamba-3 SISO Long-Ragged
 * Multi-Chunk Joint States Full VJP" (section "What You Have", steps 1-7, and
 * the dtype paragraph of "Hard Constraints"). For each packed sequence and
 * each value head h (the single Q/K head serves all of them), token by token:
 *
 *   theta = tanh(angles) * pi; phi_t = (sum_{s<=t} theta_s * dt_s[h]) mod 2 pi,
 *     one angle per rotary pair i < rot_dim
 *   q^_t = rotate(q_t + q_bias[h]), k^_t = rotate(k_t + k_bias[h]): columns
 *     (2i, 2i+1), i < rot_dim, turned by phi_t[i]; the other columns as they are
 *   p = sigmoid(trap); dt_next, p_next the next token's (zero after the last);
 *     sg = dt_next * (1 - p_next); scale = dt * p + sg
 *   h_t = exp(adt_t) h_{t-1} + scale_t * v_t (x) k^_t        (h [headdim][d_state])
 *   y_t = h_t . q^_t + d[h] * v_t - (q^_t . k^_t) * sg_t * v_t
 *   out_t = y_t * z_t * sigmoid(z_t)
 *
 * State, angle accumulation and the next-token shift reset at every sequence
 * boundary; every sequence starts from zero state. Two steps are named on the
 * page without their form; this library reads them as follows: the shifted-QK
 * correction is the term (q^_t . k^_t) sg_t v_t (the share of token t's own
 * weight that belongs to the next token), and the final K state is the
 * rotated k^ of the sequence's last token.
 *
 *   out         [rows, heads, headdim] bf16      output
 *   final_angle [num_seqs, heads, rot_dim] bf16  phi of the last token
 *   final_ssm   [num_seqs, heads, headdim, d_state] f32   h after the last token
 *   final_k     [num_seqs, heads, d_state] f32   k^ of the last token
 *   final_v     [num_seqs, heads, headdim] bf16  v of the last token (a copy)
 *   q, k        [rows, d_state] bf16             the single Q/K head
 *   v, z        [rows, heads, headdim] bf16
 *   adt, dt     [rows, heads] f32                log-decay and step per head
 *   trap        [rows, heads] bf16
 *   q_bias, k_bias [heads, d_state] f32
 *   angles      [rows, rot_dim] bf16 (angles and final_angle may be NULL when
 *               rot_dim == 0)
 *   d           [heads] f32
 *   cu_seqlens  HOST [num_seqs + 1], 0 = cu[0] <= cu[1] <= ... = rows
 *
 * An empty sequence has zero final states. Device pointers are 16-byte
 * aligned. Built shape: headdim 64, d_state 128, 0 <= rot_dim <= 64, any
 * number of heads; other headdim / d_state return MAMBA2_ERR_NOT_IMPLEMENTED.
 * Errors, all before anything is enqueued: MAMBA2_ERR_INVALID_ARGUMENT for a
 * null or misaligned pointer, negative sizes, num_seqs above MAMBA2_MAX_SEQS
 * or 2 * rot_dim > d_state; MAMBA2_ERR_RUNS_DONT_COVER_ROWS when cu_seqlens
 * does not run from 0 to rows without decreasing; MAMBA2_ERR_CUDA when the
 * launch fails.
 */
#ifndef MAMBA3_H
#define MAMBA3_H

#include "mamba2.h"

#ifdef __cplusplus
extern "C" {
#endif

mamba2_status mamba3_siso_varlen_forward(void* out, void* final_angle, float* final_ssm, float* final_k,
                                         void* final_v, const void* q, const void* k, const void* v,
                                         const float* adt, const float* dt, const void* trap,
                                         const float* q_bias, const float* k_bias, const void* angles,
                                         const float* d, const void* z, const int32_t* cu_seqlens,
                                         int32_t num_seqs, int32_t rows, int32_t heads, int32_t headdim,
                                         int32_t d_state, int32_t rot_dim, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MAMBA3_H */
