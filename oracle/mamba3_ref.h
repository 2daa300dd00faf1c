/*
 * Plain CPU oracle of the Mamba-3 SISO forward over packed variable-length
 * sequences: TEST INFRASTRUCTURE ONLY (loaded by the tests, the smoke check
 * and the benchmark's CPU-baseline leg; the CUDA product path never calls it
 * and shares no code with it).
 *
 * Semantics: the page "Mamba-3 SISO Long-Ragged Multi-Chunk Joint States Full
 * VJP", its list of the reference's forward steps (1-7) and its dtypes. Where
 * the page leaves a step open this file takes the readings listed in the
 * design notes (the form of the shifted-QK correction, the rotary pairing, the
 * final K state). Those three have no passage to pin against: parity unpinned
 * for them (the tests pin this file to the readings, not to the page). All
 * arithmetic is double; the SSM state is not rounded between tokens (the page
 * asks for no rounding there).
 *
 *   out          [T, H, P] bf16     gated output
 *   final_angle  [S, H, R] bf16     cumulative rotary angle at each sequence's last token
 *   final_ssm    [S, H, P, N] f32   SSM state after the last token
 *   final_k      [S, H, N] f32      rotated, biased K of the last token
 *   final_v      [S, H, P] bf16     V of the last token (bit copy)
 *   q, k         [T, N] bf16        the single Q/K head (expanded to H heads)
 *   v, z         [T, H, P] bf16
 *   adt, dt      [T, H] f32         per-token log-decay and step
 *   trap         [T, H] bf16        trapezoid gate (p = sigmoid(trap))
 *   q_bias, k_bias [H, N] f32
 *   angles       [T, R] bf16        rotary angles (theta = tanh(angles) * pi)
 *   d            [H] f32            skip weight
 *   out_f64      optional [T, H, P] the output before its bf16 rounding
 * A sequence of length zero gets zero final states. Returns 0, or 1 for
 * malformed arguments (nothing written).
 */
#ifndef MAMBA3_REF_H
#define MAMBA3_REF_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

int mamba3_ref_siso_forward(void* out, void* final_angle, float* final_ssm, float* final_k, void* final_v,
                            const void* q, const void* k, const void* v, const float* adt, const float* dt,
                            const void* trap, const float* q_bias, const float* k_bias, const void* angles,
                            const float* d, const void* z, int32_t num_seqs, const int32_t* cu_seqlens,
                            int32_t heads, int32_t headdim, int32_t d_state, int32_t rot_dim, double* out_f64);

#ifdef __cplusplus
}
#endif

#endif
