/*
 * Plain CPU oracle for the Mamba2 recurrent path: TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the CPU-baseline leg of the benchmark
 * load this library. The product path (the CUDA library) never calls it and
 * shares no code, header or helper with it.
 *
 * Semantics follow gllm PR #85 "feat(backend): Mamba2 ops, with CPU reference
 * implementations", section "Ops" (the four op definitions and the
 * RecurrentBatch rules) and section "CPU reference" (one token at a time, the
 * state rounded to fp32 after every token).
 *
 * All arithmetic is in double. Activations are read exactly from fp32 or bf16
 * and every interface tensor is rounded to the activation type at the end of
 * its op (double -> fp32 round-to-nearest-even -> bf16 round-to-nearest-even).
 * Optional *_f64 outputs receive the same values before that final rounding.
 */
#ifndef MAMBA2_REF_H
#define MAMBA2_REF_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Activation storage types. */
enum { MAMBA2_REF_F32 = 0, MAMBA2_REF_BF16 = 1 };

/* Status codes (numbered like the product's so tests can compare them). */
enum {
  MAMBA2_REF_OK = 0,
  MAMBA2_REF_ERR_INVALID_ARGUMENT = 1,
  MAMBA2_REF_ERR_SLOT_OUT_OF_RANGE = 2,
  MAMBA2_REF_ERR_SLOT_SHARED = 3,
  MAMBA2_REF_ERR_RUNS_DONT_COVER_ROWS = 4
};

/* RecurrentBatch validation: slot range, then shared slots, then coverage. */
int mamba2_ref_validate_batch(int32_t num_seqs, const int32_t* cu_seqlens,
                              const int32_t* slots, int32_t num_slots,
                              int32_t rows);

/* Depthwise causal conv + SiLU over each sequence's run; updates conv slots.
 * x, dst: [rows, conv_dim] act. weight: [conv_dim, kernel] f32. bias:
 * [conv_dim] f32. conv_state: [num_slots, kernel-1, conv_dim] act. */
int mamba2_ref_causal_conv1d(void* dst, const void* x, const float* weight,
                             const float* bias, void* conv_state,
                             int32_t num_slots, int32_t rows, int32_t conv_dim,
                             int32_t kernel, int32_t act, int32_t num_seqs,
                             const int32_t* cu_seqlens, const int32_t* slots,
                             const uint8_t* fresh, double* dst_f64);

/* Selective-scan recurrence. xbc: [rows, H*P + 2*G*N] act (x, then B, then
 * C). dt: [rows, H] act. A_log, dt_bias, D: [H] f32. ssm_state: [num_slots,
 * H, P, N] f32. dst: [rows, H*P] act. */
int mamba2_ref_ssd_scan(void* dst, const void* xbc, const void* dt,
                        const float* A_log, const float* dt_bias,
                        const float* D, float* ssm_state, int32_t num_slots,
                        int32_t rows, int32_t heads, int32_t headdim,
                        int32_t d_state, int32_t ngroups, int32_t act,
                        int32_t num_seqs, const int32_t* cu_seqlens,
                        const int32_t* slots, const uint8_t* fresh,
                        double* dst_f64);

/* rmsnorm(x * silu(z)) * weight with the RMS taken per group of dim/groups
 * channels. x, z, dst: [rows, dim] act. weight: [dim] f32. */
int mamba2_ref_gated_rmsnorm(void* dst, const void* x, const void* z,
                             const float* weight, int32_t rows, int32_t dim,
                             int32_t groups, float eps, int32_t act,
                             double* dst_f64);

/* One token per sequence: conv -> scan -> gated norm, with the same rounding
 * points as the three ops run one after the other. xBC: [n, conv_dim],
 * z: [n, H*P], dt: [n, H]; dst: [n, H*P]. Every run length must be 1.
 * dst_f64 (optional, [n, H*P]) receives the norm's output before its
 * rounding to act, as the gated norm's own dst_f64 does. */
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
                           double* dst_f64);

/* Bytes of recurrent state one sequence holds in one layer: the fp32 SSM
 * state plus kernel-1 conv history columns at conv_act. */
int64_t mamba2_ref_state_bytes_per_layer(int32_t heads, int32_t headdim,
                                         int32_t d_state, int32_t ngroups,
                                         int32_t conv_kernel, int32_t conv_act);

/* Worker threads the OpenMP loops use (1 without OpenMP). */
int mamba2_ref_num_threads(void);
void mamba2_ref_set_num_threads(int n);

#ifdef __cplusplus
}
#endif
#endif
