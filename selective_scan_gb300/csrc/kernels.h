// Kernel argument blocks and launchers (internal to libmamba2).
//
// Every kernel takes one argument block by value (__grid_constant__), so the
// batch table travels in the launch parameters: no device metadata buffers and
// no host->device copies per call.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mamba2.h"

namespace mamba2 {

// Batch table. Sequence i owns rows [cu[i], cu[i+1]); its slot is
// slot_fresh[i] & 0x7fffffff and it is fresh when bit 31 is set. tile[i] is
// the index of the sequence's first work tile (tile[n] = total tiles); each
// kernel defines what a tile is (conv: kConvRows rows; scan: one segment).
struct SeqTable {
  int32_t n;
  int32_t cu[MAMBA2_MAX_SEQS + 1];
  uint32_t slot_fresh[MAMBA2_MAX_SEQS];
  int32_t tile[MAMBA2_MAX_SEQS + 1];
};

// ---------------------------------------------------------------- conv ----
constexpr int kConvThreads = 256;
constexpr int kConvRows = 14;  // rows per work tile (>= kernel - 1)

struct ConvArgs {
  const void* x;
  void* dst;
  const float* weight;
  const float* bias;
  void* conv_state;
  int32_t conv_dim;
  SeqTable tab;
};
cudaError_t launch_conv1d(const ConvArgs& a, mamba2_dtype act, int kernel, cudaStream_t st);

// ---------------------------------------------------------------- scan ----
constexpr int kChunk = 64;  // tokens per chunk of the chunked scan

struct ScanArgs {
  void* dst;
  const void* xbc;
  const void* dt;
  const float* A_log;
  const float* dt_bias;
  const float* D;
  float* ssm_state;
  float* ws_state;  // [segments * state_pieces, heads, P, N] (null when unsegmented)
  float* ws_decay;  // [segments * state_pieces, heads]
  float* dtp;       // [heads, rows] dt' = softplus(dt + dt_bias) (tcgen05 path; null otherwise)
  int32_t heads, headdim, d_state, ngroups, conv_dim;
  int32_t seg_chunks;  // chunks per segment (tile = segment)
  int32_t state_pieces;  // tcgen05 state pass: entries per segment, each over an equal share of its chunks
  SeqTable tab;
};
// True when the chunked tensor-core kernels cover this shape: tcgen05 for
// headdim 64 x d_state 128 (chunks of kChunkTc tokens), mma.sync for 16 x 16.
bool scan_chunked_supported(mamba2_dtype act, int headdim, int d_state);
constexpr int kChunkTc = 128;
inline bool scan_uses_tc(mamba2_dtype act, int headdim, int d_state) {
  return act == MAMBA2_BF16 && headdim == 64 && d_state == 128;
}
inline int scan_chunk_tokens(int headdim, int d_state) {
  return (headdim == 64 && d_state == 128) ? kChunkTc : kChunk;
}
cudaError_t launch_scan_tc(const ScanArgs& a, cudaStream_t st);
unsigned int read_device_timeouts();
// Chunked scan: state pass over all but the last segment of each sequence,
// then the full pass. The serial kernel is the token-at-a-time fallback.
cudaError_t launch_scan_chunked(const ScanArgs& a, cudaStream_t st);
cudaError_t launch_scan_serial(const ScanArgs& a, mamba2_dtype act, cudaStream_t st);
constexpr int kSerialMaxN = 256;
constexpr int kSerialMaxP = 1024;

// ---------------------------------------------------------------- norm ----
struct NormArgs {
  void* dst;
  const void* x;
  const void* z;
  const float* weight;
  int32_t rows;
  int32_t dim;
  int32_t groups;
  float eps;
};
cudaError_t launch_gated_rmsnorm(const NormArgs& a, mamba2_dtype act, cudaStream_t st);

// -------------------------------------------------------------- decode ----
constexpr int kDecodeThreads = 256;
constexpr int kDecodeMaxHeadsPerCta = 8;  // heads per CTA of the state kernel for large batches
constexpr int kDecodeMaxNormGroups = 64;

struct DecodeArgs {
  void* dst;
  const void* xBC;
  const void* z;
  const void* dt;
  const float* conv_w;
  const float* conv_b;
  const float* A_log;
  const float* dt_bias;
  const float* D;
  const float* norm_w;
  void* conv_state;
  float* ssm_state;
  int32_t heads, headdim, d_state, ngroups, conv_kernel;
  int32_t norm_groups;
  float eps;
  int32_t ctas_per_seq;    // CTAs per sequence of the state kernel
  int32_t heads_per_cta;
  SeqTable tab;            // host batch: tab.n sequences; device batch: tab.n = capacity, rest unused
  // Device batch (all null for a host batch): sequence s < *dev_n has slot dev_slots[s]
  // and is fresh when dev_fresh[s] != 0; no CTA touches anything while *dev_status != 0.
  const int32_t* dev_slots;
  const uint8_t* dev_fresh;
  const int32_t* dev_n;
  const int32_t* dev_status;
};
bool decode_supported(mamba2_dtype act, const mamba2_dims& d, int norm_groups);

// ------------------------------------------------------------ GEMM ----
// dst = A[M, K] . B[N, K]^T (bf16, K contiguous in both), bf16 out. Output columns
// [seg_end[i-1], seg_end[i]) go to dst[i] (row stride ld[i], column 0 = seg_end[i-1]);
// every segment boundary is a multiple of 8 columns and every dst row 16-byte aligned.
struct GemmArgs {
  int32_t M, N, K;
  int32_t nseg;
  int32_t seg_end[3];
  void* dst[3];
  int64_t ld[3];
};
cudaError_t launch_gemm_tc(const GemmArgs& g, const void* A, const void* B, cudaStream_t st);
unsigned int read_gemm_timeouts();

// ------------------------------------------------------------ mamba3 ----
// Mamba-3 SISO varlen forward (head width 64, Q/K width 128). Sequence i owns
// rows [cu[i], cu[i+1]); order[] lists the sequences longest first (the CTAs
// take (sequence, head) items in that order).
struct Mamba3Args {
  void* out;
  void* final_angle;
  float* final_ssm;
  float* final_k;
  void* final_v;
  const void* q;
  const void* k;
  const void* v;
  const float* adt;
  const float* dt;
  const void* trap;
  const float* q_bias;
  const float* k_bias;
  const void* angles;
  const float* d;
  const void* z;
  int32_t nseq, heads, rot_dim;
  int32_t cu[MAMBA2_MAX_SEQS + 1];
  int32_t order[MAMBA2_MAX_SEQS];
};
cudaError_t launch_m3_forward(const Mamba3Args& a, int num_sms, cudaStream_t st);
unsigned int read_m3_timeouts();

// Failure-detection self-test: one bounded wait on a barrier nothing arrives at.
cudaError_t launch_bounded_wait_probe(int32_t* status, cudaStream_t st);

// ------------------------------------------------------------ pack ----
constexpr int kPackThreads = 256;
// Padded [batch, seqlen, width] <-> packed [cu[batch], width]: sequence b's tokens sit
// at padded positions [first[b], first[b] + cu[b+1] - cu[b]) of row b.
struct PackArgs {
  const void* src;
  void* dst;
  int32_t batch, seqlen, width;  // width in bytes
  int32_t cu[MAMBA2_MAX_SEQS + 1];
  int32_t first[MAMBA2_MAX_SEQS];
};
cudaError_t launch_pack_rows(const PackArgs& a, bool unpack, cudaStream_t st);
// The widest copy unit (16, 4, 2 or 1 bytes) dividing both addresses and the width.
int pack_unit_bytes(const void* dst, const void* src, int width);
cudaError_t launch_decode(const DecodeArgs& a, mamba2_dtype act, cudaStream_t st);
// Checks a device batch (count in [0, capacity], slots in range, no slot twice) and
// writes its mamba2_status to *status.
cudaError_t launch_check_device_batch(const int32_t* slots, const int32_t* n, int32_t capacity, int32_t num_slots,
                                      int32_t* status, cudaStream_t st);

}  // namespace mamba2
