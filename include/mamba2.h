/*
 * libmamba2 — C ABI of the Mamba2 layer's recurrent hot path on one
 * NVIDIA GB300 (sm_103a).
 *
 * The four operations are the ones gllm PR #85 "feat(backend): Mamba2 ops,
 * with CPU reference implementations" defines in its section "Ops":
 * CausalConv1D, SSMScan and GatedRMSNorm, plus one fused decode step that
 * chains the three for a single token per sequence (the per-token recurrence
 * over conv and SSM cache state that the page "Granite Mamba2 Inference
 * Optimization" names as the decode path), and a prefill that chains the
 * three ops over activations in host memory, streamed in pieces so the
 * host-device copies overlap the compute. The stateful calls take a
 * RecurrentBatch: per sequence a run of rows, a state slot and a fresh flag.
 * mamba2_decode_step_device takes the decode batch from device memory
 * instead, for CUDA-graph replay.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Device buffers are caller-owned device pointers, row-major and
 *    contiguous, 16-byte aligned (mamba2_prefill_host alone takes its
 *    activations and output in host memory). The library allocates no device
 *    memory and keeps no data between calls (the streamed prefill's copy
 *    streams and the static scan scratch's address are kept, per context);
 *    only `dst`, the named slots of the state pools and a caller-provided
 *    workspace are written.
 *  - Batch metadata (mamba2_recurrent_batch) is HOST memory. It is validated
 *    on the host and passed to the kernels by value in their launch
 *    parameters, so the host arrays may be reused as soon as the call returns.
 *    (mamba2_decode_step_device alone reads its batch from device memory and
 *    checks it on the device, as its comment describes.)
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream). Calls are
 *    asynchronous and ordered on that stream; the current CUDA device must be
 *    the one owning the buffers.
 *  - Activations (`act`) are fp32 or bf16. Conv weight/bias, A_log, dt_bias,
 *    D and the norm weight are fp32; the SSM state pool is fp32; the conv
 *    state pool holds activations.
 *  - Errors: every check runs on the host before anything is enqueued, so a
 *    non-OK status means no buffer was touched. Checks run in this order:
 *    arguments, slot range, shared slots, run coverage. MAMBA2_ERR_CUDA
 *    reports a failed launch (nothing else can fail after validation). The
 *    device batch of mamba2_decode_step_device is checked on the device,
 *    with the same rules in the same order.
 *  - A fresh sequence starts from zero state and never reads its slot; its
 *    slot is written with the sequence's end state.
 */
#ifndef MAMBA2_H
#define MAMBA2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mamba2_dtype {
  MAMBA2_F32 = 0,
  MAMBA2_BF16 = 1
} mamba2_dtype;

typedef enum mamba2_status {
  MAMBA2_OK = 0,
  MAMBA2_ERR_INVALID_ARGUMENT = 1,     /* null/misaligned pointer, bad size */
  MAMBA2_ERR_SLOT_OUT_OF_RANGE = 2,    /* slot < 0 or slot >= num_slots */
  MAMBA2_ERR_SLOT_SHARED = 3,          /* two sequences name one slot */
  MAMBA2_ERR_RUNS_DONT_COVER_ROWS = 4, /* cu_seqlens not 0..rows, monotone */
  MAMBA2_ERR_NOT_IMPLEMENTED = 5,      /* shape outside the built kernels */
  MAMBA2_ERR_CUDA = 6,                 /* a kernel launch failed */
  MAMBA2_ERR_WORKSPACE_TOO_SMALL = 7   /* scan workspace below the query */
} mamba2_status;

/* Most sequences one call accepts (the batch travels in launch parameters). */
#define MAMBA2_MAX_SEQS 1024

/*
 * RecurrentBatch (gllm PR #85, section "Ops"): sequence i owns packed rows
 * [cu_seqlens[i], cu_seqlens[i+1]) and state slot slots[i]; fresh[i] != 0
 * means it starts from zero state and never reads its slot. All arrays are
 * host memory; num_seqs <= MAMBA2_MAX_SEQS. cu_seqlens must start at 0, be
 * non-decreasing and end at the call's row count (zero-length runs are
 * allowed: a fresh one zeroes its slot, a resuming one leaves it unchanged).
 */
typedef struct mamba2_recurrent_batch {
  int32_t num_seqs;
  const int32_t* cu_seqlens; /* [num_seqs + 1] */
  const int32_t* slots;      /* [num_seqs] */
  const uint8_t* fresh;      /* [num_seqs] */
} mamba2_recurrent_batch;

/* Layer shape: heads x headdim = d_inner; ngroups B/C groups of d_state;
 * head h reads group h / (heads / ngroups). conv_dim = d_inner +
 * 2 * ngroups * d_state. */
typedef struct mamba2_dims {
  int32_t heads;
  int32_t headdim;
  int32_t d_state;
  int32_t ngroups;
  int32_t conv_kernel;
} mamba2_dims;

/*
 * CausalConv1D (gllm PR #85, section "Ops"): for each sequence, with u its
 * slot's kernel-1 previous inputs (zeros when fresh) followed by its rows of
 * x, row t of dst is silu(bias + sum_k weight[:, k] * u[t + k]); the last tap
 * weight[:, kernel-1] multiplies the current row. Afterwards the slot holds
 * the last kernel-1 rows of u, oldest first (a bit copy of the inputs).
 *
 *   dst        [rows, conv_dim] act      output (must not alias x)
 *   x          [rows, conv_dim] act      packed inputs (xBC columns)
 *   weight     [conv_dim, kernel] f32    depthwise taps, oldest first
 *   bias       [conv_dim] f32
 *   conv_state [num_slots, kernel-1, conv_dim] act, updated in place
 *   kernel     1..4; conv_dim * sizeof(act) must be a multiple of 16.
 */
mamba2_status mamba2_causal_conv1d(void* dst, const void* x,
                                   const float* weight, const float* bias,
                                   void* conv_state, int32_t num_slots,
                                   int32_t rows, int32_t conv_dim,
                                   int32_t kernel, mamba2_dtype act,
                                   const mamba2_recurrent_batch* rb,
                                   void* stream);

/*
 * Bytes of device workspace mamba2_ssd_scan needs for this batch on the
 * current device (0 when none). Query with the same dims, rows and batch as
 * the scan call. The figure is the larger of the needs of the two activation
 * types, so it suffices for the call with either (it is exact for bf16, whose
 * need is never the smaller). Returns 0 for arguments the scan would reject.
 */
size_t mamba2_ssd_scan_workspace_bytes(const mamba2_dims* dims, int32_t rows,
                                       const mamba2_recurrent_batch* rb);

/*
 * SSMScan (gllm PR #85, section "Ops"): per sequence and head h (group
 * g = h / (heads/ngroups)), per row t:
 *   dt'  = softplus(dt[t, h] + dt_bias[h])          (no dt clamp)
 *   h    = h * exp(-exp(A_log[h]) * dt') + dt' * B[t, g] (outer) x[t, h]
 *   y    = h . C[t, g] + D[h] * x[t, h]
 * seeded from the sequence's slot (zero when fresh) and written back to it.
 * x, B and C are read from xbc at fixed column offsets: x at h*headdim,
 * B at d_inner + g*d_state, C at d_inner + ngroups*d_state + g*d_state.
 * Long runs are computed as a chunked scan on the tensor cores.
 *
 *   dst        [rows, heads*headdim] act     y
 *   xbc        [rows, conv_dim] act          the conv output
 *   dt         [rows, heads] act
 *   A_log, dt_bias, D  [heads] f32
 *   ssm_state  [num_slots, heads, headdim, d_state] f32, updated in place
 *   workspace  device scratch of at least
 *              mamba2_ssd_scan_workspace_bytes(...) bytes (may be NULL when
 *              that is 0), 256-byte aligned; its contents need no
 *              initialisation. It holds the segment states of long runs and,
 *              on the tcgen05 path, dt' for every row and head.
 * Built shapes (any heads, ngroups): bf16 headdim 64 x d_state 128 runs on
 * the tcgen05 chunked kernel (128-token chunks), bf16 16 x 16 on the mma.sync
 * chunked kernel (64-token chunks); fp32 activations and other shapes up to
 * headdim 1024, d_state 256 run on the token-serial kernel; larger shapes
 * return MAMBA2_ERR_NOT_IMPLEMENTED.
 */
mamba2_status mamba2_ssd_scan(void* dst, const void* xbc, const void* dt,
                              const float* A_log, const float* dt_bias,
                              const float* D, float* ssm_state,
                              int32_t num_slots, int32_t rows,
                              const mamba2_dims* dims, mamba2_dtype act,
                              const mamba2_recurrent_batch* rb,
                              void* workspace, size_t workspace_bytes,
                              void* stream);

/*
 * Bytes of the library's built-in scan scratch (see
 * mamba2_ssd_scan_static_scratch).
 */
#define MAMBA2_STATIC_SCAN_SCRATCH_BYTES (32u << 20)

/*
 * mamba2_ssd_scan without a caller-provided workspace. The paper has no
 * counterpart to this entry point; it exists for callers that cannot
 * allocate device memory when they call the scan: a server whose allocator
 * has handed all device memory to its state and cache pools, a plugin host
 * that gives its kernels only their input and output buffers, or a latency-
 * critical loop where an allocation's implicit synchronisation is not
 * acceptable.
 *
 * The scratch is a fixed array of MAMBA2_STATIC_SCAN_SCRATCH_BYTES (32 MiB)
 * in the library's own device memory; every GPU that loads the library holds
 * it until the process exits. This call allocates nothing: no cudaMalloc, no
 * cudaFree, no allocating library routine. The first call in each CUDA
 * context (normally the device's primary context) looks up the array's
 * device address with cudaGetSymbolAddress, with that device current, and
 * caches it under the context's ID; make that first call before any stream
 * capture. After cudaDeviceReset the device gets a new primary context with
 * a new ID, so the next call looks the address up again.
 *
 * Arguments, semantics, results and errors are those of mamba2_ssd_scan, plus
 * MAMBA2_ERR_WORKSPACE_TOO_SMALL when the batch needs more scratch than the
 * array holds (mamba2_ssd_scan_workspace_bytes gives an upper bound of the
 * need: a batch for which it is at most the array's size is never rejected
 * for its size; long runs
 * split into many segments and batches of many sequences need more), in
 * which case nothing is enqueued.
 *
 * All calls share the one array and it keeps the last call's contents;
 * nothing in it needs to start at zero (every entry a call reads, the same
 * call wrote first). Calls whose work overlaps on the GPU (different streams,
 * or several host threads) race on it and must be serialised by the caller.
 */
mamba2_status mamba2_ssd_scan_static_scratch(void* dst, const void* xbc, const void* dt,
                                             const float* A_log, const float* dt_bias,
                                             const float* D, float* ssm_state,
                                             int32_t num_slots, int32_t rows,
                                             const mamba2_dims* dims, mamba2_dtype act,
                                             const mamba2_recurrent_batch* rb,
                                             void* stream);

/*
 * GatedRMSNorm (gllm PR #85, section "Ops"): per row and per group of
 * dim/groups consecutive channels, v = x * silu(z) and
 * dst = v / sqrt(mean(v^2) + eps) * weight (the gate is applied before the
 * norm). x, z, dst: [rows, dim] act; weight: [dim] f32. dim % groups == 0
 * and (dim/groups) * sizeof(act) a multiple of 16.
 */
mamba2_status mamba2_gated_rmsnorm(void* dst, const void* x, const void* z,
                                   const float* weight, int32_t rows,
                                   int32_t dim, int32_t groups, float eps,
                                   mamba2_dtype act, void* stream);

/*
 * One decode step: conv -> scan -> gated norm for exactly one new token per
 * sequence, fused in one kernel, with the same rounding points as the three
 * ops above (conv output and y rounded to act). Every run length must be 1:
 * rb->cu_seqlens may be NULL (meaning 0, 1, ..., num_seqs) or must equal
 * that, else MAMBA2_ERR_INVALID_ARGUMENT.
 *
 *   dst   [n, heads*headdim] act     normed output
 *   xBC   [n, conv_dim] act          the token's conv inputs
 *   z     [n, heads*headdim] act     gate
 *   dt    [n, heads] act
 *   conv_w [conv_dim, conv_kernel], conv_b [conv_dim], A_log/dt_bias/D
 *   [heads], norm_w [heads*headdim]: f32
 *   conv_state, ssm_state: the pools, updated in place at rb->slots.
 */
mamba2_status mamba2_decode_step(void* dst, const void* xBC, const void* z,
                                 const void* dt, const float* conv_w,
                                 const float* conv_b, const float* A_log,
                                 const float* dt_bias, const float* D,
                                 const float* norm_w, int32_t norm_groups,
                                 float eps, void* conv_state, float* ssm_state,
                                 int32_t num_slots, const mamba2_dims* dims,
                                 mamba2_dtype act,
                                 const mamba2_recurrent_batch* rb,
                                 void* stream);

/*
 * mamba2_decode_step with the batch in DEVICE memory, so that one captured
 * CUDA graph serves every step: the caller rewrites the slot, fresh and count
 * arrays between replays (InfiniLM PR #575, "Summary": indexed recurrent
 * Decode replayed through Decode graphs; "Benchmark / Performance Impact":
 * graphs cut the per-token latency at batch one).
 *
 *   slots_dev    [capacity] int32, device: slot of sequence s
 *   fresh_dev    [capacity] uint8, device: nonzero = fresh
 *   num_seqs_dev int32, device: n, the sequences of this step (0 <= n <= capacity)
 *   capacity     host, 1 <= capacity <= MAMBA2_MAX_SEQS: the grid is sized
 *                for it; sequence s < n uses row s of dst, xBC, z and dt
 *   status_dev   int32, device: receives this step's mamba2_status
 *
 * The other arguments, layouts and arithmetic are those of mamba2_decode_step
 * (bit-identical results when capacity equals that call's num_seqs; the
 * capacity sets the CTAs per sequence, and with it the order of the norm's
 * partial sums). Two kernels run on the
 * stream. The first checks the batch on the device, in the host check's
 * order and with its rules (gllm PR #85, "Ops": reject a slot out of range or
 * a slot shared by two sequences): n outside [0, capacity] gives
 * MAMBA2_ERR_INVALID_ARGUMENT, then MAMBA2_ERR_SLOT_OUT_OF_RANGE, then
 * MAMBA2_ERR_SLOT_SHARED, else MAMBA2_OK, written to *status_dev. The
 * second is the fused step; it touches nothing (no output row, no pool
 * entry) unless that status is MAMBA2_OK, and rows >= n of dst are never
 * written. So a rejected step leaves every buffer but *status_dev
 * bit-identical; read *status_dev once the stream has passed the call.
 * The return value covers only the host checks (null or misaligned pointers,
 * capacity, shape support: nothing enqueued) and launch failures
 * (MAMBA2_ERR_CUDA). No host synchronisation, allocation or copy: the call
 * can be captured into a CUDA graph.
 */
mamba2_status mamba2_decode_step_device(void* dst, const void* xBC, const void* z,
                                        const void* dt, const float* conv_w,
                                        const float* conv_b, const float* A_log,
                                        const float* dt_bias, const float* D,
                                        const float* norm_w, int32_t norm_groups,
                                        float eps, void* conv_state,
                                        float* ssm_state, int32_t num_slots,
                                        const mamba2_dims* dims, mamba2_dtype act,
                                        const int32_t* slots_dev,
                                        const uint8_t* fresh_dev,
                                        const int32_t* num_seqs_dev,
                                        int32_t capacity, int32_t* status_dev,
                                        void* stream);

/*
 * Bytes of device workspace mamba2_prefill_host needs for this batch, piece
 * size and activation type on the current device; 0 for arguments it would
 * reject. rb->cu_seqlens is required (the call's row count is its last entry).
 */
size_t mamba2_prefill_host_workspace_bytes(const mamba2_dims* dims, mamba2_dtype act,
                                           const mamba2_recurrent_batch* rb,
                                           int32_t piece_rows);

/*
 * Prefill from HOST memory, streamed: the three ops above, CausalConv1D ->
 * SSMScan -> GatedRMSNorm (gllm PR #85, section "Ops"), on a RecurrentBatch
 * whose activations and output live in host memory. The rows are cut into
 * pieces of piece_rows rows, except that the last piece_rows or fewer rows
 * are halved again and again while the remainder keeps at least 1024 rows
 * (pieces of at least 512 rows), so that little compute and copying remains
 * after the last input copy. For each piece, the call copies the
 * piece's xBC, z and dt rows to the device on an internal stream. It runs the
 * three ops on `stream` and copies the piece's output back on a second
 * internal stream. Inputs and outputs are double-buffered in the workspace,
 * so the copies of neighbouring pieces overlap the compute and each other.
 * A run cut by a piece edge continues in the next piece from its slots, as
 * two consecutive calls with fresh = 0 would; only its first part keeps the
 * caller's fresh flag. So conv outputs and conv state are bit-identical to
 * one call over the whole batch. y and the SSM state may differ in rounding
 * where the chunked scan's chunk boundaries move.
 *
 *   out_host  [rows, heads*headdim] act   HOST, written
 *   xBC_host  [rows, conv_dim] act        HOST
 *   z_host    [rows, heads*headdim] act   HOST
 *   dt_host   [rows, heads] act           HOST
 *     (page-locked host memory lets the copies run asynchronously; pageable
 *      memory works but serialises them)
 *   conv_w [conv_dim, conv_kernel], conv_b [conv_dim], A_log / dt_bias / D
 *   [heads], norm_w [heads*headdim]: device f32, as for the ops above
 *   conv_state, ssm_state: the device pools, updated in place at rb->slots
 *   rb         HOST batch; rb->cu_seqlens required; rows = cu_seqlens[num_seqs]
 *   piece_rows rows per piece (>= 1)
 *   workspace  device scratch of at least mamba2_prefill_host_workspace_bytes
 *              bytes, 256-byte aligned; holds the piece buffers and the scan's
 *              workspace (no initialisation needed)
 *
 * Asynchronous like the other calls: it returns once everything is enqueued
 * and `stream` completes after the last output copy. Read out_host, and
 * reuse or free the host inputs and the workspace, only after that. The two
 * internal copy streams and their nine events are created on a host thread's
 * first call in a CUDA context and kept for that thread's later calls in the
 * same context (a new context, as after a device reset, gets new ones); they
 * hold no data between calls, and every use of them is ordered after the
 * previous call's. Calls from one host thread on different caller streams
 * therefore share those copy streams and run their copies one after the
 * other. Errors: the checks of the three ops for the whole batch,
 * then MAMBA2_ERR_WORKSPACE_TOO_SMALL, all before anything is enqueued;
 * MAMBA2_ERR_CUDA if a copy, launch or stream/event creation fails.
 */
mamba2_status mamba2_prefill_host(void* out_host, const void* xBC_host,
                                  const void* z_host, const void* dt_host,
                                  const float* conv_w, const float* conv_b,
                                  const float* A_log, const float* dt_bias,
                                  const float* D, const float* norm_w,
                                  int32_t norm_groups, float eps,
                                  void* conv_state, float* ssm_state,
                                  int32_t num_slots, const mamba2_dims* dims,
                                  mamba2_dtype act,
                                  const mamba2_recurrent_batch* rb,
                                  int32_t piece_rows, void* workspace,
                                  size_t workspace_bytes, void* stream);

/*
 * Bytes of recurrent state one sequence holds in one layer: the fp32 SSM
 * state plus conv_kernel-1 history rows of conv_dim channels at
 * conv_state_dtype (InfiniLM PR #575 "feat(mamba2): integrate model loading
 * and recurrent inference", section "Motivation": about 18.25 MiB per
 * request for mamba2-130m over its 24 layers). -1 for invalid dims.
 */
int64_t mamba2_state_bytes_per_layer(const mamba2_dims* dims,
                                     mamba2_dtype conv_state_dtype);

/*
 * The projections around the recurrent path (the Mamba2 layer of the page
 * "Granite Mamba2 Inference Optimization"; gllm PR #85, "Ops": the model
 * splits in_proj into z, xBC and dt at load, so no split op is needed).
 * tcgen05 GEMMs, bf16 operands, fp32 accumulation, each output rounded once
 * to bf16.
 *
 * mamba2_in_proj: with W = w_in [d_in_proj, d_model] (row-major, the layer's
 * weight as stored: output features x input features) and
 * d_in_proj = d_inner + conv_dim + heads, the product hidden . W^T is written
 * split by columns: [0, d_inner) to z [rows, d_inner], the next conv_dim
 * columns to xBC [rows, conv_dim], the last heads to dt [rows, heads].
 *   hidden [rows, d_model] bf16, all pointers device, 16-byte aligned.
 * bf16 only; d_model, d_inner, conv_dim and heads multiples of 8 (else
 * MAMBA2_ERR_NOT_IMPLEMENTED).
 */
mamba2_status mamba2_in_proj(void* z, void* xBC, void* dt, const void* hidden,
                             const void* w_in, int32_t rows, int32_t d_model,
                             const mamba2_dims* dims, mamba2_dtype act,
                             void* stream);

/*
 * mamba2_out_proj: out [rows, d_model] = x [rows, d_inner] . w_out^T, with
 * w_out [d_model, d_inner] row-major. bf16 only; d_inner and d_model
 * multiples of 8.
 */
mamba2_status mamba2_out_proj(void* out, const void* x, const void* w_out,
                              int32_t rows, int32_t d_inner, int32_t d_model,
                              mamba2_dtype act, void* stream);

/*
 * Padded batches (page "Granite Mamba2 Inference Optimization": the layer's
 * forward takes an attention mask and must serve variable-length padded
 * batches). A padded batch is [batch, seqlen, ...] with mask[b, t] != 0 where
 * position t of row b is a token. Padding positions are not tokens of any
 * sequence, and each row's tokens must form one contiguous span (left or
 * right padding; an all-padding row is an empty sequence).
 *
 * mamba2_padded_spans (host only, no CUDA call): from mask [batch, seqlen]
 * uint8 (host), writes cu_seqlens [batch + 1] (row b's span length, prefix
 * sums from 0: the RecurrentBatch of the packed rows) and first [batch] (the
 * span's first position; 0 for an empty row). MAMBA2_ERR_INVALID_ARGUMENT for
 * a row whose tokens are not one span, batch outside [0, MAMBA2_MAX_SEQS],
 * seqlen < 0, or null pointers (mask may be NULL when batch*seqlen is 0).
 */
mamba2_status mamba2_padded_spans(const uint8_t* mask, int32_t batch,
                                  int32_t seqlen, int32_t* cu_seqlens,
                                  int32_t* first);

/*
 * Gathers the tokens of a padded batch into packed rows: packed row
 * cu_seqlens[b] + k = padded row (b, first[b] + k), width_bytes each.
 *   dst [cu_seqlens[batch], width] device; src [batch, seqlen, width] device
 *   cu_seqlens [batch + 1], first [batch]: host, as mamba2_padded_spans gives
 *   them (any spans inside the rows are accepted)
 * width_bytes > 0. The copy moves 16-, 4-, 2- or 1-byte units, the widest
 * that divides both addresses and the width (any alignment works; 16-byte
 * aligned rows are fastest).
 * MAMBA2_ERR_INVALID_ARGUMENT for a span outside its row, cu_seqlens not
 * starting at 0 or decreasing, or a bad width or null pointer (nothing
 * enqueued).
 */
mamba2_status mamba2_pack_rows(void* dst, const void* src, int32_t batch,
                               int32_t seqlen, int32_t width_bytes,
                               const int32_t* cu_seqlens, const int32_t* first,
                               void* stream);

/*
 * The inverse scatter: padded row (b, t) of dst gets packed row
 * cu_seqlens[b] + t - first[b] inside row b's span and zero bytes outside it.
 *   dst [batch, seqlen, width] device; src [cu_seqlens[batch], width] device.
 * Same checks as mamba2_pack_rows.
 */
mamba2_status mamba2_unpack_rows(void* dst, const void* src, int32_t batch,
                                 int32_t seqlen, int32_t width_bytes,
                                 const int32_t* cu_seqlens, const int32_t* first,
                                 void* stream);

/* Static description of a status code. */
const char* mamba2_status_string(mamba2_status status);

/* Text of the CUDA error behind the calling thread's last MAMBA2_ERR_CUDA. */
const char* mamba2_last_cuda_error(void);

/*
 * Failure detection: how many tensor-core CTAs (scan and projection GEMMs) on
 * the current device gave up waiting on an mbarrier (each wait is bounded; a CTA
 * that gives up writes nothing further, frees its tensor memory and exits).
 * Always 0 on a healthy GPU. Synchronous (reads a device counter);
 * 0xffffffff if the read fails.
 */
unsigned int mamba2_device_timeouts(void);

/*
 * Failure-detection self-test: launches one CTA that waits, through the same
 * bounded mbarrier wait as the tensor-core kernels, on a barrier that nothing
 * arrives at. *status_dev (device int32) becomes 2 when the wait gave up and
 * raised the CTA's abort flag (the expected outcome, after a few seconds),
 * 1 if the phase completed, 3 if it gave up without raising the flag. The
 * context stays usable. MAMBA2_ERR_INVALID_ARGUMENT for a null or misaligned
 * pointer.
 */
mamba2_status mamba2_selftest_bounded_wait(int32_t* status_dev, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MAMBA2_H */
