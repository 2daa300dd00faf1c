// C ABI of libmamba2: host-side validation of every argument and of the
// RecurrentBatch, then kernel launches on the caller's stream.
//
// RecurrentBatch rules: gllm PR #85 "feat(backend): Mamba2 ops, with CPU
// reference implementations", section "Ops": a slot out of range, a slot
// shared by two sequences, or run lengths that do not cover the rows are
// rejected before anything is written. All checks here run before the first
// launch, so a non-OK status leaves every buffer untouched.
#include <algorithm>
#include <functional>
#include <cstdio>
#include <cstring>
#include <vector>

#include "../../include/mamba3.h"
#include "kernels.h"

namespace mamba2 {
namespace {

thread_local char g_cuda_error[256] = "";

mamba2_status cuda_fail(cudaError_t e) {
  std::snprintf(g_cuda_error, sizeof g_cuda_error, "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
  return MAMBA2_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// the streamed prefill's internal copy streams and events, kept per host thread and
// CUDA context (see mamba2_prefill_host)
struct CopyLanes {
  unsigned long long ctx;
  cudaStream_t s_in, s_out;
  cudaEvent_t ev[9];
};
// the driver's ID of the current CUDA context (unique for the life of the process,
// never reused); false when there is none or the driver cannot say
bool current_context_id(unsigned long long* id);

size_t act_size(mamba2_dtype a) { return a == MAMBA2_F32 ? 4 : 2; }
bool act_ok(mamba2_dtype a) { return a == MAMBA2_F32 || a == MAMBA2_BF16; }

// Slot range, then shared slots, then coverage of [0, rows).
mamba2_status validate_batch(const mamba2_recurrent_batch* rb, int32_t num_slots, int32_t rows,
                             bool need_cu) {
  if (!rb || rb->num_seqs < 0 || rb->num_seqs > MAMBA2_MAX_SEQS || num_slots < 0 || rows < 0)
    return MAMBA2_ERR_INVALID_ARGUMENT;
  const int n = rb->num_seqs;
  if (n == 0) return rows == 0 ? MAMBA2_OK : MAMBA2_ERR_RUNS_DONT_COVER_ROWS;
  if (!rb->slots || !rb->fresh || (need_cu && !rb->cu_seqlens)) return MAMBA2_ERR_INVALID_ARGUMENT;
  for (int i = 0; i < n; ++i)
    if (rb->slots[i] < 0 || rb->slots[i] >= num_slots) return MAMBA2_ERR_SLOT_OUT_OF_RANGE;
  std::vector<int32_t> sorted(rb->slots, rb->slots + n);
  std::sort(sorted.begin(), sorted.end());
  for (int i = 1; i < n; ++i)
    if (sorted[i] == sorted[i - 1]) return MAMBA2_ERR_SLOT_SHARED;
  if (rb->cu_seqlens) {
    const int32_t* cu = rb->cu_seqlens;
    if (cu[0] != 0) return MAMBA2_ERR_RUNS_DONT_COVER_ROWS;
    for (int i = 0; i < n; ++i)
      if (cu[i + 1] < cu[i]) return MAMBA2_ERR_RUNS_DONT_COVER_ROWS;
    if (cu[n] != rows) return MAMBA2_ERR_RUNS_DONT_COVER_ROWS;
  }
  return MAMBA2_OK;
}

// Fill cu and slot/fresh; tiles are set by the caller.
void fill_table(SeqTable& t, const mamba2_recurrent_batch* rb) {
  t.n = rb->num_seqs;
  t.cu[0] = 0;
  for (int i = 0; i < t.n; ++i) {
    t.cu[i + 1] = rb->cu_seqlens ? rb->cu_seqlens[i + 1] : i + 1;
    t.slot_fresh[i] = (uint32_t)rb->slots[i] | (rb->fresh[i] ? 0x80000000u : 0u);
  }
}

int device_sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

bool dims_ok(const mamba2_dims* d) {
  return d && d->heads > 0 && d->headdim > 0 && d->d_state > 0 && d->ngroups > 0 &&
         d->heads % d->ngroups == 0 && d->conv_kernel >= 1 && d->conv_kernel <= 4 &&
         (int64_t)d->heads * d->headdim + 2LL * d->ngroups * d->d_state < (1LL << 30);
}

// Segmentation of the chunked scan: every sequence is cut into segments of
// seg_chunks chunks, sized so the grid has a few CTAs per SM.
struct ScanPlan {
  bool chunked = false;
  int seg_chunks = 1;
  int state_pieces = 1;  // tcgen05 path: state-pass entries per segment
  int total_segs = 0;
  bool segmented = false;
  size_t ws_state_floats = 0;
  size_t off_decay = 0;  // byte offsets in the workspace
  size_t off_dtp = 0;
  bool has_dtp = false;  // tcgen05 path: dt' precomputed into the workspace
  size_t ws_bytes = 0;
};

ScanPlan plan_scan(const mamba2_dims* d, mamba2_dtype act, const mamba2_recurrent_batch* rb) {
  ScanPlan p;
  p.chunked = scan_chunked_supported(act, d->headdim, d->d_state);
  const int n = rb->num_seqs;
  if (!p.chunked) {
    p.total_segs = n;
    return p;
  }
  const int Q = scan_chunk_tokens(d->headdim, d->d_state);
  const bool tc = scan_uses_tc(act, d->headdim, d->d_state);
  constexpr int kMaxStatePieces = 8;
  // Chunks per segment: both passes run one CTA per SM, so pick the segment
  // length that minimises whole waves x chunks per CTA, counting a state-pass
  // chunk (one product, no output) at about a third of a full-pass chunk and
  // about two chunks of fill and drain per CTA. On the tcgen05 path the state
  // pass may cut each segment into several pieces (one entry each, folded in
  // order by the full pass), so that its CTAs fill the SMs the segments leave.
  // the tcgen05 state pass serves two heads of one group per CTA
  const int64_t state_ctas_per_piece = (tc && (d->heads / d->ngroups) % 2 == 0) ? d->heads / 2 : d->heads;
  std::vector<int64_t> ch(n);
  for (int i = 0; i < n; ++i) ch[i] = (rb->cu_seqlens[i + 1] - rb->cu_seqlens[i] + Q - 1) / Q;
  std::sort(ch.begin(), ch.end(), std::greater<int64_t>());
  const int64_t nsm = std::max(1, device_sm_count());
  const int64_t max_ch = n > 0 ? std::max<int64_t>(1, ch[0]) : 1;
  double best = 1e300;
  p.seg_chunks = (int)max_ch;
  for (int64_t sc = 1; sc <= std::min<int64_t>(max_ch, 4096); ++sc) {
    int64_t extra = 0;  // segments beyond one per sequence = state-pass CTAs per head
    for (int i = 0; i < n && ch[i] > sc; ++i) extra += (ch[i] + sc - 1) / sc - 1;
    const int64_t full_waves = (d->heads * (n + extra) + nsm - 1) / nsm;
    double state_cost = 0.0;
    int pieces = 1;
    if (extra > 0) {
      state_cost = 1e300;
      for (int P = 1; P <= (tc ? std::min<int64_t>(kMaxStatePieces, sc) : 1); ++P) {  // no empty piece
        const int64_t state_waves = (state_ctas_per_piece * extra * P + nsm - 1) / nsm;
        const double c = (double)state_waves * (0.35 * (double)((sc + P - 1) / P) + 1.0);
        if (c < state_cost - 1e-9) {
          state_cost = c;
          pieces = P;
        }
      }
    }
    const double cost = (double)full_waves * (double)(std::min(sc, max_ch) + 2) + state_cost;
    if (cost < best - 1e-9) {
      best = cost;
      p.seg_chunks = (int)sc;
      p.state_pieces = pieces;
    }
  }
  p.total_segs = 0;
  for (int i = 0; i < n; ++i) {
    const int64_t T = rb->cu_seqlens[i + 1] - rb->cu_seqlens[i];
    const int64_t ch = (T + Q - 1) / Q;
    const int segs = (int)std::max<int64_t>(1, (ch + p.seg_chunks - 1) / p.seg_chunks);
    p.segmented |= segs > 1;
    p.total_segs += segs;
  }
  size_t bytes = 0;
  if (!p.segmented) p.state_pieces = 1;
  if (p.segmented) {
    const size_t entries = (size_t)p.total_segs * p.state_pieces;
    p.ws_state_floats = entries * d->heads * d->headdim * d->d_state;
    p.off_decay = (p.ws_state_floats * 4 + 255) / 256 * 256;
    bytes = p.off_decay + entries * d->heads * 4;
  }
  p.has_dtp = scan_uses_tc(act, d->headdim, d->d_state);
  if (p.has_dtp) {
    p.off_dtp = (bytes + 255) / 256 * 256;
    bytes = p.off_dtp + (size_t)rb->cu_seqlens[n] * d->heads * 4;
  }
  p.ws_bytes = bytes;
  return p;
}

void fill_scan_tiles(SeqTable& t, const ScanPlan& p, int Q) {
  t.tile[0] = 0;
  for (int i = 0; i < t.n; ++i) {
    int segs = 1;
    if (p.chunked) {
      const int64_t ch = ((int64_t)t.cu[i + 1] - t.cu[i] + Q - 1) / Q;
      segs = (int)std::max<int64_t>(1, (ch + p.seg_chunks - 1) / p.seg_chunks);
    }
    t.tile[i + 1] = t.tile[i] + segs;
  }
}

// ---- streamed prefill from host memory

// One piece of a streamed prefill: rows [r0, r1) of the call and the runs that
// fall in it, cut at the piece's edges. A run cut by an edge continues in the
// next piece from its slots, so only its first part keeps the caller's fresh
// flag. A zero-length run goes to the piece holding its start row (the last
// piece when it starts at the call's end).
// Pieces are piece_rows long, except that the last piece_rows or fewer rows
// are halved again and again while the remainder keeps at least
// 2 * kMinTailRows rows: once the last input copy has landed, only the last
// small piece's compute and output copy remain.
constexpr int32_t kMinTailRows = 512;
struct Piece {
  int32_t r0 = 0, r1 = 0;
  std::vector<int32_t> cu, slots;
  std::vector<uint8_t> fresh;
  mamba2_recurrent_batch batch() const {
    mamba2_recurrent_batch b;
    b.num_seqs = (int32_t)slots.size();
    b.cu_seqlens = cu.data();
    b.slots = slots.data();
    b.fresh = fresh.data();
    return b;
  }
};

std::vector<Piece> cut_pieces(const mamba2_recurrent_batch* rb, int32_t rows, int32_t piece_rows) {
  std::vector<int32_t> cuts{0};
  int32_t r = 0;
  while (rows - r > piece_rows) cuts.push_back(r += piece_rows);
  for (int32_t left = rows - r; left >= 2 * kMinTailRows; left -= left / 2) cuts.push_back(r += left / 2);
  if (rows > 0) cuts.push_back(rows);
  const size_t np = rows == 0 ? 1 : cuts.size() - 1;
  std::vector<Piece> out(np);
  const int32_t* cu = rb->cu_seqlens;
  for (size_t k = 0; k < np; ++k) {
    Piece& pc = out[k];
    pc.r0 = cuts[k];
    pc.r1 = rows == 0 ? 0 : cuts[k + 1];
    pc.cu.push_back(0);
    for (int i = 0; i < rb->num_seqs; ++i) {
      const int32_t a = cu[i], b = cu[i + 1];
      bool in;
      if (a == b)
        in = (a >= pc.r0 && a < pc.r1) || (a == rows && k == np - 1);
      else
        in = a < pc.r1 && b > pc.r0;
      if (!in) continue;
      const int32_t s0 = std::max(a, pc.r0), s1 = std::min(b, pc.r1);
      pc.cu.push_back(s1 - pc.r0);
      pc.slots.push_back(rb->slots[i]);
      pc.fresh.push_back(rb->fresh[i] && s0 == a ? 1 : 0);
    }
  }
  return out;
}

// Device workspace of a streamed prefill: two input and two output piece
// buffers, the conv output and y of one piece, then the scan's workspace.
struct PrefillLayout {
  size_t x_in[2], z_in[2], dt_in[2], out[2], xbc, y, scan, scan_bytes, total;
};

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

PrefillLayout prefill_layout(const mamba2_dims* d, mamba2_dtype act, int32_t rows, int32_t piece_rows,
                             const std::vector<Piece>& pieces) {
  PrefillLayout L;
  const size_t P = (size_t)std::max<int32_t>(1, std::min<int32_t>(piece_rows, std::max<int32_t>(rows, 1)));
  const size_t a = act_size(act);
  const size_t d_inner = (size_t)d->heads * d->headdim;
  const size_t conv_dim = d_inner + 2 * (size_t)d->ngroups * d->d_state;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  for (int b = 0; b < 2; ++b) {
    L.x_in[b] = take(P * conv_dim * a);
    L.z_in[b] = take(P * d_inner * a);
    L.dt_in[b] = take(P * d->heads * a);
    L.out[b] = take(P * d_inner * a);
  }
  L.xbc = take(P * conv_dim * a);
  L.y = take(P * d_inner * a);
  L.scan_bytes = 0;
  for (const Piece& pc : pieces) {
    const mamba2_recurrent_batch b = pc.batch();
    if (b.num_seqs > 0) L.scan_bytes = std::max(L.scan_bytes, plan_scan(d, act, &b).ws_bytes);
  }
  L.scan = take(L.scan_bytes);
  L.total = off;
  return L;
}

}  // namespace
}  // namespace mamba2

using namespace mamba2;

extern "C" {

const char* mamba2_status_string(mamba2_status s) {
  switch (s) {
    case MAMBA2_OK: return "MAMBA2_OK";
    case MAMBA2_ERR_INVALID_ARGUMENT: return "MAMBA2_ERR_INVALID_ARGUMENT";
    case MAMBA2_ERR_SLOT_OUT_OF_RANGE: return "MAMBA2_ERR_SLOT_OUT_OF_RANGE";
    case MAMBA2_ERR_SLOT_SHARED: return "MAMBA2_ERR_SLOT_SHARED";
    case MAMBA2_ERR_RUNS_DONT_COVER_ROWS: return "MAMBA2_ERR_RUNS_DONT_COVER_ROWS";
    case MAMBA2_ERR_NOT_IMPLEMENTED: return "MAMBA2_ERR_NOT_IMPLEMENTED";
    case MAMBA2_ERR_CUDA: return "MAMBA2_ERR_CUDA";
    case MAMBA2_ERR_WORKSPACE_TOO_SMALL: return "MAMBA2_ERR_WORKSPACE_TOO_SMALL";
  }
  return "MAMBA2_ERR_UNKNOWN";
}

const char* mamba2_last_cuda_error(void) { return g_cuda_error; }

mamba2_status mamba2_selftest_bounded_wait(int32_t* status_dev, void* stream) {
  if (!status_dev || (reinterpret_cast<uintptr_t>(status_dev) & 3u) != 0) return MAMBA2_ERR_INVALID_ARGUMENT;
  const cudaError_t e = launch_bounded_wait_probe(status_dev, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MAMBA2_OK : cuda_fail(e);
}

unsigned int mamba2_device_timeouts(void) {
  const unsigned int a = read_device_timeouts(), b = read_gemm_timeouts(), c = read_m3_timeouts();
  return (a == 0xffffffffu || b == 0xffffffffu || c == 0xffffffffu) ? 0xffffffffu : a + b + c;
}

mamba2_status mamba3_siso_varlen_forward(void* out, void* final_angle, float* final_ssm, float* final_k,
                                         void* final_v, const void* q, const void* k, const void* v,
                                         const float* adt, const float* dt, const void* trap, const float* q_bias,
                                         const float* k_bias, const void* angles, const float* d, const void* z,
                                         const int32_t* cu_seqlens, int32_t num_seqs, int32_t rows, int32_t heads,
                                         int32_t headdim, int32_t d_state, int32_t rot_dim, void* stream) {
  if (num_seqs < 0 || num_seqs > MAMBA2_MAX_SEQS || rows < 0 || heads <= 0 || headdim <= 0 || d_state <= 0 ||
      rot_dim < 0 || 2 * rot_dim > d_state || (num_seqs > 0 && !cu_seqlens))
    return MAMBA2_ERR_INVALID_ARGUMENT;
  if (headdim != 64 || d_state != 128) return MAMBA2_ERR_NOT_IMPLEMENTED;
  if (num_seqs > 0) {
    const void* ptrs[] = {final_ssm, final_k, final_v, q_bias, k_bias, d};
    for (const void* ptr : ptrs)
      if (!ptr || !aligned16(ptr)) return MAMBA2_ERR_INVALID_ARGUMENT;
    if (rot_dim > 0 && (!final_angle || !aligned16(final_angle))) return MAMBA2_ERR_INVALID_ARGUMENT;
  }
  if (rows > 0) {
    const void* ptrs[] = {out, q, k, v, adt, dt, trap, z};
    for (const void* ptr : ptrs)
      if (!ptr || !aligned16(ptr)) return MAMBA2_ERR_INVALID_ARGUMENT;
    if (rot_dim > 0 && (!angles || !aligned16(angles))) return MAMBA2_ERR_INVALID_ARGUMENT;
  }
  if (num_seqs == 0) return rows == 0 ? MAMBA2_OK : MAMBA2_ERR_RUNS_DONT_COVER_ROWS;
  if (cu_seqlens[0] != 0 || cu_seqlens[num_seqs] != rows) return MAMBA2_ERR_RUNS_DONT_COVER_ROWS;
  for (int i = 0; i < num_seqs; ++i)
    if (cu_seqlens[i + 1] < cu_seqlens[i]) return MAMBA2_ERR_RUNS_DONT_COVER_ROWS;
  static_assert(sizeof(Mamba3Args) < 32000, "launch parameter block");
  Mamba3Args a;
  a.out = out;
  a.final_angle = final_angle;
  a.final_ssm = final_ssm;
  a.final_k = final_k;
  a.final_v = final_v;
  a.q = q;
  a.k = k;
  a.v = v;
  a.adt = adt;
  a.dt = dt;
  a.trap = trap;
  a.q_bias = q_bias;
  a.k_bias = k_bias;
  a.angles = angles;
  a.d = d;
  a.z = z;
  a.nseq = num_seqs;
  a.heads = heads;
  a.rot_dim = rot_dim;
  for (int i = 0; i <= num_seqs; ++i) a.cu[i] = cu_seqlens[i];
  // longest sequences first, so that the CTAs that take a second item take short ones
  std::vector<int32_t> order(num_seqs);
  for (int i = 0; i < num_seqs; ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(), [&](int32_t x, int32_t y) {
    return cu_seqlens[x + 1] - cu_seqlens[x] > cu_seqlens[y + 1] - cu_seqlens[y];
  });
  for (int i = 0; i < num_seqs; ++i) a.order[i] = order[i];
  const cudaError_t e = launch_m3_forward(a, std::max(1, device_sm_count()), static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MAMBA2_OK : cuda_fail(e);
}

int64_t mamba2_state_bytes_per_layer(const mamba2_dims* d, mamba2_dtype conv_dtype) {
  if (!dims_ok(d) || !act_ok(conv_dtype)) return -1;
  const int64_t conv_dim = (int64_t)d->heads * d->headdim + 2LL * d->ngroups * d->d_state;
  return (int64_t)d->heads * d->headdim * d->d_state * 4 +
         conv_dim * (d->conv_kernel - 1) * (int64_t)act_size(conv_dtype);
}

mamba2_status mamba2_causal_conv1d(void* dst, const void* x, const float* weight, const float* bias,
                                   void* conv_state, int32_t num_slots, int32_t rows, int32_t conv_dim,
                                   int32_t kernel, mamba2_dtype act, const mamba2_recurrent_batch* rb,
                                   void* stream) {
  if (!act_ok(act) || conv_dim <= 0 || kernel < 1 || rows < 0) return MAMBA2_ERR_INVALID_ARGUMENT;
  if (kernel > 4) return MAMBA2_ERR_NOT_IMPLEMENTED;
  if (((size_t)conv_dim * act_size(act)) % 16 != 0) return MAMBA2_ERR_NOT_IMPLEMENTED;
  if (rb && rb->num_seqs > 0) {
    if (!weight || !bias || (kernel > 1 && !conv_state)) return MAMBA2_ERR_INVALID_ARGUMENT;
    if (!aligned16(weight) || !aligned16(bias)) return MAMBA2_ERR_INVALID_ARGUMENT;
    if ((kernel > 1 && !aligned16(conv_state))) return MAMBA2_ERR_INVALID_ARGUMENT;
  }
  if (rows > 0 && (!dst || !x || !aligned16(dst) || !aligned16(x))) return MAMBA2_ERR_INVALID_ARGUMENT;
  if (rows > 0 && dst == x) return MAMBA2_ERR_INVALID_ARGUMENT;
  mamba2_status st = validate_batch(rb, num_slots, rows, true);
  if (st != MAMBA2_OK) return st;
  if (rb->num_seqs == 0) return MAMBA2_OK;

  ConvArgs a;
  std::memset(&a, 0, sizeof a);
  a.x = x;
  a.dst = dst;
  a.weight = weight;
  a.bias = bias;
  a.conv_state = conv_state;
  a.conv_dim = conv_dim;
  fill_table(a.tab, rb);
  a.tab.tile[0] = 0;
  for (int i = 0; i < a.tab.n; ++i) {
    const int T = a.tab.cu[i + 1] - a.tab.cu[i];
    a.tab.tile[i + 1] = a.tab.tile[i] + std::max(1, (T + kConvRows - 1) / kConvRows);
  }
  cudaError_t e = launch_conv1d(a, act, kernel, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MAMBA2_OK : cuda_fail(e);
}

size_t mamba2_ssd_scan_workspace_bytes(const mamba2_dims* dims, int32_t rows, const mamba2_recurrent_batch* rb) {
  if (!dims_ok(dims)) return 0;
  if (!rb || rb->num_seqs <= 0 || rb->num_seqs > MAMBA2_MAX_SEQS || !rb->cu_seqlens) return 0;
  if (rb->cu_seqlens[0] != 0 || rb->cu_seqlens[rb->num_seqs] != rows) return 0;
  for (int i = 0; i < rb->num_seqs; ++i)
    if (rb->cu_seqlens[i + 1] < rb->cu_seqlens[i]) return 0;
  // the larger of the two activation types' needs: enough for the call with either
  return std::max(plan_scan(dims, MAMBA2_BF16, rb).ws_bytes, plan_scan(dims, MAMBA2_F32, rb).ws_bytes);
}

mamba2_status mamba2_ssd_scan(void* dst, const void* xbc, const void* dt, const float* A_log,
                              const float* dt_bias, const float* D, float* ssm_state, int32_t num_slots,
                              int32_t rows, const mamba2_dims* dims, mamba2_dtype act,
                              const mamba2_recurrent_batch* rb, void* workspace, size_t workspace_bytes,
                              void* stream) {
  if (!act_ok(act) || !dims_ok(dims) || rows < 0) return MAMBA2_ERR_INVALID_ARGUMENT;
  const bool chunked = scan_chunked_supported(act, dims->headdim, dims->d_state);
  if (!chunked && (dims->headdim > kSerialMaxP || dims->d_state > kSerialMaxN))
    return MAMBA2_ERR_NOT_IMPLEMENTED;
  if (rb && rb->num_seqs > 0 && (!ssm_state || !A_log || !dt_bias || !D || !aligned16(ssm_state)))
    return MAMBA2_ERR_INVALID_ARGUMENT;
  if (rows > 0 && (!dst || !xbc || !dt || !aligned16(dst) || !aligned16(xbc)))
    return MAMBA2_ERR_INVALID_ARGUMENT;
  mamba2_status st = validate_batch(rb, num_slots, rows, true);
  if (st != MAMBA2_OK) return st;
  if (rb->num_seqs == 0) return MAMBA2_OK;

  const ScanPlan plan = plan_scan(dims, act, rb);
  if (plan.ws_bytes > 0 && (!workspace || workspace_bytes < plan.ws_bytes))
    return MAMBA2_ERR_WORKSPACE_TOO_SMALL;
  if (plan.ws_bytes > 0 && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return MAMBA2_ERR_INVALID_ARGUMENT;

  ScanArgs a;
  std::memset(&a, 0, sizeof a);
  a.dst = dst;
  a.xbc = xbc;
  a.dt = dt;
  a.A_log = A_log;
  a.dt_bias = dt_bias;
  a.D = D;
  a.ssm_state = ssm_state;
  a.heads = dims->heads;
  a.headdim = dims->headdim;
  a.d_state = dims->d_state;
  a.ngroups = dims->ngroups;
  a.conv_dim = dims->heads * dims->headdim + 2 * dims->ngroups * dims->d_state;
  a.seg_chunks = plan.seg_chunks;
  a.state_pieces = plan.state_pieces;
  if (plan.segmented) {
    a.ws_state = static_cast<float*>(workspace);
    a.ws_decay = reinterpret_cast<float*>(static_cast<char*>(workspace) + plan.off_decay);
  }
  if (plan.has_dtp) a.dtp = reinterpret_cast<float*>(static_cast<char*>(workspace) + plan.off_dtp);
  fill_table(a.tab, rb);
  fill_scan_tiles(a.tab, plan, scan_chunk_tokens(dims->headdim, dims->d_state));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = plan.chunked ? launch_scan_chunked(a, s) : launch_scan_serial(a, act, s);
  return e == cudaSuccess ? MAMBA2_OK : cuda_fail(e);
}

mamba2_status mamba2_gated_rmsnorm(void* dst, const void* x, const void* z, const float* weight, int32_t rows,
                                   int32_t dim, int32_t groups, float eps, mamba2_dtype act, void* stream) {
  if (!act_ok(act) || rows < 0 || dim <= 0 || groups <= 0 || dim % groups != 0 || !(eps >= 0.0f))
    return MAMBA2_ERR_INVALID_ARGUMENT;
  if (((size_t)(dim / groups) * act_size(act)) % 16 != 0) return MAMBA2_ERR_NOT_IMPLEMENTED;
  if (rows == 0) return MAMBA2_OK;
  if (!dst || !x || !z || !weight || !aligned16(dst) || !aligned16(x) || !aligned16(z) || !aligned16(weight))
    return MAMBA2_ERR_INVALID_ARGUMENT;
  NormArgs a{dst, x, z, weight, rows, dim, groups, eps};
  cudaError_t e = launch_gated_rmsnorm(a, act, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MAMBA2_OK : cuda_fail(e);
}

namespace {
// Heads per CTA of the decode state kernel over n sequences: the fewest (a power
// of two, at most 8) that keep the grid near four CTAs per SM or more, so a single
// sequence spreads over one CTA per head and large batches take 8 heads a CTA.
void decode_split(int64_t n, int heads, DecodeArgs& a) {
  const int64_t target = 4 * (int64_t)std::max(1, device_sm_count());
  int hpc = 1;
  while (hpc < kDecodeMaxHeadsPerCta && hpc < heads && n * ((heads + hpc - 1) / hpc) > 2 * target) hpc *= 2;
  a.heads_per_cta = hpc;
  a.ctas_per_seq = (heads + hpc - 1) / hpc;
}
}  // namespace

mamba2_status mamba2_decode_step(void* dst, const void* xBC, const void* z, const void* dt, const float* conv_w,
                                 const float* conv_b, const float* A_log, const float* dt_bias, const float* D,
                                 const float* norm_w, int32_t norm_groups, float eps, void* conv_state,
                                 float* ssm_state, int32_t num_slots, const mamba2_dims* dims, mamba2_dtype act,
                                 const mamba2_recurrent_batch* rb, void* stream) {
  if (!act_ok(act) || !dims_ok(dims) || !(eps >= 0.0f) || norm_groups <= 0) return MAMBA2_ERR_INVALID_ARGUMENT;
  if (!decode_supported(act, *dims, norm_groups)) return MAMBA2_ERR_NOT_IMPLEMENTED;
  if (!rb) return MAMBA2_ERR_INVALID_ARGUMENT;
  const int n = rb->num_seqs;
  if (n > 0) {
    const void* ptrs[] = {dst, xBC, z, dt, conv_w, conv_b, A_log, dt_bias, D, norm_w, ssm_state};
    for (const void* p : ptrs)
      if (!p) return MAMBA2_ERR_INVALID_ARGUMENT;
    if (dims->conv_kernel > 1 && !conv_state) return MAMBA2_ERR_INVALID_ARGUMENT;
    if (!aligned16(dst) || !aligned16(xBC) || !aligned16(z) || !aligned16(ssm_state) ||
        (dims->conv_kernel > 1 && !aligned16(conv_state)) || !aligned16(norm_w))
      return MAMBA2_ERR_INVALID_ARGUMENT;
  }
  mamba2_status st = validate_batch(rb, num_slots, n, false);
  if (st != MAMBA2_OK) return st;
  if (rb->cu_seqlens)
    for (int i = 0; i <= n; ++i)
      if (rb->cu_seqlens[i] != i) return MAMBA2_ERR_INVALID_ARGUMENT;
  if (n == 0) return MAMBA2_OK;

  DecodeArgs a;
  std::memset(&a, 0, sizeof a);
  a.dst = dst;
  a.xBC = xBC;
  a.z = z;
  a.dt = dt;
  a.conv_w = conv_w;
  a.conv_b = conv_b;
  a.A_log = A_log;
  a.dt_bias = dt_bias;
  a.D = D;
  a.norm_w = norm_w;
  a.conv_state = conv_state;
  a.ssm_state = ssm_state;
  a.heads = dims->heads;
  a.headdim = dims->headdim;
  a.d_state = dims->d_state;
  a.ngroups = dims->ngroups;
  a.conv_kernel = dims->conv_kernel;
  a.norm_groups = norm_groups;
  a.eps = eps;
  decode_split(n, dims->heads, a);
  fill_table(a.tab, rb);
  for (int i = 0; i <= n; ++i) a.tab.tile[i] = i;
  cudaError_t e = launch_decode(a, act, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MAMBA2_OK : cuda_fail(e);
}

mamba2_status mamba2_decode_step_device(void* dst, const void* xBC, const void* z, const void* dt,
                                        const float* conv_w, const float* conv_b, const float* A_log,
                                        const float* dt_bias, const float* D, const float* norm_w,
                                        int32_t norm_groups, float eps, void* conv_state, float* ssm_state,
                                        int32_t num_slots, const mamba2_dims* dims, mamba2_dtype act,
                                        const int32_t* slots_dev, const uint8_t* fresh_dev,
                                        const int32_t* num_seqs_dev, int32_t capacity, int32_t* status_dev,
                                        void* stream) {
  if (!act_ok(act) || !dims_ok(dims) || !(eps >= 0.0f) || norm_groups <= 0) return MAMBA2_ERR_INVALID_ARGUMENT;
  if (!decode_supported(act, *dims, norm_groups)) return MAMBA2_ERR_NOT_IMPLEMENTED;
  if (capacity < 1 || capacity > MAMBA2_MAX_SEQS || num_slots < 0) return MAMBA2_ERR_INVALID_ARGUMENT;
  const void* ptrs[] = {dst, xBC, z, dt, conv_w, conv_b, A_log, dt_bias, D, norm_w, ssm_state,
                        slots_dev, fresh_dev, num_seqs_dev, status_dev};
  for (const void* p : ptrs)
    if (!p) return MAMBA2_ERR_INVALID_ARGUMENT;
  if (dims->conv_kernel > 1 && !conv_state) return MAMBA2_ERR_INVALID_ARGUMENT;
  if (!aligned16(dst) || !aligned16(xBC) || !aligned16(z) || !aligned16(ssm_state) ||
      (dims->conv_kernel > 1 && !aligned16(conv_state)) || !aligned16(norm_w))
    return MAMBA2_ERR_INVALID_ARGUMENT;
  const auto aligned4 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 3u) == 0; };
  if (!aligned4(slots_dev) || !aligned4(num_seqs_dev) || !aligned4(status_dev)) return MAMBA2_ERR_INVALID_ARGUMENT;

  DecodeArgs a;
  std::memset(&a, 0, sizeof a);
  a.dst = dst;
  a.xBC = xBC;
  a.z = z;
  a.dt = dt;
  a.conv_w = conv_w;
  a.conv_b = conv_b;
  a.A_log = A_log;
  a.dt_bias = dt_bias;
  a.D = D;
  a.norm_w = norm_w;
  a.conv_state = conv_state;
  a.ssm_state = ssm_state;
  a.heads = dims->heads;
  a.headdim = dims->headdim;
  a.d_state = dims->d_state;
  a.ngroups = dims->ngroups;
  a.conv_kernel = dims->conv_kernel;
  a.norm_groups = norm_groups;
  a.eps = eps;
  // the grid is sized for the capacity (CTAs past the device count leave at once)
  decode_split(capacity, dims->heads, a);
  a.tab.n = capacity;
  a.dev_slots = slots_dev;
  a.dev_fresh = fresh_dev;
  a.dev_n = num_seqs_dev;
  a.dev_status = status_dev;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_check_device_batch(slots_dev, num_seqs_dev, capacity, num_slots, status_dev, st);
  if (e == cudaSuccess) e = launch_decode(a, act, st);
  return e == cudaSuccess ? MAMBA2_OK : cuda_fail(e);
}

mamba2_status mamba2_in_proj(void* z, void* xBC, void* dt, const void* hidden, const void* w_in, int32_t rows,
                             int32_t d_model, const mamba2_dims* dims, mamba2_dtype act, void* stream) {
  if (!act_ok(act) || !dims_ok(dims) || rows < 0 || d_model <= 0) return MAMBA2_ERR_INVALID_ARGUMENT;
  const int32_t d_inner = dims->heads * dims->headdim;
  const int32_t conv_dim = d_inner + 2 * dims->ngroups * dims->d_state;
  if (act != MAMBA2_BF16 || d_model % 8 != 0 || d_inner % 8 != 0 || conv_dim % 8 != 0 || dims->heads % 8 != 0)
    return MAMBA2_ERR_NOT_IMPLEMENTED;
  if (rows == 0) return MAMBA2_OK;
  const void* ptrs[] = {z, xBC, dt, hidden, w_in};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return MAMBA2_ERR_INVALID_ARGUMENT;
  GemmArgs g;
  std::memset(&g, 0, sizeof g);
  g.M = rows;
  g.N = d_inner + conv_dim + dims->heads;
  g.K = d_model;
  g.nseg = 3;
  g.seg_end[0] = d_inner;
  g.seg_end[1] = d_inner + conv_dim;
  g.seg_end[2] = g.N;
  g.dst[0] = z;
  g.dst[1] = xBC;
  g.dst[2] = dt;
  g.ld[0] = d_inner;
  g.ld[1] = conv_dim;
  g.ld[2] = dims->heads;
  const cudaError_t e = launch_gemm_tc(g, hidden, w_in, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MAMBA2_OK : cuda_fail(e);
}

mamba2_status mamba2_out_proj(void* out, const void* x, const void* w_out, int32_t rows, int32_t d_inner,
                              int32_t d_model, mamba2_dtype act, void* stream) {
  if (!act_ok(act) || rows < 0 || d_inner <= 0 || d_model <= 0) return MAMBA2_ERR_INVALID_ARGUMENT;
  if (act != MAMBA2_BF16 || d_inner % 8 != 0 || d_model % 8 != 0) return MAMBA2_ERR_NOT_IMPLEMENTED;
  if (rows == 0) return MAMBA2_OK;
  const void* ptrs[] = {out, x, w_out};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return MAMBA2_ERR_INVALID_ARGUMENT;
  GemmArgs g;
  std::memset(&g, 0, sizeof g);
  g.M = rows;
  g.N = d_model;
  g.K = d_inner;
  g.nseg = 1;
  g.seg_end[0] = d_model;
  g.dst[0] = out;
  g.ld[0] = d_model;
  const cudaError_t e = launch_gemm_tc(g, x, w_out, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MAMBA2_OK : cuda_fail(e);
}

mamba2_status mamba2_padded_spans(const uint8_t* mask, int32_t batch, int32_t seqlen, int32_t* cu_seqlens,
                                  int32_t* first) {
  if (batch < 0 || batch > MAMBA2_MAX_SEQS || seqlen < 0 || !cu_seqlens || !first) return MAMBA2_ERR_INVALID_ARGUMENT;
  if (batch > 0 && seqlen > 0 && !mask) return MAMBA2_ERR_INVALID_ARGUMENT;
  int64_t rows = 0;
  cu_seqlens[0] = 0;
  for (int b = 0; b < batch; ++b) {
    const uint8_t* m = mask ? mask + (int64_t)b * seqlen : nullptr;
    int f = 0;
    while (f < seqlen && m[f] == 0) ++f;
    int e = f;
    while (e < seqlen && m[e] != 0) ++e;
    for (int t = e; t < seqlen; ++t)
      if (m[t] != 0) return MAMBA2_ERR_INVALID_ARGUMENT;  // a hole: two spans in one row
    first[b] = e > f ? f : 0;
    rows += e - f;
    if (rows > INT32_MAX) return MAMBA2_ERR_INVALID_ARGUMENT;
    cu_seqlens[b + 1] = (int32_t)rows;
  }
  return MAMBA2_OK;
}

namespace {
mamba2_status pack_common(void* dst, const void* src, int32_t batch, int32_t seqlen, int32_t width_bytes,
                          const int32_t* cu_seqlens, const int32_t* first, bool unpack, void* stream) {
  if (batch < 0 || batch > MAMBA2_MAX_SEQS || seqlen < 0 || width_bytes <= 0 || !cu_seqlens || (batch > 0 && !first))
    return MAMBA2_ERR_INVALID_ARGUMENT;
  if (cu_seqlens[0] != 0) return MAMBA2_ERR_INVALID_ARGUMENT;
  for (int b = 0; b < batch; ++b) {
    const int64_t len = (int64_t)cu_seqlens[b + 1] - cu_seqlens[b];
    if (len < 0 || first[b] < 0 || first[b] + len > seqlen) return MAMBA2_ERR_INVALID_ARGUMENT;
  }
  const int64_t moved = unpack ? (int64_t)batch * seqlen : (int64_t)cu_seqlens[batch];
  if (moved > 0 && (!dst || !src)) return MAMBA2_ERR_INVALID_ARGUMENT;
  if (moved == 0) return MAMBA2_OK;
  PackArgs a;
  std::memset(&a, 0, sizeof a);
  a.src = src;
  a.dst = dst;
  a.batch = batch;
  a.seqlen = seqlen;
  a.width = width_bytes;
  for (int b = 0; b <= batch; ++b) a.cu[b] = cu_seqlens[b];
  for (int b = 0; b < batch; ++b) a.first[b] = first[b];
  const cudaError_t e = launch_pack_rows(a, unpack, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MAMBA2_OK : cuda_fail(e);
}
}  // namespace

mamba2_status mamba2_pack_rows(void* dst, const void* src, int32_t batch, int32_t seqlen, int32_t width_bytes,
                               const int32_t* cu_seqlens, const int32_t* first, void* stream) {
  return pack_common(dst, src, batch, seqlen, width_bytes, cu_seqlens, first, false, stream);
}

mamba2_status mamba2_unpack_rows(void* dst, const void* src, int32_t batch, int32_t seqlen, int32_t width_bytes,
                                 const int32_t* cu_seqlens, const int32_t* first, void* stream) {
  return pack_common(dst, src, batch, seqlen, width_bytes, cu_seqlens, first, true, stream);
}

size_t mamba2_prefill_host_workspace_bytes(const mamba2_dims* dims, mamba2_dtype act,
                                           const mamba2_recurrent_batch* rb, int32_t piece_rows) {
  if (!act_ok(act) || !dims_ok(dims) || piece_rows < 1 || !rb || !rb->cu_seqlens || rb->num_seqs < 0 ||
      rb->num_seqs > MAMBA2_MAX_SEQS || !rb->slots || !rb->fresh)
    return 0;
  const int n = rb->num_seqs;
  if (rb->cu_seqlens[0] != 0) return 0;
  for (int i = 0; i < n; ++i)
    if (rb->cu_seqlens[i + 1] < rb->cu_seqlens[i]) return 0;
  const int32_t rows = rb->cu_seqlens[n];
  return prefill_layout(dims, act, rows, piece_rows, cut_pieces(rb, rows, piece_rows)).total;
}

mamba2_status mamba2_prefill_host(void* out_host, const void* xBC_host, const void* z_host, const void* dt_host,
                                  const float* conv_w, const float* conv_b, const float* A_log,
                                  const float* dt_bias, const float* D, const float* norm_w, int32_t norm_groups,
                                  float eps, void* conv_state, float* ssm_state, int32_t num_slots,
                                  const mamba2_dims* dims, mamba2_dtype act, const mamba2_recurrent_batch* rb,
                                  int32_t piece_rows, void* workspace, size_t workspace_bytes, void* stream) {
  // ---- every check before anything is enqueued
  if (!act_ok(act) || !dims_ok(dims) || piece_rows < 1 || norm_groups <= 0 || !(eps >= 0.0f))
    return MAMBA2_ERR_INVALID_ARGUMENT;
  const int32_t d_inner = dims->heads * dims->headdim;
  const int32_t conv_dim = d_inner + 2 * dims->ngroups * dims->d_state;
  if (d_inner % norm_groups != 0) return MAMBA2_ERR_INVALID_ARGUMENT;
  if (((size_t)(d_inner / norm_groups) * act_size(act)) % 16 != 0) return MAMBA2_ERR_NOT_IMPLEMENTED;
  if (((size_t)conv_dim * act_size(act)) % 16 != 0) return MAMBA2_ERR_NOT_IMPLEMENTED;
  if (!scan_chunked_supported(act, dims->headdim, dims->d_state) &&
      (dims->headdim > kSerialMaxP || dims->d_state > kSerialMaxN))
    return MAMBA2_ERR_NOT_IMPLEMENTED;
  if (!rb || !rb->cu_seqlens) return MAMBA2_ERR_INVALID_ARGUMENT;
  if (rb->num_seqs < 0 || rb->num_seqs > MAMBA2_MAX_SEQS) return MAMBA2_ERR_INVALID_ARGUMENT;
  const int32_t rows = rb->num_seqs > 0 ? rb->cu_seqlens[rb->num_seqs] : 0;
  if (rb->num_seqs > 0) {
    if (!conv_w || !conv_b || !A_log || !dt_bias || !D || !norm_w || !ssm_state ||
        (dims->conv_kernel > 1 && !conv_state))
      return MAMBA2_ERR_INVALID_ARGUMENT;
    if (!aligned16(conv_w) || !aligned16(conv_b) || !aligned16(norm_w) || !aligned16(ssm_state) ||
        (dims->conv_kernel > 1 && !aligned16(conv_state)))
      return MAMBA2_ERR_INVALID_ARGUMENT;
  }
  if (rows > 0 && (!out_host || !xBC_host || !z_host || !dt_host)) return MAMBA2_ERR_INVALID_ARGUMENT;
  mamba2_status st = validate_batch(rb, num_slots, rows, true);
  if (st != MAMBA2_OK) return st;
  if (rb->num_seqs == 0) return MAMBA2_OK;
  const std::vector<Piece> pieces = cut_pieces(rb, rows, piece_rows);
  const PrefillLayout L = prefill_layout(dims, act, rows, piece_rows, pieces);
  if (!workspace || workspace_bytes < L.total) return MAMBA2_ERR_WORKSPACE_TOO_SMALL;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MAMBA2_ERR_INVALID_ARGUMENT;

  // ---- two copy streams and their events: made on a host thread's first call in a
  // CUDA context and kept for that thread (a new context, as after a device reset, gets
  // new ones), so a call creates nothing; without a context ID to key on, each call
  // makes its own and releases them at its end (destruction waits for the work already
  // enqueued on them). Every use is stream-ordered, so a later call may re-record an
  // event an earlier call's work has yet to reach.
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  CopyLanes lanes = {};
  bool cached = false;
  static thread_local std::vector<CopyLanes> t_lanes;
  unsigned long long ctx = 0;
  const bool keyed = current_context_id(&ctx);
  if (keyed)
    for (const CopyLanes& l : t_lanes)
      if (l.ctx == ctx) {
        lanes = l;
        cached = true;
        break;
      }
  auto release = [&]() {
    if (cached) return;
    for (cudaEvent_t& ev : lanes.ev)
      if (ev) cudaEventDestroy(ev);
    if (lanes.s_in) cudaStreamDestroy(lanes.s_in);
    if (lanes.s_out) cudaStreamDestroy(lanes.s_out);
  };
  cudaError_t e = cudaSuccess;
  if (!cached) {
    e = cudaStreamCreateWithFlags(&lanes.s_in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&lanes.s_out, cudaStreamNonBlocking);
    for (int i = 0; i < 9 && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(&lanes.ev[i], cudaEventDisableTiming);
    if (e != cudaSuccess) {
      release();
      return cuda_fail(e);
    }
    if (keyed) {
      lanes.ctx = ctx;
      t_lanes.push_back(lanes);
      cached = true;
    }
  }
  cudaStream_t s_in = lanes.s_in, s_out = lanes.s_out;
  cudaEvent_t* ev = lanes.ev;  // start, in_ready[2], in_free[2], out_ready[2], out_free[2]
  cudaEvent_t ev_start = ev[0], *in_ready = ev + 1, *in_free = ev + 3, *out_ready = ev + 5, *out_free = ev + 7;

  char* ws = static_cast<char*>(workspace);
  const size_t a = act_size(act);
  // work already on the caller's stream (pools, weights) comes first
  e = cudaEventRecord(ev_start, cs);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s_in, ev_start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s_out, ev_start, 0);
  for (size_t k = 0; k < pieces.size() && e == cudaSuccess; ++k) {
    const Piece& pc = pieces[k];
    const int b = (int)(k & 1);
    const size_t pr = (size_t)(pc.r1 - pc.r0);
    // inputs of piece k into buffer b once piece k-2 has consumed it
    if (k >= 2) e = cudaStreamWaitEvent(s_in, in_free[b], 0);
    if (e == cudaSuccess && pr > 0)
      e = cudaMemcpyAsync(ws + L.x_in[b], static_cast<const char*>(xBC_host) + (size_t)pc.r0 * conv_dim * a,
                          pr * conv_dim * a, cudaMemcpyHostToDevice, s_in);
    if (e == cudaSuccess && pr > 0)
      e = cudaMemcpyAsync(ws + L.z_in[b], static_cast<const char*>(z_host) + (size_t)pc.r0 * d_inner * a,
                          pr * d_inner * a, cudaMemcpyHostToDevice, s_in);
    if (e == cudaSuccess && pr > 0)
      e = cudaMemcpyAsync(ws + L.dt_in[b], static_cast<const char*>(dt_host) + (size_t)pc.r0 * dims->heads * a,
                          pr * dims->heads * a, cudaMemcpyHostToDevice, s_in);
    if (e == cudaSuccess) e = cudaEventRecord(in_ready[b], s_in);
    // conv -> scan -> norm on the caller's stream, into output buffer b once piece k-2's copy-out is done
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, in_ready[b], 0);
    if (e == cudaSuccess && k >= 2) e = cudaStreamWaitEvent(cs, out_free[b], 0);
    if (e != cudaSuccess) break;
    const mamba2_recurrent_batch pb = pc.batch();
    st = mamba2_causal_conv1d(ws + L.xbc, ws + L.x_in[b], conv_w, conv_b, conv_state, num_slots, (int32_t)pr,
                              conv_dim, dims->conv_kernel, act, &pb, cs);
    if (st == MAMBA2_OK)
      st = mamba2_ssd_scan(ws + L.y, ws + L.xbc, ws + L.dt_in[b], A_log, dt_bias, D, ssm_state, num_slots,
                           (int32_t)pr, dims, act, &pb, L.scan_bytes ? ws + L.scan : nullptr, L.scan_bytes, cs);
    if (st == MAMBA2_OK)
      st = mamba2_gated_rmsnorm(ws + L.out[b], ws + L.y, ws + L.z_in[b], norm_w, (int32_t)pr, d_inner,
                                norm_groups, eps, act, cs);
    if (st != MAMBA2_OK) {
      release();
      return st;
    }
    e = cudaEventRecord(in_free[b], cs);
    if (e == cudaSuccess) e = cudaEventRecord(out_ready[b], cs);
    // output of piece k back to the host
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s_out, out_ready[b], 0);
    if (e == cudaSuccess && pr > 0)
      e = cudaMemcpyAsync(static_cast<char*>(out_host) + (size_t)pc.r0 * d_inner * a, ws + L.out[b],
                          pr * d_inner * a, cudaMemcpyDeviceToHost, s_out);
    if (e == cudaSuccess) e = cudaEventRecord(out_free[b], s_out);
  }
  // the caller's stream finishes after the last copy-out
  if (e == cudaSuccess) e = cudaEventRecord(ev_start, s_out);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, ev_start, 0);
  release();
  return e == cudaSuccess ? MAMBA2_OK : cuda_fail(e);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Scan with the library's own scratch, for callers that cannot allocate.
// ---------------------------------------------------------------------------
#include <cuda.h>

#include <mutex>

namespace mamba2 {
namespace {

// The built-in scan scratch: one fixed array in every device that loads the
// library. Host code must not use its name as an address (on the host it is
// only a stand-in); the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_scan_scratch[MAMBA2_STATIC_SCAN_SCRATCH_BYTES];

// The address is cached per CUDA context, identified by the driver's context
// ID (unique for the life of the process, never reused): a device reset or a
// new primary context gets a new ID, so a stale address is never used.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
struct ScratchEntry {
  unsigned long long ctx_id;
  void* addr;
};
constexpr int kMaxScratchEntries = 64;
std::mutex g_scratch_mutex;
ScratchEntry g_scratch_cache[kMaxScratchEntries] = {};
int g_scratch_entries = 0;

template <typename Fn>
Fn driver_fn(const char* name) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<Fn>(fn);
}

bool current_context_id(unsigned long long* id) {
  static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  CUcontext ctx = nullptr;
  return get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx && get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_scan_scratch in the current context. The first call in
// each context looks it up with cudaGetSymbolAddress (which also makes the
// current device's primary context current if none is); later calls in the
// same context take it from the cache.
mamba2_status scan_scratch_address(void** out) {
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  unsigned long long id = 0;
  if (current_context_id(&id))
    for (int i = 0; i < g_scratch_entries; ++i)
      if (g_scratch_cache[i].ctx_id == id) {
        *out = g_scratch_cache[i].addr;
        return MAMBA2_OK;
      }
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_scan_scratch);
  if (e != cudaSuccess) return cuda_fail(e);
  // without a context ID to key on, nothing is cached and every call looks the address up
  if (current_context_id(&id) && g_scratch_entries < kMaxScratchEntries) g_scratch_cache[g_scratch_entries++] = {id, p};
  *out = p;
  return MAMBA2_OK;
}

}  // namespace
}  // namespace mamba2

extern "C" mamba2_status mamba2_ssd_scan_static_scratch(void* dst, const void* xbc, const void* dt,
                                                        const float* A_log, const float* dt_bias, const float* D,
                                                        float* ssm_state, int32_t num_slots, int32_t rows,
                                                        const mamba2_dims* dims, mamba2_dtype act,
                                                        const mamba2_recurrent_batch* rb, void* stream) {
  // Scratch this batch needs (arguments the scan rejects need none; the scan
  // below then reports them).
  size_t need = 0;
  if (act_ok(act) && dims_ok(dims) && rows >= 0 && validate_batch(rb, num_slots, rows, true) == MAMBA2_OK &&
      rb->num_seqs > 0)
    need = plan_scan(dims, act, rb).ws_bytes;
  if (need > MAMBA2_STATIC_SCAN_SCRATCH_BYTES) return MAMBA2_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  const mamba2_status st = scan_scratch_address(&scratch);
  if (st != MAMBA2_OK) return st;
  return mamba2_ssd_scan(dst, xbc, dt, A_log, dt_bias, D, ssm_state, num_slots, rows, dims, act, rb, scratch,
                         MAMBA2_STATIC_SCAN_SCRATCH_BYTES, stream);
}
