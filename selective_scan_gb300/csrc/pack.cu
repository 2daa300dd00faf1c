// Padded batch <-> packed rows: the gathers between a [batch, seqlen, width]
// padded tensor whose row b holds its sequence's tokens in one contiguous span
// [first[b], first[b] + len_b) and the packed [rows, width] layout the ops take
// (sequence b on rows [cu[b], cu[b+1])). The Granite Mamba2 inference page asks
// the layer to serve variable-length padded batches with an attention mask;
// padding positions are not tokens of any sequence.
#include <algorithm>

#include "common.cuh"

namespace mamba2 {
namespace {

// The sequence owning packed row r: largest b with cu[b] <= r (cu non-decreasing).
__device__ __forceinline__ int owner(const PackArgs& a, int64_t r) {
  int lo = 0, hi = a.batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.cu[mid] <= r) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// one packed row per CTA iteration; the row's units (U: 16, 4, 2 or 1 bytes) across the threads
template <typename U>
__global__ void __launch_bounds__(kPackThreads) pack_rows_kernel(const __grid_constant__ PackArgs a) {
  const int vec = a.width / (int)sizeof(U);
  const U* __restrict__ src = static_cast<const U*>(a.src);
  U* __restrict__ dst = static_cast<U*>(a.dst);
  const int64_t rows = a.cu[a.batch];
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const int b = owner(a, r);
    const int64_t from = (int64_t)b * a.seqlen + a.first[b] + (r - a.cu[b]);
    for (int v = threadIdx.x; v < vec; v += blockDim.x) dst[r * vec + v] = src[from * vec + v];
  }
}

// one padded row per CTA iteration: a copy of its packed row inside the span, zeros outside
template <typename U>
__global__ void __launch_bounds__(kPackThreads) unpack_rows_kernel(const __grid_constant__ PackArgs a) {
  const int vec = a.width / (int)sizeof(U);
  const U* __restrict__ src = static_cast<const U*>(a.src);
  U* __restrict__ dst = static_cast<U*>(a.dst);
  const int64_t total = (int64_t)a.batch * a.seqlen;
  U zero;
  memset(&zero, 0, sizeof zero);
  for (int64_t pr = blockIdx.x; pr < total; pr += gridDim.x) {
    const int b = (int)(pr / a.seqlen), t = (int)(pr - (int64_t)b * a.seqlen);
    const int k = t - a.first[b];
    const bool in_span = k >= 0 && k < a.cu[b + 1] - a.cu[b];
    const int64_t from = in_span ? (int64_t)a.cu[b] + k : 0;
    for (int v = threadIdx.x; v < vec; v += blockDim.x) dst[pr * vec + v] = in_span ? src[from * vec + v] : zero;
  }
}

int grid_for(int64_t rows) {
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 152;
  return (int)std::min<int64_t>(rows, (int64_t)sms * 8);
}

template <typename U>
void launch_unit(const PackArgs& a, bool unpack, int64_t n, cudaStream_t st) {
  if (unpack)
    unpack_rows_kernel<U><<<grid_for(n), kPackThreads, 0, st>>>(a);
  else
    pack_rows_kernel<U><<<grid_for(n), kPackThreads, 0, st>>>(a);
}

}  // namespace

int pack_unit_bytes(const void* dst, const void* src, int width) {
  const uintptr_t bits = reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src) | (uintptr_t)width;
  return (bits & 15u) == 0 ? 16 : (bits & 3u) == 0 ? 4 : (bits & 1u) == 0 ? 2 : 1;
}

cudaError_t launch_pack_rows(const PackArgs& a, bool unpack, cudaStream_t st) {
  const int64_t n = unpack ? (int64_t)a.batch * a.seqlen : (int64_t)a.cu[a.batch];
  if (n == 0) return cudaSuccess;
  switch (pack_unit_bytes(a.dst, a.src, a.width)) {
    case 16: launch_unit<uint4>(a, unpack, n, st); break;
    case 4: launch_unit<uint32_t>(a, unpack, n, st); break;
    case 2: launch_unit<uint16_t>(a, unpack, n, st); break;
    default: launch_unit<uint8_t>(a, unpack, n, st); break;
  }
  return cudaGetLastError();
}

}  // namespace mamba2
