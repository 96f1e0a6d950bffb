// moe_index.cu -- expert index of a routed batch on the GPU: a stable counting
// sort of the flat (token, slot) routes by expert id, giving expert_offsets
// [E+1] and token_index [n] such that expert e's rows are
// token_index[offsets[e] .. offsets[e+1]-1], in ascending flat order.
//
// Three passes over chunks of 1024 routes:
//   1. per-chunk histograms (shared-memory atomics) -> counts[chunk][e];
//   2. per expert (a block each) an exclusive scan of its counts over the chunks (the
//      chunk's base within the expert's rows) and its total; then one block scans the
//      totals into the offsets;
//   3. per chunk (each expert's cursor starting at its offset plus the chunk's base),
//      the 32 warps take turns in route order; inside a warp the lanes
//      that share an expert rank themselves by __match_any_sync and a popcount
//      of the lower lanes, which keeps equal keys in route order (stable).
// The result is the same permutation on every run (no atomics decide order).
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "situ_internal.h"
#include "situ_ptx.cuh"

namespace situ {
namespace {

constexpr int kChunk = 1024;
constexpr int32_t kMaxExperts = 16384;  // the ABI's bound on E

__global__ void index_count_kernel(const int32_t* __restrict__ ids, int64_t n, int32_t E,
                                   int32_t* __restrict__ counts, uint32_t* status) {
  extern __shared__ int32_t hist[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kChunk;
  for (int i = threadIdx.x; i < kChunk; i += blockDim.x) {
    const int64_t r = base + i;
    if (r < n) {
      const int32_t e = __ldg(ids + r);
      if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
      else record_status(status, SITU_ERR_INDEX);
    }
  }
  __syncthreads();
  int32_t* row = counts + static_cast<int64_t>(blockIdx.x) * E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) row[e] = hist[e];
}

// Per expert (one block each): counts[c][e] <- sum_{c' < c} counts[c'][e], the chunk's base
// within its expert's rows, and offsets[e] <- the expert's total.  Each thread scans a run
// of consecutive chunks; a block-wide scan of the runs' sums joins them.
constexpr int kScanThreads = 256;
__global__ void __launch_bounds__(kScanThreads)
    index_scan_chunks_kernel(int32_t* __restrict__ counts, int32_t nchunks, int32_t E,
                             int32_t* __restrict__ offsets) {
  __shared__ int32_t part[kScanThreads];
  const int e = blockIdx.x;
  const int per = (nchunks + kScanThreads - 1) / kScanThreads;
  const int c0 = threadIdx.x * per;
  const int c1 = min(c0 + per, nchunks);
  int32_t sum = 0;
  for (int c = c0; c < c1; ++c) sum += counts[static_cast<int64_t>(c) * E + e];
  part[threadIdx.x] = sum;
  __syncthreads();
  for (int d = 1; d < kScanThreads; d <<= 1) {
    const int32_t v = threadIdx.x >= static_cast<unsigned>(d) ? part[threadIdx.x - d] : 0;
    __syncthreads();
    part[threadIdx.x] += v;
    __syncthreads();
  }
  int32_t run = part[threadIdx.x] - sum;  // exclusive prefix of this thread's run
  for (int c = c0; c < c1; ++c) {
    int32_t* p = counts + static_cast<int64_t>(c) * E + e;
    const int32_t v = *p;
    *p = run;
    run += v;
  }
  if (threadIdx.x == kScanThreads - 1) offsets[e] = part[threadIdx.x];
}

// offsets[0..E-1] (the experts' totals) <- their exclusive scan; offsets[E] <- the sum.
// One block of 1024 threads.
__global__ void index_scan_experts_kernel(int32_t E, int32_t* __restrict__ offsets) {
  extern __shared__ int32_t tot[];  // [E] totals, then [blockDim] partial sums
  int32_t* partial = tot + E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) tot[e] = offsets[e];
  __syncthreads();
  const int per = (E + blockDim.x - 1) / blockDim.x;
  const int e0 = threadIdx.x * per;
  int32_t sum = 0;
  for (int e = e0; e < e0 + per && e < E; ++e) sum += tot[e];
  partial[threadIdx.x] = sum;
  __syncthreads();
  for (int d = 1; d < static_cast<int>(blockDim.x); d <<= 1) {
    const int32_t v = threadIdx.x >= static_cast<unsigned>(d) ? partial[threadIdx.x - d] : 0;
    __syncthreads();
    partial[threadIdx.x] += v;
    __syncthreads();
  }
  int32_t run = threadIdx.x == 0 ? 0 : partial[threadIdx.x - 1];
  for (int e = e0; e < e0 + per && e < E; ++e) {
    offsets[e] = run;
    run += tot[e];
  }
  if (threadIdx.x == blockDim.x - 1) offsets[E] = partial[threadIdx.x];
}

__global__ void __launch_bounds__(kChunk)
    index_place_kernel(const int32_t* __restrict__ ids, int64_t n, int32_t E,
                       const int32_t* __restrict__ bases, const int32_t* __restrict__ offsets,
                       int32_t* __restrict__ token_index) {
  extern __shared__ int32_t cursor[];
  const int32_t* row = bases + static_cast<int64_t>(blockIdx.x) * E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) cursor[e] = offsets[e] + row[e];
  __syncthreads();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * kChunk + threadIdx.x;
  int32_t e = -1;
  if (r < n) e = __ldg(ids + r);
  const bool valid = r < n && e >= 0 && e < E;
  const unsigned vmask = __ballot_sync(0xFFFFFFFFu, valid);
  for (int w = 0; w < kChunk / 32; ++w) {
    if (warp == w && valid) {
      const unsigned peers = __match_any_sync(vmask, e);
      const unsigned lower = peers & ((1u << lane) - 1u);
      const int32_t pos = cursor[e] + __popc(lower);
      token_index[pos] = static_cast<int32_t>(r);
      // The highest lane of each peer group advances that expert's cursor.
      if ((peers >> lane) == 1u) cursor[e] += __popc(peers);
    }
    __syncthreads();
  }
}

}  // namespace

size_t index_workspace_bytes(int64_t n, int32_t E) {
  const int64_t nchunks = (n + kChunk - 1) / kChunk;
  return static_cast<size_t>(nchunks > 0 ? nchunks : 1) * static_cast<size_t>(E) * 4;
}

cudaError_t launch_build_index(const int32_t* expert_ids, int32_t* offsets,
                               int32_t* token_index, void* workspace, int64_t n, int32_t E,
                               uint32_t* status, cudaStream_t stream) {
  const int32_t nchunks = static_cast<int32_t>((n + kChunk - 1) / kChunk);
  int32_t* counts = static_cast<int32_t*>(workspace);
  const size_t hist_bytes = static_cast<size_t>(E) * 4;
  const size_t scan_bytes = hist_bytes + 1024 * 4;
  cudaError_t e;
  // The shared-memory opt-ins, set once per device for the largest expert count (a
  // per-device property of each kernel; threads racing on the first call each set it).
  static std::atomic<bool> smem_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!smem_set[dev].load(std::memory_order_acquire)) {
    const int max_hist = static_cast<int>(kMaxExperts) * 4;
    for (auto fn : {reinterpret_cast<const void*>(index_count_kernel),
                    reinterpret_cast<const void*>(index_place_kernel)}) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, max_hist);
      if (e != cudaSuccess) return e;
    }
    e = cudaFuncSetAttribute(reinterpret_cast<const void*>(index_scan_experts_kernel),
                             cudaFuncAttributeMaxDynamicSharedMemorySize, max_hist + 1024 * 4);
    if (e != cudaSuccess) return e;
    smem_set[dev].store(true, std::memory_order_release);
  }
  if (E > kMaxExperts) return cudaErrorInvalidValue;
  if (nchunks > 0) {
    index_count_kernel<<<nchunks, 256, hist_bytes, stream>>>(expert_ids, n, E, counts, status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // Per expert, the chunks' bases within its rows and its total (in offsets); then the
  // offsets; the placement adds an expert's offset to its chunk bases.
  index_scan_chunks_kernel<<<E, kScanThreads, 0, stream>>>(counts, nchunks, E, offsets);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  index_scan_experts_kernel<<<1, 1024, scan_bytes, stream>>>(E, offsets);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (nchunks > 0) {
    index_place_kernel<<<nchunks, kChunk, hist_bytes, stream>>>(expert_ids, n, E, counts,
                                                                offsets, token_index);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace situ
