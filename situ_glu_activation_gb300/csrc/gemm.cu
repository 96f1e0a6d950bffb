// gemm.cu -- the bf16 tcgen05 GEMMs of the SiTU-GLU feed-forward on sm_103a
// (the kernel itself is in gemm_kernel.cuh): dispatch of the forward GEMMs
//   gate_up + SiTU-GLU:  h[r, j] = SiTU-GLU(x[r] . Wgu[j], x[r] . Wgu[I + j])
//   down:                y[r, m] = h[r] . Wd[m]
// ("DenseFFN and SituGLU - Docs - Kimi K3 from Scratch", "Two linear maps and a
// guarded compiled branch"), dense or grouped over experts, and of the backward
// GEMMs (the activation's derivative in the dh epilogue; MN-major operands; the
// K-grouped per-expert weight gradients); plus the small kernels of the grouped
// path (per-group tile and unit prefixes, row gather) and the bounded-wait self test.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include <cstring>
#include <vector>

#include "gemm_kernel.cuh"

namespace situ {
namespace {

// ---------------------------------------------------------------------------
// Small helper kernels of the grouped path
// ---------------------------------------------------------------------------

// Per-group work prefixes of the grouped GEMMs, and validation of the offsets:
//   tiles[g]    = sum over g' < g of m_g'            (m_g = ceil(rows_g / 128))
//   units_gu[g] = sum over g' < g of units(m_g', n_gu) (work units, gate_up GEMM)
//   units_dn[g] = sum over g' < g of units(m_g', n_dn) (work units, down GEMM)
// Invalid offsets (not starting at 0, decreasing, not ending at R) zero all three
// so the GEMMs do nothing, and record SITU_ERR_INDEX.  One block of 1024 threads.
// Rank of each group by (row count descending, index ascending) -- a strict total order,
// so order[] is a permutation of 0..G-1 for any offsets (invalid offsets are caught by
// group_tiles_kernel, which then stops the GEMMs).
__global__ void group_order_kernel(const int32_t* __restrict__ off, int32_t G,
                                   int32_t* __restrict__ order) {
  for (int32_t g = threadIdx.x; g < G; g += blockDim.x) {
    const int32_t rows = __ldg(off + g + 1) - __ldg(off + g);
    int32_t rank = 0;
    for (int32_t h = 0; h < G; ++h) {
      const int32_t rh = __ldg(off + h + 1) - __ldg(off + h);
      rank += (rh > rows || (rh == rows && h < g)) ? 1 : 0;
    }
    order[rank] = g;
  }
}

__global__ void group_tiles_kernel(const int32_t* __restrict__ off, int32_t G, int64_t R,
                                   int32_t n_gu, int32_t n_dn, int32_t* __restrict__ tiles,
                                   int32_t* __restrict__ units_gu,
                                   int32_t* __restrict__ units_dn, uint32_t* status,
                                   int two_cta) {
  // Units of a group with m m-tiles: two-CTA pairs (ceil(m / 2) per n-tile), or tiles.
  auto units = [two_cta](int32_t m, int32_t n) { return two_cta ? ((m + 1) >> 1) * n : m * n; };
  __shared__ int32_t partial[3][1024];
  __shared__ int bad;
  if (threadIdx.x == 0) bad = 0;
  __syncthreads();
  const int per = (G + blockDim.x - 1) / blockDim.x;
  const int g0 = threadIdx.x * per;
  int32_t sum[3] = {0, 0, 0};
  for (int g = g0; g < g0 + per && g < G; ++g) {
    const int32_t a = off[g], b = off[g + 1];
    if (b < a) bad = 1;
    const int32_t m = (b - a + kBM - 1) / kBM;
    sum[0] += m;
    sum[1] += units(m, n_gu);
    sum[2] += units(m, n_dn);
  }
  if (threadIdx.x == 0 && (off[0] != 0 || static_cast<int64_t>(off[G]) != R)) bad = 1;
  for (int k = 0; k < 3; ++k) partial[k][threadIdx.x] = sum[k];
  __syncthreads();
  // Inclusive scans of the per-thread sums (Hillis-Steele over one block).
  for (int d = 1; d < static_cast<int>(blockDim.x); d <<= 1) {
    int32_t v[3];
    for (int k = 0; k < 3; ++k)
      v[k] = threadIdx.x >= static_cast<unsigned>(d) ? partial[k][threadIdx.x - d] : 0;
    __syncthreads();
    for (int k = 0; k < 3; ++k) partial[k][threadIdx.x] += v[k];
    __syncthreads();
  }
  if (bad) {
    for (int g = threadIdx.x; g <= G; g += blockDim.x) tiles[g] = units_gu[g] = units_dn[g] = 0;
    if (threadIdx.x == 0) record_status(status, SITU_ERR_INDEX);
    return;
  }
  int32_t run[3];
  for (int k = 0; k < 3; ++k) run[k] = threadIdx.x == 0 ? 0 : partial[k][threadIdx.x - 1];
  for (int g = g0; g < g0 + per && g < G; ++g) {
    tiles[g] = run[0];
    units_gu[g] = run[1];
    units_dn[g] = run[2];
    const int32_t m = (off[g + 1] - off[g] + kBM - 1) / kBM;
    run[0] += m;
    run[1] += units(m, n_gu);
    run[2] += units(m, n_dn);
  }
  if (threadIdx.x == blockDim.x - 1) {
    tiles[G] = partial[0][threadIdx.x];
    units_gu[G] = partial[1][threadIdx.x];
    units_dn[G] = partial[2][threadIdx.x];
  }
}

// One warp per gathered row: x_perm[r] = x[token_index[r] / k_eff] (16-byte copies, eight
// loads in flight per lane before their stores).
__global__ void gather_rows_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ tix,
                                   uint4* __restrict__ xp, int64_t R, int32_t k_eff,
                                   int64_t vec_per_row, int64_t T, uint32_t* status) {
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       r < R; r += warps) {
    const int32_t flat = __ldg(tix + r);
    const int64_t t = flat / k_eff;
    uint4* dst = xp + r * vec_per_row;
    if (flat < 0 || t >= T) {
      if ((threadIdx.x & 31) == 0) record_status(status, SITU_ERR_INDEX);
      for (int64_t v = threadIdx.x & 31; v < vec_per_row; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const uint4* src = x + t * vec_per_row;
    int64_t v = threadIdx.x & 31;
    for (; v + 7 * 32 < vec_per_row; v += 8 * 32) {
      uint4 q[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) q[j] = __ldg(src + v + 32 * j);
#pragma unroll
      for (int j = 0; j < 8; ++j) dst[v + 32 * j] = q[j];
    }
    for (; v < vec_per_row; v += 32) dst[v] = __ldg(src + v);
  }
}

__global__ void bounded_wait_selftest_kernel(uint64_t limit_ns, uint32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
    // Nothing ever arrives on this barrier: the wait must give up by itself.
    mbar_wait(smem_u32(&bar), 0, status, limit_ns);
  }
}

}  // namespace

cudaError_t launch_gemm_situ(const GemmShape& s, const SituParams& p, Caps caps,
                             uint32_t* status, int num_sms, cudaStream_t stream) {
  // Storing the pre-activation (training forward) is a separate instantiation,
  // so the inference epilogue carries none of it.
  if (s.gu_store) {
    switch (caps) {
      case Caps::kBoth:
        return launch<Epi::kSitu, Caps::kBoth, true, Major::kKMajor, 0, true>(s, p, status, num_sms, stream);
      case Caps::kGateOnly:
        return launch<Epi::kSitu, Caps::kGateOnly, true, Major::kKMajor, 0, true>(s, p, status, num_sms, stream);
      case Caps::kUpOnly:
        return launch<Epi::kSitu, Caps::kUpOnly, true, Major::kKMajor, 0, true>(s, p, status, num_sms, stream);
      case Caps::kNone:
        return launch<Epi::kSitu, Caps::kNone, true, Major::kKMajor, 0, true>(s, p, status, num_sms, stream);
    }
    return cudaErrorInvalidValue;
  }
  switch (caps) {
    case Caps::kBoth: return launch<Epi::kSitu, Caps::kBoth, false, Major::kKMajor, 0, true>(s, p, status, num_sms, stream);
    case Caps::kGateOnly:
      return launch<Epi::kSitu, Caps::kGateOnly, false, Major::kKMajor, 0, true>(s, p, status, num_sms, stream);
    case Caps::kUpOnly: return launch<Epi::kSitu, Caps::kUpOnly, false, Major::kKMajor, 0, true>(s, p, status, num_sms, stream);
    case Caps::kNone: return launch<Epi::kSitu, Caps::kNone, false, Major::kKMajor, 0, true>(s, p, status, num_sms, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_plain(const GemmShape& s, uint32_t* status, int num_sms,
                              cudaStream_t stream) {
  if (s.a_mn_major && s.b_mn_major && s.k_group_offsets)
    return launch<Epi::kPlain, Caps::kBoth, false, Major::kABMNGrouped, 0, true>(
        s, SituParams{}, status, num_sms, stream);
  if (s.a_mn_major && s.b_mn_major)
    return launch<Epi::kPlain, Caps::kBoth, false, Major::kABMN, 0, true>(s, SituParams{}, status,
                                                                         num_sms, stream);
  if (s.b_mn_major)
    return launch<Epi::kPlain, Caps::kBoth, false, Major::kBMN, 0, true>(s, SituParams{}, status,
                                                                        num_sms, stream);
  if (s.a_mn_major) return cudaErrorInvalidValue;
  return launch<Epi::kPlain, Caps::kBoth, false, Major::kKMajor, 0, true>(s, SituParams{}, status,
                                                                        num_sms, stream);
}

cudaError_t launch_gemm_situ_bwd(const GemmShape& s, const SituParams& p, Caps caps,
                                 uint32_t* status, int num_sms, cudaStream_t stream) {
  if (s.a_mn_major) return cudaErrorInvalidValue;
  if (s.b_mn_major) {
    switch (caps) {
      case Caps::kBoth:
        return launch<Epi::kSituBwd, Caps::kBoth, false, Major::kBMN, 0, true>(s, p, status, num_sms, stream);
      case Caps::kGateOnly:
        return launch<Epi::kSituBwd, Caps::kGateOnly, false, Major::kBMN, 0, true>(s, p, status, num_sms,
                                                                         stream);
      case Caps::kUpOnly:
        return launch<Epi::kSituBwd, Caps::kUpOnly, false, Major::kBMN, 0, true>(s, p, status, num_sms,
                                                                       stream);
      case Caps::kNone:
        return launch<Epi::kSituBwd, Caps::kNone, false, Major::kBMN, 0, true>(s, p, status, num_sms, stream);
    }
    return cudaErrorInvalidValue;
  }
  switch (caps) {
    case Caps::kBoth: return launch<Epi::kSituBwd, Caps::kBoth, false, Major::kKMajor, 0, true>(s, p, status, num_sms, stream);
    case Caps::kGateOnly:
      return launch<Epi::kSituBwd, Caps::kGateOnly, false, Major::kKMajor, 0, true>(s, p, status, num_sms, stream);
    case Caps::kUpOnly:
      return launch<Epi::kSituBwd, Caps::kUpOnly, false, Major::kKMajor, 0, true>(s, p, status, num_sms, stream);
    case Caps::kNone: return launch<Epi::kSituBwd, Caps::kNone, false, Major::kKMajor, 0, true>(s, p, status, num_sms, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_ffn_fused(const GemmShape& s_gu, const GemmShape& s_dn, const SituParams& p,
                             Caps caps, int32_t* h_ready, uint32_t* status, int num_sms,
                             cudaStream_t stream) {
  switch (caps) {
    case Caps::kBoth:
      return launch_ffn_fused_impl<Caps::kBoth>(s_gu, s_dn, p, h_ready, status, num_sms, stream);
    case Caps::kGateOnly:
      return launch_ffn_fused_impl<Caps::kGateOnly>(s_gu, s_dn, p, h_ready, status, num_sms,
                                                    stream);
    case Caps::kUpOnly:
      return launch_ffn_fused_impl<Caps::kUpOnly>(s_gu, s_dn, p, h_ready, status, num_sms, stream);
    case Caps::kNone:
      return launch_ffn_fused_impl<Caps::kNone>(s_gu, s_dn, p, h_ready, status, num_sms, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_plain2(const GemmShape& s1, const GemmShape& s2, uint32_t* status,
                               int num_sms, cudaStream_t stream) {
  if (s1.a_mn_major != s2.a_mn_major || s1.b_mn_major != s2.b_mn_major || s1.group_offsets ||
      s2.group_offsets || s1.k_group_offsets || s2.k_group_offsets)
    return cudaErrorInvalidValue;
  if (s1.a_mn_major && s1.b_mn_major)
    return launch_plain2_impl<Major::kABMN>(s1, s2, status, num_sms, stream);
  if (!s1.a_mn_major && s1.b_mn_major)
    return launch_plain2_impl<Major::kBMN>(s1, s2, status, num_sms, stream);
  if (!s1.a_mn_major && !s1.b_mn_major)
    return launch_plain2_impl<Major::kKMajor>(s1, s2, status, num_sms, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_group_order(const int32_t* group_offsets, int32_t G, int32_t* order,
                               cudaStream_t stream) {
  if (G <= 0) return cudaSuccess;
  group_order_kernel<<<1, 1024, 0, stream>>>(group_offsets, G, order);
  return cudaGetLastError();
}

cudaError_t launch_group_tiles(const int32_t* group_offsets, int32_t G, int64_t R,
                               int32_t n_tiles_1, int32_t n_tiles_2, int32_t* tile_offsets,
                               int32_t* units_1, int32_t* units_2, uint32_t* status,
                               cudaStream_t stream, bool two_cta) {
  group_tiles_kernel<<<1, 1024, 0, stream>>>(group_offsets, G, R, n_tiles_1, n_tiles_2,
                                             tile_offsets, units_1, units_2, status,
                                             two_cta ? 1 : 0);
  return cudaGetLastError();
}

bool gemm_two_cta_available() {
  return max_pair_clusters<Epi::kPlain, Caps::kBoth, false, Major::kKMajor, 0>(
             smem_bytes_pair()) > 0;
}

int32_t gemm_n_tiles_situ(int64_t n_out) { return static_cast<int32_t>((n_out + 127) / 128); }
int32_t gemm_n_tiles_wide(int64_t n_out) { return static_cast<int32_t>((n_out + kBN - 1) / kBN); }

cudaError_t launch_gather_rows(const void* x, const int32_t* token_index, void* x_perm,
                               int64_t R, int32_t k_eff, int64_t M, uint32_t* status,
                               cudaStream_t stream) {
  if (R == 0) return cudaSuccess;
  const int64_t T = R / k_eff;
  const int threads = 256;
  int64_t blocks = (R + (threads / 32) - 1) / (threads / 32);
  if (blocks > 65535) blocks = 65535;
  gather_rows_kernel<<<static_cast<int>(blocks), threads, 0, stream>>>(
      static_cast<const uint4*>(x), token_index, static_cast<uint4*>(x_perm), R, k_eff, M / 8,
      T, status);
  return cudaGetLastError();
}

// Writes per-group row extents into device copies of two host-encoded maps and compares
// each with the driver's own encoding of that base and extent (no copy uses the maps):
// mismatches[2g], [2g + 1] = 1 where group g's A or B map differs.
cudaError_t group_maps_selftest(const int32_t* k_offsets, int32_t groups, int64_t rows,
                                int64_t cols, int32_t* mismatches, cudaStream_t stream) {
  for (int32_t i = 0; i < 2 * groups; ++i) mismatches[i] = -1;
  void* alloc = nullptr;
  int32_t* d_off = nullptr;
  CUtensorMap* d_maps = nullptr;
  cudaError_t e = cudaMalloc(&alloc, 2048);
  if (e == cudaSuccess) e = cudaMalloc(&d_off, sizeof(int32_t) * (groups + 1));
  if (e == cudaSuccess) e = cudaMalloc(&d_maps, sizeof(CUtensorMap) * 2 * groups);
  std::vector<CUtensorMap> got(2 * static_cast<size_t>(groups));
  // Operand A [rows, cols] at base_a, B [rows, 2 cols] at base_b (only encoded).
  uint8_t* base_a = static_cast<uint8_t*>(alloc) + 1024;
  uint8_t* base_b = base_a + 512;
  const int64_t ld_a = cols * 2, ld_b = 4 * cols;
  CUtensorMap ta, tb;
  if (e == cudaSuccess && !(make_map(&ta, base_a, rows, cols, 64, cols) &&
                            make_map(&tb, base_b, rows, 2 * cols, 64, 2 * cols)))
    e = cudaErrorInvalidValue;
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(d_off, k_offsets, sizeof(int32_t) * (groups + 1), cudaMemcpyHostToDevice,
                        stream);
  if (e == cudaSuccess) {
    group_maps_kernel<<<(groups + 127) / 128, 128, 0, stream>>>(ta, tb, base_a, base_b, ld_a,
                                                                 ld_b, d_off, groups, d_maps);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(got.data(), d_maps, sizeof(CUtensorMap) * 2 * groups,
                        cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  for (int32_t g = 0; e == cudaSuccess && g < groups; ++g) {
    const int32_t k0 = k_offsets[g], k_end = k_offsets[g + 1];
    CUtensorMap ea = ta, eb = tb;
    if (k_end > k0 && k0 >= 0) {
      const int32_t shift = group_map_shift(k_end);
      if (!(make_map(&ea, base_a - shift * ld_a, k_end + shift, cols, 64, cols) &&
            make_map(&eb, base_b - shift * ld_b, k_end + shift, 2 * cols, 64, 2 * cols))) {
        e = cudaErrorInvalidValue;
        break;
      }
    }
    mismatches[2 * g] = std::memcmp(&got[2 * g], &ea, sizeof(CUtensorMap)) != 0;
    mismatches[2 * g + 1] = std::memcmp(&got[2 * g + 1], &eb, sizeof(CUtensorMap)) != 0;
  }
  cudaFree(d_maps);
  cudaFree(d_off);
  cudaFree(alloc);
  return e;
}

cudaError_t launch_bounded_wait_selftest(uint64_t limit_ns, uint32_t* status,
                                         cudaStream_t stream) {
  bounded_wait_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns, status);
  return cudaGetLastError();
}

}  // namespace situ
