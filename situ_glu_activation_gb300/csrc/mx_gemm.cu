// mx_gemm.cu -- MXFP8 (OCP Microscaling E4M3 codes, one E8M0 scale per 32 along
// K) block-scaled GEMMs of the SiTU-GLU feed-forward on sm_103a -- with MXFP8 or
// MXFP4 (E2M1) expert weights -- and the quantization kernels that produce their
// operands.
//
// The "SiTU-GLU" chapter ("Pourquoi un plafond doux") motivates the activation's
// bound by experts that run in MXFP8 / MXFP4: a bounded h never drives a block
// scale to the format's limits.  Here the two projections run as
// tcgen05.mma kind::mxf8f6f4 block-scaled MMAs in the same persistent
// warp-specialised kernel as the bf16 GEMMs (gemm_kernel.cuh, MXFP8 geometry):
// 128 x 192 tiles, 128 K a stage, the stage's E8M0 scale tiles copied into TMEM
// with tcgen05.cp before its MMAs.  The gate_up GEMM's epilogue can emit h directly
// as MXFP8 (bf16 rounding, then block quantization), the input of the down GEMM.
//
// Scale-tile layout (the hardware's): a 128-row tile's scales for one 128-wide K
// stage are 512 bytes, byte l * 16 + g * 4 + k holding row 32 g + l, block k.
// Activations (GEMM A): one such tile per (128-row m-tile, K stage); grouped rows
// follow the groups' m-tiles.  Weights (GEMM B): 1024 bytes per (group, n-tile, K
// stage) -- the tile's 192 rows as rows 0..127 and 128..191 of two 512-byte tiles;
// for the gate_up weights an n-tile's rows are 96 gate rows then the 96 matching up
// rows.
#include "gemm_kernel.cuh"

namespace situ {
namespace {

constexpr int kQuantThreads = 256;

// Group of row r (largest g with off[g] <= r; empty groups repeat an offset).
__device__ __forceinline__ int32_t group_of(const int32_t* off, int32_t G, int64_t r) {
  int32_t lo = 0, hi = G - 1;
  while (lo < hi) {
    const int32_t mid = (lo + hi + 1) >> 1;
    if (__ldg(off + mid) <= r) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// One thread per 32-wide block of one row: 64 bytes of bf16 in, 32 code bytes and
// one scale byte out.
__global__ void __launch_bounds__(kQuantThreads)
    mx_quant_act_kernel(const uint4* __restrict__ src, const int32_t* __restrict__ row_index,
                        int32_t k_eff, int64_t src_rows, uint8_t* __restrict__ codes,
                        uint8_t* __restrict__ scales, int64_t sf_tiles, int64_t R, int64_t K,
                        int32_t G, const int32_t* __restrict__ off,
                        const int32_t* __restrict__ tiles, uint32_t* status) {
  const int64_t bpr = K / 32;
  const int64_t total = R * bpr;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kQuantThreads + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * kQuantThreads) {
    const int64_t r = i / bpr;
    const int64_t b = i - r * bpr;
    int64_t sr = r;
    if (row_index) {
      const int32_t f = __ldg(row_index + r);
      sr = f >= 0 ? f / k_eff : -1;
      if (sr < 0 || sr >= src_rows) {
        record_status(status, SITU_ERR_INDEX);
        sr = -1;
      }
    }
    uint32_t w[16];
    if (sr >= 0) {
      const uint4* p = src + sr * (K / 8) + b * 4;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 v = __ldg(p + j);
        w[4 * j] = v.x;
        w[4 * j + 1] = v.y;
        w[4 * j + 2] = v.z;
        w[4 * j + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) w[j] = 0;
    }
    uint32_t q[8];
    const uint32_t sc = mx_quantize32(w, q);
    uint4* d = reinterpret_cast<uint4*>(codes + r * K + b * 32);
    d[0] = make_uint4(q[0], q[1], q[2], q[3]);
    d[1] = make_uint4(q[4], q[5], q[6], q[7]);
    int64_t m_tile = r / kBM;
    int32_t rit = static_cast<int32_t>(r % kBM);
    if (off) {
      const int32_t g = group_of(off, G, r);
      const int64_t local = r - __ldg(off + g);
      m_tile = local >= 0 ? __ldg(tiles + g) + local / kBM : -1;
      rit = static_cast<int32_t>(local % kBM);
    }
    // Offsets that failed validation can point outside the scale tiles: skip.
    if (m_tile < 0 || m_tile >= sf_tiles) {
      record_status(status, SITU_ERR_INDEX);
      continue;
    }
    scales[sf_tile_offset(m_tile, K / 128, rit, b)] = static_cast<uint8_t>(sc);
  }
}

// MXFP4 quantization of one block of 32 bf16 values (as mx_quantize32, with E2M1
// elements): scale 2^(floor(log2 amax) - 2), i.e. code max(E - 2, 0); 16 bytes of
// packed codes, element 2i in the low nibble of byte i.
__device__ __forceinline__ uint32_t mx_quantize32_e2m1(const uint32_t (&w)[16], uint32_t (&q)[4]) {
  uint32_t amax = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = max(amax, max(w[i] & 0x7FFFu, (w[i] >> 16) & 0x7FFFu));
  const uint32_t e = amax >> 7;
  const uint32_t code = e > 2u ? e - 2u : 0u;
  const float inv = __uint_as_float((254u - code) << 23);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[4 * j + i] << 16) * inv;
      v[2 * i + 1] = __uint_as_float(w[4 * j + i] & 0xFFFF0000u) * inv;
    }
    q[j] = cvt_e2m1x8(v);
  }
  return code;
}

// Weight rows: codes keep the row-major layout (E4M3 one a byte, or E2M1 two a
// byte); scales go to the B tiles.
template <bool kFp4>
__global__ void __launch_bounds__(kQuantThreads)
    mx_quant_weight_kernel(const uint4* __restrict__ w, uint8_t* __restrict__ codes,
                           uint8_t* __restrict__ scales, int64_t rows_total, int64_t rows_g,
                           int64_t K, int64_t split, int32_t n_tiles) {
  const int64_t bpr = K / 32;
  const int64_t total = rows_total * bpr;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kQuantThreads + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * kQuantThreads) {
    const int64_t row = i / bpr;
    const int64_t b = i - row * bpr;
    uint32_t v[16];
    const uint4* p = w + row * (K / 8) + b * 4;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 x = __ldg(p + j);
      v[4 * j] = x.x;
      v[4 * j + 1] = x.y;
      v[4 * j + 2] = x.z;
      v[4 * j + 3] = x.w;
    }
    uint32_t sc;
    if (kFp4) {
      uint32_t q[4];
      sc = mx_quantize32_e2m1(v, q);
      *reinterpret_cast<uint4*>(codes + row * (K / 2) + b * 16) = make_uint4(q[0], q[1], q[2], q[3]);
    } else {
      uint32_t q[8];
      sc = mx_quantize32(v, q);
      uint4* d = reinterpret_cast<uint4*>(codes + row * K + b * 32);
      d[0] = make_uint4(q[0], q[1], q[2], q[3]);
      d[1] = make_uint4(q[4], q[5], q[6], q[7]);
    }
    const int64_t g = row / rows_g;
    const int64_t r = row - g * rows_g;
    int64_t t, n;
    if (split > 0) {
      const bool up = r >= split;
      const int64_t j = up ? r - split : r;
      t = j / kMxSituCols;
      n = (up ? kMxSituCols : 0) + j % kMxSituCols;
    } else {
      t = r / kMxPlainCols;
      n = r % kMxPlainCols;
    }
    const int64_t chunk = ((g * n_tiles + t) * (K / 128) + b / 4) * kSfbStageBytes;
    scales[chunk + (n / 128) * kSfTileBytes + (n % 32) * 16 + ((n % 128) / 32) * 4 + b % 4] =
        static_cast<uint8_t>(sc);
  }
}

int quant_grid(int64_t items) {
  int64_t b = (items + kQuantThreads - 1) / kQuantThreads;
  if (b > 152 * 32) b = 152 * 32;
  return b < 1 ? 1 : static_cast<int>(b);
}

int32_t weight_n_tiles(int64_t rows_per_group, int64_t split) {
  return static_cast<int32_t>(split > 0 ? (split + kMxSituCols - 1) / kMxSituCols
                                        : (rows_per_group + kMxPlainCols - 1) / kMxPlainCols);
}

}  // namespace

size_t mx_act_scale_bytes(int64_t R, int64_t K) {
  return static_cast<size_t>((R + kBM - 1) / kBM) * static_cast<size_t>(K / 128) * kSfTileBytes;
}

size_t mx_weight_scale_bytes(int32_t G, int64_t rows_per_group, int64_t K, int64_t split) {
  return static_cast<size_t>(G) * weight_n_tiles(rows_per_group, split) *
         static_cast<size_t>(K / 128) * kSfbStageBytes;
}

cudaError_t launch_mx_quantize_act(const void* src, const int32_t* row_index, int32_t k_eff,
                                   int64_t src_rows, void* codes, void* scales, int64_t sf_tiles,
                                   int64_t R, int64_t K, int32_t num_groups,
                                   const int32_t* group_offsets, const int32_t* tile_offsets,
                                   uint32_t* status, cudaStream_t stream) {
  if (R == 0) return cudaSuccess;
  if (K % 128 != 0) return cudaErrorInvalidValue;
  mx_quant_act_kernel<<<quant_grid(R * (K / 32)), kQuantThreads, 0, stream>>>(
      static_cast<const uint4*>(src), row_index, k_eff, src_rows, static_cast<uint8_t*>(codes),
      static_cast<uint8_t*>(scales), sf_tiles, R, K, num_groups, group_offsets, tile_offsets,
      status);
  return cudaGetLastError();
}

cudaError_t launch_mx_quantize_weights(const void* w, void* codes, void* scales, int32_t G,
                                       int64_t rows_per_group, int64_t K, int64_t split,
                                       bool fp4, cudaStream_t stream) {
  if (K % 128 != 0) return cudaErrorInvalidValue;
  // Tile positions no weight row maps to (a partial last tile, the unused fourth
  // 32-row group of the second 512-byte tile) read as scale code 0.
  cudaError_t e =
      cudaMemsetAsync(scales, 0, mx_weight_scale_bytes(G, rows_per_group, K, split), stream);
  if (e != cudaSuccess) return e;
  const int64_t rows = static_cast<int64_t>(G) * rows_per_group;
  auto kernel = fp4 ? mx_quant_weight_kernel<true> : mx_quant_weight_kernel<false>;
  kernel<<<quant_grid(rows * (K / 32)), kQuantThreads, 0, stream>>>(
      static_cast<const uint4*>(w), static_cast<uint8_t*>(codes), static_cast<uint8_t*>(scales),
      rows, rows_per_group, K, split, weight_n_tiles(rows_per_group, split));
  return cudaGetLastError();
}

namespace {

template <int kMx>
cudaError_t mx_situ(const GemmShape& s, const SituParams& p, Caps caps, uint32_t* status,
                    int num_sms, cudaStream_t stream) {
  constexpr Major K = Major::kKMajor;
  if (s.h_codes) {
    switch (caps) {
      case Caps::kBoth:
        return launch<Epi::kSituMx, Caps::kBoth, false, K, kMx, true>(s, p, status, num_sms, stream);
      case Caps::kGateOnly:
        return launch<Epi::kSituMx, Caps::kGateOnly, false, K, kMx, true>(s, p, status, num_sms, stream);
      case Caps::kUpOnly:
        return launch<Epi::kSituMx, Caps::kUpOnly, false, K, kMx, true>(s, p, status, num_sms, stream);
      case Caps::kNone:
        return launch<Epi::kSituMx, Caps::kNone, false, K, kMx, true>(s, p, status, num_sms, stream);
    }
    return cudaErrorInvalidValue;
  }
  switch (caps) {
    case Caps::kBoth:
      return launch<Epi::kSitu, Caps::kBoth, false, K, kMx, true>(s, p, status, num_sms, stream);
    case Caps::kGateOnly:
      return launch<Epi::kSitu, Caps::kGateOnly, false, K, kMx, true>(s, p, status, num_sms, stream);
    case Caps::kUpOnly:
      return launch<Epi::kSitu, Caps::kUpOnly, false, K, kMx, true>(s, p, status, num_sms, stream);
    case Caps::kNone:
      return launch<Epi::kSitu, Caps::kNone, false, K, kMx, true>(s, p, status, num_sms, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_mx_gemm_situ(const GemmShape& s, const SituParams& p, Caps caps,
                                uint32_t* status, int num_sms, cudaStream_t stream) {
  return s.b_fp4 ? mx_situ<2>(s, p, caps, status, num_sms, stream)
                 : mx_situ<1>(s, p, caps, status, num_sms, stream);
}

template <int kMx>
cudaError_t mx_ffn_fused(const GemmShape& s_gu, const GemmShape& s_dn, const SituParams& p,
                         Caps caps, int32_t* h_ready, uint32_t* status, int num_sms,
                         cudaStream_t stream) {
  switch (caps) {
    case Caps::kBoth:
      return launch_ffn_fused_impl<Caps::kBoth, kMx>(s_gu, s_dn, p, h_ready, status, num_sms,
                                                     stream);
    case Caps::kGateOnly:
      return launch_ffn_fused_impl<Caps::kGateOnly, kMx>(s_gu, s_dn, p, h_ready, status, num_sms,
                                                         stream);
    case Caps::kUpOnly:
      return launch_ffn_fused_impl<Caps::kUpOnly, kMx>(s_gu, s_dn, p, h_ready, status, num_sms,
                                                       stream);
    case Caps::kNone:
      return launch_ffn_fused_impl<Caps::kNone, kMx>(s_gu, s_dn, p, h_ready, status, num_sms,
                                                     stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_mx_ffn_fused(const GemmShape& s_gu, const GemmShape& s_dn, const SituParams& p,
                                Caps caps, int32_t* h_ready, uint32_t* status, int num_sms,
                                cudaStream_t stream) {
  return s_gu.b_fp4 ? mx_ffn_fused<2>(s_gu, s_dn, p, caps, h_ready, status, num_sms, stream)
                    : mx_ffn_fused<1>(s_gu, s_dn, p, caps, h_ready, status, num_sms, stream);
}

cudaError_t launch_mx_gemm_plain(const GemmShape& s, uint32_t* status, int num_sms,
                                 cudaStream_t stream) {
  if (s.b_fp4)
    return launch<Epi::kPlain, Caps::kBoth, false, Major::kKMajor, 2, true>(s, SituParams{}, status,
                                                                    num_sms, stream);
  return launch<Epi::kPlain, Caps::kBoth, false, Major::kKMajor, 1, true>(s, SituParams{}, status,
                                                                  num_sms, stream);
}

}  // namespace situ
