// act.cu -- standalone SiTU-GLU activation (memory-bound) and the FP32
// small-shape feed-forward.
//
// Standalone activation: gate_up [rows, 2I] -> out [rows, I], out[r, j] =
// SiTU-GLU(gate_up[r, j], gate_up[r, I + j]) ("SiTU-GLU" problem page,
// "Implementation order"; "DenseFFN and SituGLU - Docs", "one split, two softly
// bounded branches").  Every input byte is read once and every output byte
// written once, so the kernel is bound by HBM bandwidth: 128-bit loads of 8
// gate and 8 up bf16 values and one 128-bit store of 8 outputs per vector step,
// streaming cache hints (the data is touched once), a grid of up to 32 blocks of
// 256 threads per SM with each thread keeping two vector steps (four 16-byte
// loads) in flight.  The activation costs four special-function ops and eight
// FP32 ops per output, with no select (situ_math.cuh), which keeps instruction
// issue below the memory time.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "situ_internal.h"
#include "situ_math.cuh"

namespace situ {
namespace {

constexpr int kActThreads = 256;
constexpr int kActBlocksPerSm = 32;
constexpr int kActUnroll = 2;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // round to nearest even
  return *reinterpret_cast<uint32_t*>(&v);
}

template <Caps kC>
__device__ __forceinline__ uint32_t situ_word(uint32_t gw, uint32_t uw, const SituParams& p) {
  return pack_bf16x2(situ_act<kC>(bf16_lo(gw), bf16_lo(uw), p),
                     situ_act<kC>(bf16_hi(gw), bf16_hi(uw), p));
}

// Vector path, bf16: one step = 8 consecutive outputs of one row.  vpr = I / 8
// steps per row; (row, c) walks the flattened [rows, vpr] space with a
// grid-wide stride split as stride = q * vpr + rem so no division is needed
// inside the loop.
template <Caps kC>
__global__ void __launch_bounds__(kActThreads)
    act_bf16_vec_kernel(const uint4* __restrict__ in, uint4* __restrict__ out, uint32_t rows,
                        uint32_t vpr, uint32_t q, uint32_t rem, SituParams p) {
  const uint32_t tid = blockIdx.x * kActThreads + threadIdx.x;
  uint32_t row = tid / vpr;
  uint32_t c = tid - row * vpr;
  while (row < rows) {
    uint4 gv[kActUnroll], uv[kActUnroll];
    uint32_t rr[kActUnroll], cc[kActUnroll];
#pragma unroll
    for (int k = 0; k < kActUnroll; ++k) {
      rr[k] = row;
      cc[k] = c;
      if (row < rows) {
        const uint4* src = in + static_cast<size_t>(row) * (2u * vpr) + c;
        gv[k] = __ldcs(src);
        uv[k] = __ldcs(src + vpr);
      }
      row += q;
      c += rem;
      if (c >= vpr) {
        c -= vpr;
        ++row;
      }
    }
#pragma unroll
    for (int k = 0; k < kActUnroll; ++k) {
      if (rr[k] < rows) {
        uint4 o;
        o.x = situ_word<kC>(gv[k].x, uv[k].x, p);
        o.y = situ_word<kC>(gv[k].y, uv[k].y, p);
        o.z = situ_word<kC>(gv[k].z, uv[k].z, p);
        o.w = situ_word<kC>(gv[k].w, uv[k].w, p);
        __stcs(out + static_cast<size_t>(rr[k]) * vpr + cc[k], o);
      }
    }
  }
}

// Vector path, float32: one step = 4 consecutive outputs.
template <Caps kC>
__global__ void __launch_bounds__(kActThreads)
    act_f32_vec_kernel(const float4* __restrict__ in, float4* __restrict__ out, uint32_t rows,
                       uint32_t vpr, uint32_t q, uint32_t rem, SituParams p) {
  const uint32_t tid = blockIdx.x * kActThreads + threadIdx.x;
  uint32_t row = tid / vpr;
  uint32_t c = tid - row * vpr;
  while (row < rows) {
    const float4* src = in + static_cast<size_t>(row) * (2u * vpr) + c;
    const float4 g = __ldcs(src);
    const float4 u = __ldcs(src + vpr);
    float4 o;
    o.x = situ_act_accurate<kC>(g.x, u.x, p);
    o.y = situ_act_accurate<kC>(g.y, u.y, p);
    o.z = situ_act_accurate<kC>(g.z, u.z, p);
    o.w = situ_act_accurate<kC>(g.w, u.w, p);
    __stcs(out + static_cast<size_t>(row) * vpr + c, o);
    row += q;
    c += rem;
    if (c >= vpr) {
      c -= vpr;
      ++row;
    }
  }
}

// Scalar path for rows that do not start 16-byte aligned.
template <typename T>
__device__ __forceinline__ float load_elem(const T* p, size_t i);
template <>
__device__ __forceinline__ float load_elem<float>(const float* p, size_t i) {
  return p[i];
}
template <>
__device__ __forceinline__ float load_elem<__nv_bfloat16>(const __nv_bfloat16* p, size_t i) {
  return __bfloat162float(p[i]);
}
template <typename T>
__device__ __forceinline__ void store_elem(T* p, size_t i, float v);
template <>
__device__ __forceinline__ void store_elem<float>(float* p, size_t i, float v) {
  p[i] = v;
}
template <>
__device__ __forceinline__ void store_elem<__nv_bfloat16>(__nv_bfloat16* p, size_t i, float v) {
  p[i] = __float2bfloat16_rn(v);
}

template <typename T, Caps kC>
__global__ void __launch_bounds__(kActThreads)
    act_scalar_kernel(const T* __restrict__ in, T* __restrict__ out, uint64_t rows, uint64_t I,
                      SituParams p) {
  const uint64_t total = rows * I;
  for (uint64_t idx = static_cast<uint64_t>(blockIdx.x) * kActThreads + threadIdx.x; idx < total;
       idx += static_cast<uint64_t>(gridDim.x) * kActThreads) {
    const uint64_t r = idx / I;
    const uint64_t j = idx - r * I;
    const float g = load_elem(in, r * 2 * I + j);
    const float u = load_elem(in, r * 2 * I + I + j);
    // float32 outputs take the accurate variant; bf16 outputs the fast one.
    const float h = sizeof(T) == 4 ? situ_act_accurate<kC>(g, u, p) : situ_act<kC>(g, u, p);
    store_elem(out, idx, h);
  }
}

// FP32 small-shape FFN, first half: h[r, j] = SiTU-GLU(x[r] . Wgu[j], x[r] . Wgu[I + j]).
template <Caps kC>
__global__ void ffn_f32_gate_up_kernel(const float* __restrict__ x, const float* __restrict__ w,
                                       float* __restrict__ h, int64_t R, int64_t M, int64_t I,
                                       SituParams p) {
  const int64_t total = R * I;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = idx / I;
    const int64_t j = idx - r * I;
    const float* xr = x + r * M;
    const float* wg = w + j * M;
    const float* wu = w + (I + j) * M;
    float g = 0.0f, u = 0.0f;
    for (int64_t k = 0; k < M; ++k) {
      g = fmaf(xr[k], wg[k], g);
      u = fmaf(xr[k], wu[k], u);
    }
    h[idx] = situ_act_accurate<kC>(g, u, p);
  }
}

// FP32 small-shape FFN, second half: y[r, m] = h[r] . Wd[m].
__global__ void ffn_f32_down_kernel(const float* __restrict__ h, const float* __restrict__ w,
                                    float* __restrict__ y, int64_t R, int64_t M, int64_t I) {
  const int64_t total = R * M;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = idx / M;
    const int64_t m = idx - r * M;
    const float* hr = h + r * I;
    const float* wm = w + m * I;
    float s = 0.0f;
    for (int64_t j = 0; j < I; ++j) s = fmaf(hr[j], wm[j], s);
    y[idx] = s;
  }
}

inline int grid_for(int64_t work_items, int threads, int max_blocks) {
  int64_t b = (work_items + threads - 1) / threads;
  if (b > max_blocks) b = max_blocks;
  return b < 1 ? 1 : static_cast<int>(b);
}

template <Caps kC>
cudaError_t launch_situ_act_caps(const void* gate_up, void* out, int64_t rows, int64_t I,
                                 const SituParams& p, situ_dtype dt, int num_sms,
                                 cudaStream_t stream) {
  const int max_blocks = num_sms * kActBlocksPerSm;
  const size_t esz = dtype_size(dt);
  const int elems_per_vec = static_cast<int>(16 / esz);
  const bool aligned = (reinterpret_cast<uintptr_t>(gate_up) % 16 == 0) &&
                       (reinterpret_cast<uintptr_t>(out) % 16 == 0) && (I % elems_per_vec == 0);
  const int64_t vpr = I / elems_per_vec;
  const int64_t total_vec = rows * vpr;
  if (aligned && total_vec + static_cast<int64_t>(max_blocks) * kActThreads < (int64_t(1) << 32)) {
    const int grid = grid_for(total_vec, kActThreads, max_blocks);
    const uint32_t stride = static_cast<uint32_t>(grid) * kActThreads;
    const uint32_t q = stride / static_cast<uint32_t>(vpr);
    const uint32_t rem = stride - q * static_cast<uint32_t>(vpr);
    if (dt == SITU_BF16) {
      act_bf16_vec_kernel<kC><<<grid, kActThreads, 0, stream>>>(
          static_cast<const uint4*>(gate_up), static_cast<uint4*>(out),
          static_cast<uint32_t>(rows), static_cast<uint32_t>(vpr), q, rem, p);
    } else {
      act_f32_vec_kernel<kC><<<grid, kActThreads, 0, stream>>>(
          static_cast<const float4*>(gate_up), static_cast<float4*>(out),
          static_cast<uint32_t>(rows), static_cast<uint32_t>(vpr), q, rem, p);
    }
  } else {
    const int grid = grid_for(rows * I, kActThreads, max_blocks);
    if (dt == SITU_BF16) {
      act_scalar_kernel<__nv_bfloat16, kC><<<grid, kActThreads, 0, stream>>>(
          static_cast<const __nv_bfloat16*>(gate_up), static_cast<__nv_bfloat16*>(out),
          static_cast<uint64_t>(rows), static_cast<uint64_t>(I), p);
    } else {
      act_scalar_kernel<float, kC><<<grid, kActThreads, 0, stream>>>(
          static_cast<const float*>(gate_up), static_cast<float*>(out),
          static_cast<uint64_t>(rows), static_cast<uint64_t>(I), p);
    }
  }
  return cudaGetLastError();
}

template <Caps kC>
cudaError_t launch_ffn_f32_caps(const float* x, const float* w_gate_up, const float* w_down,
                                float* h, float* y, int64_t R, int64_t M, int64_t I,
                                const SituParams& p, cudaStream_t stream) {
  constexpr int threads = 128;
  ffn_f32_gate_up_kernel<kC><<<grid_for(R * I, threads, 4096), threads, 0, stream>>>(
      x, w_gate_up, h, R, M, I, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ffn_f32_down_kernel<<<grid_for(R * M, threads, 4096), threads, 0, stream>>>(h, w_down, y, R,
                                                                              M, I);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_situ_act(const void* gate_up, void* out, int64_t rows, int64_t I,
                            const SituParams& p, Caps caps, situ_dtype dt, int num_sms,
                            cudaStream_t stream) {
  if (rows == 0 || I == 0) return cudaSuccess;
  switch (caps) {
    case Caps::kBoth:
      return launch_situ_act_caps<Caps::kBoth>(gate_up, out, rows, I, p, dt, num_sms, stream);
    case Caps::kGateOnly:
      return launch_situ_act_caps<Caps::kGateOnly>(gate_up, out, rows, I, p, dt, num_sms, stream);
    case Caps::kUpOnly:
      return launch_situ_act_caps<Caps::kUpOnly>(gate_up, out, rows, I, p, dt, num_sms, stream);
    case Caps::kNone:
      return launch_situ_act_caps<Caps::kNone>(gate_up, out, rows, I, p, dt, num_sms, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_ffn_f32(const float* x, const float* w_gate_up, const float* w_down,
                           float* h, float* y, int64_t R, int64_t M, int64_t I,
                           const SituParams& p, Caps caps, cudaStream_t stream) {
  if (R == 0) return cudaSuccess;
  switch (caps) {
    case Caps::kBoth:
      return launch_ffn_f32_caps<Caps::kBoth>(x, w_gate_up, w_down, h, y, R, M, I, p, stream);
    case Caps::kGateOnly:
      return launch_ffn_f32_caps<Caps::kGateOnly>(x, w_gate_up, w_down, h, y, R, M, I, p, stream);
    case Caps::kUpOnly:
      return launch_ffn_f32_caps<Caps::kUpOnly>(x, w_gate_up, w_down, h, y, R, M, I, p, stream);
    case Caps::kNone:
      return launch_ffn_f32_caps<Caps::kNone>(x, w_gate_up, w_down, h, y, R, M, I, p, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace situ
