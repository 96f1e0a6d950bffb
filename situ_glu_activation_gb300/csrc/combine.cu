// combine.cu -- the router-weighted combine of a routed layer:
//   out[t, :] = sum over slots s of w[t, s] * y[t, s, :]   (FP32, slot order)
// A null w means weight 1 for every slot (the sum the grouped backward needs).
// Memory bound: every y byte is read once, every out byte written once.  One
// thread owns 16 bytes of one token's output row (8 bf16 / 4 float columns) and
// walks that token's k_eff slot rows with 128-bit streaming loads.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "situ_internal.h"

namespace situ {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], uint4 v, float w) {
  const uint32_t q[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc[2 * i] = fmaf(w, __uint_as_float(q[i] << 16), acc[2 * i]);
    acc[2 * i + 1] = fmaf(w, __uint_as_float(q[i] & 0xFFFF0000u), acc[2 * i + 1]);
  }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__global__ void __launch_bounds__(kThreads)
    combine_bf16_vec_kernel(const uint4* __restrict__ y, const float* __restrict__ w,
                            uint4* __restrict__ out, int64_t T, int32_t k_eff, int64_t vpr) {
  const int64_t total = T * vpr;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int64_t t = i / vpr;
    const int64_t c = i - t * vpr;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    const uint4* row = y + t * k_eff * vpr + c;
    for (int32_t s = 0; s < k_eff; ++s)
      add_bf16x8(acc, __ldcs(row + s * vpr), w ? __ldg(w + t * k_eff + s) : 1.0f);
    __stcs(out + i, make_uint4(pack2(acc[0], acc[1]), pack2(acc[2], acc[3]),
                               pack2(acc[4], acc[5]), pack2(acc[6], acc[7])));
  }
}

__global__ void __launch_bounds__(kThreads)
    combine_f32_vec_kernel(const float4* __restrict__ y, const float* __restrict__ w,
                           float4* __restrict__ out, int64_t T, int32_t k_eff, int64_t vpr) {
  const int64_t total = T * vpr;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int64_t t = i / vpr;
    const int64_t c = i - t * vpr;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4* row = y + t * k_eff * vpr + c;
    for (int32_t s = 0; s < k_eff; ++s) {
      const float ws = w ? __ldg(w + t * k_eff + s) : 1.0f;
      const float4 v = __ldcs(row + s * vpr);
      acc.x = fmaf(ws, v.x, acc.x);
      acc.y = fmaf(ws, v.y, acc.y);
      acc.z = fmaf(ws, v.z, acc.z);
      acc.w = fmaf(ws, v.w, acc.w);
    }
    __stcs(out + i, acc);
  }
}

template <typename T>
__device__ __forceinline__ float ld(const T* p, int64_t i);
template <>
__device__ __forceinline__ float ld<float>(const float* p, int64_t i) { return p[i]; }
template <>
__device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16* p, int64_t i) {
  return __bfloat162float(p[i]);
}
__device__ __forceinline__ void st(float* p, int64_t i, float v) { p[i] = v; }
__device__ __forceinline__ void st(__nv_bfloat16* p, int64_t i, float v) {
  p[i] = __float2bfloat16_rn(v);
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
    combine_scalar_kernel(const T* __restrict__ y, const float* __restrict__ w,
                          T* __restrict__ out, int64_t T_, int32_t k_eff, int64_t M) {
  const int64_t total = T_ * M;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int64_t t = i / M;
    const int64_t m = i - t * M;
    float acc = 0.0f;
    for (int32_t s = 0; s < k_eff; ++s)
      acc = fmaf(w ? __ldg(w + t * k_eff + s) : 1.0f, ld(y, (t * k_eff + s) * M + m), acc);
    st(out, i, acc);
  }
}

// FP32 -> bf16 (round to nearest even), 8 values a thread when aligned.
__global__ void __launch_bounds__(kThreads)
    f32_to_bf16_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ out, int64_t n) {
  const int64_t n8 = n / 8;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * kThreads) {
    const float4 a = __ldcs(reinterpret_cast<const float4*>(acc) + 2 * i);
    const float4 b = __ldcs(reinterpret_cast<const float4*>(acc) + 2 * i + 1);
    __stcs(reinterpret_cast<uint4*>(out) + i,
           make_uint4(pack2(a.x, a.y), pack2(a.z, a.w), pack2(b.x, b.y), pack2(b.z, b.w)));
  }
  for (int64_t i = n8 * 8 + static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * kThreads)
    out[i] = __float2bfloat16_rn(acc[i]);
}

int grid_of(int64_t items, int num_sms) {
  int64_t b = (items + kThreads - 1) / kThreads;
  const int64_t cap = static_cast<int64_t>(num_sms) * 16;
  if (b > cap) b = cap;
  return b < 1 ? 1 : static_cast<int>(b);
}

}  // namespace

cudaError_t launch_f32_to_bf16(const float* acc, void* out, int64_t n, int num_sms,
                               cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  f32_to_bf16_kernel<<<grid_of((n + 7) / 8, num_sms), kThreads, 0, stream>>>(
      acc, static_cast<__nv_bfloat16*>(out), n);
  return cudaGetLastError();
}

cudaError_t launch_combine(const void* y, const float* w, void* out, int64_t T, int32_t k_eff,
                           int64_t M, situ_dtype dt, int num_sms, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const int per_vec = dt == SITU_BF16 ? 8 : 4;
  const bool vec = M % per_vec == 0 && reinterpret_cast<uintptr_t>(y) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(out) % 16 == 0;
  if (vec) {
    const int64_t vpr = M / per_vec;
    const int grid = grid_of(T * vpr, num_sms);
    if (dt == SITU_BF16) {
      combine_bf16_vec_kernel<<<grid, kThreads, 0, stream>>>(
          static_cast<const uint4*>(y), w, static_cast<uint4*>(out), T, k_eff, vpr);
    } else {
      combine_f32_vec_kernel<<<grid, kThreads, 0, stream>>>(
          static_cast<const float4*>(y), w, static_cast<float4*>(out), T, k_eff, vpr);
    }
  } else {
    const int grid = grid_of(T * M, num_sms);
    if (dt == SITU_BF16) {
      combine_scalar_kernel<__nv_bfloat16><<<grid, kThreads, 0, stream>>>(
          static_cast<const __nv_bfloat16*>(y), w, static_cast<__nv_bfloat16*>(out), T, k_eff, M);
    } else {
      combine_scalar_kernel<float><<<grid, kThreads, 0, stream>>>(
          static_cast<const float*>(y), w, static_cast<float*>(out), T, k_eff, M);
    }
  }
  return cudaGetLastError();
}

}  // namespace situ
