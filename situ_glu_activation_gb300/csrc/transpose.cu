// transpose.cu -- out[c, r] = in[r, c] (bf16), the operand re-layout of the
// backward GEMMs: the library's tcgen05 GEMMs read both operands K-major, and the
// weight gradients contract over the token rows, so dy, h, d(g,u) and x are
// transposed to [features, rows] (and the weights to [in, out]).  Columns of the
// output beyond `rows` (up to ld_out, a multiple of 8) are zero, so a 16-byte
// aligned row stride can be used by the tensor-memory-access loads.
//
// One block moves a 64 x 64 tile through shared memory: 16-byte loads along the
// input rows, 16-byte stores along the output rows.  Memory bound.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "situ_internal.h"

namespace situ {
namespace {

constexpr int kTile = 64;
constexpr int kPad = 8;  // elements of padding per shared row (16 bytes)

__global__ void __launch_bounds__(256)
    transpose_kernel(const uint16_t* __restrict__ in, int64_t rows, int64_t cols,
                     uint16_t* __restrict__ out, int64_t ld_out) {
  __shared__ __align__(16) uint16_t tile[kTile][kTile + kPad];
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * kTile;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kTile;
  // Load: 64 rows x 8 chunks of 8 columns.
  for (int i = threadIdx.x; i < kTile * (kTile / 8); i += blockDim.x) {
    const int rr = i / (kTile / 8), cc = (i % (kTile / 8)) * 8;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r0 + rr < rows && c0 + cc < cols)
      v = *reinterpret_cast<const uint4*>(in + (r0 + rr) * cols + c0 + cc);
    *reinterpret_cast<uint4*>(&tile[rr][cc]) = v;
  }
  __syncthreads();
  // Store: 64 output rows (input columns) x 8 chunks of 8 output columns (input rows).
  for (int i = threadIdx.x; i < kTile * (kTile / 8); i += blockDim.x) {
    const int cr = i / (kTile / 8), rc = (i % (kTile / 8)) * 8;
    if (c0 + cr >= cols || r0 + rc >= ld_out) continue;
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t lo = tile[rc + 2 * k][cr], hi = tile[rc + 2 * k + 1][cr];
      w[k] = lo | (hi << 16);
    }
    *reinterpret_cast<uint4*>(out + (c0 + cr) * ld_out + r0 + rc) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace

cudaError_t launch_transpose(const void* in, int64_t rows, int64_t cols, void* out,
                             int64_t ld_out, cudaStream_t stream) {
  if (cols == 0 || ld_out == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>((cols + kTile - 1) / kTile),
                  static_cast<unsigned>((ld_out + kTile - 1) / kTile));
  transpose_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(in), rows, cols,
                                             static_cast<uint16_t*>(out), ld_out);
  return cudaGetLastError();
}

}  // namespace situ
