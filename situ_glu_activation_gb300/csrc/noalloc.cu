// noalloc.cu -- situ_ffn_forward_noalloc: the dense SiTU-GLU FFN for callers
// that cannot allocate device memory (see include/situ.h).  The intermediate h
// lives in a file-scope device array compiled into the library instead of a
// caller-provided workspace; the kernels are the ones situ_ffn_forward launches.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "situ.h"
#include "situ_internal.h"
#include "situ_math.cuh"

namespace {

using namespace situ;

constexpr int kMaxDevices = 64;
constexpr size_t kScratchBytes = SITU_NOALLOC_SCRATCH_BYTES;

// h scratch.  Every GPU that loads the library holds these bytes until exit.
// In host code the name is only a handle for cudaGetSymbolAddress; kernels get
// the device address looked up below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_address[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per
// device (with that device current) and cached.
situ_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return report_cuda_error(e);
  if (dev < 0 || dev >= kMaxDevices) return SITU_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_address[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return report_cuda_error(e);
    g_scratch_address[dev] = p;
  }
  *out = g_scratch_address[dev];
  return SITU_OK;
}

bool ranges_overlap(const void* a, size_t an, const void* b, size_t bn) {
  if (!a || !b || an == 0 || bn == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + bn && b0 < a0 + an;
}

bool is_aligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

}  // namespace

extern "C" situ_status situ_ffn_forward_noalloc(const void* x, const void* W_gate_up,
                                                const void* W_down, void* y, int64_t R,
                                                int64_t M, int64_t I, float beta,
                                                float linear_beta, situ_dtype dt,
                                                void* stream) {
  // The same checks as situ_ffn_forward, then the scratch limit.
  situ_status s = ffn_arg_checks(dt, R, M, I, beta, linear_beta);
  if (s != SITU_OK || R == 0) return s;
  if (!x || !W_gate_up || !W_down || !y) return SITU_ERR_ARG;
  const size_t esz = dtype_size(dt);
  // The limit of the built-in scratch: h is R x I elements.
  if (static_cast<uint64_t>(R) * static_cast<uint64_t>(I) > kScratchBytes / esz)
    return SITU_ERR_WORKSPACE;
  const size_t y_bytes = static_cast<size_t>(R) * M * esz;
  if (ranges_overlap(y, y_bytes, x, static_cast<size_t>(R) * M * esz) ||
      ranges_overlap(y, y_bytes, W_gate_up, static_cast<size_t>(2 * I) * M * esz) ||
      ranges_overlap(y, y_bytes, W_down, static_cast<size_t>(M) * I * esz))
    return SITU_ERR_ALIAS;
  void* scratch = nullptr;
  s = scratch_address(&scratch);
  if (s != SITU_OK) return s;
  int num_sms = 0;
  uint32_t* status = nullptr;
  if ((s = current_device_context(&num_sms, &status)) != SITU_OK) return s;
  const SituParams p = make_situ_params(beta, linear_beta);
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (dt == SITU_F32) {
    if (!is_aligned(x, 4) || !is_aligned(W_gate_up, 4) || !is_aligned(W_down, 4) ||
        !is_aligned(y, 4))
      return SITU_ERR_ALIGN;
    e = launch_ffn_f32(static_cast<const float*>(x), static_cast<const float*>(W_gate_up),
                       static_cast<const float*>(W_down), static_cast<float*>(scratch),
                       static_cast<float*>(y), R, M, I, p, caps_of(beta, linear_beta), cs);
    return e == cudaSuccess ? SITU_OK : report_cuda_error(e);
  }
  if ((s = ffn_bf16_operand_checks(x, W_gate_up, W_down, M, I)) != SITU_OK) return s;
  if (!is_aligned(y, 16)) return SITU_ERR_ALIGN;
  GemmShape g{};
  g.a = x;
  g.a_rows = R;
  g.b = W_gate_up;
  g.b_rows = 2 * I;
  g.K = M;
  g.num_groups = 1;
  g.b_group_rows = 2 * I;
  g.b_up_offset = I;
  g.n_out = I;
  g.out = scratch;  // h [R, I]
  g.ldo = I;
  g.out_rows = R;
  if ((e = launch_gemm_situ(g, p, caps_of(beta, linear_beta), status, num_sms, cs)) !=
      cudaSuccess)
    return report_cuda_error(e);
  GemmShape d{};
  d.a = scratch;
  d.a_rows = R;
  d.b = W_down;
  d.b_rows = M;
  d.K = I;
  d.num_groups = 1;
  d.b_group_rows = M;
  d.n_out = M;
  d.out = y;
  d.ldo = M;
  d.out_rows = R;
  e = launch_gemm_plain(d, status, num_sms, cs);
  return e == cudaSuccess ? SITU_OK : report_cuda_error(e);
}
