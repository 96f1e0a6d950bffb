// hostio.cu -- situ_ffn_forward_host: the dense FFN with x and y in host memory,
// pipelined in row chunks so that host->device copies, the two GEMMs and
// device->host copies of neighbouring chunks overlap (see include/situ.h).
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "situ.h"
#include "situ_internal.h"

namespace {

using namespace situ;

constexpr int kMaxDevices = 64;
constexpr int64_t kDefaultChunk = 4096;

struct CopyEngines {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr;
  cudaEvent_t loaded[2] = {}, computed[2] = {}, stored[2] = {};
};

CopyEngines g_engines[kMaxDevices];
std::mutex g_mutex;

size_t round256(size_t v) { return (v + 255) / 256 * 256; }

situ_status engines(CopyEngines** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return report_cuda_error(e);
  if (dev < 0 || dev >= kMaxDevices) return SITU_ERR_UNSUPPORTED;
  CopyEngines& c = g_engines[dev];
  if (!c.ready) {
    if ((e = cudaStreamCreateWithFlags(&c.in, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&c.out, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&c.start, cudaEventDisableTiming)) != cudaSuccess)
      return report_cuda_error(e);
    for (int i = 0; i < 2; ++i) {
      if ((e = cudaEventCreateWithFlags(&c.loaded[i], cudaEventDisableTiming)) != cudaSuccess ||
          (e = cudaEventCreateWithFlags(&c.computed[i], cudaEventDisableTiming)) != cudaSuccess ||
          (e = cudaEventCreateWithFlags(&c.stored[i], cudaEventDisableTiming)) != cudaSuccess)
        return report_cuda_error(e);
    }
    c.ready = true;
  }
  *out = &c;
  return SITU_OK;
}

}  // namespace

extern "C" size_t situ_ffn_host_workspace_size(int64_t R, int64_t M, int64_t I, situ_dtype dt,
                                               int64_t chunk_rows) {
  if (R <= 0 || M <= 0 || I <= 0 || (dt != SITU_BF16 && dt != SITU_F32) || chunk_rows < 0)
    return 0;
  const int64_t c = chunk_rows == 0 ? kDefaultChunk : chunk_rows;
  const int64_t rows = c < R ? c : R;
  const size_t esz = dtype_size(dt);
  const size_t xb = round256(static_cast<size_t>(rows) * M * esz);
  const size_t hb = situ_ffn_workspace_size(rows, M, I, dt);
  return 4 * xb + hb;  // x[2], y[2], the FFN's workspace (h)
}

extern "C" situ_status situ_ffn_forward_host(const void* x_host, const void* W_gate_up,
                                             const void* W_down, void* y_host, void* workspace,
                                             size_t workspace_bytes, int64_t R, int64_t M,
                                             int64_t I, int64_t chunk_rows, float beta,
                                             float linear_beta, situ_dtype dt, void* stream) {
  if ((dt != SITU_BF16 && dt != SITU_F32) || R < 0 || M < 1 || I < 1 || chunk_rows < 0)
    return SITU_ERR_ARG;
  if (R == 0) return SITU_OK;
  if (!x_host || !y_host || !W_gate_up || !W_down) return SITU_ERR_ARG;
  const size_t need = situ_ffn_host_workspace_size(R, M, I, dt, chunk_rows);
  if (!workspace || workspace_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 256)
    return SITU_ERR_WORKSPACE;
  const int64_t chunk = chunk_rows == 0 ? kDefaultChunk : chunk_rows;
  const int64_t rows = chunk < R ? chunk : R;
  const size_t esz = dtype_size(dt);
  const size_t xb = round256(static_cast<size_t>(rows) * M * esz);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* xbuf[2] = {ws, ws + xb};
  void* ybuf[2] = {ws + 2 * xb, ws + 3 * xb};
  void* hbuf = ws + 4 * xb;
  const size_t hbytes = need - 4 * xb;

  std::lock_guard<std::mutex> lock(g_mutex);
  CopyEngines* ce = nullptr;
  situ_status s = engines(&ce);
  if (s != SITU_OK) return s;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  // The copy streams start after whatever the caller queued before this call.
  if ((e = cudaEventRecord(ce->start, cs)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(ce->in, ce->start, 0)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(ce->out, ce->start, 0)) != cudaSuccess)
    return report_cuda_error(e);
  const int64_t nchunks = (R + chunk - 1) / chunk;
  const uint8_t* xh = static_cast<const uint8_t*>(x_host);
  uint8_t* yh = static_cast<uint8_t*>(y_host);
  for (int64_t c = 0; c < nchunks; ++c) {
    const int slot = static_cast<int>(c & 1);
    const int64_t r0 = c * chunk;
    const int64_t n = (R - r0) < chunk ? (R - r0) : chunk;
    const size_t bytes = static_cast<size_t>(n) * M * esz;
    // copy in (the slot's x buffer is free once chunk c-2's GEMMs finished)
    if (c >= 2 && (e = cudaStreamWaitEvent(ce->in, ce->computed[slot], 0)) != cudaSuccess)
      return report_cuda_error(e);
    if ((e = cudaMemcpyAsync(xbuf[slot], xh + static_cast<size_t>(r0) * M * esz, bytes,
                             cudaMemcpyHostToDevice, ce->in)) != cudaSuccess ||
        (e = cudaEventRecord(ce->loaded[slot], ce->in)) != cudaSuccess)
      return report_cuda_error(e);
    // compute (the slot's y buffer is free once chunk c-2's results were copied out)
    if ((e = cudaStreamWaitEvent(cs, ce->loaded[slot], 0)) != cudaSuccess)
      return report_cuda_error(e);
    if (c >= 2 && (e = cudaStreamWaitEvent(cs, ce->stored[slot], 0)) != cudaSuccess)
      return report_cuda_error(e);
    s = situ_ffn_forward(xbuf[slot], W_gate_up, W_down, ybuf[slot], hbuf, hbytes, n, M, I, beta,
                         linear_beta, dt, stream);
    if (s != SITU_OK) return s;
    if ((e = cudaEventRecord(ce->computed[slot], cs)) != cudaSuccess) return report_cuda_error(e);
    // copy out
    if ((e = cudaStreamWaitEvent(ce->out, ce->computed[slot], 0)) != cudaSuccess ||
        (e = cudaMemcpyAsync(yh + static_cast<size_t>(r0) * M * esz, ybuf[slot], bytes,
                             cudaMemcpyDeviceToHost, ce->out)) != cudaSuccess ||
        (e = cudaEventRecord(ce->stored[slot], ce->out)) != cudaSuccess)
      return report_cuda_error(e);
  }
  // The caller's stream completes after the last copy-out.
  for (int i = 0; i < 2 && i < nchunks; ++i) {
    if ((e = cudaStreamWaitEvent(cs, ce->stored[i], 0)) != cudaSuccess)
      return report_cuda_error(e);
  }
  return SITU_OK;
}
