// abi.cu -- the extern "C" entry points of libsitu (declared and documented in
// include/situ.h): argument validation, workspace carving and kernel launches.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>

#include "situ.h"
#include "situ_internal.h"
#include "situ_math.cuh"

namespace {

using namespace situ;

constexpr int kMaxDevices = 64;
// Grouped bf16 GEMMs run two-CTA MMAs when the experts average at least this many rows.
constexpr int64_t kTwoCtaMinRows = 128;

// Bound of every pipeline wait in the GEMM kernels (situ_set_wait_limit_ns).
constexpr uint64_t kDefaultWaitLimitNs = 10ull * 1000 * 1000 * 1000;  // 10 s
std::atomic<uint64_t> g_wait_limit_ns{kDefaultWaitLimitNs};

// Per-device status word: the first device-side failure since the last clear.
__device__ uint32_t g_device_status;

struct DeviceState {
  bool ready = false;
  int num_sms = 0;
  uint32_t* status = nullptr;  // device address of g_device_status
};

DeviceState g_devices[kMaxDevices];
std::mutex g_mutex;
thread_local char t_last_cuda_error[256] = "";
thread_local int t_ffn_path = 0;  // the path of this thread's last bf16 dense forward
std::atomic<int> g_ffn_single_launch{1};
// The grouped backward's K-grouped weight gradients on two-CTA MMAs (per-expert tensor
// maps); off: one CTA per tile (the path taken where two-CTA clusters cannot launch).
std::atomic<int> g_kgrouped_two_cta{1};

situ_status cuda_fail(cudaError_t e) {
  std::snprintf(t_last_cuda_error, sizeof t_last_cuda_error, "%s: %s", cudaGetErrorName(e),
                cudaGetErrorString(e));
  return SITU_ERR_CUDA;
}

// Set-up of the current device (once): SM count and the status word's address.
situ_status device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return SITU_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& st = g_devices[dev];
  if (!st.ready) {
    int major = 0;
    if ((e = cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev)) !=
        cudaSuccess)
      return cuda_fail(e);
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) !=
        cudaSuccess)
      return cuda_fail(e);
    if (major < 10) return SITU_ERR_UNSUPPORTED;
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_device_status)) != cudaSuccess) return cuda_fail(e);
    st.status = static_cast<uint32_t*>(p);
    st.ready = true;
  }
  *out = &st;
  return SITU_OK;
}

// Each cap is either finite in (0, 2^20] or +infinity (that branch uncapped).
bool caps_ok(float beta, float linear_beta) {
  auto one = [](float b) { return b == INFINITY || (b > 0.0f && b <= kMaxFiniteCap); };
  return one(beta) && one(linear_beta);
}

bool dtype_ok(situ_dtype dt) { return dt == SITU_BF16 || dt == SITU_F32; }

bool overlap(const void* a, size_t an, const void* b, size_t bn) {
  if (!a || !b || an == 0 || bn == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + bn && b0 < a0 + an;
}

bool aligned16(const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

situ_status finish(cudaError_t e) { return e == cudaSuccess ? SITU_OK : cuda_fail(e); }

}  // namespace

extern "C" {

int situ_abi_version(void) { return SITU_ABI_VERSION; }

const char* situ_status_string(situ_status s) {
  switch (s) {
    case SITU_OK: return "SITU_OK";
    case SITU_ERR_ARG: return "SITU_ERR_ARG";
    case SITU_ERR_ALIGN: return "SITU_ERR_ALIGN";
    case SITU_ERR_ALIAS: return "SITU_ERR_ALIAS";
    case SITU_ERR_CUDA: return "SITU_ERR_CUDA";
    case SITU_ERR_TIMEOUT: return "SITU_ERR_TIMEOUT";
    case SITU_ERR_UNSUPPORTED: return "SITU_ERR_UNSUPPORTED";
    case SITU_ERR_INDEX: return "SITU_ERR_INDEX";
    case SITU_ERR_WORKSPACE: return "SITU_ERR_WORKSPACE";
  }
  return "SITU_ERR_UNKNOWN";
}

const char* situ_last_cuda_error(void) { return t_last_cuda_error; }

int situ_ffn_last_path(void) { return t_ffn_path; }

int situ_ffn_set_single_launch(int enable) {
  return g_ffn_single_launch.exchange(enable ? 1 : 0);
}

int situ_moe_set_kgrouped_two_cta(int enable) {
  return g_kgrouped_two_cta.exchange(enable ? 1 : 0);
}

situ_status situ_device_status(int clear) {
  DeviceState* st = nullptr;
  situ_status s = device_state(&st);
  if (s != SITU_OK) return s;
  uint32_t v = 0;
  cudaError_t e = cudaMemcpy(&v, st->status, sizeof v, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  if (clear) {
    const uint32_t zero = 0;
    e = cudaMemcpy(st->status, &zero, sizeof zero, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return static_cast<situ_status>(v);
}

situ_status situ_glu_act(const void* gate_up, void* out, int64_t rows, int64_t I, float beta,
                         float linear_beta, situ_dtype dt, void* stream) {
  if (!dtype_ok(dt) || rows < 0 || I < 1 || !caps_ok(beta, linear_beta)) return SITU_ERR_ARG;
  if (rows == 0) return SITU_OK;
  if (!gate_up || !out) return SITU_ERR_ARG;
  const size_t esz = dtype_size(dt);
  if (overlap(gate_up, static_cast<size_t>(rows) * 2 * I * esz, out,
              static_cast<size_t>(rows) * I * esz))
    return SITU_ERR_ALIAS;
  if (reinterpret_cast<uintptr_t>(gate_up) % esz || reinterpret_cast<uintptr_t>(out) % esz)
    return SITU_ERR_ALIGN;
  DeviceState* st = nullptr;
  situ_status s = device_state(&st);
  if (s != SITU_OK) return s;
  return finish(launch_situ_act(gate_up, out, rows, I, make_situ_params(beta, linear_beta),
                                caps_of(beta, linear_beta), dt, st->num_sms,
                                static_cast<cudaStream_t>(stream)));
}

size_t situ_ffn_workspace_size(int64_t R, int64_t M, int64_t I, situ_dtype dt) {
  (void)M;
  if (R <= 0 || I <= 0 || !dtype_ok(dt)) return 0;
  const size_t h = round_up(static_cast<size_t>(R) * I * dtype_size(dt), 256);
  if (dt == SITU_F32) return h;
  // bf16: h, then one int32 per 128-row m-tile (the fused launch's h-ready counts).
  return h + round_up(static_cast<size_t>((R + 127) / 128) * 4, 256);
}

namespace {

// Shared argument checks of the dense FFN calls.
situ_status ffn_common_checks(situ_dtype dt, int64_t R, int64_t M, int64_t I, float beta,
                              float linear_beta) {
  if (!dtype_ok(dt) || R < 0 || M < 1 || I < 1 || !caps_ok(beta, linear_beta))
    return SITU_ERR_ARG;
  if (R >= (int64_t(1) << 31) || 2 * I >= (int64_t(1) << 31) || M >= (int64_t(1) << 31))
    return SITU_ERR_UNSUPPORTED;
  return SITU_OK;
}

situ_status bf16_gemm_checks(const void* a, const void* b, const void* c, int64_t M, int64_t I) {
  if (M % 8 || I % 8) return SITU_ERR_UNSUPPORTED;
  if (!aligned16(a) || !aligned16(b) || !aligned16(c)) return SITU_ERR_ALIGN;
  return SITU_OK;
}

cudaError_t run_gate_up(const DeviceState* st, const void* x, const void* W_gate_up, void* h,
                        int64_t R, int64_t M, int64_t I, float beta, float linear_beta,
                        cudaStream_t cs) {
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
  g.out = h;
  g.ldo = I;
  g.out_rows = R;
  return launch_gemm_situ(g, make_situ_params(beta, linear_beta), caps_of(beta, linear_beta),
                          st->status, st->num_sms, cs);
}

cudaError_t run_down(const DeviceState* st, const void* h, const void* W_down, void* y,
                     int64_t R, int64_t M, int64_t I, cudaStream_t cs) {
  GemmShape d{};
  d.a = h;
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
  return launch_gemm_plain(d, st->status, st->num_sms, cs);
}

}  // namespace

situ_status situ_ffn_forward(const void* x, const void* W_gate_up, const void* W_down, void* y,
                             void* workspace, size_t workspace_bytes, int64_t R, int64_t M,
                             int64_t I, float beta, float linear_beta, situ_dtype dt,
                             void* stream) {
  situ_status s = ffn_common_checks(dt, R, M, I, beta, linear_beta);
  if (s != SITU_OK || R == 0) return s;
  if (!x || !W_gate_up || !W_down || !y) return SITU_ERR_ARG;
  const size_t esz = dtype_size(dt);
  const size_t need = situ_ffn_workspace_size(R, M, I, dt);
  if (!workspace || workspace_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 256)
    return SITU_ERR_WORKSPACE;
  const size_t y_bytes = static_cast<size_t>(R) * M * esz;
  if (overlap(y, y_bytes, x, static_cast<size_t>(R) * M * esz) ||
      overlap(y, y_bytes, W_gate_up, static_cast<size_t>(2 * I) * M * esz) ||
      overlap(y, y_bytes, W_down, static_cast<size_t>(M) * I * esz) ||
      overlap(y, y_bytes, workspace, need) ||
      overlap(workspace, need, x, static_cast<size_t>(R) * M * esz) ||
      overlap(workspace, need, W_gate_up, static_cast<size_t>(2 * I) * M * esz) ||
      overlap(workspace, need, W_down, static_cast<size_t>(M) * I * esz))
    return SITU_ERR_ALIAS;
  DeviceState* st = nullptr;
  if ((s = device_state(&st)) != SITU_OK) return s;
  const SituParams p = make_situ_params(beta, linear_beta);
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (dt == SITU_F32) {
    if (reinterpret_cast<uintptr_t>(x) % 4 || reinterpret_cast<uintptr_t>(W_gate_up) % 4 ||
        reinterpret_cast<uintptr_t>(W_down) % 4 || reinterpret_cast<uintptr_t>(y) % 4)
      return SITU_ERR_ALIGN;
    return finish(launch_ffn_f32(static_cast<const float*>(x),
                                 static_cast<const float*>(W_gate_up),
                                 static_cast<const float*>(W_down),
                                 static_cast<float*>(workspace), static_cast<float*>(y), R, M,
                                 I, p, caps_of(beta, linear_beta), cs));
  }
  if ((s = bf16_gemm_checks(x, W_gate_up, W_down, M, I)) != SITU_OK) return s;
  if (!aligned16(y)) return SITU_ERR_ALIGN;
  // One persistent launch for both GEMMs (down tiles start as the gate_up tiles of
  // their rows complete); two launches when that grid cannot be co-resident.
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
  g.out = workspace;
  g.ldo = I;
  g.out_rows = R;
  GemmShape d{};
  d.a = workspace;
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
  int32_t* h_ready = reinterpret_cast<int32_t*>(
      static_cast<uint8_t*>(workspace) + round_up(static_cast<size_t>(R) * I * 2, 256));
  cudaError_t e = cudaSuccess;
  if (g_ffn_single_launch.load(std::memory_order_relaxed)) {
    e = launch_ffn_fused(g, d, p, caps_of(beta, linear_beta), h_ready, st->status, st->num_sms,
                         cs);
    if (e == cudaSuccess) {
      t_ffn_path = SITU_FFN_PATH_FUSED;
      return SITU_OK;
    }
    // A refused launch configuration is not sticky: clear it and take the two launches
    // (a sticky error fails them as well and is reported from there).
    (void)cudaGetLastError();
  }
  t_ffn_path = SITU_FFN_PATH_TWO_LAUNCHES;
  e = run_gate_up(st, x, W_gate_up, workspace, R, M, I, beta, linear_beta, cs);
  if (e != cudaSuccess) return cuda_fail(e);
  return finish(run_down(st, workspace, W_down, y, R, M, I, cs));
}

situ_status situ_ffn_gate_up(const void* x, const void* W_gate_up, void* h, int64_t R,
                             int64_t M, int64_t I, float beta, float linear_beta,
                             situ_dtype dt, void* stream) {
  situ_status s = ffn_common_checks(dt, R, M, I, beta, linear_beta);
  if (s != SITU_OK || R == 0) return s;
  if (!x || !W_gate_up || !h) return SITU_ERR_ARG;
  const size_t esz = dtype_size(dt);
  const size_t h_bytes = static_cast<size_t>(R) * I * esz;
  if (overlap(h, h_bytes, x, static_cast<size_t>(R) * M * esz) ||
      overlap(h, h_bytes, W_gate_up, static_cast<size_t>(2 * I) * M * esz))
    return SITU_ERR_ALIAS;
  if (dt == SITU_F32) return SITU_ERR_UNSUPPORTED;
  if ((s = bf16_gemm_checks(x, W_gate_up, h, M, I)) != SITU_OK) return s;
  DeviceState* st = nullptr;
  if ((s = device_state(&st)) != SITU_OK) return s;
  return finish(run_gate_up(st, x, W_gate_up, h, R, M, I, beta, linear_beta,
                            static_cast<cudaStream_t>(stream)));
}

situ_status situ_ffn_down(const void* h, const void* W_down, void* y, int64_t R, int64_t M,
                          int64_t I, situ_dtype dt, void* stream) {
  situ_status s = ffn_common_checks(dt, R, M, I, 1.0f, 1.0f);
  if (s != SITU_OK || R == 0) return s;
  if (!h || !W_down || !y) return SITU_ERR_ARG;
  const size_t esz = dtype_size(dt);
  const size_t y_bytes = static_cast<size_t>(R) * M * esz;
  if (overlap(y, y_bytes, h, static_cast<size_t>(R) * I * esz) ||
      overlap(y, y_bytes, W_down, static_cast<size_t>(M) * I * esz))
    return SITU_ERR_ALIAS;
  if (dt == SITU_F32) return SITU_ERR_UNSUPPORTED;
  if ((s = bf16_gemm_checks(h, W_down, y, M, I)) != SITU_OK) return s;
  DeviceState* st = nullptr;
  if ((s = device_state(&st)) != SITU_OK) return s;
  return finish(run_down(st, h, W_down, y, R, M, I, static_cast<cudaStream_t>(stream)));
}

situ_status situ_ffn_forward_train(const void* x, const void* W_gate_up, const void* W_down,
                                   void* y, void* gu, void* h, int64_t R, int64_t M,
                                   int64_t I, float beta, float linear_beta, situ_dtype dt,
                                   void* stream) {
  situ_status s = ffn_common_checks(dt, R, M, I, beta, linear_beta);
  if (s != SITU_OK || R == 0) return s;
  if (dt != SITU_BF16) return SITU_ERR_UNSUPPORTED;
  if (!x || !W_gate_up || !W_down || !y || !gu || !h) return SITU_ERR_ARG;
  if ((s = bf16_gemm_checks(x, W_gate_up, W_down, M, I)) != SITU_OK) return s;
  if (!aligned16(y) || !aligned16(gu) || !aligned16(h)) return SITU_ERR_ALIGN;
  const size_t xb = static_cast<size_t>(R) * M * 2, wgb = static_cast<size_t>(2 * I) * M * 2,
               wdb = static_cast<size_t>(M) * I * 2, gub = static_cast<size_t>(R) * 2 * I * 2,
               hb = static_cast<size_t>(R) * I * 2;
  const void* ins[] = {x, W_gate_up, W_down};
  const size_t inb[] = {xb, wgb, wdb};
  void* outs[] = {y, gu, h};
  const size_t outb[] = {xb, gub, hb};
  for (int o = 0; o < 3; ++o) {
    for (int i = 0; i < 3; ++i)
      if (overlap(outs[o], outb[o], ins[i], inb[i])) return SITU_ERR_ALIAS;
    for (int j = o + 1; j < 3; ++j)
      if (overlap(outs[o], outb[o], outs[j], outb[j])) return SITU_ERR_ALIAS;
  }
  DeviceState* st = nullptr;
  if ((s = device_state(&st)) != SITU_OK) return s;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
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
  g.out = h;
  g.ldo = I;
  g.out_rows = R;
  g.gu_store = gu;
  g.split = I;
  cudaError_t e = launch_gemm_situ(g, make_situ_params(beta, linear_beta),
                                   caps_of(beta, linear_beta), st->status, st->num_sms, cs);
  if (e != cudaSuccess) return cuda_fail(e);
  return finish(run_down(st, h, W_down, y, R, M, I, cs));
}

size_t situ_ffn_backward_workspace_size(int64_t R, int64_t M, int64_t I, situ_dtype dt) {
  (void)M;
  if (R <= 0 || I <= 0 || dt != SITU_BF16) return 0;
  return round_up(static_cast<size_t>(R) * 2 * I * 2, 256);  // dgu [R, 2I]
}

situ_status situ_ffn_backward(const void* x, const void* W_gate_up, const void* W_down,
                              const void* gu, const void* h, const void* dy, void* dx,
                              void* dW_gate_up, void* dW_down, void* workspace,
                              size_t workspace_bytes, int64_t R, int64_t M, int64_t I,
                              float beta, float linear_beta, situ_dtype dt, void* stream) {
  situ_status s = ffn_common_checks(dt, R, M, I, beta, linear_beta);
  if (s != SITU_OK) return s;
  if (dt != SITU_BF16) return SITU_ERR_UNSUPPORTED;
  if (R < 1) return SITU_ERR_ARG;
  if (!x || !W_gate_up || !W_down || !gu || !h || !dy || !dx || !dW_gate_up || !dW_down)
    return SITU_ERR_ARG;
  if (M % 8 || I % 8) return SITU_ERR_UNSUPPORTED;
  const void* ptrs[] = {x, W_gate_up, W_down, gu, h, dy, dx, dW_gate_up, dW_down};
  for (const void* q : ptrs)
    if (!aligned16(q)) return SITU_ERR_ALIGN;
  const size_t need = situ_ffn_backward_workspace_size(R, M, I, dt);
  if (!workspace || workspace_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 256)
    return SITU_ERR_WORKSPACE;
  const size_t xb = static_cast<size_t>(R) * M * 2, wgb = static_cast<size_t>(2 * I) * M * 2,
               wdb = static_cast<size_t>(M) * I * 2, gub = static_cast<size_t>(R) * 2 * I * 2,
               hb = static_cast<size_t>(R) * I * 2;
  const void* ins[] = {x, W_gate_up, W_down, gu, h, dy, workspace};
  const size_t inb[] = {xb, wgb, wdb, gub, hb, xb, need};
  void* outs[] = {dx, dW_gate_up, dW_down};
  const size_t outb[] = {xb, wgb, wdb};
  for (int o = 0; o < 3; ++o) {
    for (int i = 0; i < 7; ++i)
      if (overlap(outs[o], outb[o], ins[i], inb[i])) return SITU_ERR_ALIAS;
    for (int j = o + 1; j < 3; ++j)
      if (overlap(outs[o], outb[o], outs[j], outb[j])) return SITU_ERR_ALIAS;
  }
  DeviceState* st = nullptr;
  if ((s = device_state(&st)) != SITU_OK) return s;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  void* dgu = workspace;
  cudaError_t e;
  // dh = dy W_down (W_down [M, I] read as an MN-major [K = M, N = I] operand);
  // the epilogue turns dh into d(g, u) at the saved gu.
  {
    GemmShape g{};
    g.a = dy;
    g.a_rows = R;
    g.b = W_down;
    g.b_rows = I;
    g.b_mn_major = true;
    g.K = M;
    g.num_groups = 1;
    g.n_out = I;
    g.out = dgu;
    g.ldo = 2 * I;
    g.out_rows = R;
    g.gu_in = gu;
    g.dgu_out = dgu;
    g.split = I;
    e = launch_gemm_situ_bwd(g, make_situ_params(beta, linear_beta), caps_of(beta, linear_beta),
                             st->status, st->num_sms, cs);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  // dx = dgu W_gate_up (W_gate_up [2I, M] read as MN-major [K = 2I, N = M]).
  {
    GemmShape g{};
    g.a = dgu;
    g.a_rows = R;
    g.b = W_gate_up;
    g.b_rows = M;
    g.b_mn_major = true;
    g.K = 2 * I;
    g.num_groups = 1;
    g.n_out = M;
    g.out = dx;
    g.ldo = M;
    g.out_rows = R;
    if ((e = launch_gemm_plain(g, st->status, st->num_sms, cs)) != cudaSuccess)
      return cuda_fail(e);
  }
  // The weight gradients, both operands read MN-major, contracting over the R rows,
  // in one launch (their tiles together fill the last wave better than either alone):
  // dW_down = dy^T h and dW_gate_up = dgu^T x.
  {
    GemmShape g{};
    g.a = dy;
    g.a_rows = M;
    g.a_mn_major = true;
    g.b = h;
    g.b_rows = I;
    g.b_mn_major = true;
    g.K = R;
    g.num_groups = 1;
    g.n_out = I;
    g.out = dW_down;
    g.ldo = I;
    g.out_rows = M;
    GemmShape g2{};
    g2.a = dgu;
    g2.a_rows = 2 * I;
    g2.a_mn_major = true;
    g2.b = x;
    g2.b_rows = M;
    g2.b_mn_major = true;
    g2.K = R;
    g2.num_groups = 1;
    g2.n_out = M;
    g2.out = dW_gate_up;
    g2.ldo = M;
    g2.out_rows = 2 * I;
    if ((e = launch_gemm_plain2(g, g2, st->status, st->num_sms, cs)) != cudaSuccess)
      return cuda_fail(e);
  }
  return SITU_OK;
}

size_t situ_moe_index_workspace_size(int64_t n_routes, int32_t E) {
  if (n_routes < 0 || E < 1) return 0;
  return round_up(index_workspace_bytes(n_routes, E), 256);
}

situ_status situ_moe_build_index(const int32_t* expert_ids, int32_t* expert_offsets,
                                 int32_t* token_index, void* workspace, size_t workspace_bytes,
                                 int64_t n_routes, int32_t E, void* stream) {
  if (n_routes < 0 || n_routes >= (int64_t(1) << 31) || E < 1 || E > 16384) return SITU_ERR_ARG;
  if (!expert_offsets || (n_routes > 0 && (!expert_ids || !token_index))) return SITU_ERR_ARG;
  const size_t need = situ_moe_index_workspace_size(n_routes, E);
  if (!workspace || workspace_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 16)
    return SITU_ERR_WORKSPACE;
  const size_t ids_b = static_cast<size_t>(n_routes) * 4, off_b = static_cast<size_t>(E + 1) * 4;
  if (overlap(expert_offsets, off_b, expert_ids, ids_b) ||
      overlap(token_index, ids_b, expert_ids, ids_b) ||
      overlap(token_index, ids_b, expert_offsets, off_b) ||
      overlap(workspace, need, expert_ids, ids_b) ||
      overlap(workspace, need, expert_offsets, off_b) ||
      overlap(workspace, need, token_index, ids_b))
    return SITU_ERR_ALIAS;
  DeviceState* st = nullptr;
  situ_status s = device_state(&st);
  if (s != SITU_OK) return s;
  return finish(launch_build_index(expert_ids, expert_offsets, token_index, workspace, n_routes,
                                   E, st->status, static_cast<cudaStream_t>(stream)));
}

size_t situ_moe_workspace_size(int64_t R, int32_t E, int64_t M, int64_t I, situ_dtype dt) {
  if (R < 0 || E < 1 || M < 1 || I < 1 || dt != SITU_BF16) return 0;
  // m-tile prefix + work-unit prefixes of the two GEMMs
  const size_t tiles = 3 * round_up(static_cast<size_t>(E + 1) * 4, 256);
  const size_t xperm = round_up(static_cast<size_t>(R) * M * 2, 256);
  const size_t h = round_up(static_cast<size_t>(R) * I * 2, 256);
  return tiles + xperm + h;
}

// Shared argument checks of the grouped entry points.
situ_status moe_common_checks(const void* x, const int32_t* expert_offsets,
                              const int32_t* token_index, const void* W_gate_up,
                              const void* W_down, int64_t T, int32_t k_eff, int32_t E, int64_t M,
                              int64_t I, float beta, float linear_beta, situ_dtype dt) {
  if (dt != SITU_BF16) return dt == SITU_F32 ? SITU_ERR_UNSUPPORTED : SITU_ERR_ARG;
  if (T < 0 || k_eff < 1 || E < 1 || E > 65536 || M < 1 || I < 1 || !caps_ok(beta, linear_beta))
    return SITU_ERR_ARG;
  const int64_t R = T * k_eff;
  if (R == 0) return SITU_OK;
  if (!x || !expert_offsets || !token_index || !W_gate_up || !W_down) return SITU_ERR_ARG;
  if (R >= (int64_t(1) << 31) || static_cast<int64_t>(E) * 2 * I >= (int64_t(1) << 31) ||
      static_cast<int64_t>(E) * M >= (int64_t(1) << 31))
    return SITU_ERR_UNSUPPORTED;
  if (M % 8 || I % 8) return SITU_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(W_gate_up) || !aligned16(W_down)) return SITU_ERR_ALIGN;
  return SITU_OK;
}

// The grouped forward; gu_store (training) additionally keeps the pre-activation;
// with combine_w the down GEMM adds the weighted rows into combine_acc instead of
// writing y.
situ_status moe_forward_impl(const void* x, const int32_t* expert_offsets,
                             const int32_t* token_index, const void* W_gate_up,
                             const void* W_down, void* y, void* h_perm, void* gu_store,
                             void* workspace, int64_t T, int32_t k_eff, int32_t E, int64_t M,
                             int64_t I, float beta, float linear_beta, cudaStream_t cs,
                             const float* combine_w = nullptr, float* combine_acc = nullptr) {
  const int64_t R = T * k_eff;
  DeviceState* st = nullptr;
  situ_status s = device_state(&st);
  if (s != SITU_OK) return s;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t prefix_bytes = round_up(static_cast<size_t>(E + 1) * 4, 256);
  int32_t* tile_offsets = reinterpret_cast<int32_t*>(ws);
  int32_t* units_gu = reinterpret_cast<int32_t*>(ws + prefix_bytes);
  int32_t* units_dn = reinterpret_cast<int32_t*>(ws + 2 * prefix_bytes);
  void* x_perm = ws + 3 * prefix_bytes;

  // Experts averaging at least 128 rows run as two-CTA MMAs (M = 256 over a CTA pair; an
  // expert's odd last m-tile as an M = 128 pair, 64 rows per CTA); experts of a few
  // rows (decode) stream their weights through the one-CTA kernel's 64-row MMAs.
  const bool two_cta = R >= kTwoCtaMinRows * static_cast<int64_t>(E) && gemm_two_cta_available();
  cudaError_t e = launch_group_tiles(expert_offsets, E, R, gemm_n_tiles_situ(I),
                                     gemm_n_tiles_wide(M), tile_offsets, units_gu, units_dn,
                                     st->status, cs, two_cta);
  if (e != cudaSuccess) return cuda_fail(e);
  e = launch_gather_rows(x, token_index, x_perm, R, k_eff, M, st->status, cs);
  if (e != cudaSuccess) return cuda_fail(e);
  const SituParams p = make_situ_params(beta, linear_beta);
  GemmShape g{};
  g.a = x_perm;
  g.a_rows = R;
  g.b = W_gate_up;
  g.b_rows = static_cast<int64_t>(E) * 2 * I;
  g.K = M;
  g.num_groups = E;
  g.group_offsets = expert_offsets;
  g.tile_offsets = tile_offsets;
  g.unit_offsets = units_gu;
  g.pair_units = two_cta;
  g.b_group_rows = 2 * I;
  g.b_up_offset = I;
  g.n_out = I;
  g.out = h_perm;
  g.ldo = I;
  g.out_rows = R;
  g.gu_store = gu_store;
  g.split = I;
  e = launch_gemm_situ(g, p, caps_of(beta, linear_beta), st->status, st->num_sms, cs);
  if (e != cudaSuccess) return cuda_fail(e);
  GemmShape d{};
  d.a = h_perm;
  d.a_rows = R;
  d.b = W_down;
  d.b_rows = static_cast<int64_t>(E) * M;
  d.K = I;
  d.num_groups = E;
  d.group_offsets = expert_offsets;
  d.tile_offsets = tile_offsets;
  d.unit_offsets = units_dn;
  d.pair_units = two_cta;
  d.b_group_rows = M;
  d.n_out = M;
  d.out = y;
  d.ldo = M;
  d.out_rows = R;
  d.out_row_index = token_index;
  d.combine_w = combine_w;
  d.combine_out = combine_acc;
  d.combine_k = k_eff;
  return finish(launch_gemm_plain(d, st->status, st->num_sms, cs));
}

situ_status situ_moe_grouped_forward(const void* x, const int32_t* expert_offsets,
                                     const int32_t* token_index, const void* W_gate_up,
                                     const void* W_down, void* y, void* workspace,
                                     size_t workspace_bytes, int64_t T, int32_t k_eff,
                                     int32_t E, int64_t M, int64_t I, float beta,
                                     float linear_beta, situ_dtype dt, void* stream) {
  situ_status s = moe_common_checks(x, expert_offsets, token_index, W_gate_up, W_down, T, k_eff,
                                    E, M, I, beta, linear_beta, dt);
  const int64_t R = T * k_eff;
  if (s != SITU_OK || R == 0) return s;
  if (!y) return SITU_ERR_ARG;
  if (!aligned16(y)) return SITU_ERR_ALIGN;
  const size_t need = situ_moe_workspace_size(R, E, M, I, dt);
  if (!workspace || workspace_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 256)
    return SITU_ERR_WORKSPACE;
  const size_t x_b = static_cast<size_t>(T) * M * 2, y_b = static_cast<size_t>(R) * M * 2;
  const size_t wgu_b = static_cast<size_t>(E) * 2 * I * M * 2, wd_b = static_cast<size_t>(E) * M * I * 2;
  const size_t off_b = static_cast<size_t>(E + 1) * 4, tix_b = static_cast<size_t>(R) * 4;
  const void* ins[] = {x, W_gate_up, W_down, expert_offsets, token_index};
  const size_t in_b[] = {x_b, wgu_b, wd_b, off_b, tix_b};
  for (int i = 0; i < 5; ++i) {
    if (overlap(y, y_b, ins[i], in_b[i]) || overlap(workspace, need, ins[i], in_b[i]))
      return SITU_ERR_ALIAS;
  }
  if (overlap(y, y_b, workspace, need)) return SITU_ERR_ALIAS;
  const size_t prefix_bytes = round_up(static_cast<size_t>(E + 1) * 4, 256);
  void* h_perm = static_cast<uint8_t*>(workspace) + 3 * prefix_bytes +
                 round_up(static_cast<size_t>(R) * M * 2, 256);
  return moe_forward_impl(x, expert_offsets, token_index, W_gate_up, W_down, y, h_perm, nullptr,
                          workspace, T, k_eff, E, M, I, beta, linear_beta,
                          static_cast<cudaStream_t>(stream));
}

situ_status situ_moe_grouped_forward_train(const void* x, const int32_t* expert_offsets,
                                           const int32_t* token_index, const void* W_gate_up,
                                           const void* W_down, void* y, void* gu, void* h,
                                           void* workspace, size_t workspace_bytes, int64_t T,
                                           int32_t k_eff, int32_t E, int64_t M, int64_t I,
                                           float beta, float linear_beta, situ_dtype dt,
                                           void* stream) {
  situ_status s = moe_common_checks(x, expert_offsets, token_index, W_gate_up, W_down, T, k_eff,
                                    E, M, I, beta, linear_beta, dt);
  const int64_t R = T * k_eff;
  if (s != SITU_OK || R == 0) return s;
  if (!y || !gu || !h) return SITU_ERR_ARG;
  if (!aligned16(y) || !aligned16(gu) || !aligned16(h)) return SITU_ERR_ALIGN;
  const size_t need = situ_moe_workspace_size(R, E, M, I, dt);
  if (!workspace || workspace_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 256)
    return SITU_ERR_WORKSPACE;
  const size_t x_b = static_cast<size_t>(T) * M * 2, y_b = static_cast<size_t>(R) * M * 2;
  const size_t wgu_b = static_cast<size_t>(E) * 2 * I * M * 2, wd_b = static_cast<size_t>(E) * M * I * 2;
  const size_t off_b = static_cast<size_t>(E + 1) * 4, tix_b = static_cast<size_t>(R) * 4;
  const size_t gu_b = static_cast<size_t>(R) * 2 * I * 2, h_b = static_cast<size_t>(R) * I * 2;
  const void* ins[] = {x, W_gate_up, W_down, expert_offsets, token_index};
  const size_t in_b[] = {x_b, wgu_b, wd_b, off_b, tix_b};
  void* outs[] = {y, gu, h, workspace};
  const size_t out_b[] = {y_b, gu_b, h_b, need};
  for (int o = 0; o < 4; ++o) {
    for (int i = 0; i < 5; ++i)
      if (overlap(outs[o], out_b[o], ins[i], in_b[i])) return SITU_ERR_ALIAS;
    for (int j = o + 1; j < 4; ++j)
      if (overlap(outs[o], out_b[o], outs[j], out_b[j])) return SITU_ERR_ALIAS;
  }
  return moe_forward_impl(x, expert_offsets, token_index, W_gate_up, W_down, y, h, gu, workspace,
                          T, k_eff, E, M, I, beta, linear_beta,
                          static_cast<cudaStream_t>(stream));
}

size_t situ_moe_combined_workspace_size(int64_t T, int32_t k_eff, int32_t E, int64_t M,
                                        int64_t I, situ_dtype dt) {
  if (T < 0 || k_eff < 1) return 0;
  const size_t base = situ_moe_workspace_size(T * k_eff, E, M, I, dt);
  if (base == 0) return 0;
  return base + round_up(static_cast<size_t>(T) * M * 4, 256);  // FP32 accumulator [T, M]
}

situ_status situ_moe_grouped_forward_combined(const void* x, const int32_t* expert_offsets,
                                              const int32_t* token_index, const void* W_gate_up,
                                              const void* W_down, const float* weights,
                                              void* out, void* workspace, size_t workspace_bytes,
                                              int64_t T, int32_t k_eff, int32_t E, int64_t M,
                                              int64_t I, float beta, float linear_beta,
                                              situ_dtype dt, void* stream) {
  situ_status s = moe_common_checks(x, expert_offsets, token_index, W_gate_up, W_down, T, k_eff,
                                    E, M, I, beta, linear_beta, dt);
  const int64_t R = T * k_eff;
  if (s != SITU_OK || R == 0) return s;
  if (!weights || !out) return SITU_ERR_ARG;
  if (!aligned16(out)) return SITU_ERR_ALIGN;
  const size_t need = situ_moe_combined_workspace_size(T, k_eff, E, M, I, dt);
  if (!workspace || workspace_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 256)
    return SITU_ERR_WORKSPACE;
  const size_t x_b = static_cast<size_t>(T) * M * 2, out_b = x_b;
  const size_t wgu_b = static_cast<size_t>(E) * 2 * I * M * 2, wd_b = static_cast<size_t>(E) * M * I * 2;
  const size_t off_b = static_cast<size_t>(E + 1) * 4, tix_b = static_cast<size_t>(R) * 4,
               w_b = static_cast<size_t>(R) * 4;
  const void* ins[] = {x, W_gate_up, W_down, expert_offsets, token_index, weights};
  const size_t in_b[] = {x_b, wgu_b, wd_b, off_b, tix_b, w_b};
  for (int i = 0; i < 6; ++i)
    if (overlap(out, out_b, ins[i], in_b[i]) || overlap(workspace, need, ins[i], in_b[i]))
      return SITU_ERR_ALIAS;
  if (overlap(out, out_b, workspace, need)) return SITU_ERR_ALIAS;
  DeviceState* st = nullptr;
  if ((s = device_state(&st)) != SITU_OK) return s;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const size_t base = situ_moe_workspace_size(R, E, M, I, dt);
  float* acc = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + base);
  cudaError_t e = cudaMemsetAsync(acc, 0, static_cast<size_t>(T) * M * 4, cs);
  if (e != cudaSuccess) return cuda_fail(e);
  const size_t prefix_bytes = round_up(static_cast<size_t>(E + 1) * 4, 256);
  void* h_perm = static_cast<uint8_t*>(workspace) + 3 * prefix_bytes +
                 round_up(static_cast<size_t>(R) * M * 2, 256);
  s = moe_forward_impl(x, expert_offsets, token_index, W_gate_up, W_down, nullptr, h_perm,
                       nullptr, workspace, T, k_eff, E, M, I, beta, linear_beta, cs, weights, acc);
  if (s != SITU_OK) return s;
  return finish(launch_f32_to_bf16(acc, out, T * M, st->num_sms, cs));
}

}  // extern "C"

namespace {
// Bytes of one GEMM's per-expert tensor maps (two 128-byte maps per expert).
size_t moe_group_maps_bytes(int32_t E) {
  return round_up(static_cast<size_t>(E) * 2 * 128, 256);
}
}  // namespace

extern "C" {

size_t situ_moe_backward_workspace_size(int64_t R, int32_t E, int64_t M, int64_t I,
                                        situ_dtype dt) {
  if (R < 0 || E < 1 || M < 1 || I < 1 || dt != SITU_BF16) return 0;
  // m-tile prefix + work-unit prefixes of the dh and dx GEMMs + the experts by
  // descending rows, the per-expert tensor maps of the two weight-gradient GEMMs, one
  // [R, M] buffer (dy in expert order, then the per-route dx, then x in expert order)
  // and d(g, u) [R, 2I] in expert order.
  const size_t tiles = 4 * round_up(static_cast<size_t>(E + 1) * 4, 256);
  const size_t maps = 2 * moe_group_maps_bytes(E);
  const size_t rows_m = round_up(static_cast<size_t>(R) * M * 2, 256);
  const size_t dgu = round_up(static_cast<size_t>(R) * 2 * I * 2, 256);
  return tiles + maps + rows_m + dgu;
}

situ_status situ_moe_grouped_backward(const void* x, const int32_t* expert_offsets,
                                      const int32_t* token_index, const void* W_gate_up,
                                      const void* W_down, const void* gu, const void* h,
                                      const void* dy, void* dx, void* dW_gate_up, void* dW_down,
                                      void* workspace, size_t workspace_bytes, int64_t T,
                                      int32_t k_eff, int32_t E, int64_t M, int64_t I, float beta,
                                      float linear_beta, situ_dtype dt, void* stream) {
  situ_status s = moe_common_checks(x, expert_offsets, token_index, W_gate_up, W_down, T, k_eff,
                                    E, M, I, beta, linear_beta, dt);
  if (s != SITU_OK) return s;
  const int64_t R = T * k_eff;
  if (!dW_gate_up || !dW_down) return SITU_ERR_ARG;
  if (!aligned16(dW_gate_up) || !aligned16(dW_down)) return SITU_ERR_ALIGN;
  if (M % 8 || I % 8) return SITU_ERR_UNSUPPORTED;
  const size_t wgu_b = static_cast<size_t>(E) * 2 * I * M * 2, wd_b = static_cast<size_t>(E) * M * I * 2;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (R == 0) {
    // No routes: every expert's weight gradient is zero and dx is empty.
    if (overlap(dW_gate_up, wgu_b, dW_down, wd_b)) return SITU_ERR_ALIAS;
    DeviceState* st = nullptr;
    if ((s = device_state(&st)) != SITU_OK) return s;
    cudaError_t e = cudaMemsetAsync(dW_gate_up, 0, wgu_b, cs);
    if (e == cudaSuccess) e = cudaMemsetAsync(dW_down, 0, wd_b, cs);
    return finish(e);
  }
  if (!gu || !h || !dy || !dx) return SITU_ERR_ARG;
  if (!aligned16(gu) || !aligned16(h) || !aligned16(dy) || !aligned16(dx)) return SITU_ERR_ALIGN;
  const size_t need = situ_moe_backward_workspace_size(R, E, M, I, dt);
  if (!workspace || workspace_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 256)
    return SITU_ERR_WORKSPACE;
  const size_t x_b = static_cast<size_t>(T) * M * 2, dy_b = static_cast<size_t>(R) * M * 2;
  const size_t off_b = static_cast<size_t>(E + 1) * 4, tix_b = static_cast<size_t>(R) * 4;
  const size_t gu_b = static_cast<size_t>(R) * 2 * I * 2, h_b = static_cast<size_t>(R) * I * 2;
  const void* ins[] = {x, W_gate_up, W_down, expert_offsets, token_index, gu, h, dy};
  const size_t in_b[] = {x_b, wgu_b, wd_b, off_b, tix_b, gu_b, h_b, dy_b};
  void* outs[] = {dx, dW_gate_up, dW_down, workspace};
  const size_t out_b[] = {x_b, wgu_b, wd_b, need};
  for (int o = 0; o < 4; ++o) {
    for (int i = 0; i < 8; ++i)
      if (overlap(outs[o], out_b[o], ins[i], in_b[i])) return SITU_ERR_ALIAS;
    for (int j = o + 1; j < 4; ++j)
      if (overlap(outs[o], out_b[o], outs[j], out_b[j])) return SITU_ERR_ALIAS;
  }
  DeviceState* st = nullptr;
  if ((s = device_state(&st)) != SITU_OK) return s;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t prefix_bytes = round_up(static_cast<size_t>(E + 1) * 4, 256);
  int32_t* tile_offsets = reinterpret_cast<int32_t*>(ws);
  int32_t* units_dh = reinterpret_cast<int32_t*>(ws + prefix_bytes);
  int32_t* units_dx = reinterpret_cast<int32_t*>(ws + 2 * prefix_bytes);
  int32_t* expert_order = reinterpret_cast<int32_t*>(ws + 3 * prefix_bytes);
  void* maps_dwd = ws + 4 * prefix_bytes;  // per-expert tensor maps of dW_down
  void* maps_dwg = static_cast<uint8_t*>(maps_dwd) + moe_group_maps_bytes(E);  // of dW_gate_up
  void* rows_m = static_cast<uint8_t*>(maps_dwg) + moe_group_maps_bytes(E);  // [R, M]
  void* dgu = static_cast<uint8_t*>(rows_m) + round_up(static_cast<size_t>(R) * M * 2, 256);
  const SituParams p = make_situ_params(beta, linear_beta);
  // The dh and dx GEMMs run as two-CTA MMAs when experts average >= 128 rows (as the
  // forward); the K-grouped weight gradients always do (one CTA per tile only where
  // two-CTA clusters cannot be launched, or with situ_moe_set_kgrouped_two_cta(0)).
  const bool kg_two_cta = g_kgrouped_two_cta.load() != 0;
  const bool two_cta = R >= kTwoCtaMinRows * static_cast<int64_t>(E) && gemm_two_cta_available();
  cudaError_t e = launch_group_tiles(expert_offsets, E, R, gemm_n_tiles_wide(I),
                                     gemm_n_tiles_wide(M), tile_offsets, units_dh, units_dx,
                                     st->status, cs, two_cta);
  if (e != cudaSuccess) return cuda_fail(e);
  if ((e = launch_group_order(expert_offsets, E, expert_order, cs)) != cudaSuccess)
    return cuda_fail(e);
  // dy in expert order: dy_perm[r] = dy[token_index[r]] (one row per route).
  e = launch_gather_rows(dy, token_index, rows_m, R, 1, M, st->status, cs);
  if (e != cudaSuccess) return cuda_fail(e);
  // dh = dy W_down[e] per expert (W_down[e] [M, I] read as MN-major [K = M, N = I]);
  // the epilogue turns dh into d(g, u) at the saved pre-activation.
  {
    GemmShape g{};
    g.a = rows_m;
    g.a_rows = R;
    g.b = W_down;
    g.b_rows = I;
    g.b_mn_major = true;
    g.K = M;
    g.num_groups = E;
    g.group_offsets = expert_offsets;
    g.tile_offsets = tile_offsets;
    g.unit_offsets = units_dh;
    g.pair_units = two_cta;
    g.b_group_rows = M;
    g.n_out = I;
    g.out = dgu;
    g.ldo = 2 * I;
    g.out_rows = R;
    g.gu_in = gu;
    g.dgu_out = dgu;
    g.split = I;
    e = launch_gemm_situ_bwd(g, p, caps_of(beta, linear_beta), st->status, st->num_sms, cs);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  // dW_down[e] = dy_e^T h_e: contraction over each expert's own rows.
  {
    GemmShape g{};
    g.a = rows_m;
    g.a_rows = M;
    g.a_mn_major = true;
    g.b = h;
    g.b_rows = I;
    g.b_mn_major = true;
    g.K = R;
    g.num_groups = E;
    g.tile_offsets = tile_offsets;
    g.k_group_offsets = expert_offsets;
    g.group_order = expert_order;
    g.group_maps = kg_two_cta ? maps_dwd : nullptr;
    g.out_group_rows = M;
    g.n_out = I;
    g.out = dW_down;
    g.ldo = I;
    g.out_rows = static_cast<int64_t>(E) * M;
    if ((e = launch_gemm_plain(g, st->status, st->num_sms, cs)) != cudaSuccess)
      return cuda_fail(e);
  }
  // Per-route dx = d(g, u) W_gate_up[e] (W_gate_up[e] [2I, M] as MN-major
  // [K = 2I, N = M]), written in (token, slot) order over the dy rows.
  {
    GemmShape g{};
    g.a = dgu;
    g.a_rows = R;
    g.b = W_gate_up;
    g.b_rows = M;
    g.b_mn_major = true;
    g.K = 2 * I;
    g.num_groups = E;
    g.group_offsets = expert_offsets;
    g.tile_offsets = tile_offsets;
    g.unit_offsets = units_dx;
    g.pair_units = two_cta;
    g.b_group_rows = 2 * I;
    g.n_out = M;
    g.out = rows_m;
    g.ldo = M;
    g.out_rows = R;
    g.out_row_index = token_index;
    if ((e = launch_gemm_plain(g, st->status, st->num_sms, cs)) != cudaSuccess)
      return cuda_fail(e);
  }
  // dx[t] = sum over the token's slots of the per-route dx (FP32, slot order).
  if ((e = launch_combine(rows_m, nullptr, dx, T, k_eff, M, SITU_BF16, st->num_sms, cs)) !=
      cudaSuccess)
    return cuda_fail(e);
  // x in expert order, then dW_gate_up[e] = d(g, u)_e^T x_e.
  if ((e = launch_gather_rows(x, token_index, rows_m, R, k_eff, M, st->status, cs)) !=
      cudaSuccess)
    return cuda_fail(e);
  {
    GemmShape g{};
    g.a = dgu;
    g.a_rows = 2 * I;
    g.a_mn_major = true;
    g.b = rows_m;
    g.b_rows = M;
    g.b_mn_major = true;
    g.K = R;
    g.num_groups = E;
    g.tile_offsets = tile_offsets;
    g.k_group_offsets = expert_offsets;
    g.group_order = expert_order;
    g.group_maps = kg_two_cta ? maps_dwg : nullptr;
    g.out_group_rows = 2 * I;
    g.n_out = M;
    g.out = dW_gate_up;
    g.ldo = M;
    g.out_rows = static_cast<int64_t>(E) * 2 * I;
    if ((e = launch_gemm_plain(g, st->status, st->num_sms, cs)) != cudaSuccess)
      return cuda_fail(e);
  }
  return SITU_OK;
}

// ---------------------------------------------------------------------------
// MXFP8
// ---------------------------------------------------------------------------
namespace {

int64_t mx_weight_rows(int kind, int64_t M, int64_t I) { return kind == SITU_MX_GATE_UP ? 2 * I : M; }
int64_t mx_weight_k(int kind, int64_t M, int64_t I) { return kind == SITU_MX_GATE_UP ? M : I; }
int64_t mx_weight_split(int kind, int64_t I) { return kind == SITU_MX_GATE_UP ? I : 0; }

bool mx_shape_ok(int64_t M, int64_t I) { return M >= 128 && I >= 128 && M % 128 == 0 && I % 128 == 0; }
bool mx_fmt_ok(int fmt) { return fmt == SITU_MX_E4M3 || fmt == SITU_MX_E2M1; }
// Bytes of the codes of E weight matrices [rows, K] in format fmt.
size_t mx_weight_code_bytes(int32_t E, int64_t rows, int64_t K, int fmt) {
  return static_cast<size_t>(E) * rows * (fmt == SITU_MX_E2M1 ? K / 2 : K);
}

}  // namespace

size_t situ_mx_act_scales_size(int64_t R, int64_t K) {
  if (R < 0 || K <= 0 || K % 128 != 0) return 0;
  return mx_act_scale_bytes(R, K);
}

size_t situ_mx_weight_scales_size(int32_t E, int64_t M, int64_t I, int kind) {
  if (E < 1 || (kind != SITU_MX_GATE_UP && kind != SITU_MX_DOWN) || !mx_shape_ok(M, I)) return 0;
  return mx_weight_scale_bytes(E, mx_weight_rows(kind, M, I), mx_weight_k(kind, M, I),
                               mx_weight_split(kind, I));
}

situ_status situ_mx_quantize_act(const void* x, void* codes, void* scales, int64_t R, int64_t K,
                                 void* stream) {
  if (R < 0 || K <= 0) return SITU_ERR_ARG;
  if (K % 128 != 0) return SITU_ERR_UNSUPPORTED;
  if (R == 0) return SITU_OK;
  if (!x || !codes || !scales) return SITU_ERR_ARG;
  if (!aligned16(x) || !aligned16(codes)) return SITU_ERR_ALIGN;
  const size_t xb = static_cast<size_t>(R) * K * 2, cb = static_cast<size_t>(R) * K,
               sb = mx_act_scale_bytes(R, K);
  if (overlap(codes, cb, x, xb) || overlap(scales, sb, x, xb) || overlap(codes, cb, scales, sb))
    return SITU_ERR_ALIAS;
  DeviceState* st = nullptr;
  situ_status s = device_state(&st);
  if (s != SITU_OK) return s;
  return finish(launch_mx_quantize_act(x, nullptr, 1, R, codes, scales, (R + 127) / 128, R, K, 0,
                                       nullptr, nullptr, st->status,
                                       static_cast<cudaStream_t>(stream)));
}

situ_status situ_mx_quantize_weights(const void* W, void* codes, void* scales, int32_t E,
                                     int64_t M, int64_t I, int kind, int fmt, void* stream) {
  if (E < 1 || M < 1 || I < 1 || (kind != SITU_MX_GATE_UP && kind != SITU_MX_DOWN) ||
      !mx_fmt_ok(fmt))
    return SITU_ERR_ARG;
  if (!mx_shape_ok(M, I)) return SITU_ERR_UNSUPPORTED;
  if (!W || !codes || !scales) return SITU_ERR_ARG;
  if (!aligned16(W) || !aligned16(codes)) return SITU_ERR_ALIGN;
  const int64_t rows = mx_weight_rows(kind, M, I), K = mx_weight_k(kind, M, I);
  const size_t wb = static_cast<size_t>(E) * rows * K * 2,
               cb = mx_weight_code_bytes(E, rows, K, fmt),
               sb = situ_mx_weight_scales_size(E, M, I, kind);
  if (overlap(codes, cb, W, wb) || overlap(scales, sb, W, wb) || overlap(codes, cb, scales, sb))
    return SITU_ERR_ALIAS;
  DeviceState* st = nullptr;
  situ_status s = device_state(&st);
  if (s != SITU_OK) return s;
  return finish(launch_mx_quantize_weights(W, codes, scales, E, rows, K,
                                           mx_weight_split(kind, I), fmt == SITU_MX_E2M1,
                                           static_cast<cudaStream_t>(stream)));
}

namespace {

// The MXFP8 gate_up GEMM (+ SiTU-GLU): bf16 h into h, or MXFP8 h into h_codes / h_sf.
cudaError_t run_mx_gate_up(const DeviceState* st, const void* x_codes, const void* x_scales,
                           const void* wgu_codes, const void* wgu_scales, void* h, void* h_codes,
                           void* h_sf, int64_t R, int64_t M, int64_t I, float beta,
                           float linear_beta, int32_t E, const int32_t* offsets,
                           const int32_t* tiles, const int32_t* units, bool fp4,
                           cudaStream_t cs, bool pair_units = false) {
  GemmShape g{};
  g.b_fp4 = fp4;
  g.pair_units = pair_units;
  g.a = x_codes;
  g.a_rows = R;
  g.b = wgu_codes;
  g.b_rows = static_cast<int64_t>(E) * 2 * I;
  g.K = M;
  g.num_groups = offsets ? E : 1;
  g.group_offsets = offsets;
  g.tile_offsets = tiles;
  g.unit_offsets = units;
  g.b_group_rows = 2 * I;
  g.b_up_offset = I;
  g.n_out = I;
  g.out = h;
  g.ldo = I;
  g.out_rows = R;
  g.sfa = x_scales;
  g.sfb = wgu_scales;
  g.h_codes = h_codes;
  g.h_sf = h_sf;
  return launch_mx_gemm_situ(g, make_situ_params(beta, linear_beta), caps_of(beta, linear_beta),
                             st->status, st->num_sms, cs);
}

cudaError_t run_mx_down(const DeviceState* st, const void* h_codes, const void* h_sf,
                        const void* wd_codes, const void* wd_scales, void* y, int64_t R,
                        int64_t M, int64_t I, int32_t E, const int32_t* offsets,
                        const int32_t* tiles, const int32_t* units, const int32_t* row_index,
                        bool fp4, cudaStream_t cs, bool pair_units = false) {
  GemmShape d{};
  d.b_fp4 = fp4;
  d.pair_units = pair_units;
  d.a = h_codes;
  d.a_rows = R;
  d.b = wd_codes;
  d.b_rows = static_cast<int64_t>(E) * M;
  d.K = I;
  d.num_groups = offsets ? E : 1;
  d.group_offsets = offsets;
  d.tile_offsets = tiles;
  d.unit_offsets = units;
  d.b_group_rows = M;
  d.n_out = M;
  d.out = y;
  d.ldo = M;
  d.out_rows = R;
  d.out_row_index = row_index;
  d.sfa = h_sf;
  d.sfb = wd_scales;
  return launch_mx_gemm_plain(d, st->status, st->num_sms, cs);
}

// Carving of the dense MXFP8 FFN workspace: x codes, x scales, h codes, h scales, and
// one int32 per 128-row m-tile (the one-launch FFN's h-ready counts).
struct MxFfnWs {
  size_t x_codes, x_sf, h_codes, h_sf, h_ready, total;
};
MxFfnWs mx_ffn_ws(int64_t R, int64_t M, int64_t I) {
  MxFfnWs w;
  w.x_codes = 0;
  w.x_sf = round_up(static_cast<size_t>(R) * M, 256);
  w.h_codes = w.x_sf + round_up(mx_act_scale_bytes(R, M), 256);
  w.h_sf = w.h_codes + round_up(static_cast<size_t>(R) * I, 256);
  w.h_ready = w.h_sf + round_up(mx_act_scale_bytes(R, I), 256);
  w.total = w.h_ready + round_up(static_cast<size_t>((R + 127) / 128) * 4, 256);
  return w;
}

}  // namespace

situ_status situ_ffn_gate_up_mxfp8(const void* x_codes, const void* x_scales,
                                   const void* wgu_codes, const void* wgu_scales, int weight_fmt,
                                   void* h, int64_t R, int64_t M, int64_t I, float beta,
                                   float linear_beta, void* stream) {
  if (R < 0 || M < 1 || I < 1 || !caps_ok(beta, linear_beta) || !mx_fmt_ok(weight_fmt))
    return SITU_ERR_ARG;
  if (!mx_shape_ok(M, I)) return SITU_ERR_UNSUPPORTED;
  if (R == 0) return SITU_OK;
  if (!x_codes || !x_scales || !wgu_codes || !wgu_scales || !h) return SITU_ERR_ARG;
  if (!aligned16(x_codes) || !aligned16(x_scales) || !aligned16(wgu_codes) ||
      !aligned16(wgu_scales) || !aligned16(h))
    return SITU_ERR_ALIGN;
  if (R >= (int64_t(1) << 31)) return SITU_ERR_UNSUPPORTED;
  const size_t hb = static_cast<size_t>(R) * I * 2;
  if (overlap(h, hb, x_codes, static_cast<size_t>(R) * M) ||
      overlap(h, hb, x_scales, mx_act_scale_bytes(R, M)) ||
      overlap(h, hb, wgu_codes, mx_weight_code_bytes(1, 2 * I, M, weight_fmt)) ||
      overlap(h, hb, wgu_scales, situ_mx_weight_scales_size(1, M, I, SITU_MX_GATE_UP)))
    return SITU_ERR_ALIAS;
  DeviceState* st = nullptr;
  situ_status s = device_state(&st);
  if (s != SITU_OK) return s;
  return finish(run_mx_gate_up(st, x_codes, x_scales, wgu_codes, wgu_scales, h, nullptr, nullptr,
                               R, M, I, beta, linear_beta, 1, nullptr, nullptr, nullptr,
                               weight_fmt == SITU_MX_E2M1, static_cast<cudaStream_t>(stream)));
}

size_t situ_ffn_mxfp8_workspace_size(int64_t R, int64_t M, int64_t I) {
  if (R < 0 || !mx_shape_ok(M, I)) return 0;
  return mx_ffn_ws(R, M, I).total;
}

situ_status situ_ffn_forward_mxfp8(const void* x, const void* wgu_codes, const void* wgu_scales,
                                   const void* wd_codes, const void* wd_scales, int weight_fmt,
                                   void* y, void* workspace, size_t workspace_bytes, int64_t R,
                                   int64_t M, int64_t I, float beta, float linear_beta,
                                   void* stream) {
  if (R < 0 || M < 1 || I < 1 || !caps_ok(beta, linear_beta) || !mx_fmt_ok(weight_fmt))
    return SITU_ERR_ARG;
  if (!mx_shape_ok(M, I)) return SITU_ERR_UNSUPPORTED;
  if (R == 0) return SITU_OK;
  if (!x || !wgu_codes || !wgu_scales || !wd_codes || !wd_scales || !y) return SITU_ERR_ARG;
  const void* ptrs[] = {x, wgu_codes, wgu_scales, wd_codes, wd_scales, y};
  for (const void* q : ptrs)
    if (!aligned16(q)) return SITU_ERR_ALIGN;
  if (R >= (int64_t(1) << 31)) return SITU_ERR_UNSUPPORTED;
  const MxFfnWs w = mx_ffn_ws(R, M, I);
  if (!workspace || workspace_bytes < w.total || reinterpret_cast<uintptr_t>(workspace) % 256)
    return SITU_ERR_WORKSPACE;
  const size_t xb = static_cast<size_t>(R) * M * 2;
  const void* ins[] = {x, wgu_codes, wgu_scales, wd_codes, wd_scales};
  const size_t inb[] = {xb, mx_weight_code_bytes(1, 2 * I, M, weight_fmt),
                        situ_mx_weight_scales_size(1, M, I, SITU_MX_GATE_UP),
                        mx_weight_code_bytes(1, M, I, weight_fmt),
                        situ_mx_weight_scales_size(1, M, I, SITU_MX_DOWN)};
  for (int i = 0; i < 5; ++i)
    if (overlap(y, xb, ins[i], inb[i]) || overlap(workspace, w.total, ins[i], inb[i]))
      return SITU_ERR_ALIAS;
  if (overlap(y, xb, workspace, w.total)) return SITU_ERR_ALIAS;
  DeviceState* st = nullptr;
  situ_status s = device_state(&st);
  if (s != SITU_OK) return s;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaError_t e = launch_mx_quantize_act(x, nullptr, 1, R, ws + w.x_codes, ws + w.x_sf,
                                         (R + 127) / 128, R, M, 0, nullptr, nullptr, st->status,
                                         cs);
  if (e != cudaSuccess) return cuda_fail(e);
  const bool fp4 = weight_fmt == SITU_MX_E2M1;
  if (g_ffn_single_launch.load(std::memory_order_relaxed)) {
    // Both projections in one persistent launch, as the bf16 forward.
    GemmShape g{};
    g.b_fp4 = fp4;
    g.a = ws + w.x_codes;
    g.a_rows = R;
    g.b = wgu_codes;
    g.b_rows = 2 * I;
    g.K = M;
    g.num_groups = 1;
    g.b_group_rows = 2 * I;
    g.b_up_offset = I;
    g.n_out = I;
    g.ldo = I;
    g.out_rows = R;
    g.sfa = ws + w.x_sf;
    g.sfb = wgu_scales;
    g.h_codes = ws + w.h_codes;
    g.h_sf = ws + w.h_sf;
    GemmShape d{};
    d.b_fp4 = fp4;
    d.a = ws + w.h_codes;
    d.a_rows = R;
    d.b = wd_codes;
    d.b_rows = M;
    d.K = I;
    d.num_groups = 1;
    d.b_group_rows = M;
    d.n_out = M;
    d.out = y;
    d.ldo = M;
    d.out_rows = R;
    d.sfa = ws + w.h_sf;
    d.sfb = wd_scales;
    e = launch_mx_ffn_fused(g, d, make_situ_params(beta, linear_beta), caps_of(beta, linear_beta),
                            reinterpret_cast<int32_t*>(ws + w.h_ready), st->status, st->num_sms,
                            cs);
    if (e == cudaSuccess) {
      t_ffn_path = SITU_FFN_PATH_FUSED;
      return SITU_OK;
    }
    (void)cudaGetLastError();  // a refused launch configuration: take the two launches
  }
  t_ffn_path = SITU_FFN_PATH_TWO_LAUNCHES;
  e = run_mx_gate_up(st, ws + w.x_codes, ws + w.x_sf, wgu_codes, wgu_scales, nullptr,
                     ws + w.h_codes, ws + w.h_sf, R, M, I, beta, linear_beta, 1, nullptr, nullptr,
                     nullptr, fp4, cs);
  if (e != cudaSuccess) return cuda_fail(e);
  return finish(run_mx_down(st, ws + w.h_codes, ws + w.h_sf, wd_codes, wd_scales, y, R, M, I, 1,
                            nullptr, nullptr, nullptr, nullptr, fp4, cs));
}

namespace {

// Carving of the grouped MXFP8 workspace: three prefixes, x codes (expert order),
// x scales, h codes, h scales.  Grouped m-tiles number at most ceil(R/128) + E.
struct MxMoeWs {
  size_t tiles, units_gu, units_dn, x_codes, x_sf, h_codes, h_sf, total;
};
MxMoeWs mx_moe_ws(int64_t R, int32_t E, int64_t M, int64_t I) {
  MxMoeWs w;
  const size_t pre = round_up(static_cast<size_t>(E + 1) * 4, 256);
  const int64_t tile_rows = ((R + 127) / 128 + E) * 128;
  w.tiles = 0;
  w.units_gu = pre;
  w.units_dn = 2 * pre;
  w.x_codes = 3 * pre;
  w.x_sf = w.x_codes + round_up(static_cast<size_t>(R) * M, 256);
  w.h_codes = w.x_sf + round_up(mx_act_scale_bytes(tile_rows, M), 256);
  w.h_sf = w.h_codes + round_up(static_cast<size_t>(R) * I, 256);
  w.total = w.h_sf + round_up(mx_act_scale_bytes(tile_rows, I), 256);
  return w;
}

}  // namespace

size_t situ_moe_mxfp8_workspace_size(int64_t R, int32_t E, int64_t M, int64_t I) {
  if (R < 0 || E < 1 || !mx_shape_ok(M, I)) return 0;
  return mx_moe_ws(R, E, M, I).total;
}

situ_status situ_moe_grouped_forward_mxfp8(const void* x, const int32_t* expert_offsets,
                                           const int32_t* token_index, const void* wgu_codes,
                                           const void* wgu_scales, const void* wd_codes,
                                           const void* wd_scales, int weight_fmt, void* y,
                                           void* workspace, size_t workspace_bytes, int64_t T,
                                           int32_t k_eff, int32_t E, int64_t M, int64_t I,
                                           float beta, float linear_beta, void* stream) {
  if (T < 0 || k_eff < 1 || E < 1 || E > 65536 || M < 1 || I < 1 || !caps_ok(beta, linear_beta) ||
      !mx_fmt_ok(weight_fmt))
    return SITU_ERR_ARG;
  if (!mx_shape_ok(M, I)) return SITU_ERR_UNSUPPORTED;
  const int64_t R = T * k_eff;
  if (R == 0) return SITU_OK;
  if (!x || !expert_offsets || !token_index || !wgu_codes || !wgu_scales || !wd_codes ||
      !wd_scales || !y)
    return SITU_ERR_ARG;
  if (R >= (int64_t(1) << 31) || static_cast<int64_t>(E) * 2 * I >= (int64_t(1) << 31) ||
      static_cast<int64_t>(E) * M >= (int64_t(1) << 31))
    return SITU_ERR_UNSUPPORTED;
  const void* ptrs[] = {x, wgu_codes, wgu_scales, wd_codes, wd_scales, y};
  for (const void* q : ptrs)
    if (!aligned16(q)) return SITU_ERR_ALIGN;
  const MxMoeWs w = mx_moe_ws(R, E, M, I);
  if (!workspace || workspace_bytes < w.total || reinterpret_cast<uintptr_t>(workspace) % 256)
    return SITU_ERR_WORKSPACE;
  const size_t x_b = static_cast<size_t>(T) * M * 2, y_b = static_cast<size_t>(R) * M * 2;
  const void* ins[] = {x, expert_offsets, token_index, wgu_codes, wgu_scales, wd_codes, wd_scales};
  const size_t in_b[] = {x_b, static_cast<size_t>(E + 1) * 4, static_cast<size_t>(R) * 4,
                         mx_weight_code_bytes(E, 2 * I, M, weight_fmt),
                         situ_mx_weight_scales_size(E, M, I, SITU_MX_GATE_UP),
                         mx_weight_code_bytes(E, M, I, weight_fmt),
                         situ_mx_weight_scales_size(E, M, I, SITU_MX_DOWN)};
  for (int i = 0; i < 7; ++i)
    if (overlap(y, y_b, ins[i], in_b[i]) || overlap(workspace, w.total, ins[i], in_b[i]))
      return SITU_ERR_ALIAS;
  if (overlap(y, y_b, workspace, w.total)) return SITU_ERR_ALIAS;
  DeviceState* st = nullptr;
  situ_status s = device_state(&st);
  if (s != SITU_OK) return s;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* tiles = reinterpret_cast<int32_t*>(ws + w.tiles);
  int32_t* units_gu = reinterpret_cast<int32_t*>(ws + w.units_gu);
  int32_t* units_dn = reinterpret_cast<int32_t*>(ws + w.units_dn);
  // Two-CTA MMAs when the experts average at least 512 rows (as for bf16).
  const bool two_cta = R >= 512 * static_cast<int64_t>(E) && gemm_two_cta_available();
  cudaError_t e = launch_group_tiles(expert_offsets, E, R,
                                     static_cast<int32_t>((I + kMxSituCols - 1) / kMxSituCols),
                                     static_cast<int32_t>((M + kMxPlainCols - 1) / kMxPlainCols),
                                     tiles, units_gu, units_dn, st->status, cs, two_cta);
  if (e != cudaSuccess) return cuda_fail(e);
  // Gather x into expert order and quantize it, scales tiled by the experts' m-tiles.
  e = launch_mx_quantize_act(x, token_index, k_eff, T, ws + w.x_codes, ws + w.x_sf,
                             (R + 127) / 128 + E, R, M, E, expert_offsets, tiles, st->status, cs);
  if (e != cudaSuccess) return cuda_fail(e);
  const bool fp4 = weight_fmt == SITU_MX_E2M1;
  e = run_mx_gate_up(st, ws + w.x_codes, ws + w.x_sf, wgu_codes, wgu_scales, nullptr,
                     ws + w.h_codes, ws + w.h_sf, R, M, I, beta, linear_beta, E, expert_offsets,
                     tiles, units_gu, fp4, cs, two_cta);
  if (e != cudaSuccess) return cuda_fail(e);
  return finish(run_mx_down(st, ws + w.h_codes, ws + w.h_sf, wd_codes, wd_scales, y, R, M, I, E,
                            expert_offsets, tiles, units_dn, token_index, fp4, cs, two_cta));
}

situ_status situ_moe_combine(const void* y, const float* weights, void* out, int64_t T,
                             int32_t k_eff, int64_t M, situ_dtype dt, void* stream) {
  if (!dtype_ok(dt) || T < 0 || k_eff < 1 || M < 1) return SITU_ERR_ARG;
  if (T == 0) return SITU_OK;
  if (!y || !weights || !out) return SITU_ERR_ARG;
  const size_t esz = dtype_size(dt);
  const size_t out_b = static_cast<size_t>(T) * M * esz;
  if (overlap(out, out_b, y, static_cast<size_t>(T) * k_eff * M * esz) ||
      overlap(out, out_b, weights, static_cast<size_t>(T) * k_eff * 4))
    return SITU_ERR_ALIAS;
  if (reinterpret_cast<uintptr_t>(y) % esz || reinterpret_cast<uintptr_t>(out) % esz ||
      reinterpret_cast<uintptr_t>(weights) % 4)
    return SITU_ERR_ALIGN;
  DeviceState* st = nullptr;
  situ_status s = device_state(&st);
  if (s != SITU_OK) return s;
  return finish(launch_combine(y, weights, out, T, k_eff, M, dt, st->num_sms,
                               static_cast<cudaStream_t>(stream)));
}

uint64_t situ_set_wait_limit_ns(uint64_t ns) {
  return g_wait_limit_ns.exchange(ns == 0 ? kDefaultWaitLimitNs : ns);
}

situ_status situ_selftest_group_maps(const int32_t* k_offsets, int32_t groups, int64_t rows,
                                     int64_t cols, int32_t* mismatches, void* stream) {
  if (!k_offsets || !mismatches || groups < 1 || groups > (1 << 16) || rows < 1 ||
      rows >= (int64_t(1) << 31) || cols < 8 || cols % 8 || cols >= (int64_t(1) << 30))
    return SITU_ERR_ARG;
  for (int32_t g = 0; g < groups; ++g)
    if (k_offsets[g] < 0 || k_offsets[g + 1] < k_offsets[g] || k_offsets[g + 1] > rows)
      return SITU_ERR_ARG;
  DeviceState* st = nullptr;
  situ_status s = device_state(&st);
  if (s != SITU_OK) return s;
  const cudaError_t e = group_maps_selftest(k_offsets, groups, rows, cols, mismatches,
                                            static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SITU_OK : report_cuda_error(e);
}

situ_status situ_selftest_bounded_wait(uint32_t limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000) return SITU_ERR_ARG;
  DeviceState* st = nullptr;
  situ_status s = device_state(&st);
  if (s != SITU_OK) return s;
  return finish(launch_bounded_wait_selftest(static_cast<uint64_t>(limit_us) * 1000, st->status,
                                             static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Internal accessors for other translation units of the library.
// ---------------------------------------------------------------------------
namespace situ {

situ_status current_device_context(int* num_sms, uint32_t** status) {
  DeviceState* st = nullptr;
  situ_status s = device_state(&st);
  if (s != SITU_OK) return s;
  *num_sms = st->num_sms;
  *status = st->status;
  return SITU_OK;
}

situ_status report_cuda_error(cudaError_t e) { return cuda_fail(e); }

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

situ_status ffn_arg_checks(situ_dtype dt, int64_t R, int64_t M, int64_t I, float beta,
                           float linear_beta) {
  return ffn_common_checks(dt, R, M, I, beta, linear_beta);
}

situ_status ffn_bf16_operand_checks(const void* x, const void* W_gate_up, const void* W_down,
                                    int64_t M, int64_t I) {
  return bf16_gemm_checks(x, W_gate_up, W_down, M, I);
}

}  // namespace situ
