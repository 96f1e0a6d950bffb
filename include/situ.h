/*
 * situ.h -- C ABI of libsitu, the GB300 (sm_103a) SiTU-GLU expert feed-forward.
 *
 * SiTU-GLU (Sigmoid-Tanh-Unit GLU) is the activation of every feed-forward
 * network of Kimi K3.  For a gate projection g and an up projection u,
 *
 *     h = [beta1 * tanh(g / beta1) * sigmoid(g)] * [beta2 * tanh(u / beta2)],
 *
 * with beta1 = 4 and beta2 = 25 in Kimi K3, so that |h| <= beta1 * beta2 = 100.
 * Sources, by page title and section:
 *   - "SiTU-GLU" problem page (ai-engineer-exhaustive.pages.dev): "Theory",
 *     "Implementation order", "Requirements", "Constraints", "Starter Code";
 *   - "Kimi K3 - Bound the up branch" (atlas.klimoza.dev): the up-branch formula
 *     and the expert MLP / activation-module code excerpts;
 *   - "DenseFFN and SituGLU - Docs - Kimi K3 from Scratch": the packed
 *     gate_up_proj (M -> 2I) and down_proj (I -> M), FP32 activation math, cast
 *     back to the input dtype;
 *   - "SiTU-GLU" architecture chapter (mkdocs.reaper.mx): the boxed equation, the
 *     beta values and the bound.
 *
 * Conventions shared by every call:
 *   - Every pointer named as device memory must be a CUDA device pointer on the
 *     current device.  The caller allocates and owns every buffer; the library
 *     keeps only a per-device status word.
 *   - Every call is asynchronous on `stream` (a cudaStream_t, NULL for the legacy
 *     default stream).  A non-OK return means nothing was launched.  Device-side
 *     failures (a bounded wait that gave up, a route index out of range) are
 *     recorded in the per-device status word: read them with
 *     situ_device_status() after synchronising the stream.
 *   - Inputs are never written ("Do not mutate any input tensor", problem page,
 *     "Requirements").  An output that overlaps an input returns SITU_ERR_ALIAS.
 *   - Each cap (beta, linear_beta) is either finite in (0, 2^20] ("Both cap
 *     values are positive", problem page, "Constraints") or +infinity, which
 *     leaves that branch uncapped: beta tanh(x / beta) -> x as beta -> infinity.
 *     An infinite up cap is the activation module's linear_beta = None ("Kimi K3 -
 *     Bound the up branch", SituAndMul excerpt); both caps infinite is SwiGLU
 *     ("SiTU-GLU" chapter, "Les proprietes").  Anything else returns SITU_ERR_ARG.
 *     The bound |h| <= beta * linear_beta holds when both caps are finite.  With
 *     the up branch uncapped, outputs are within 1 bf16 ulp for |u| <= 2^50.
 *   - The output dtype equals the input dtype ("Preserve the floating-point dtype",
 *     problem page, "Requirements").  Activation math is FP32 in every path.
 *   - Matrices are row-major.  Weights use the [out, in] orientation of a
 *     bias-free linear layer: W_gate_up is [2I, M] with rows 0..I-1 the gate
 *     projection and rows I..2I-1 the up projection; W_down is [M, I].
 *   - Zero rows is a valid no-op.
 */
#ifndef SITU_H
#define SITU_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SITU_ABI_VERSION 2

typedef enum {
  SITU_BF16 = 0, /* bfloat16 storage, FP32 accumulation and activation math */
  SITU_F32 = 1   /* float32 storage (small-shape SIMT path) */
} situ_dtype;

typedef enum {
  SITU_OK = 0,
  SITU_ERR_ARG = 1,         /* bad size, NULL pointer, bad cap, bad dtype */
  SITU_ERR_ALIGN = 2,       /* a pointer lacks the alignment the kernel requires */
  SITU_ERR_ALIAS = 3,       /* an output overlaps an input */
  SITU_ERR_CUDA = 4,        /* a CUDA runtime or driver call failed */
  SITU_ERR_TIMEOUT = 5,     /* a bounded device-side wait gave up (device status) */
  SITU_ERR_UNSUPPORTED = 6, /* shape/dtype combination the kernels do not cover */
  SITU_ERR_INDEX = 7,       /* expert id, route index or expert offsets invalid */
  SITU_ERR_WORKSPACE = 8    /* workspace NULL, too small or misaligned */
} situ_status;

/* ABI version of the loaded library (SITU_ABI_VERSION). */
int situ_abi_version(void);

/* Static, NUL-terminated name of a status code. */
const char* situ_status_string(situ_status s);

/* Text of the last CUDA error seen by this host thread inside the library
 * ("" if none).  Static storage per thread; valid until the next call. */
const char* situ_last_cuda_error(void);

/* Which path this host thread's last successful bf16 situ_ffn_forward or
 * situ_ffn_forward_mxfp8 took:
 * SITU_FFN_PATH_FUSED (one persistent launch for both projections),
 * SITU_FFN_PATH_TWO_LAUNCHES (the device refused that grid as co-resident, so the
 * projections ran as two launches), or 0 before the first such call.  Both paths
 * produce the same bits. */
#define SITU_FFN_PATH_FUSED 1
#define SITU_FFN_PATH_TWO_LAUNCHES 2
int situ_ffn_last_path(void);

/* Process-wide switch for that single launch (on by default); returns the previous
 * setting.  With it off, bf16 situ_ffn_forward and situ_ffn_forward_mxfp8 always run
 * the two launches.  The
 * single launch is a cooperative launch of thread-block clusters, which tools that
 * intercept and replay launches (kernel profilers) may not reproduce faithfully:
 * turn it off under such a tool. */
int situ_ffn_set_single_launch(int enable);

/* Process-wide switch (on by default; returns the previous setting) for the form of
 * situ_moe_grouped_backward's per-expert weight gradients: on, two-CTA MMAs reading each
 * expert through tensor maps that end at its last row; off, one CTA per tile with the
 * rows past an expert's end zeroed in shared memory (the form used where two-CTA
 * clusters cannot be launched).  Both produce the same bits. */
int situ_moe_set_kgrouped_two_cta(int enable);

/* Device-side status of the current device: SITU_OK, or the first failure a
 * kernel recorded since the last clear (SITU_ERR_TIMEOUT, SITU_ERR_INDEX).
 * Synchronous: call it after synchronising the streams the kernels ran on.
 * clear != 0 resets the word to SITU_OK. */
situ_status situ_device_status(int clear);

/* -------------------------------------------------------------------------
 * situ_glu_act -- standalone SiTU-GLU activation.
 *
 * Operation (problem page "Implementation order"; docs page "SiTU-GLU: one split,
 * two softly bounded branches"; bound page, SituAndMul excerpt): for every row r
 * and column j < I, with g = gate_up[r, j] and u = gate_up[r, I + j],
 *   out[r, j] = dtype( beta * tanh(g / beta) * sigmoid(g)
 *                      * linear_beta * tanh(u / linear_beta) ).
 *
 *   gate_up  device, [rows, 2I] of `dt`, row-major, read only.
 *   out      device, [rows, I] of `dt`, row-major, written; must not overlap
 *            gate_up.
 *   rows     >= 0; leading dimensions flattened by the caller.
 *   I        >= 1 (half the width of gate_up).
 *   beta, linear_beta   gate and up caps (see the conventions above).
 * Rows whose start is 16-byte aligned (bf16: I % 8 == 0, f32: I % 4 == 0, and
 * 16-byte aligned base pointers) take the 128-bit vector path; other shapes take
 * a scalar path, never an error.  |out| <= beta * linear_beta holds exactly.
 * Errors: SITU_ERR_ARG, SITU_ERR_ALIAS, SITU_ERR_CUDA.
 * ------------------------------------------------------------------------- */
situ_status situ_glu_act(const void* gate_up, void* out, int64_t rows, int64_t I,
                         float beta, float linear_beta, situ_dtype dt, void* stream);

/* -------------------------------------------------------------------------
 * situ_ffn_forward -- dense SiTU-GLU feed-forward (one expert, or a dense layer).
 *
 * Operation (docs page "Two linear maps and a guarded compiled branch": packed
 * gate_up_proj M -> 2I, activation, down_proj I -> M; bound page,
 * KimiBlockSparseMLP forward):
 *   gu = x W_gate_up^T            (FP32 accumulation, kept on chip for bf16)
 *   h  = dtype(SiTU-GLU(gu[:, :I], gu[:, I:]))   (FP32 math, as situ_glu_act)
 *   y  = dtype(h W_down^T)        (FP32 accumulation)
 * For bf16 the gate_up product and the activation run in one tcgen05 GEMM whose
 * epilogue applies SiTU-GLU to the FP32 accumulators, so the [R, 2I] tensor never
 * reaches memory; h ([R, I], bf16) is written to the workspace and read back by the
 * down GEMM.  Both GEMMs run in one persistent launch: a down tile starts once every
 * gate_up tile of its 128 rows has stored its h (two launches when the grid cannot be
 * made co-resident).
 *
 *   x          device, [R, M] of `dt`.
 *   W_gate_up  device, [2I, M] of `dt`.
 *   W_down     device, [M, I] of `dt`.
 *   y          device, [R, M] of `dt`, written; must not overlap any input or the
 *              workspace.
 *   workspace  device, >= situ_ffn_workspace_size(R, M, I, dt) bytes, 256-byte
 *              aligned; its contents are overwritten: h [R, I] first (rounded up to
 *              256 bytes) then, for bf16, one int32 per 128-row tile of h-ready counts.
 *   R >= 0, M >= 1, I >= 1.  bf16 requires M % 8 == 0, I % 8 == 0 and 16-byte
 *   aligned x, W_gate_up, W_down and y (tensor-memory-access rules); otherwise
 *   SITU_ERR_UNSUPPORTED / SITU_ERR_ALIGN.  f32 accepts any shape.
 * Errors: SITU_ERR_ARG, SITU_ERR_ALIGN, SITU_ERR_ALIAS, SITU_ERR_WORKSPACE,
 *         SITU_ERR_UNSUPPORTED, SITU_ERR_CUDA; SITU_ERR_TIMEOUT on the device.
 * ------------------------------------------------------------------------- */
size_t situ_ffn_workspace_size(int64_t R, int64_t M, int64_t I, situ_dtype dt);

situ_status situ_ffn_forward(const void* x, const void* W_gate_up, const void* W_down,
                             void* y, void* workspace, size_t workspace_bytes,
                             int64_t R, int64_t M, int64_t I, float beta,
                             float linear_beta, situ_dtype dt, void* stream);

/* -------------------------------------------------------------------------
 * situ_ffn_gate_up -- the first half of situ_ffn_forward on its own:
 *   h = dtype(SiTU-GLU(x W_gate_up^T))          h: device, [R, I] of `dt`
 * (docs page "Two linear maps": packed gate_up_proj followed by the activation;
 * for bf16 one tcgen05 GEMM with the activation in its epilogue).  Arguments,
 * shape and alignment rules as situ_ffn_forward; h must not overlap the inputs.
 * Errors: SITU_ERR_ARG, SITU_ERR_ALIGN, SITU_ERR_ALIAS, SITU_ERR_UNSUPPORTED,
 *         SITU_ERR_CUDA; SITU_ERR_TIMEOUT on the device.
 * ------------------------------------------------------------------------- */
situ_status situ_ffn_gate_up(const void* x, const void* W_gate_up, void* h, int64_t R,
                             int64_t M, int64_t I, float beta, float linear_beta,
                             situ_dtype dt, void* stream);

/* -------------------------------------------------------------------------
 * situ_ffn_down -- the second half of situ_ffn_forward on its own:
 *   y = dtype(h W_down^T)                        y: device, [R, M] of `dt`
 * (docs page "Two linear maps": down_proj I -> M, no bias).  h is [R, I], W_down
 * [M, I]; bf16 needs M % 8 == 0, I % 8 == 0 and 16-byte aligned pointers.
 * Errors: SITU_ERR_ARG, SITU_ERR_ALIGN, SITU_ERR_ALIAS, SITU_ERR_UNSUPPORTED,
 *         SITU_ERR_CUDA; SITU_ERR_TIMEOUT on the device.
 * ------------------------------------------------------------------------- */
situ_status situ_ffn_down(const void* h, const void* W_down, void* y, int64_t R, int64_t M,
                          int64_t I, situ_dtype dt, void* stream);

/* -------------------------------------------------------------------------
 * situ_ffn_forward_train / situ_ffn_backward -- training pair of the dense FFN.
 *
 * The forward also keeps what the backward needs: the pre-activation pair
 * gu = x W_gate_up^T (bf16, [R, 2I]: gate columns then up columns) and the
 * activation h ([R, I]); y as situ_ffn_forward.
 *
 * The backward, for an upstream gradient dy [R, M], computes (FP32 accumulation,
 * bf16 outputs), by differentiating the steps of "Implementation order"
 * (problem page) -- the soft caps keep the gradient nonzero where a hard clamp
 * would not ("SiTU-GLU" chapter, "Pourquoi un plafond doux"):
 *   dh   = dy W_down                                   [R, I]
 *   dg   = dh * b(u) * a'(g),  a'(g) = sech^2(g/b1) sigmoid(g)
 *                                    + b1 tanh(g/b1) sigmoid(g) sigmoid(-g)
 *   du   = dh * a(g) * sech^2(u/b2)          (dgu = [dg, du], [R, 2I], bf16)
 *   dx   = dgu W_gate_up                              [R, M]
 *   dW_down    = dy^T h                                [M, I]
 *   dW_gate_up = dgu^T x                               [2I, M]
 * evaluated at the saved bf16 gu.  Caps as everywhere (+inf = uncapped).
 * The activation derivative runs in the epilogue of the dy W_down GEMM (dgu
 * lives in the workspace); every GEMM reads its operands in their stored layout
 * (the weights and the row-contracted operands as MN-major tiles), so nothing is
 * transposed.
 *
 *   all tensors device, bf16, row-major; gu and h as written by
 *   situ_ffn_forward_train.  dx, dW_gate_up, dW_down are written and must not
 *   overlap the inputs or the workspace.
 *   workspace  >= situ_ffn_backward_workspace_size(R, M, I, dt) bytes, 256-byte
 *              aligned.
 *   bf16 only; M % 8 == 0, I % 8 == 0, R >= 1, 16-byte aligned pointers.
 * Errors: SITU_ERR_ARG, SITU_ERR_ALIGN, SITU_ERR_ALIAS, SITU_ERR_WORKSPACE,
 *         SITU_ERR_UNSUPPORTED, SITU_ERR_CUDA; SITU_ERR_TIMEOUT on the device.
 * ------------------------------------------------------------------------- */
situ_status situ_ffn_forward_train(const void* x, const void* W_gate_up, const void* W_down,
                                   void* y, void* gu, void* h, int64_t R, int64_t M,
                                   int64_t I, float beta, float linear_beta, situ_dtype dt,
                                   void* stream);

size_t situ_ffn_backward_workspace_size(int64_t R, int64_t M, int64_t I, situ_dtype dt);

situ_status situ_ffn_backward(const void* x, const void* W_gate_up, const void* W_down,
                              const void* gu, const void* h, const void* dy, void* dx,
                              void* dW_gate_up, void* dW_down, void* workspace,
                              size_t workspace_bytes, int64_t R, int64_t M, int64_t I,
                              float beta, float linear_beta, situ_dtype dt, void* stream);

/* -------------------------------------------------------------------------
 * situ_ffn_forward_host -- situ_ffn_forward with x and y in host memory.
 *
 * Same operation as situ_ffn_forward (docs page "Two linear maps"), for callers
 * whose activations live on the host.  The rows are processed in chunks of
 * `chunk_rows`: while chunk c runs on the GPU, chunk c+1 is copied in and chunk
 * c-1 copied out on two library-owned copy streams, ordered with events, so the
 * host<->device traffic overlaps the GEMMs.  The call returns once everything is
 * enqueued; `stream` completes only after the last result row has reached y_host.
 *
 *   x_host     host, [R, M] of `dt`, read only.  Use page-locked (pinned) memory:
 *              pageable memory works but its copies do not overlap.
 *   y_host     host, [R, M] of `dt`, written.
 *   W_gate_up, W_down   device, as situ_ffn_forward.
 *   workspace  device, >= situ_ffn_host_workspace_size(R, M, I, dt, chunk_rows)
 *              bytes, 256-byte aligned (two x chunks, two y chunks, one h chunk).
 *   chunk_rows rows per chunk, >= 1; 0 picks 4096.
 * The copy streams and events are created once per device on first use.
 * Errors: those of situ_ffn_forward.
 * ------------------------------------------------------------------------- */
size_t situ_ffn_host_workspace_size(int64_t R, int64_t M, int64_t I, situ_dtype dt,
                                    int64_t chunk_rows);

situ_status situ_ffn_forward_host(const void* x_host, const void* W_gate_up,
                                  const void* W_down, void* y_host, void* workspace,
                                  size_t workspace_bytes, int64_t R, int64_t M, int64_t I,
                                  int64_t chunk_rows, float beta, float linear_beta,
                                  situ_dtype dt, void* stream);

/* -------------------------------------------------------------------------
 * situ_ffn_forward_noalloc -- situ_ffn_forward for callers that cannot allocate
 * device memory.  The pages have no counterpart: this is a library service.
 *
 * Some callers have no way to hand the library a workspace: a plugin whose
 * enqueue hook runs inside another engine's execution phase, where every buffer
 * was planned before execution began; a latency-bound serving loop that must not
 * call cudaMalloc (it can synchronise the whole device); code with no allocator
 * of its own.  For them this call keeps the intermediate h in a scratch array
 * built into the library: a file-scope device array of SITU_NOALLOC_SCRATCH_BYTES
 * bytes that every GPU which loads libsitu holds until the process exits.  The
 * call itself allocates nothing: no cudaMalloc, no cudaFree, no allocating
 * library routine.
 *
 *   x, W_gate_up, W_down, y, R, M, I, beta, linear_beta, dt, stream: exactly as
 *   situ_ffn_forward (same shapes, alignment rules and result).
 *   The caller still passes (and owns) every input and output.
 *   Limit: R * I * sizeof(dt) <= SITU_NOALLOC_SCRATCH_BYTES (at I = 3072 and bf16,
 *   up to 2730 rows); larger calls return SITU_ERR_WORKSPACE and launch nothing.
 *
 * Set-up: the first call on a device, with that device current, looks up the
 * scratch array's device address once (cudaGetSymbolAddress) and caches it; make
 * that first call before any stream capture on the device.
 * Sharing: every call on a device uses the same scratch array, which keeps the
 * previous call's h.  Nothing in it needs to start at zero (each call writes every
 * h element it reads), but two calls whose kernels overlap on the GPU (different
 * streams without ordering) race on it: order them on one stream or with events.
 * Errors: those of situ_ffn_forward, with SITU_ERR_WORKSPACE for a size above
 * the limit.
 * ------------------------------------------------------------------------- */
#define SITU_NOALLOC_SCRATCH_BYTES (16u << 20) /* 16 MiB */

situ_status situ_ffn_forward_noalloc(const void* x, const void* W_gate_up, const void* W_down,
                                     void* y, int64_t R, int64_t M, int64_t I, float beta,
                                     float linear_beta, situ_dtype dt, void* stream);

/* -------------------------------------------------------------------------
 * situ_moe_build_index -- expert index of a routed batch.
 *
 * Operation: a stable counting sort of the n_routes = T * k_eff flat routes
 * (route t*k_eff + s is slot s of token t) by expert id.  After the call,
 * expert_offsets[e] .. expert_offsets[e+1]-1 are the positions in token_index of
 * expert e's routes, listed in ascending flat order.  The pages call the expert
 * FFN on a varying number of expert-token rows (docs page, "Two linear maps and
 * a guarded compiled branch"); this builds those row groups.
 *
 *   expert_ids      device, [n_routes] int32, each in [0, E).
 *   expert_offsets  device, [E + 1] int32, written.
 *   token_index     device, [n_routes] int32, written.
 *   workspace       device, >= situ_moe_index_workspace_size(n_routes, E) bytes.
 *   0 <= n_routes < 2^31, 1 <= E <= 16384.
 * An id outside [0, E) records SITU_ERR_INDEX in the device status and that route
 * is dropped (expert_offsets[E] is then < n_routes).
 * Errors: SITU_ERR_ARG, SITU_ERR_ALIAS, SITU_ERR_WORKSPACE, SITU_ERR_CUDA.
 * ------------------------------------------------------------------------- */
size_t situ_moe_index_workspace_size(int64_t n_routes, int32_t E);

situ_status situ_moe_build_index(const int32_t* expert_ids, int32_t* expert_offsets,
                                 int32_t* token_index, void* workspace,
                                 size_t workspace_bytes, int64_t n_routes, int32_t E,
                                 void* stream);

/* -------------------------------------------------------------------------
 * situ_moe_grouped_forward -- SiTU-GLU experts over variable row groups.
 *
 * Operation: for every expert e and every position r in
 * [expert_offsets[e], expert_offsets[e+1]), with flat = token_index[r] and token
 * t = flat / k_eff,
 *   y[flat, :] = SiTU-GLU FFN of expert e applied to x[t, :]
 * (the dense operation of situ_ffn_forward with expert e's weights).  Each routed
 * and shared expert of Kimi K3 is such an FFN ("SiTU-GLU" chapter, "Ou SiTU-GLU
 * est utilise"; bound page, "Direct evidence": each routed expert is its own
 * gated MLP).  There are no combine weights: the output has one row per
 * (token, slot), shape [T, k_eff, M].  Shared experts are extra experts whose
 * groups hold every token.
 *
 *   x               device, [T, M] of `dt` (bf16 only).
 *   expert_offsets  device, [E + 1] int32: offsets[0] = 0, non-decreasing,
 *                   offsets[E] = R = T * k_eff.
 *   token_index     device, [R] int32, a permutation of 0..R-1 (as written by
 *                   situ_moe_build_index).
 *   W_gate_up       device, [E, 2I, M] of `dt`: the experts' packed gate_up
 *                   weights stacked in one allocation.
 *   W_down          device, [E, M, I] of `dt`, stacked likewise.
 *   y               device, [T * k_eff, M] of `dt`; every row listed in
 *                   token_index is written.
 *   workspace       device, >= situ_moe_workspace_size(T * k_eff, E, M, I, dt)
 *                   bytes, 256-byte aligned.
 *   M % 8 == 0, I % 8 == 0, 16-byte aligned pointers.
 * Offsets that are not monotone or do not end at R record SITU_ERR_INDEX in the
 * device status and the call writes nothing.
 * Errors: SITU_ERR_ARG, SITU_ERR_ALIGN, SITU_ERR_ALIAS, SITU_ERR_WORKSPACE,
 *         SITU_ERR_UNSUPPORTED, SITU_ERR_CUDA; SITU_ERR_TIMEOUT / SITU_ERR_INDEX
 *         on the device.
 * ------------------------------------------------------------------------- */
size_t situ_moe_workspace_size(int64_t R, int32_t E, int64_t M, int64_t I, situ_dtype dt);

situ_status situ_moe_grouped_forward(const void* x, const int32_t* expert_offsets,
                                     const int32_t* token_index, const void* W_gate_up,
                                     const void* W_down, void* y, void* workspace,
                                     size_t workspace_bytes, int64_t T, int32_t k_eff,
                                     int32_t E, int64_t M, int64_t I, float beta,
                                     float linear_beta, situ_dtype dt, void* stream);

/* -------------------------------------------------------------------------
 * situ_moe_grouped_forward_combined -- the routed layer output in one pass:
 *   out[t, :] = dtype( sum over slots s of weights[t, s] * FFN_{e(t,s)}(x[t, :]) )
 * i.e. situ_moe_grouped_forward followed by situ_moe_combine, with the combine fused
 * into the down projection's epilogue as a scatter-add: each (token, slot) row is
 * multiplied by its weight and added into an FP32 [T, M] accumulator with atomic
 * vector adds, then cast to dtype.  The per-route rows are never written, and they
 * are added unrounded.  The order of the additions depends on scheduling, so the
 * result can differ from run to run in the last bits (situ_moe_combine is the
 * deterministic path).  Each routed and shared expert of Kimi K3 runs on its tokens
 * ("SiTU-GLU" chapter, "Ou SiTU-GLU est utilise"), and the layer output is their
 * router-weighted sum.
 *
 *   x, expert_offsets, token_index, W_gate_up, W_down, T, k_eff, E, M, I, caps, dt:
 *               as situ_moe_grouped_forward (bf16 only).
 *   weights     device, [T, k_eff] float32.
 *   out         device, [T, M] bf16, written.
 *   workspace   device, >= situ_moe_combined_workspace_size(T, k_eff, E, M, I, dt)
 *               bytes, 256-byte aligned.
 * Errors: those of situ_moe_grouped_forward.
 * ------------------------------------------------------------------------- */
size_t situ_moe_combined_workspace_size(int64_t T, int32_t k_eff, int32_t E, int64_t M,
                                        int64_t I, situ_dtype dt);

situ_status situ_moe_grouped_forward_combined(const void* x, const int32_t* expert_offsets,
                                              const int32_t* token_index, const void* W_gate_up,
                                              const void* W_down, const float* weights,
                                              void* out, void* workspace, size_t workspace_bytes,
                                              int64_t T, int32_t k_eff, int32_t E, int64_t M,
                                              int64_t I, float beta, float linear_beta,
                                              situ_dtype dt, void* stream);

/* -------------------------------------------------------------------------
 * situ_moe_grouped_forward_train / situ_moe_grouped_backward -- training step of
 * the grouped experts.
 *
 * The forward is situ_moe_grouped_forward (same arguments, same y) that also
 * keeps, in expert order (row r belongs to route token_index[r]), what the
 * backward needs: the pre-activation pair gu [R, 2I] (gate columns then up
 * columns, bf16) and the activation h [R, I], R = T * k_eff.
 *
 * The backward takes dy [T, k_eff, M], the gradient of the per-route outputs y
 * (apply the combine weights to dy first: the combine is linear), and computes,
 * every route (t, s) of expert e being one row of expert e's dense FFN on x[t]
 * (as situ_ffn_backward, whose derivative it uses: "SiTU-GLU" chapter, "Pourquoi
 * un plafond doux"; docs page, "Two linear maps and a guarded compiled branch"):
 *   dx[t]          = sum over the token's slots s of d(g, u)[t, s] W_gate_up[e]
 *   dW_gate_up[e]  = sum over expert e's routes of d(g, u)^T x[t]     [2I, M]
 *   dW_down[e]     = sum over expert e's routes of dy[t, s]^T h       [M, I]
 * FP32 accumulation, bf16 results; an expert without routes gets zero weight
 * gradients.  The per-expert weight gradients contract over each expert's own
 * rows; the per-route dx rows are summed over slots in FP32, slot order
 * (deterministic, no atomics).
 *
 *   x, expert_offsets, token_index, W_gate_up, W_down, T, k_eff, E, M, I, caps:
 *               as situ_moe_grouped_forward.
 *   gu, h       device, as written by situ_moe_grouped_forward_train with the same
 *               expert_offsets and token_index.
 *   dy          device, [T, k_eff, M] bf16.
 *   dx          device, [T, M] bf16, written.
 *   dW_gate_up  device, [E, 2I, M] bf16, written;  dW_down  [E, M, I] bf16, written.
 *   workspace   forward: >= situ_moe_workspace_size(R, E, M, I, dt) bytes;
 *               backward: >= situ_moe_backward_workspace_size(R, E, M, I, dt) bytes;
 *               256-byte aligned.  Outputs must not overlap inputs or workspace.
 * T = 0: the backward zeroes dW_gate_up and dW_down.  Invalid offsets record
 * SITU_ERR_INDEX in the device status and the GEMMs write nothing.
 * Errors: those of situ_moe_grouped_forward.
 * ------------------------------------------------------------------------- */
situ_status situ_moe_grouped_forward_train(const void* x, const int32_t* expert_offsets,
                                           const int32_t* token_index, const void* W_gate_up,
                                           const void* W_down, void* y, void* gu, void* h,
                                           void* workspace, size_t workspace_bytes, int64_t T,
                                           int32_t k_eff, int32_t E, int64_t M, int64_t I,
                                           float beta, float linear_beta, situ_dtype dt,
                                           void* stream);

size_t situ_moe_backward_workspace_size(int64_t R, int32_t E, int64_t M, int64_t I,
                                        situ_dtype dt);

situ_status situ_moe_grouped_backward(const void* x, const int32_t* expert_offsets,
                                      const int32_t* token_index, const void* W_gate_up,
                                      const void* W_down, const void* gu, const void* h,
                                      const void* dy, void* dx, void* dW_gate_up, void* dW_down,
                                      void* workspace, size_t workspace_bytes, int64_t T,
                                      int32_t k_eff, int32_t E, int64_t M, int64_t I, float beta,
                                      float linear_beta, situ_dtype dt, void* stream);

/* -------------------------------------------------------------------------
 * MX experts -- the SiTU-GLU FFN with block-scaled operands: MXFP8 activations
 * and MXFP8 or MXFP4 expert weights.
 *
 * The "SiTU-GLU" chapter ("Pourquoi un plafond doux"; "Ou SiTU-GLU est utilise")
 * motivates the activation's +/-100 bound by experts that run in MXFP8 / MXFP4.
 * The format is the OCP Microscaling (MX) v1.0 MXFP8: E4M3 element codes (largest
 * magnitude 448), one E8M0 scale 2^(floor(log2 amax) - 8) per 32 consecutive
 * elements along K (amax the block's largest magnitude; zero blocks take 2^-127);
 * each code is the element divided by its scale, rounded to nearest even, clamped
 * to 448.  Quantization reads bf16 values, so every rounding decision is taken on
 * the bf16 input.
 *
 * MXFP4 weights (weight_fmt SITU_MX_E2M1) are the specification's MXFP4: E2M1 codes
 * (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), one E8M0 scale 2^(floor(log2 amax) - 2)
 * per 32 elements, codes past 6 clamped, packed two a byte with element 2j in the
 * low nibble of byte j; they run on the same block-scaled MMA (E4M3 x E2M1) with half
 * the weight bytes to stream.
 *
 * Codes keep the operand's row-major layout (K contiguous).  Scales are stored
 * in the tiles the block-scaled MMA consumes:
 *   activations (x, h): per 128-row tile and 128-wide K stage, 512 bytes, byte
 *     l * 16 + g * 4 + k = scale of row 32 g + l of the tile, 32-wide block k of the
 *     stage; tiles ordered (row tile, K stage); situ_mx_act_scales_size bytes.
 *   weights: per (expert, n-tile, K stage) 1024 bytes holding the n-tile's 192
 *     rows as rows 0..127 and 128..191 of two such 512-byte tiles.  SITU_MX_GATE_UP
 *     (W_gate_up [E, 2I, M], K = M): n-tile t = gate rows 96t..96t+95 then up rows
 *     I + 96t..; SITU_MX_DOWN (W_down [E, M, I], K = I): n-tile t = rows
 *     192t..192t+191.  situ_mx_weight_scales_size bytes; positions no row maps to
 *     hold code 0.
 * All MXFP8 calls need M and I multiples of 128 (SITU_ERR_UNSUPPORTED otherwise)
 * and 16-byte aligned code and scale pointers.
 * ------------------------------------------------------------------------- */
#define SITU_MX_GATE_UP 0
#define SITU_MX_DOWN 1
#define SITU_MX_E4M3 0 /* MXFP8 weight codes, one a byte */
#define SITU_MX_E2M1 1 /* MXFP4 weight codes, two a byte */

size_t situ_mx_act_scales_size(int64_t R, int64_t K);
size_t situ_mx_weight_scales_size(int32_t E, int64_t M, int64_t I, int kind);

/* x [R, K] bf16 (device) -> codes [R, K] uint8 and scales (activation tiles),
 * both device, written.  K % 128 == 0.  Errors: SITU_ERR_ARG, SITU_ERR_ALIGN,
 * SITU_ERR_ALIAS, SITU_ERR_UNSUPPORTED, SITU_ERR_CUDA. */
situ_status situ_mx_quantize_act(const void* x, void* codes, void* scales, int64_t R, int64_t K,
                                 void* stream);

/* Stacked expert weights W [E, rows, K] bf16 (kind SITU_MX_GATE_UP: rows = 2I,
 * K = M; SITU_MX_DOWN: rows = M, K = I) -> codes (fmt SITU_MX_E4M3: [E, rows, K]
 * bytes; SITU_MX_E2M1: [E, rows, K / 2] bytes) and scales (weight tiles), written.
 * A one-time conversion: the weights then stay resident as MXFP8 / MXFP4.
 * Errors: as situ_mx_quantize_act. */
situ_status situ_mx_quantize_weights(const void* W, void* codes, void* scales, int32_t E,
                                     int64_t M, int64_t I, int kind, int fmt, void* stream);

/* The packed gate_up projection of MXFP8 x (codes [R, M] + activation scales) by
 * W_gate_up (one expert, SITU_MX_GATE_UP layout, weight_fmt SITU_MX_E4M3 or
 * SITU_MX_E2M1), FP32 accumulation, with the SiTU-GLU activation on the
 * accumulators; h [R, I] bf16 written.  Caps as situ_glu_act.  Errors: SITU_ERR_ARG,
 * SITU_ERR_ALIGN, SITU_ERR_ALIAS, SITU_ERR_UNSUPPORTED, SITU_ERR_CUDA;
 * SITU_ERR_TIMEOUT on the device. */
situ_status situ_ffn_gate_up_mxfp8(const void* x_codes, const void* x_scales,
                                   const void* wgu_codes, const void* wgu_scales, int weight_fmt,
                                   void* h, int64_t R, int64_t M, int64_t I, float beta,
                                   float linear_beta, void* stream);

/* The dense FFN with MXFP8 experts: x [R, M] bf16 is quantized to MXFP8; the gate_up
 * GEMM (block-scaled, FP32 accumulation) applies SiTU-GLU, rounds h to bf16 (the
 * pages' cast back to the input dtype) and writes it as MXFP8 in its epilogue; the
 * down GEMM (block-scaled) writes y [R, M] bf16.  Both GEMMs run in one persistent
 * launch as in situ_ffn_forward (two launches when that grid cannot be co-resident).
 *   wgu_*, wd_*   device, one expert's weights as situ_mx_quantize_weights wrote them,
 *                 in format weight_fmt.
 *   workspace     device, >= situ_ffn_mxfp8_workspace_size(R, M, I) bytes, 256-byte
 *                 aligned; regions (each starting 256-byte aligned, in order): x codes
 *                 [R, M], x scales, h codes [R, I], h scales, one int32 per 128-row
 *                 tile of h-ready counts -- after the call the first four hold the
 *                 quantized x and h.
 * Errors: those of situ_ffn_gate_up_mxfp8, SITU_ERR_WORKSPACE. */
size_t situ_ffn_mxfp8_workspace_size(int64_t R, int64_t M, int64_t I);
situ_status situ_ffn_forward_mxfp8(const void* x, const void* wgu_codes, const void* wgu_scales,
                                   const void* wd_codes, const void* wd_scales, int weight_fmt,
                                   void* y, void* workspace, size_t workspace_bytes, int64_t R,
                                   int64_t M, int64_t I, float beta, float linear_beta,
                                   void* stream);

/* situ_moe_grouped_forward with MXFP8 experts: x is gathered into expert order and
 * quantized (scale tiles following each expert's 128-row tiles), then the grouped
 * block-scaled gate_up (h written as MXFP8) and down GEMMs; y [T, k_eff, M] bf16 per
 * (token, slot) as situ_moe_grouped_forward.  Weights [E, ...] as
 * situ_mx_quantize_weights wrote them, in format weight_fmt.  workspace >= situ_moe_mxfp8_workspace_size
 * (T * k_eff, E, M, I) bytes, 256-byte aligned.  Errors: those of
 * situ_moe_grouped_forward. */
size_t situ_moe_mxfp8_workspace_size(int64_t R, int32_t E, int64_t M, int64_t I);
situ_status situ_moe_grouped_forward_mxfp8(const void* x, const int32_t* expert_offsets,
                                           const int32_t* token_index, const void* wgu_codes,
                                           const void* wgu_scales, const void* wd_codes,
                                           const void* wd_scales, int weight_fmt, void* y,
                                           void* workspace, size_t workspace_bytes, int64_t T,
                                           int32_t k_eff, int32_t E, int64_t M, int64_t I,
                                           float beta, float linear_beta, void* stream);

/* -------------------------------------------------------------------------
 * situ_moe_combine -- the layer output of a routed batch: for every token t,
 *   out[t, :] = dtype( sum over slots s = 0 .. k_eff-1 of w[t, s] * y[t, s, :] ),
 * accumulated in FP32 in slot order (deterministic; no atomics).  Each routed and
 * shared expert of Kimi K3 runs on its tokens ("SiTU-GLU" chapter, "Ou SiTU-GLU
 * est utilise"); the layer output is the router-weighted sum of a token's expert
 * outputs, with shared experts as extra slots (weight 1 for a plain sum).
 *
 *   y        device, [T, k_eff, M] of `dt` (as situ_moe_grouped_forward writes it).
 *   weights  device, [T, k_eff] float32 combine weights.
 *   out      device, [T, M] of `dt`; must not overlap y or weights.
 *   T >= 0, k_eff >= 1, M >= 1.  Rows start 16-byte aligned (M % 8 == 0 for bf16,
 *   M % 4 == 0 for f32, aligned pointers) use 128-bit accesses, others a scalar path.
 * Errors: SITU_ERR_ARG, SITU_ERR_ALIAS, SITU_ERR_CUDA.
 * ------------------------------------------------------------------------- */
situ_status situ_moe_combine(const void* y, const float* weights, void* out, int64_t T,
                             int32_t k_eff, int64_t M, situ_dtype dt, void* stream);

/* -------------------------------------------------------------------------
 * situ_selftest_group_maps -- self test of the per-group tensor maps of the
 * K-grouped weight-gradient GEMMs (no counterpart on the pages).  Encodes two tensor
 * maps over MN-major operands of `rows` x `cols` (and 2 * cols) bf16 elements on the
 * host, lets a kernel write one copy of each per group with its row extent set to the
 * group's end k_offsets[g + 1], copies them back and compares each byte for byte with
 * the driver's own encoding of that base and extent (a group ending before row 32 gets
 * 32 rows from a base moved that many rows earlier; a group without rows keeps the
 * template).  No copy reads through the maps.
 *   k_offsets   host, [groups + 1] int32, non-decreasing, k_offsets[0] >= 0,
 *               k_offsets[groups] <= rows.
 *   groups      1 .. 65536;  rows 1 .. 2^31 - 1;  cols a multiple of 8.
 *   mismatches  host, out, [2 * groups] int32: entry 2g (A) and 2g + 1 (B) are 1 where
 *               group g's map differs from the driver's encoding, else 0.
 * Synchronises `stream`; allocates and frees a little device memory.
 * Errors: SITU_ERR_ARG, SITU_ERR_CUDA.
 * ------------------------------------------------------------------------- */
situ_status situ_selftest_group_maps(const int32_t* k_offsets, int32_t groups, int64_t rows,
                                     int64_t cols, int32_t* mismatches, void* stream);

/* -------------------------------------------------------------------------
 * situ_selftest_bounded_wait -- failure-detection self test (no counterpart on
 * the pages).  Launches one block that waits on a shared-memory barrier nothing
 * ever completes, with a wait limit of `limit_us` microseconds (1..1000000).
 * The wait gives up, records SITU_ERR_TIMEOUT in the device status and the
 * kernel returns normally, leaving the context usable.  This is the same bounded
 * wait every pipelined kernel of the library uses.
 * Errors: SITU_ERR_ARG, SITU_ERR_CUDA.
 * ------------------------------------------------------------------------- */
situ_status situ_selftest_bounded_wait(uint32_t limit_us, void* stream);

/* -------------------------------------------------------------------------
 * situ_set_wait_limit_ns -- bound of the GEMM kernels' waits (failure detection;
 * no counterpart on the pages).  Every wait of the pipelined GEMM kernels (a stage's
 * copies, an accumulator, the one-launch FFN's wait for another CTA's h rows) gives
 * up after `ns` nanoseconds of wall time: the kernel then records SITU_ERR_TIMEOUT in
 * the device status, drains its own copies and MMAs with bounded waits, frees its
 * tensor memory and returns; the results of that call are undefined, the context
 * stays usable.  Process-wide, read by each launch when it is enqueued; ns = 0
 * restores the default of 10 s (far above any legitimate wait).  A bound shorter
 * than the kernels' normal waits (a few microseconds) makes them time out: that is
 * how the failure path is exercised.  Returns the previous bound.
 * ------------------------------------------------------------------------- */
uint64_t situ_set_wait_limit_ns(uint64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* SITU_H */
