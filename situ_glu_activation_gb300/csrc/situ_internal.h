// situ_internal.h -- host-side launchers shared between the library's
// translation units (not part of the public ABI; see include/situ.h).
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "situ.h"
#include "situ_math.cuh"

namespace situ {

// Bytes of one element of a library dtype.
inline size_t dtype_size(situ_dtype dt) { return dt == SITU_F32 ? 4 : 2; }

// Largest finite cap the kernels accept (2^20); +infinity means "no cap".
constexpr float kMaxFiniteCap = 1048576.0f;

// Cap configuration from the two cap arguments (+infinity = uncapped branch).
inline Caps caps_of(float beta, float linear_beta) {
  const bool gi = beta > kMaxFiniteCap, ui = linear_beta > kMaxFiniteCap;
  return gi ? (ui ? Caps::kNone : Caps::kUpOnly) : (ui ? Caps::kGateOnly : Caps::kBoth);
}

// ----- standalone activation (act.cu) --------------------------------------
// gate_up [rows, 2I] -> out [rows, I]; picks the 128-bit path when rows start
// 16-byte aligned, else the scalar path.
cudaError_t launch_situ_act(const void* gate_up, void* out, int64_t rows, int64_t I,
                            const SituParams& p, Caps caps, situ_dtype dt, int num_sms,
                            cudaStream_t stream);

// ----- FP32 small-shape FFN (act.cu) ----------------------------------------
// h [R, I] = SiTU-GLU(x W_gate_up^T) then y [R, M] = h W_down^T, all float32.
cudaError_t launch_ffn_f32(const float* x, const float* w_gate_up, const float* w_down,
                           float* h, float* y, int64_t R, int64_t M, int64_t I,
                           const SituParams& p, Caps caps, cudaStream_t stream);

// ----- tcgen05 GEMMs (gemm.cu) ------------------------------------------------
struct GemmShape {
  // A operand: [a_rows, K] bf16 row-major (dense x / gathered rows / h).
  const void* a;
  int64_t a_rows;
  // B operand: [b_rows, K] bf16 row-major (one or E stacked weight matrices).
  const void* b;
  int64_t b_rows;
  int64_t K;
  // Row groups (experts).  group_offsets / tile_offsets are device arrays of
  // G + 1 int32 each, or NULL for a single dense group of a_rows rows.
  int32_t num_groups;
  const int32_t* group_offsets;
  const int32_t* tile_offsets;
  // Work-unit prefix per group for this GEMM (from launch_group_tiles), or NULL.
  const int32_t* unit_offsets;
  // unit_offsets count two-CTA units (ceil(m-tiles / 2) per output tile; the group's
  // pairs run as cta_group::2 MMAs); otherwise the grouped GEMM runs one CTA per tile
  // over tile_offsets.
  bool pair_units;
  int64_t b_group_rows;  // B rows per group
  int64_t b_up_offset;   // SiTU epilogue: row offset of the up half inside a group
  int64_t n_out;         // valid output columns
  // Output [out_rows, ldo] bf16; row of A-row r is out_row_index[r] if given.
  void* out;
  int64_t ldo;
  int64_t out_rows;
  const int32_t* out_row_index;
  // Row strides (elements) of A and B when they differ from K (0 = K), or, for
  // MN-major operands, from their row / N extent.
  int64_t a_ld;
  int64_t b_ld;
  // MN-major operands: A stored [K, a_rows], B stored [K, b_rows] (the row / N
  // index contiguous).  Supported: B alone, or A and B; the SiTU epilogue needs a
  // K-major B.
  bool a_mn_major;
  bool b_mn_major;
  // K-grouped contraction (A and B both MN-major, grouped by K rows): group g
  // contracts over the K rows k_group_offsets[g] .. k_group_offsets[g+1]-1 of both
  // operands ([G+1] int32, device) and writes its [a_rows, n_out] result at output
  // row g * out_group_rows.  K is then the operands' total row count.  With
  // tile_offsets given, a zero tile_offsets[num_groups] (offsets that failed
  // validation) makes the GEMM do nothing.
  const int32_t* k_group_offsets;
  // K-grouped: an optional permutation of the groups (device, [num_groups]), the
  // order their units run in (largest row count first balances the CTAs).
  const int32_t* group_order;
  int64_t out_group_rows;
  // K-grouped: device scratch for two tensor maps per group ([2 * num_groups]
  // CUtensorMap, 128-byte aligned), written by the launch; with it the contraction runs
  // as two-CTA MMAs (without it, one CTA per tile).
  void* group_maps;
  // MXFP8 operands (launch_mx_gemm_*): A and B are E4M3 codes (row-major, K
  // contiguous, K a multiple of 128); sfa / sfb their E8M0 scale tiles (A: 512 bytes
  // per 128-row m-tile and 128-wide K stage; B: 1024 bytes per (group, n-tile) and K
  // stage).  h_codes / h_sf: the SiTU epilogue's MXFP8 output (codes [rows, ldo],
  // scale tiles in the A layout with n_out / 128 K stages), or null for bf16 h.
  const void* sfa;
  const void* sfb;
  void* h_codes;
  void* h_sf;
  // MXFP4 B: E2M1 codes packed two a byte ([b_rows, K / 2] bytes).
  bool b_fp4;
  // Plain epilogue with a fused combine (routed down projection): output row r (flat
  // route token * combine_k + slot, from out_row_index) is added, times combine_w[r],
  // into combine_out[r / combine_k] (FP32 [tokens, n_out], 16-byte aligned rows) by
  // atomic adds instead of being stored.
  const float* combine_w;
  void* combine_out;
  int32_t combine_k;
  // SiTU epilogue: optional bf16 store of the pre-activation (g, u), [rows, 2*split].
  void* gu_store;
  // Backward epilogue: saved (g, u) in, d(g, u) out, both [rows, 2*split] bf16.
  const void* gu_in;
  void* dgu_out;
  int64_t split;
};

// gu = A B^T with the SiTU-GLU epilogue: output column j of group tile n pairs B
// row n*128 + j (gate) with B row b_up_offset + n*128 + j (up).
cudaError_t launch_gemm_situ(const GemmShape& s, const SituParams& p, Caps caps,
                             uint32_t* status, int num_sms, cudaStream_t stream);
// C = A B^T, bf16 output.
cudaError_t launch_gemm_plain(const GemmShape& s, uint32_t* status, int num_sms,
                              cudaStream_t stream);
// Two independent plain GEMMs (same operand layouts, dense) in one persistent launch:
// the tiles of s1, then those of s2.
cudaError_t launch_gemm_plain2(const GemmShape& s1, const GemmShape& s2, uint32_t* status,
                               int num_sms, cudaStream_t stream);
// The dense bf16 FFN in one persistent cooperative launch: s_gu is the gate_up GEMM
// (SiTU epilogue into h), s_dn the down GEMM (A = h, out = y); h_ready holds one int32
// per 128-row m-tile of scratch.  Returns an error (and launches nothing) when the
// grid cannot be co-resident.
cudaError_t launch_ffn_fused(const GemmShape& s_gu, const GemmShape& s_dn, const SituParams& p,
                             Caps caps, int32_t* h_ready, uint32_t* status, int num_sms,
                             cudaStream_t stream);
// dh = A B^T (B 256-wide tiles like the plain GEMM), epilogue: d(g, u) = dh * the
// activation's partial derivatives at the saved (g, u).
cudaError_t launch_gemm_situ_bwd(const GemmShape& s, const SituParams& p, Caps caps,
                                 uint32_t* status, int num_sms, cudaStream_t stream);

// ----- MXFP8 block-scaled GEMMs (mx_gemm.cu) ------------------------------------
// Tile widths of the MXFP8 GEMMs: 96 activation columns per SiTU tile (gate rows
// and up rows of B in two 96-row halves), 192 output columns per plain tile.
constexpr int kMxSituCols = 96;
constexpr int kMxPlainCols = 192;
// gu = A B^T (MXFP8) with the SiTU-GLU epilogue: bf16 h into s.out, or MXFP8 h into
// s.h_codes / s.h_sf when s.h_codes is set.
cudaError_t launch_mx_gemm_situ(const GemmShape& s, const SituParams& p, Caps caps,
                                uint32_t* status, int num_sms, cudaStream_t stream);
// C = A B^T (MXFP8), bf16 output.
cudaError_t launch_mx_gemm_plain(const GemmShape& s, uint32_t* status, int num_sms,
                                 cudaStream_t stream);
// The dense MXFP8 FFN in one persistent cooperative launch: s_gu the gate_up GEMM (h as
// MXFP8 into h_codes / h_sf), s_dn the down GEMM (A = h codes, sfa = h scales); h_ready
// holds one int32 per 128-row m-tile.  Launches nothing and returns an error when the
// grid cannot be co-resident.
cudaError_t launch_mx_ffn_fused(const GemmShape& s_gu, const GemmShape& s_dn, const SituParams& p,
                                Caps caps, int32_t* h_ready, uint32_t* status, int num_sms,
                                cudaStream_t stream);
// MXFP8 quantization of bf16 rows [R, K] (K % 128 == 0) into codes [R, K] and A-layout
// scale tiles.  Row r is read from src row (row_index ? row_index[r] / k_eff : r);
// with group offsets (and their m-tile prefix) the tiles follow the groups' m-tiles.
// sf_tiles bounds the scale tiles written (a row mapping outside is recorded as
// SITU_ERR_INDEX and skipped).
cudaError_t launch_mx_quantize_act(const void* src, const int32_t* row_index, int32_t k_eff,
                                   int64_t src_rows, void* codes, void* scales, int64_t sf_tiles,
                                   int64_t R, int64_t K, int32_t num_groups,
                                   const int32_t* group_offsets, const int32_t* tile_offsets,
                                   uint32_t* status, cudaStream_t stream);
// MXFP8 quantization of G stacked weight matrices [rows_per_group, K] into codes and
// B-layout scale tiles: split > 0 pairs gate row j < split with up row split + j in
// tiles of 96 + 96 rows (the SiTU GEMM's B); split == 0 cuts plain 192-row tiles.
// fp4: E2M1 codes, two a byte ([rows, K / 2] bytes), scale 2^(floor(log2 amax) - 2).
cudaError_t launch_mx_quantize_weights(const void* w, void* codes, void* scales, int32_t G,
                                       int64_t rows_per_group, int64_t K, int64_t split,
                                       bool fp4, cudaStream_t stream);
// Scale bytes of those layouts.
size_t mx_act_scale_bytes(int64_t R, int64_t K);
size_t mx_weight_scale_bytes(int32_t G, int64_t rows_per_group, int64_t K, int64_t split);

// Per-group prefixes of m-tiles and of the work units of two grouped GEMMs with
// n_tiles_1 and n_tiles_2 output tiles per m-tile, plus validation of the offsets.
// order[rank] = group, ranking groups by descending row count (ties by index): the
// K-grouped weight-gradient GEMMs run the largest contractions first.
cudaError_t launch_group_order(const int32_t* group_offsets, int32_t G, int32_t* order,
                               cudaStream_t stream);
// two_cta: the unit prefixes count two-CTA units (ceil(m/2) per output tile); otherwise
// tiles (m per output tile).
cudaError_t launch_group_tiles(const int32_t* group_offsets, int32_t G, int64_t R,
                               int32_t n_tiles_1, int32_t n_tiles_2, int32_t* tile_offsets,
                               int32_t* units_1, int32_t* units_2, uint32_t* status,
                               cudaStream_t stream, bool two_cta = false);
// Whether the two-CTA MMA kernels can run on this device (2-CTA clusters fit).
bool gemm_two_cta_available();
// Output tiles per m-tile: of the SiTU GEMM (128 activation columns per tile) and
// of the plain / backward GEMMs (256 columns per tile), for n_out output columns.
int32_t gemm_n_tiles_situ(int64_t n_out);
int32_t gemm_n_tiles_wide(int64_t n_out);
// x_perm[r, :] = x[token_index[r] / k_eff, :]  (M bf16 columns).
cudaError_t launch_gather_rows(const void* x, const int32_t* token_index, void* x_perm,
                               int64_t R, int32_t k_eff, int64_t M, uint32_t* status,
                               cudaStream_t stream);
// Per-group tensor-map extents written on the device against the driver's encoding
// (host k_offsets [groups + 1]); mismatches [2 * groups]: 1 where a map differs.
cudaError_t group_maps_selftest(const int32_t* k_offsets, int32_t groups, int64_t rows,
                                int64_t cols, int32_t* mismatches, cudaStream_t stream);
// One block waiting on a barrier nothing completes, bounded by limit_ns.
cudaError_t launch_bounded_wait_selftest(uint64_t limit_ns, uint32_t* status,
                                         cudaStream_t stream);

// ----- routed-layer combine (combine.cu) --------------------------------------
// out[i] = bf16(acc[i]) for n FP32 values (the fused combine's cast).
cudaError_t launch_f32_to_bf16(const float* acc, void* out, int64_t n, int num_sms,
                               cudaStream_t stream);
// out[t, :] = sum_s w[t, s] * y[t, s, :] in FP32, slot order (w == NULL: all 1).
cudaError_t launch_combine(const void* y, const float* w, void* out, int64_t T, int32_t k_eff,
                           int64_t M, situ_dtype dt, int num_sms, cudaStream_t stream);

// ----- expert index (moe_index.cu) -------------------------------------------
size_t index_workspace_bytes(int64_t n, int32_t E);
cudaError_t launch_build_index(const int32_t* expert_ids, int32_t* offsets,
                               int32_t* token_index, void* workspace, int64_t n, int32_t E,
                               uint32_t* status, cudaStream_t stream);

}  // namespace situ

namespace situ {

// ----- shared with abi.cu ------------------------------------------------------
// Wall-time bound of every pipeline wait in the GEMM kernels, read at each launch
// (situ_set_wait_limit_ns; default 10 s).
uint64_t wait_limit_ns();
// The argument checks situ_ffn_forward applies: dtype, sizes, caps (SITU_ERR_ARG) and the
// kernels' size limits (SITU_ERR_UNSUPPORTED); for bf16, M and I multiples of 8
// (SITU_ERR_UNSUPPORTED) and 16-byte aligned x and weights (SITU_ERR_ALIGN).
situ_status ffn_arg_checks(situ_dtype dt, int64_t R, int64_t M, int64_t I, float beta,
                           float linear_beta);
situ_status ffn_bf16_operand_checks(const void* x, const void* W_gate_up, const void* W_down,
                                    int64_t M, int64_t I);
// SM count and device address of the status word of the current device (the
// library's one-time per-device set-up runs on first use; it allocates nothing).
situ_status current_device_context(int* num_sms, uint32_t** status);
// Record a CUDA error for situ_last_cuda_error() and return SITU_ERR_CUDA.
situ_status report_cuda_error(cudaError_t e);

}  // namespace situ
