// gemm_kernel.cuh -- the persistent, warp-specialised tcgen05 GEMM kernel shared
// by the bf16 GEMMs (gemm.cu) and the MXFP8 block-scaled GEMMs (mx_gemm.cu), with
// its host-side launch.  Included by exactly those translation units; everything
// is in an anonymous namespace, so each unit instantiates what it launches.
//
// One CTA per SM (persistent); 192 threads (224 for MXFP8, 320 for the activation-
// derivative epilogue):
//   warp 0      TMA producer: per k-block, the A box(es) and B rows into a ring of
//               128-byte-swizzled shared-memory stages (bf16: 4 stages of A 128x64 +
//               B 256x64, or 6 stages of A 128x64 + half of B with two-CTA MMAs;
//               MXFP8: 5 stages of A 128x128 + B 192x128 codes and the scale tiles,
//               or 7 stages of A 128x128 + half of B and the scale tiles with two-CTA
//               MMAs).
//   warp 1      MMA issuer: tcgen05.mma (kind::f16 M=128 N=256 K=16, M=64 for tiles with
//               at most 64 rows, or cta_group::2 M=256 over a CTA pair; kind::mxf8f6f4
//               block-scaled M=128 or M=256 N=192 K=32), accumulating in tensor memory;
//               tcgen05.commit frees each stage and publishes each finished accumulator.
//               Two accumulators let the epilogue of tile i overlap the MMAs of tile i+1.
//   warps 2..   epilogue (4 warps, 8 for the derivative): tcgen05.ld (thread = tile row);
//               SiTU-GLU on (gate column j, up column BN/2 + j) with bf16 or MXFP8 output,
//               plain conversion, the activation's derivative (backward), or a fused
//               weighted scatter-add.
//   last warp   (MXFP8) copies each stage's scale tiles into TMEM as it lands (with
//               two-CTA MMAs: the even CTA's warp copies both CTAs' tiles, the odd
//               CTA's relays the landing of its own to the even CTA's barrier).
// Every CTA loads its own operands with plain TMA tile copies into its own shared
// memory (no copy is multicast).  One-CTA kernels take one tile per work unit, in
// (group, m-tile, n-tile) order, so the n-tiles of one m-tile run side by side and
// share A in L2, and the m-tiles of one group follow each other and share B there; a
// tile with at most 64 valid rows fetches only those 64 A rows.  With two-CTA MMAs
// (dense GEMMs, large-expert grouped GEMMs, the K-grouped weight gradients, the dense
// MXFP8 GEMMs) a cluster of two CTAs takes m-tiles 2p and 2p+1 of one n-tile as one
// M=256 MMA: each CTA stages its own A rows and its half of B, both CTAs' copies count
// on the even CTA's barrier, and its MMA thread issues for both.  Operands are K-major,
// or MN-major ({64, 64} boxes) for the backward, which also has a K-grouped schedule
// (each group contracts over its own row range, read through tensor maps that end at
// the group's end; groups largest first, rounds in serpentine order).
// Two GEMMs can share one launch: the whole FFN (down tiles wait, across CTAs, for the
// h rows of their m-tile; a cooperative launch) or two independent plain GEMMs.  Every
// wait is bounded (ctl_wait / mbar_wait / wait_count); on a timeout the CTA records
// SITU_ERR_TIMEOUT, drains its in-flight copies and MMAs with bounded waits, frees its
// tensor memory and exits.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <type_traits>

#include "situ_internal.h"
#include "situ_math.cuh"
#include "situ_ptx.cuh"

namespace situ {
namespace {

constexpr int kBM = 128;  // tile rows (UMMA M)
constexpr int kBN = 256;  // accumulator columns per tile (UMMA N)
constexpr int kBK = 64;   // K per stage: one 128-byte swizzle row of bf16
constexpr int kUK = 16;   // K per tcgen05.mma for 16-bit inputs
constexpr int kAccBufs = 2;
constexpr uint32_t kTmemCols = 512;
constexpr int kEpiThreads = 128;
// Every wait of the pipeline is bounded by the launch's wait limit (wait_limit_ns(),
// default 10 s); the drains after an abort by 100 ms.  After an abort, a CTA of a
// two-CTA pair stays resident kAbortLingerNs before the final cluster barrier: its
// operand copies complete on the even CTA's barriers, which it cannot wait on, and
// the linger lets every copy it issued land while both CTAs' shared memory is live.
constexpr uint64_t kDrainLimitNs = 100ull * 1000 * 1000;  // 100 ms
constexpr uint64_t kAbortLingerNs = 1000ull * 1000;       // 1 ms
constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kBN);
// Tiles with at most 64 valid rows (an expert's tail, a small group) issue M=64
// MMAs: half the tensor work.  Their accumulator rows 16q..16q+15 sit in TMEM lanes
// 32q..32q+15 (the first 16 lanes of each warp's quarter), measured on GB300.
constexpr uint32_t kIdescHalf = idesc_bf16_f32(64, kBN);
// Operand layouts: kKMajor -- A [rows, K] and B [N, K] with K contiguous (the
// forward); kBMN -- B stored [K, N] (N contiguous), e.g. W_down when the
// backward multiplies by it untransposed; kABMN -- A stored [K, rows] and B
// stored [K, N], e.g. dy and h when the weight gradient contracts over tokens.
// MN-major tiles arrive as {64, 64} boxes (8 KB): A takes two, B four.
// kABMNGrouped -- the kABMN layouts with a K-grouped schedule: each group (expert)
// contracts over its own row range (per-expert weight gradients).
enum class Major { kKMajor = 0, kBMN = 1, kABMN = 2, kABMNGrouped = 3 };
__host__ __device__ constexpr bool a_mn_major(Major m) { return m == Major::kABMN || m == Major::kABMNGrouped; }
constexpr uint32_t kAMnBit = 1u << 15, kBMnBit = 1u << 16;
constexpr uint32_t kMnAtomBytes = 64 * 64 * 2;
// Two-CTA K-grouped contractions read each group through tensor maps whose rows end at
// the group's end (group_maps_kernel); such a map spans at least kMinGroupMapRows rows, a
// group ending before that row is read through a map based group_map_shift rows earlier.
constexpr int32_t kMinGroupMapRows = 32;
__host__ __device__ __forceinline__ int32_t group_map_shift(int32_t k_end) {
  return k_end < kMinGroupMapRows ? kMinGroupMapRows - k_end : 0;
}

// Tile geometry per operand type.  Both stage 128-byte rows of K (one 128-byte
// swizzle row): 64 bf16 or 128 MXFP8 codes.
//   bf16: N = 256 accumulator columns, 4 stages of A 128x64 + B 256x64 (48 KB).
//   MXFP8 (E4M3 codes, one E8M0 scale per 32 along K): N = 192 (two accumulators
//     of 192 columns leave TMEM room for the scales), 5 stages of A 128x128 +
//     B 192x128 codes + the A and B scale tiles of the stage (512 + 1024 bytes),
//     K = 32 per MMA.  B arrives as two 96-row halves.
// kMx: 0 bf16; 1 MXFP8 A and B; 2 MXFP8 A and MXFP4 B (E2M1 weights, packed two a
// byte in memory; TMA unpacks each 16 codes into a 16-byte chunk of shared memory --
// 8 bytes of codes, 8 bytes of gap -- the layout the block-scaled MMA reads for 4-bit
// operands, so the stage keeps the MXFP8 geometry and only half the B bytes travel).
template <int kMx>
struct Geo {
  static constexpr int BN = 256, BK = 64, UK = 16, Stages = 4, BHalfRows = 128;
  static constexpr uint32_t ABytes = 16384, BBytes = 32768, SfBytes = 0;
  static constexpr uint32_t TxBytes = ABytes + BBytes;  // bytes the copies of a stage bring
  static constexpr uint32_t StageBytes = TxBytes;
};
template <>
struct Geo<1> {
  // A seventh warp copies each stage's scale tiles into TMEM as soon as the stage
  // lands, so the MMA warp never issues a tcgen05.cp in front of its own MMAs (a
  // copy issued right before the MMAs that read it held the tensor pipe ~20 % idle,
  // measured on GB300).
  static constexpr int BN = 192, BK = 128, UK = 32, Stages = 5, BHalfRows = 96;
  static constexpr uint32_t ABytes = 16384, BBytes = 24576, SfBytes = 512 + 1024;
  static constexpr uint32_t TxBytes = ABytes + BBytes + SfBytes;
  static constexpr uint32_t StageBytes = 43008;  // TxBytes rounded up to 1 KB
};
template <>
struct Geo<2> : Geo<1> {
  static constexpr uint32_t TxBytes = ABytes + BBytes / 2 + SfBytes;  // B arrives packed
};
// Two-CTA MMA (dense bf16): each CTA of the pair stages its own A tile and its half of
// B (32 KB), so six stages fit where four shared-B stages did; the even CTA's barrier
// counts both CTAs' bytes.
struct GeoPair {
  static constexpr int BN = 256, BK = 64, UK = 16, Stages = 6, BHalfRows = 128;
  static constexpr uint32_t ABytes = 16384, BBytes = 16384, SfBytes = 0;
  static constexpr uint32_t TxBytes = 2 * (ABytes + BBytes);  // both CTAs' copies
  static constexpr uint32_t StageBytes = ABytes + BBytes;
};
// Two-CTA MMA (MXFP8 / MXFP4 B): M = 256, N = 192; each CTA stages its own A codes, its
// 96-row half of B and its own A and B scale tiles (the pair MMA reads both from each
// CTA's own tensor memory), 30 KB a stage, seven stages.  The even CTA's barrier counts
// both CTAs' codes and its own scales; the odd CTA's scales land on a barrier of its own
// and are relayed (see the scale copier).
template <int kMx>
struct GeoPairT : GeoPair {};
template <>
struct GeoPairT<1> {
  static constexpr int BN = 192, BK = 128, UK = 32, Stages = 7, BHalfRows = 96;
  static constexpr uint32_t ABytes = 16384, BBytes = 12288, SfBytes = 512 + 1024;
  static constexpr uint32_t TxBytes = 2 * (ABytes + BBytes) + SfBytes;
  static constexpr uint32_t StageBytes = 30720;  // A + B + scales rounded up to 1 KB
};
template <>
struct GeoPairT<2> : GeoPairT<1> {
  static constexpr uint32_t TxBytes = 2 * (ABytes + BBytes / 2) + SfBytes;  // B arrives packed
};
// The two-CTA activation-derivative GEMM (dh): five operand stages, and kGuSlots
// 16 KB slots in which a loader warp stages the saved (g, u) of the epilogue's
// 32-column chunks ahead of the accumulator.  A slot holds the chunk's g columns for
// the CTA's 128 rows (64 bytes a row), then its u columns, each with the 64-byte
// swizzle: 16-byte piece v of slot row r sits at piece v ^ ((r >> 1) & 3) of the row,
// so that eight threads reading piece v of eight consecutive rows hit distinct banks.
struct GeoPairBwd : GeoPair {
  static constexpr int Stages = 5;
};
constexpr int kGuSlots = 4;
constexpr uint32_t kGuSlotBytes = 16384;
constexpr uint32_t kGuHalfBytes = kGuSlotBytes / 2;  // the g (or u) part of a slot
constexpr int kMaxStages = 7;
// MXFP8 scale tiles.  The block-scaled MMA reads the E8M0 scale of A row m for its
// k-th 32-wide K block (k = 0..3 within a 128-K stage) from TMEM lane m, column
// base + m / 32, byte k; that of B row n from column base + n / 32, byte k, in the
// lane quadrant of the accumulator row it is producing (measured on GB300 with an
// in-bounds probe).  tcgen05.cp.32x128b.warpx4 copies 32 rows x 16 bytes into all
// four quadrants, so a 128-row scale tile is stored as 512 bytes, byte
// l * 16 + g * 4 + k holding row 32 g + l, block k; B's 192 rows take two such tiles
// (1024 bytes, groups 6 and 7 unused).
constexpr uint32_t kSfTileBytes = 512;
constexpr uint32_t kSfbStageBytes = 1024;
constexpr uint32_t kSfTmemCols = 12;  // per stage: A 4 columns, B 8 columns

// Epilogues: kSitu applies SiTU-GLU to (gate, up) accumulator pairs (and can
// also store the pre-activation pair); kPlain converts to bf16; kSituBwd turns
// dh accumulators into d(gate, up) through the activation's derivative, reading
// the saved pre-activation pair.
// kSituMx (MXFP8 only) applies SiTU-GLU, rounds h to bf16 and stores it as MXFP8
// codes and scales, the input format of the next block-scaled GEMM.  kFfn is the
// whole dense FFN in one persistent launch: units [0, fused_units1) are gate_up
// tiles with the SiTU epilogue (h), the rest are down tiles with the plain epilogue
// (y); a down tile starts once every gate_up tile of its rows has stored its h.
// kPlain2 runs two independent plain GEMMs of the same operand layout in one
// persistent launch (units of the first, then of the second): the weight gradients of
// the dense backward, whose own tile counts (192 and 384) leave partial last waves.
enum class Epi { kSitu, kPlain, kSituBwd, kSituMx, kFfn, kPlain2 };

// Epilogue warps: 4 (one per TMEM lane quarter), or 8 for the activation-derivative
// epilogue, whose per-element work (eight SFU ops, about 30 FP32 ops, the saved (g, u)
// reads and the d(g, u) stores) is of the order of the tile's MMAs: with one warp per SM
// sub-partition its latency was exposed (the dh GEMM ran at 40 % of the dx GEMM's rate,
// measured on GB300).  With 8, warps e and e + 4 share a lane quarter and split the
// columns.
template <Epi kEpi>
__host__ __device__ constexpr int epi_warps() {
  return kEpi == Epi::kSituBwd ? 8 : 4;
}
// Column groups of epilogue warps: warps e, e + 4, ... share a TMEM lane quarter and
// split a tile's columns.
template <Epi kEpi>
__host__ __device__ constexpr int epi_col_groups() {
  return epi_warps<kEpi>() / 4;
}
// Threads per CTA: producer and MMA warps, the epilogue warps, and (MXFP8) the scale
// copier or (activation derivative) the loader of the saved (g, u).
template <Epi kEpi, int kMx>
__host__ __device__ constexpr int block_threads() {
  return 32 * (2 + epi_warps<kEpi>() + ((kMx || kEpi == Epi::kSituBwd) ? 1 : 0));
}

struct Args {
  int32_t num_groups;
  const int32_t* group_offsets;  // [G+1] device or null (dense)
  const int32_t* tile_offsets;   // [G+1] device or null (dense): m-tile prefix
  const int32_t* unit_offsets;   // [G+1] device or null (dense): two-CTA unit prefix
  int32_t dense_rows;
  int32_t n_tiles;
  int32_t k_blocks;
  int64_t b_group_rows;
  int64_t b_up_offset;
  int64_t n_out;
  __nv_bfloat16* out;
  int64_t ldo;
  int64_t out_rows;
  const int32_t* out_row_index;
  SituParams sp;
  uint32_t* status;
  // kSitu: optional store of the pre-activation (g, u) as bf16 [rows, 2*split];
  // kSituBwd: the saved (g, u) to read and d(g, u) to write, same layout.
  __nv_bfloat16* gu_store;
  const __nv_bfloat16* gu_in;
  __nv_bfloat16* dgu_out;
  int64_t split;
  // K-grouped contraction (MN-major A and B only): group g contracts over the K
  // rows k_group_offsets[g] .. k_group_offsets[g+1]-1 of both operands and writes
  // its [dense_rows, n_out] result at output rows g * out_group_rows.  Every group
  // has units_per_group work units.  A nonzero tile_offsets[num_groups] marks the
  // offsets as validated (zero: nothing runs).
  const int32_t* k_group_offsets;
  const int32_t* group_order;  // K-grouped: the groups in this order (null: index order)
  // Two-CTA K-grouped: per group, the A and B maps whose row extent ends at the group's
  // end (2g, 2g + 1; see group_maps_kernel).
  const CUtensorMap* group_maps;
  int32_t units_per_group;
  int64_t out_group_rows;
  // MXFP8: the scale tiles of A (per global m-tile and k-block, 512 bytes) and of
  // B (per (group, n-tile) and k-block, 1024 bytes); kSituMx output: h codes
  // [rows, ldo] and h scale tiles (A layout, n_out / 128 k-blocks per m-tile).
  const uint8_t* sfa;
  const uint8_t* sfb;
  const uint8_t* sfa2;  // kFfn with MXFP8: the down GEMM's scale tiles (h, W_down)
  const uint8_t* sfb2;
  uint8_t* h_codes;
  uint8_t* h_sf;
  // kPlain with a fused combine: instead of storing output row r (a route, flat
  // token * k_eff + slot), add combine_w[r] * row into combine_out[r / combine_k]
  // (FP32 [tokens, n_out]) with vector atomics.
  const float* combine_w;
  float* combine_out;
  int32_t combine_k;
  // kFfn: the down GEMM's geometry and output, and the per-m-tile count of gate_up
  // tiles whose h rows are stored (zeroed before the launch; ready at h_ready_target).
  // kPlain2: the second GEMM's geometry and output (its A rows: dense_rows2).
  int32_t fused_units1, fused_units2;
  int32_t dense_rows2;
  int32_t n_tiles2, k_blocks2;
  int64_t n_out2, ldo2;
  __nv_bfloat16* out2;
  int32_t* h_ready;
  int32_t h_ready_target;
  // Two-CTA grouped bf16 GEMMs: a group's odd last m-tile runs as an M = 128 pair
  // (64 rows per CTA) instead of an M = 256 pair with a phantom half.
  int32_t pair_tails;
  uint64_t wait_limit_ns;  // bound of every pipeline wait (wall time)
};

struct SharedCtl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t acc_full[kAccBufs];
  uint64_t acc_empty[kAccBufs];
  uint64_t drain;
  uint64_t sf_ready[kMaxStages];  // MXFP8: the stage's scales are in TMEM
  uint64_t sf_drain;
  uint64_t gu_full[kGuSlots];   // dh GEMM: a slot's saved (g, u) have landed
  uint64_t gu_done[kGuSlots];   // dh GEMM: the epilogue warps are done with the slot
  uint64_t wait_limit_ns;
  uint32_t tmem_base;
  volatile int abort;
};

struct TileCoord {
  int32_t a_row0;   // first A row of the tile
  int32_t row_end;  // one past the last valid A row (group end)
  int32_t group;
  int32_t n_tile;
  int32_t half_pair;  // two-CTA M = 128 pair: this CTA holds 64 rows from a_row0
  int32_t k0;       // first K row of the contraction (K-grouped; 0 otherwise)
  int32_t k_end;    // one past its last K row (K-grouped)
  int32_t k_blocks; // k-blocks of this tile
  int32_t phase2;   // kFfn: a down tile; kPlain2: a tile of the second GEMM
};

__device__ __forceinline__ int32_t total_tiles(const Args& a) {
  const int32_t m_tiles = a.tile_offsets ? __ldg(a.tile_offsets + a.num_groups)
                                         : (a.dense_rows + kBM - 1) / kBM;
  return m_tiles * a.n_tiles;
}

__device__ __forceinline__ TileCoord decode_tile(const Args& a, int32_t t) {
  TileCoord c;
  const int32_t mt = t / a.n_tiles;
  c.n_tile = t - mt * a.n_tiles;
  if (!a.tile_offsets) {
    c.group = 0;
    c.a_row0 = mt * kBM;
    c.row_end = a.dense_rows;
    c.half_pair = 0;
    return c;
  }
  // Largest g with tile_offsets[g] <= mt (empty groups repeat an offset; the
  // last of a run of equal offsets is the group that owns the tile).
  int32_t lo = 0, hi = a.num_groups - 1;
  while (lo < hi) {
    const int32_t mid = (lo + hi + 1) >> 1;
    if (__ldg(a.tile_offsets + mid) <= mt) lo = mid; else hi = mid - 1;
  }
  c.group = lo;
  c.a_row0 = __ldg(a.group_offsets + lo) + (mt - __ldg(a.tile_offsets + lo)) * kBM;
  c.row_end = __ldg(a.group_offsets + lo + 1);
  c.half_pair = 0;
  return c;
}

// Tile `local` of one group's rows row0 .. row_end-1 (m-tile-major).
__device__ __forceinline__ TileCoord in_group_tile(int32_t n_tiles, int32_t local, int32_t row0,
                                                   int32_t row_end) {
  TileCoord c;
  const int32_t mt = local / n_tiles;
  c.n_tile = local - mt * n_tiles;
  c.a_row0 = row0 + mt * kBM;
  c.row_end = row_end;
  c.group = 0;
  c.half_pair = 0;
  return c;
}

// Work units.  One-CTA kernels: one unit = one tile (decode_tile; K-grouped:
// in_group_tile within each group).  Two-CTA kernels (clusters of two CTAs, CTA rank
// r): unit (p, n) of a group gives rank r m-tile 2p + r of n-tile n (pair_unit); dense
// calls are one group of all rows, grouped calls read the per-group unit prefix from
// unit_offsets.
template <bool kPair, bool kKG, bool kTwo = false>
__device__ __forceinline__ int32_t num_units(const Args& a) {
  if (kTwo) return a.fused_units1 + a.fused_units2;
  if (kKG) {
    if (a.tile_offsets && __ldg(a.tile_offsets + a.num_groups) == 0) return 0;
    return a.num_groups * a.units_per_group;
  }
  if (kPair) {
    if (a.unit_offsets) return __ldg(a.unit_offsets + a.num_groups);
    return ((a.dense_rows + 2 * kBM - 1) / (2 * kBM)) * a.n_tiles;
  }
  return total_tiles(a);
}

// The unit of a CTA's i-th round: round i covers units [i * stride, (i + 1) * stride),
// one per CTA (pair).  K-grouped schedules walk alternate rounds in reverse
// (serpentine): their units cost in proportion to their group's rows, and with the
// groups ordered by descending rows this keeps the CTAs' totals within about 1 % of
// each other, against 5-14 % for a fixed CTA-to-offset assignment (Zipf-routed
// experts).  Every role of a CTA walks the same rounds.
template <bool kSerpentine>
__device__ __forceinline__ int32_t round_unit(int32_t i, int32_t u0, int32_t stride) {
  return i * stride + ((kSerpentine && (i & 1)) ? stride - 1 - u0 : u0);
}

// Two-CTA unit `local` of a group's rows row0 .. row_end-1: CTA r of the pair takes
// m-tile 2p + r of n-tile n (a last pair past the rows computes fill that is not
// stored).  With half-pair tails, a group's odd last m-tile (at most 128 rows) is an
// M = 128 pair instead: CTA r takes its rows 64r .. 64r+63 (half_pair).
__device__ __forceinline__ TileCoord pair_unit(int32_t n_tiles, int32_t local, uint32_t rank,
                                               int32_t row0, int32_t row_end, bool tails) {
  TileCoord c;
  const int32_t p = local / n_tiles;
  c.n_tile = local - p * n_tiles;
  const int32_t m = (row_end - row0 + kBM - 1) / kBM;
  c.half_pair = (tails && (m & 1) && 2 * p == m - 1) ? 1 : 0;
  c.a_row0 = row0 + 2 * p * kBM + static_cast<int32_t>(rank) * (c.half_pair ? 64 : kBM);
  c.row_end = row_end;
  c.group = 0;
  return c;
}

template <bool kPair, bool kKG, bool kTwo = false>
__device__ __forceinline__ TileCoord unit_tile(const Args& a, int32_t u, uint32_t rank) {
  TileCoord c;
  if (kTwo) {
    // The first GEMM's units (gate_up), then the second's (down).
    const bool p2 = u >= a.fused_units1;
    const int32_t local = p2 ? u - a.fused_units1 : u;
    const int32_t nt = p2 ? a.n_tiles2 : a.n_tiles;
    const int32_t rows = p2 ? a.dense_rows2 : a.dense_rows;
    c = kPair ? pair_unit(nt, local, rank, 0, rows, false) : in_group_tile(nt, local, 0, rows);
    c.group = 0;
    c.k0 = 0;
    c.k_end = 0;
    c.k_blocks = p2 ? a.k_blocks2 : a.k_blocks;
    c.phase2 = p2 ? 1 : 0;
    return c;
  }
  c.phase2 = 0;
  if (kKG) {
    // Every group has the same output tiles (one-CTA tiles, or two-CTA units of m-tile
    // pairs); its K range is its row range.
    const int32_t gi = u / a.units_per_group;
    const int32_t local = u - gi * a.units_per_group;
    const int32_t g = a.group_order ? __ldg(a.group_order + gi) : gi;
    c = kPair ? pair_unit(a.n_tiles, local, rank, 0, a.dense_rows, false)
              : in_group_tile(a.n_tiles, local, 0, a.dense_rows);
    c.phase2 = 0;
    c.group = g;
    c.k0 = __ldg(a.k_group_offsets + g);
    c.k_end = __ldg(a.k_group_offsets + g + 1);
    c.k_blocks = c.k_end > c.k0 ? (c.k_end - c.k0 + kBK - 1) / kBK : 0;
    return c;
  }
  if (kPair) {
    // Dense, or grouped with a per-group prefix of two-CTA units.
    int32_t g = 0, row0 = 0, row_end = a.dense_rows, local = u;
    if (a.unit_offsets) {
      int32_t lo = 0, hi = a.num_groups - 1;
      while (lo < hi) {
        const int32_t mid = (lo + hi + 1) >> 1;
        if (__ldg(a.unit_offsets + mid) <= u) lo = mid; else hi = mid - 1;
      }
      g = lo;
      row0 = __ldg(a.group_offsets + g);
      row_end = __ldg(a.group_offsets + g + 1);
      local = u - __ldg(a.unit_offsets + g);
    }
    c = pair_unit(a.n_tiles, local, rank, row0, row_end, a.pair_tails != 0);
    c.group = g;
    c.phase2 = 0;
    c.k0 = 0;
    c.k_end = 0;
    c.k_blocks = a.k_blocks;
    return c;
  }
  c = decode_tile(a, u);
  c.phase2 = 0;
  c.k0 = 0;
  c.k_end = 0;
  c.k_blocks = a.k_blocks;
  return c;
}

// dh GEMM: whether the d(g, u) of a unit's chunks may leave as one TMA box store of the
// CTA's 128 rows: all of them inside the unit's group, or running past the tensor's last
// row (the store does not write those).  Half-pair tiles and CTAs without rows store
// from registers.
__device__ __forceinline__ bool gu_tma_out_rows(const TileCoord& c, bool hp, int32_t total_rows) {
  return !hp && c.a_row0 < c.row_end && (c.a_row0 + kBM <= c.row_end || c.row_end == total_rows);
}

// kCluster: acquire at cluster scope (a barrier the peer CTA arrives on).
template <bool kCluster = false>
__device__ __forceinline__ bool ctl_wait(SharedCtl* ctl, uint64_t* bar, uint32_t parity,
                                         uint32_t* status) {
  const uint32_t b = smem_u32(bar);
  auto try_wait = [&]() {
    return kCluster ? mbar_try_wait_cluster(b, parity) : mbar_try_wait(b, parity);
  };
  if (try_wait()) return true;
  const uint64_t t0 = global_timer_ns();
  uint32_t polls = 0;
  while (true) {
    if (try_wait()) return true;
    // Each try_wait may suspend the thread for a while: check the clock every few.
    if ((++polls & 7u) == 0u) {
      if (ctl->abort) return false;
      if (global_timer_ns() - t0 > ctl->wait_limit_ns) {
        record_status(status, SITU_ERR_TIMEOUT);
        ctl->abort = 1;
        return false;
      }
    }
  }
}

// Zero K rows kv..63 of a stage's MN-major operand tiles (2 A atoms, 4 B
// atoms): row k of a {64 MN, 64 K} 128-byte-swizzled atom is the 128 bytes at
// k * 128 (the swizzle permutes 16-byte pieces within a row), so the tail is one
// contiguous range per atom.  Warp-collective.
__device__ __forceinline__ void zero_k_tail(uint32_t sa, uint32_t sb, int32_t kv, int lane) {
  const uint32_t first = static_cast<uint32_t>(kv) * 128u;
  const uint32_t n = (kMnAtomBytes - first) / 16u;
#pragma unroll 1
  for (int at = 0; at < 6; ++at) {
    const uint32_t base = (at < 2 ? sa + at * kMnAtomBytes : sb + (at - 2) * kMnAtomBytes) + first;
    for (uint32_t i = lane; i < n; i += 32) st_shared_zero16(base + 16u * i);
  }
}

// Bounded wait (as ctl_wait) until the int32 at p reaches target (acquire).
__device__ __forceinline__ bool wait_count(SharedCtl* ctl, const int32_t* p, int32_t target,
                                           uint32_t* status) {
  if (ld_acquire_gpu(p) >= target) return true;
  const uint64_t t0 = global_timer_ns();
  uint32_t polls = 0;
  while (true) {
    __nanosleep(64);
    if (ld_acquire_gpu(p) >= target) return true;
    if ((++polls & 15u) == 0u) {
      if (ctl->abort) return false;
      if (global_timer_ns() - t0 > ctl->wait_limit_ns) {
        record_status(status, SITU_ERR_TIMEOUT);
        ctl->abort = 1;
        return false;
      }
    }
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Store up to 32 bf16 (16 packed words) of one row; columns >= n_valid are not
// written (n_valid is a multiple of 8, so a 16-byte piece is all in or all out).
__device__ __forceinline__ void store_row_chunk(__nv_bfloat16* dst, const uint32_t (&w)[16],
                                                int64_t col0, int64_t n_valid) {
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    if (col0 + 8 * v + 8 <= n_valid) {
      st_global_v4(dst + 8 * v, w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
    }
  }
}

// MXFP8 quantization of one block of 32 values given as bf16 (16 packed words,
// element 2i in the low half of word i), per the OCP MX conversion: scale
// 2^(floor(log2 amax) - 8), i.e. E8M0 code max(E - 8, 0) with E the biased exponent
// of the largest magnitude (zero and tiny blocks take the smallest scale 2^-127);
// each code is E4M3(v * 2^(127 - code)), an exact power-of-two scaling followed by
// one rounding to nearest even, clamped to 448.  Fills 8 words of codes (element
// 4j + b in byte b of word j) and returns the scale code.
__device__ __forceinline__ uint32_t mx_quantize32(const uint32_t (&w)[16], uint32_t (&q)[8]) {
  uint32_t amax = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = max(amax, max(w[i] & 0x7FFFu, (w[i] >> 16) & 0x7FFFu));
  const uint32_t e = amax >> 7;
  const uint32_t code = e > 8u ? e - 8u : 0u;
  const float inv = __uint_as_float((254u - code) << 23);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float v0 = __uint_as_float(w[2 * j] << 16) * inv;
    const float v1 = __uint_as_float(w[2 * j] & 0xFFFF0000u) * inv;
    const float v2 = __uint_as_float(w[2 * j + 1] << 16) * inv;
    const float v3 = __uint_as_float(w[2 * j + 1] & 0xFFFF0000u) * inv;
    q[j] = cvt_e4m3x2(v0, v1) | (cvt_e4m3x2(v2, v3) << 16);
  }
  return code;
}

// Byte offset of the scale of row r (r_in_tile = its row within its 128-row tile
// m_tile) and 32-wide block b in a 128-row scale-tile array with k_stages 128-wide
// K stages per tile.
__host__ __device__ __forceinline__ int64_t sf_tile_offset(int64_t m_tile, int64_t k_stages,
                                                           int32_t r_in_tile, int64_t b) {
  return (m_tile * k_stages + b / 4) * kSfTileBytes + (r_in_tile % 32) * 16 +
         (r_in_tile / 32) * 4 + (b % 4);
}

// kPair: clusters of two CTAs whose MMAs are tcgen05 cta_group::2 (M = 256 over the
// pair, or M = 128 for a grouped GEMM's half-pair tail); otherwise one CTA per tile
// with cta_group::1 MMAs.
template <Epi kEpi, Caps kC, bool kPair, bool kStoreGu, Major kMajor, int kMx = 0>
__global__ void __launch_bounds__(block_threads<kEpi, kMx>(), 1)
    ffn_gemm_kernel(const __grid_constant__ CUtensorMap map_a,
                    const __grid_constant__ CUtensorMap map_a64,
                    const __grid_constant__ CUtensorMap map_b,
                    const __grid_constant__ CUtensorMap map_a2,
                    const __grid_constant__ CUtensorMap map_a2_64,
                    const __grid_constant__ CUtensorMap map_b2, const Args args) {
  constexpr bool k2Cta = kPair;
  // The two-CTA dh GEMM stages the saved (g, u) through shared memory (a loader warp);
  // its one-CTA form reads them from global memory in the epilogue.
  constexpr bool kGuStage = k2Cta && kEpi == Epi::kSituBwd;
  using G = std::conditional_t<k2Cta,
                               std::conditional_t<kGuStage, GeoPairBwd, GeoPairT<kMx>>, Geo<kMx>>;
  constexpr uint32_t kGuBytes = kGuStage ? kGuSlots * kGuSlotBytes : 0u;
  static_assert(G::Stages * G::StageBytes + kGuBytes + sizeof(SharedCtl) + 1024 <= 232448,
                "shared memory per CTA");
  static_assert(!kMx || 2 * G::BN + kSfTmemCols * G::Stages <= kTmemCols,
                "accumulators and scale slots fit in tensor memory");
  static_assert(!kMx || kMajor == Major::kKMajor, "MXFP8 operands are K-major");
  static_assert(kMx || kEpi != Epi::kSituMx, "the MXFP8 epilogue needs MXFP8 GEMMs");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled operand buffers.
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  // Operand stages, then (dh GEMM) the (g, u) slots, then the control block.
  uint8_t* gu_smem = smem + G::Stages * G::StageBytes;
  SharedCtl* ctl = reinterpret_cast<SharedCtl*>(gu_smem + kGuBytes);
  constexpr bool kSituEpi = kEpi == Epi::kSitu || kEpi == Epi::kSituMx;
  constexpr bool kFfn = kEpi == Epi::kFfn;
  static_assert(!kFfn || kMajor == Major::kKMajor, "the one-launch FFN is K-major");
  // Two GEMMs in one launch: the one-launch FFN, or two independent plain GEMMs.
  constexpr bool kTwo = kFfn || kEpi == Epi::kPlain2;
  static_assert(kEpi != Epi::kPlain2 || (!kMx && kMajor != Major::kABMNGrouped),
                "two plain GEMMs: bf16, not K-grouped");

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  // Contractions over rows (both operands MN-major) may be K-grouped.
  constexpr bool kKG = kMajor == Major::kABMNGrouped;
  // A two-CTA M = 128 pair tile: a grouped bf16 GEMM's half-pair tail (K-major A; the
  // launch passes the 64-row B box map in map_b2, which only two-GEMM launches use
  // otherwise, and those have no half pairs).
  auto pair_half_tile = [](const TileCoord& c) {
    return k2Cta && kMx == 0 && !a_mn_major(kMajor) && c.half_pair != 0;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < G::Stages; ++s) {
      // Two-CTA MXFP8: the even CTA's own arrival and the odd CTA's relayed one.
      mbar_init(smem_u32(&ctl->full[s]), (k2Cta && kMx) ? 2 : 1);
      // Two-CTA: one commit of the even CTA frees the stage in both.
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    for (int b = 0; b < kAccBufs; ++b) {
      mbar_init(smem_u32(&ctl->acc_full[b]), 1);
      // Two-CTA: the even CTA's MMAs wait for both CTAs' epilogues.
      mbar_init(smem_u32(&ctl->acc_empty[b]), (k2Cta ? 2 : 1) * 32 * epi_warps<kEpi>());
    }
    mbar_init(smem_u32(&ctl->drain), 1);
    if (kMx) {
      for (int s = 0; s < G::Stages; ++s) mbar_init(smem_u32(&ctl->sf_ready[s]), 1);
      mbar_init(smem_u32(&ctl->sf_drain), 1);
    }
    if (kGuStage) {
      for (int s = 0; s < kGuSlots; ++s) {
        mbar_init(smem_u32(&ctl->gu_full[s]), 1);
        // Every thread of the column group that reads the slot.
        mbar_init(smem_u32(&ctl->gu_done[s]), 128);
      }
    }
    ctl->abort = 0;
    ctl->wait_limit_ns = args.wait_limit_ns;
    fence_mbar_init();
    tma_prefetch_map(&map_a);
    if (!kPair) tma_prefetch_map(&map_a64);
    tma_prefetch_map(&map_b);
    if (kTwo) {
      tma_prefetch_map(&map_a2);
      if (!kPair) tma_prefetch_map(&map_a2_64);
      tma_prefetch_map(&map_b2);
    }
    if (kGuStage) {
      // The dh GEMM's saved-(g, u) maps ride in the second-GEMM A slots, its d(g, u) map
      // in the 64-row B slot.
      tma_prefetch_map(&map_a2);
      tma_prefetch_map(&map_a2_64);
      tma_prefetch_map(&map_b2);
    }
  }
  if (warp == 1) {
    if constexpr (k2Cta) {
      tmem_alloc_pair(smem_u32(&ctl->tmem_base), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(&ctl->tmem_base), kTmemCols);
      tmem_relinquish();
    }
    tc_fence_before_sync();
  }
  __syncthreads();
  if (kPair) cluster_sync();  // the peer's barriers exist before any copy or MMA names them
  tc_fence_after_sync();
  const uint32_t tmem_base = ctl->tmem_base;
  const int32_t n_total = num_units<kPair, kKG, kTwo>(args);
  const int32_t u0 = kPair ? static_cast<int32_t>(blockIdx.x >> 1) : static_cast<int32_t>(blockIdx.x);
  const int32_t ustride = kPair ? static_cast<int32_t>(gridDim.x >> 1) : static_cast<int32_t>(gridDim.x);

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      uint32_t issued = 0;
      bool ok = true;
      int32_t last_group = -1;  // two-CTA K-grouped: the group whose maps were acquired
      (void)last_group;
      for (int32_t i = 0; i * ustride < n_total && ok; ++i) {
        const int32_t t = round_unit<kKG>(i, u0, ustride);
        if (t >= n_total) continue;
        const TileCoord tc = unit_tile<kPair, kKG, kTwo>(args, t, rank);
        const int64_t gbase = static_cast<int64_t>(tc.group) * args.b_group_rows;
        // Second-GEMM tiles read the second pair of operands (kFfn: h and W_down).
        const bool p2 = kTwo && tc.phase2;
        const CUtensorMap* pm_a = p2 ? &map_a2 : &map_a;
        const CUtensorMap* pm_a64 = p2 ? &map_a2_64 : &map_a64;
        const CUtensorMap* pm_b = p2 ? &map_b2 : &map_b;
        // Two-CTA K-grouped: the group's own maps, whose rows end at the group's end, so
        // that its last k-block reads zeros past it (a group ending before row
        // kMinGroupMapRows: maps based that many rows earlier, coordinates shifted).
        int32_t k_shift = 0;
        if constexpr (kKG && k2Cta) {
          if (tc.k_blocks > 0) {
            pm_a = args.group_maps + 2 * tc.group;
            pm_b = pm_a + 1;
            k_shift = group_map_shift(tc.k_end);
            if (tc.group != last_group) {
              fence_tensormap_acquire(pm_a);
              fence_tensormap_acquire(pm_b);
              last_group = tc.group;
            }
          }
        }
        const bool situ_tile = kSituEpi || (kFfn && !p2);
        constexpr bool kBMNp = kMajor != Major::kKMajor;
        // K-major B: a group's weights are b_group_rows further down the N rows.
        // MN-major B: they are b_group_rows further down the K rows (grouped by
        // rows), or the contraction itself starts at k0 (K-grouped).
        int32_t b_row0, b_row1, kb_off = 0;
        if (situ_tile) {
          b_row0 = static_cast<int32_t>(gbase + static_cast<int64_t>(tc.n_tile) * (G::BN / 2));
          b_row1 = static_cast<int32_t>(gbase + args.b_up_offset +
                                        static_cast<int64_t>(tc.n_tile) * (G::BN / 2));
        } else if (kBMNp) {
          b_row0 = tc.n_tile * G::BN;
          b_row1 = b_row0 + 128;
          kb_off = kKG ? tc.k0 : static_cast<int32_t>(gbase);
        } else {
          b_row0 = static_cast<int32_t>(gbase + static_cast<int64_t>(tc.n_tile) * G::BN);
          b_row1 = b_row0 + G::BHalfRows;
        }
        // MXFP8: the unit's scale tiles (A per global m-tile, B per (group, n-tile)).
        const uint8_t* sfa_unit = nullptr;
        const uint8_t* sfb_unit = nullptr;
        if constexpr (kMx) {
          // A two-CTA pair's m-tile past the rows has no scale tile: it reads its
          // partner's (its products are not stored).
          const int32_t a_row_sf =
              (k2Cta && tc.a_row0 >= tc.row_end) ? tc.a_row0 - kBM : tc.a_row0;
          const int32_t a_tile =
              args.tile_offsets ? __ldg(args.tile_offsets + tc.group) +
                                      (a_row_sf - __ldg(args.group_offsets + tc.group)) / kBM
                                : a_row_sf / kBM;
          const uint8_t* sfa = p2 ? args.sfa2 : args.sfa;
          const uint8_t* sfb = p2 ? args.sfb2 : args.sfb;
          const int32_t nt = p2 ? args.n_tiles2 : args.n_tiles;
          sfa_unit = sfa + static_cast<int64_t>(a_tile) * tc.k_blocks * kSfTileBytes;
          sfb_unit = sfb + (static_cast<int64_t>(tc.group) * nt + tc.n_tile) * tc.k_blocks *
                               kSfbStageBytes;
        }
        if (kFfn && p2 && tc.a_row0 < tc.row_end) {
          // The h rows of this tile's m-tile must be stored by every gate_up tile:
          // acquire the count, then order the TMA reads of h after it.  (A two-CTA
          // pair's m-tile past the rows has no count and loads only fill.)
          const int32_t mt = tc.a_row0 / kBM;
          if (!wait_count(ctl, args.h_ready + mt, args.h_ready_target, args.status)) {
            ok = false;
            break;
          }
          fence_proxy_async_all();
        }
        for (int32_t kb = 0; kb < tc.k_blocks; ++kb) {
          if (!ctl_wait(ctl, &ctl->empty[stage], phase ^ 1u, args.status)) {
            ok = false;
            break;
          }
          const uint32_t full = smem_u32(&ctl->full[stage]);
          const uint32_t sa = smem_u32(smem + stage * G::StageBytes);
          const uint32_t sb = sa + G::ABytes;
          if constexpr (k2Cta) {
            // This CTA's A rows and its half of B (K-major: one 128-row box; MN-major:
            // two {64, 64} atoms); both CTAs' copies count on the even CTA's barrier,
            // which expects them all.  An M = 128 pair (half_pair) stages 64 A rows per
            // CTA, and its SiTU tile's B half in CTA r is gate rows n0 + 64r .. +63 then
            // the matching up rows, so each accumulator lane pairs gate and up columns.
            const bool hp = pair_half_tile(tc);
            const uint32_t full0 = map_to_rank(full, 0);
            if (rank == 0) mbar_arrive_expect_tx(full, hp ? G::TxBytes - G::ABytes : G::TxBytes);
            const int32_t kxa = kb * G::BK + tc.k0 + k_shift, kxb2 = kb * G::BK + kb_off + k_shift;
            const int32_t brow = rank == 0 ? b_row0 : b_row1;
            if constexpr (a_mn_major(kMajor)) {
              for (int j = 0; j < 2; ++j)
                tma_load_2d_pair(sa + j * kMnAtomBytes, pm_a, tc.a_row0 + 64 * j, kxa, full0);
            } else {
              tma_load_2d_pair(sa, hp ? pm_a64 : pm_a, kxa, tc.a_row0, full0);
            }
            if constexpr (kMajor != Major::kKMajor) {
              for (int j = 0; j < 2; ++j)
                tma_load_2d_pair(sb + j * kMnAtomBytes, pm_b, brow + 64 * j, kxb2, full0);
            } else if (hp && situ_tile) {
              const int32_t off = 64 * static_cast<int32_t>(rank);
              tma_load_2d_pair(sb, &map_b2, kxb2, b_row0 + off, full0);
              tma_load_2d_pair(sb + 64 * 128, &map_b2, kxb2, b_row1 + off, full0);
            } else {
              tma_load_2d_pair(sb, pm_b, kxb2, brow, full0);
            }
            if constexpr (kMx) {
              // This CTA's own scale tiles: the even CTA's land on its full barrier,
              // the odd CTA's on its sf_ready barrier, from where they are relayed.
              const uint32_t ssf = sb + G::BBytes;
              uint32_t sf_bar = full;
              if (rank != 0) {
                sf_bar = smem_u32(&ctl->sf_ready[stage]);
                mbar_arrive_expect_tx(sf_bar, G::SfBytes);
              }
              bulk_load(ssf, sfa_unit + static_cast<int64_t>(kb) * kSfTileBytes, kSfTileBytes,
                        sf_bar);
              bulk_load(ssf + kSfTileBytes, sfb_unit + static_cast<int64_t>(kb) * kSfbStageBytes,
                        kSfbStageBytes, sf_bar);
            }
            ++issued;
            if (++stage == G::Stages) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          // A tile with at most 64 valid rows needs only A rows 0..63 (the 64-row MMA reads
          // no more; with MXFP8, rows 64..127 only feed output rows that are not stored):
          // one 64-row box, and the stage expects that many bytes less.
          const bool a_half = tc.row_end - tc.a_row0 <= 64;
          mbar_arrive_expect_tx(full, a_half ? G::TxBytes - G::ABytes / 2 : G::TxBytes);
          constexpr bool kAMN = a_mn_major(kMajor);
          constexpr bool kBMN = kMajor != Major::kKMajor;
          const int32_t kx = kb * G::BK + tc.k0;     // A's K coordinate
          const int32_t kxb = kb * G::BK + kb_off;   // B's K coordinate
          // A: rows a_row0 .. +127, or the first 64 of them (MN-major: one {64, 64} atom
          // per 64 rows; K-major: one 128-row box, or one 64-row box).
          if (kAMN) {
            for (int j = 0; j < (a_half ? 1 : 2); ++j)
              tma_load_2d(sa + j * kMnAtomBytes, pm_a, tc.a_row0 + 64 * j, kx, full);
          } else if (a_half) {
            tma_load_2d(sa, pm_a64, kx, tc.a_row0, full);
          } else {
            tma_load_2d(sa, pm_a, kx, tc.a_row0, full);
          }
          // B: two halves of BHalfRows rows (MN-major: two {64, 64} atoms each).
          constexpr uint32_t kBHalf = G::BHalfRows * 128;  // bytes of one B half
          for (int h = 0; h < 2; ++h) {
            const uint32_t dst = sb + h * kBHalf;
            const int32_t row = h == 0 ? b_row0 : b_row1;
            if (kBMN) {
              for (int j = 0; j < 2; ++j)
                tma_load_2d(dst + j * kMnAtomBytes, pm_b, row + 64 * j, kxb, full);
            } else {
              tma_load_2d(dst, pm_b, kxb, row, full);
            }
          }
          if constexpr (kMx) {
            // The stage's A and B scale tiles.
            const uint32_t ssf = sb + G::BBytes;
            bulk_load(ssf, sfa_unit + static_cast<int64_t>(kb) * kSfTileBytes, kSfTileBytes, full);
            bulk_load(ssf + kSfTileBytes, sfb_unit + static_cast<int64_t>(kb) * kSfbStageBytes,
                      kSfbStageBytes, full);
          }
          ++issued;
          if (++stage == G::Stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Two-CTA: the odd CTA's operand copies count on the even CTA's barriers, drained
      // there (the odd CTA leaves only after the even one, at the final cluster
      // barrier); its own MXFP8 scale copies land on its sf_ready barriers.
      const bool drain_sf = k2Cta && kMx && rank != 0;
      if (!ok && (!(k2Cta && rank != 0) || drain_sf)) {
        // Drain: wait (bounded) for the copies of the last stages issued.
        const uint32_t n = issued < G::Stages ? issued : G::Stages;
        for (uint32_t i = 0; i < n; ++i) {
          stage = (stage + G::Stages - 1) % G::Stages;
          if (stage == G::Stages - 1) phase ^= 1u;
          mbar_wait(smem_u32(drain_sf ? &ctl->sf_ready[stage] : &ctl->full[stage]), phase,
                    nullptr, kDrainLimitNs);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    // Lane 0 waits and issues.  One-CTA K-grouped contractions run the whole warp: the
    // last k-block of a group holds the next group's first rows (or fill) past
    // k_end, and the warp zeroes those K rows of both operands before the MMAs (two-CTA:
    // the group's tensor maps end at k_end, so those rows arrive as zeros).
    // Two-CTA: the even CTA's thread issues the pair's MMAs; the odd CTA's MMA warp idles.
    constexpr bool kWarpZero = kKG && !k2Cta;
    if ((kWarpZero || lane == 0) && (!k2Cta || rank == 0)) {
      uint32_t stage = 0, phase = 0;
      uint32_t local = 0;
      bool ok = true;
      auto wait = [&](uint64_t* bar, uint32_t par) {
        int w = 1;
        if (lane == 0) w = ctl_wait(ctl, bar, par, args.status) ? 1 : 0;
        if (kWarpZero) w = __shfl_sync(0xFFFFFFFFu, w, 0);
        return w != 0;
      };
      for (int32_t i = 0; i * ustride < n_total && ok; ++i) {
        const int32_t t = round_unit<kKG>(i, u0, ustride);
        if (t >= n_total) continue;
        const uint32_t acc = local & 1u;
        const uint32_t acc_phase = (local >> 1) & 1u;
        if (!wait(&ctl->acc_empty[acc], acc_phase ^ 1u)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * G::BN;
        const TileCoord tcm = unit_tile<kPair, kKG, kTwo>(args, t, rank);
        const uint32_t idesc = kMx      ? idesc_mxf8(k2Cta ? 2 * kBM : kBM, G::BN,
                                                kMx == 2 ? kMxE2M1 : kMxE4M3)
                               : (k2Cta ? idesc_bf16_f32(pair_half_tile(tcm) ? kBM : 2 * kBM, G::BN)
                                        : (tcm.row_end - tcm.a_row0 <= 64 ? kIdescHalf : kIdesc)) |
                                         (a_mn_major(kMajor) ? kAMnBit : 0u) |
                                         (kMajor != Major::kKMajor ? kBMnBit : 0u);
        for (int32_t kb = 0; kb < tcm.k_blocks; ++kb) {
          // MXFP8: the scale warp signals once the stage's data and scales are in.
          if (!wait(kMx ? &ctl->sf_ready[stage] : &ctl->full[stage], phase)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t sa = smem_u32(smem + stage * G::StageBytes);
          const uint32_t sb = sa + G::ABytes;
          if (kWarpZero) {
            const int32_t kv = tcm.k_end - (tcm.k0 + kb * G::BK);
            if (kv < G::BK) {
              zero_k_tail(sa, sb, kv, lane);
              fence_proxy_async_smem();
            }
            __syncwarp();
          }
          if (kMx && lane == 0) {
            // Four K=32 block-scaled MMAs, the k-th reading byte k of the stage's
            // scales in its TMEM slot (A: 4 columns, B: 8).
            const uint32_t sf_t = tmem_base + 2 * G::BN + kSfTmemCols * stage;
#pragma unroll
            for (int k = 0; k < G::BK / G::UK; ++k) {
              if constexpr (k2Cta) {
                umma_mxf8_pair(d_tmem, sw128_kmajor_desc(sa + k * 32),
                               sw128_kmajor_desc(sb + k * 32), idesc | idesc_mxf8_ids(k, k), sf_t,
                               sf_t + 4, (kb | k) != 0 ? 1u : 0u);
              } else {
                umma_mxf8(d_tmem, sw128_kmajor_desc(sa + k * 32), sw128_kmajor_desc(sb + k * 32),
                          idesc | idesc_mxf8_ids(k, k), sf_t, sf_t + 4, (kb | k) != 0 ? 1u : 0u);
              }
            }
            if constexpr (k2Cta) {
              umma_commit_pair(smem_u32(&ctl->empty[stage]), 0x3);
            } else {
              umma_commit(smem_u32(&ctl->empty[stage]));
            }
          } else if (lane == 0) {
#pragma unroll
            for (int k = 0; k < kBK / kUK; ++k) {
              // K-major: 16 K elements = 32 bytes along the row; MN-major: 16 K
              // rows = 2048 bytes.
              const uint64_t ad = a_mn_major(kMajor)
                                      ? sw128_mnmajor_desc(sa + k * 2048, kMnAtomBytes)
                                      : sw128_kmajor_desc(sa + k * kUK * 2);
              const uint64_t bd = kMajor != Major::kKMajor
                                      ? sw128_mnmajor_desc(sb + k * 2048, kMnAtomBytes)
                                      : sw128_kmajor_desc(sb + k * kUK * 2);
              if constexpr (k2Cta) umma_bf16_pair(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
              else umma_bf16(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
            }
            if constexpr (k2Cta) {
              umma_commit_pair(smem_u32(&ctl->empty[stage]), 0x3);
            } else {
              umma_commit(smem_u32(&ctl->empty[stage]));
            }
          }
          if (++stage == G::Stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        // A group without rows issues no MMA: the commit arrives at once and the
        // epilogue writes zeros.
        if (lane == 0) {
          if constexpr (k2Cta) umma_commit_pair(smem_u32(&ctl->acc_full[acc]), 0x3);
          else umma_commit(smem_u32(&ctl->acc_full[acc]));
        }
        ++local;
      }
      if (!ok && lane == 0) {
        // Drain the MMAs already issued before the tensor memory is freed.
        if constexpr (k2Cta) umma_commit_pair(smem_u32(&ctl->drain), 0x1);
        else umma_commit(smem_u32(&ctl->drain));
        mbar_wait(smem_u32(&ctl->drain), 0, nullptr, kDrainLimitNs);
      }
    }
  } else if (kMx && warp == 2 + epi_warps<kEpi>()) {
    // ---------------- scale copier (MXFP8) ----------------
    // Per stage, once its copies landed: the A and B scale tiles into the stage's
    // TMEM slot, then a commit that tells the MMA warp.  A slot is rewritten only
    // after its stage was refilled, i.e. after the MMAs that read it completed.
    // Two-CTA: the even CTA's copies move both CTAs' scale tiles, each into its own
    // CTA's tensor memory, once the even CTA's full barrier has seen both CTAs' codes,
    // its own scales and the odd CTA's relay; the odd CTA's warp is that relay: once its
    // own scale tiles of a stage have landed it arrives on the even CTA's full barrier.
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      const bool relay = k2Cta && rank != 0;
      for (int32_t i = 0; i * ustride < n_total && ok; ++i) {
        const int32_t t = round_unit<kKG>(i, u0, ustride);
        if (t >= n_total) continue;
        const TileCoord tcs = unit_tile<kPair, kKG, kTwo>(args, t, rank);
        for (int32_t kb = 0; kb < tcs.k_blocks; ++kb) {
          const bool landed = relay ? ctl_wait(ctl, &ctl->sf_ready[stage], phase, args.status)
                                    : ctl_wait<k2Cta>(ctl, &ctl->full[stage], phase, args.status);
          if (!landed) {
            ok = false;
            break;
          }
          if (relay) {
            mbar_arrive_remote(map_to_rank(smem_u32(&ctl->full[stage]), 0));
          } else {
            tc_fence_after_sync();
            const uint32_t ssf = smem_u32(smem + stage * G::StageBytes) + G::ABytes + G::BBytes;
            const uint32_t sf_t = tmem_base + 2 * G::BN + kSfTmemCols * stage;
            if constexpr (k2Cta) {
              tmem_cp_32x128b_x4_pair(sf_t, ssf);
              tmem_cp_32x128b_x4_pair(sf_t + 4, ssf + kSfTileBytes);
              tmem_cp_32x128b_x4_pair(sf_t + 8, ssf + 2 * kSfTileBytes);
              umma_commit_pair(smem_u32(&ctl->sf_ready[stage]), 0x1);
            } else {
              tmem_cp_32x128b_x4(sf_t, ssf);
              tmem_cp_32x128b_x4(sf_t + 4, ssf + kSfTileBytes);
              tmem_cp_32x128b_x4(sf_t + 8, ssf + 2 * kSfTileBytes);
              umma_commit(smem_u32(&ctl->sf_ready[stage]));
            }
          }
          if (++stage == G::Stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && !relay) {
        // Drain the copies already issued before the tensor memory is freed.
        if constexpr (k2Cta) umma_commit_pair(smem_u32(&ctl->sf_drain), 0x1);
        else umma_commit(smem_u32(&ctl->sf_drain));
        mbar_wait(smem_u32(&ctl->sf_drain), 0, nullptr, kDrainLimitNs);
      }
    }
  } else if (kGuStage && warp == 2 + epi_warps<kEpi>()) {
    // ---------------- saved (g, u) loader and d(g, u) storer (two-CTA dh GEMM) ----------
    // For each unit, the epilogue's 32-column chunks in the order in which the two
    // column groups of epilogue warps take them (group 0's first chunk, group 1's
    // first, group 0's second, ...), each copied into the next slot.  A slot takes this
    // CTA's rows of the chunk (an M = 128 pair: slot rows 0..63 are the CTA's 64 rows at
    // the tile's column offset 0, rows 64..127 the same rows at offset 128, the columns
    // of the accumulator lanes 64..127).  A CTA whose rows all lie past its group's end
    // (the idle half of a group's last pair) loads nothing and only arrives.
    // The epilogue writes a chunk's d(g, u) over its (g, u) in the slot when the chunk's
    // box may be stored whole (gu_tma_out); this warp then stores the slot to dgu with
    // TMA before it copies the slot's next chunk in.  Other chunks' d(g, u) the epilogue
    // stores itself, releasing the slot as soon as it has read it.
    if (lane == 0) {
      uint32_t seq = 0;  // chunks issued
      bool ok = true;
      const int32_t split = static_cast<int32_t>(args.split);
      int32_t out_x[kGuSlots], out_y[kGuSlots];  // pending TMA store of a slot (y < 0: none)
      for (int q = 0; q < kGuSlots; ++q) {
        out_x[q] = 0;
        out_y[q] = -1;
      }
      // Waits until the epilogue is done with chunk sq, then stores its d(g, u) if the
      // epilogue left them in the slot; the slot is free once the store has read it.
      auto retire = [&](uint32_t sq) {
        const uint32_t slot = sq % kGuSlots;
        if (!ctl_wait(ctl, &ctl->gu_done[slot], (sq / kGuSlots) & 1u, args.status)) return false;
        if (out_y[slot] >= 0) {
          const uint32_t src = smem_u32(gu_smem + slot * kGuSlotBytes);
          tma_store_2d(&map_b2, src, out_x[slot], out_y[slot]);
          tma_store_2d(&map_b2, src + kGuHalfBytes, split + out_x[slot], out_y[slot]);
          bulk_commit_group();
          bulk_wait_group_read<0>();
          out_y[slot] = -1;
        }
        return true;
      };
      for (int32_t i = 0; i * ustride < n_total && ok; ++i) {
        const int32_t t = round_unit<kKG>(i, u0, ustride);
        if (t >= n_total) continue;
        const TileCoord tc = unit_tile<kPair, kKG, kTwo>(args, t, rank);
        const bool hp = pair_half_tile(tc);
        const bool rows = tc.a_row0 < tc.row_end;
        const bool out_rows = gu_tma_out_rows(tc, hp, args.dense_rows);
        constexpr int kGroups = epi_col_groups<kEpi>();
        const int per_group = (hp ? 4 : 8) / kGroups;
        const int32_t col_base = tc.n_tile * G::BN;
        for (int j = 0; j < per_group && ok; ++j) {
          for (int cg = 0; cg < kGroups; ++cg, ++seq) {
            if (seq >= static_cast<uint32_t>(kGuSlots) && !retire(seq - kGuSlots)) {
              ok = false;
              break;
            }
            const uint32_t slot = seq % kGuSlots;
            const uint32_t full = smem_u32(&ctl->gu_full[slot]);
            if (!rows) {
              mbar_arrive(full);
              continue;
            }
            mbar_arrive_expect_tx(full, kGuSlotBytes);
            const uint32_t dst = smem_u32(gu_smem + slot * kGuSlotBytes);
            const int32_t x = col_base + (cg * per_group + j) * 32;
            if (hp) {
              for (int h = 0; h < 2; ++h) {
                tma_load_2d(dst + h * (kGuHalfBytes / 2), &map_a2_64, x + 128 * h, tc.a_row0,
                            full);
                tma_load_2d(dst + kGuHalfBytes + h * (kGuHalfBytes / 2), &map_a2_64,
                            split + x + 128 * h, tc.a_row0, full);
              }
            } else {
              tma_load_2d(dst, &map_a2, x, tc.a_row0, full);
              tma_load_2d(dst + kGuHalfBytes, &map_a2, split + x, tc.a_row0, full);
            }
            if (out_rows && x + 32 <= args.n_out) {
              out_x[slot] = x;
              out_y[slot] = tc.a_row0;
            }
          }
        }
      }
      // The last chunks' stores.
      for (uint32_t sq = seq > static_cast<uint32_t>(kGuSlots) ? seq - kGuSlots : 0u;
           ok && sq < seq; ++sq)
        ok = retire(sq);
      if (!ok || ctl->abort) {
        // Aborted: wait (bounded) for the copies of the last slots issued, which land in
        // this CTA's shared memory, before the CTA may leave.
        const uint32_t n = seq < static_cast<uint32_t>(kGuSlots) ? seq : kGuSlots;
        for (uint32_t k = 1; k <= n; ++k) {
          const uint32_t sq = seq - k;
          mbar_wait(smem_u32(&ctl->gu_full[sq % kGuSlots]), (sq / kGuSlots) & 1u, nullptr,
                    kDrainLimitNs);
        }
      }
      bulk_wait_group<0>();  // the stores' writes are performed
    }
  } else if (warp >= 2 && warp < 2 + epi_warps<kEpi>()) {
    // ---------------- epilogue (warps 2 .. 2 + epi_warps - 1) ----------------
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    // With 8 epilogue warps, warps 2..5 take the first half of the tile's 32-column
    // chunks and warps 6..9 the second half.
    const int col_group = (warp - 2) >> 2;
    const int row_in_tile = quarter * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t local = 0;
    uint32_t gseq = 0;  // dh GEMM: (g, u) chunks of the units before this one
    for (int32_t i = 0; i * ustride < n_total; ++i, ++local) {
      const int32_t t = round_unit<kKG>(i, u0, ustride);
      if (t >= n_total) {
        --local;  // no unit this round
        continue;
      }
      const uint32_t acc = local & 1u;
      const uint32_t acc_phase = (local >> 1) & 1u;
      int ok = 1;
      if (lane == 0) ok = ctl_wait(ctl, &ctl->acc_full[acc], acc_phase, args.status) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      tc_fence_after_sync();
      const TileCoord tc = unit_tile<kPair, kKG, kTwo>(args, t, rank);
      const bool p2 = kTwo && tc.phase2;
      // M=64 tiles (bf16 only): only the first 16 lanes of each quarter hold rows
      // (16q + lane).
      const bool half = !kMx && !k2Cta && tc.row_end - tc.a_row0 <= 64;
      // Two-CTA M = 128 pair: lane L holds this CTA's row L mod 64, accumulator columns
      // 0..127 being the tile's columns 128 (L div 64) .. +127 (lh).
      const bool hp = pair_half_tile(tc);
      const int lh = hp ? (row_in_tile >> 6) : 0;
      const int32_t row =
          tc.a_row0 + (half ? quarter * 16 + lane : hp ? (row_in_tile & 63) : row_in_tile);
      bool valid = row < tc.row_end && (!half || lane < 16);
      int64_t out_row = row;
      // K-grouped: group g's result starts at output row g * out_group_rows; a
      // group without rows has a zero result.
      bool zero = false;
      if (kKG) {
        out_row += static_cast<int64_t>(tc.group) * args.out_group_rows;
        zero = tc.k_blocks == 0;
      }
      if (valid && args.out_row_index) {
        out_row = __ldg(args.out_row_index + row);
        valid = out_row >= 0 && out_row < args.out_rows;
      }
      const uint32_t t_acc = tmem_base + lane_addr + acc * G::BN;
      if (kSituEpi || (kFfn && !p2)) {
        // Gate column j of the tile pairs with up column BN/2 + j (a half pair: the
        // lane's 64 gate columns, then their 64 up columns, are the activation's
        // columns 64 lh .. +63 of the tile).
        constexpr int kHalfN = G::BN / 2;
        const int pair_cols = hp ? 64 : kHalfN;
        __nv_bfloat16* dst_row = args.out + out_row * args.ldo;
        int64_t h_tile = 0;
        if constexpr (kEpi == Epi::kSituMx || (kFfn && kMx != 0)) {
          h_tile = args.tile_offsets
                       ? __ldg(args.tile_offsets + tc.group) +
                             (tc.a_row0 - __ldg(args.group_offsets + tc.group)) / kBM
                       : tc.a_row0 / kBM;
        }
#pragma unroll 1
        for (int c = 0; c < pair_cols / 32; ++c) {
          __syncwarp();  // tcgen05.ld is warp-collective (.sync.aligned)
          uint32_t g[32], u[32];
          tmem_ld32(t_acc + c * 32, g);
          tmem_ld32(t_acc + pair_cols + c * 32, u);
          tmem_ld_wait2(g, u);
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            w[i] = pack_bf16x2(
                situ_act<kC>(__uint_as_float(g[2 * i]), __uint_as_float(u[2 * i]), args.sp),
                situ_act<kC>(__uint_as_float(g[2 * i + 1]), __uint_as_float(u[2 * i + 1]),
                             args.sp));
          }
          const int64_t col0 = static_cast<int64_t>(tc.n_tile) * kHalfN + lh * 64 + c * 32;
          if constexpr (kEpi == Epi::kSituMx || (kFfn && kMx != 0)) {
            // h rounded to bf16 (w), then one 32-wide MXFP8 block: 32 codes and the
            // block's scale in the A-operand scale tiles of the next GEMM.
            if (valid && col0 < args.n_out) {
              uint32_t q[8];
              const uint32_t sc = mx_quantize32(w, q);
              uint8_t* dst = args.h_codes + out_row * args.ldo + col0;
              st_global_v4(dst, q[0], q[1], q[2], q[3]);
              st_global_v4(dst + 16, q[4], q[5], q[6], q[7]);
              args.h_sf[sf_tile_offset(h_tile, args.n_out / 128, row - tc.a_row0, col0 / 32)] =
                  static_cast<uint8_t>(sc);
            }
          } else {
            if (valid) store_row_chunk(dst_row + col0, w, col0, args.n_out);
          }
          if (kStoreGu && valid) {
            // Pre-activation (g, u) for the backward pass, bf16.
            uint32_t wg[16], wu[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              wg[i] = pack_bf16x2(__uint_as_float(g[2 * i]), __uint_as_float(g[2 * i + 1]));
              wu[i] = pack_bf16x2(__uint_as_float(u[2 * i]), __uint_as_float(u[2 * i + 1]));
            }
            __nv_bfloat16* gu_row = args.gu_store + out_row * 2 * args.split;
            store_row_chunk(gu_row + col0, wg, col0, args.n_out);
            store_row_chunk(gu_row + args.split + col0, wu, col0, args.n_out);
          }
        }
        if (kFfn) {
          // Publish this tile's h rows: each epilogue thread orders its stores, the
          // epilogue warps meet, and one release add counts the tile for its m-tile (a
          // two-CTA pair's m-tile past the rows stores nothing and does not count).
          __threadfence();
          named_barrier_sync(1, kEpiThreads);
          if (threadIdx.x == 64 && tc.n_tile < args.n_tiles && tc.a_row0 < tc.row_end)
            red_release_add_gpu(args.h_ready + tc.a_row0 / kBM, 1);
        }
      } else if (kGuStage) {
        // The saved (g, u) of each chunk come from the slot the loader filled: this
        // thread's slot row is its accumulator lane.  It reads its 64 bytes of g and of
        // u and forms d(g, u).  A chunk whose box leaves by TMA store (the loader's) gets
        // d(g, u) written over (g, u) in the slot before the slot is released; otherwise
        // the slot is released as soon as it is read and d(g, u) is stored from registers.
        __nv_bfloat16* dgu_row = args.dgu_out + static_cast<int64_t>(row) * 2 * args.split;
        const int64_t col_base = static_cast<int64_t>(tc.n_tile) * G::BN + lh * 128;
        const int chunks = (hp ? 4 : 8) / epi_col_groups<kEpi>();  // this warp's chunks
        const bool out_rows = gu_tma_out_rows(tc, hp, args.dense_rows);
        const uint32_t srow = static_cast<uint32_t>(row_in_tile) * 64u;
        const uint32_t swz = static_cast<uint32_t>((row_in_tile >> 1) & 3);
        bool gu_ok = true;
#pragma unroll 1
        for (int j = 0; j < chunks; ++j) {
          const uint32_t seq = gseq + epi_col_groups<kEpi>() * j + col_group;
          const uint32_t slot = seq % kGuSlots, par = (seq / kGuSlots) & 1u;
          int w = 1;
          if (lane == 0) w = ctl_wait(ctl, &ctl->gu_full[slot], par, args.status) ? 1 : 0;
          w = __shfl_sync(0xFFFFFFFFu, w, 0);
          if (!w) {
            gu_ok = false;
            break;
          }
          // Each lane's own acquire of the landed bytes (the phase is complete: one try).
          (void)mbar_try_wait(smem_u32(&ctl->gu_full[slot]), par);
          const int c = col_group * chunks + j;
          __syncwarp();  // tcgen05.ld is warp-collective
          uint32_t a[32];
          tmem_ld32(t_acc + c * 32, a);
          const uint32_t sg = smem_u32(gu_smem + slot * kGuSlotBytes) + srow;
          uint4 gq[4], uq[4];
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const uint32_t piece = 16u * (static_cast<uint32_t>(v) ^ swz);
            gq[v] = ld_shared_v4(sg + piece);
            uq[v] = ld_shared_v4(sg + kGuHalfBytes + piece);
          }
          const int64_t col0 = col_base + c * 32;
          const bool tma_out = out_rows && col0 + 32 <= args.n_out;
          const uint32_t done = smem_u32(&ctl->gu_done[slot]);
          if (!tma_out) mbar_arrive(done);
          tmem_ld_wait(a);
          // Rows past the tensor's end (a dense GEMM's last tile) compute nothing; the
          // TMA store does not write them.
          if (valid) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const int64_t cv = col0 + 8 * v;
              if (!tma_out && cv + 8 > args.n_out) continue;
              const uint32_t gw[4] = {gq[v].x, gq[v].y, gq[v].z, gq[v].w};
              const uint32_t uw[4] = {uq[v].x, uq[v].y, uq[v].z, uq[v].w};
              uint32_t og[4], ou[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                uint64_t dg2, du2;
                situ_act_grad_x2<kC>(__uint_as_float(gw[e] << 16),
                                     __uint_as_float(gw[e] & 0xFFFF0000u),
                                     __uint_as_float(uw[e] << 16),
                                     __uint_as_float(uw[e] & 0xFFFF0000u),
                                     f2_pack(__uint_as_float(a[8 * v + 2 * e]),
                                             __uint_as_float(a[8 * v + 2 * e + 1])),
                                     args.sp, dg2, du2);
                float lo, hi;
                f2_unpack(dg2, lo, hi);
                og[e] = pack_bf16x2(lo, hi);
                f2_unpack(du2, lo, hi);
                ou[e] = pack_bf16x2(lo, hi);
              }
              if (tma_out) {
                const uint32_t piece = 16u * (static_cast<uint32_t>(v) ^ swz);
                st_shared_v4(sg + piece, og[0], og[1], og[2], og[3]);
                st_shared_v4(sg + kGuHalfBytes + piece, ou[0], ou[1], ou[2], ou[3]);
              } else {
                st_global_v4(dgu_row + cv, og[0], og[1], og[2], og[3]);
                st_global_v4(dgu_row + args.split + cv, ou[0], ou[1], ou[2], ou[3]);
              }
            }
          }
          if (tma_out) {
            // The slot's d(g, u) are visible to the loader's TMA store once it has seen
            // every thread's arrival.
            fence_proxy_async_smem();
            mbar_arrive(done);
          }
        }
        gseq += static_cast<uint32_t>(epi_col_groups<kEpi>() * chunks);
        if (!gu_ok) break;
      } else if (kEpi == Epi::kSituBwd) {
        const __nv_bfloat16* gu_row = args.gu_in + static_cast<int64_t>(row) * 2 * args.split;
        __nv_bfloat16* dgu_row = args.dgu_out + static_cast<int64_t>(row) * 2 * args.split;
        // The saved (g, u) of a 32-column chunk are loaded one chunk ahead, through the
        // read-only path: loaded in the loop, each 16-byte load would wait behind the
        // previous stores (whose asm carries a memory clobber) and the tile's epilogue
        // would serialise 32 global-load latencies.
        uint4 gq[4], uq[4];
        // A half pair's lane holds 128 columns (4 chunks) starting at column 128 lh.
        const int64_t col_base = static_cast<int64_t>(tc.n_tile) * G::BN + lh * 128;
        auto load_gu = [&](int c, uint4 (&gd)[4], uint4 (&ud)[4]) {
          const int64_t col0 = col_base + c * 32;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const int64_t cv = col0 + 8 * v;
            if (valid && cv + 8 <= args.n_out) {
              gd[v] = __ldg(reinterpret_cast<const uint4*>(gu_row + cv));
              ud[v] = __ldg(reinterpret_cast<const uint4*>(gu_row + args.split + cv));
            } else {
              gd[v] = make_uint4(0, 0, 0, 0);
              ud[v] = make_uint4(0, 0, 0, 0);
            }
          }
        };
        constexpr int kChunks = 8 / (epi_warps<kEpi>() / 4);  // chunks per warp
        const int chunks = hp ? kChunks / 2 : kChunks;
        const int c_begin = col_group * chunks, c_end = c_begin + chunks;
        load_gu(c_begin, gq, uq);
#pragma unroll 1
        for (int c = c_begin; c < c_end; ++c) {
          uint4 gn[4], un[4];
          if (c + 1 < c_end) load_gu(c + 1, gn, un);
          __syncwarp();
          uint32_t a[32];
          tmem_ld32(t_acc + c * 32, a);
          tmem_ld_wait(a);
          const int64_t col0 = col_base + c * 32;
          if (valid) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const int64_t cv = col0 + 8 * v;
              if (cv + 8 > args.n_out) continue;
              const uint32_t gw[4] = {gq[v].x, gq[v].y, gq[v].z, gq[v].w};
              const uint32_t uw[4] = {uq[v].x, uq[v].y, uq[v].z, uq[v].w};
              uint32_t og[4], ou[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                uint64_t dg2, du2;
                situ_act_grad_x2<kC>(__uint_as_float(gw[i] << 16),
                                     __uint_as_float(gw[i] & 0xFFFF0000u),
                                     __uint_as_float(uw[i] << 16),
                                     __uint_as_float(uw[i] & 0xFFFF0000u),
                                     f2_pack(__uint_as_float(a[8 * v + 2 * i]),
                                             __uint_as_float(a[8 * v + 2 * i + 1])),
                                     args.sp, dg2, du2);
                float lo, hi;
                f2_unpack(dg2, lo, hi);
                og[i] = pack_bf16x2(lo, hi);
                f2_unpack(du2, lo, hi);
                ou[i] = pack_bf16x2(lo, hi);
              }
              st_global_v4(dgu_row + cv, og[0], og[1], og[2], og[3]);
              st_global_v4(dgu_row + args.split + cv, ou[0], ou[1], ou[2], ou[3]);
            }
          }
          if (c + 1 < c_end) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              gq[v] = gn[v];
              uq[v] = un[v];
            }
          }
        }
      } else {
        const int64_t n_out = p2 ? args.n_out2 : args.n_out;
        __nv_bfloat16* dst_row = p2 ? args.out2 + out_row * args.ldo2 : args.out + out_row * args.ldo;
#pragma unroll 1
        for (int c = 0; c < (hp ? G::BN / 64 : G::BN / 32); ++c) {
          __syncwarp();
          uint32_t a[32];
          tmem_ld32(t_acc + c * 32, a);
          tmem_ld_wait(a);
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            w[i] = zero ? 0u
                        : pack_bf16x2(__uint_as_float(a[2 * i]), __uint_as_float(a[2 * i + 1]));
          }
          const int64_t col0 = static_cast<int64_t>(tc.n_tile) * G::BN + lh * 128 + c * 32;
          if (kEpi == Epi::kPlain && args.combine_w) {
            // Fused combine: FP32 atomic adds of the weighted row (order-dependent
            // rounding).
            if (valid) {
              const float wr = __ldg(args.combine_w + out_row);
              float* dst = args.combine_out + (out_row / args.combine_k) * n_out + col0;
#pragma unroll
              for (int v = 0; v < 8; ++v) {
                if (col0 + 4 * v + 4 <= n_out)
                  red_add_v4_f32(dst + 4 * v, wr * __uint_as_float(a[4 * v]),
                                 wr * __uint_as_float(a[4 * v + 1]), wr * __uint_as_float(a[4 * v + 2]),
                                 wr * __uint_as_float(a[4 * v + 3]));
              }
            }
          } else if (valid) {
            store_row_chunk(dst_row + col0, w, col0, n_out);
          }
        }
      }
      tc_fence_before_sync();
      // Two-CTA: the accumulator is free once both CTAs' epilogues have read it; they
      // arrive on the even CTA's barrier, where its MMA thread waits.
      if (k2Cta && rank != 0)
        mbar_arrive_remote(map_to_rank(smem_u32(&ctl->acc_empty[acc]), 0));
      else
        mbar_arrive(smem_u32(&ctl->acc_empty[acc]));
    }
  }

  __syncthreads();
  if (k2Cta && ctl->abort) {
    // Aborted: let this CTA's copies that complete on the peer's barriers land.
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < kAbortLingerNs) __nanosleep(1000);
  }
  // Paired: neither CTA leaves while the peer may still write into it.
  if (kPair) cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    if constexpr (k2Cta) tmem_dealloc_pair(tmem_base, kTmemCols);
    else tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  // Resolved once; the static's initialisation is thread-safe.
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

// 2-D map over a row-major [rows, cols] matrix -- elem 0: bf16 (64 x box_rows
// boxes); 1: bytes (MXFP8 codes, 128 x box_rows); 2: packed 4-bit codes (128 x
// box_rows, two a byte in memory, unpacked to 16-byte chunks) -- 128 bytes a box row in
// shared memory, 128-byte swizzle (the layout sw128_kmajor_desc describes), zero fill
// out of bounds.  ld: row stride in elements (0 = cols).
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols,
              uint32_t box_rows = 128, int64_t ld = 0, int elem = 0) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode_fn();
  if (!enc) return false;
  const int64_t ldv = ld > 0 ? ld : cols;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(elem == 0 ? ldv * 2 : elem == 1 ? ldv : ldv / 2)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(elem == 0 ? 64 : 128), box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType type = elem == 0   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                   : elem == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                               : CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B;
  CUresult r = enc(m, type, 2, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D map over the saved pre-activation pair, bf16 [rows, cols] row-major (cols = 2 *
// split: g columns, then u columns): {32 columns, box_rows} boxes, 64 bytes a box row
// in shared memory with the 64-byte swizzle (16-byte piece v of box row r lands at
// piece v ^ ((r >> 1) & 3)), zero fill out of bounds.
bool make_map_gu(CUtensorMap* m, const void* base, int64_t rows, int64_t cols,
                 uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * 2)};
  cuuint32_t box[2] = {32, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Per-group copies of two tensor maps over row-major [K rows, cols] operands (the
// MN-major operands of a K-grouped contraction, at base_a and base_b with row pitches
// ld_a and ld_b bytes) whose rows end at the group's end, k_offsets[g + 1]: a copy of
// the group's last k-block then reads zeros past the group's end instead of the next
// group's rows.  Thread g writes out[2g] (from ta) and out[2g + 1] (from tb).  The
// device-written extent is at least kMinGroupMapRows rows (the driver encodes smaller
// extents differently from what the replacement writes): a group ending before that
// row gets a map of kMinGroupMapRows rows whose base lies kMinGroupMapRows - end rows
// before the operand's, and its loads add that many rows to their row coordinate
// (group_map_shift); they never reach below the group's first row.  A group without
// rows keeps the templates.
__global__ void group_maps_kernel(const __grid_constant__ CUtensorMap ta,
                                  const __grid_constant__ CUtensorMap tb, const uint8_t* base_a,
                                  const uint8_t* base_b, int64_t ld_a, int64_t ld_b,
                                  const int32_t* k_offsets, int32_t groups, CUtensorMap* out) {
  const int32_t g = static_cast<int32_t>(blockIdx.x * blockDim.x + threadIdx.x);
  if (g >= groups) return;
  const int32_t k0 = __ldg(k_offsets + g), k_end = __ldg(k_offsets + g + 1);
  out[2 * g] = ta;
  out[2 * g + 1] = tb;
  if (k_end > k0 && k0 >= 0) {
    const int32_t shift = group_map_shift(k_end);
    if (shift > 0) {
      tensormap_set_base(out + 2 * g, base_a - shift * ld_a);
      tensormap_set_base(out + 2 * g + 1, base_b - shift * ld_b);
    }
    tensormap_set_rows(out + 2 * g, k_end + shift);
    tensormap_set_rows(out + 2 * g + 1, k_end + shift);
  }
  fence_tensormap_release();
}

template <int kMx>
constexpr size_t smem_bytes() {
  return Geo<kMx>::Stages * Geo<kMx>::StageBytes + sizeof(SharedCtl) + 1024;
}
// Shared memory of the two-CTA kernels (the pair geometry).
template <int kMx = 0>
constexpr size_t smem_bytes_pair() {
  return GeoPairT<kMx>::Stages * GeoPairT<kMx>::StageBytes + sizeof(SharedCtl) + 1024;
}
// Shared memory of a two-CTA kernel of epilogue kEpi: the dh GEMM's five stages and
// (g, u) slots, or the pair geometry's stages.
template <Epi kEpi, int kMx = 0>
constexpr size_t smem_bytes_pair_epi() {
  return kEpi == Epi::kSituBwd ? GeoPairBwd::Stages * GeoPairBwd::StageBytes +
                                     kGuSlots * kGuSlotBytes + sizeof(SharedCtl) + 1024
                               : smem_bytes_pair<kMx>();
}
static_assert(smem_bytes_pair_epi<Epi::kSituBwd>() <= 232448, "shared memory per CTA");
static_assert(smem_bytes<1>() <= 232448 && smem_bytes<2>() <= 232448 &&
                  smem_bytes<0>() <= 232448 && smem_bytes_pair<0>() <= 232448 &&
                  smem_bytes_pair<1>() <= 232448 && smem_bytes_pair<2>() <= 232448,
              "shared memory per CTA");

// Most 2-CTA clusters of the two-CTA kernel ffn_gemm_kernel<kEpi, kC, true, ...>
// resident at once, per device (0 if the query fails: the one-CTA kernel is used
// then).  Cached per device as the count + 1 (0: not queried yet); threads that race
// on the first call each query and store the same value.
template <Epi kEpi, Caps kC, bool kStoreGu, Major kMajor, int kMx>
int max_pair_clusters(size_t smem) {
  static std::atomic<int> cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int c = cached[dev].load(std::memory_order_acquire);
  if (c == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(block_threads<kEpi, kMx>(), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    // The query counts the dynamic shared memory against the kernel's opt-in limit:
    // raise it first (it may not have been launched yet).
    auto fn = ffn_gemm_kernel<kEpi, kC, true, kStoreGu, kMajor, kMx>;
    if (!(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem)) == cudaSuccess &&
          cudaOccupancyMaxActiveClusters(&n, fn, &cfg) == cudaSuccess)) {
      (void)cudaGetLastError();
      n = 0;
    }
    c = n + 1;
    cached[dev].store(c, std::memory_order_release);
  }
  return c - 1;
}

// k2Cta: a dense (ungrouped) call runs the two-CTA MMA kernel when 2-CTA clusters fit.
template <Epi kEpi, Caps kC, bool kStoreGu = false, Major kMajor = Major::kKMajor,
          int kMx = 0, bool k2Cta = false>
cudaError_t launch(const GemmShape& s, const SituParams& p, uint32_t* status, int num_sms,
                   cudaStream_t stream) {
  using G = Geo<kMx>;
  constexpr size_t kSmem = smem_bytes<kMx>();
  static_assert(kEpi != Epi::kSitu || kMajor == Major::kKMajor,
                "the SiTU epilogue pairs gate and up rows of a K-major B");
  if (s.a_rows == 0 && !s.tile_offsets) return cudaSuccess;
  if (kMx && (!s.sfa || !s.sfb || s.K % G::BK != 0)) return cudaErrorInvalidValue;
  if ((s.k_group_offsets != nullptr) != (kMajor == Major::kABMNGrouped))
    return cudaErrorInvalidValue;
  CUtensorMap ma, ma64, mb;
  bool ok;
  if (a_mn_major(kMajor)) {
    // A stored [K, rows]: {64 rows, 64 K} boxes.
    ok = make_map(&ma, s.a, s.K, s.a_rows, 64, s.a_ld);
    ma64 = ma;
  } else {
    ok = make_map(&ma, s.a, s.a_rows, s.K, 128, s.a_ld, kMx ? 1 : 0) &&
         make_map(&ma64, s.a, s.a_rows, s.K, 64, s.a_ld, kMx ? 1 : 0);
  }
  if (kMajor != Major::kKMajor) {
    // B stored [K, N]; grouped by rows, the groups' K-row blocks are stacked.
    const int64_t b_k_rows =
        (s.group_offsets && !s.k_group_offsets) ? s.b_group_rows * s.num_groups : s.K;
    ok = ok && make_map(&mb, s.b, b_k_rows, s.b_rows, 64, s.b_ld);
  } else {
    ok = ok && make_map(&mb, s.b, s.b_rows, s.K, G::BHalfRows, s.b_ld, kMx);
  }
  if (!ok) return cudaErrorInvalidValue;
  Args a{};
  a.num_groups = s.num_groups;
  a.group_offsets = s.group_offsets;
  a.tile_offsets = s.tile_offsets;
  a.unit_offsets = nullptr;
  a.dense_rows = static_cast<int32_t>(s.a_rows);
  const int64_t out_cols_per_tile =
      (kEpi == Epi::kSitu || kEpi == Epi::kSituMx) ? G::BN / 2 : G::BN;
  a.n_tiles = static_cast<int32_t>((s.n_out + out_cols_per_tile - 1) / out_cols_per_tile);
  a.k_blocks = static_cast<int32_t>((s.K + G::BK - 1) / G::BK);
  a.b_group_rows = s.b_group_rows;
  a.b_up_offset = s.b_up_offset;
  a.n_out = s.n_out;
  a.out = static_cast<__nv_bfloat16*>(s.out);
  a.ldo = s.ldo;
  a.out_rows = s.out_rows;
  a.out_row_index = s.out_row_index;
  a.sp = p;
  a.status = status;
  a.wait_limit_ns = wait_limit_ns();
  a.gu_store = static_cast<__nv_bfloat16*>(s.gu_store);
  a.gu_in = static_cast<const __nv_bfloat16*>(s.gu_in);
  a.dgu_out = static_cast<__nv_bfloat16*>(s.dgu_out);
  a.split = s.split;
  a.k_group_offsets = s.k_group_offsets;
  a.group_order = s.group_order;
  a.out_group_rows = s.out_group_rows;
  a.units_per_group = 0;
  a.sfa = static_cast<const uint8_t*>(s.sfa);
  a.sfb = static_cast<const uint8_t*>(s.sfb);
  a.h_codes = static_cast<uint8_t*>(s.h_codes);
  a.h_sf = static_cast<uint8_t*>(s.h_sf);
  a.combine_w = s.combine_w;
  a.combine_out = static_cast<float*>(s.combine_out);
  a.combine_k = s.combine_k > 0 ? s.combine_k : 1;
  const int64_t m_tiles = (s.a_rows + kBM - 1) / kBM;
  // The shared-memory opt-in is a per-device property of each kernel: set once (threads
  // racing on the first call each set it; the flag is published after the settings).
  static std::atomic<bool> smem_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!smem_set[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(ffn_gemm_kernel<kEpi, kC, false, kStoreGu, kMajor, kMx>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmem));
    if (e != cudaSuccess) return e;
    if constexpr (k2Cta) {
      e = cudaFuncSetAttribute(ffn_gemm_kernel<kEpi, kC, true, kStoreGu, kMajor, kMx>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem_bytes_pair_epi<kEpi, kMx>()));
      if (e != cudaSuccess) return e;
    }
    smem_set[dev].store(true, std::memory_order_release);
  }
  if constexpr (k2Cta) {
    // Two-CTA MMA for a dense call, a grouped call whose unit prefix counts two-CTA
    // units (pair_units), or a K-grouped contraction.
    const bool dense = !s.group_offsets && !s.tile_offsets && !s.k_group_offsets &&
                       !s.out_row_index && !s.combine_w;
    const bool kgrouped = kMajor == Major::kABMNGrouped && s.k_group_offsets && s.group_maps;
    const bool use2 = dense || kgrouped || (s.pair_units && s.unit_offsets && !s.k_group_offsets);
    int clusters2 =
        use2 ? max_pair_clusters<kEpi, kC, kStoreGu, kMajor, kMx>(
                   smem_bytes_pair_epi<kEpi, kMx>())
             : 0;
    if (s.pair_units && clusters2 == 0) return cudaErrorNotSupported;
    if (clusters2 > 0) {
      // Unit (p, n) gives CTA r m-tile 2p + r of n-tile n (of its group).  Grouped bf16
      // GEMMs with K-major A run each group's odd last m-tile as an M = 128 pair (64
      // rows per CTA); its SiTU B halves are 64-row boxes (the map in the second-GEMM
      // slot, unused by one-GEMM launches).
      a.unit_offsets = s.pair_units ? s.unit_offsets : nullptr;
      CUtensorMap mb64 = mb;
      if (kMx == 0 && !a_mn_major(kMajor) && s.pair_units) {
        a.pair_tails = 1;
        if (kMajor == Major::kKMajor &&
            !make_map(&mb64, s.b, s.b_rows, s.K, 64, s.b_ld, 0))
          return cudaErrorInvalidValue;
      }
      // The dh GEMM: maps over the saved (g, u) for its loader warp (128- and 64-row
      // boxes) in the second-GEMM slots, and over d(g, u) for its TMA stores in the
      // 64-row B slot (its B is never a SiTU tile's).
      CUtensorMap mg = ma, mg64 = ma64;
      if (kEpi == Epi::kSituBwd &&
          !(make_map_gu(&mg, s.gu_in, s.a_rows, 2 * s.split, 128) &&
            make_map_gu(&mg64, s.gu_in, s.a_rows, 2 * s.split, 64) &&
            make_map_gu(&mb64, s.dgu_out, s.a_rows, 2 * s.split, 128)))
        return cudaErrorInvalidValue;
      if (dense) {
        const int64_t units = ((m_tiles + 1) / 2) * a.n_tiles;
        if (units < clusters2) clusters2 = static_cast<int>(units);
      } else if (kgrouped) {
        // Every group: units (p, n) over the output's m-tile pairs and n-tiles; its own
        // A and B maps end at the group's last row.
        a.units_per_group = static_cast<int32_t>(((m_tiles + 1) / 2) * a.n_tiles);
        const int64_t units = static_cast<int64_t>(a.units_per_group) * s.num_groups;
        if (units < clusters2) clusters2 = static_cast<int>(units < 1 ? 1 : units);
        a.group_maps = static_cast<const CUtensorMap*>(s.group_maps);
        group_maps_kernel<<<(s.num_groups + 127) / 128, 128, 0, stream>>>(
            ma, mb, static_cast<const uint8_t*>(s.a), static_cast<const uint8_t*>(s.b),
            (s.a_ld > 0 ? s.a_ld : s.a_rows) * 2, (s.b_ld > 0 ? s.b_ld : s.b_rows) * 2,
            s.k_group_offsets, s.num_groups, static_cast<CUtensorMap*>(s.group_maps));
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
      }
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * clusters2, 1, 1);
      cfg.blockDim = dim3(block_threads<kEpi, kMx>(), 1, 1);
      cfg.dynamicSmemBytes = smem_bytes_pair_epi<kEpi, kMx>();
      cfg.stream = stream;
      cudaLaunchAttribute attr;
      attr.id = cudaLaunchAttributeClusterDimension;
      attr.val.clusterDim.x = 2;
      attr.val.clusterDim.y = 1;
      attr.val.clusterDim.z = 1;
      cfg.attrs = &attr;
      cfg.numAttrs = 1;
      return cudaLaunchKernelEx(&cfg, ffn_gemm_kernel<kEpi, kC, true, kStoreGu, kMajor, kMx>,
                                ma, ma64, mb, mg, mg64, mb64, a);
    }
  }
  // One CTA per tile, persistent: tiles in (group, m-tile, n-tile) order (K-grouped:
  // every group has the same m_tiles x n_tiles output tiles).
  int grid = num_sms;
  if (s.k_group_offsets) {
    a.units_per_group = static_cast<int32_t>(m_tiles * a.n_tiles);
    const int64_t units = m_tiles * a.n_tiles * s.num_groups;
    if (units < grid) grid = static_cast<int>(units < 1 ? 1 : units);
  } else if (!s.tile_offsets) {
    const int64_t tiles = m_tiles * a.n_tiles;
    if (tiles < grid) grid = static_cast<int>(tiles);
  }
  ffn_gemm_kernel<kEpi, kC, false, kStoreGu, kMajor, kMx>
      <<<grid, block_threads<kEpi, kMx>(), kSmem, stream>>>(ma, ma64, mb, ma, ma64, mb, a);
  return cudaGetLastError();
}

// The dense FFN in one persistent launch (Epi::kFfn): s_gu describes the gate_up
// GEMM (A = x, B = W_gate_up, out = h), s_dn the down GEMM (A = h, B = W_down, out = y);
// h_ready: one int32 per 128-row m-tile, zeroed here.  Every CTA must be resident at
// once (down tiles wait for gate_up tiles of other CTAs), so the launch is cooperative:
// a grid that cannot be co-resident fails to launch instead of waiting.
template <Caps kC, int kMx = 0>
cudaError_t launch_ffn_fused_impl(const GemmShape& s_gu, const GemmShape& s_dn,
                                  const SituParams& p, int32_t* h_ready, uint32_t* status,
                                  int num_sms, cudaStream_t stream) {
  using G = Geo<kMx>;
  // The cluster kernel is the two-CTA MMA one (its N, BK and B half match Geo<kMx>).
  static_assert(GeoPairT<kMx>::BN == G::BN && GeoPairT<kMx>::BK == G::BK &&
                    GeoPairT<kMx>::BHalfRows == G::BHalfRows,
                "tile geometry of the two-CTA kernel");
  // One opt-in size serves the two-CTA kernel and the one-CTA fallback.
  constexpr size_t kSmem = smem_bytes_pair<kMx>() > smem_bytes<kMx>() ? smem_bytes_pair<kMx>()
                                                                       : smem_bytes<kMx>();
  if (s_gu.a_rows == 0) return cudaSuccess;
  if (kMx && (!s_gu.sfa || !s_gu.sfb || !s_gu.h_codes || !s_gu.h_sf || !s_dn.sfa || !s_dn.sfb ||
              s_gu.K % G::BK != 0 || s_dn.K % G::BK != 0))
    return cudaErrorInvalidValue;
  // bf16: 64-element boxes; MXFP8: 128-byte boxes of codes (B: packed 4-bit for MXFP4).
  const int ea = kMx ? 1 : 0, eb = kMx == 2 ? 2 : ea;
  CUtensorMap ma, ma64, mb, ma2, ma2_64, mb2;
  if (!make_map(&ma, s_gu.a, s_gu.a_rows, s_gu.K, 128, 0, ea) ||
      !make_map(&ma64, s_gu.a, s_gu.a_rows, s_gu.K, 64, 0, ea) ||
      !make_map(&mb, s_gu.b, s_gu.b_rows, s_gu.K, G::BHalfRows, 0, eb) ||
      !make_map(&ma2, s_dn.a, s_dn.a_rows, s_dn.K, 128, 0, ea) ||
      !make_map(&ma2_64, s_dn.a, s_dn.a_rows, s_dn.K, 64, 0, ea) ||
      !make_map(&mb2, s_dn.b, s_dn.b_rows, s_dn.K, G::BHalfRows, 0, eb))
    return cudaErrorInvalidValue;
  const int64_t m_tiles = (s_gu.a_rows + kBM - 1) / kBM;
  cudaError_t e = cudaMemsetAsync(h_ready, 0, static_cast<size_t>(m_tiles) * 4, stream);
  if (e != cudaSuccess) return e;
  Args a{};
  a.num_groups = 1;
  a.dense_rows = static_cast<int32_t>(s_gu.a_rows);
  a.n_tiles = static_cast<int32_t>((s_gu.n_out + G::BN / 2 - 1) / (G::BN / 2));
  a.k_blocks = static_cast<int32_t>((s_gu.K + G::BK - 1) / G::BK);
  a.b_group_rows = s_gu.b_group_rows;
  a.b_up_offset = s_gu.b_up_offset;
  a.n_out = s_gu.n_out;
  a.out = static_cast<__nv_bfloat16*>(s_gu.out);
  a.ldo = s_gu.ldo;
  a.out_rows = s_gu.a_rows;
  a.sp = p;
  a.status = status;
  a.wait_limit_ns = wait_limit_ns();
  a.combine_k = 1;
  a.sfa = static_cast<const uint8_t*>(s_gu.sfa);
  a.sfb = static_cast<const uint8_t*>(s_gu.sfb);
  a.h_codes = static_cast<uint8_t*>(s_gu.h_codes);
  a.h_sf = static_cast<uint8_t*>(s_gu.h_sf);
  a.sfa2 = static_cast<const uint8_t*>(s_dn.sfa);
  a.sfb2 = static_cast<const uint8_t*>(s_dn.sfb);
  a.n_tiles2 = static_cast<int32_t>((s_dn.n_out + G::BN - 1) / G::BN);
  a.k_blocks2 = static_cast<int32_t>((s_dn.K + G::BK - 1) / G::BK);
  a.n_out2 = s_dn.n_out;
  a.out2 = static_cast<__nv_bfloat16*>(s_dn.out);
  a.ldo2 = s_dn.ldo;
  a.h_ready = h_ready;
  a.h_ready_target = a.n_tiles;
  a.dense_rows2 = a.dense_rows;
  static std::atomic<bool> smem_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!smem_set[dev].load(std::memory_order_acquire)) {
    for (auto fn : {ffn_gemm_kernel<Epi::kFfn, kC, false, false, Major::kKMajor, kMx>,
                    ffn_gemm_kernel<Epi::kFfn, kC, true, false, Major::kKMajor, kMx>}) {
      if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(kSmem))) != cudaSuccess)
        return e;
    }
    smem_set[dev].store(true, std::memory_order_release);
  }
  const int clusters = max_pair_clusters<Epi::kFfn, kC, false, Major::kKMajor, kMx>(kSmem);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeCooperative;
  attrs[0].val.cooperative = 1;
  cfg.blockDim = dim3(block_threads<Epi::kFfn, kMx>(), 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cfg.attrs = attrs;
  if (clusters > 0) {
    const int32_t mt = static_cast<int32_t>(m_tiles);
    a.fused_units1 = ((mt + 1) / 2) * a.n_tiles;
    a.fused_units2 = ((mt + 1) / 2) * a.n_tiles2;
    attrs[1].id = cudaLaunchAttributeClusterDimension;
    attrs[1].val.clusterDim.x = 2;
    attrs[1].val.clusterDim.y = 1;
    attrs[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    return cudaLaunchKernelEx(&cfg,
                              ffn_gemm_kernel<Epi::kFfn, kC, true, false, Major::kKMajor, kMx>,
                              ma, ma64, mb, ma2, ma2_64, mb2, a);
  }
  a.fused_units1 = static_cast<int32_t>(m_tiles) * a.n_tiles;
  a.fused_units2 = static_cast<int32_t>(m_tiles) * a.n_tiles2;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(num_sms, 1, 1);
  return cudaLaunchKernelEx(&cfg, ffn_gemm_kernel<Epi::kFfn, kC, false, false, Major::kKMajor, kMx>,
                            ma, ma64, mb, ma2, ma2_64, mb2, a);
}

// Two independent plain GEMMs of one operand layout in one persistent launch
// (Epi::kPlain2): the units of s1, then those of s2.  No CTA waits on another.
template <Major kMajor>
cudaError_t launch_plain2_impl(const GemmShape& s1, const GemmShape& s2, uint32_t* status,
                               int num_sms, cudaStream_t stream) {
  constexpr size_t kSmem = smem_bytes<0>();
  static_assert(smem_bytes<0>() == smem_bytes_pair<0>(), "one opt-in size for both kernels");
  static_assert(kMajor != Major::kABMNGrouped, "not K-grouped");
  if (s1.a_rows == 0 || s2.a_rows == 0) return cudaErrorInvalidValue;
  CUtensorMap ma, ma64, mb, ma2, ma2_64, mb2;
  auto maps = [&](const GemmShape& s, CUtensorMap* a, CUtensorMap* a64, CUtensorMap* b) {
    bool ok;
    if (a_mn_major(kMajor)) {
      ok = make_map(a, s.a, s.K, s.a_rows, 64, s.a_ld);
      *a64 = *a;
    } else {
      ok = make_map(a, s.a, s.a_rows, s.K, 128, s.a_ld) &&
           make_map(a64, s.a, s.a_rows, s.K, 64, s.a_ld);
    }
    if (kMajor != Major::kKMajor) return ok && make_map(b, s.b, s.K, s.b_rows, 64, s.b_ld);
    return ok && make_map(b, s.b, s.b_rows, s.K, 128, s.b_ld);
  };
  if (!maps(s1, &ma, &ma64, &mb) || !maps(s2, &ma2, &ma2_64, &mb2)) return cudaErrorInvalidValue;
  Args a{};
  a.num_groups = 1;
  a.dense_rows = static_cast<int32_t>(s1.a_rows);
  a.dense_rows2 = static_cast<int32_t>(s2.a_rows);
  a.n_tiles = static_cast<int32_t>((s1.n_out + kBN - 1) / kBN);
  a.k_blocks = static_cast<int32_t>((s1.K + kBK - 1) / kBK);
  a.n_out = s1.n_out;
  a.out = static_cast<__nv_bfloat16*>(s1.out);
  a.ldo = s1.ldo;
  a.out_rows = s1.a_rows;
  a.status = status;
  a.wait_limit_ns = wait_limit_ns();
  a.combine_k = 1;
  a.n_tiles2 = static_cast<int32_t>((s2.n_out + kBN - 1) / kBN);
  a.k_blocks2 = static_cast<int32_t>((s2.K + kBK - 1) / kBK);
  a.n_out2 = s2.n_out;
  a.out2 = static_cast<__nv_bfloat16*>(s2.out);
  a.ldo2 = s2.ldo;
  const int32_t m1 = static_cast<int32_t>((s1.a_rows + kBM - 1) / kBM);
  const int32_t m2 = static_cast<int32_t>((s2.a_rows + kBM - 1) / kBM);
  static std::atomic<bool> smem_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaError_t e;
  if (!smem_set[dev].load(std::memory_order_acquire)) {
    for (auto fn : {ffn_gemm_kernel<Epi::kPlain2, Caps::kBoth, false, false, kMajor, 0>,
                    ffn_gemm_kernel<Epi::kPlain2, Caps::kBoth, true, false, kMajor, 0>}) {
      if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(kSmem))) != cudaSuccess)
        return e;
    }
    smem_set[dev].store(true, std::memory_order_release);
  }
  // Pairs of CTAs run two-CTA MMAs (unit (p, n): CTA r takes m-tile 2p + r).
  int clusters = max_pair_clusters<Epi::kPlain2, Caps::kBoth, false, kMajor, 0>(kSmem);
  if (clusters > 0) {
    a.fused_units1 = ((m1 + 1) / 2) * a.n_tiles;
    a.fused_units2 = ((m2 + 1) / 2) * a.n_tiles2;
    const int32_t units = a.fused_units1 + a.fused_units2;
    if (units < clusters) clusters = units;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(block_threads<Epi::kPlain2, 0>(), 1, 1);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg,
                              ffn_gemm_kernel<Epi::kPlain2, Caps::kBoth, true, false, kMajor, 0>,
                              ma, ma64, mb, ma2, ma2_64, mb2, a);
  }
  a.fused_units1 = m1 * a.n_tiles;
  a.fused_units2 = m2 * a.n_tiles2;
  int grid = num_sms;
  if (a.fused_units1 + a.fused_units2 < grid) grid = a.fused_units1 + a.fused_units2;
  ffn_gemm_kernel<Epi::kPlain2, Caps::kBoth, false, false, kMajor, 0>
      <<<grid, block_threads<Epi::kPlain2, 0>(), kSmem, stream>>>(ma, ma64, mb, ma2, ma2_64, mb2,
                                                                   a);
  return cudaGetLastError();
}

}  // namespace
}  // namespace situ
