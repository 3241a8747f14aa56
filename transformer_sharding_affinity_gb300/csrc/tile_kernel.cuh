// tile_kernel.cuh -- parameters shared by the tcgen05 tile kernel and its host launcher.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "scales.cuh"

namespace aff {

// A job of the tile kernel stages, per K block of 64 fp16 elements (128-byte
// rows), three 128-row tiles, and runs one N = 256 MMA per K slice.  Head
// passes (FO, ADD, LOO): A = 128 interleaved gate / up weight rows of 64
// neurons, B = 256 tokens.  Fold: A = the same 128 weight rows, B = 256
// columns of gamma*Wo^T (its hi part, then its lo part, along K).  Alpha, x',
// c_h, ||b_gk||^2: A = the third tile (tokens; neurons for ||b_gk||^2), B = the
// first two.  Gate / up weights (W16, M16) are stored in
// groups of 16 neurons: 16 gate rows, then the same neurons' 16 up rows.
constexpr int kBlockM = 128;      // rows per tile (TMEM lanes)
constexpr int kBlockN = 128;      // TMEM columns per tile of the accumulator
constexpr int kBlockK = 64;       // fp16 elements per K block (one 128 B swizzle row)
constexpr int kTileBytes = kBlockM * kBlockK * 2;     // 16 KB
constexpr int kStageBytes = 3 * kTileBytes;           // three tiles = 48 KB
// Epilogue warps: 8 (two per TMEM lane quarter), or 16 (four per lane
// quarter) for the x' pass of the down edge and the two leave-one-out passes:
// the x' and c_h passes wait on loads of x and the LOO pass on its heavier
// per-token arithmetic, all latency-bound with 8 (LOO 2.09 ms with 16 warps,
// 2.98 ms with 8).  The block is one TMA warp, one MMA warp and the epilogue
// warps.
constexpr int kWideEpiWarps = 16;
constexpr int kEpiWarps = 8;
constexpr __host__ __device__ int epi_warps(int mode) {
  return (mode == 4 || mode == 6 || mode == 7) ? kWideEpiWarps : kEpiWarps;
}
constexpr __host__ __device__ int block_threads(int mode) { return 64 + 32 * epi_warps(mode); }
// FO / ADD / LOO units: sets of 256 tokens per unit (one partial sum per unit)
constexpr int kHeadSets = 2;
constexpr int kTmemCols = 512;                        // 2 accumulator buffers x 256 columns
constexpr int kUnitRing = 4;                          // unit ids the TMA warp publishes ahead of the others
constexpr int kMaxDynSmem = 232448;                   // 227 KB opt-in limit per block

enum TileMode : int {
  kModeFold = 0,   // M_h = Wg/Wu * diag(gamma) * Wo^(h)   -> fp16 [H][2 I_pad][dh], interleaved rows
  kModeFO = 1,     // per (512 tokens, 64 neurons): operating point, then every head's Delta^2
  kModeADD = 2,    // per (512 tokens, 64 neurons): every head's (p.w^g)^2 + (p.w^u)^2
  kModeAlpha = 3,  // per token tile: alpha = silu(g) u  -> fp16 [T_pad][I_pad]
  kModeXPrime = 4, // x' = x + alpha Wd^T per (token tile, 256 columns d): partial sums of x'^2
  kModeQNorm = 5,  // ||b_gk||^2 = sum over group g's q/k/v rows r of ((Wqkv' diag(gamma'))_r . w^d_k)^2
  kModeCNorm = 6,  // per (token tile, 256 columns d), every head h: c_h/r = (a_h/r) Wo^(h)^T; sums of (c/r)^2, x (c/r)
  kModeLOO = 7     // per (512 tokens, 64 neurons): g, u, then every head's exact leave-one-out change
};

struct TileParams {
  int32_t mode;
  int32_t unit0;           // first unit of this launch (a pass may be split over launches)
  int32_t n_units;         // one past the last unit
  int32_t stages;
  int32_t T, D, H, G, dh, I, I_pad, T_pad;
  int32_t n_ktiles;        // neuron tiles of 128 (I_pad / 128); head passes: blocks of 64 = 2 n_ktiles
  int32_t n_ttiles;        // token tiles of 128 (T_pad / 128)
  int32_t tiles_per_unit;  // token tiles per alpha unit
  int32_t n_ntiles;        // fold: column tiles of 256 over H*dh; x', c_h: tiles of 256 over D; qnorm: row tiles of 256 per group
  int32_t rows_per_group;  // qnorm: (H/G + 2) * dh
  int32_t nkb_D, nkb_dh, nkb_I;
  int32_t ls_D, ls_dh;     // 16-wide K slices in the last K block of D and of dh
  int32_t stream_heads;    // FO / ADD / LOO: 1 = the heads' K ranges are streamed back to back
                           // (d_head % 16 == 0 but not % 64): M16 is [2 I_pad][H*dh], a16 read as [T][H*dh]
  int32_t nkb_HD, ls_HD;   // streaming: K blocks over H*dh, 16-wide slices in the last one
  int32_t spp;             // streaming: 16-wide K slices per head (d_head / 16)
  uint32_t* status;
  uint32_t* ucount;        // when set, CTAs claim units from this counter (zero at launch) instead of
                           // taking every gridDim-th unit; each unit writes its own slots either way
  float* partial;          // FO/ADD/LOO: [H][I_pad / 64][n_chunks][column group][64]; x': [column tile][group][T_pad]
  __half* M16;             // fold output
  __half* alpha16;         // alpha output
  const uint16_t* x_bf16;  // x' epilogue reads x (bf16 bits) [T][D]
  float* inv_rp2;          // x' output 1/r'^2 [T_pad]
  float* bnorm;            // qnorm output [I_pad][G]
  const float* rho;        // LOO: sigma = 1 - r / rms(x - c_h), [H][T_pad]
  const DevScales* sc;     // maxima that fix the power-of-two scales of the fp16 operands
  float eps;
};

}  // namespace aff
