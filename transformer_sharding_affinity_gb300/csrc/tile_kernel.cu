// tile_kernel.cu -- the persistent tcgen05 kernel behind every dense
// contraction of the affinity pass ("Affinity-Aware Sharding for Delayed
// Tensor Parallelism", §3 "Affinity scores").
//
// One CTA per SM (227 KB of shared memory, all 512 TMEM columns).  Warp
// roles:
//   warp 0       TMA producer: a ring of `stages` 48 KB stages, each holding
//                three 128 x 64 tiles (fp16, 128 B swizzle);
//   warp 1       MMA issuer (one thread): for every K slice of 16 one
//                tcgen05.mma with M = 128 and N = 256 (two of the tiles back
//                to back) into an fp32 accumulator of 256 TMEM columns.
//                Two accumulator buffers alternate so the epilogue of one job
//                overlaps the MMAs of the next;
//   warps 2..    epilogue: TMEM -> registers with tcgen05.ld; warp w reads
//                TMEM lanes 32*(w%4)..+31 and one column group (w-2)/4.
// FO / ADD / LOO: A = 128 weight rows of 64 neurons, in groups of 16 per lane
// quarter: lanes 32q..32q+15 hold the gate rows (g, or p.w^g) of neurons
// 16q..16q+15 and lanes 32q+16..32q+31 their up rows; B = 256 tokens.  The
// epilogue reads them with the 16x32bx2 TMEM shape: thread l and thread l + 16
// of a warp both get neuron 16q + l's gate and up values, for the first and
// the second half of the warp's columns, so the sum over tokens stays within
// a thread.  The fold: A = the same 128 weight rows, B = 256 columns of
// gamma*Wo^T.  The alpha, x', c_h and ||b_gk||^2 passes: A = the third tile
// (tokens, or neurons), B = the first two.
// Work is a fixed list of units, each a short list of jobs.  The TMA warp
// picks a CTA's next unit -- every gridDim-th, except that in the head passes
// the last two rounds are claimed from a counter, so that CTAs on faster SMs
// take more of them -- and publishes its id through a small shared-memory ring
// that the MMA thread and the epilogue warps read in order.  Which CTA computes a unit never changes
// its result, and every unit writes its own partial sums, so the outputs do
// not depend on the grid size or on which CTA claimed what.
#include "launch.cuh"
#include "sm103_primitives.cuh"
#include "tile_kernel.cuh"

#include <cuda_fp16.h>

namespace aff {

enum JobKind : int {
  kJobGateUp = 0, kJobHead = 1, kJobFold = 2, kJobXPrime = 3, kJobQNorm = 4, kJobCNorm = 5,
  kJobStream = 6   // producer / MMA view of all H head jobs of a 256-token set, K ranges back to back
};

struct Job {
  int kind;
  int nkb;       // K blocks of 64 in the job
  int nkb_part;  // K blocks per part (fold / qnorm run the K range twice: hi then lo)
  int last_nks;  // 16-wide K slices in the last block of a part
  int head;      // head index (kJobHead)
  int t0;        // first token
  int kt;        // neuron tile of 128 (fold, alpha) or block of 64 (head passes)
  int nt;        // column / row tile
  int g;         // KV group (qnorm)
};

struct Unit {
  int njobs;     // jobs as the epilogue sees them
  int njobs_pm;  // jobs as the producer and the MMA issuer see them (fewer when heads are streamed)
  int chunk;    // FO/ADD/LOO/alpha: token chunk index
  int kt;       // as Job::kt; cnorm: the column tile of 256
  int tile0;    // FO/ADD/LOO/alpha: first token tile
  int base;     // x', cnorm: first token; qnorm: first neuron
  int head;     // x': the column tile of 256; qnorm: KV group
};

// Unit u of the schedule.
template <bool STREAM = false>
__device__ __forceinline__ Unit unit_info(const TileParams& p, int u) {
  Unit U{};
  switch (p.mode) {
    case kModeFold:   // one unit per (128 rows of W16 / M16, 256 columns of H*dh)
      U.kt = u % (2 * p.n_ktiles);
      U.njobs = 1;
      U.base = u / (2 * p.n_ktiles);  // column tile of 256
      break;
    case kModeFO:
    case kModeLOO:
    case kModeADD: {   // one unit per (kHeadSets x 256 tokens, 64 neurons): kt = the 64-neuron block
      const int nblk = 2 * p.n_ktiles;
      U.kt = u % nblk;
      U.chunk = u / nblk;
      U.tile0 = 2 * kHeadSets * U.chunk;
      const bool op = p.mode != kModeADD;   // with an operating-point job
      U.njobs = kHeadSets * (op ? 1 + p.H : p.H);
      U.njobs_pm = STREAM ? kHeadSets * (op ? 2 : 1) : U.njobs;
      return U;
    }
    case kModeAlpha: {
      U.kt = u % p.n_ktiles;
      U.chunk = u / p.n_ktiles;
      U.tile0 = U.chunk * p.tiles_per_unit;
      U.njobs = min(p.tiles_per_unit, p.n_ttiles - U.tile0);
      U.njobs_pm = U.njobs;
      return U;
    }
    case kModeCNorm:   // one unit per (token tile, 256 columns d); jobs: the H heads
      U.kt = u % p.n_ntiles;   // the column tile
      U.base = (u / p.n_ntiles) * kBlockM;
      U.njobs = p.H;
      break;
    case kModeXPrime:   // one unit per (token tile, 256 columns d)
      U.base = (u / p.n_ntiles) * kBlockM;
      U.head = u % p.n_ntiles;   // the column tile
      U.njobs = 1;
      break;
    case kModeQNorm:   // one unit per (128 neurons, KV group); jobs: the group's row tiles of 256
      U.base = (u / p.G) * kBlockM;
      U.head = u % p.G;
      U.njobs = p.n_ntiles;
      break;
  }
  U.njobs_pm = U.njobs;
  return U;
}

// Position within a unit's job list, advanced without divisions: FO / ADD /
// LOO: a = the unit's set of 256 tokens, b = job within the set; the other
// modes count jobs in b.
struct JobIter {
  int a, b;
};

// The next job of unit U.  Every role walks the same sequence, except that
// with streamed heads the producer and the MMA issuer (pm) see one kJobStream
// where the epilogue sees the H head jobs of a 256-token set.
template <int MODE, bool STREAM = false>
__device__ __forceinline__ Job job_next(const TileParams& p, const Unit& U, JobIter& it, bool pm = false) {
  Job J{};
  J.kt = U.kt;
  if constexpr (MODE == kModeFold) {
    J.kind = kJobFold; J.nkb = 2 * p.nkb_D; J.nkb_part = p.nkb_D; J.last_nks = p.ls_D; J.nt = U.base;
  } else if constexpr (MODE == kModeFO || MODE == kModeLOO || MODE == kModeADD) {
    // a = the unit's set of 256 tokens, b = the job within the set
    J.t0 = (U.tile0 + 2 * it.a) * kBlockN;
    const bool op = MODE != kModeADD;
    const int j = it.b;
    const int per = (STREAM && pm) ? (op ? 2 : 1) : (op ? 1 + p.H : p.H);
    if (++it.b == per) { it.b = 0; ++it.a; }
    if (op && j == 0) {
      J.kind = kJobGateUp; J.nkb = p.nkb_D; J.nkb_part = p.nkb_D; J.last_nks = p.ls_D;
    } else if (STREAM && pm) {
      J.kind = kJobStream; J.nkb = p.nkb_HD; J.nkb_part = p.nkb_HD; J.last_nks = p.ls_HD;
    } else {
      J.kind = kJobHead; J.head = op ? j - 1 : j; J.nkb = p.nkb_dh; J.nkb_part = p.nkb_dh; J.last_nks = p.ls_dh;
    }
  } else if constexpr (MODE == kModeAlpha) {
    J.t0 = (U.tile0 + it.b) * kBlockN;
    J.kind = kJobGateUp; J.nkb = p.nkb_D; J.nkb_part = p.nkb_D; J.last_nks = p.ls_D;
    ++it.b;
  } else if constexpr (MODE == kModeXPrime) {
    J.kind = kJobXPrime; J.nkb = p.nkb_I; J.nkb_part = p.nkb_I; J.last_nks = 4;
    J.t0 = U.base; J.nt = U.head;
  } else if constexpr (MODE == kModeCNorm) {
    J.kind = kJobCNorm; J.nkb = p.nkb_dh; J.nkb_part = p.nkb_dh; J.last_nks = p.ls_dh;
    J.t0 = U.base; J.head = it.b++; J.nt = U.kt;
  } else {   // kModeQNorm
    J.kind = kJobQNorm; J.nkb = 2 * p.nkb_D; J.nkb_part = p.nkb_D; J.last_nks = p.ls_D;
    J.g = U.head; J.nt = it.b++;
  }
  return J;
}

struct Smem {
  uint64_t* full;
  uint64_t* empty;
  uint64_t* tfull;
  uint64_t* tempty;
  uint64_t* drain;
  uint32_t* tmem_slot;
  volatile int* abort_flag;
  uint64_t* ufull;         // unit ring: the TMA warp published the slot's unit id
  uint64_t* uempty;        // unit ring: the MMA thread and every epilogue warp have read it
  volatile int* uring;     // unit ids (-1: no more units)
  float* sacc;     // FO / ADD / LOO: the unit's sums [column group][H][128 neurons]
  float4* rsc;     // LOO: per epilogue warp, sigma of its column group's tokens for the current head job
  uint8_t* stage0;
};

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// STREAM: the producer and MMA issuer walk the heads' K ranges back to back
// (FO / ADD / LOO with p.stream_heads); a separate instantiation, so the
// issue loop of the other shapes carries no extra branch.
template <int MODE, bool STREAM>
__global__ void __launch_bounds__(block_threads(MODE), 1)
    affinity_tile_kernel(const __grid_constant__ CUtensorMap map0, const __grid_constant__ CUtensorMap map1,
                         const __grid_constant__ CUtensorMap map2, const __grid_constant__ CUtensorMap map3,
                         const TileParams p) {
  pdl_enter();
  // The next kernel in the stream may be placed beside this one's CTAs at once (it waits
  // for this kernel to complete before touching memory).  Not in the FO pass: there the
  // early arrivals (the reduction's 512-thread blocks) measured 10 us slower per launch.
  if constexpr (MODE != kModeFO) pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* base = smem_raw + (((raw + 1023u) & ~1023u) - raw);

  constexpr int EW = epi_warps(MODE);   // epilogue warps
  constexpr int NG = EW / 4;              // column groups of a 128-column accumulator
  constexpr int CW = kBlockN / NG;        // columns per epilogue thread (of each accumulator)
  constexpr bool kHeads = MODE == kModeFO || MODE == kModeADD || MODE == kModeLOO;
  // one N = 256 MMA per K slice (see the file comment): A = the first tile for the
  // head passes and the fold, the third for the others
  constexpr bool kAFirst = kHeads || MODE == kModeFold;
  constexpr int CWW = 2 * kBlockN / NG;   // columns of the 256 per epilogue thread
  const int S = p.stages;
  constexpr int kSB = kStageBytes;        // bytes of one pipeline stage
  constexpr int kBOff = 2 * kTileBytes;   // offset of the third tile within a stage
  Smem sm;
  sm.stage0 = base;
  uint8_t* cur = base + (size_t)S * kSB;
  sm.sacc = reinterpret_cast<float*>(cur);
  const int sacc_floats = kHeads ? NG * p.H * kBlockM : 0;
  cur += (size_t)sacc_floats * 4;
  sm.rsc = reinterpret_cast<float4*>(cur);
  if constexpr (MODE == kModeLOO) cur += (size_t)EW * (CWW / 4) * 16;
  sm.full = reinterpret_cast<uint64_t*>(cur);
  sm.empty = sm.full + S;
  sm.tfull = sm.empty + S;
  sm.tempty = sm.tfull + 2;
  sm.drain = sm.tempty + 2;
  sm.tmem_slot = reinterpret_cast<uint32_t*>(sm.drain + 1);
  sm.abort_flag = reinterpret_cast<volatile int*>(sm.tmem_slot + 1);
  sm.ufull = reinterpret_cast<uint64_t*>(sm.tmem_slot + 2);   // 8-byte aligned: drain + 16 bytes
  sm.uempty = sm.ufull + kUnitRing;
  sm.uring = reinterpret_cast<volatile int*>(sm.uempty + kUnitRing);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cid = (int)blockIdx.x;
  const int ncl = (int)gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.tfull[b], 1);
      mbar_init(&sm.tempty[b], EW);
    }
    mbar_init(sm.drain, 1);
    for (int r = 0; r < kUnitRing; ++r) {
      mbar_init(&sm.ufull[r], 1);
      mbar_init(&sm.uempty[r], 1 + EW);   // the MMA thread and one lane of every epilogue warp
    }
    *sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&map0);
    prefetch_tmap(&map1);
    prefetch_tmap(&map2);
    prefetch_tmap(&map3);
  }
  if (warp == 1) {
    tmem_alloc(sm.tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp >= 2) {
    for (int i = threadIdx.x - 64; i < sacc_floats; i += EW * 32) sm.sacc[i] = 0.f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_slot;
  // Powers of two that undo the operand scales (see scales.cuh): g, u come out of
  // the gate/up job times 2^(e_n + e_w), head-job values times 2^(e_m + e_a), the
  // fold's accumulator times 2^(e_w + e_g).
  // The head-job sums keep their 2^2(e_m + e_a); reduce_finalize removes it.
  const ScaleExps ex = scale_exps(*p.sc, p.D);
  const float f_gu = pow2f(-(ex.e_n + ex.e_w));   // -> g, u
  const float f_up = pow2f(ex.e_m + ex.e_a);      // LOO: g, u onto the head jobs' scale

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int s = 0, issued = 0;
      uint32_t ph = 0;                 // phase parity of the current use of stage s
      bool ok = true;
      int ur = 0;
      uint32_t urph = 0;               // unit ring slot and its phase parity
      // With a counter, the units before the last two rounds still go every gridDim-th (the
      // CTAs then walk the token tiles in step, which keeps them in L2) and the rest are
      // claimed, which evens out the CTAs' finishing times.
      const int fixed_rounds = p.ucount ? max(0, (p.n_units - p.unit0) / ncl - 2) : 1 << 30;
      for (int k = 0; ok; ++k) {
        // the next unit, published to the ring
        const int u = k < fixed_rounds ? p.unit0 + cid + k * ncl
                                       : p.unit0 + fixed_rounds * ncl + (int)atomicAdd(p.ucount, 1u);
        const bool done = u >= p.n_units;
        if (!mbar_wait(&sm.uempty[ur], urph ^ 1u, sm.abort_flag, p.status)) { ok = false; break; }
        sm.uring[ur] = done ? -1 : u;
        mbar_arrive(&sm.ufull[ur]);
        if (++ur == kUnitRing) { ur = 0; urph ^= 1u; }
        if (done) break;
        const Unit U = unit_info<STREAM>(p, u);
        JobIter jt{0, 0};
        for (int j = 0; ok && j < U.njobs_pm; ++j) {
          const Job J = job_next<MODE, STREAM>(p, U, jt, true);
          for (int kb = 0, kb_in = 0, part = 0; kb < J.nkb; ++kb) {
            if (!mbar_wait(&sm.empty[s], ph ^ 1u, sm.abort_flag, p.status)) { ok = false; break; }
            uint8_t* st = sm.stage0 + s * kSB;
            uint64_t* fb = &sm.full[s];
            const int kx = kb_in * kBlockK;
            mbar_arrive_expect_tx(fb, kStageBytes);
            switch (J.kind) {
              case kJobGateUp:
                if (MODE == kModeAlpha) {
                  // the gate and up rows of 128 neurons (the MMA's B, through the 4-D view
                  // of W16), n16 token rows (its A)
                  tma_load_4d(st, &map0, fb, kx, 0, 0, J.kt * 8);
                  tma_load_4d(st + kTileBytes, &map0, fb, kx, 0, 1, J.kt * 8);
                  tma_load_2d(st + kBOff, &map1, fb, kx, J.t0);
                } else {
                  // A = the 128 interleaved W16 rows of 64 neurons, B = 256 n16 token rows
                  tma_load_2d(st, &map0, fb, kx, J.kt * kBlockM);
                  tma_load_2d(st + kTileBytes, &map1, fb, kx, J.t0);
                  tma_load_2d(st + kBOff, &map1, fb, kx, J.t0 + kBlockN);
                }
                break;
              case kJobStream:   // M16 rows of 64 neurons, 256 a16 tokens; K runs over all heads' columns
                tma_load_2d(st, &map2, fb, kx, J.kt * kBlockM);
                tma_load_2d(st + kTileBytes, &map3, fb, kx, J.t0);
                tma_load_2d(st + kBOff, &map3, fb, kx, J.t0 + kBlockN);
                break;
              case kJobHead:     // M16 rows of 64 neurons for head h, 256 a16 head h tokens
                tma_load_3d(st, &map2, fb, kx, J.kt * kBlockM, J.head);
                tma_load_3d(st + kTileBytes, &map3, fb, kx, J.head, J.t0);
                tma_load_3d(st + kBOff, &map3, fb, kx, J.head, J.t0 + kBlockN);
                break;
              case kJobFold:     // A = 128 rows of W16, B = 256 columns of gamma*Wo^T (hi, then lo)
                tma_load_2d(st, &map0, fb, kx, J.kt * kBlockM);
                tma_load_3d(st + kTileBytes, &map1, fb, kx, part, J.nt * 2 * kBlockN);
                tma_load_3d(st + kBOff, &map1, fb, kx, part, J.nt * 2 * kBlockN + kBlockN);
                break;
              case kJobXPrime:   // Wd16 rows d (256, the MMA's B), alpha16 token rows (its A)
                tma_load_2d(st, &map1, fb, kx, J.nt * 2 * kBlockN);
                tma_load_2d(st + kTileBytes, &map1, fb, kx, J.nt * 2 * kBlockN + kBlockN);
                tma_load_2d(st + kBOff, &map0, fb, kx, J.t0);
                break;
              case kJobCNorm:    // Wo16 rows d (256), head h's columns (B); a16 head h token rows (A)
                tma_load_2d(st, &map1, fb, J.head * p.dh + kx, J.nt * 2 * kBlockN);
                tma_load_2d(st + kTileBytes, &map1, fb, J.head * p.dh + kx, J.nt * 2 * kBlockN + kBlockN);
                tma_load_3d(st + kBOff, &map0, fb, kx, J.head, J.t0);
                break;
              case kJobQNorm:    // group g's gamma'-scaled q/k/v rows, hi | lo along K (256, B); Wd^T neuron rows (A)
                tma_load_4d(st, &map1, fb, kx, part, J.nt * 2 * kBlockN, J.g);
                tma_load_4d(st + kTileBytes, &map1, fb, kx, part, J.nt * 2 * kBlockN + kBlockN, J.g);
                tma_load_2d(st + kBOff, &map0, fb, kx, U.base);
                break;
            }
            ++issued;
            if (++s == S) { s = 0; ph ^= 1u; }
            if (++kb_in == J.nkb_part) { kb_in = 0; ++part; }
          }
        }
      }
      if (!ok) {
        // Let every copy already issued land before shared memory is released.
        const int n = issued < S ? issued : S;
        for (int i = 1; i <= n; ++i) {
          const int q = issued - i;
          volatile int dummy = 0;
          mbar_wait(&sm.full[q % S], (uint32_t)((q / S) & 1), &dummy, p.status, 100000000ull);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // A lean loop: this one thread must issue MMAs as fast as the tensor pipe
    // retires them, so no divisions, and descriptors advance by constants.
    if (lane == 0) {
      // N = 256: one MMA reads 12 KB of shared memory where two N = 128 MMAs read 16 KB
      constexpr uint32_t idesc = idesc_f16(kBlockM, 2 * kBlockN, 0);
      const uint64_t dbase = smem_desc_k_sw128(smem_u32(sm.stage0));   // first tile of stage 0
      constexpr uint64_t kStageDesc = (uint64_t)(kSB >> 4);             // descriptor step per stage
      constexpr uint64_t kA2 = (uint64_t)(kTileBytes >> 4), kB = (uint64_t)(kBOff >> 4);
      int s = 0, b = 0;
      uint32_t ph = 0, tph = 0;        // stage phase; TMEM buffer phase (flips every second job)
      bool ok = true;
      int ur = 0;
      uint32_t urph = 0;
      while (ok) {
        if (!mbar_wait(&sm.ufull[ur], urph, sm.abort_flag, p.status)) { ok = false; break; }
        const int u = sm.uring[ur];
        mbar_arrive(&sm.uempty[ur]);
        if (++ur == kUnitRing) { ur = 0; urph ^= 1u; }
        if (u < 0) break;
        const Unit U = unit_info<STREAM>(p, u);
        JobIter jt{0, 0};
        for (int j = 0; ok && j < U.njobs_pm; ++j) {
          const Job J = job_next<MODE, STREAM>(p, U, jt, true);
          if (!mbar_wait(&sm.tempty[b], tph ^ 1u, sm.abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          if constexpr (STREAM) {
           if (J.kind == kJobStream) {
            // The H heads' K slices arrive back to back; a stage may hold the end of one
            // head and the start of the next.  When a head's last slice is issued its
            // accumulator is committed and the next head moves to the other buffer.
            int sih = 0, heads_left = p.H;
            for (int kb = 0; ok && kb < J.nkb; ++kb) {
              if (!mbar_wait(&sm.full[s], ph, sm.abort_flag, p.status)) { ok = false; break; }
              tc_fence_after();
              const uint64_t da = dbase + (uint64_t)s * kStageDesc, dt = da + kA2;
              const int nks = (kb == J.nkb - 1) ? J.last_nks : 4;
#pragma unroll
              for (int ks = 0; ks < 4; ++ks) {
                if (ks < nks && heads_left > 0) {
                  const uint32_t d = tmem + (uint32_t)(b * 2 * kBlockN);
                  mma_f16_ss(d, da + 2 * ks, dt + 2 * ks, idesc, sih > 0 ? 1u : 0u);
                  if (++sih == p.spp) {
                    mma_commit(&sm.tfull[b]);
                    if (++b == 2) { b = 0; tph ^= 1u; }
                    sih = 0;
                    if (--heads_left > 0) {
                      if (!mbar_wait(&sm.tempty[b], tph ^ 1u, sm.abort_flag, p.status)) { ok = false; break; }
                      tc_fence_after();
                    }
                  }
                }
              }
              mma_commit(&sm.empty[s]);   // also on the way out, so the producer can drain
              if (++s == S) { s = 0; ph ^= 1u; }
            }
            continue;
           }
          }
          const uint32_t d1 = tmem + (uint32_t)(b * 2 * kBlockN);
          uint32_t acc = 0u;
          for (int kb = 0, kb_in = 0; kb < J.nkb; ++kb) {
            if (!mbar_wait(&sm.full[s], ph, sm.abort_flag, p.status)) { ok = false; break; }
            tc_fence_after();
            const uint64_t da1 = dbase + (uint64_t)s * kStageDesc;
            const uint64_t da2 = da1 + kA2, db = da1 + kB;
            const int nks = (kb_in == J.nkb_part - 1) ? J.last_nks : 4;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              if (ks < nks) {
                if constexpr (kAFirst) {   // A = the first tile (weights), B = the next 256 rows
                  mma_f16_ss(d1, da1 + 2 * ks, da2 + 2 * ks, idesc, acc);
                } else {
                  mma_f16_ss(d1, db + 2 * ks, da1 + 2 * ks, idesc, acc);
                }
                acc = 1u;
              }
            }
            mma_commit(&sm.empty[s]);
            if (++s == S) { s = 0; ph ^= 1u; }
            if (++kb_in == J.nkb_part) kb_in = 0;
          }
          if (!ok) break;
          mma_commit(&sm.tfull[b]);
          if (++b == 2) { b = 0; tph ^= 1u; }
        }
      }
      if (!ok) {
        mma_commit(sm.drain);
        volatile int dummy = 0;
        mbar_wait(sm.drain, 0, &dummy, p.status, 100000000ull);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;            // TMEM lane quarter this warp may read
    const int hf = (warp - 2) >> 2;    // which group of CW columns of the tile
    const int row = q * 32 + lane;     // TMEM lane = row of the MMA's A
    const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
    // Head passes: thread l and thread l + 16 both work on neuron 16q + l of the unit's
    // 64, on the first and the last CW tokens of the column group.
    const bool upl = lane >= 16;
    const uint32_t tg = tmem + ((uint32_t)(q * 32) << 16);        // the quarter's gate lanes
    const uint32_t tu = tmem + ((uint32_t)(q * 32 + 16) << 16);   // ... and its up lanes
    // FO: f32x2 pairs of silu'(g)u and silu(g), CW tokens; LOO: g and u
    uint64_t abA[CW / 2], abB[CW / 2];
#pragma unroll
    for (int i = 0; i < CW / 2; ++i) { abA[i] = 0ull; abB[i] = 0ull; }
    uint64_t ssp = pk(0.f, 0.f);       // x' / qnorm running sums, a packed pair (even and odd columns)
    // c_h pass: x of the thread's token and CWW columns, loaded at a unit's first head
    uint32_t xr[MODE == kModeCNorm ? CWW / 2 : 1];
    int b = 0;
    uint32_t tph = 0;                  // TMEM buffer phase (flips every second job)
    bool ok = true;
    int ur = 0;
    uint32_t urph = 0;
    while (ok) {
      int u = -1, u_ok = 1;
      if (lane == 0) {
        u_ok = mbar_wait(&sm.ufull[ur], urph, sm.abort_flag, p.status) ? 1 : 0;
        if (u_ok) {
          u = sm.uring[ur];
          mbar_arrive(&sm.uempty[ur]);
        }
      }
      u_ok = __shfl_sync(0xffffffffu, u_ok, 0);
      u = __shfl_sync(0xffffffffu, u, 0);
      if (!u_ok) { ok = false; break; }
      if (++ur == kUnitRing) { ur = 0; urph ^= 1u; }
      if (u < 0) break;
      const Unit U = unit_info<STREAM>(p, u);
      JobIter jt{0, 0};
      for (int j = 0; j < U.njobs; ++j, b ^= 1, tph ^= (uint32_t)(b == 0)) {
        const Job J = job_next<MODE, STREAM>(p, U, jt);
        // LOO head job: lanes 0..15 fetch sigma of the column group's CWW tokens (one float4
        // each) before the accumulator wait, which hides the load; the token loop takes
        // its values from them with shuffles
        float4 rho_v = make_float4(0.f, 0.f, 0.f, 0.f);
        if constexpr (MODE == kModeLOO) {
          if (J.kind == kJobHead && lane < CWW / 4)
            rho_v = __ldg(reinterpret_cast<const float4*>(p.rho + (size_t)J.head * p.T_pad + J.t0 + hf * CWW) + lane);
        }
        int w_ok = 1;
        if (lane == 0) w_ok = mbar_wait(&sm.tfull[b], tph, sm.abort_flag, p.status) ? 1 : 0;
        w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
        if (!w_ok) { ok = false; break; }
        tc_fence_after();
        const uint32_t c1 = tl + (uint32_t)(b * 2 * kBlockN + hf * CW);
        const uint32_t c2 = c1 + kBlockN;
        float4* rsw = sm.rsc + (warp - 2) * (CWW / 4);   // LOO: this warp's sigma slots
        if constexpr (MODE == kModeLOO) {
          if (J.kind == kJobHead) {
            __syncwarp();   // the previous head job's reads of the slots are done
            if (lane < CWW / 4) rsw[lane] = rho_v;
            __syncwarp();
          }
        }

        if constexpr (MODE == kModeFO || MODE == kModeLOO) {
          if (J.kind == kJobGateUp) {
            // Phase 1: stash g, u in the registers that will hold A', B' and hand the
            // accumulator buffer back at once, so the MMAs of the next two head
            // jobs run while phase 2 (exp + reciprocal per element) computes.
            const uint32_t col = (uint32_t)(b * 2 * kBlockN + hf * CWW);
#pragma unroll
            for (int c = 0; c < CW / 8; ++c) {
              uint32_t gr[8], ur[8];
              tmem_ld8_x2<CW>(tg + col + c * 8, gr);
              tmem_ld8_x2<CW>(tu + col + c * 8, ur);
              tmem_ld_wait();
              if (c == CW / 8 - 1) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.tempty[b]);
              }
#pragma unroll
              for (int i = 0; i < 8; i += 2) {
                abA[(c * 8 + i) / 2] = pk_u(gr[i], gr[i + 1]);
                abB[(c * 8 + i) / 2] = pk_u(ur[i], ur[i + 1]);
              }
            }
            {
              // FO: the accumulators' 2^(e_n + e_w) removed (g, u exact);  LOO: g, u onto the scale
              // of the head jobs' p_h.w, at which g - g^(-h) is formed
              const float fs = MODE == kModeLOO ? f_gu * f_up : f_gu;
              const uint64_t fl = pk(fs, fs);
#pragma unroll
              for (int i = 0; i < CW / 2; ++i) {
                abA[i] = mul2(abA[i], fl);
                abB[i] = mul2(abB[i], fl);
              }
            }
            // Phase 2 (FO): (g, u) -> (A', B') = (silu'(g) u, silu(g)) in place; LOO keeps g and u.
            if constexpr (MODE == kModeFO) {
#pragma unroll
              for (int i = 0; i < CW / 2; ++i) {
                const float2 g2 = unpk(abA[i]), u2 = unpk(abB[i]);
                float gA[2], gB[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  const float g = e ? g2.y : g2.x;
                  const float uu = e ? u2.y : u2.x;
                  const float sg = __fdividef(1.0f, 1.0f + __expf(-g));  // sigmoid(g)
                  gA[e] = sg * fmaf(g, 1.0f - sg, 1.0f) * uu;           // silu'(g) u
                  gB[e] = g * sg;                                       // silu(g)
                }
                abA[i] = pk(gA[0], gA[1]);
                abB[i] = pk(gB[0], gB[1]);
              }
            }
            continue;
          }
        }
        if constexpr (MODE == kModeAlpha) {
          {   // kJobGateUp: TMEM lane = token J.t0 + row, columns = g (first 128) and u of
              // the neuron tile; alpha = silu(g) u, 16 neurons (32 B) stored at a time
            __half* dst = p.alpha16 + (size_t)(J.t0 + row) * p.I_pad + J.kt * kBlockM + hf * CW;
#pragma unroll
            for (int c = 0; c < CW / 16; ++c) {
              uint32_t gr[16], ur[16];
              tmem_ld16(c1 + c * 16, gr);
              tmem_ld16(c2 + c * 16, ur);
              tmem_ld_wait();
              if (c == CW / 16 - 1) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.tempty[b]);
              }
              uint32_t hv[8];
#pragma unroll
              for (int i = 0; i < 16; i += 2) {
                float a2[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  const float g = __uint_as_float(gr[i + e]) * f_gu;
                  const float sg = __fdividef(1.0f, 1.0f + __expf(-g));
                  a2[e] = g * sg * (__uint_as_float(ur[i + e]) * f_gu);
                }
                hv[i / 2] = pack_h2(a2[0], a2[1]);
              }
              uint4* d4 = reinterpret_cast<uint4*>(dst + c * 16);
              d4[0] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
              d4[1] = make_uint4(hv[4], hv[5], hv[6], hv[7]);
            }
            continue;
          }
        }
        if constexpr (kHeads) {
          // kJobHead.  FO: Delta = A' pg + B' pu per token, Delta^2 summed over the thread's CW
          // tokens; LOO: g - g^(-h) = pg + sigma (g - pg) with sigma = 1 - r / rms(x - c_h),
          // likewise for u, both squared; ADD: each lane sums the squares of its own 2 CW values.
          const uint32_t col = (uint32_t)(b * 2 * kBlockN + hf * CWW);
          uint64_t acc = pk(0.f, 0.f);
          if constexpr (MODE == kModeADD) {
            // own lane, both halves of the group, 16 columns per read: ADD has registers to
            // spare, and fewer, wider reads leave fewer TMEM load latencies in the job
#pragma unroll
            for (int c = 0; c < CW / 16; ++c) {
              uint32_t v1[16], v2[16];
              tmem_ld16(tl + col + c * 16, v1);
              tmem_ld16(tl + col + CW + c * 16, v2);
              tmem_ld_wait();
              if (c == CW / 16 - 1) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.tempty[b]);
              }
#pragma unroll
              for (int i = 0; i < 16; i += 2) {
                const uint64_t w1 = pk_u(v1[i], v1[i + 1]), w2 = pk_u(v2[i], v2[i + 1]);
                acc = fma2(w1, w1, acc);
                acc = fma2(w2, w2, acc);
              }
            }
          } else {
          // TMEM columns per read: 8, or 4 in LOO mode (its arithmetic needs more registers)
          constexpr int kW = MODE == kModeLOO ? 4 : 8;
#pragma unroll
          for (int c = 0; c < CW / kW; ++c) {
            // LOO: sigma of the slice's 4 tokens, a broadcast read issued before the TMEM reads
            // so that its latency overlaps theirs
            float4 rq = make_float4(0.f, 0.f, 0.f, 0.f);
            if constexpr (MODE == kModeLOO) {
              static_assert(kW == 4, "one float4 of sigma per slice");
              rq = rsw[(upl ? CW / 4 : 0) + c];
            }
            uint32_t pg[kW], pu[kW];
            if constexpr (kW == 8) {
              tmem_ld8_x2<CW>(tg + col + c * kW, pg);
              tmem_ld8_x2<CW>(tu + col + c * kW, pu);
            } else {
              tmem_ld4_x2<CW>(tg + col + c * kW, pg);
              tmem_ld4_x2<CW>(tu + col + c * kW, pu);
            }
            tmem_ld_wait();
            if (c == CW / kW - 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&sm.tempty[b]);
            }
#pragma unroll
            for (int i = 0; i < kW; i += 2) {
              const uint64_t vg = pk_u(pg[i], pg[i + 1]);
              const uint64_t vu = pk_u(pu[i], pu[i + 1]);
              const int ai = (c * kW + i) / 2;   // token pair within the thread's CW tokens
              if constexpr (MODE == kModeFO) {
                uint64_t d = mul2(abA[ai], vg);
                d = fma2(abB[ai], vu, d);
                acc = fma2(d, d, acc);
              } else {   // LOO: g - g^(-h) = p.w + sigma (g - p.w), sigma = 1 - rho
                const uint64_t rr = i == 0 ? pk(rq.x, rq.y) : pk(rq.z, rq.w), neg1 = pk(-1.0f, -1.0f);
                const uint64_t dg = fma2(rr, fma2(vg, neg1, abA[ai]), vg);
                const uint64_t du = fma2(rr, fma2(vu, neg1, abB[ai]), vu);
                acc = fma2(dg, dg, acc);
                acc = fma2(du, du, acc);
              }
            }
          }
          }
          const float2 s2 = unpk(acc);
          sm.sacc[(hf * p.H + J.head) * kBlockM + row] += s2.x + s2.y;   // times 2^2(e_m + e_a)
        }
        static_assert(EW == kWideEpiWarps || CW == 64, "the 8-warp epilogues read 64 columns per thread");

        if constexpr (MODE == kModeFold) {
          // TMEM lane = row R of W16 and M16 (groups of 16 neurons: 16 gate rows, then the same
          // neurons' 16 up rows), columns n = nt*256 + hf*128 + ... of H*dh, times 2^(e_w + e_g)
          // from the operands; stored times 2^e_m.  d_head % 8 == 0, so an 8-column group lies
          // in one head.
          const size_t R = (size_t)J.kt * kBlockM + row;
          const float fm1 = pow2f(ex.e_m), fm2 = pow2f(-(ex.e_w + ex.e_g));
          const uint32_t col = (uint32_t)(b * 2 * kBlockN + hf * CWW);
#pragma unroll
          for (int c = 0; c < CWW / 32; ++c) {
            uint32_t v[32];
            tmem_ld16(tl + col + c * 32, *reinterpret_cast<uint32_t(*)[16]>(v));
            tmem_ld16(tl + col + c * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(v + 16));
            tmem_ld_wait();
            if (c == CWW / 32 - 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&sm.tempty[b]);
            }
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
              const int n = J.nt * 2 * kBlockN + hf * CWW + c * 32 + i;
              if (n < p.H * p.dh) {
                float f[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(v[i + e]) * fm1 * fm2;
                uint4 w;
                w.x = pack_h2(f[0], f[1]);
                w.y = pack_h2(f[2], f[3]);
                w.z = pack_h2(f[4], f[5]);
                w.w = pack_h2(f[6], f[7]);
                if (p.stream_heads) {   // [2 I_pad][H*dh]: heads back to back along K
                  *reinterpret_cast<uint4*>(p.M16 + R * ((size_t)p.H * p.dh) + n) = w;
                } else {                // [H][2 I_pad][dh]
                  const int h = n / p.dh, jj = n % p.dh;
                  *reinterpret_cast<uint4*>(p.M16 + ((size_t)h * 2 * p.I_pad + R) * p.dh + jj) = w;
                }
              }
            }
          }
        }
        if constexpr (MODE == kModeCNorm) {
          // lane = token t; columns d = J.nt * 256 + hf * CWW + ... of (c_h / r)[t][d] for head
          // J.head: sum (c/r)^2 and x (c/r) over them.  x is read once per unit.  Columns past
          // D hold zeros (the B tiles were zero-filled), so only x needs a guard; D % 8 == 0,
          // so an 8-column group is wholly inside or wholly past D.
          const int t = J.t0 + row;
          if (j == 0) {
#pragma unroll
            for (int q8 = 0; q8 < CWW / 8; ++q8) {
              const int d = J.nt * 2 * kBlockN + hf * CWW + q8 * 8;
              uint4 w = make_uint4(0u, 0u, 0u, 0u);
              if (d < p.D && t < p.T) w = __ldg(reinterpret_cast<const uint4*>(p.x_bf16 + (size_t)t * p.D + d));
              xr[q8 * 4 + 0] = w.x;
              xr[q8 * 4 + 1] = w.y;
              xr[q8 * 4 + 2] = w.z;
              xr[q8 * 4 + 3] = w.w;
            }
          }
          const uint32_t c0 = tl + (uint32_t)(b * 2 * kBlockN + hf * CWW);
          uint64_t s1p = pk(0.f, 0.f), s2p = pk(0.f, 0.f);   // packed pairs: even and odd columns
#pragma unroll
          for (int c = 0; c < CWW / 16; ++c) {
            uint32_t v[16];
            tmem_ld16(c0 + c * 16, v);
            tmem_ld_wait();
            if (c == CWW / 16 - 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&sm.tempty[b]);
            }
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
              const uint32_t e = xr[(c * 16 + i) / 2];
              const uint64_t v2 = pk_u(v[i], v[i + 1]);
              s1p = fma2(v2, v2, s1p);
              s2p = fma2(pk_u(e << 16, e & 0xFFFF0000u), v2, s2p);
            }
          }
          const float2 f1 = unpk(s1p), f2 = unpk(s2p);
          const float s1 = f1.x + f1.y, s2 = f2.x + f2.y;
          // [column tile][column group][quantity][H][T_pad]: quantity 0 = sum (c/r)^2, 1 = sum x (c/r)
          float* dst = p.partial + ((size_t)((U.kt * NG + hf) * 2) * p.H + J.head) * p.T_pad + t;
          dst[0] = s1;
          dst[(size_t)p.H * p.T_pad] = s2;
        }
        if constexpr (MODE == kModeXPrime) {
          // lane = token t; columns d = J.nt * 256 + hf * CWW + ...: (alpha Wd^T)[t][d],
          // x' = x + that, accumulate x'^2 over d.  Columns past D hold zeros (the B tiles were
          // zero-filled), so only x needs a guard; D % 8 == 0, so an 8-column group is wholly
          // inside or wholly past D.
          const int t = J.t0 + row;
          const uint32_t c0 = tl + (uint32_t)(b * 2 * kBlockN + hf * CWW);
#pragma unroll
          for (int c = 0; c < CWW / 16; ++c) {
            uint32_t v[16];
            tmem_ld16(c0 + c * 16, v);
            tmem_ld_wait();
            if (c == CWW / 16 - 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&sm.tempty[b]);
            }
            const int d0 = J.nt * 2 * kBlockN + hf * CWW + c * 16;
#pragma unroll
            for (int q8 = 0; q8 < 2; ++q8) {
              const int d = d0 + q8 * 8;
              if (d < p.D && t < p.T) {
                const uint4 w = __ldg(reinterpret_cast<const uint4*>(p.x_bf16 + (size_t)t * p.D + d));
                const uint32_t e[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  // x' = x + alpha Wd^T for two columns at once (x * 1 + v rounds as x + v)
                  const uint64_t x2 = pk_u(e[i] << 16, e[i] & 0xFFFF0000u);
                  const uint64_t y2 = fma2(x2, pk(1.0f, 1.0f), pk_u(v[q8 * 8 + 2 * i], v[q8 * 8 + 2 * i + 1]));
                  ssp = fma2(y2, y2, ssp);
                }
              }
            }
          }
        }
        if constexpr (MODE == kModeQNorm) {
          // lane = neuron k = U.base + row; columns = 256 rows r of group J.g (hi and lo
          // parts already summed along K): accumulate Q[k][r]^2 over the group's rows
          const uint32_t c0 = tl + (uint32_t)(b * 2 * kBlockN + hf * CWW);
#pragma unroll
          for (int c = 0; c < CWW / 16; ++c) {
            uint32_t v[16];
            tmem_ld16(c0 + c * 16, v);
            tmem_ld_wait();
            if (c == CWW / 16 - 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&sm.tempty[b]);
            }
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
              const uint64_t v2 = pk_u(v[i], v[i + 1]);
              ssp = fma2(v2, v2, ssp);
            }
          }
          if (J.nt == p.n_ntiles - 1) {
            // rows past the group's end were zero-filled, so the sum is this column group's share
            const int k = U.base + row;
            const float2 s2 = unpk(ssp);
            if (k < p.I_pad) p.bnorm[((size_t)hf * p.I_pad + k) * p.G + J.g] = s2.x + s2.y;
            ssp = pk(0.f, 0.f);
          }
        }
      }
      if (!ok) break;
      // ---- end of unit
      if constexpr (kHeads) {
        // [H][I_pad / 64][chunk][column group][64]: each (head, 64-neuron block) owns one
        // contiguous run of its chunks' sums, which the reduction streams.  Threads l and
        // l + 16 add their sums (the same value in both) and thread l writes it.
        const int n_chunks = p.n_units / (2 * p.n_ktiles);
        const size_t run = (size_t)n_chunks * NG * 64;   // floats per (head, neuron block)
        float* dst = p.partial + (size_t)U.kt * run + ((size_t)U.chunk * NG + hf) * 64 + q * 16 + (lane & 15);
        const size_t hstride = (size_t)(p.I_pad / 64) * run;
        for (int h = 0; h < p.H; ++h) {
          float* sp = &sm.sacc[(hf * p.H + h) * kBlockM + row];
          const float v = *sp;
          *sp = 0.f;
          const float t = v + __shfl_xor_sync(0xffffffffu, v, 16);
          if (!upl) dst[(size_t)h * hstride] = t;
        }
      }
      if constexpr (MODE == kModeXPrime) {
        // [column tile][column group][T_pad]; token tiles are whole, so t < T_pad
        const float2 s2 = unpk(ssp);
        p.partial[(size_t)(U.head * NG + hf) * p.T_pad + U.base + row] = s2.x + s2.y;
        ssp = pk(0.f, 0.f);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

size_t tile_smem_bytes(int mode, int stages, int H) {
  const bool heads = mode == kModeFO || mode == kModeADD || mode == kModeLOO;
  const size_t sacc = heads ? (size_t)(epi_warps(mode) / 4) * H * kBlockM * 4 : 0;
  // LOO: a 16-byte sigma slot per 4 tokens of each epilogue warp's column group
  const size_t rsc = mode == kModeLOO ? (size_t)epi_warps(mode) * (2 * kBlockN / (epi_warps(mode) / 4) / 4) * 16 : 0;
  return 1024 + (size_t)stages * kStageBytes + sacc + rsc + (size_t)(2 * stages + 5) * 8 + 8 + (size_t)kUnitRing * 20;
}

// Launches `grid` CTAs.  With grid == 0 it only reports in *grid how many CTAs
// fit on the device at once.
template <int MODE, bool STREAM = false>
static cudaError_t launch_mode(const CUtensorMap* maps, const TileParams& p, int* grid, cudaStream_t stream) {
  const size_t smem = tile_smem_bytes(MODE, p.stages, p.H);
  auto* fn = affinity_tile_kernel<MODE, STREAM>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (*grid <= 0) {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    *grid = n;   // shared memory and TMEM allow one CTA per SM
    return e;
  }
  if (cudaError_t e_ = launch_pdl(fn, *grid, block_threads(MODE), smem, stream, maps[0], maps[1], maps[2], maps[3], p); e_ != cudaSuccess)
    return e_;
  return cudaGetLastError();
}

cudaError_t launch_tile_kernel(const CUtensorMap* maps, const TileParams& p, int* grid, cudaStream_t stream) {
  switch (p.mode) {
    case kModeFold: return launch_mode<kModeFold>(maps, p, grid, stream);
    case kModeFO:
      return p.stream_heads ? launch_mode<kModeFO, true>(maps, p, grid, stream)
                            : launch_mode<kModeFO>(maps, p, grid, stream);
    case kModeADD:
      return p.stream_heads ? launch_mode<kModeADD, true>(maps, p, grid, stream)
                            : launch_mode<kModeADD>(maps, p, grid, stream);
    case kModeAlpha: return launch_mode<kModeAlpha>(maps, p, grid, stream);
    case kModeXPrime: return launch_mode<kModeXPrime>(maps, p, grid, stream);
    case kModeQNorm: return launch_mode<kModeQNorm>(maps, p, grid, stream);
    case kModeCNorm: return launch_mode<kModeCNorm>(maps, p, grid, stream);
    case kModeLOO:
      return p.stream_heads ? launch_mode<kModeLOO, true>(maps, p, grid, stream)
                            : launch_mode<kModeLOO>(maps, p, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace aff
