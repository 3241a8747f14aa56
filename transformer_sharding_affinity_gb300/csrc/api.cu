// api.cu -- the C ABI declared in include/affinity.h: argument validation,
// workspace layout, TMA descriptor encoding and the launch sequence of the
// affinity pass ("Affinity-Aware Sharding for Delayed Tensor Parallelism",
// §3 "Affinity scores").  The host-only layout helpers live in layout.cu.
#include "affinity.h"
#include "aux_kernels.cuh"
#include "internal.h"
#include "moment_kernel.cuh"
#include "tile_kernel.cuh"

#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <deque>
#include <mutex>
#include <string>
#include <vector>

namespace aff {
cudaError_t launch_tile_kernel(const CUtensorMap* maps, const TileParams& p, int* grid, cudaStream_t stream);
size_t tile_smem_bytes(int mode, int stages, int H);
}  // namespace aff

using namespace aff;

namespace {
thread_local std::string g_last_cuda_error;
thread_local cudaEvent_t g_timing_start = nullptr;  // see affinity_set_timing_events
thread_local cudaEvent_t g_timing_stop = nullptr;
}  // namespace

aff_status aff::cuda_fail(cudaError_t e, const char* where) {
  g_last_cuda_error = std::string(where) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
  return AFF_ERR_CUDA;
}

// ---------------------------------------------------------------- device checks
aff_status aff::check_device(int* sm_count) {
  static std::mutex mu;
  static std::vector<int> sms;  // per device: 0 unknown, -1 wrong arch, >0 SM count
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return AFF_ERR_ARCH;
  }
  std::lock_guard<std::mutex> lk(mu);
  if ((int)sms.size() <= dev) sms.resize(dev + 1, 0);
  if (sms[dev] == 0) {
    int maj = 0, min = 0, n = 0;
    if (cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return AFF_ERR_ARCH;
    }
    sms[dev] = (maj == 10 && min == 3) ? n : -1;
  }
  if (sms[dev] < 0) return AFF_ERR_ARCH;
  *sm_count = sms[dev];
  return AFF_OK;
}

namespace {

constexpr int64_t kMaxDim = (int64_t)1 << 30;
constexpr int kTilesPerUnit = 2;      // token tiles (of 128) per alpha unit
constexpr int kDownTokenChunk = 256;  // tokens per partial sum of E_t[alpha^2 / r'^2]

inline int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

// Partial sums of x'^2 per token that the x' pass writes: one per column tile
// of 256 and column group of its epilogue.
inline int xprime_groups(int64_t D) { return (int)((D + 255) / 256) * (epi_warps(kModeXPrime) / 4); }

// Partial sums per (token, head) that the c_h pass writes: one per column tile of 256
// and column group of its epilogue.
inline int cnorm_groups(int64_t D) { return (int)((D + 255) / 256) * (epi_warps(kModeCNorm) / 4); }
inline int64_t ceil_div(int64_t v, int64_t m) { return (v + m - 1) / m; }

aff_status check_dims(const aff_dims* d) {
  if (!d) return AFF_ERR_INVALID_ARG;
  if (d->dtype != AFF_BF16 && d->dtype != AFF_FP32) return AFF_ERR_UNSUPPORTED_DTYPE;
  if (d->flags & ~AFF_FLAG_ADD_DIRECT) return AFF_ERR_INVALID_ARG;
  if (d->T < 1 || d->D < 1 || d->H < 1 || d->G < 1 || d->d_head < 1 || d->I < 1) return AFF_ERR_INVALID_ARG;
  if (!(std::isfinite(d->eps) && d->eps >= 0.f)) return AFF_ERR_INVALID_ARG;
  if (d->T > kMaxDim || d->D > kMaxDim || d->H > 4096 || d->d_head > 4096 || d->I > kMaxDim)
    return AFF_ERR_UNSUPPORTED_SHAPE;
  if (d->H % d->G) return AFF_ERR_UNSUPPORTED_SHAPE;
  if (d->dtype == AFF_BF16) {
    if (d->D % 8 || d->d_head % 8 || d->I % 8) return AFF_ERR_UNSUPPORTED_SHAPE;
    // per-thread head sums live in shared memory next to 2+ pipeline stages
    if (tile_smem_bytes(kModeFO, 2, (int)d->H) > (size_t)kMaxDynSmem) return AFF_ERR_UNSUPPORTED_SHAPE;
    if (d->H * d->d_head > kMaxDim) return AFF_ERR_UNSUPPORTED_SHAPE;
  }
  return AFF_OK;
}

// Workspace carve-up; every buffer starts on a 1024-byte boundary.
struct Layout {
  size_t total = 0;
  size_t status = 0;
  size_t scales = 0;   // DevScales (bf16 path)
  // bf16 path
  size_t W16 = 0, GWo16 = 0, M16 = 0, n16 = 0, a16 = 0, partial = 0, headsum = 0, wdn = 0;
  size_t alpha16 = 0, Wd16 = 0, WdT16 = 0, Wqkv16 = 0, ssx = 0, cpart = 0, bnorm = 0;
  size_t Wo16 = 0, cn = 0, rho = 0, inv_r = 0;   // leave-one-out score
  size_t ir = 0, gram = 0, cmax = 0, CC = 0, gscale = 0;  // ADD, second-moment form
  // fp32 path
  size_t n32 = 0, a32 = 0, M32 = 0, ab = 0, alpha32 = 0;
  int64_t I_pad = 0, T_pad = 0, n_chunks = 0, n_tchunks = 0, Rg = 0;

  size_t take(size_t bytes) {
    total = (size_t)round_up((int64_t)total, 1024);
    size_t off = total;
    total += bytes;
    return off;
  }
};

// ADD through each head's second moment (moment_kernel.cuh): AFF_BF16, d_head
// <= 128 (one 128-row tile per head), unless the caller asks for the direct form.
bool moment_form(const aff_dims& d, int mode) {
  return d.dtype == AFF_BF16 && mode == AFF_MODE_ADD && !(d.flags & AFF_FLAG_ADD_DIRECT) && d.d_head <= 128;
}

Layout make_layout(const aff_dims& d, int mode, bool down) {
  Layout L;
  const int64_t T = d.T, D = d.D, H = d.H, G = d.G, dh = d.d_head, I = d.I;
  L.status = L.take(256);
  if (d.dtype == AFF_BF16) {
    L.scales = L.take(256);
    L.I_pad = round_up(I, 256);
    L.T_pad = round_up(T, down ? 128 : 256 * kHeadSets);   // head-pass units take 512 tokens
    L.W16 = L.take((size_t)2 * L.I_pad * D * 2);
    if (down || mode != AFF_MODE_ADD) L.n16 = L.take((size_t)T * D * 2);   // ADD has no operating point
    if (!down && moment_form(d, mode)) {
      const GramSplit gs = gram_split(T, H);
      L.n_chunks = 1;
      L.GWo16 = L.take((size_t)H * dh * 2 * D * 2);
      L.M16 = L.take((size_t)2 * H * L.I_pad * dh * 2);
      L.ir = L.take((size_t)gs.nkb * 64 * 4);
      L.gram = L.take((size_t)gs.n_chunks * H * kMomentRows * kMomentRows * 4);
      L.cmax = L.take((size_t)gs.n_chunks * H * 4);
      L.CC = L.take((size_t)2 * H * kMomentRows * kMomentRows * 2);
      L.gscale = L.take((size_t)H * 4);
      L.partial = L.take((size_t)H * L.I_pad * 4);   // [H][I_pad] token sums
    } else if (!down) {
      L.n_chunks = L.T_pad / (256 * kHeadSets);
      L.GWo16 = L.take((size_t)H * dh * 2 * D * 2);
      L.M16 = L.take((size_t)2 * H * L.I_pad * dh * 2);
      L.a16 = L.take((size_t)T * H * dh * 2);
      // one slot per (chunk, column group of the epilogue, head, neuron)
      const int tile_mode = mode == AFF_MODE_LOO ? kModeLOO : (mode == AFF_MODE_ADD ? kModeADD : kModeFO);
      L.partial = L.take((size_t)L.n_chunks * (epi_warps(tile_mode) / 4) * H * L.I_pad * 4);
      if (mode == AFF_MODE_FO) L.wdn = L.take((size_t)L.I_pad * 4);
      L.inv_r = L.take((size_t)L.T_pad * 4);   // 1/r per token (restaging of a16, LOO's rho)
      if (mode == AFF_MODE_LOO) {
        L.Wo16 = L.take((size_t)D * H * dh * 2);
        L.cn = L.take((size_t)2 * cnorm_groups(D) * H * L.T_pad * 4);
        L.rho = L.take((size_t)H * L.T_pad * 4);
      }
    } else {
      L.Rg = (H / G + 2) * dh;
      L.n_tchunks = ceil_div(T, kDownTokenChunk);
      L.alpha16 = L.take((size_t)L.T_pad * L.I_pad * 2);
      L.Wd16 = L.take((size_t)D * L.I_pad * 2);
      L.WdT16 = L.take((size_t)L.I_pad * D * 2);
      L.Wqkv16 = L.take((size_t)G * L.Rg * 2 * D * 2);
      L.ssx = L.take((size_t)xprime_groups(D) * L.T_pad * 4);
      L.cpart = L.take((size_t)L.n_tchunks * L.I_pad * 4);
      L.bnorm = L.take((size_t)2 * L.I_pad * G * 4);
    }
  } else {
    L.I_pad = I;
    L.T_pad = T;
    L.n32 = L.take((size_t)T * D * 4);
    if (!down) {
      L.n_chunks = ceil_div(T, 128);
      L.a32 = L.take((size_t)T * H * dh * 4);
      L.M32 = L.take((size_t)2 * H * I * dh * 4);
      if (mode == AFF_MODE_FO) L.ab = L.take((size_t)T * I * 8);
      L.partial = L.take((size_t)L.n_chunks * H * I * 4);
      L.headsum = L.take((size_t)H * I * 8);
      if (mode == AFF_MODE_FO) L.wdn = L.take((size_t)I * 4);
    } else {
      L.n_tchunks = ceil_div(T, kDownTokenChunk);
      L.alpha32 = L.take((size_t)T * I * 4);
      L.ssx = L.take((size_t)2 * T * 4);
      L.cpart = L.take((size_t)L.n_tchunks * I * 4);
      L.bnorm = L.take((size_t)I * G * 4);
    }
  }
  L.total = (size_t)round_up((int64_t)L.total, 1024);
  return L;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    cudaGetLastError();
  });
  return fn;
}

// fp16 tensor of `rank` dims (dims[0] innermost, contiguous), 128 B swizzle,
// box = 64 innermost elements x box1 (x 1 in the other dims); OOB reads zero.
aff_status make_map(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims, const uint64_t* strides,
                    uint32_t box1, int box1_dim, uint32_t box2 = 1, int box2_dim = -1) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    g_last_cuda_error = "cuTensorMapEncodeTiled unavailable";
    return AFF_ERR_CUDA;
  }
  cuuint64_t gd[5], gs[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = 1;
    es[i] = 1;
  }
  for (int i = 0; i < rank - 1; ++i) gs[i] = strides[i];
  bx[0] = 64;
  bx[box1_dim] = box1;
  if (box2_dim > 0) bx[box2_dim] = box2;
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, (cuuint32_t)rank, const_cast<void*>(ptr), gd, gs, bx, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[96];
    std::snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    g_last_cuda_error = buf;
    return AFF_ERR_CUDA;
  }
  return AFF_OK;
}

// 16-bit tensor [rows][inner] (row stride inner * 2 bytes), box (32 innermost
// elements = 64 bytes, box1 rows), 64-byte swizzle; OOB reads zero.
aff_status map_sw64_2d(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows, uint32_t box1) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    g_last_cuda_error = "cuTensorMapEncodeTiled unavailable";
    return AFF_ERR_CUDA;
  }
  cuuint64_t gd[2] = {inner, rows}, gs[1] = {inner * 2};
  cuuint32_t bx[2] = {32, box1}, es[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(ptr), gd, gs, bx, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[96];
    std::snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    g_last_cuda_error = buf;
    return AFF_ERR_CUDA;
  }
  return AFF_OK;
}

// The gate (part 0) or up (part 1) rows of 128 consecutive neurons of W16
// ([I_pad / 16][2][16][D]) as one box: dims (D, 16, 2, I_pad / 16), box (64, 16, 1, 8).
aff_status map_gate_up(CUtensorMap* m, const void* W16, uint64_t D, uint64_t I_pad) {
  uint64_t d[4] = {D, 16, 2, I_pad / 16}, s[3] = {D * 2, 16 * D * 2, 32 * D * 2};
  return make_map(m, W16, 4, d, s, 16, 1, 8, 3);
}

aff_status map2(CUtensorMap* m, const void* p, uint64_t inner, uint64_t rows) {
  uint64_t d[2] = {inner, rows}, s[1] = {inner * 2};
  return make_map(m, p, 2, d, s, 128, 1);
}

int pick_stages(int mode, int H) {
  for (int s = 6; s >= 2; --s)
    if (tile_smem_bytes(mode, s, H) <= (size_t)kMaxDynSmem) return s;
  return 0;
}

// Heads whose width is a multiple of 16 but not of 64 (e.g. 96) leave the last
// 64-wide K block of every head job partly empty.  Streaming all heads' K
// ranges back to back fills every block; AFFINITY_STREAM_HEADS=0 turns it off.
bool stream_heads(const aff_dims& d) {
  static const bool allowed = [] {
    const char* e = std::getenv("AFFINITY_STREAM_HEADS");
    return !(e && e[0] == '0');
  }();
  return allowed && d.d_head % 16 == 0 && d.d_head % 64 != 0;
}

// ADD in the second-moment form: fold units run before the Gram pass, beside 1/r --
// those past the last whole round of one unit per SM, so that the rest take whole
// rounds after it.  AFFINITY_FOLD_EARLY=<n> sets the count (0: none).
int fold_early_units(int n_units, int sm_count) {
  const char* e = std::getenv("AFFINITY_FOLD_EARLY");   // read per call: tests vary it
  const int forced = e ? std::atoi(e) : -1;
  int n = forced >= 0 ? forced : (n_units > sm_count && sm_count > 0 ? n_units % sm_count : 0);
  return n < n_units ? n : n_units;
}

TileParams base_params(const aff_dims& d, const Layout& L, uint8_t* ws, int mode) {
  TileParams p{};
  p.mode = mode;
  p.T = (int)d.T;
  p.D = (int)d.D;
  p.H = (int)d.H;
  p.G = (int)d.G;
  p.dh = (int)d.d_head;
  p.I = (int)d.I;
  p.I_pad = (int)L.I_pad;
  p.T_pad = (int)L.T_pad;
  p.n_ktiles = (int)(L.I_pad / 128);
  p.n_ttiles = (int)(L.T_pad / 128);
  p.tiles_per_unit = kTilesPerUnit;
  p.nkb_D = (int)ceil_div(d.D, 64);
  p.nkb_dh = (int)ceil_div(d.d_head, 64);
  p.nkb_I = (int)(L.I_pad / 64);
  p.ls_D = (int)(((d.D - 1) % 64) / 16 + 1);          // 16-wide K slices in the last block of D
  p.ls_dh = (int)(((d.d_head - 1) % 64) / 16 + 1);    // ... and of d_head
  p.stages = pick_stages(mode, p.H);
  if (stream_heads(d)) {
    const int64_t slices = d.H * d.d_head / 16;
    p.stream_heads = 1;
    p.nkb_HD = (int)ceil_div(slices, 4);
    p.ls_HD = (int)((slices - 1) % 4 + 1);
    p.spp = (int)(d.d_head / 16);
  }
  p.status = reinterpret_cast<uint32_t*>(ws + L.status);
  p.sc = reinterpret_cast<const DevScales*>(ws + L.scales);
  p.eps = d.eps;
  return p;
}

aff_status run_tile(const CUtensorMap* maps, TileParams& p, cudaStream_t s, bool dominant = false, int max_ctas = 0) {
  if (p.n_units - p.unit0 <= 0) return AFF_OK;
  // CTAs resident at once, cached per device and configuration
  static std::mutex mu;
  static std::vector<std::pair<std::vector<int>, int>> cache;
  int dev = 0;
  AFF_CUDA(cudaGetDevice(&dev));
  const std::vector<int> key = {dev, p.mode, p.stages, p.H};
  int fit = 0;
  {
    std::lock_guard<std::mutex> lk(mu);
    for (auto& kv : cache)
      if (kv.first == key) fit = kv.second;
  }
  if (fit <= 0) {
    cudaError_t e = launch_tile_kernel(maps, p, &fit, s);
    if (e != cudaSuccess) return cuda_fail(e, "tile kernel occupancy query");
    if (fit <= 0) {
      g_last_cuda_error = "the tile kernel does not fit on this device";
      return AFF_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(mu);
    cache.push_back({key, fit});
  }
  int grid = p.n_units - p.unit0 < fit ? p.n_units - p.unit0 : fit;
  if (max_ctas > 0 && grid > max_ctas) grid = max_ctas;
  const bool timed = dominant && g_timing_start && g_timing_stop;
  if (timed) AFF_CUDA(cudaEventRecord(g_timing_start, s));
  cudaError_t e = launch_tile_kernel(maps, p, &grid, s);
  if (e != cudaSuccess) return cuda_fail(e, "affinity_tile_kernel");
  if (timed) AFF_CUDA(cudaEventRecord(g_timing_stop, s));
  return AFF_OK;
}

// A second stream (and two events) per host thread and device: the weight-side
// preparation runs on it concurrently with the token-side preparation, forked
// from and joined back into the caller's stream, so ordering relative to the
// caller's other work is unchanged.  Created on first use, kept for the life
// of the process (no device memory is involved).
struct SideStream {
  int dev = -1;
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr, join_late = nullptr, mid = nullptr;
};

aff_status side_stream(SideStream** out) {
  thread_local std::deque<SideStream> per_dev;   // a deque keeps earlier entries in place
  int dev = 0;
  AFF_CUDA(cudaGetDevice(&dev));
  for (auto& ss : per_dev)
    if (ss.dev == dev) {
      *out = &ss;
      return AFF_OK;
    }
  SideStream ss;
  ss.dev = dev;
  AFF_CUDA(cudaStreamCreateWithFlags(&ss.stream, cudaStreamNonBlocking));
  AFF_CUDA(cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming));
  AFF_CUDA(cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming));
  AFF_CUDA(cudaEventCreateWithFlags(&ss.join_late, cudaEventDisableTiming));
  AFF_CUDA(cudaEventCreateWithFlags(&ss.mid, cudaEventDisableTiming));
  per_dev.push_back(ss);
  *out = &per_dev.back();
  return AFF_OK;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

aff_status check_ws(const Layout& L, void* ws, size_t bytes) {
  if (!ws) return AFF_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) & 255u) return AFF_ERR_WORKSPACE;
  if (bytes < L.total) return AFF_ERR_WORKSPACE;
  return AFF_OK;
}

}  // namespace

extern "C" {

int32_t affinity_version(void) { return 100; }

aff_status affinity_set_timing_events(void* start_event, void* stop_event) {
  if ((start_event == nullptr) != (stop_event == nullptr)) return AFF_ERR_INVALID_ARG;
  g_timing_start = static_cast<cudaEvent_t>(start_event);
  g_timing_stop = static_cast<cudaEvent_t>(stop_event);
  return AFF_OK;
}

const char* affinity_strerror(aff_status s) {
  switch (s) {
    case AFF_OK: return "success";
    case AFF_ERR_INVALID_ARG: return "invalid argument (NULL pointer, bad enum value or non-positive size)";
    case AFF_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case AFF_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype";
    case AFF_ERR_ARCH: return "no sm_103 (GB300) device is current";
    case AFF_ERR_WORKSPACE: return "workspace missing, misaligned (256 B) or smaller than affinity_workspace_size()";
    case AFF_ERR_CUDA: return "a CUDA call failed (see affinity_last_cuda_error())";
    case AFF_ERR_DEVICE_TIMEOUT: return "a kernel's bounded wait expired";
    case AFF_ERR_RANGE: return "a non-finite input, or an fp16 intermediate overflowed where nothing rescales it";
    case AFF_ERR_ALIGNMENT: return "a device pointer is not 16-byte aligned";
    case AFF_ERR_NO_CONVERGENCE: return "an iterative solver reached its iteration cap";
  }
  return "unknown status";
}

const char* affinity_last_cuda_error(void) { return g_last_cuda_error.c_str(); }

aff_status affinity_workspace_size(const aff_dims* dims, int32_t mode, int32_t down, size_t* bytes) {
  if (!bytes) return AFF_ERR_INVALID_ARG;
  aff_status st = check_dims(dims);
  if (st != AFF_OK) return st;
  if (!down && mode != AFF_MODE_FO && mode != AFF_MODE_ADD && mode != AFF_MODE_LOO) return AFF_ERR_INVALID_ARG;
  if (!down && mode == AFF_MODE_LOO && dims->dtype != AFF_BF16) return AFF_ERR_UNSUPPORTED_DTYPE;
  *bytes = make_layout(*dims, mode, down != 0).total;
  return AFF_OK;
}

aff_status affinity_up(const void* a, const void* x, const void* Wo, const void* gamma, const void* Wg,
                       const void* Wu, const void* Wd, const aff_dims* dims, int32_t mode, float* S_out,
                       float* S_head_out, void* workspace, size_t workspace_bytes, aff_stream_t stream) {
  aff_status st = check_dims(dims);
  if (st != AFF_OK) return st;
  if (mode != AFF_MODE_FO && mode != AFF_MODE_ADD && mode != AFF_MODE_LOO) return AFF_ERR_INVALID_ARG;
  const bool fo = mode == AFF_MODE_FO;
  const bool loo = mode == AFF_MODE_LOO;
  if (loo && dims->dtype != AFF_BF16) return AFF_ERR_UNSUPPORTED_DTYPE;
  if (!a || !x || !Wo || !gamma || !Wg || !Wu || (fo && !Wd) || !S_out) return AFF_ERR_INVALID_ARG;
  const void* ptrs[] = {a, x, Wo, gamma, Wg, Wu, fo ? Wd : nullptr, S_out, S_head_out};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return AFF_ERR_ALIGNMENT;
  const aff_dims& d = *dims;
  Layout L = make_layout(d, mode, false);
  if ((st = check_ws(L, workspace, workspace_bytes)) != AFF_OK) return st;
  int sm_count = 0;
  if ((st = check_device(&sm_count)) != AFF_OK) return st;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws + L.status);
  AFF_CUDA(cudaMemsetAsync(status, 0, 4, s));
  const int T = (int)d.T, D = (int)d.D, H = (int)d.H, G = (int)d.G, dh = (int)d.d_head, I = (int)d.I;
  const int I_pad = (int)L.I_pad;
  float* wdn = fo ? reinterpret_cast<float*>(ws + L.wdn) : nullptr;
  double* headsum = reinterpret_cast<double*>(ws + L.headsum);

  if (d.dtype == AFF_FP32) {
    F32UpArgs A{};
    A.a = (const float*)a; A.x = (const float*)x; A.Wo = (const float*)Wo; A.gamma = (const float*)gamma;
    A.Wg = (const float*)Wg; A.Wu = (const float*)Wu;
    A.n32 = reinterpret_cast<float*>(ws + L.n32); A.a32 = reinterpret_cast<float*>(ws + L.a32);
    A.M32 = reinterpret_cast<float*>(ws + L.M32); A.partial = reinterpret_cast<float*>(ws + L.partial);
    A.ab = fo ? reinterpret_cast<float2*>(ws + L.ab) : nullptr;
    A.T = T; A.D = D; A.H = H; A.dh = dh; A.I = I; A.n_chunks = (int)L.n_chunks; A.chunk = 128; A.fo = fo;
    A.eps = d.eps;
    AFF_CUDA(launch_f32_up(A, s));
    AFF_CUDA(launch_reduce_partials(A.partial, headsum, (int)L.n_chunks, 1, H, I, s));
    if (fo) AFF_CUDA(launch_wd_colnorm_f32((const float*)Wd, wdn, D, I, s));
    AFF_CUDA(launch_finalize_up(headsum, wdn, fo, T, H, G, I, I, S_out, S_head_out, s));
    return AFF_OK;
  }

  // ---- bf16 path: stage fp16 operands, fold, contract, reduce
  __half* W16 = reinterpret_cast<__half*>(ws + L.W16);
  __half* GWo16 = reinterpret_cast<__half*>(ws + L.GWo16);
  __half* M16 = reinterpret_cast<__half*>(ws + L.M16);
  __half* n16 = reinterpret_cast<__half*>(ws + L.n16);
  __half* a16 = reinterpret_cast<__half*>(ws + L.a16);
  float* partial = reinterpret_cast<float*>(ws + L.partial);
  const uint16_t* a_b = static_cast<const uint16_t*>(a);
  const uint16_t* x_b = static_cast<const uint16_t*>(x);
  const uint16_t* g_b = static_cast<const uint16_t*>(gamma);

  // Power-of-two scales of the fp16 operands (scales.cuh): their maxima start at zero.
  DevScales* sc = reinterpret_cast<DevScales*>(ws + L.scales);
  AFF_CUDA(cudaMemsetAsync(sc, 0, sizeof(DevScales), s));
  // weight side (weight maxima, fp16 gate/up rows, gamma*Wo^T, ||w^d||^2, the fold) on the side stream
  SideStream* side = nullptr;
  if ((st = side_stream(&side)) != AFF_OK) return st;
  const cudaStream_t ws2 = side->stream;
  AFF_CUDA(cudaEventRecord(side->fork, s));
  AFF_CUDA(cudaStreamWaitEvent(ws2, side->fork, 0));
  // The weight side (maxima, fp16 gate/up rows, gamma*Wo^T, the fold) runs on the side stream.
  // FO / LOO / direct ADD: beside the token staging on the caller's stream.  ADD in the
  // second-moment form: 1/r and then the Gram pass run first on the caller's stream (the Gram
  // reading a through an L2 that holds no dirty lines of this call yet); the fold, which wants
  // every SM as the Gram pass does, follows the Gram on the caller's stream, and the Gram
  // reduction runs beside it on the side stream, so that the path from the Gram through the
  // fold to the quadratic forms crosses no stream.  The fold's units past its last whole round
  // run before the Gram instead, beside 1/r.
  const bool moment = moment_form(d, mode);
  const cudaStream_t wst = ws2;
  float* ir_m = moment ? reinterpret_cast<float*>(ws + L.ir) : nullptr;
  if (moment) AFF_CUDA(launch_inv_r(x_b, ir_m, T, gram_split(T, H).nkb * 64, D, d.eps, sm_count, s));
  // weights staged unscaled with their maxima recorded, then staged again only if a
  // maximum lies outside fp16's comfortable range (scales.cuh)
  AFF_CUDA(launch_weight_stage((const uint16_t*)Wg, (const uint16_t*)Wu, W16, I, I_pad, D, (const uint16_t*)Wo, g_b,
                               GWo16, H * dh, sc, sm_count, wst));
  __half* Wo16 = loo ? reinterpret_cast<__half*>(ws + L.Wo16) : nullptr;
  float* inv_r = moment ? nullptr : reinterpret_cast<float*>(ws + L.inv_r);
  if (loo) AFF_CUDA(launch_to_fp16((const uint16_t*)Wo, Wo16, (size_t)D * H * dh, status, wst));
  AFF_CUDA(launch_weight_restage((const uint16_t*)Wg, (const uint16_t*)Wu, W16, I, I_pad, D, (const uint16_t*)Wo, g_b,
                                 GWo16, Wo16, H * dh, sc, status, sm_count, wst));

  // fold: M_h = [Wg; Wu] diag(gamma) Wo^(h), units of (128 rows of W16, 256 columns of H*dh):
  // A = W16 rows, B = gamma*Wo^T hi, then lo
  CUtensorMap fmaps[4];
  std::memset(fmaps, 0, sizeof fmaps);
  if ((st = map2(&fmaps[0], W16, (uint64_t)D, (uint64_t)2 * I_pad)) != AFF_OK) return st;
  {
    uint64_t dm[3] = {(uint64_t)D, 2, (uint64_t)H * dh}, sd[2] = {(uint64_t)D * 2, (uint64_t)D * 4};
    if ((st = make_map(&fmaps[1], GWo16, 3, dm, sd, 128, 2)) != AFF_OK) return st;
  }
  fmaps[2] = fmaps[0];
  fmaps[3] = fmaps[0];
  TileParams fp = base_params(d, L, ws, kModeFold);
  fp.n_ntiles = (int)ceil_div((int64_t)H * dh, 256);
  fp.n_units = 2 * fp.n_ktiles * fp.n_ntiles;
  fp.M16 = M16;
  // ADD, second-moment form: the units past the last whole round of the fold run first, on
  // the side stream beside 1/r (which needs few SMs); the rest follow the Gram pass
  const int fold_early = moment ? fold_early_units(fp.n_units, sm_count) : 0;
  if (moment) {
    AFF_CUDA(cudaEventRecord(side->join_late, ws2));   // the staged weights are ready
    if (fold_early > 0) {
      TileParams p1 = fp;
      p1.unit0 = fp.n_units - fold_early;
      if ((st = run_tile(fmaps, p1, ws2)) != AFF_OK) return st;
    }
  }
  // token side on the caller's stream meanwhile
  if (!moment) {
    AFF_CUDA(launch_prep_tokens(x_b, a_b, g_b, (fo || loo) ? n16 : nullptr, a16, inv_r, T, D, H * dh, d.eps, status,
                                sm_count, sc, s));
    AFF_CUDA(launch_restage_a(a_b, inv_r, a16, T, H * dh, sc, status, sm_count, s));
  }

  // ADD, second-moment form: C_h over the tokens (Gram pass), then m^T C_h m for every
  // folded row, then the group sums
  const GramSplit gs = gram_split(T, H);
  float* gram = moment ? reinterpret_cast<float*>(ws + L.gram) : nullptr;
  float* cmax = moment ? reinterpret_cast<float*>(ws + L.cmax) : nullptr;
  __half* CC = moment ? reinterpret_cast<__half*>(ws + L.CC) : nullptr;
  float* gscale = moment ? reinterpret_cast<float*>(ws + L.gscale) : nullptr;
  CUtensorMap mm[2];
  std::memset(mm, 0, sizeof mm);
  if (moment) {
    // a (bf16 bits) as [T][H*dh], boxes of 32 columns x 64 tokens, 64-byte swizzle
    if ((st = map_sw64_2d(&mm[0], a, (uint64_t)H * dh, (uint64_t)T, 64)) != AFF_OK) return st;
    mm[1] = mm[0];
    MomentParams mp{};
    mp.mode = kMomentGram;
    mp.n_units = gs.n_chunks * H;
    mp.H = H; mp.dh = dh; mp.HD = H * dh; mp.I_pad = I_pad;
    mp.nkb = gs.nkb; mp.kpc = gs.kpc;
    mp.status = status;
    mp.gram = gram;
    mp.cmax = cmax;
    mp.inv_r = ir_m;
    const bool timed = g_timing_start && g_timing_stop;
    if (timed) AFF_CUDA(cudaEventRecord(g_timing_start, s));
    AFF_CUDA(launch_moment(mm, mp, s));
    if (timed) AFF_CUDA(cudaEventRecord(g_timing_stop, s));
    // the Gram reduction on the side stream once the Gram pass is done; the fold next on
    // this stream once the staged weights are ready (recorded before the side stream
    // waits for the Gram, so that this wait is already met)
    AFF_CUDA(cudaEventRecord(side->mid, s));
    AFF_CUDA(cudaStreamWaitEvent(ws2, side->mid, 0));
    AFF_CUDA(cudaStreamWaitEvent(s, side->join_late, 0));
    AFF_CUDA(launch_gram_reduce(gram, cmax, CC, gscale, gs.n_chunks, H, dh, status, a_b, ir_m, T, sc, ws2));
  }

  {
    TileParams p2 = fp;
    p2.n_units = fp.n_units - fold_early;   // moment form: the units not run before the Gram pass
    if ((st = run_tile(fmaps, p2, moment ? s : wst)) != AFF_OK) return st;
  }
  CUtensorMap maps[4];
  std::memset(maps, 0, sizeof maps);
  AFF_CUDA(cudaEventRecord(side->join, ws2));
  if (moment) {
    AFF_CUDA(cudaStreamWaitEvent(s, side->join, 0));
    {
      if (stream_heads(d)) {
        if ((st = map2(&mm[0], M16, (uint64_t)H * dh, (uint64_t)2 * I_pad)) != AFF_OK) return st;
      } else {
        uint64_t dm[3] = {(uint64_t)dh, (uint64_t)2 * I_pad, (uint64_t)H};
        uint64_t sd[2] = {(uint64_t)dh * 2, (uint64_t)2 * I_pad * dh * 2};
        if ((st = make_map(&mm[0], M16, 3, dm, sd, kMomentRows, 1)) != AFF_OK) return st;
      }
      if ((st = map2(&mm[1], CC, (uint64_t)kMomentRows, (uint64_t)2 * H * kMomentRows)) != AFF_OK) return st;
      MomentParams mp{};
      mp.mode = kMomentQuad;
      mp.n_units = (int)(2 * L.I_pad / kMomentRows) * H;
      mp.H = H; mp.dh = dh; mp.HD = H * dh; mp.I_pad = I_pad;
      mp.nkb = (int)ceil_div(dh, 64);
      mp.stream = stream_heads(d) ? 1 : 0;
      mp.ctas = 2 * sm_count;
      mp.status = status;
      mp.scale = gscale;
      mp.M16 = M16;
      mp.out = partial;
      AFF_CUDA(launch_moment(mm, mp, s));
    }
    AFF_CUDA(launch_moment_finalize(partial, T, H, G, I, I_pad, S_out, S_head_out, sc, D, s));
    return AFF_OK;
  }
  AFF_CUDA(cudaStreamWaitEvent(s, side->join, 0));
  // ||w^d||^2 is needed only by the last kernel: computed after the fold, joined late
  if (fo) AFF_CUDA(launch_wd_colnorm((const uint16_t*)Wd, wdn, D, I, I_pad, ws2));
  AFF_CUDA(cudaEventRecord(side->join_late, ws2));
  float* rho = loo ? reinterpret_cast<float*>(ws + L.rho) : nullptr;
  if (loo) {
    // sigma[h][t] = 1 - r / rms(x - c_h): tensor-core pass over (a_h / r) Wo^(h)^T with the
    // per-token sums over d in the epilogue, then a small kernel
    float* cn = reinterpret_cast<float*>(ws + L.cn);
    uint64_t da[3] = {(uint64_t)dh, (uint64_t)H, (uint64_t)T};
    uint64_t sa[2] = {(uint64_t)dh * 2, (uint64_t)H * dh * 2};
    if ((st = make_map(&maps[0], a16, 3, da, sa, 128, 2)) != AFF_OK) return st;
    if ((st = map2(&maps[1], Wo16, (uint64_t)H * dh, (uint64_t)D)) != AFF_OK) return st;
    maps[2] = maps[0];
    maps[3] = maps[0];
    TileParams p = base_params(d, L, ws, kModeCNorm);
    p.n_ntiles = (int)ceil_div(D, 256);
    p.n_units = (int)(L.T_pad / 128 * p.n_ntiles);
    p.partial = cn;
    p.x_bf16 = x_b;
    if ((st = run_tile(maps, p, s)) != AFF_OK) return st;
    AFF_CUDA(launch_loo_rho(cn, inv_r, rho, T, (int)L.T_pad, H, D, cnorm_groups(D), sc, s));
  }
  int epi_groups = 2;   // column groups of the epilogue in the partial sums (set below)
  // FO / ADD / LOO: per (256 tokens, 64 neurons), operating point (FO, LOO) then every head
  {
    const uint32_t brows = 128u;
    uint64_t dx[2] = {(uint64_t)D, (uint64_t)T}, sx[1] = {(uint64_t)D * 2};
    if ((st = map2(&maps[0], W16, (uint64_t)D, (uint64_t)2 * I_pad)) != AFF_OK) return st;
    if (fo || loo) {
      if ((st = make_map(&maps[1], n16, 2, dx, sx, brows, 1)) != AFF_OK) return st;
    } else {
      maps[1] = maps[0];
    }
    if (stream_heads(d)) {
      // M16 as [2 I_pad][H*dh] and a16 as [T][H*dh]: K blocks run across head boundaries
      if ((st = map2(&maps[2], M16, (uint64_t)H * dh, (uint64_t)2 * I_pad)) != AFF_OK) return st;
      if ((st = map2(&maps[3], a16, (uint64_t)H * dh, (uint64_t)T)) != AFF_OK) return st;
    } else {
      uint64_t dm[3] = {(uint64_t)dh, (uint64_t)2 * I_pad, (uint64_t)H};
      uint64_t sd[2] = {(uint64_t)dh * 2, (uint64_t)2 * I_pad * dh * 2};
      if ((st = make_map(&maps[2], M16, 3, dm, sd, 128, 1)) != AFF_OK) return st;
      uint64_t da[3] = {(uint64_t)dh, (uint64_t)H, (uint64_t)T};
      uint64_t sa[2] = {(uint64_t)dh * 2, (uint64_t)H * dh * 2};
      if ((st = make_map(&maps[3], a16, 3, da, sa, brows, 2)) != AFF_OK) return st;
    }
    TileParams p = base_params(d, L, ws, fo ? kModeFO : (loo ? kModeLOO : kModeADD));
    // CTAs claim units from a counter (zeroed with the scales at the start of the call), so
    // that CTAs on faster SMs take more of them and the pass ends with less of a tail
    p.ucount = &reinterpret_cast<DevScales*>(ws + L.scales)->units;
    p.rho = rho;
    p.n_units = (int)(L.n_chunks * 2 * p.n_ktiles);   // (512 tokens, 64 neurons)
    p.partial = partial;
    epi_groups = epi_warps(p.mode) / 4;
    if ((st = run_tile(maps, p, s, true)) != AFF_OK) return st;
  }
  AFF_CUDA(cudaStreamWaitEvent(s, side->join_late, 0));
  AFF_CUDA(launch_reduce_finalize(partial, wdn, fo, (int)L.n_chunks, epi_groups, T, H, G, I, I_pad, S_out,
                                  S_head_out, reinterpret_cast<const DevScales*>(ws + L.scales), D, s));
  return AFF_OK;
}

aff_status affinity_down(const void* x, const void* gamma, const void* Wg, const void* Wu, const void* Wd,
                         const void* gamma_next, const void* Wq_next, const void* Wk_next, const void* Wv_next,
                         const aff_dims* dims, float* S_out, void* workspace, size_t workspace_bytes,
                         aff_stream_t stream) {
  aff_status st = check_dims(dims);
  if (st != AFF_OK) return st;
  if (!x || !gamma || !Wg || !Wu || !Wd || !gamma_next || !Wq_next || !Wk_next || !Wv_next || !S_out)
    return AFF_ERR_INVALID_ARG;
  const void* ptrs[] = {x, gamma, Wg, Wu, Wd, gamma_next, Wq_next, Wk_next, Wv_next, S_out};
  for (const void* p : ptrs)
    if (!aligned16(p)) return AFF_ERR_ALIGNMENT;
  const aff_dims& d = *dims;
  Layout L = make_layout(d, 0, true);
  if ((st = check_ws(L, workspace, workspace_bytes)) != AFF_OK) return st;
  int sm_count = 0;
  if ((st = check_device(&sm_count)) != AFF_OK) return st;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws + L.status);
  AFF_CUDA(cudaMemsetAsync(status, 0, 4, s));
  const int T = (int)d.T, D = (int)d.D, H = (int)d.H, G = (int)d.G, dh = (int)d.d_head, I = (int)d.I;
  const int I_pad = (int)L.I_pad, T_pad = (int)L.T_pad;
  float* ssx = reinterpret_cast<float*>(ws + L.ssx);
  float* cpart = reinterpret_cast<float*>(ws + L.cpart);
  float* bnorm = reinterpret_cast<float*>(ws + L.bnorm);

  if (d.dtype == AFF_FP32) {
    F32DownArgs A{};
    A.x = (const float*)x; A.gamma = (const float*)gamma; A.Wg = (const float*)Wg; A.Wu = (const float*)Wu;
    A.Wd = (const float*)Wd; A.gamma_next = (const float*)gamma_next; A.Wq = (const float*)Wq_next;
    A.Wk = (const float*)Wk_next; A.Wv = (const float*)Wv_next;
    A.n32 = reinterpret_cast<float*>(ws + L.n32); A.alpha32 = reinterpret_cast<float*>(ws + L.alpha32);
    A.ssx = ssx; A.cpart = cpart; A.bnorm = bnorm;
    A.T = T; A.D = D; A.H = H; A.G = G; A.dh = dh; A.I = I; A.n_chunks = (int)L.n_tchunks;
    A.chunk = kDownTokenChunk; A.eps = d.eps;
    AFF_CUDA(launch_f32_down(A, s));
    AFF_CUDA(launch_finalize_down(cpart, bnorm, (int)L.n_tchunks, 1, T, I, I, G, S_out, s));
    return AFF_OK;
  }

  __half* W16 = reinterpret_cast<__half*>(ws + L.W16);
  __half* n16 = reinterpret_cast<__half*>(ws + L.n16);
  __half* alpha16 = reinterpret_cast<__half*>(ws + L.alpha16);
  __half* Wd16 = reinterpret_cast<__half*>(ws + L.Wd16);
  __half* WdT16 = reinterpret_cast<__half*>(ws + L.WdT16);
  __half* Wqkv16 = reinterpret_cast<__half*>(ws + L.Wqkv16);

  // The weight side is staged on a side stream while the tokens are normalised on
  // the caller's stream; the side stream later runs the ||b_gk||^2 pass, which
  // needs only weights, beside the token-weight pass.
  SideStream* side = nullptr;
  if ((st = side_stream(&side)) != AFF_OK) return st;
  const cudaStream_t ws2 = side->stream;
  DevScales* sc = reinterpret_cast<DevScales*>(ws + L.scales);
  AFF_CUDA(cudaMemsetAsync(sc, 0, sizeof(DevScales), s));
  AFF_CUDA(cudaEventRecord(side->fork, s));
  AFF_CUDA(cudaStreamWaitEvent(ws2, side->fork, 0));
  AFF_CUDA(launch_prep_gate_up((const uint16_t*)Wg, (const uint16_t*)Wu, W16, I, I_pad, D, sc, ws2));
  AFF_CUDA(launch_weight_restage((const uint16_t*)Wg, (const uint16_t*)Wu, W16, I, I_pad, D, nullptr, nullptr, nullptr,
                                 nullptr, 0, sc, status, sm_count, ws2));
  AFF_CUDA(launch_prep_wd((const uint16_t*)Wd, Wd16, WdT16, D, I, I_pad, status, ws2));
  AFF_CUDA(launch_prep_qkv((const uint16_t*)Wq_next, (const uint16_t*)Wk_next, (const uint16_t*)Wv_next,
                           (const uint16_t*)gamma_next, Wqkv16, G, H / G, dh, D, status, ws2));
  AFF_CUDA(cudaEventRecord(side->join, ws2));
  AFF_CUDA(launch_prep_tokens((const uint16_t*)x, nullptr, (const uint16_t*)gamma, n16, nullptr, nullptr, T, D, 0,
                              d.eps, status, sm_count, sc, s));
  AFF_CUDA(cudaStreamWaitEvent(s, side->join, 0));
  CUtensorMap maps[4];
  std::memset(maps, 0, sizeof maps);
  // alpha = silu(g) u for every (token, neuron)
  {
    if ((st = map_gate_up(&maps[0], W16, (uint64_t)D, (uint64_t)I_pad)) != AFF_OK) return st;
    if ((st = map2(&maps[1], n16, (uint64_t)D, (uint64_t)T)) != AFF_OK) return st;
    maps[2] = maps[0];
    maps[3] = maps[0];
    TileParams p = base_params(d, L, ws, kModeAlpha);
    p.n_units = (int)(ceil_div(p.n_ttiles, kTilesPerUnit) * p.n_ktiles);
    p.alpha16 = alpha16;
    if ((st = run_tile(maps, p, s, true)) != AFF_OK) return st;
  }
  // x' = x + alpha Wd^T and sum_d x'^2 per token
  {
    if ((st = map2(&maps[0], alpha16, (uint64_t)I_pad, (uint64_t)T_pad)) != AFF_OK) return st;
    if ((st = map2(&maps[1], Wd16, (uint64_t)I_pad, (uint64_t)D)) != AFF_OK) return st;
    maps[2] = maps[0];
    maps[3] = maps[0];
    TileParams p = base_params(d, L, ws, kModeXPrime);
    p.n_ntiles = (int)ceil_div(D, 256);
    p.n_units = (int)(T_pad / 128 * p.n_ntiles);
    p.partial = ssx;
    p.x_bf16 = (const uint16_t*)x;
    if ((st = run_tile(maps, p, s)) != AFF_OK) return st;
  }
  // ||b_gk||^2 for every neuron and group, on the side stream once the tensor-core
  // passes before it are done
  AFF_CUDA(cudaEventRecord(side->fork, s));
  AFF_CUDA(cudaStreamWaitEvent(ws2, side->fork, 0));
  {
    if ((st = map2(&maps[0], WdT16, (uint64_t)D, (uint64_t)I_pad)) != AFF_OK) return st;
    uint64_t dm[4] = {(uint64_t)D, 2, (uint64_t)L.Rg, (uint64_t)G};
    uint64_t sd[3] = {(uint64_t)D * 2, (uint64_t)D * 4, (uint64_t)L.Rg * D * 4};
    if ((st = make_map(&maps[1], Wqkv16, 4, dm, sd, 128, 2)) != AFF_OK) return st;
    maps[2] = maps[0];
    maps[3] = maps[0];
    TileParams p = base_params(d, L, ws, kModeQNorm);
    p.n_ntiles = (int)ceil_div(L.Rg, 256);
    p.rows_per_group = (int)L.Rg;
    p.n_units = (int)(I_pad / 128 * G);
    p.bnorm = bnorm;
    if ((st = run_tile(maps, p, ws2)) != AFF_OK) return st;
  }
  AFF_CUDA(cudaEventRecord(side->join_late, ws2));
  AFF_CUDA(launch_down_token_weights(alpha16, ssx, cpart, T, T_pad, D, I_pad, kDownTokenChunk, d.eps,
                                     xprime_groups(D), s));
  AFF_CUDA(cudaStreamWaitEvent(s, side->join_late, 0));
  AFF_CUDA(launch_finalize_down(cpart, bnorm, (int)L.n_tchunks, 2, T, I, I_pad, G, S_out, s));
  return AFF_OK;
}

aff_status affinity_selftest_timeout(void* workspace, size_t workspace_bytes, int64_t limit_ns, aff_stream_t stream) {
  if (!workspace || workspace_bytes < 256 || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return AFF_ERR_WORKSPACE;
  if (limit_ns < 1000 || limit_ns > 10000000000LL) return AFF_ERR_INVALID_ARG;
  int sm_count = 0;
  aff_status st = check_device(&sm_count);
  if (st != AFF_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t* status = static_cast<uint32_t*>(workspace);
  AFF_CUDA(cudaMemsetAsync(status, 0, 4, s));
  AFF_CUDA(launch_wait_selftest(status, (unsigned long long)limit_ns, s));
  return AFF_OK;
}

aff_status affinity_device_status(void* workspace, aff_stream_t stream) {
  if (!workspace) return AFF_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  AFF_CUDA(cudaStreamSynchronize(s));
  AFF_CUDA(cudaMemcpy(&v, workspace, 4, cudaMemcpyDeviceToHost));
  AFF_CUDA(cudaMemset(workspace, 0, 4));
  return static_cast<aff_status>(v);
}

}  // extern "C"
