// bfp8_api.cu -- the libbfp8 C ABI: argument validation, device checks,
// schedule planning, TMA tensor maps and kernel launches.  See include/bfp8.h
// for the contract of every entry point.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/bfp8.h"
#include "bfp8_gemm_kernel.cuh"
#include "bfp8_internal.h"
#include "bfp8_ptx.cuh"

namespace bfp8 {
namespace {

// Library-owned device state: the failure word kernels report into.
__device__ int g_dev_err;
__device__ unsigned long long g_selftest_elapsed;
__device__ int g_selftest_ok;

constexpr unsigned long long kWaitLimitCycles = 1ull << 31;  // ~1 s at 2 GHz
constexpr int kMaxDevices = 64;

thread_local std::string t_last_error;

bfp8_status fail(bfp8_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return st;
}

bfp8_status ok() {
  t_last_error.clear();
  return BFP8_OK;
}

}  // namespace

bfp8_status set_last_error(bfp8_status st, const char* msg) {
  t_last_error = msg ? msg : "";
  return st;
}

namespace {

constexpr int kMaxCluster = 8;   // portable cluster size

struct DevInfo {
  bool ready = false;
  int cc_major = 0, cc_minor = 0, sms = 0;
  int* err = nullptr;
  bool caps_ready = false;
  // co-resident GEMM clusters of each size: one-CTA-per-SM instantiations,
  // and the swap-AB ones sized for two CTAs per SM
  int cluster_cap[kMaxCluster + 1] = {};
  int cluster_cap2[kMaxCluster + 1] = {};
};
DevInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Checks the current device is an sm_103 part and caches its properties.
bfp8_status current_device(DevInfo* out, int* dev_out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(BFP8_ERR_UNSUPPORTED, "no CUDA device: %s", cudaGetErrorString(e));
  }
  if (dev < 0 || dev >= kMaxDevices) return fail(BFP8_ERR_UNSUPPORTED, "device index %d", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return fail(BFP8_ERR_CUDA, "cudaDeviceGetAttribute failed on device %d", dev);
    }
    if (d.cc_major == 10 && d.cc_minor == 3) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_dev_err);
      if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(BFP8_ERR_CUDA, "cudaGetSymbolAddress(failure word): %s", cudaGetErrorString(e));
      }
      d.err = static_cast<int*>(p);
    }
    d.ready = true;
  }
  if (!(d.cc_major == 10 && d.cc_minor == 3))
    return fail(BFP8_ERR_UNSUPPORTED, "device %d is sm_%d%d; libbfp8 is built for sm_103a only", dev,
                d.cc_major, d.cc_minor);
  *out = d;
  if (dev_out) *dev_out = dev;
  return BFP8_OK;
}

// current_device plus the device's GEMM cluster capacities (asked once).
bfp8_status current_device_with_caps(DevInfo* out) {
  int dev = 0;
  bfp8_status st = current_device(out, &dev);
  if (st != BFP8_OK) return st;
  if (out->caps_ready) return BFP8_OK;
  int cap[kMaxCluster + 1] = {};
  int cap2[kMaxCluster + 1] = {};
  cap[0] = cap[1] = out->sms;
  cap2[0] = cap2[1] = 2 * out->sms;
  for (int cs = 2; cs <= kMaxCluster; ++cs) {
    cudaError_t e = gemm_cluster_capacity(cs, false, &cap[cs]);
    if (e == cudaSuccess) e = gemm_cluster_capacity(cs, true, &cap2[cs]);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(BFP8_ERR_CUDA, "cluster occupancy query (size %d): %s", cs, cudaGetErrorString(e));
    }
  }
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& d = g_dev[dev];
  std::memcpy(d.cluster_cap, cap, sizeof(cap));
  std::memcpy(d.cluster_cap2, cap2, sizeof(cap2));
  d.caps_ready = true;
  *out = d;
  return BFP8_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bfp8_status get_encoder(PFN_cuTensorMapEncodeTiled_v12000* fn) {
  std::call_once(g_encode_once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    cudaGetLastError();
  });
  if (!g_encode) return fail(BFP8_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  *fn = g_encode;
  return BFP8_OK;
}

// Tensor map over a [rows, inner] uint8 matrix (row stride `inner` bytes),
// box 128 (K) x box_rows, 128-byte swizzle, zero fill outside the matrix.
bfp8_status encode_operand(CUtensorMap* map, const void* ptr, int64_t rows, int64_t inner,
                           int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  bfp8_status st = get_encoder(&enc);
  if (st != BFP8_OK) return st;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner)};
  const cuuint32_t box[2] = {128u, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1u, 1u};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(BFP8_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for [%lld x %lld] box %d", (int)r,
                (long long)rows, (long long)inner, box_rows);
  return BFP8_OK;
}

// Tensor map over a [rows, K] uint8 matrix (row stride K bytes, K % 128 == 0)
// viewed as 128-byte k-block lines indexed (byte, row, k-block) -- strides K
// and 128 bytes: box 128 x box_rows x 8, i.e. eight k-blocks of box_rows rows,
// landing as [k-block][row][128 bytes]; 128-byte swizzle, zero fill outside
// the matrix (rows past `rows`, k-blocks past K / 128).
bfp8_status encode_kblocks(CUtensorMap* map, const void* ptr, int64_t rows, int64_t K,
                           int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  bfp8_status st = get_encoder(&enc);
  if (st != BFP8_OK) return st;
  const cuuint64_t dims[3] = {128u, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(K / 128)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K), 128u};
  const cuuint32_t box[3] = {128u, static_cast<cuuint32_t>(box_rows), 8u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(BFP8_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for [%lld x %lld] in k-blocks, box %d",
                (int)r, (long long)rows, (long long)K, box_rows);
  return BFP8_OK;
}

// Tensor map over the bf16 output [rows, cols] (row stride cols * 2 bytes,
// 16-byte aligned), box 32 x 32 with the 64-byte swizzle, for the wide
// tiles' TMA stores.
bfp8_status encode_output(CUtensorMap* map, void* ptr, int64_t rows, int64_t cols) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  bfp8_status st = get_encoder(&enc);
  if (st != BFP8_OK) return st;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2u};
  const cuuint32_t box[2] = {32u, 32u};
  const cuuint32_t estr[2] = {1u, 1u};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(BFP8_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for the [%lld x %lld] output",
                (int)r, (long long)rows, (long long)cols);
  return BFP8_OK;
}

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct Plan {
  bool swap = false;
  int bn = 0;
  int mr = 128;              // wide tiles: activation rows loaded per stage
  bool gemv = false;         // the matrix-vector kernel (few activation rows)
  bool pair = false;         // 256 x 256 tiles on CTA pairs (sched counts pairs)
  bool relayout = false;
  int64_t kp = 0;            // inner extent of the operand tensor maps
  Sched sched{};
  size_t off_counters = 0, off_partials = 0, off_a = 0, off_b = 0, off_as = 0, off_bs = 0,
         total = 0;
};

bfp8_status check_options(const bfp8_gemm_options* opt) {
  if (!opt) return BFP8_OK;
  if (opt->schedule < 0 || opt->schedule > 3)
    return fail(BFP8_ERR_INVALID_ARG, "options.schedule = %d (expected 0 .. 3)", opt->schedule);
  if (opt->max_ctas < 0) return fail(BFP8_ERR_INVALID_ARG, "options.max_ctas = %d", opt->max_ctas);
  if (opt->tile_n != 0 && opt->tile_n != 16 && opt->tile_n != 32 && opt->tile_n != 64 &&
      opt->tile_n != 128 && opt->tile_n != 256)
    return fail(BFP8_ERR_INVALID_ARG, "options.tile_n = %d (expected 0, 16, 32, 64, 128 or 256)",
                opt->tile_n);
  if (opt->schedule == BFP8_SCHEDULE_WIDE && opt->tile_n != 0 && opt->tile_n != 128 &&
      opt->tile_n != 256)
    return fail(BFP8_ERR_INVALID_ARG, "options.tile_n = %d: wide tiles are 128 or 256 wide",
                opt->tile_n);
  if (opt->prefetch_weights != 0 && opt->prefetch_weights != 1)
    return fail(BFP8_ERR_INVALID_ARG, "options.prefetch_weights = %d (expected 0 or 1)",
                opt->prefetch_weights);
  if (opt->k_split < 0 || opt->k_split > 3)
    return fail(BFP8_ERR_INVALID_ARG, "options.k_split = %d (expected 0 .. 3)", opt->k_split);
  if (opt->cluster_size != 0 && (opt->cluster_size < 2 || opt->cluster_size > kMaxCluster))
    return fail(BFP8_ERR_INVALID_ARG, "options.cluster_size = %d (expected 0 or 2..8)",
                opt->cluster_size);
  if (opt->pairs < 0 || opt->pairs > 2)
    return fail(BFP8_ERR_INVALID_ARG, "options.pairs = %d (expected 0, 1 or 2)", opt->pairs);
  return BFP8_OK;
}

// Co-resident clusters of each size on a device with `sms` SMs when the
// device itself cannot be asked (host-only planning): its GPCs are not all
// alike, so a little less than sms / cs, and clearly less for 7 and 8
// (ctas_per_sm CTAs of the instantiation fit on one SM).
void estimate_cluster_caps(int sms, int ctas_per_sm, int* cap) {
  const int slots = sms * ctas_per_sm;
  for (int cs = 0; cs <= kMaxCluster; ++cs)
    cap[cs] = cs < 2 ? slots : static_cast<int>(slots * (cs >= 7 ? 0.75 : 0.94) / cs);
}

// Relative time of the ways of sharing the work among CTAs, in units of one
// (tile, k-block) step of one CTA (a cost model, calibrated on this GB300).
//
// Stream-K: the busiest CTA's whole-tile steps and stream-K steps, plus, for
// each segment end it meets, writing its fp32 partial tile (128 x bn) and,
// for the tile it finishes, reading the c - 1 other contributors' partials
// one after another.  Fitted to measured times on this GPU, per 256 columns
// of partial: writing 12 steps on wide tiles and 4 on swap-AB tiles (whose
// steps are shorter-lived weight streams), reading 3.5 steps on wide tiles
// and 1.5 + bn / 128 per partial on swap-AB tiles.
double stream_k_cost(int64_t tiles, int64_t G, int bn, bool swap, int64_t max_ctas) {
  const int64_t units = tiles * G;
  const int64_t grid = max_ctas < units ? max_ctas : units;
  const int64_t dp_per = (tiles / grid) * G;
  const double sk_per = static_cast<double>((tiles % grid) * G) / static_cast<double>(grid);
  if (sk_per <= 0.0) return static_cast<double>(dp_per);
  const double ctas_per_tile = sk_per >= static_cast<double>(G) ? 1.0 : G / sk_per + 1.0;
  const double segments = 1.0 + sk_per / static_cast<double>(G);
  const double write = (swap ? 4.0 : 12.0) * bn / 256.0;
  const double read = swap ? 1.5 + bn / 128.0 : 3.5 * bn / 256.0;
  return static_cast<double>(dp_per) + std::ceil(sk_per) + segments * write +
         (ctas_per_tile - 1.0) * read;
}
// Whole tiles only: waves of tiles over at most max_ctas CTAs, nothing split.
double whole_tiles_cost(int64_t tiles, int64_t G, int64_t max_ctas) {
  return static_cast<double>((tiles + max_ctas - 1) / max_ctas * G);
}
// Cluster split-K of size cs: ceil(G / cs) steps per wave of co-resident
// clusters, plus the reduction through distributed shared memory.
double cluster_cost(int64_t tiles, int64_t G, int bn, int cs, int cap) {
  const int64_t waves = cap > 0 ? (tiles + cap - 1) / cap : tiles;
  return static_cast<double>(waves) *
         (static_cast<double>((G + cs - 1) / cs) + 0.5 + 0.5 * bn / 128.0);
}

enum class Split { kStreamK, kWholeTiles, kCluster };
struct SplitChoice {
  Split kind = Split::kStreamK;
  uint32_t cs = 0;
  double cost = 0.0;    // the model's relative time of the chosen split
};

// How the tiles and their k-blocks are shared out.  Explicit k_split values
// are honoured (cluster only when the tiles alone would leave SMs idle, with
// tiles * cs <= max_ctas and cs <= G; an explicit cluster_size is taken as
// given, clamped to G); under AUTO the cheapest of the three by the model.
SplitChoice choose_split(int64_t tiles, int64_t G, int bn, bool swap, int64_t max_ctas,
                         const bfp8_gemm_options* opt, const int* cap) {
  const int ks = opt ? opt->k_split : BFP8_KSPLIT_AUTO;
  SplitChoice c;
  const double sk = stream_k_cost(tiles, G, bn, swap, max_ctas);
  const double whole = whole_tiles_cost(tiles, G, max_ctas);
  c.cost = sk;
  if (ks == BFP8_KSPLIT_STREAM_K) return c;
  if (ks == BFP8_KSPLIT_NONE) {
    c.kind = Split::kWholeTiles;
    c.cost = whole;
    return c;
  }
  int best_cs = 0;
  double best_cl = 0.0;
  if (tiles < max_ctas && G >= 2) {
    if (opt && opt->cluster_size > 0) {
      best_cs = static_cast<int>(opt->cluster_size < G ? opt->cluster_size : G);
      best_cl = cluster_cost(tiles, G, bn, best_cs, cap[best_cs]);
    } else {
      for (int cs = 2; cs <= kMaxCluster && cs <= G && tiles * cs <= max_ctas; ++cs) {
        const double v = cluster_cost(tiles, G, bn, cs, cap[cs]);
        if (best_cs == 0 || v < best_cl) {
          best_cs = cs;
          best_cl = v;
        }
      }
    }
  }
  if (ks == BFP8_KSPLIT_CLUSTER) {
    if (best_cs >= 2) {
      c.kind = Split::kCluster;
      c.cs = static_cast<uint32_t>(best_cs);
      c.cost = best_cl;
    }
    return c;
  }
  // AUTO
  if (whole < c.cost) {
    c.cost = whole;
    c.kind = Split::kWholeTiles;
  }
  if (best_cs >= 2 && best_cl < c.cost) {
    c.kind = Split::kCluster;
    c.cs = static_cast<uint32_t>(best_cs);
    c.cost = best_cl;
  }
  return c;
}

// Stream-K tiles of a schedule (they each need a counter in the header).
int64_t stream_k_tiles(const Sched& s) {
  return s.cluster > 1 ? 0 : static_cast<int64_t>(s.tiles) - s.dp_tiles;
}

// Small M: the weights fill the 128-row MMA slot and the activation rows the
// N slot, padded to the next supported width.
int swap_tile_n(int64_t M) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  if (M <= 128) return 128;
  return 256;
}

constexpr int64_t kSwapMaxM = 256;
// AUTO runs the warp-MMA kernel for M <= 24 when its 16-row tiles fit in one
// wave of two CTAs per SM, and for M <= 16 past that when they keep the SMs
// balanced or the weight stream is short: the CTAs take whole tiles
// round-robin (all CTAs streaming the same k offsets together, which the
// DRAM favours: a stream-K split of (tile, stage) ranges measured slower
// everywhere), so an SM carries ceil(tiles / SMs) tiles against tiles / SMs
// on average; below 3/4 of that balance the tcgen05 split-K plan wins on
// long streams, while up to 64 MB of weights the tcgen05 plans pay more for
// their cluster reductions.  Measured on this GPU (µs, against the tcgen05
// plan AUTO would otherwise take): M = 1: N = K = 4096 4.9 against 9.1,
// N = 576, K = 7168 4.7 against 8.5, N = 51200, K = 5120 40.3 against 60.6,
// N = 5120, K = 25600 26.3 against 26.4 (balance 0.70, 131 MB); M = 16:
// N = K = 4096 5.9 against 9.6, N = 4880 7.95 against 10.3 (305 tiles,
// balance 0.67), N = 5120, K = 8192 12.8 against 13.4 (0.70, 42 MB), N =
// 10240, K = 5120 12.8 against 12.8 (0.84), N = 51200 50.9 against 61.3,
// N = 5120, K = 25600 34.2 against 27.6 (0.70, 131 MB).  M = 17 .. 24 (three
// MMA column groups, two CTAs per SM) only in one wave: N = K = 4096 at
// M = 24 6.8 against 8.9, but N = 10240, K = 5120 16.5 against 15.0 and
// N = 51200 65.3 against 61.2; M = 25 .. 32 (one CTA per SM) loses (N = K =
// 4096 at M = 32: 9.4 against 8.9).
bool gemv_preferred(int64_t M, int64_t N, int64_t K, int num_sms) {
  if (M > 24) return false;
  const int64_t tiles = (N + 15) / 16;
  const int64_t sms = num_sms > 0 ? num_sms : 1;
  if (tiles <= 2 * sms) return true;
  if (M > 16) return false;
  const int64_t most = (tiles + sms - 1) / sms;          // tiles on the busiest SM
  const bool balanced = 4 * tiles >= 3 * most * sms;
  return balanced || N * K <= (int64_t{64} << 20);
}

// AUTO never takes the paired tiles: on this GPU they ran slower than 128-row
// tiles at every size measured (N = K = 4096: M = 256 24.3 against 14.0 us,
// M = 2048 47.2 against 37.9, M = 8192 155.2 against 124.1; M = 2048,
// N = 5120, K = 25600 386.7 against 246.7).  Both kernels are bound by the
// promotion warps, and a pair's promotion costs more per unit (its activation
// scales come through a ring the warps wait on, its TMEM releases cross the
// pair); whole-tile schedules on pairs also leave SMs idle at small M.
bool pairs_preferred(int64_t /*M*/) { return false; }

// `dev` = the device's cached properties, whose co-resident cluster counts
// the planner uses (nullptr: host-only planning, counts estimated from
// num_sms).  `experts` > 1: M-grouped mode, B and Bs hold that many experts'
// weights.
bfp8_status make_plan(int64_t M, int64_t N, int64_t K, int num_sms, const bfp8_gemm_options* opt,
                      bool unaligned, const DevInfo* dev, Plan* p, int64_t experts = 1) {
  const int schedule = opt ? opt->schedule : BFP8_SCHEDULE_AUTO;
  p->gemv = experts == 1 && !unaligned && K % 128 == 0 && M <= kGemvMaxM &&
            (schedule == BFP8_SCHEDULE_GEMV ||
             (schedule == BFP8_SCHEDULE_AUTO && gemv_preferred(M, N, K, num_sms)));
  if (schedule == BFP8_SCHEDULE_GEMV && !p->gemv)
    return fail(BFP8_ERR_UNSUPPORTED,
                "options.schedule = GEMV needs M <= %d, K %% 128 == 0 and 16-byte aligned A and B "
                "(got M=%lld K=%lld)", kGemvMaxM, (long long)M, (long long)K);
  const int tn = opt ? opt->tile_n : 0;
  // swap-AB when asked for, and under AUTO only for the tile widths that
  // exist only as swap-AB tiles (16, 32, 64)
  p->swap = schedule == BFP8_SCHEDULE_SWAP_AB || schedule == BFP8_SCHEDULE_GEMV ||
            (schedule == BFP8_SCHEDULE_AUTO && M <= kSwapMaxM && tn != 0 && tn < 128);
  if (!p->swap && tn != 0 && tn != 128 && tn != 256)
    return fail(BFP8_ERR_INVALID_ARG, "options.tile_n = %d: wide tiles are 128 or 256 wide", tn);
  const int64_t G = cdiv(K, 128);
  int max_ctas = num_sms;
  if (opt && opt->max_ctas > 0 && opt->max_ctas < max_ctas) max_ctas = opt->max_ctas;
  // the split of one tile shape, with the cluster capacities of its class
  auto split_for = [&](bool swap, int bn, int64_t tiles) -> SplitChoice {
    const bool two = gemm_two_per_sm(swap, bn);
    int est[kMaxCluster + 1];
    const int* cap = nullptr;
    if (dev) {
      cap = two ? dev->cluster_cap2 : dev->cluster_cap;
    } else {
      estimate_cluster_caps(num_sms, two ? 2 : 1, est);
      cap = est;
    }
    return choose_split(tiles, G, bn, swap, max_ctas, opt, cap);
  };
  if (p->swap) {
    p->bn = tn ? tn : swap_tile_n(M);
  } else if (tn) {
    p->bn = tn;
  } else if (schedule == BFP8_SCHEDULE_AUTO && M <= kSwapMaxM && experts == 1 &&
             !(opt && opt->pairs == BFP8_PAIRS_ALWAYS)) {
    // up to 256 rows: 256- or 128-wide tiles by the split model, a 128-wide
    // step weighted 0.7 of a 256-wide one (fitted to this GPU's times at
    // M = 9 .. 256 on the sweep and Qwen3-32B shapes; swap-AB tiles, the
    // pages' small-M design, were never faster by more than 1 % there and
    // up to 1.6x slower, so AUTO does not take them)
    const int64_t mt = cdiv(M, 128);
    const double c256 = split_for(false, 256, mt * cdiv(N, 256)).cost;
    const double c128 = 0.7 * split_for(false, 128, mt * cdiv(N, 128)).cost;
    p->bn = c128 < c256 ? 128 : 256;
  } else {
    p->bn = 256;
  }
  // plain 256-wide tiles of a decode-sized M load only the rows that exist
  // (M-grouped calls keep whole 128-row tiles: experts start on them)
  p->mr = (!p->swap && p->bn == 256 && experts == 1 && M <= 64) ? (M <= 32 ? 32 : 64) : 128;
  const int64_t p_tiles = p->swap ? cdiv(N, 128) : cdiv(M, 128);
  const int64_t q_tiles = p->swap ? cdiv(M, p->bn) : cdiv(N, p->bn);
  if (p_tiles * q_tiles * G >= (int64_t{1} << 31))
    return fail(BFP8_ERR_UNSUPPORTED, "problem too large: %lld tiles x %lld k-blocks",
                (long long)(p_tiles * q_tiles), (long long)G);
  const SplitChoice sc = split_for(p->swap, p->bn, p_tiles * q_tiles);
  const uint32_t pt = static_cast<uint32_t>(p_tiles), qt = static_cast<uint32_t>(q_tiles);
  const uint32_t g32 = static_cast<uint32_t>(G), mc = static_cast<uint32_t>(max_ctas);
  if (sc.kind == Split::kCluster)
    p->sched = make_sched_cluster(pt, qt, g32, sc.cs);
  else if (sc.kind == Split::kWholeTiles)
    p->sched = make_sched_whole_tiles(pt, qt, g32, mc);
  else
    p->sched = make_sched(pt, qt, g32, mc);
  // 256 x 256 tiles on CTA pairs (bfp8_pairs), whole tiles over the pairs
  const int pairs_opt = opt ? opt->pairs : BFP8_PAIRS_AUTO;
  const int ks = opt ? opt->k_split : BFP8_KSPLIT_AUTO;
  const bool pair_ok = !p->gemv && !p->swap && p->bn == 256 && p->mr == 128 && experts == 1 &&
                       (ks == BFP8_KSPLIT_AUTO || ks == BFP8_KSPLIT_NONE);
  if (pairs_opt == BFP8_PAIRS_ALWAYS && !pair_ok)
    return fail(BFP8_ERR_UNSUPPORTED,
                "options.pairs = ALWAYS needs a plain call on 256-wide tiles with more than 64 rows "
                "and no explicit stream-K or cluster split (M=%lld N=%lld)", (long long)M, (long long)N);
  if (pair_ok && (pairs_opt == BFP8_PAIRS_ALWAYS || (pairs_opt == BFP8_PAIRS_AUTO && pairs_preferred(M)))) {
    int est2[kMaxCluster + 1];
    if (!dev) estimate_cluster_caps(num_sms, 1, est2);
    const int cap_pairs = dev ? dev->cluster_cap[2] : est2[2];
    int64_t max_pairs = max_ctas / 2;
    if (cap_pairs > 0 && cap_pairs < max_pairs) max_pairs = cap_pairs;
    if (max_pairs < 1) max_pairs = 1;
    p->pair = true;
    p->sched = make_sched_whole_tiles(static_cast<uint32_t>(cdiv(M, 256)), static_cast<uint32_t>(cdiv(N, 256)),
                                      g32, static_cast<uint32_t>(max_pairs));
  }
  p->relayout = unaligned || (K % 16) != 0;
  p->kp = p->relayout ? cdiv(K, 16) * 16 : K;
  size_t off = 0;
  // The counters live in a fixed-size header at the start of every workspace,
  // whatever the problem: a later call with a different shape must find zeros
  // there, never an earlier call's partial sums.  Stream-K covers fewer tiles
  // than the grid has CTAs (whole waves are handed out round-robin first).
  // It is always reserved, so that nothing but counters (which every
  // completed call returns to zero) is ever written there.
  p->off_counters = off;
  off += kCounterHeaderBytes;
  p->off_partials = off;
  if (p->sched.sk_units > 0)
    off += align256(static_cast<size_t>(p->sched.grid) * 2 * 128 * p->bn * sizeof(float));
  p->off_a = off;
  if (p->relayout) off += align256(static_cast<size_t>(M) * p->kp);
  p->off_b = off;
  if (p->relayout) off += align256(static_cast<size_t>(experts * N) * p->kp);
  // room for the scales in the kernel's layout (used when the caller's As is
  // row-major or not 16-byte aligned, or Bs does not meet the 16-byte rules)
  p->off_as = off;
  off += align256(static_cast<size_t>(G) * static_cast<size_t>(cdiv(M, 4) * 4) * sizeof(float));
  p->off_bs = off;
  off += align256(static_cast<size_t>(experts * cdiv(N, 128) * G + 4) * sizeof(float));
  p->total = off;
  return BFP8_OK;
}

bfp8_status check_gemm_sizes(int64_t M, int64_t N, int64_t K) {
  const int64_t lim = 0x7FFFFFFF;
  if (M < 1 || N < 1 || K < 1)
    return fail(BFP8_ERR_INVALID_ARG, "M, N, K must be >= 1 (got %lld, %lld, %lld)", (long long)M,
                (long long)N, (long long)K);
  if (M > lim || N > lim || K > lim)
    return fail(BFP8_ERR_INVALID_ARG, "M, N, K must be < 2^31");
  return BFP8_OK;
}

bool misaligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) != 0; }

// One bounded wait on a barrier nothing arrives on.
__global__ void selftest_wait_kernel(unsigned long long limit) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    fence_barrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) {
    const long long t0 = clock64();
    const bool done = mbar_wait_bounded(smem_addr(&bar), 0, limit);
    g_selftest_elapsed = static_cast<unsigned long long>(clock64() - t0);
    g_selftest_ok = done ? 1 : 0;
  }
}

}  // namespace

#if defined(BFP8_TRACE)
__device__ unsigned long long g_bfp8_trace[1024 * kTraceEvents];
#endif

}  // namespace bfp8

using namespace bfp8;

#if defined(BFP8_TRACE)
// Trace builds only: copies the per-CTA milestone timestamps of the last
// traced launch (kTraceEvents per CTA, up to 1024 CTAs) to host memory.
extern "C" int bfp8_trace_events(void) { return kTraceEvents; }
extern "C" int bfp8_trace_read(unsigned long long* host, int max_ctas) {
  if (max_ctas > 1024) max_ctas = 1024;
  if (cudaDeviceSynchronize() != cudaSuccess) return -1;
  return cudaMemcpyFromSymbol(host, g_bfp8_trace, sizeof(unsigned long long) * kTraceEvents * max_ctas) ==
                 cudaSuccess ? 0 : -1;
}
#endif

extern "C" {

int bfp8_version(void) { return BFP8_VERSION; }

const char* bfp8_last_error(void) { return t_last_error.c_str(); }

const char* bfp8_status_string(int status) {
  switch (status) {
    case BFP8_OK: return "BFP8_OK";
    case BFP8_ERR_INVALID_ARG: return "BFP8_ERR_INVALID_ARG";
    case BFP8_ERR_ALIGNMENT: return "BFP8_ERR_ALIGNMENT";
    case BFP8_ERR_UNSUPPORTED: return "BFP8_ERR_UNSUPPORTED";
    case BFP8_ERR_CUDA: return "BFP8_ERR_CUDA";
    case BFP8_ERR_WORKSPACE: return "BFP8_ERR_WORKSPACE";
    case BFP8_ERR_DEVICE_TIMEOUT: return "BFP8_ERR_DEVICE_TIMEOUT";
    default: return "BFP8_ERR_UNKNOWN";
  }
}

int64_t bfp8_scale_ld(int64_t M) { return M <= 0 ? 0 : (M + 3) / 4 * 4; }

bfp8_status bfp8_group_quant_ex(const void* x, int in_dtype, int64_t M, int64_t K, int64_t ld_x,
                                int group, int col_major, int scale_fmt, void* q, int64_t ld_q,
                                float* s, int64_t ld_s, void* stream) {
  if (scale_fmt != BFP8_SCALE_FP32 && scale_fmt != BFP8_SCALE_UE8M0)
    return fail(BFP8_ERR_INVALID_ARG, "scale_fmt = %d (expected BFP8_SCALE_FP32 or BFP8_SCALE_UE8M0)",
                scale_fmt);
  if (in_dtype != BFP8_IN_BF16 && in_dtype != BFP8_IN_F32)
    return fail(BFP8_ERR_INVALID_ARG, "in_dtype = %d (expected BFP8_IN_BF16 or BFP8_IN_F32)", in_dtype);
  if (group != 128) return fail(BFP8_ERR_INVALID_ARG, "group = %d: only 128 is supported", group);
  if (col_major != 0 && col_major != 1)
    return fail(BFP8_ERR_INVALID_ARG, "col_major = %d (expected 0 or 1)", col_major);
  if (M < 0 || K < 0) return fail(BFP8_ERR_INVALID_ARG, "negative size M=%lld K=%lld", (long long)M, (long long)K);
  if (M == 0 || K == 0) return ok();
  const int64_t G = (K + 127) / 128;
  if (!x || !q || !s) return fail(BFP8_ERR_INVALID_ARG, "null pointer (x=%p q=%p s=%p)", x, q, (void*)s);
  if (ld_x < K) return fail(BFP8_ERR_INVALID_ARG, "ld_x = %lld < K = %lld", (long long)ld_x, (long long)K);
  if (ld_q < K) return fail(BFP8_ERR_INVALID_ARG, "ld_q = %lld < K = %lld", (long long)ld_q, (long long)K);
  if (col_major ? ld_s < M : ld_s < G)
    return fail(BFP8_ERR_INVALID_ARG, "ld_s = %lld too small for the %s layout", (long long)ld_s,
                col_major ? "column-major" : "row-major");
  if (misaligned(x, in_dtype == BFP8_IN_F32 ? 4 : 2))
    return fail(BFP8_ERR_ALIGNMENT, "x is not aligned to its element size");
  if (misaligned(s, 4)) return fail(BFP8_ERR_ALIGNMENT, "s is not 4-byte aligned");
  if (M * ((G + 1) / 2) >= (int64_t{1} << 30))
    return fail(BFP8_ERR_UNSUPPORTED, "M x K too large for one quantisation launch");
  DevInfo d;
  bfp8_status st = current_device(&d, nullptr);
  if (st != BFP8_OK) return st;
  cudaError_t e = launch_group_quant(x, in_dtype == BFP8_IN_F32, M, K, ld_x, static_cast<uint8_t*>(q),
                                     ld_q, s, col_major, ld_s, scale_fmt == BFP8_SCALE_UE8M0, d.sms,
                                     static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(BFP8_ERR_CUDA, "quantisation launch: %s", cudaGetErrorString(e));
  return ok();
}

bfp8_status bfp8_group_quant(const void* x, int in_dtype, int64_t M, int64_t K, int64_t ld_x,
                             int group, int col_major, void* q, int64_t ld_q, float* s,
                             int64_t ld_s, void* stream) {
  return bfp8_group_quant_ex(x, in_dtype, M, K, ld_x, group, col_major, BFP8_SCALE_FP32, q, ld_q, s,
                             ld_s, stream);
}

bfp8_status bfp8_scale_ceil_ue8m0(const float* in, float* out, int64_t n, void* stream) {
  if (n < 0) return fail(BFP8_ERR_INVALID_ARG, "n = %lld", (long long)n);
  if (n == 0) return ok();
  if (!in || !out) return fail(BFP8_ERR_INVALID_ARG, "null pointer (in=%p out=%p)", (const void*)in,
                               (void*)out);
  if (misaligned(in, 4) || misaligned(out, 4))
    return fail(BFP8_ERR_ALIGNMENT, "in and out must be 4-byte aligned");
  DevInfo d;
  bfp8_status st = current_device(&d, nullptr);
  if (st != BFP8_OK) return st;
  cudaError_t e = launch_scale_ceil_ue8m0(in, out, n, d.sms, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(BFP8_ERR_CUDA, "scale rounding launch: %s", cudaGetErrorString(e));
  return ok();
}

bfp8_status bfp8_gemm_plan(int64_t M, int64_t N, int64_t K, int num_sms,
                           const bfp8_gemm_options* opt, int operands_unaligned,
                           bfp8_plan_info* info) {
  bfp8_status st = check_gemm_sizes(M, N, K);
  if (st != BFP8_OK) return st;
  if ((st = check_options(opt)) != BFP8_OK) return st;
  if (num_sms < 0) return fail(BFP8_ERR_INVALID_ARG, "num_sms = %d", num_sms);
  if (!info) return fail(BFP8_ERR_INVALID_ARG, "info is null");
  DevInfo d;
  const DevInfo* dp = nullptr;
  if (num_sms == 0) {
    if ((st = current_device_with_caps(&d)) != BFP8_OK) return st;
    num_sms = d.sms;
    dp = &d;
  }
  Plan p;
  if ((st = make_plan(M, N, K, num_sms, opt, operands_unaligned != 0, dp, &p)) != BFP8_OK) return st;
  if (stream_k_tiles(p.sched) > static_cast<int64_t>(kCounterHeaderBytes / sizeof(int)))
    return fail(BFP8_ERR_UNSUPPORTED, "more stream-K tiles than the workspace header holds");
  info->swap_ab = p.swap;
  info->tile_n = p.bn;
  info->stages = p.pair ? gemm_pair_stages() : gemm_stages(p.swap, p.bn, p.mr);
  info->grid = p.pair ? 2 * p.sched.grid : p.sched.grid;
  info->tiles = p.sched.tiles;
  info->k_blocks = p.sched.G;
  info->dp_tiles = p.sched.dp_tiles;
  info->sk_units = p.sched.sk_units;
  info->relayout = p.relayout;
  info->workspace_bytes = p.total;
  info->cluster = p.sched.cluster > 1 ? static_cast<int>(p.sched.cluster) : 1;
  info->gemv = p.gemv ? 1 : 0;
  info->pair = p.pair ? 1 : 0;
  return ok();
}

bfp8_status bfp8_plan_unit(int64_t M, int64_t N, int64_t K, int num_sms,
                           const bfp8_gemm_options* opt, int cta, int64_t j, int64_t* num_units_out,
                           int64_t* tile, int64_t* k_block) {
  bfp8_status st = check_gemm_sizes(M, N, K);
  if (st != BFP8_OK) return st;
  if ((st = check_options(opt)) != BFP8_OK) return st;
  if (num_sms < 0) return fail(BFP8_ERR_INVALID_ARG, "num_sms = %d", num_sms);
  DevInfo d;
  const DevInfo* dp = nullptr;
  if (num_sms == 0) {
    if ((st = current_device_with_caps(&d)) != BFP8_OK) return st;
    num_sms = d.sms;
    dp = &d;
  }
  Plan p;
  if ((st = make_plan(M, N, K, num_sms, opt, false, dp, &p)) != BFP8_OK) return st;
  if (cta < 0 || static_cast<uint32_t>(cta) >= p.sched.grid)
    return fail(BFP8_ERR_INVALID_ARG, "cta %d out of range", cta);
  const int64_t n = num_units(p.sched, static_cast<uint32_t>(cta));
  if (num_units_out) *num_units_out = n;
  if (j >= 0) {
    if (j >= n) return fail(BFP8_ERR_INVALID_ARG, "unit %lld out of range", (long long)j);
    // walk the same cursor the kernel's roles walk
    Cursor c;
    c.init(p.sched, static_cast<uint32_t>(cta));
    for (int64_t i = 0; i < j; ++i) c.next();
    if (tile) *tile = c.tile;
    if (k_block) *k_block = c.kb;
  }
  return ok();
}

bfp8_status bfp8_gemm_workspace_size(int64_t M, int64_t N, int64_t K,
                                     const bfp8_gemm_options* opt, int operands_unaligned,
                                     size_t* bytes) {
  bfp8_status st = check_gemm_sizes(M, N, K);
  if (st != BFP8_OK) return st;
  if ((st = check_options(opt)) != BFP8_OK) return st;
  if (!bytes) return fail(BFP8_ERR_INVALID_ARG, "bytes is null");
  DevInfo d;
  if ((st = current_device_with_caps(&d)) != BFP8_OK) return st;
  Plan p;
  if ((st = make_plan(M, N, K, d.sms, opt, operands_unaligned != 0, &d, &p)) != BFP8_OK)
    return st;
  *bytes = p.total;
  return ok();
}

// What a call adds to the plain GEMM: M-grouped experts and / or the fused
// epilogue (bias, next-layer quantisation, optional bf16 output).
struct GemmExtras {
  const int32_t* psum = nullptr;
  int64_t experts = 1;
  const void* bias = nullptr;
  void* q = nullptr;
  float* s = nullptr;
  int s_col_major = 1;
  int64_t ld_s = 0;
  bool store_out = true;
};

// Options a call actually runs with: grouped and fused calls use the wide
// schedule (128 activation rows per tile, inside one expert; one 128-column
// group per promotion thread), and fused calls the stream-K split (the
// cluster reduction stores outside the fused epilogue).
static bfp8_gemm_options effective_options(const bfp8_gemm_options* opt, bool grouped,
                                           bool fused) {
  bfp8_gemm_options o{};
  if (opt) o = *opt;
  if (grouped || fused) {
    o.schedule = BFP8_SCHEDULE_WIDE;
    o.pairs = BFP8_PAIRS_NEVER;
  }
  if (fused) o.k_split = BFP8_KSPLIT_STREAM_K;
  return o;
}

// Timeline-trace builds: the kernels record into g_bfp8_trace.
static void set_trace(GemmArgs* a) {
  a->trace = nullptr;
#if defined(BFP8_TRACE)
  void* tp = nullptr;
  if (cudaGetSymbolAddress(&tp, g_bfp8_trace) == cudaSuccess) a->trace = static_cast<unsigned long long*>(tp);
  cudaGetLastError();
#endif
}

// The GEMM proper (internal linkage: not part of the exported interface).
static bfp8_status gemm_impl(const void* A, const void* B, const float* As, int as_col_major,
                             int64_t ld_as, const float* Bs, void* out, int64_t M, int64_t N,
                             int64_t K, void* workspace, size_t workspace_bytes,
                             const bfp8_gemm_options* opt_in, void* stream, const GemmExtras& x) {
  bfp8_status st = check_gemm_sizes(M, N, K);
  if (st != BFP8_OK) return st;
  if ((st = check_options(opt_in)) != BFP8_OK) return st;
  const int32_t* psum = x.psum;
  const int64_t experts = x.experts;
  const bool fused = x.bias != nullptr || x.q != nullptr;
  if (fused && psum)
    return fail(BFP8_ERR_UNSUPPORTED, "the fused epilogue is not available for grouped GEMMs");
  const bfp8_gemm_options eff = effective_options(opt_in, psum != nullptr, fused);
  const bfp8_gemm_options* opt = (psum || fused) ? &eff : opt_in;
  if (!A || !B || !As || !Bs || (!out && x.store_out))
    return fail(BFP8_ERR_INVALID_ARG, "null pointer (A=%p B=%p As=%p Bs=%p out=%p)", A, B,
                (const void*)As, (const void*)Bs, out);
  if (as_col_major != 0 && as_col_major != 1)
    return fail(BFP8_ERR_INVALID_ARG, "as_col_major = %d (expected 0 or 1)", as_col_major);
  const int64_t G = cdiv(K, 128);
  if (as_col_major ? ld_as < M : ld_as < G)
    return fail(BFP8_ERR_INVALID_ARG, "ld_as = %lld too small for the %s layout", (long long)ld_as,
                as_col_major ? "column-major" : "row-major");
  if (misaligned(As, 4) || misaligned(Bs, 4))
    return fail(BFP8_ERR_ALIGNMENT, "As and Bs must be 4-byte aligned");
  if (misaligned(out, 2)) return fail(BFP8_ERR_ALIGNMENT, "out must be 2-byte aligned");
  DevInfo d;
  if ((st = current_device_with_caps(&d)) != BFP8_OK) return st;
  const bool unaligned = misaligned(A, 16) || misaligned(B, 16);
  Plan p;
  if ((st = make_plan(M, N, K, d.sms, opt, unaligned, &d, &p, experts)) != BFP8_OK)
    return st;
  if (stream_k_tiles(p.sched) > static_cast<int64_t>(kCounterHeaderBytes / sizeof(int)))
    return fail(BFP8_ERR_UNSUPPORTED, "more stream-K tiles than the workspace header holds");
  if (p.total > 0) {
    if (!workspace)
      return fail(BFP8_ERR_WORKSPACE, "this problem needs %zu workspace bytes; got none", p.total);
    if (workspace_bytes < p.total)
      return fail(BFP8_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu needed",
                  workspace_bytes, p.total);
    if (misaligned(workspace, 256))
      return fail(BFP8_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  }
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (p.gemv) {
    // warp-MMA kernel: A and B streamed by TMA in k-block boxes; As (either
    // layout) and Bs read where they are
    CUtensorMap tmW, tmX;
    if ((st = encode_kblocks(&tmW, B, N, K, 16)) != BFP8_OK) return st;
    if ((st = encode_kblocks(&tmX, A, M, K, static_cast<int>(M))) != BFP8_OK) return st;
    GemvArgs ga{};
    ga.As = As;
    ga.ld_as = ld_as;
    ga.as_col_major = as_col_major;
    ga.Bs = Bs;
    ga.out = static_cast<__nv_bfloat16*>(out);
    ga.M = static_cast<int32_t>(M);
    ga.N = N;
    ga.G = K / 128;
    ga.prefetch_b = (opt && opt->prefetch_weights == 1) ? 1 : 0;
    ga.err = d.err;
    ga.wait_limit = kWaitLimitCycles;
    ga.as_bulk = (as_col_major && ld_as % 4 == 0 && ld_as <= 8 * cdiv(M, 8) && !misaligned(As, 16)) ? 1 : 0;
    const cudaError_t e =
        launch_gemv(tmW, tmX, ga, d.sms, (opt && opt->max_ctas > 0) ? opt->max_ctas : 0, cs);
    if (e != cudaSuccess) return fail(BFP8_ERR_CUDA, "GEMV launch: %s", cudaGetErrorString(e));
    return ok();
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const void* a_op = A;
  const void* b_op = B;
  if (p.relayout) {
    cudaError_t e = launch_relayout(static_cast<const uint8_t*>(A), M, K, ws + p.off_a, p.kp, d.sms, cs);
    if (e == cudaSuccess)
      e = launch_relayout(static_cast<const uint8_t*>(B), experts * N, K, ws + p.off_b, p.kp, d.sms,
                          cs);
    if (e != cudaSuccess) return fail(BFP8_ERR_CUDA, "operand re-layout launch: %s", cudaGetErrorString(e));
    a_op = ws + p.off_a;
    b_op = ws + p.off_b;
  }
  const int64_t NTv = cdiv(N, 128);
  // scales in the layout the kernel bulk-copies
  const bool as_ok = as_col_major && ld_as % 4 == 0 && !misaligned(As, 16);
  const bool bs_ok = !misaligned(Bs, 16) && (experts * NTv * G) % 4 == 0;
  const float* as_k = As;
  int64_t ld_k = ld_as;
  const float* bs_k = Bs;
  if (!as_ok || !bs_ok) {
    float* as_out = as_ok ? nullptr : reinterpret_cast<float*>(ws + p.off_as);
    float* bs_out = bs_ok ? nullptr : reinterpret_cast<float*>(ws + p.off_bs);
    const int64_t ld_out = cdiv(M, 4) * 4;
    cudaError_t e = launch_scale_relayout(As, as_col_major, ld_as, M, G, as_out, ld_out, Bs,
                                          experts * NTv * G, bs_out, d.sms, cs);
    if (e != cudaSuccess) return fail(BFP8_ERR_CUDA, "scale re-layout launch: %s", cudaGetErrorString(e));
    if (as_out) { as_k = as_out; ld_k = ld_out; }
    if (bs_out) bs_k = bs_out;
  }
  CUtensorMap tmP, tmQ;
  const void* p_ptr = p.swap ? b_op : a_op;
  const void* q_ptr = p.swap ? a_op : b_op;
  const int64_t p_rows = p.swap ? N : M;
  const int64_t q_rows = p.swap ? M : experts * N;
  const int mode = psum ? kModeGrouped : (fused ? kModeFused : kModePlain);
  const int mr = mode == kModePlain ? p.mr : 128;
  if ((st = encode_operand(&tmP, p_ptr, p_rows, p.kp, p.swap ? 128 : mr)) != BFP8_OK) return st;
  if ((st = encode_operand(&tmQ, q_ptr, q_rows, p.kp, p.pair ? p.bn / 2 : p.bn)) != BFP8_OK) return st;

  GemmArgs a{};
  a.As = as_k;
  a.ld_as = ld_k;
  a.NT = static_cast<int32_t>(NTv);
  a.Bs = bs_k;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.M = M;
  a.N = N;
  a.sched = p.sched;
  a.counters = reinterpret_cast<int*>(ws ? ws + p.off_counters : nullptr);
  a.partials = reinterpret_cast<float*>(ws ? ws + p.off_partials : nullptr);
  a.vec_store = (!misaligned(out, 16) && (N % 8) == 0) ? 1 : 0;
  // wide plain / fused tiles store through TMA (grouped tiles mask rows)
  a.tma_store = 0;
  if (!p.swap && !psum && a.vec_store) {
    if ((st = encode_output(&a.tmO, out, M, N)) != BFP8_OK) return st;
    a.tma_store = 1;
  }
  // weight prefetch also needs the weight operand untouched by re-layout (and,
  // in grouped mode, the expert of each tile, known only after the wait)
  a.prefetch_b = (opt && opt->prefetch_weights == 1 && !p.relayout && bs_ok && !psum) ? 1 : 0;
  a.psum = psum;
  a.experts = static_cast<int32_t>(experts);
  a.bias = static_cast<const __nv_bfloat16*>(x.bias);
  a.bias_vec = (x.bias && !misaligned(x.bias, 16) && N % 8 == 0) ? 1 : 0;
  a.store_out = x.store_out ? 1 : 0;
  a.q_out = static_cast<uint8_t*>(x.q);
  a.s_out = x.s;
  a.s_col_major = x.s_col_major;
  a.ld_s = x.ld_s;
  a.q_vec = (x.q && !misaligned(x.q, 16) && N % 16 == 0) ? 1 : 0;
  a.err = d.err;
  a.wait_limit = kWaitLimitCycles;
  set_trace(&a);
  cudaError_t e = p.pair ? launch_gemm_pair(tmP, tmQ, a, cs)
                 : p.swap ? launch_gemm_swap(p.bn, tmP, tmQ, a, cs)
                          : launch_gemm_wide(p.bn, mode, mr, tmP, tmQ, a, cs);
  if (e != cudaSuccess) return fail(BFP8_ERR_CUDA, "GEMM launch: %s", cudaGetErrorString(e));
  return ok();
}

bfp8_status bfp8_gemm_ex(const void* A, const void* B, const float* As, int as_col_major,
                         int64_t ld_as, const float* Bs, void* out, int64_t M, int64_t N,
                         int64_t K, void* workspace, size_t workspace_bytes,
                         const bfp8_gemm_options* opt, void* stream) {
  return gemm_impl(A, B, As, as_col_major, ld_as, Bs, out, M, N, K, workspace, workspace_bytes,
                   opt, stream, GemmExtras{});
}

static bfp8_status check_grouped(const int32_t* grouped_layout, int num_experts, int64_t N, int64_t K) {
  if (num_experts < 1 || num_experts > kMaxExperts)
    return fail(BFP8_ERR_INVALID_ARG, "num_experts = %d (expected 1..%d)", num_experts, kMaxExperts);
  if (!grouped_layout) return fail(BFP8_ERR_INVALID_ARG, "grouped_layout is null");
  if (misaligned(grouped_layout, 4))
    return fail(BFP8_ERR_ALIGNMENT, "grouped_layout must be 4-byte aligned");
  const int64_t G = cdiv(K, 128);
  if (static_cast<int64_t>(num_experts) * N >= (int64_t{1} << 31) ||
      static_cast<int64_t>(num_experts) * cdiv(N, 128) * G >= (int64_t{1} << 31))
    return fail(BFP8_ERR_UNSUPPORTED, "num_experts x N too large");
  return BFP8_OK;
}

bfp8_status bfp8_gemm_grouped(const void* A, const void* B, const float* As, int as_col_major,
                              int64_t ld_as, const float* Bs, const int32_t* grouped_layout,
                              int num_experts, void* out, int64_t M, int64_t N, int64_t K,
                              void* workspace, size_t workspace_bytes,
                              const bfp8_gemm_options* opt, void* stream) {
  bfp8_status st = check_gemm_sizes(M, N, K);
  if (st != BFP8_OK) return st;
  if ((st = check_grouped(grouped_layout, num_experts, N, K)) != BFP8_OK) return st;
  GemmExtras x;
  x.psum = grouped_layout;
  x.experts = num_experts;
  return gemm_impl(A, B, As, as_col_major, ld_as, Bs, out, M, N, K, workspace, workspace_bytes,
                   opt, stream, x);
}

bfp8_status bfp8_gemm_grouped_workspace_size(int64_t M, int64_t N, int64_t K, int num_experts,
                                             const bfp8_gemm_options* opt,
                                             int operands_unaligned, size_t* bytes) {
  bfp8_status st = check_gemm_sizes(M, N, K);
  if (st != BFP8_OK) return st;
  if ((st = check_options(opt)) != BFP8_OK) return st;
  if (num_experts < 1 || num_experts > kMaxExperts)
    return fail(BFP8_ERR_INVALID_ARG, "num_experts = %d (expected 1..%d)", num_experts, kMaxExperts);
  if (!bytes) return fail(BFP8_ERR_INVALID_ARG, "bytes is null");
  DevInfo d;
  if ((st = current_device_with_caps(&d)) != BFP8_OK) return st;
  const bfp8_gemm_options g = effective_options(opt, true, false);
  Plan p;
  if ((st = make_plan(M, N, K, d.sms, &g, operands_unaligned != 0, &d, &p,
                      num_experts)) != BFP8_OK)
    return st;
  *bytes = p.total;
  return ok();
}

bfp8_status bfp8_gemm_fused(const void* A, const void* B, const float* As, int as_col_major,
                            int64_t ld_as, const float* Bs, const void* bias, void* out, void* q,
                            float* s, int s_col_major, int64_t ld_s, int64_t M, int64_t N,
                            int64_t K, void* workspace, size_t workspace_bytes,
                            const bfp8_gemm_options* opt, void* stream) {
  bfp8_status st = check_gemm_sizes(M, N, K);
  if (st != BFP8_OK) return st;
  if (!out && !q) return fail(BFP8_ERR_INVALID_ARG, "out and q are both null: nothing to produce");
  if ((q == nullptr) != (s == nullptr))
    return fail(BFP8_ERR_INVALID_ARG, "q and s must be given together");
  if (q) {
    if (s_col_major != 0 && s_col_major != 1)
      return fail(BFP8_ERR_INVALID_ARG, "s_col_major = %d (expected 0 or 1)", s_col_major);
    const int64_t Gn = cdiv(N, 128);
    if (s_col_major ? ld_s < M : ld_s < Gn)
      return fail(BFP8_ERR_INVALID_ARG, "ld_s = %lld too small for the %s layout", (long long)ld_s,
                  s_col_major ? "column-major" : "row-major");
    if (misaligned(s, 4)) return fail(BFP8_ERR_ALIGNMENT, "s must be 4-byte aligned");
  }
  if (bias && misaligned(bias, 2)) return fail(BFP8_ERR_ALIGNMENT, "bias must be 2-byte aligned");
  GemmExtras x;
  x.bias = bias;
  x.q = q;
  x.s = s;
  x.s_col_major = s_col_major;
  x.ld_s = ld_s;
  x.store_out = out != nullptr;
  if (!bias && !q) {
    // nothing to fuse: the plain GEMM
    return gemm_impl(A, B, As, as_col_major, ld_as, Bs, out, M, N, K, workspace, workspace_bytes,
                     opt, stream, GemmExtras{});
  }
  return gemm_impl(A, B, As, as_col_major, ld_as, Bs, out, M, N, K, workspace, workspace_bytes,
                   opt, stream, x);
}

bfp8_status bfp8_gemm_fused_workspace_size(int64_t M, int64_t N, int64_t K,
                                           const bfp8_gemm_options* opt, int operands_unaligned,
                                           size_t* bytes) {
  bfp8_status st = check_gemm_sizes(M, N, K);
  if (st != BFP8_OK) return st;
  if ((st = check_options(opt)) != BFP8_OK) return st;
  if (!bytes) return fail(BFP8_ERR_INVALID_ARG, "bytes is null");
  DevInfo d;
  if ((st = current_device_with_caps(&d)) != BFP8_OK) return st;
  const bfp8_gemm_options g = effective_options(opt, false, true);
  Plan p;
  if ((st = make_plan(M, N, K, d.sms, &g, operands_unaligned != 0, &d, &p)) != BFP8_OK)
    return st;
  *bytes = p.total;
  return ok();
}

bfp8_status bfp8_gemm(const void* A, const void* B, const float* As, int as_col_major,
                      int64_t ld_as, const float* Bs, void* out, int64_t M, int64_t N, int64_t K,
                      void* workspace, size_t workspace_bytes, void* stream) {
  return bfp8_gemm_ex(A, B, As, as_col_major, ld_as, Bs, out, M, N, K, workspace, workspace_bytes,
                      nullptr, stream);
}

bfp8_status bfp8_device_status(int* code, int clear) {
  if (!code) return fail(BFP8_ERR_INVALID_ARG, "code is null");
  DevInfo d;
  bfp8_status st = current_device(&d, nullptr);
  if (st != BFP8_OK) return st;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(code, g_dev_err, sizeof(int));
  if (e == cudaSuccess && clear) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_dev_err, &zero, sizeof(int));
  }
  if (e != cudaSuccess) return fail(BFP8_ERR_CUDA, "reading the failure word: %s", cudaGetErrorString(e));
  return ok();
}

bfp8_status bfp8_selftest_bounded_wait(uint64_t limit_cycles, uint64_t* elapsed, void* stream) {
  DevInfo d;
  bfp8_status st = current_device(&d, nullptr);
  if (st != BFP8_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  selftest_wait_kernel<<<1, 32, 0, cs>>>(limit_cycles);
  cudaError_t e = cudaGetLastError();
  unsigned long long el = 0;
  int done = 0;
  if (e == cudaSuccess) e = cudaMemcpyFromSymbolAsync(&el, g_selftest_elapsed, sizeof(el), 0, cudaMemcpyDeviceToHost, cs);
  if (e == cudaSuccess) e = cudaMemcpyFromSymbolAsync(&done, g_selftest_ok, sizeof(done), 0, cudaMemcpyDeviceToHost, cs);
  if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
  if (e != cudaSuccess) return fail(BFP8_ERR_CUDA, "bounded-wait self-test: %s", cudaGetErrorString(e));
  if (elapsed) *elapsed = el;
  if (!done) return fail(BFP8_ERR_DEVICE_TIMEOUT, "the wait gave up after %llu cycles", el);
  return ok();
}


// bfp8_linear: workspace = [GEMM workspace | q (M x K e4m3) | s (G x ld fp32)].
static bfp8_status linear_plan(int64_t M, int64_t N, int64_t K, const bfp8_gemm_options* opt,
                               bool b_unaligned, const DevInfo& d, Plan* p, size_t* off_q,
                               size_t* off_s, size_t* total) {
  bfp8_status st = check_gemm_sizes(M, N, K);
  if (st != BFP8_OK) return st;
  if ((st = check_options(opt)) != BFP8_OK) return st;
  if ((st = make_plan(M, N, K, d.sms, opt, b_unaligned, &d, p)) != BFP8_OK) return st;
  if (stream_k_tiles(p->sched) > static_cast<int64_t>(kCounterHeaderBytes / sizeof(int)))
    return fail(BFP8_ERR_UNSUPPORTED, "more stream-K tiles than the workspace header holds");
  *off_q = p->total;
  *off_s = *off_q + align256(static_cast<size_t>(M) * static_cast<size_t>(K));
  *total = *off_s + align256(static_cast<size_t>(cdiv(K, 128)) * static_cast<size_t>(bfp8_scale_ld(M)) *
                             sizeof(float));
  return BFP8_OK;
}

bfp8_status bfp8_linear_workspace_size(int64_t M, int64_t N, int64_t K, const bfp8_gemm_options* opt,
                                       int weights_unaligned, size_t* bytes) {
  if (!bytes) return fail(BFP8_ERR_INVALID_ARG, "bytes is null");
  bfp8_status st = check_gemm_sizes(M, N, K);
  if (st != BFP8_OK) return st;
  if ((st = check_options(opt)) != BFP8_OK) return st;
  DevInfo d;
  st = current_device_with_caps(&d);
  if (st != BFP8_OK) return st;
  Plan p;
  size_t oq = 0, os = 0;
  if ((st = linear_plan(M, N, K, opt, weights_unaligned != 0, d, &p, &oq, &os, bytes)) != BFP8_OK)
    return st;
  return ok();
}

bfp8_status bfp8_linear(const void* x, int64_t ld_x, const void* B, const float* Bs, void* out,
                        int64_t M, int64_t N, int64_t K, void* workspace, size_t workspace_bytes,
                        const bfp8_gemm_options* opt, void* stream) {
  bfp8_status st = check_gemm_sizes(M, N, K);
  if (st != BFP8_OK) return st;
  if ((st = check_options(opt)) != BFP8_OK) return st;
  if (!x || !B || !Bs || !out)
    return fail(BFP8_ERR_INVALID_ARG, "null pointer (x=%p B=%p Bs=%p out=%p)", x, B,
                (const void*)Bs, out);
  if (ld_x < K) return fail(BFP8_ERR_INVALID_ARG, "ld_x = %lld < K = %lld", (long long)ld_x, (long long)K);
  if (misaligned(x, 2) || misaligned(out, 2)) return fail(BFP8_ERR_ALIGNMENT, "x and out must be 2-byte aligned");
  if (misaligned(Bs, 4)) return fail(BFP8_ERR_ALIGNMENT, "Bs must be 4-byte aligned");
  DevInfo d;
  st = current_device_with_caps(&d);
  if (st != BFP8_OK) return st;
  Plan p;
  size_t off_q = 0, off_s = 0, total = 0;
  if ((st = linear_plan(M, N, K, opt, misaligned(B, 16), d, &p, &off_q, &off_s, &total)) != BFP8_OK)
    return st;
  if (!workspace) return fail(BFP8_ERR_WORKSPACE, "this layer needs %zu workspace bytes; got none", total);
  if (workspace_bytes < total)
    return fail(BFP8_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu needed",
                workspace_bytes, total);
  if (misaligned(workspace, 256)) return fail(BFP8_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  // quantise into the workspace, then the GEMM (which may stream the weights
  // while the quantisation runs: it writes neither B nor Bs)
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* q = ws + off_q;
  float* s = reinterpret_cast<float*>(ws + off_s);
  const int64_t ld_s = bfp8_scale_ld(M);
  cudaError_t e = launch_group_quant(x, 0, M, K, ld_x, q, K, s, 1, ld_s, 0, d.sms, cs);
  if (e != cudaSuccess) return fail(BFP8_ERR_CUDA, "quantisation launch: %s", cudaGetErrorString(e));
  bfp8_gemm_options o{};
  if (opt) o = *opt;
  o.prefetch_weights = 1;
  return gemm_impl(q, B, s, 1, ld_s, Bs, out, M, N, K, workspace, off_q, &o, stream, GemmExtras{});
}

}  // extern "C"
