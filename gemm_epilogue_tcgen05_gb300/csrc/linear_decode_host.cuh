// Host side of the decode-shaped Linear kernels (decode_linear_kernel.cuh): launch shapes (cluster
// size, one or two CTAs per SM), the choice between them, and the parameters every kind shares.
// Each entry point lives in its own translation unit (k_linear_decode_*.cu), so the kernel
// variants of the kinds compile in parallel.  kDecodeNotTaken sends a call to the GEMM kernel.
#pragma once
#include <algorithm>
#include <cmath>
#include <mutex>

#include "decode_linear_kernel.cuh"
#include "host_common.h"

namespace fl {
namespace {


template <int C, int KIND, int S>
void ld_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, int grid, cudaStream_t s) {
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = ld_smem_bytes(S);
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // programmatic dependent launch: the weight prefetch may overlap the preceding kernel's tail
  // (everything the kernel reads or writes besides W waits in griddepcontrol.wait)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
}

// Clusters of C CTAs of this kernel the device holds at once (cached per device).
template <int C, int KIND, int S>
int ld_fit(const DeviceInfo& di) {
  static std::mutex mu;
  static int cache[64];
  static bool known[64];
  if (di.device < 0 || di.device >= 64) return 0;
  std::lock_guard<std::mutex> lk(mu);
  if (!known[di.device]) {
    int n = 0;
    const void* kfn = reinterpret_cast<const void*>(&linear_decode_kernel<C, KIND, S>);
    if (ensure_smem_attr(kfn, di.device, ld_smem_bytes(S))) {
      cudaLaunchConfig_t cfg;
      cudaLaunchAttribute attr[2];
      ld_config<C, KIND, S>(cfg, attr, C * (di.num_sms / C), nullptr);
      cfg.numAttrs = 1;  // the occupancy query takes the cluster shape only
      if (cudaOccupancyMaxActiveClusters(&n, kfn, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
      }
    }
    cache[di.device] = n;
    known[di.device] = true;
  }
  return cache[di.device];
}

// Launches tiles [p.f0, p.f0 + tiles) (the whole call unless it takes several launches).
template <int C, int KIND, int S>
int ld_launch(const LinearDecodeParams& p, const DeviceInfo& di, cudaStream_t s, int tiles) {
  const void* kfn = reinterpret_cast<const void*>(&linear_decode_kernel<C, KIND, S>);
  if (!ensure_smem_attr(kfn, di.device, ld_smem_bytes(S))) return kDecodeNotTaken;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  ld_config<C, KIND, S>(cfg, attr, tiles * C, s);
  if (cudaLaunchKernelEx(&cfg, linear_decode_kernel<C, KIND, S>, p) != cudaSuccess) {
    cudaGetLastError();  // a refused launch configuration: the GEMM kernel takes the call
    return kDecodeNotTaken;
  }
  return FL_OK;
}

// One launch shape: C CTAs per tile, and one CTA per SM (10 stages) or two (5 stages each).  The
// list is in the order of preference between shapes that stream equally many k blocks per CTA.
struct LdShape {
  int C;
  bool pair;
};
constexpr LdShape kLdShapes[] = {{1, false}, {2, false}, {2, true}, {3, true},
                                 {4, false}, {4, true},  {8, false}, {8, true}};

template <int KIND>
int ld_fit_single(int C, const DeviceInfo& di) {
  switch (C) {
    case 1: return ld_fit<1, KIND, kLdStages>(di);
    case 2: return ld_fit<2, KIND, kLdStages>(di);
    case 4: return ld_fit<4, KIND, kLdStages>(di);
    default: return ld_fit<8, KIND, kLdStages>(di);
  }
}

// Stand-in with the block size and shared memory of the two-per-SM decode kernel; never launched.
__global__ void __launch_bounds__(kThreads, 2) ld_pair_stand_in_kernel() {}

// Clusters of C CTAs at two per SM the device holds at once (cached per device).  The occupancy
// query reports one block per SM for the two-per-SM decode kernel itself, although the hardware runs
// two (measured: the 288 CTAs of QKV 32 x 12288 x 4096 in one wave; Nsight's occupancy analysis
// gives two), so it is asked about the stand-in.  Its counts match what ran on 152 SMs: 97 clusters
// of 3 (96 ran in one wave, 100 in two) and 46 of 6 (48 ran in two waves).
int ld_fit_pair(int C, const DeviceInfo& di) {
  static std::mutex mu;
  static int cache[64][9];
  static bool known[64][9];
  if (di.device < 0 || di.device >= 64 || C < 1 || C > 8) return 0;
  std::lock_guard<std::mutex> lk(mu);
  if (!known[di.device][C]) {
    int n = 0;
    const void* kfn = reinterpret_cast<const void*>(&ld_pair_stand_in_kernel);
    if (ensure_smem_attr(kfn, di.device, ld_smem_bytes(kLdStagesPair))) {
      cudaLaunchConfig_t cfg;
      std::memset(&cfg, 0, sizeof(cfg));
      cudaLaunchAttribute attr[1];
      cfg.gridDim = dim3(C * (2 * di.num_sms / C));
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = ld_smem_bytes(kLdStagesPair);
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = C;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, kfn, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
      }
    }
    cache[di.device][C] = n;
    known[di.device][C] = true;
  }
  return cache[di.device][C];
}

template <int KIND>
int ld_fit_of(const LdShape& c, const DeviceInfo& di) {
  return c.pair ? ld_fit_pair(c.C, di) : ld_fit_single<KIND>(c.C, di);
}

template <int KIND>
int ld_launch_of(const LdShape& c, const LinearDecodeParams& p, const DeviceInfo& di, cudaStream_t s,
                 int tiles) {
  if (!c.pair) {
    switch (c.C) {
      case 1: return ld_launch<1, KIND, kLdStages>(p, di, s, tiles);
      case 2: return ld_launch<2, KIND, kLdStages>(p, di, s, tiles);
      case 4: return ld_launch<4, KIND, kLdStages>(p, di, s, tiles);
      default: return ld_launch<8, KIND, kLdStages>(p, di, s, tiles);
    }
  }
  switch (c.C) {
    case 1: return ld_launch<1, KIND, kLdStagesPair>(p, di, s, tiles);
    case 2: return ld_launch<2, KIND, kLdStagesPair>(p, di, s, tiles);
    case 3: return ld_launch<3, KIND, kLdStagesPair>(p, di, s, tiles);
    case 4: return ld_launch<4, KIND, kLdStagesPair>(p, di, s, tiles);
    default: return ld_launch<8, KIND, kLdStagesPair>(p, di, s, tiles);
  }
}

// k blocks a CTA streams below which a further split of the tile no longer pays: 16 blocks are
// 256 KB of W (measured on 32 tiles of K = 4096, 20 back-to-back calls: clusters of 4 9.3-9.4 us,
// of 8 9.6 us, of 6 9.7 us).
constexpr int kLdMinKbPerCta = 16;

// The launches of one call: shape, and the tiles of each launch (launches = 0: the call goes to the
// GEMM kernel).
struct LdPlan {
  LdShape shape;
  int launches;
  int share;  // tiles per launch (the last takes the rest)
};

// Launch shape.  Every cluster must be resident at once (a cluster that did not fit would run in a
// later wave), with at most one (10 stages) or two (5 stages) CTAs per SM and at least one k block
// per CTA.  Measured per point: 20 back-to-back calls, K = 4096.
// - More tiles than SMs: one CTA per tile at two per SM keeps every tile resident at once (SwiGLU
//   32 x 14336 x 4096, 224 tiles, 37.8 us against 45.3 in two waves of one per SM and 45.9 on the
//   GEMM kernel; GELU 32 x 20480 x 4096, 160 tiles, 28.3 us against 42.8 and 37.2).  More tiles
//   than that holds run as several such launches of equal shares, back to back on the stream.
// - One CTA per tile already engaging 3/4 of the SMs: W streams close to the HBM rate and a split
//   would add only its reduction (128 tiles: 21.9 us on one CTA per tile and SM, 24.6 at two per SM,
//   22.4-22.9 on clusters of 2 at two per SM).
// - Otherwise the per-CTA stream is the limit (each CTA keeps at most its ring of stages in flight):
//   the shape with the fewest k blocks per CTA wins, counting no fewer than kLdMinKbPerCta; ties go
//   to the smaller C, then to one CTA per SM (the order of kLdShapes).  48 tiles: 12.6 us on clusters
//   of 4 at two per SM against 13.4 on clusters of 3 and 14.9 on clusters of 2; 64 tiles: 13.2
//   against 14.1 on clusters of 2; 80 and 96 tiles on clusters of 3 at two per SM (15.6 and 18.7 us)
//   against 17.0 and 20.2 on clusters of 2.
template <int KIND>
LdPlan ld_plan(int num_f, int num_kb, const DeviceInfo& di) {
  const int cap = max_ctas_override();
  const int sms = cap > 0 && cap < di.num_sms ? cap : di.num_sms;
  LdPlan none{{1, false}, 0, 0};
  if (num_f < 1 || num_kb < 1) return none;
  if (num_f > sms) {
    const int per_launch = std::min(2 * sms, ld_fit_pair(1, di));  // tiles resident at once
    if (per_launch < 1) return none;
    const int launches = cdiv(num_f, per_launch);
    return LdPlan{{1, true}, launches, cdiv(num_f, launches)};
  }
  if (4 * num_f >= 3 * sms) return LdPlan{{1, false}, 1, num_f};
  const LdShape* best = nullptr;
  int best_kb = 0;
  for (const LdShape& c : kLdShapes) {
    const long long ctas = static_cast<long long>(num_f) * c.C;
    if (c.C > num_kb || ctas > static_cast<long long>(c.pair ? 2 : 1) * sms) continue;
    const int kb = std::max(cdiv(num_kb, c.C), kLdMinKbPerCta);
    if (best != nullptr && kb >= best_kb) continue;
    if (ld_fit_of<KIND>(c, di) < num_f) continue;
    best = &c;
    best_kb = kb;
  }
  if (best == nullptr) return none;
  return LdPlan{*best, 1, num_f};
}

template <int KIND>
int ld_run(const LinearDecodeParams& p, const DeviceInfo& di, cudaStream_t s) {
  const LdPlan pl = ld_plan<KIND>(p.num_f, p.num_kb, di);
  if (pl.launches == 0) return kDecodeNotTaken;
  LinearDecodeParams q = p;
  for (q.f0 = 0; q.f0 < p.num_f; q.f0 += pl.share) {
    const int st = ld_launch_of<KIND>(pl.shape, q, di, s, std::min(pl.share, p.num_f - q.f0));
    // a refused first launch leaves the call to the GEMM kernel; a later one cannot
    if (st != FL_OK) return q.f0 == 0 ? st : FL_ERR_CUDA;
  }
  return FL_OK;
}

// The plan as the query entry point reports it.
template <int KIND>
void ld_plan_out(int num_f, int num_kb, const DeviceInfo& di, int* cluster, int* ctas_per_sm, int* launches) {
  const LdPlan pl = ld_plan<KIND>(num_f, num_kb, di);
  *cluster = pl.launches > 0 ? pl.shape.C : 0;
  *ctas_per_sm = pl.launches > 0 ? (pl.shape.pair ? 2 : 1) : 0;
  *launches = pl.launches;
}

inline bool ld_common(LinearDecodeParams& p, const void* X, int M, int K, int64_t ldx, const DeviceInfo& di) {
  std::memset(&p, 0, sizeof(p));
  if (!encode_2d(&p.map_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, X, K, M, ldx, kBK, kLdTokens,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return false;
  p.M = M;
  p.K = K;
  p.num_kb = cdiv(K, kBK);
  p.status = device_status_ptr(di.device);
  p.timeout_ns = wait_timeout_ns();
  return p.status != nullptr;
}

inline bool ld_taken(int M, int K) { return linear_decode_mode() != 0 && M > 0 && M <= kLdTokens && K > 0; }

}  // namespace
}  // namespace fl
