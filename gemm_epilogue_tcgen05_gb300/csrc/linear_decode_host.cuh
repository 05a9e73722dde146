// Host side of the decode-shaped Linear kernels (decode_linear_kernel.cuh): launch shapes (cluster
// size, one or two CTAs per SM), the choice between them, and the parameters every kind shares.
// Each entry point lives in its own translation unit (k_linear_decode_*.cu), so the kernel
// variants of the kinds compile in parallel.  kDecodeNotTaken sends a call to the GEMM kernel.
#pragma once
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

template <int C, int KIND, int S>
int ld_launch(const LinearDecodeParams& p, const DeviceInfo& di, cudaStream_t s) {
  const void* kfn = reinterpret_cast<const void*>(&linear_decode_kernel<C, KIND, S>);
  if (!ensure_smem_attr(kfn, di.device, ld_smem_bytes(S))) return kDecodeNotTaken;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  ld_config<C, KIND, S>(cfg, attr, p.num_f * C, s);
  if (cudaLaunchKernelEx(&cfg, linear_decode_kernel<C, KIND, S>, p) != cudaSuccess) {
    cudaGetLastError();  // a refused launch configuration: the GEMM kernel takes the call
    return kDecodeNotTaken;
  }
  return FL_OK;
}

// One launch shape: C CTAs per tile, and one CTA per SM (10 stages) or two (5 stages each).  Of
// the two-per-SM shapes only C = 3 ever wins the choice below outright (77 to 101 tiles on 152
// SMs, e.g. the 96 head tiles of a 32-head QKV); the others tie with a one-per-SM shape.
struct LdShape {
  int C;
  bool pair;
};
constexpr LdShape kLdShapes[] = {{1, false}, {2, false}, {3, false}, {4, false}, {6, false}, {8, false}, {3, true}};

template <int KIND>
int ld_fit_of(const LdShape& c, const DeviceInfo& di) {
  switch (c.C) {  // one CTA per SM
    case 1: return ld_fit<1, KIND, kLdStages>(di);
    case 2: return ld_fit<2, KIND, kLdStages>(di);
    case 3: return ld_fit<3, KIND, kLdStages>(di);
    case 4: return ld_fit<4, KIND, kLdStages>(di);
    case 6: return ld_fit<6, KIND, kLdStages>(di);
    default: return ld_fit<8, KIND, kLdStages>(di);
  }
}

template <int KIND>
int ld_launch_of(const LdShape& c, const LinearDecodeParams& p, const DeviceInfo& di, cudaStream_t s) {
  if (!c.pair) {
    switch (c.C) {
      case 1: return ld_launch<1, KIND, kLdStages>(p, di, s);
      case 2: return ld_launch<2, KIND, kLdStages>(p, di, s);
      case 3: return ld_launch<3, KIND, kLdStages>(p, di, s);
      case 4: return ld_launch<4, KIND, kLdStages>(p, di, s);
      case 6: return ld_launch<6, KIND, kLdStages>(p, di, s);
      default: return ld_launch<8, KIND, kLdStages>(p, di, s);
    }
  }
  return ld_launch<3, KIND, kLdStagesPair>(p, di, s);
}

// Launch shape: every cluster resident at once, each CTA with at least one k block, and the
// fewest W bytes on the busiest SM: ceil(tiles C / SMs) CTAs there, each streaming 1/C of a tile.
// Ties go to one CTA per SM, then to the smaller C.  The resident-cluster count of the one-per-SM
// shapes comes from the occupancy query; for the two-per-SM shape the query reports one block per
// SM although the hardware runs two (measured, 20 back-to-back calls: QKV 32 x 12288 x 4096 on 288
// CTAs 18.2 us against 23.5 us on 96), so that shape relies on its per-SM bound alone; a cluster
// that did not fit would only wait for a later wave, as the tiles are independent.  With more tiles than SMs the stream would run
// in two uneven waves (measured: SwiGLU 32 x 14336 x 4096, 224 tiles, 45.0 us against 42.9 us
// on the GEMM kernel), so the GEMM kernel takes those calls.
template <int KIND>
int ld_run(const LinearDecodeParams& p, const DeviceInfo& di, cudaStream_t s) {
  const int cap = max_ctas_override();
  const int sms = cap > 0 && cap < di.num_sms ? cap : di.num_sms;
  if (p.num_f > sms) return kDecodeNotTaken;
  const LdShape* best = nullptr;
  long long best_per_sm = 0;  // CTAs on the busiest SM
  for (const LdShape& c : kLdShapes) {
    const long long ctas = static_cast<long long>(p.num_f) * c.C;
    const long long per_sm = (ctas + sms - 1) / sms;
    if (c.C > p.num_kb || per_sm > (c.pair ? 2 : 1)) continue;
    // per-SM load per_sm / C: compare per_sm * best.C against best_per_sm * C
    if (best != nullptr && per_sm * best->C >= best_per_sm * c.C) continue;
    if (!c.pair && ld_fit_of<KIND>(c, di) < p.num_f) continue;
    best = &c;
    best_per_sm = per_sm;
  }
  if (best == nullptr) return kDecodeNotTaken;
  return ld_launch_of<KIND>(*best, p, di, s);
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
