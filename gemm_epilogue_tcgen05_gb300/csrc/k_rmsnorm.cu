// fused_linear_residual_rmsnorm_fp8: h = X W^T (+ b) + Z; y = r h (.) gamma with
// r = 1/sqrt(mean h^2 + eps); Yq = e4m3(y / s), s = max|y| / 448 per row.
//   "GEMM Epilogue 完全拆解" (pinghaoyang.com.cn), §模式 A and §仿射量化与尾声的五步.
// M > 32: persistent tcgen05 kernel; the 256-column tiles of one 128-row block
//         exchange per-row partials through the workspace inside the kernel.
// M <= 32: swap-AB decode kernels: one cluster per 128-feature tile with the split-K partials
//          reduced in distributed shared memory (decode_cluster_kernel.cuh) when every tile's
//          cluster fits on the device at once, else split-K over all SMs (decode_kernel.cuh).
#include <mutex>

#include "decode_cluster_kernel.cuh"
#include "decode_kernel.cuh"
#include "host_common.h"

namespace fl {
namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Byte offset, inside the status area at the workspace's start, of the decode epoch word (a fixed
// place whatever the shape, past the status words that fl_check_device_status reads and clears).
constexpr size_t kEpochOffset = 128;

struct WsLayout {
  bool decode;
  size_t counters, recs, partials, hbuf, stats, total;  // byte offsets (total = size); the status record is at 0
  int grid, seg_max;                              // decode only
  bool units_ok;                                  // decode unit indices fit 32-bit arithmetic
};

bool use_decode(int M, int K) { return M <= kDecTokens && K > 0; }

// Cluster decode kernel: launch configuration and the number of its clusters the device
// can hold at once (cached per device and cluster size).
template <int C>
void cluster_cfg(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, int grid, cudaStream_t s) {
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kDcSmemBytes;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // programmatic dependent launch, as for the flat decode kernel
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
}

template <int C>
int max_active_clusters(const DeviceInfo& di) {
  static std::mutex mu;
  static int cache[64];
  static bool known[64];
  if (di.device < 0 || di.device >= 64) return 0;
  std::lock_guard<std::mutex> lk(mu);
  if (!known[di.device]) {
    int n = 0;
    const void* kfn = reinterpret_cast<const void*>(&rmsnorm_fp8_decode_cluster_kernel<C>);
    if (ensure_smem_attr(kfn, di.device, kDcSmemBytes)) {
      cudaLaunchConfig_t cfg;
      cudaLaunchAttribute attr[2];
      cluster_cfg<C>(cfg, attr, C * di.num_sms / C, nullptr);
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

// Cluster size for the cluster decode kernel, or 0 to run the flat split-K kernel: every
// feature tile gets a resident cluster of C CTAs and each CTA streams at least one k block.
// The cluster kernel wins whenever it fits, even on few SMs (measured, 20 back-to-back calls:
// 32 x 14336 x 4096 on 112 SMs 27.1 us against 33.3 us flat; 32 x 1024 x 14336 on 64 SMs 14.6
// against 18.7 us), so the flat kernel serves only more tiles than SMs, or a CTA cap.
int pick_decode_cluster(const DeviceInfo& di, int num_f, int num_kb, int sms) {
  const int cs[4] = {8, 4, 2, 1};
  for (int C : cs) {
    if (C > num_kb || static_cast<long long>(num_f) * C > sms) continue;
    const int fit = C == 8   ? max_active_clusters<8>(di)
                    : C == 4 ? max_active_clusters<4>(di)
                    : C == 2 ? max_active_clusters<2>(di)
                             : max_active_clusters<1>(di);
    if (fit >= num_f) return C;
  }
  return 0;
}

template <int C>
int launch_decode_cluster(const DecodeParams& p, const DeviceInfo& di, cudaStream_t s, PreLaunchClear* clear) {
  const void* kfn = reinterpret_cast<const void*>(&rmsnorm_fp8_decode_cluster_kernel<C>);
  if (!ensure_smem_attr(kfn, di.device, kDcSmemBytes)) return FL_ERR_CUDA;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  cluster_cfg<C>(cfg, attr, p.num_f * C, s);
  if (run_clear(clear, s) != FL_OK) return FL_ERR_CUDA;
  return cudaLaunchKernelEx(&cfg, rmsnorm_fp8_decode_cluster_kernel<C>, p) == cudaSuccess ? FL_OK : FL_ERR_CUDA;
}

// SMs the decode grid may use: all of them, or fewer under fl_set_max_ctas.
int decode_sms(const DeviceInfo& di) {
  const int cap = max_ctas_override();
  return cap > 0 && cap < di.num_sms ? cap : di.num_sms;
}

WsLayout layout(int M, int N, int K, int num_sms) {
  WsLayout w{};
  if (M <= 0 || N <= 0) return w;
  if (use_decode(M, K)) {
    w.decode = true;
    const int num_f = cdiv(N, 128);
    const int num_kb = cdiv(K, kBK);
    const long long units_ll = static_cast<long long>(num_f) * num_kb;
    w.grid = static_cast<int>(units_ll < num_sms ? units_ll : num_sms);
    w.units_ok = units_ll * (w.grid + 1) < (1LL << 31);
    const int units = static_cast<int>(w.units_ok ? units_ll : 0);
    w.seg_max = 1;
    for (int c = 0; c < w.grid && w.units_ok; ++c) {
      const int b = dec_unit_begin(c, units, w.grid), e = dec_unit_begin(c + 1, units, w.grid);
      if (e > b) {
        const int segs = static_cast<int>((e - 1) / num_kb - b / num_kb + 1);
        if (segs > w.seg_max) w.seg_max = segs;
      }
    }
    w.counters = kWsStatusBytes;
    w.recs = w.counters + align_up(static_cast<size_t>(num_f + 2) * sizeof(unsigned));
    w.partials = w.recs + align_up(static_cast<size_t>(num_f) * kDecTokens * 2 * sizeof(unsigned long long));
    w.hbuf = w.partials + align_up(static_cast<size_t>(w.grid) * w.seg_max * 128 * kDecTokens * sizeof(float));
    w.stats = w.hbuf + align_up(static_cast<size_t>(num_f) * kDecTokens * 128 * sizeof(float));
    w.total = w.stats + align_up(static_cast<size_t>(num_f) * kDecTokens * sizeof(float2));
  } else {
    const int num_m = cdiv(M, kBM), num_n = cdiv(N, 256);
    w.counters = kWsStatusBytes;
    w.partials = w.counters + align_up(static_cast<size_t>(2 * num_m) * sizeof(unsigned));
    w.total = w.partials + align_up(static_cast<size_t>(num_m) * num_n * kBM * sizeof(float2));
  }
  return w;
}

// Byte ranges [a, a + na) and [b, b + nb) overlap.
bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

}  // namespace

int rmsnorm_fp8_enqueue(const void* X, const void* W, const void* b, const void* Z, const void* gamma, float eps,
                        void* Yq, float* row_scale, void* h_out, int M, int N, int K, int64_t ldx, int64_t ldw,
                        int64_t ldz, int64_t ldq, void* workspace, size_t workspace_bytes, cudaStream_t s,
                        bool scratch_mode) {
  if (M < 0 || N < 0 || K < 0) return FL_ERR_INVALID_ARG;
  if (!(eps >= 0.f)) return FL_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return FL_OK;
  if (Z == nullptr || gamma == nullptr || Yq == nullptr || row_scale == nullptr ||
      (K > 0 && (X == nullptr || W == nullptr)))
    return FL_ERR_INVALID_ARG;
  if (ldz < N || ldq < N || (K > 0 && (ldx < K || ldw < K))) return FL_ERR_INVALID_ARG;
  // h_out shares the residual's layout (pitch ldz) and must not overlap it: both passes of the
  // prefill epilogue read Z after the first one has started writing h.
  const size_t zbytes = (static_cast<size_t>(M - 1) * static_cast<size_t>(ldz) + static_cast<size_t>(N)) * 2;
  if (h_out != nullptr && overlaps(h_out, zbytes, Z, zbytes)) return FL_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(W) || !aligned16(b) || !aligned16(Z) || !aligned16(gamma) || !aligned16(Yq) ||
      !aligned16(row_scale) || !aligned16(h_out))
    return FL_ERR_ALIGNMENT;
  if (!pitch_ok(ldz, 2) || !pitch_ok(ldq, 1) || (K > 0 && (!pitch_ok(ldx, 2) || !pitch_ok(ldw, 2))))
    return FL_ERR_ALIGNMENT;
  DeviceInfo di;
  int st = current_device(&di);
  if (st != FL_OK) return st;
  const WsLayout wl = layout(M, N, K, decode_sms(di));
  if (workspace == nullptr || workspace_bytes < wl.total) return FL_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return FL_ERR_ALIGNMENT;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  // A caller-owned workspace records failures in its own status record, so concurrent calls
  // on different workspaces never see each other's; the no-allocation entry point's shared
  // scratch uses the device-wide word instead, and clears its counters before the launch.
  int* status = scratch_mode ? device_status_ptr(di.device) : reinterpret_cast<int*>(ws);
  if (status == nullptr) return FL_ERR_CUDA;
  PreLaunchClear clear;
  if (scratch_mode) {
    clear.ptr = ws;
    clear.bytes = wl.partials;  // status area (with the decode epoch word), counters and decode records
  }

  if (wl.decode) {
    if (!wl.units_ok || wl.seg_max > kDecMaxSeg) return FL_ERR_UNSUPPORTED;
    DecodeParams p;
    std::memset(&p, 0, sizeof(p));
    if (!encode_2d(&p.map_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, W, K, N, ldw, kBK, 128,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&p.map_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, X, K, M, ldx, kBK, kDecTokens,
                   CU_TENSOR_MAP_SWIZZLE_128B))
      return FL_ERR_CUDA;
    p.M = M;
    p.N = N;
    p.K = K;
    p.num_f = cdiv(N, 128);
    p.num_kb = cdiv(K, kBK);
    p.units = p.num_f * p.num_kb;
    p.seg_max = wl.seg_max;
    p.bias = static_cast<const __nv_bfloat16*>(b);
    p.resid = static_cast<const __nv_bfloat16*>(Z);
    p.ldz = ldz;
    p.gamma = static_cast<const __nv_bfloat16*>(gamma);
    p.eps = eps;
    p.yq = static_cast<uint8_t*>(Yq);
    p.ldq = ldq;
    p.row_scale = row_scale;
    p.hout = static_cast<__nv_bfloat16*>(h_out);
    p.ldh = ldz;
    p.counters = reinterpret_cast<unsigned*>(ws + wl.counters);
    p.partials = reinterpret_cast<float*>(ws + wl.partials);
    p.hbuf = reinterpret_cast<float*>(ws + wl.hbuf);
    p.stats = reinterpret_cast<float2*>(ws + wl.stats);
    p.recs = reinterpret_cast<unsigned long long*>(ws + wl.recs);
    p.epoch = reinterpret_cast<unsigned*>(ws + kEpochOffset);
    p.status = status;
    p.timeout_ns = wait_timeout_ns();
    switch (pick_decode_cluster(di, p.num_f, p.num_kb, decode_sms(di))) {
      case 8: return launch_decode_cluster<8>(p, di, s, &clear);
      case 4: return launch_decode_cluster<4>(p, di, s, &clear);
      case 2: return launch_decode_cluster<2>(p, di, s, &clear);
      case 1: return launch_decode_cluster<1>(p, di, s, &clear);
      default: break;
    }
    const void* kfn = reinterpret_cast<const void*>(&rmsnorm_fp8_decode_kernel);
    if (!ensure_smem_attr(kfn, di.device, kDecSmemBytes)) return FL_ERR_CUDA;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(wl.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kDecSmemBytes;
    cfg.stream = s;
    // Programmatic dependent launch: the kernel may start on SMs the preceding kernel has left
    // and prefetch weights into L2, then waits for that kernel (griddepcontrol.wait).  The grid
    // never exceeds one CTA per SM, so every CTA is resident once the preceding kernel's CTAs,
    // which never wait on this one, have left.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (run_clear(&clear, s) != FL_OK) return FL_ERR_CUDA;
    return cudaLaunchKernelEx(&cfg, rmsnorm_fp8_decode_kernel, p) == cudaSuccess ? FL_OK : FL_ERR_CUDA;
  }

  const int num_n = cdiv(N, 256);
  if (num_n > di.num_sms) return FL_ERR_UNSUPPORTED;
  auto setup = [&](int cg, GemmParams& p) -> bool {
    init_params(p, M, N, K, 256, cg);
    p.group_m = 1;  // row-major tile order: the tiles of one row block run side by side
    if (K > 0 &&
        (!encode_2d(&p.map_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, X, K, M, ldx, kBK, kBM,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
         !encode_2d(&p.map_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, W, K, N, ldw, kBK, 256 / cg,
                    CU_TENSOR_MAP_SWIZZLE_128B)))
      return false;
    if (!encode_2d(&p.map_out[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Yq, N, M, ldq, 128, 32,
                   CU_TENSOR_MAP_SWIZZLE_128B))
      return false;
    if (h_out != nullptr && !encode_2d(&p.map_out[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, h_out, N, M, ldz, 64, 32,
                                       CU_TENSOR_MAP_SWIZZLE_128B))
      return false;
    p.store_h1 = h_out != nullptr;
    p.status = status;
    p.bias = static_cast<const __nv_bfloat16*>(b);
    p.resid = static_cast<const __nv_bfloat16*>(Z);
    p.ldz = ldz;
    p.gamma = static_cast<const __nv_bfloat16*>(gamma);
    p.eps = eps;
    p.row_scale = row_scale;
    p.counters = reinterpret_cast<unsigned*>(ws + wl.counters);
    p.partials = reinterpret_cast<float2*>(ws + wl.partials);
    return true;
  };
  // Every tile of a row block must be resident together: at least one row block's
  // worth of tiles runs at once and all CTAs are co-scheduled (cooperative launch).
  return run_gemm<EPI_RMSNORM_FP8>(M, setup, di, s, true, num_n, &clear);
}

}  // namespace fl

extern "C" size_t fl_rmsnorm_fp8_workspace_bytes(int M, int N, int K) {
  using namespace fl;
  DeviceInfo di;
  if (current_device(&di) == FL_ERR_CUDA) return 0;
  return layout(M, N, K, decode_sms(di)).total;
}

extern "C" int fused_linear_residual_rmsnorm_fp8(const void* X, const void* W, const void* b, const void* Z,
                                                 const void* gamma, float eps, void* Yq, float* row_scale,
                                                 void* h_out, int M, int N, int K, int64_t ldx, int64_t ldw,
                                                 int64_t ldz, int64_t ldq, void* workspace, size_t workspace_bytes,
                                                 void* stream) {
  return fl::rmsnorm_fp8_enqueue(X, W, b, Z, gamma, eps, Yq, row_scale, h_out, M, N, K, ldx, ldw, ldz, ldq,
                                 workspace, workspace_bytes, static_cast<cudaStream_t>(stream), false);
}
