// fused_linear_cross_entropy: LM-head logits h = X W^T (+ b) and per-row cross-entropy
// loss = logsumexp(h) - h[label] without materialising the logits (optional copy).
//   "GEMM Epilogue 完全拆解" (pinghaoyang.com.cn), §模式 C: per-tile (max, sum-exp) state,
//   merged per row with m = max(m1, m2), s = s1 e^{m1-m} + s2 e^{m2-m}, in a fixed order
//   (deterministic, no atomics on the values).
#include "host_common.h"

namespace fl {
namespace {
constexpr size_t kCeAlign = 256;
inline size_t ce_align(size_t x) { return (x + kCeAlign - 1) / kCeAlign * kCeAlign; }
struct CeLayout {
  size_t counters, partials, label_logit, total;  // byte offsets; the status record is at 0
};
CeLayout ce_layout(int M, int V) {
  CeLayout l{};
  if (M <= 0 || V <= 0) return l;
  const size_t num_m = cdiv(M, kBM), num_n = cdiv(V, 256);
  l.counters = kWsStatusBytes;
  l.partials = l.counters + ce_align(num_m * sizeof(unsigned));
  l.label_logit = l.partials + ce_align(num_n * static_cast<size_t>(M) * sizeof(float2));
  l.total = l.label_logit + ce_align(static_cast<size_t>(M) * sizeof(float));
  return l;
}
}  // namespace
}  // namespace fl

extern "C" size_t fl_cross_entropy_workspace_bytes(int M, int V) { return fl::ce_layout(M, V).total; }

extern "C" int fused_linear_cross_entropy(const void* X, const void* W, const void* b, const int32_t* labels,
                                          float* loss, void* logits, int M, int V, int K, int64_t ldx, int64_t ldw,
                                          int64_t ldl, void* workspace, size_t workspace_bytes, void* stream) {
  using namespace fl;
  if (M < 0 || V < 0 || K < 0) return FL_ERR_INVALID_ARG;
  if (M == 0) return FL_OK;
  if (V == 0 || labels == nullptr || loss == nullptr || (K > 0 && (X == nullptr || W == nullptr)))
    return FL_ERR_INVALID_ARG;
  if ((logits != nullptr && ldl < V) || (K > 0 && (ldx < K || ldw < K))) return FL_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(W) || !aligned16(b) || !aligned16(logits)) return FL_ERR_ALIGNMENT;
  if ((logits != nullptr && !pitch_ok(ldl, 2)) || (K > 0 && (!pitch_ok(ldx, 2) || !pitch_ok(ldw, 2))))
    return FL_ERR_ALIGNMENT;
  DeviceInfo di;
  int st = current_device(&di);
  if (st != FL_OK) return st;
  const CeLayout wl = ce_layout(M, V);
  if (workspace == nullptr || workspace_bytes < wl.total) return FL_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & (kCeAlign - 1)) != 0) return FL_ERR_ALIGNMENT;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto setup = [&](int cg, GemmParams& p) -> bool {
    init_params(p, M, V, K, 256, cg);
    if (K > 0 &&
        (!encode_2d(&p.map_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, X, K, M, ldx, kBK, kBM,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
         !encode_2d(&p.map_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, W, K, V, ldw, kBK, 256 / cg,
                    CU_TENSOR_MAP_SWIZZLE_128B)))
      return false;
    if (logits != nullptr && !encode_2d(&p.map_out[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, logits, V, M, ldl, 64,
                                        32, CU_TENSOR_MAP_SWIZZLE_128B))
      return false;
    p.store_logits = logits != nullptr;
    p.bias = static_cast<const __nv_bfloat16*>(b);
    p.labels = labels;
    p.loss = loss;
    p.status = reinterpret_cast<int*>(ws);  // this workspace's status record
    p.counters = reinterpret_cast<unsigned*>(ws + wl.counters);
    p.ce_partials = reinterpret_cast<float2*>(ws + wl.partials);
    p.label_logit = reinterpret_cast<float*>(ws + wl.label_logit);
    return true;
  };
  return run_gemm<EPI_CE>(M, setup, di, static_cast<cudaStream_t>(stream), false, 1);
}
