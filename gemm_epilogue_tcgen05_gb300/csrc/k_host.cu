// fused_linear_gelu_host: Linear + bias + GELU on host buffers, with the copies in, the
// GEMM and the copies out overlapped.
//   The operation is fused_linear_gelu's ("Triton 算子融合: Linear 与 Attention", §Linear算子剖析
//   and §GELU激活融合).  The pipeline is this library's own: X is cut into row blocks and W into
//   blocks of output columns, uploaded alternately (X0, W0, X1, W1, ..., then the rest of the
//   longer list); the GEMM of output block (r, c) starts as soon as X_r and W_c have landed, and
//   the block goes back to the host (one 2-D copy of a strided region of the row-major array) on
//   a second copy stream while later blocks are still uploading or computing.  The first output
//   leaves after one row block of X and one column block of W; alternating keeps the landed row
//   and column blocks balanced, so each upload completes as many output blocks as it can and the
//   copies back (more bytes than the copies in, over a link each direction of which is slower
//   than the GEMMs) start early and do not run dry.
#include <mutex>

#include "host_common.h"

namespace fl {
namespace {

constexpr int kHostColBlocks = 8;      // target number of column blocks (of whole 256-column tiles)
constexpr int kHostRowBlocks = 4;      // target number of row blocks (of whole 128-row tiles)
constexpr int kHostMaxCol = 16;
constexpr int kHostMaxRow = 8;
constexpr int kMaxHostDevices = 64;

struct HostPipe {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t x_ready[kHostMaxRow] = {};
  cudaEvent_t w_ready[kHostMaxCol] = {};
  cudaEvent_t y_ready[kHostMaxRow * kHostMaxCol] = {};
};
std::mutex g_host_mu;
HostPipe g_pipe[kMaxHostDevices];

bool init_pipe(HostPipe& hp) {
  if (hp.ready) return true;
  const unsigned ev = cudaEventDisableTiming;
  if (cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&hp.start, ev) != cudaSuccess || cudaEventCreateWithFlags(&hp.done, ev) != cudaSuccess)
    return false;
  for (int i = 0; i < kHostMaxRow; ++i)
    if (cudaEventCreateWithFlags(&hp.x_ready[i], ev) != cudaSuccess) return false;
  for (int i = 0; i < kHostMaxCol; ++i)
    if (cudaEventCreateWithFlags(&hp.w_ready[i], ev) != cudaSuccess) return false;
  for (int i = 0; i < kHostMaxRow * kHostMaxCol; ++i)
    if (cudaEventCreateWithFlags(&hp.y_ready[i], ev) != cudaSuccess) return false;
  hp.ready = true;
  return true;
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Device buffer layout: X [M][K] | W [N][K] | b [N] | Y [M][N], each 256-byte aligned.
struct HostLayout {
  size_t x, w, b, y, total;
  HostLayout(int M, int N, int K) {
    x = 0;
    w = x + align256(static_cast<size_t>(M) * K * 2);
    b = w + align256(static_cast<size_t>(N) * K * 2);
    y = b + align256(static_cast<size_t>(N) * 2);
    total = y + align256(static_cast<size_t>(M) * N * 2);
  }
};

}  // namespace
}  // namespace fl

extern "C" size_t fl_linear_gelu_host_buffer_bytes(int M, int N, int K) {
  if (M < 0 || N < 0 || K < 0) return 0;
  return fl::HostLayout(M, N, K).total;
}

extern "C" int fused_linear_gelu_host(const void* X, const void* W, const void* b, void* Y, int M, int N, int K,
                                      int mode, void* dev_buf, size_t dev_buf_bytes, void* stream) {
  using namespace fl;
  if (M < 0 || N < 0 || K < 0) return FL_ERR_INVALID_ARG;
  if (mode != FL_GELU_ERF && mode != FL_GELU_TANH) return FL_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return FL_OK;
  if (Y == nullptr || dev_buf == nullptr || (K > 0 && (X == nullptr || W == nullptr))) return FL_ERR_INVALID_ARG;
  if ((N % 8) != 0 || (K % 8) != 0) return FL_ERR_ALIGNMENT;  // 16-byte row pitches for TMA
  if ((reinterpret_cast<uintptr_t>(dev_buf) & 255u) != 0) return FL_ERR_ALIGNMENT;
  const HostLayout L(M, N, K);
  if (dev_buf_bytes < L.total) return FL_ERR_WORKSPACE;
  DeviceInfo di;
  int st = current_device(&di);
  if (st != FL_OK) return st;
  if (di.device >= kMaxHostDevices) return FL_ERR_UNSUPPORTED;

  std::lock_guard<std::mutex> lk(g_host_mu);
  HostPipe& hp = g_pipe[di.device];
  if (!init_pipe(hp)) return FL_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(dev_buf);
  auto* dX = reinterpret_cast<__nv_bfloat16*>(base + L.x);
  auto* dW = reinterpret_cast<__nv_bfloat16*>(base + L.w);
  auto* db = reinterpret_cast<__nv_bfloat16*>(base + L.b);
  auto* dY = reinterpret_cast<__nv_bfloat16*>(base + L.y);
  const int nc = ((cdiv(N, kHostColBlocks) + 255) / 256) * 256;  // columns per block
  const int mr = ((cdiv(M, kHostRowBlocks) + 127) / 128) * 128;    // rows per block
  const int cols = cdiv(N, nc), rows = cdiv(M, mr);
  if (cols > kHostMaxCol || rows > kHostMaxRow) return FL_ERR_UNSUPPORTED;

  // uploads wait for earlier work on the caller's stream (which may still read dev_buf)
  if (cudaEventRecord(hp.start, s) != cudaSuccess || cudaStreamWaitEvent(hp.in, hp.start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(hp.out, hp.start, 0) != cudaSuccess)
    return FL_ERR_CUDA;
  auto up_x = [&](int r) -> bool {
    const int m0 = r * mr, mrr = M - m0 < mr ? M - m0 : mr;
    if (K > 0 && cudaMemcpyAsync(dX + static_cast<size_t>(m0) * K,
                                 static_cast<const __nv_bfloat16*>(X) + static_cast<size_t>(m0) * K,
                                 static_cast<size_t>(mrr) * K * 2, cudaMemcpyHostToDevice, hp.in) != cudaSuccess)
      return false;
    return cudaEventRecord(hp.x_ready[r], hp.in) == cudaSuccess;
  };
  auto up_w = [&](int c) -> bool {
    const int n0 = c * nc, ncc = N - n0 < nc ? N - n0 : nc;
    if (K > 0 && cudaMemcpyAsync(dW + static_cast<size_t>(n0) * K,
                                 static_cast<const __nv_bfloat16*>(W) + static_cast<size_t>(n0) * K,
                                 static_cast<size_t>(ncc) * K * 2, cudaMemcpyHostToDevice, hp.in) != cudaSuccess)
      return false;
    return cudaEventRecord(hp.w_ready[c], hp.in) == cudaSuccess;
  };
  // output block (r, c) on the caller's stream once X_r and W_c have landed, then back to the host
  bool x_waited[kHostMaxRow] = {}, w_waited[kHostMaxCol] = {};
  auto emit = [&](int r, int c) -> int {
    if (!x_waited[r] && cudaStreamWaitEvent(s, hp.x_ready[r], 0) != cudaSuccess) return FL_ERR_CUDA;
    if (!w_waited[c] && cudaStreamWaitEvent(s, hp.w_ready[c], 0) != cudaSuccess) return FL_ERR_CUDA;
    x_waited[r] = w_waited[c] = true;
    const int m0 = r * mr, mrr = M - m0 < mr ? M - m0 : mr;
    const int n0 = c * nc, ncc = N - n0 < nc ? N - n0 : nc;
    const int rc = fused_linear_gelu(dX + static_cast<size_t>(m0) * K, dW + static_cast<size_t>(n0) * K,
                                     b != nullptr ? db + n0 : nullptr, dY + static_cast<size_t>(m0) * N + n0, mrr, ncc,
                                     K, K, K, N, FL_BF16, mode, s);
    if (rc != FL_OK) return rc;
    cudaEvent_t e = hp.y_ready[r * kHostMaxCol + c];
    if (cudaEventRecord(e, s) != cudaSuccess || cudaStreamWaitEvent(hp.out, e, 0) != cudaSuccess ||
        cudaMemcpy2DAsync(static_cast<__nv_bfloat16*>(Y) + static_cast<size_t>(m0) * N + n0,
                          static_cast<size_t>(N) * 2, dY + static_cast<size_t>(m0) * N + n0,
                          static_cast<size_t>(N) * 2, static_cast<size_t>(ncc) * 2, mrr, cudaMemcpyDeviceToHost,
                          hp.out) != cudaSuccess)
      return FL_ERR_CUDA;
    return FL_OK;
  };
  // upload order: b, then X0, W0, X1, W1, ... and the rest of the longer list; after each upload,
  // the output blocks it completes (every landed column block for a row block, and vice versa)
  if (b != nullptr && cudaMemcpyAsync(db, b, static_cast<size_t>(N) * 2, cudaMemcpyHostToDevice, hp.in) != cudaSuccess)
    return FL_ERR_CUDA;
  int xr = 0, wc = 0;  // row and column blocks uploaded so far
  while (xr < rows || wc < cols) {
    if (xr < rows && (wc == cols || xr <= wc)) {
      if (!up_x(xr)) return FL_ERR_CUDA;
      for (int c = 0; c < wc; ++c)
        if ((st = emit(xr, c)) != FL_OK) return st;
      ++xr;
    } else {
      if (!up_w(wc)) return FL_ERR_CUDA;
      for (int r = 0; r < xr; ++r)
        if ((st = emit(r, wc)) != FL_OK) return st;
      ++wc;
    }
  }
  // the caller's stream resumes once every column block is back on the host
  if (cudaEventRecord(hp.done, hp.out) != cudaSuccess || cudaStreamWaitEvent(s, hp.done, 0) != cudaSuccess)
    return FL_ERR_CUDA;
  return FL_OK;
}
