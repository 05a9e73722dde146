// fused_linear_gelu_host: Linear + bias + GELU on host buffers, with the copies in, the
// GEMM and the copies out overlapped.
//   The operation is fused_linear_gelu's ("Triton 算子融合: Linear 与 Attention", §Linear算子剖析
//   and §GELU激活融合).  The pipeline is this library's own: X and b go up first, then W in
//   blocks of output columns; the GEMM of a column block starts as soon as its rows of W
//   have landed, and its columns of Y go back on a second copy stream while later blocks
//   are still uploading or computing, so both copy engines and the tensor cores run at
//   once.  A column block of Y is a strided region of the row-major host array and is
//   copied with one 2-D copy.
#include <mutex>

#include "host_common.h"

namespace fl {
namespace {

constexpr int kHostChunks = 8;         // target number of column blocks
constexpr int kHostMaxChunks = 16;
constexpr int kMaxHostDevices = 64;

struct HostPipe {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t w_ready[kHostMaxChunks] = {};
  cudaEvent_t y_ready[kHostMaxChunks] = {};
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
  for (int i = 0; i < kHostMaxChunks; ++i)
    if (cudaEventCreateWithFlags(&hp.w_ready[i], ev) != cudaSuccess ||
        cudaEventCreateWithFlags(&hp.y_ready[i], ev) != cudaSuccess)
      return false;
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
  const int nc = ((cdiv(N, kHostChunks) + 255) / 256) * 256;  // columns per block, whole 256-column tiles
  const int chunks = cdiv(N, nc);
  if (chunks > kHostMaxChunks) return FL_ERR_UNSUPPORTED;

  bool ok = true;
  // uploads wait for earlier work on the caller's stream (which may still read dev_buf)
  ok = ok && cudaEventRecord(hp.start, s) == cudaSuccess && cudaStreamWaitEvent(hp.in, hp.start, 0) == cudaSuccess &&
       cudaStreamWaitEvent(hp.out, hp.start, 0) == cudaSuccess;
  if (K > 0)
    ok = ok && cudaMemcpyAsync(dX, X, static_cast<size_t>(M) * K * 2, cudaMemcpyHostToDevice, hp.in) == cudaSuccess;
  if (b != nullptr)
    ok = ok && cudaMemcpyAsync(db, b, static_cast<size_t>(N) * 2, cudaMemcpyHostToDevice, hp.in) == cudaSuccess;
  for (int j = 0; j < chunks && ok; ++j) {
    const int n0 = j * nc, ncj = N - n0 < nc ? N - n0 : nc;
    if (K > 0)
      ok = cudaMemcpyAsync(dW + static_cast<size_t>(n0) * K, static_cast<const __nv_bfloat16*>(W) +
                                                                 static_cast<size_t>(n0) * K,
                           static_cast<size_t>(ncj) * K * 2, cudaMemcpyHostToDevice, hp.in) == cudaSuccess;
    ok = ok && cudaEventRecord(hp.w_ready[j], hp.in) == cudaSuccess;
  }
  if (!ok) return FL_ERR_CUDA;
  for (int j = 0; j < chunks; ++j) {
    const int n0 = j * nc, ncj = N - n0 < nc ? N - n0 : nc;
    if (cudaStreamWaitEvent(s, hp.w_ready[j], 0) != cudaSuccess) return FL_ERR_CUDA;
    st = fused_linear_gelu(dX, dW + static_cast<size_t>(n0) * K, b != nullptr ? db + n0 : nullptr, dY + n0, M, ncj,
                           K, K, K, N, FL_BF16, mode, s);
    if (st != FL_OK) return st;
    if (cudaEventRecord(hp.y_ready[j], s) != cudaSuccess || cudaStreamWaitEvent(hp.out, hp.y_ready[j], 0) != cudaSuccess ||
        cudaMemcpy2DAsync(static_cast<__nv_bfloat16*>(Y) + n0, static_cast<size_t>(N) * 2, dY + n0,
                          static_cast<size_t>(N) * 2, static_cast<size_t>(ncj) * 2, M, cudaMemcpyDeviceToHost,
                          hp.out) != cudaSuccess)
      return FL_ERR_CUDA;
  }
  // the caller's stream resumes once every column block is back on the host
  if (cudaEventRecord(hp.done, hp.out) != cudaSuccess || cudaStreamWaitEvent(s, hp.done, 0) != cudaSuccess)
    return FL_ERR_CUDA;
  return FL_OK;
}
