// Library-wide host state: device query cache, the per-device status word,
// wait limits, tensor-map encoding (with its descriptor cache) and the small
// exported utility calls.
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "host_common.h"

namespace fl {

// Status word written by kernels that give up a bounded wait (see ptx.cuh).
__device__ int g_fl_status[ST_WORDS];

namespace {
constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
bool g_dev_known[kMaxDevices];
int* g_status_ptr[kMaxDevices];
std::atomic<uint64_t> g_timeout_ns{kDefaultTimeoutNs};
std::atomic<int> g_max_ctas{0};
std::atomic<int> g_pairing{1};
std::atomic<int> g_linear_decode{1};
std::atomic<int> g_cooperative{1};

struct SmemAttr {
  const void* fn;
  int device;
  int bytes;
};
SmemAttr g_smem_attr[256];
int g_smem_attr_n = 0;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}
}  // namespace

int current_device(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FL_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_dev_known[dev]) {
      *out = g_dev[dev];
      return out->cc == 103 ? FL_OK : FL_ERR_ARCH;
    }
  }
  DeviceInfo d{dev, 0, 0};
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FL_ERR_CUDA;
  d.cc = major * 10 + minor;
  std::lock_guard<std::mutex> lk(g_mu);
  g_dev[dev] = d;
  g_dev_known[dev] = true;
  *out = d;
  return d.cc == 103 ? FL_OK : FL_ERR_ARCH;
}

int* device_status_ptr(int device) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (device < 0 || device >= kMaxDevices) return nullptr;
  if (g_status_ptr[device] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fl_status) != cudaSuccess) return nullptr;
    g_status_ptr[device] = static_cast<int*>(p);
  }
  return g_status_ptr[device];
}

uint64_t wait_timeout_ns() { return g_timeout_ns.load(); }
int max_ctas_override() { return g_max_ctas.load(); }
int cta_pairing_mode() { return g_pairing.load(); }
int linear_decode_mode() { return g_linear_decode.load(); }

int cooperative_launch_mode() { return g_cooperative.load(); }

bool ensure_smem_attr(const void* kernel, int device, int smem_bytes) {
  std::lock_guard<std::mutex> lk(g_mu);
  for (int i = 0; i < g_smem_attr_n; ++i)
    if (g_smem_attr[i].fn == kernel && g_smem_attr[i].device == device && g_smem_attr[i].bytes >= smem_bytes)
      return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) != cudaSuccess)
    return false;
  // All of the unified L1/shared storage as shared memory, so that the carveout leaves room for a
  // second CTA of the decode variant that runs two per SM (103 KB each).
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared) !=
      cudaSuccess)
    return false;
  if (g_smem_attr_n < 256) g_smem_attr[g_smem_attr_n++] = SmemAttr{kernel, device, smem_bytes};
  return true;
}

namespace {
// Descriptor cache.  A tensor map is a pure function of its arguments (address, extents, pitch,
// box, element type, swizzle): it holds no device state, so an entry stays valid for as long as
// its key is unchanged, even across frees and reallocations, and any change of pointer or shape
// is a different key.  Decode-shaped calls re-encode the same few maps on every call; the cache
// takes that work off the enqueue path.  Fixed size, round-robin replacement, one mutex.
struct MapKey {
  const void* base;
  uint64_t inner, outer, ld_elems;
  uint32_t box_inner, box_outer;
  int dt, elem_bytes, sw;
  bool operator==(const MapKey& o) const {
    return base == o.base && inner == o.inner && outer == o.outer && ld_elems == o.ld_elems &&
           box_inner == o.box_inner && box_outer == o.box_outer && dt == o.dt && elem_bytes == o.elem_bytes &&
           sw == o.sw;
  }
};
constexpr int kMapCacheSize = 128;
std::mutex g_map_mu;
MapKey g_map_key[kMapCacheSize];
CUtensorMap g_map_val[kMapCacheSize];
int g_map_n = 0, g_map_next = 0;
std::atomic<int> g_map_cache_on{1};
std::atomic<unsigned long long> g_map_hits{0}, g_map_misses{0};

bool encode_uncached(CUtensorMap* map, const MapKey& k) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {k.inner, k.outer};
  cuuint64_t strides[1] = {k.ld_elems * static_cast<uint64_t>(k.elem_bytes)};
  cuuint32_t box[2] = {k.box_inner, k.box_outer};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, static_cast<CUtensorMapDataType>(k.dt), 2, const_cast<void*>(k.base), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, static_cast<CUtensorMapSwizzle>(k.sw),
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}
}  // namespace

bool encode_2d(CUtensorMap* map, CUtensorMapDataType dt, int elem_bytes, const void* base, uint64_t inner,
               uint64_t outer, uint64_t ld_elems, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  const MapKey k{base, inner, outer, ld_elems, box_inner, box_outer, static_cast<int>(dt), elem_bytes,
                 static_cast<int>(sw)};
  if (g_map_cache_on.load() == 0) return encode_uncached(map, k);
  {
    std::lock_guard<std::mutex> lk(g_map_mu);
    for (int i = 0; i < g_map_n; ++i)
      if (g_map_key[i] == k) {
        *map = g_map_val[i];
        g_map_hits.fetch_add(1);
        return true;
      }
  }
  if (!encode_uncached(map, k)) return false;  // failures are not cached
  g_map_misses.fetch_add(1);
  std::lock_guard<std::mutex> lk(g_map_mu);
  int slot;
  if (g_map_n < kMapCacheSize) {
    slot = g_map_n++;
  } else {
    slot = g_map_next;
    g_map_next = (g_map_next + 1) % kMapCacheSize;
  }
  g_map_key[slot] = k;
  g_map_val[slot] = *map;
  return true;
}

namespace {
// Reads the status words at `rec` and clears them if a failure is recorded.  The read and the
// clear are ordered on `stream` (the caller's, already synchronised), so neither can overtake work
// the caller enqueues there later; the clear is complete when this returns.
int read_and_clear_status(void* rec, cudaStream_t stream) {
  int words[ST_WORDS];
  if (cudaMemcpyAsync(words, rec, sizeof(words), cudaMemcpyDeviceToHost, stream) != cudaSuccess) return FL_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FL_ERR_CUDA;
  if (words[ST_CODE] == 0) return FL_OK;
  if (cudaMemsetAsync(rec, 0, sizeof(words), stream) != cudaSuccess) return FL_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FL_ERR_CUDA;
  return words[ST_CODE];
}
}  // namespace

}  // namespace fl

extern "C" {

int fl_device_status(void* stream) {
  using namespace fl;
  DeviceInfo di;
  const int st = current_device(&di);
  if (st == FL_ERR_CUDA) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FL_ERR_CUDA;
  int* dptr = device_status_ptr(di.device);
  if (dptr == nullptr) return FL_ERR_CUDA;
  return read_and_clear_status(dptr, static_cast<cudaStream_t>(stream));
}

int fl_check_device_status(void* workspace, void* stream) {
  using namespace fl;
  if (workspace == nullptr) return fl_device_status(stream);
  if ((reinterpret_cast<uintptr_t>(workspace) & (kWsStatusBytes - 1)) != 0) return FL_ERR_ALIGNMENT;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FL_ERR_CUDA;
  return read_and_clear_status(workspace, static_cast<cudaStream_t>(stream));
}

void fl_set_cooperative_launch(int enable) { fl::g_cooperative.store(enable != 0 ? 1 : 0); }

void fl_set_descriptor_cache(int enable) {
  fl::g_map_cache_on.store(enable != 0 ? 1 : 0);
  if (enable == 0) {
    std::lock_guard<std::mutex> lk(fl::g_map_mu);
    fl::g_map_n = 0;
    fl::g_map_next = 0;
  }
}

void fl_descriptor_cache_stats(unsigned long long* hits, unsigned long long* misses) {
  if (hits != nullptr) *hits = fl::g_map_hits.load();
  if (misses != nullptr) *misses = fl::g_map_misses.load();
}

void fl_set_wait_timeout_ns(uint64_t ns) { fl::g_timeout_ns.store(ns == 0 ? fl::kDefaultTimeoutNs : ns); }

void fl_set_max_ctas(int n) { fl::g_max_ctas.store(n < 0 ? 0 : n); }

void fl_set_cta_pairing(int enable) { fl::g_pairing.store(enable != 0 ? 1 : 0); }

void fl_set_linear_decode(int enable) { fl::g_linear_decode.store(enable != 0 ? 1 : 0); }

int fl_linear_decode_shape(int kind, int M, int N, int K, int* cluster, int* ctas_per_sm, int* launches) {
  using namespace fl;
  if (cluster == nullptr || ctas_per_sm == nullptr || launches == nullptr) return FL_ERR_INVALID_ARG;
  *cluster = *ctas_per_sm = *launches = 0;
  if (M < 0 || N < 0 || K < 0 || kind < FL_DECODE_GELU || kind > FL_DECODE_ROWSCALE) return FL_ERR_INVALID_ARG;
  if (linear_decode_mode() == 0 || M == 0 || M > 32 || N == 0 || K == 0) return FL_OK;  // not a decode call
  DeviceInfo di;
  const int st = current_device(&di);
  if (st != FL_OK) return st;
  const int num_kb = cdiv(K, kBK);
  switch (kind) {
    case FL_DECODE_GELU: linear_decode_plan_gelu(cdiv(N, 128), num_kb, di, cluster, ctas_per_sm, launches); break;
    case FL_DECODE_SWIGLU: linear_decode_plan_swiglu(cdiv(N, 64), num_kb, di, cluster, ctas_per_sm, launches); break;
    case FL_DECODE_QKV: linear_decode_plan_qkv(cdiv(N, 128), num_kb, di, cluster, ctas_per_sm, launches); break;
    case FL_DECODE_QKV_FP8KV:
      linear_decode_plan_qkv_fp8kv(cdiv(N, 128), num_kb, di, cluster, ctas_per_sm, launches);
      break;
    case FL_DECODE_QUANT: linear_decode_plan_quant(cdiv(N, 128), num_kb, di, cluster, ctas_per_sm, launches); break;
    case FL_DECODE_RESID_GAMMA:
      linear_decode_plan_resgamma(cdiv(N, 128), num_kb, di, cluster, ctas_per_sm, launches);
      break;
    default: linear_decode_plan_rowscale(cdiv(N, 128), num_kb, di, cluster, ctas_per_sm, launches); break;
  }
  return FL_OK;
}

const char* fl_status_string(int status) {
  switch (status) {
    case FL_OK: return "ok";
    case FL_ERR_INVALID_ARG: return "invalid argument";
    case FL_ERR_UNSUPPORTED: return "unsupported shape or option";
    case FL_ERR_ALIGNMENT: return "pointer or row pitch not 16-byte aligned";
    case FL_ERR_WORKSPACE: return "workspace missing or too small";
    case FL_ERR_CUDA: return "CUDA runtime error";
    case FL_ERR_TIMEOUT: return "device-side wait timed out";
    case FL_ERR_ARCH: return "device is not sm_103";
    default: return "unknown status";
  }
}

int fl_version(void) { return 200; }

}  // extern "C"
