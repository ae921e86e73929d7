// api.cu -- status strings, the device error word, launch flags and
// per-device properties shared by the three entry points.
#include <map>
#include <tuple>
#include <mutex>
#include <utility>

#include "common.cuh"

namespace {

// One error word per device that loads the library.  Bounded device waits
// and candidate overflows OR their bit in; sv_last_device_error() reads and
// clears it.
__device__ unsigned g_error_word;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned *g_err_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};
std::atomic<unsigned> g_flags{0};
std::atomic<uint64_t> g_launches{0};

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
  return d;
}

}  // namespace

namespace sv {

unsigned *device_error_word() {
  int d = current_device();
  if (d < 0) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[d]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    g_err_ptr[d] = static_cast<unsigned *>(p);
  }
  return g_err_ptr[d];
}

int device_sm_count() {
  int d = current_device();
  if (d < 0) return 0;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sm_count[d]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess) return 0;
    g_sm_count[d] = n;
  }
  return g_sm_count[d];
}

cudaError_t raise_smem_limit(const void *kernel, size_t bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void *, int>, size_t> done;
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  size_t &cur = done[{kernel, d}];
  if (bytes <= cur) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) cur = bytes;
  return e;
}

int max_active_clusters(const void *kern, int block, size_t smem, int cl) {
  static std::mutex mu;
  static std::map<std::tuple<const void *, int, size_t, int, int>, int> cache;
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return 0;
  const auto key = std::make_tuple(kern, cl, smem, block, d);
  {
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  if (raise_smem_limit(kern, smem) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)cl);
  cfg.blockDim = dim3((unsigned)block);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  std::lock_guard<std::mutex> lk(mu);
  cache[key] = n;
  return n;
}

unsigned launch_flags() { return g_flags.load(std::memory_order_relaxed); }
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

}  // namespace sv

extern "C" {

const char *sv_status_string(sv_status s) {
  switch (s) {
    case SV_OK: return "ok";
    case SV_ERR_INVALID_ARG: return "invalid argument";
    case SV_ERR_UNSUPPORTED: return "unsupported shape or setting";
    case SV_ERR_CUDA: return "CUDA error";
    case SV_ERR_TIMEOUT: return "bounded device wait expired";
    case SV_ERR_WORKSPACE: return "workspace missing or too small";
    case SV_ERR_OVERFLOW: return "candidate set overflow (top-k ties)";
  }
  return "unknown status";
}

sv_status sv_last_device_error(sv_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return SV_ERR_CUDA;
  unsigned *p = sv::device_error_word();
  if (!p) return SV_ERR_CUDA;
  unsigned v = 0, zero = 0;
  if (cudaMemcpy(&v, p, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return SV_ERR_CUDA;
  if (v != 0 && cudaMemcpy(p, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
    return SV_ERR_CUDA;
  if (v & sv::ERR_TIMEOUT) return SV_ERR_TIMEOUT;
  if (v & sv::ERR_LISTS) return SV_ERR_INVALID_ARG;  // (the chain also flags the bad lists)
  if (v & sv::ERR_OVERFLOW) return SV_ERR_OVERFLOW;
  return SV_OK;
}

void sv_set_launch_flags(unsigned flags) {
  g_flags.store(flags & (SV_LAUNCH_PDL | SV_LAUNCH_QMM_CUDA_CORES | SV_LAUNCH_ATTN_MMA_SYNC |
                         SV_LAUNCH_ATTN_TCGEN05 | SV_LAUNCH_TEST_STALL_COPY));
}
unsigned sv_get_launch_flags(void) { return g_flags.load(); }
uint64_t sv_kernel_launch_count(void) { return g_launches.load(); }

}  // extern "C"
