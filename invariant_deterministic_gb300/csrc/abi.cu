// Library-wide entry points of the C ABI: status strings, device class, build
// id and the device status word that bounded waits report through.
#include <cuda.h>

#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"

namespace kinv {

namespace {
// One status word per device.  Device code reaches it through the pointer
// the host passes at launch; host code reads it in kinv_last_device_status.
__device__ int g_status_word;

constexpr int kMaxDevices = 64;
std::once_flag g_once[kMaxDevices];
int g_sm_count[kMaxDevices];
int g_smem_optin[kMaxDevices];
int g_smem_per_sm[kMaxDevices];
int g_smem_reserved[kMaxDevices];

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

void init_device(int dev) {
  cudaDeviceGetAttribute(&g_sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
  cudaDeviceGetAttribute(&g_smem_optin[dev], cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaDeviceGetAttribute(&g_smem_per_sm[dev], cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  cudaDeviceGetAttribute(&g_smem_reserved[dev], cudaDevAttrReservedSharedMemoryPerBlock, dev);
}

int ensure() {
  const int dev = current_device();
  if (dev < 0) return -1;
  std::call_once(g_once[dev], init_device, dev);
  return dev;
}

using PFN_ctxGetCurrent = CUresult (*)(CUcontext*);
using PFN_ctxGetId = CUresult (*)(CUcontext, unsigned long long*);

struct CtxFns {
  PFN_ctxGetCurrent get_current = nullptr;
  PFN_ctxGetId get_id = nullptr;
};

const CtxFns& ctx_fns() {
  static CtxFns f;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_current = reinterpret_cast<PFN_ctxGetCurrent>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_id = reinterpret_cast<PFN_ctxGetId>(p);
  });
  return f;
}

// Device addresses of the status word, one per CUDA context (a context torn
// down and created again -- cudaDeviceReset -- loads the module afresh, so an
// address from the old context must not be reused).
std::mutex g_ctx_mu;
std::map<unsigned long long, int*> g_status_by_ctx;
std::map<std::pair<unsigned long long, const void*>, size_t> g_smem_by_ctx;
}  // namespace

unsigned long long context_id() {
  const CtxFns& f = ctx_fns();
  CUcontext c = nullptr;
  if (!f.get_current || f.get_current(&c) != CUDA_SUCCESS || !c) return 0;
  unsigned long long id = 0;
  if (f.get_id && f.get_id(c, &id) == CUDA_SUCCESS) return id;
  return static_cast<unsigned long long>(reinterpret_cast<uintptr_t>(c));
}

int* device_status_word() {
  if (ensure() < 0) return nullptr;
  std::lock_guard<std::mutex> lock(g_ctx_mu);
  unsigned long long ctx = context_id();
  if (ctx != 0) {
    auto it = g_status_by_ctx.find(ctx);
    if (it != g_status_by_ctx.end()) return it->second;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
  ctx = context_id();  // the lookup makes the device's primary context current if none was
  if (ctx != 0) g_status_by_ctx[ctx] = static_cast<int*>(p);
  return static_cast<int*>(p);
}

kinv_status ensure_smem(const void* kernel, size_t bytes) {
  // without the attribute a block may hold 48 KB of static and dynamic
  // shared memory together
  if (bytes == 0) return KINV_OK;
  std::lock_guard<std::mutex> lock(g_ctx_mu);
  const auto key = std::make_pair(context_id(), kernel);
  auto it = g_smem_by_ctx.find(key);
  if (key.first != 0 && it != g_smem_by_ctx.end() && it->second >= bytes) return KINV_OK;
  cudaFuncAttributes fa{};
  if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess) return KINV_ERR_CUDA;
  if (bytes + fa.sharedSizeBytes > 48 * 1024 &&
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)) !=
          cudaSuccess)
    return KINV_ERR_CUDA;
  if (key.first != 0) g_smem_by_ctx[key] = bytes;
  return KINV_OK;
}

int sm_count() {
  const int dev = ensure();
  return dev < 0 ? 0 : g_sm_count[dev];
}
int max_smem_optin() {
  const int dev = ensure();
  return dev < 0 ? 0 : g_smem_optin[dev];
}
int smem_per_sm() {
  const int dev = ensure();
  return dev < 0 ? 0 : g_smem_per_sm[dev];
}
int smem_reserved_per_block() {
  const int dev = ensure();
  return dev < 0 ? 0 : g_smem_reserved[dev];
}

// One thread waits on a barrier nothing completes, for at most limit_ns,
// through the bounded wait every kernel pipeline uses; it then records the
// time-out and the block exits.
__global__ void bounded_wait_test_kernel(unsigned long long limit_ns, int* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    fence_mbar_init();
    mbar_wait_bounded(smem_addr(&bar), 0, status, DEV_TIMEOUT_TEST, limit_ns);
  }
}

}  // namespace kinv

extern "C" {

kinv_status kinv_test_bounded_wait(int64_t limit_ns, kinv_stream stream) {
  if (limit_ns < 1000 || limit_ns > 100000000) return KINV_ERR_INVALID_ARG;
  int* status = kinv::device_status_word();
  if (!status) return KINV_ERR_CUDA;
  kinv::bounded_wait_test_kernel<<<1, 32, 0, stream>>>(static_cast<unsigned long long>(limit_ns), status);
  return kinv::launch_status();
}

const char* kinv_status_string(int status) {
  switch (status) {
    case KINV_OK: return "KINV_OK";
    case KINV_ERR_INVALID_ARG: return "KINV_ERR_INVALID_ARG";
    case KINV_ERR_UNSUPPORTED: return "KINV_ERR_UNSUPPORTED";
    case KINV_ERR_ALIGNMENT: return "KINV_ERR_ALIGNMENT";
    case KINV_ERR_WORKSPACE: return "KINV_ERR_WORKSPACE";
    case KINV_ERR_CUDA: return "KINV_ERR_CUDA";
    case KINV_ERR_TIMEOUT: return "KINV_ERR_TIMEOUT";
    default: return "KINV_ERR_UNKNOWN";
  }
}

const char* kinv_device_class(void) { return "cuda-sm103a"; }

const char* kinv_build_id(void) { return KINV_BUILD_ID; }

int kinv_last_device_status(kinv_stream stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return KINV_ERR_CUDA;
  int* p = kinv::device_status_word();
  if (!p) return KINV_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return KINV_ERR_CUDA;
  if (word == 0) return KINV_OK;
  const int zero = 0;
  if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return KINV_ERR_CUDA;
  // Low byte holds the status (as a signed byte); the rest says where.
  return static_cast<int>(static_cast<int8_t>(word & 0xFF));
}

}  // extern "C"
