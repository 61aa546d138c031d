// Library-wide entry points of the C ABI: status strings, device class, build
// id and the device status word that bounded waits report through.
#include <mutex>

#include "common.cuh"

namespace kinv {

namespace {
// One status word per device.  Device code reaches it through the pointer
// the host passes at launch; host code reads it in kinv_last_device_status.
__device__ int g_status_word;

constexpr int kMaxDevices = 64;
std::once_flag g_once[kMaxDevices];
int* g_status_ptr[kMaxDevices];
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
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_status_word) == cudaSuccess) g_status_ptr[dev] = static_cast<int*>(p);
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
}  // namespace

int* device_status_word() {
  const int dev = ensure();
  return dev < 0 ? nullptr : g_status_ptr[dev];
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

}  // namespace kinv

extern "C" {

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
