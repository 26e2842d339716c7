// Host side of the C ABI: error reporting, the device status word, device
// properties, and the one-time kernel attributes.  The per-device caches are
// filled under a mutex, so host threads may make their first calls at once.
#include <stdarg.h>
#include <stdio.h>

#include <map>
#include <mutex>
#include <set>
#include <tuple>

#include "common.cuh"

namespace {

thread_local char g_last_error[512] = "";

// Device status word: kernels OR MOE_DEV_* bits into it; moe_device_status()
// reads and clears it.  One word per device (a module-scope device variable).
__device__ unsigned g_device_status = 0;

struct DeviceInfo {
  unsigned *status = nullptr;  // device address of g_device_status
  int sms = 0;
};

std::mutex g_info_mu;
std::map<int, DeviceInfo> g_info;                        // by device ordinal
std::set<std::tuple<const void *, int, int>> g_attr_set;  // (kernel, device, bytes) already configured

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return dev;
}

// The current device's cached properties (filled on first use), or null.
const DeviceInfo *device_info() {
  const int dev = current_device();
  if (dev < 0) return nullptr;
  std::lock_guard<std::mutex> lock(g_info_mu);
  DeviceInfo &d = g_info[dev];
  if (!d.status) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return nullptr;
    d.sms = n;
    d.status = static_cast<unsigned *>(p);
  }
  return &d;
}

}  // namespace

namespace moe {

moe_status fail(moe_status s, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return s;
}

moe_status cuda_fail(cudaError_t e, const char *what) {
  return fail(MOE_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

unsigned *device_status_word() {
  const DeviceInfo *d = device_info();
  return d ? d->status : nullptr;
}

int sm_count() {
  const DeviceInfo *d = device_info();
  return d ? d->sms : 1;
}

moe_status ensure_smem_attr(const void *kern, int bytes, const char *name) {
  const int dev = current_device();
  if (dev < 0) return fail(MOE_ERR_CUDA, "%s: no current CUDA device", name);
  std::lock_guard<std::mutex> lock(g_info_mu);
  const auto key = std::make_tuple(kern, dev, bytes);
  if (g_attr_set.count(key)) return MOE_OK;
  const cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (err != cudaSuccess) return cuda_fail(err, name);
  g_attr_set.insert(key);
  return MOE_OK;
}

}  // namespace moe

extern "C" const char *moe_last_error(void) { return g_last_error; }

extern "C" int moe_abi_version(void) { return MOE_ABI_VERSION; }

extern "C" moe_status moe_device_status(void *stream, uint32_t *flags) {
  cudaError_t err = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return moe::cuda_fail(err, "moe_device_status: stream synchronize");
  unsigned v = 0;
  err = cudaMemcpyFromSymbol(&v, g_device_status, sizeof v);
  if (err != cudaSuccess) return moe::cuda_fail(err, "moe_device_status: read");
  if (v) {
    const unsigned zero = 0;
    err = cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero);
    if (err != cudaSuccess) return moe::cuda_fail(err, "moe_device_status: clear");
  }
  if (flags) *flags = v;
  if (v) return moe::fail(MOE_ERR_DEVICE, "device status word 0x%x", v);
  return MOE_OK;
}
