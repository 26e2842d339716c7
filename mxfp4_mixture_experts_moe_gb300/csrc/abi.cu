// Host side of the C ABI: error reporting, the device status word, device
// properties.
#include <stdarg.h>
#include <stdio.h>

#include "common.cuh"

namespace {

thread_local char g_last_error[512] = "";

// Device status word: kernels OR MOE_DEV_* bits into it; moe_device_status()
// reads and clears it.  One word per device (a module-scope device variable).
__device__ unsigned g_device_status = 0;

unsigned *g_status_ptr[64] = {nullptr};
int g_sm_count[64] = {0};

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return dev;
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
  const int dev = current_device();
  if (dev < 0 || dev >= 64) return nullptr;
  if (!g_status_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<unsigned *>(p);
  }
  return g_status_ptr[dev];
}

int sm_count() {
  const int dev = current_device();
  if (dev < 0 || dev >= 64) return 1;
  if (!g_sm_count[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
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
