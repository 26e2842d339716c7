// Allocation-free variant of the single-launch decode path.
//
// Some callers cannot call cudaMalloc at the point where they run the layer:
// serving loops whose latency budget rules out the device-wide
// synchronisation an allocation can cause, runtimes whose device memory is
// owned by a pool that this library cannot reach, or embedders that forbid
// allocation after start-up.  For them,
// moe_decode_forward_noalloc keeps every intermediate of moe_decode_forward
// (grid-barrier counters, router logits, top-k ids and weights, the SwiGLU
// activations exchanged between the two projections) in one fixed array of
// device memory that belongs to this library.  The caller passes only the
// inputs and the layer output.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds kScratchBytes of it until the process exits.  Host code must
// never use the variable's name as a pointer: on the host it is a stand-in
// symbol, not a device address.  Its device address is looked up with
// cudaGetSymbolAddress on every call, with the caller's device current (a
// host-side query, no stream work; the first call on a device also loads the
// module there, which is why that first call should come before any stream
// capture).  Looking it up each time keeps a call correct after
// cudaDeviceReset or in a new primary context.
#include "common.cuh"

namespace moe {
namespace {

// Limits of the fixed scratch array.
constexpr int kScratchMaxSlots = 64;        // T * k
constexpr int kScratchMaxLogits = 32768;    // T * E
constexpr int kScratchMaxI = 4096;          // expert intermediate width
constexpr size_t kBarBytes = 1024;          // grid-barrier and readiness words (>= moe_decode_workspace_bytes)
constexpr size_t kOffBar = 0;
constexpr size_t kOffIds = kBarBytes;       // int32 [T*k]
constexpr size_t kOffW = kOffIds + 4 * kScratchMaxSlots;
constexpr size_t kOffLogits = kOffW + 4 * kScratchMaxSlots;  // fp32 [T][E]
constexpr size_t kOffH = kOffLogits + 4 * (size_t)kScratchMaxLogits;  // fp32 [T*k][I]
constexpr size_t kScratchBytes = kOffH + 4 * (size_t)kScratchMaxSlots * kScratchMaxI;
static_assert(kOffH % 256 == 0, "h rows must stay 16-byte aligned");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of the current device's copy of the scratch array.
moe_status scratch_for_current_device(unsigned char **out) {
  void *ptr = nullptr;
  const cudaError_t err = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
  if (err != cudaSuccess || !ptr) return cuda_fail(err, "moe_decode_forward_noalloc: cudaGetSymbolAddress");
  *out = static_cast<unsigned char *>(ptr);
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_decode_forward_noalloc(const void *x, moe_dtype x_dtype, int64_t ld_x, const void *w_router,
                                                 moe_dtype w_dtype, const float *bias, const uint8_t *wg,
                                                 const uint8_t *sg, const uint8_t *wu, const uint8_t *su,
                                                 const uint8_t *wd, const uint8_t *sd, int T, int H, int E, int k,
                                                 int I, float *out, int64_t ld_out, void *stream) {
  const char *name = "moe_decode_forward_noalloc";
  if (T < 0 || E <= 0 || k <= 0 || I <= 0) return fail(MOE_ERR_INVALID_ARG, "%s: T=%d E=%d k=%d I=%d", name, T, E, k, I);
  if (T == 0) return MOE_OK;
  if ((int64_t)T * k > kScratchMaxSlots)
    return fail(MOE_ERR_UNSUPPORTED, "%s: T*k=%lld exceeds the fixed scratch limit of %d", name, (long long)T * k, kScratchMaxSlots);
  if ((int64_t)T * E > kScratchMaxLogits)
    return fail(MOE_ERR_UNSUPPORTED, "%s: T*E=%lld exceeds the fixed scratch limit of %d", name, (long long)T * E, kScratchMaxLogits);
  if (I > kScratchMaxI) return fail(MOE_ERR_UNSUPPORTED, "%s: I=%d exceeds the fixed scratch limit of %d", name, I, kScratchMaxI);
  if (moe_decode_workspace_bytes() > kBarBytes) return fail(MOE_ERR_UNSUPPORTED, "%s: workspace layout", name);
  unsigned char *s = nullptr;
  moe_status st = scratch_for_current_device(&s);
  if (st != MOE_OK) return st;
  // The barrier counter and its hold word must start at zero (the kernel
  // clears the readiness words itself); the other regions are written before
  // they are read within one launch.  decode_forward clears the barrier
  // words on the stream only after every argument check has passed, so a
  // rejected call enqueues nothing.
  return decode_forward(name, x, x_dtype, ld_x, w_router, w_dtype, bias, wg, sg, wu, su, wd, sd, T, H, E, k, I, out,
                        ld_out, reinterpret_cast<float *>(s + kOffLogits), reinterpret_cast<int32_t *>(s + kOffIds),
                        reinterpret_cast<float *>(s + kOffW), reinterpret_cast<float *>(s + kOffH), I, nullptr, 0,
                        s + kOffBar, kBarBytes, nullptr, true, stream);
}
