// Throughput probe of the block-scaled FP4 tensor-core MMA this library's
// tensor-core expert kernel issues (tcgen05.mma kind::mxf4 with E8M0 block
// scales, scale_vec::2X, M = 128, K = 64, A 128-byte swizzled, B without
// swizzle, operands in shared memory, scales and accumulators in tensor
// memory): the measured dense FP4 peak against which the prefill projections
// are reported.  A measurement aid beside the layer, not a step of it.
//
// One CTA per SM; one elected thread issues `iters` accumulating MMAs back to
// back, alternating between two accumulators when tensor memory holds two,
// then commits them to an mbarrier.  Operands are zero (the tensor pipe's
// rate does not depend on the values).  Every wait is bounded: a wait that
// runs out sets MOE_DEV_WAIT_TIMEOUT and waits once more (bounded) before the
// tensor memory is released.
#include "mx_device.cuh"
#include "tc_device.cuh"

namespace moe {
namespace {

constexpr int kProbeThreads = 128;
constexpr uint32_t kProbeA = 128 * 128;  // A: 128 rows x 128 bytes (K = 256, four K-steps)
constexpr uint32_t kProbeTmemCols = 512;
constexpr uint32_t kProbeSfb = 0, kProbeSfa = 16, kProbeD = 128;

// Bounded wait on an mbarrier phase measured in time (the MMAs of one launch
// take milliseconds; the bound is two seconds).
MOE_DEVFN bool probe_wait(uint32_t bar, unsigned *status) {
  uint64_t t0;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t0));
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, 0)) return true;
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    if ((i > (1u << 14) && t - t0 > 2000000000ull) || i > (1u << 30)) {  // (time counts after 2^14 polls)
      if (status) atomicOr(status, MOE_DEV_WAIT_TIMEOUT);
      return false;
    }
    __nanosleep(256);
  }
}

__global__ void __launch_bounds__(kProbeThreads, 1) mxf4_probe_kernel(int n, int iters, unsigned *status) {
  extern __shared__ __align__(1024) uint8_t smem_dyn[];
  __shared__ __align__(8) uint64_t done;
  __shared__ uint32_t tmem_slot;
  const uint32_t dyn = smem_addr(smem_dyn);
  const uint32_t base = (dyn + 1023u) & ~1023u;
  const uint32_t s_a = base, s_b = base + kProbeA;
  const uint32_t bbytes = (uint32_t)n * 128u;
  const int tid = threadIdx.x, warp = tid >> 5;

  for (uint32_t o = 16u * tid; o < kProbeA + bbytes; o += 16u * kProbeThreads) sts128(base + o, make_uint4(0, 0, 0, 0));
  fence_proxy_async();
  if (tid == 0) {
    mbar_init(smem_addr(&done), 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_addr(&tmem_slot), kProbeTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(&tmem_slot);
  {
    // scales 1.0 (E8M0 127) for both blocks of a K-step: B scales in
    // columns 0..3, A scales in columns 16 + quadrant, as the expert kernel
    // lays them out
    const uint32_t lanes = (uint32_t)(32 * warp) << 16;
#pragma unroll
    for (int c = 0; c < 4; ++c) tmem_st1(tmem + lanes + kProbeSfb + c, 0x7F7F7F7Fu);
    tmem_st1(tmem + lanes + kProbeSfa + warp, 0x7F7Fu);
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) {
    const uint32_t idesc = idesc_mxf4(128, n);
    const uint64_t adesc = smem_desc_sw128(s_a), bdesc = smem_desc(s_b, 128u, 1024u);
    const bool two = kProbeD + 2u * (uint32_t)n <= kProbeTmemCols;
    for (int i = 0; i < iters; ++i) {
      const uint32_t s = (uint32_t)(i & 3);  // the four K-steps of the staged tiles
      const uint32_t d = tmem + kProbeD + (two && (i & 1) ? (uint32_t)n : 0u);
      mma_mxf4(d, adesc + ((32u * s) >> 4), bdesc + ((256u * s) >> 4), idesc, tmem + kProbeSfa, tmem + kProbeSfb,
               true);
    }
    mma_commit(smem_addr(&done));
    if (!probe_wait(smem_addr(&done), status)) probe_wait(smem_addr(&done), status);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kProbeTmemCols);
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_mxf4_mma_probe(int n, int iters, double *flops, void *stream) {
  const char *name = "moe_mxf4_mma_probe";
  if (n != 64 && n != 128 && n != 256) return fail(MOE_ERR_INVALID_ARG, "%s: n=%d (64, 128 or 256)", name, n);
  if (iters < 1 || iters > (1 << 20)) return fail(MOE_ERR_INVALID_ARG, "%s: iters=%d (1 .. 2^20)", name, iters);
  const int G = sm_count();
  const int smem = (int)(kProbeA + 128u * (uint32_t)n + 1024u);
  const moe_status ast = ensure_smem_attr(reinterpret_cast<const void *>(mxf4_probe_kernel), smem, name);
  if (ast != MOE_OK) return ast;
  mxf4_probe_kernel<<<G, kProbeThreads, smem, static_cast<cudaStream_t>(stream)>>>(n, iters, device_status_word());
  const cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return cuda_fail(err, name);
  if (flops) *flops = 2.0 * 128.0 * n * 64.0 * (double)iters * (double)G;
  return MOE_OK;
}
