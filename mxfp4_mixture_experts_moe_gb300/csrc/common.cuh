// Shared device helpers for the sm_103a MXFP4 MoE kernels: inline-PTX
// wrappers (mbarrier, bulk copies, streaming loads), the E2M1 -> int8 nibble
// conversion and the E8M0 scale decode.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_mxfp4.h"

#define MOE_DEVFN __device__ __forceinline__

namespace moe {

// ------------------------------------------------------------------ host glue
// (defined in abi.cu)
moe_status fail(moe_status s, const char *fmt, ...);
moe_status cuda_fail(cudaError_t e, const char *what);
unsigned *device_status_word();  // per-device address of the status word, or NULL
int sm_count();
// cudaFuncSetAttribute(kern, MaxDynamicSharedMemorySize, bytes) on the current
// device, once per (kernel, device, bytes); thread-safe.
moe_status ensure_smem_attr(const void *kern, int bytes, const char *name);

// Tensor-core path of the expert projections (tc_expert.cu): mode 0 gate/up
// with SwiGLU into out0, 1 gate into out0 and up into out1, 2 down into out0.
// Tile policy of the stage calls ("Optimizing DeepSeek V4 Flash Inference on
// a Strix Halo Pair", "MXFP4 routed-expert kernels": a direct route for small
// batches instead of partially filled expert tiles): a call of fewer than
// kTensorMinRows rows runs every expert on the CUDA-core kernel (the exact-
// rows range); a larger call splits its experts on the device by their row
// counts in `offsets`: at most kLightExpertRows rows on the CUDA-core kernel,
// more on the tensor-core kernel, in two launches on disjoint experts.
constexpr int kTensorMinRows = 17;
#ifndef MOE_LIGHT_EXPERT_ROWS
#define MOE_LIGHT_EXPERT_ROWS 4
#endif
constexpr int kLightExpertRows = MOE_LIGHT_EXPERT_ROWS;
bool tc_expert_supported(int K, int N);
moe_status launch_tc_expert(int mode, const int8_t *aq, int64_t ld_aq, const float *as, int64_t ld_as,
                            const uint8_t *w0, const uint8_t *s0, const uint8_t *w1, const uint8_t *s1,
                            const int32_t *offsets, const int32_t *sorted, int64_t cap, int A, int k, int E,
                            int K, int N, int bytoken, int min_rows, float *out0, float *out1, int64_t ld_out,
                            cudaStream_t stream, const char *name);

// The expert projections of 1-16-row calls (krow.cu): mode 0 gate/up with
// SwiGLU into out0, 1 gate into out0 and up into out1, 2 down into out0 (and
// the slot-ordered combine into cout when cout is given), over the experts
// with at most max_rows rows.  MOE_ERR_UNSUPPORTED (nothing enqueued) when the
// shape does not fit its shared-memory plan.
moe_status launch_krow(int mode, const int8_t *aq, int64_t ld_aq, const float *as, int64_t ld_as, const uint8_t *w0,
                       const uint8_t *s0, const uint8_t *w1, const uint8_t *s1, const int32_t *offsets,
                       const int32_t *sorted, int64_t cap, int T, int k, int E, int K, int N, int max_rows,
                       float *out0, float *out1, int64_t ld_out, const float *wts, float *cout, int64_t ld_cout,
                       cudaStream_t stream, const char *name);

// The single-launch decode forward (decode.cu) behind moe_decode_forward and
// moe_decode_forward_shared: their arguments, the shared expert's (sh, or
// null), and clear_ws: zero the workspace on the stream right before the
// launch, once every argument check has passed.
struct SharedArgs {
  const uint8_t *wg, *sg, *wu, *su, *wd, *sd;
  float *h;
  int64_t ld_h;
  float *y;
  int64_t ld_y;
};
moe_status decode_forward(const char *name, const void *x, moe_dtype x_dtype, int64_t ld_x, const void *w_router,
                          moe_dtype w_dtype, const float *bias, const uint8_t *wg, const uint8_t *sg, const uint8_t *wu,
                          const uint8_t *su, const uint8_t *wd, const uint8_t *sd, int T, int H, int E, int k, int I,
                          float *out, int64_t ld_out, float *logits, int32_t *ids, float *weights, float *h,
                          int64_t ld_h, float *y, int64_t ld_y, void *workspace, size_t ws_bytes,
                          const SharedArgs *sh, bool clear_ws, void *stream);

// Token of assignment a = t*k + j, i.e. a / k, as a multiply-high by
// kdiv_of(k) = ceil(2^32 / k), exact for a < 2^28 and k <= 8.  k = 1 is
// encoded as 0 (ceil(2^32 / 1) does not fit 32 bits) and is the identity.
inline uint32_t kdiv_of(int k) { return k <= 1 ? 0u : (uint32_t)((0x100000000ull + (uint64_t)k - 1) / (uint64_t)k); }
MOE_DEVFN int token_of(int a, uint32_t kdiv) { return kdiv ? (int)__umulhi((unsigned)a, kdiv) : a; }

// ------------------------------------------------------------------ formats

// E8M0 byte u -> 2^(u-128) as fp32 (the E8M0 factor 2^(u-127) halved, because
// the integer block dots count twice the E2M1 values).  Exact for every byte
// (subnormal for u < 2); byte 255 is NaN.
MOE_DEVFN float e8m0_half(uint32_t u) {
  if (u - 2u < 253u) return __uint_as_float((u - 1u) << 23);  // bytes 2..254: normal fp32
  const uint32_t bits = (u == 255u) ? 0x7FC00000u : (0x00400000u >> (1u - u));
  return __uint_as_float(bits);
}

// PTX prmt.b32 in its default mode: each 4-bit selector picks one of the 8
// bytes of {b, a} with its low 3 bits; a set top bit replicates that byte's
// sign bit instead.  (The CUDA __byte_perm intrinsic documents only the low
// 3 bits, so the sign mode is reached through PTX.)
MOE_DEVFN uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// 8 E2M1 codes (one 32-bit word, element i in nibble i) -> 8 bytes holding
// 12 + 2*value, i.e. 12 + {0,1,2,3,4,6,8,12} for positive codes and
// 12 - {..} for negative ones, all in [0, 24].  Two byte-permute lookups per
// 4 codes: the first table answers codes 0..7 and yields 0 for codes 8..15
// (the selector's top bit replicates the table byte's sign bit, which is 0);
// the second answers the sign-flipped codes the same way; OR merges them.
// dot(x, 12 + 2v) - 12 * sum(x) = dot(x, 2v).
MOE_DEVFN void e2m1x8_to_off12(uint32_t w, uint32_t &lo, uint32_t &hi) {
  const uint32_t P0 = 0x0F0E0D0Cu, P1 = 0x18141210u;  // 12 + {0,1,2,3 | 4,6,8,12}
  const uint32_t N0 = 0x090A0B0Cu, N1 = 0x00040608u;  // 12 - {0,1,2,3 | 4,6,8,12}
  uint32_t wx = w ^ 0x88888888u;
  lo = prmt(P0, P1, w) | prmt(N0, N1, wx);
  hi = prmt(P0, P1, w >> 16) | prmt(N0, N1, wx >> 16);
}

// ------------------------------------------------------------------ loads

MOE_DEVFN uint4 ldg_stream(const void *p) {  // weights: read once, keep out of L1
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

MOE_DEVFN uint4 ldg_nc(const void *p) {  // activations: re-read by many warps
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

MOE_DEVFN uint4 lds128(uint32_t addr) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(addr));
  return r;
}

MOE_DEVFN uint32_t lds_u8(uint32_t addr) {
  uint32_t r;
  asm volatile("ld.shared.u8 %0, [%1];" : "=r"(r) : "r"(addr));
  return r;
}

MOE_DEVFN uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier

MOE_DEVFN void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

MOE_DEVFN void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

MOE_DEVFN void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

MOE_DEVFN void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One poll of an mbarrier phase.  The thread may be suspended inside the
// poll until the phase completes; the hint caps that at 20 us, so that the
// bounds below are bounds in time.
MOE_DEVFN bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(20000u)
      : "memory");
  return ok != 0;
}

MOE_DEVFN uint64_t gtimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Limits of a bounded mbarrier wait: two seconds of global time, counted
// only once kWaitMinPolls polls have passed (so that a step of the global
// timer, which can be re-synchronised, never ends a wait of normal length),
// or kWaitMaxPolls polls.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kWaitMinPolls = 1u << 12;
constexpr uint32_t kWaitMaxPolls = 1u << 24;

// Bounded wait: gives up at the limits above, raises MOE_DEV_WAIT_TIMEOUT
// and returns false.
MOE_DEVFN bool mbar_wait(uint32_t bar, uint32_t parity, unsigned *status) {
  uint64_t t0 = 0;
  for (uint32_t i = 0; i < kWaitMaxPolls; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (i >= 16) __nanosleep(64);
    if (i == 64) t0 = gtimer_ns();
    else if (i > kWaitMinPolls && (i & 255u) == 0 && gtimer_ns() - t0 > kWaitLimitNs) break;
  }
  if (status) atomicOr(status, MOE_DEV_WAIT_TIMEOUT);
  return false;
}

// ------------------------------------------------------------------ async copies

// Bulk global -> shared copy (TMA unit) completing on an mbarrier's tx count.
// dst, src 16-byte aligned, bytes a multiple of 16.
MOE_DEVFN void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

MOE_DEVFN uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
MOE_DEVFN uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Per-thread async 4- or 16-byte copies (cp.async), tracked by an mbarrier.
MOE_DEVFN void cp_async4(uint32_t dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
MOE_DEVFN void cp_async16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
MOE_DEVFN void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
MOE_DEVFN void cp_async_wait() {  // at most N of this thread's committed groups still pending
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
MOE_DEVFN void cp_async_mbar_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

}  // namespace moe
