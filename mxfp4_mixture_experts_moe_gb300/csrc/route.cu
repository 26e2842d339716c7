// Router logits and top-k selection.
//
// "DeepSeek-V4-Flash on AMD gfx90a: Correctness Recovery and Inference
// Performance Engineering", Fig. 1 (router top-6 of 256 routed experts) and
// §5.3 (deterministic index selection: ties fixed by logical id, selected
// positions in a fixed order).
#include <math_constants.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kRouteWarps = 4;   // warps per CTA, one expert each
constexpr int kRouteTokens = 8;  // tokens per warp pass (register tile)

template <bool BF16>
MOE_DEVFN void load8(const void *base, int64_t elem, float (&v)[8]) {
  if (BF16) {
    uint4 r = ldg_nc(static_cast<const uint16_t *>(base) + elem);
    uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[2 * j] = __uint_as_float(w[j] << 16);
      v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
  } else {
    const float *p = static_cast<const float *>(base) + elem;
    uint4 a = ldg_nc(p), b = ldg_nc(p + 4);
    v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y);
    v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
    v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y);
    v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
  }
}

// logits[t, e] for one expert per warp and kRouteTokens tokens per pass.  Lane
// l owns chunks l, l+32, ... of 8 consecutive inputs and accumulates them in
// increasing order with one fma per element; the 32 partial sums are then
// added by an xor butterfly (lane 0's sum is ((p0+p16)+(p8+p24))+...).
template <bool XBF, bool WBF>
__global__ void __launch_bounds__(kRouteWarps * 32)
route_logits_kernel(const void *x, int64_t ld_x, const void *wr, int T, int H, int E, float *logits) {
  const int lane = threadIdx.x & 31;
  const int e = blockIdx.x * kRouteWarps + (threadIdx.x >> 5);
  const int t0 = blockIdx.y * kRouteTokens;
  if (e >= E) return;
  const int nch = H / 8;
  float p[kRouteTokens];
#pragma unroll
  for (int j = 0; j < kRouteTokens; ++j) p[j] = 0.0f;
  for (int c = lane; c < nch; c += 32) {
    float wv[8];
    load8<WBF>(wr, (int64_t)e * H + 8 * c, wv);
#pragma unroll
    for (int j = 0; j < kRouteTokens; ++j) {
      if (t0 + j < T) {
        float xv[8];
        load8<XBF>(x, (int64_t)(t0 + j) * ld_x + 8 * c, xv);
#pragma unroll
        for (int q = 0; q < 8; ++q) p[j] = __fmaf_rn(xv[q], wv[q], p[j]);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kRouteTokens; ++j) {
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) p[j] = __fadd_rn(p[j], __shfl_xor_sync(0xffffffffu, p[j], s));
    if (lane == 0 && t0 + j < T) logits[(int64_t)(t0 + j) * E + e] = p[j];
  }
}

// (score, id) ordering: larger score first, then lower id.
MOE_DEVFN bool better(float s, int i, float bs, int bi) {
  return s > bs || (s == bs && i < bi);
}

// Top-k per token, one warp per token.  Lane l holds the scores of experts
// l, l+32, ...; each of the k rounds takes the best unselected expert by an
// xor-butterfly argmax, so slots come out in descending score order.
__global__ void __launch_bounds__(128)
topk_kernel(const float *logits, const float *bias, int T, int E, int k, int32_t *ids, float *weights) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (t >= T) return;
  const int ns = (E + 31) / 32;
  float sc[32];
#pragma unroll
  for (int s = 0; s < 32; ++s) {
    const int e = lane + 32 * s;
    float v = -CUDART_INF_F;
    if (s < ns && e < E) {
      v = logits[(int64_t)t * E + e];
      if (bias) v = __fadd_rn(v, bias[e]);
    }
    sc[s] = v;
  }
  uint32_t taken = 0;
  float sel_s[8];
  int sel_i[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < k) {
      float bs = -CUDART_INF_F;
      int bi = 0x7fffffff;
#pragma unroll
      for (int s = 0; s < 32; ++s) {
        const int e = lane + 32 * s;
        if (s < ns && e < E && !((taken >> s) & 1u) && better(sc[s], e, bs, bi)) {
          bs = sc[s];
          bi = e;
        }
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        const float os = __shfl_xor_sync(0xffffffffu, bs, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (better(os, oi, bs, bi)) {
          bs = os;
          bi = oi;
        }
      }
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
      sel_s[j] = bs;
      sel_i[j] = bi;
    }
  }
  if (lane == 0) {
    float sig[8];
    float total = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < k) {
        sig[j] = __frcp_rn(__fadd_rn(1.0f, expf(-sel_s[j])));
        total = __fadd_rn(total, sig[j]);
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < k) {
        ids[(int64_t)t * k + j] = sel_i[j];
        weights[(int64_t)t * k + j] = __fdiv_rn(sig[j], total);
      }
    }
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_route_topk(const void *x, moe_dtype x_dtype, int64_t ld_x, const void *w_router,
                                     moe_dtype w_dtype, const float *bias, int T, int H, int E, int k,
                                     float *logits, int32_t *ids, float *weights, void *stream) {
  if (T < 0 || H <= 0 || E <= 0 || k <= 0) return fail(MOE_ERR_INVALID_ARG, "moe_route_topk: T=%d H=%d E=%d k=%d", T, H, E, k);
  if (x_dtype != MOE_F32 && x_dtype != MOE_BF16) return fail(MOE_ERR_INVALID_ARG, "moe_route_topk: bad x dtype");
  if (w_dtype != MOE_F32 && w_dtype != MOE_BF16) return fail(MOE_ERR_INVALID_ARG, "moe_route_topk: bad router dtype");
  if (H % 8) return fail(MOE_ERR_INVALID_ARG, "moe_route_topk: H=%d must be a multiple of 8", H);
  if (E > 1024) return fail(MOE_ERR_UNSUPPORTED, "moe_route_topk: E=%d > 1024", E);
  if (k > 8 || k > E) return fail(MOE_ERR_INVALID_ARG, "moe_route_topk: k=%d must be <= min(E, 8)", k);
  if (T == 0) return MOE_OK;
  const int xes = x_dtype == MOE_BF16 ? 2 : 4;
  if (!x || !w_router || !logits || !ids || !weights) return fail(MOE_ERR_INVALID_ARG, "moe_route_topk: null pointer");
  if (ld_x < H || (ld_x * xes) % 16) return fail(MOE_ERR_INVALID_ARG, "moe_route_topk: ld_x=%lld", (long long)ld_x);
  if ((uintptr_t)x % 16 || (uintptr_t)w_router % 16) return fail(MOE_ERR_INVALID_ARG, "moe_route_topk: x and w_router must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  dim3 grid((E + kRouteWarps - 1) / kRouteWarps, (T + kRouteTokens - 1) / kRouteTokens);
  if (grid.y > 65535) return fail(MOE_ERR_UNSUPPORTED, "moe_route_topk: T=%d too large", T);
  const bool xb = x_dtype == MOE_BF16, wb = w_dtype == MOE_BF16;
  if (xb && wb) route_logits_kernel<true, true><<<grid, kRouteWarps * 32, 0, s>>>(x, ld_x, w_router, T, H, E, logits);
  else if (xb) route_logits_kernel<true, false><<<grid, kRouteWarps * 32, 0, s>>>(x, ld_x, w_router, T, H, E, logits);
  else if (wb) route_logits_kernel<false, true><<<grid, kRouteWarps * 32, 0, s>>>(x, ld_x, w_router, T, H, E, logits);
  else route_logits_kernel<false, false><<<grid, kRouteWarps * 32, 0, s>>>(x, ld_x, w_router, T, H, E, logits);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return cuda_fail(err, "moe_route_topk: logits launch");
  topk_kernel<<<(T + 3) / 4, 128, 0, s>>>(logits, bias, T, E, k, ids, weights);
  err = cudaGetLastError();
  if (err != cudaSuccess) return cuda_fail(err, "moe_route_topk: top-k launch");
  return MOE_OK;
}
