// Router logits and top-k selection.
//
// "DeepSeek-V4-Flash on AMD gfx90a: Correctness Recovery and Inference
// Performance Engineering", Fig. 1 (router top-6 of 256 routed experts) and
// §5.3 (deterministic index selection: ties fixed by logical id, selected
// positions in a fixed order).
#include "mx_device.cuh"

namespace moe {
namespace {

constexpr int kRouteWarps = 4;   // warps per CTA, one expert each
constexpr int kRouteTokens = 8;  // tokens per warp pass (register tile)

// logits[t, e] for one expert per warp and kRouteTokens tokens per CTA row.
__global__ void __launch_bounds__(kRouteWarps * 32)
route_logits_kernel(const void *x, bool xbf, int64_t ld_x, const void *wr, bool wbf, int T, int H, int E,
                    float *logits) {
  const int lane = threadIdx.x & 31;
  const int e = blockIdx.x * kRouteWarps + (threadIdx.x >> 5);
  const int t0 = blockIdx.y * kRouteTokens;
  if (e >= E) return;
  const int nt = min(kRouteTokens, T - t0);
  float p[8];
  router_logits_warp(x, xbf, ld_x, wr, wbf, e, t0, nt, H, p);
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (lane == 0 && j < nt) logits[(int64_t)(t0 + j) * E + e] = p[j];
}

// Top-k per token, one warp per token.
__global__ void __launch_bounds__(128)
topk_kernel(const float *logits, const float *bias, int T, int E, int k, int32_t *ids, float *weights) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (t >= T) return;
  int id[8];
  float w[8];
  topk_warp(logits + (int64_t)t * E, bias, E, k, id, w);
  if (lane < k) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j == lane) {
        ids[(int64_t)t * k + j] = id[j];
        weights[(int64_t)t * k + j] = w[j];
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
  route_logits_kernel<<<grid, kRouteWarps * 32, 0, s>>>(x, x_dtype == MOE_BF16, ld_x, w_router, w_dtype == MOE_BF16,
                                                        T, H, E, logits);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return cuda_fail(err, "moe_route_topk: logits launch");
  topk_kernel<<<(T + 3) / 4, 128, 0, s>>>(logits, bias, T, E, k, ids, weights);
  err = cudaGetLastError();
  if (err != cudaSuccess) return cuda_fail(err, "moe_route_topk: top-k launch");
  return MOE_OK;
}
