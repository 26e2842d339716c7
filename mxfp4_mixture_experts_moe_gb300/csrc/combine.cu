// Routing-weighted combine of the per-slot down outputs, in slot order.
//
// "DeepSeek-V4-Flash on AMD gfx90a", §8.2: the down consumer "retains the
// existing FP32 top-k partial and fixed reduction"; Table 4 ("BF16 down
// partial ... retain FP32 partials").  out[t,n] = fma chain over j = 0..k-1,
// fp32, the same for every token whatever T is.  A slot whose weight is
// exactly 0 adds nothing and its y row is not read: top-k gives that weight
// to a slot with no expert (only NaN scores were left for it), whose y row
// no projection writes.
#include "common.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(256)
combine_kernel(const float *y, int64_t ld_y, const float *w, int T, int k, int H, float *out, int64_t ld_out) {
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= (int64_t)T * H) return;
  const int t = (int)(gid / H), n = (int)(gid % H);
  const float *wt = w + (int64_t)t * k;
  const float *yt = y + (int64_t)t * k * ld_y + n;
  float acc = wt[0] != 0.0f ? __fmul_rn(wt[0], yt[0]) : 0.0f;
  for (int j = 1; j < k; ++j)
    if (wt[j] != 0.0f) acc = __fmaf_rn(wt[j], yt[(int64_t)j * ld_y], acc);
  out[(int64_t)t * ld_out + n] = acc;
}

// The join of the shared expert onto the routed output: out[t,n] += ys[t,n].
__global__ void __launch_bounds__(256)
join_add_kernel(const float *ys, int64_t ld_ys, int T, int H, float *out, int64_t ld_out) {
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= (int64_t)T * H) return;
  const int t = (int)(gid / H), n = (int)(gid % H);
  float *o = out + (int64_t)t * ld_out + n;
  *o = __fadd_rn(*o, ys[(int64_t)t * ld_ys + n]);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_combine(const float *y, int64_t ld_y, const float *w, int T, int k, int H, float *out,
                                  int64_t ld_out, void *stream) {
  if (T < 0 || k <= 0 || H <= 0) return fail(MOE_ERR_INVALID_ARG, "moe_combine: T=%d k=%d H=%d", T, k, H);
  if (T == 0) return MOE_OK;
  if (!y || !w || !out) return fail(MOE_ERR_INVALID_ARG, "moe_combine: null pointer");
  if (ld_y < H || ld_out < H) return fail(MOE_ERR_INVALID_ARG, "moe_combine: ld_y=%lld ld_out=%lld < H=%d", (long long)ld_y, (long long)ld_out, H);
  const int64_t n = (int64_t)T * H;
  const int64_t grid = (n + 255) / 256;
  if (grid > 0x7fffffff) return fail(MOE_ERR_UNSUPPORTED, "moe_combine: too large");
  combine_kernel<<<(unsigned)grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(y, ld_y, w, T, k, H, out, ld_out);
  cudaError_t err = cudaGetLastError();
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_combine: launch");
}

extern "C" moe_status moe_join_add(const float *ys, int64_t ld_ys, int T, int H, float *out, int64_t ld_out,
                                   void *stream) {
  if (T < 0 || H <= 0) return fail(MOE_ERR_INVALID_ARG, "moe_join_add: T=%d H=%d", T, H);
  if (T == 0) return MOE_OK;
  if (!ys || !out) return fail(MOE_ERR_INVALID_ARG, "moe_join_add: null pointer");
  if (ld_ys < H || ld_out < H) return fail(MOE_ERR_INVALID_ARG, "moe_join_add: ld_ys=%lld ld_out=%lld < H=%d", (long long)ld_ys, (long long)ld_out, H);
  const int64_t n = (int64_t)T * H;
  const int64_t grid = (n + 255) / 256;
  if (grid > 0x7fffffff) return fail(MOE_ERR_UNSUPPORTED, "moe_join_add: too large");
  join_add_kernel<<<(unsigned)grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(ys, ld_ys, T, H, out, ld_out);
  cudaError_t err = cudaGetLastError();
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_join_add: launch");
}
