// Q8 activation quantisation, per row and per block of 32 columns.
//
// "DeepSeek-V4-Flash on AMD gfx90a", §6.1 ("online BF16 activation
// quantization to INT8 per 32 elements") and §8.2 ("forms group32 INT8
// values/scales").  scale = amax/127 (IEEE division), q = rne(x * (1/scale))
// clamped to [-127, 127]; every step is an IEEE-rounded fp32 operation, so the
// codes are the same bits on any IEEE machine.
#include "mx_device.cuh"

namespace moe {
namespace {

template <bool BF16>
__global__ void __launch_bounds__(256)
quant_q8_kernel(const void *x, int64_t ld_x, int rows, int nblk, int8_t *q, int64_t ld_q, float *scale,
                int64_t ld_s) {
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= (int64_t)rows * nblk) return;
  const int r = (int)(gid / nblk), b = (int)(gid % nblk);
  float v[32];
  if (BF16) {
    const uint16_t *p = static_cast<const uint16_t *>(x) + r * ld_x + 32 * b;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint4 w = ldg_nc(p + 8 * c);
      uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[8 * c + 2 * j] = __uint_as_float(u[j] << 16);
        v[8 * c + 2 * j + 1] = __uint_as_float(u[j] & 0xFFFF0000u);
      }
    }
  } else {
    const float *p = static_cast<const float *>(x) + r * ld_x + 32 * b;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint4 w = ldg_nc(p + 4 * c);
      v[4 * c] = __uint_as_float(w.x);
      v[4 * c + 1] = __uint_as_float(w.y);
      v[4 * c + 2] = __uint_as_float(w.z);
      v[4 * c + 3] = __uint_as_float(w.w);
    }
  }
  uint32_t packed[8];
  const float d = q8_block(v, packed, nullptr);
  uint4 *dst = reinterpret_cast<uint4 *>(q + r * ld_q + 32 * b);
  dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
  scale[r * ld_s + b] = d;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status act_quant_q8(const void *x, moe_dtype x_dtype, int rows, int cols, int64_t ld_x, int8_t *q,
                                   int64_t ld_q, float *scale, int64_t ld_s, void *stream) {
  if (rows < 0 || cols < 0 || cols % 32) return fail(MOE_ERR_INVALID_ARG, "act_quant_q8: rows=%d cols=%d (cols %% 32 == 0)", rows, cols);
  if (x_dtype != MOE_F32 && x_dtype != MOE_BF16) return fail(MOE_ERR_INVALID_ARG, "act_quant_q8: bad dtype");
  if (rows == 0 || cols == 0) return MOE_OK;
  const int es = x_dtype == MOE_BF16 ? 2 : 4;
  if (!x || !q || !scale) return fail(MOE_ERR_INVALID_ARG, "act_quant_q8: null pointer");
  if (ld_x < cols || (ld_x * es) % 16 || (uintptr_t)x % 16) return fail(MOE_ERR_INVALID_ARG, "act_quant_q8: x must be 16-byte aligned with a 16-byte multiple row stride (ld_x=%lld)", (long long)ld_x);
  if (ld_q < cols || ld_q % 16 || (uintptr_t)q % 16) return fail(MOE_ERR_INVALID_ARG, "act_quant_q8: q must be 16-byte aligned with ld_q a multiple of 16 (ld_q=%lld)", (long long)ld_q);
  if (ld_s < cols / 32 || (uintptr_t)scale % 4) return fail(MOE_ERR_INVALID_ARG, "act_quant_q8: ld_s=%lld", (long long)ld_s);
  const int nblk = cols / 32;
  const int64_t n = (int64_t)rows * nblk;
  const int64_t grid = (n + 255) / 256;
  if (grid > 0x7fffffff) return fail(MOE_ERR_UNSUPPORTED, "act_quant_q8: too many rows");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (x_dtype == MOE_BF16) quant_q8_kernel<true><<<(unsigned)grid, 256, 0, s>>>(x, ld_x, rows, nblk, q, ld_q, scale, ld_s);
  else quant_q8_kernel<false><<<(unsigned)grid, 256, 0, s>>>(x, ld_x, rows, nblk, q, ld_q, scale, ld_s);
  cudaError_t err = cudaGetLastError();
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "act_quant_q8: launch");
}
