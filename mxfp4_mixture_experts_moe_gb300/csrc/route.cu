// Router logits and top-k selection.
//
// "DeepSeek-V4-Flash on AMD gfx90a: Correctness Recovery and Inference
// Performance Engineering", Fig. 1 (router top-6 of 256 routed experts) and
// §5.3 (deterministic index selection: ties fixed by logical id, selected
// positions in a fixed order).
#include "mx_device.cuh"

namespace moe {
namespace {

constexpr int kRouteWarps = 4;   // warps per CTA, each on its own EW experts
constexpr int kRouteTokens = 8;  // tokens per CTA (register tile)
constexpr int kRouteSlab = 64;   // 8-element chunks per shared-memory slab (512 inputs)

// logits[t, e] for a tile of kRouteWarps*EW experts x kRouteTokens tokens.
// The tile's router rows and activation rows pass through shared memory in
// slabs of 512 inputs (cp.async, double-buffered), so each input is read
// from L2 once per tile instead of once per (expert, token).  Every logit
// keeps the fixed order of the layer's router: lane l accumulates the
// 8-element chunks l, l+32, l+64, ... in increasing order, one fma per
// element, then the 32 partial sums meet in an xor butterfly (whose value is
// the same in every lane, IEEE addition being commutative).  So the bits of
// a logit depend neither on T nor on the tile it falls in.
template <int EW, bool XBF, bool WBF>
__global__ void __launch_bounds__(kRouteWarps * 32)
route_logits_kernel(const void *x, int64_t ld_x, const void *wr, int T, int H, int E, float *logits) {
  extern __shared__ __align__(128) uint8_t rsm[];
  constexpr uint32_t xsz = XBF ? 2 : 4, wsz = WBF ? 2 : 4;
  constexpr uint32_t wrow = kRouteSlab * 8 * wsz, xrow = kRouteSlab * 8 * xsz;  // bytes per row and slab
  constexpr int nw = kRouteWarps * EW;                                            // router rows per tile
  constexpr uint32_t wbytes = nw * wrow, slab_bytes = wbytes + kRouteTokens * xrow;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int e0 = blockIdx.x * nw, t0 = blockIdx.y * kRouteTokens;
  const int nch = H / 8, nslab = (nch + kRouteSlab - 1) / kRouteSlab;
  const uint32_t base = smem_addr(rsm);

  // rows past E or T are read from the last valid row; their sums are never stored
  auto stage = [&](int sl, int buf) {
    const uint32_t dst = base + (uint32_t)buf * slab_bytes;
    const int elem0 = sl * kRouteSlab * 8;
    constexpr int wp = wrow / 16, xp = xrow / 16;
    for (int i = tid; i < nw * wp; i += kRouteWarps * 32) {
      const int r = i / wp, q = i - r * wp;
      const int elem = elem0 + q * (16 / wsz);
      if (elem < H)
        cp_async16(dst + r * wrow + q * 16,
                   static_cast<const uint8_t *>(wr) + ((int64_t)min(e0 + r, E - 1) * H + elem) * wsz);
    }
    for (int i = tid; i < kRouteTokens * xp; i += kRouteWarps * 32) {
      const int r = i / xp, q = i - r * xp;
      const int elem = elem0 + q * (16 / xsz);
      if (elem < H)
        cp_async16(dst + wbytes + r * xrow + q * 16,
                   static_cast<const uint8_t *>(x) + ((int64_t)min(t0 + r, T - 1) * ld_x + elem) * xsz);
    }
    cp_async_commit();
  };

  float p[EW][kRouteTokens];
#pragma unroll
  for (int i = 0; i < EW; ++i)
#pragma unroll
    for (int j = 0; j < kRouteTokens; ++j) p[i][j] = 0.0f;
  stage(0, 0);
#pragma unroll 1
  for (int sl = 0; sl < nslab; ++sl) {
    if (sl + 1 < nslab) {
      stage(sl + 1, (sl + 1) & 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint32_t sb = base + (uint32_t)(sl & 1) * slab_bytes;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int cl = lane + 32 * h;  // chunk within the slab
      if (sl * kRouteSlab + cl < nch) {
        float wv[EW][8];
#pragma unroll
        for (int i = 0; i < EW; ++i) load8_smem(sb + (uint32_t)(warp * EW + i) * wrow + (uint32_t)cl * 8 * wsz, WBF, wv[i]);
#pragma unroll
        for (int j = 0; j < kRouteTokens; ++j) {
          float xv[8];
          load8_smem(sb + wbytes + (uint32_t)j * xrow + (uint32_t)cl * 8 * xsz, XBF, xv);
#pragma unroll
          for (int i = 0; i < EW; ++i)
#pragma unroll
            for (int q = 0; q < 8; ++q) p[i][j] = __fmaf_rn(xv[q], wv[i][q], p[i][j]);
        }
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < EW; ++i)
#pragma unroll
    for (int j = 0; j < kRouteTokens; ++j)
#pragma unroll
      for (int s = 16; s >= 1; s >>= 1) p[i][j] = __fadd_rn(p[i][j], __shfl_xor_sync(0xffffffffu, p[i][j], s));
#pragma unroll
  for (int i = 0; i < EW; ++i) {
#pragma unroll
    for (int j = 0; j < kRouteTokens; ++j) {
      const int e = e0 + warp * EW + i, t = t0 + j;
      if (lane == i * kRouteTokens + j && e < E && t < T) logits[(int64_t)t * E + e] = p[i][j];
    }
  }
}

// Small batches (T <= kSmallMaxT): one CTA per kSmallE experts x kSmallT
// tokens takes its whole router rows and token rows in one round of bulk
// copies (no slab pipeline: at a few tokens the slabs' serial round trips
// were the whole cost), then warp w dots expert w / 2 against four tokens
// at once.  Same per-logit order as route_logits_kernel.
constexpr int kSmallE = 2, kSmallT = 8, kSmallWarps = 4, kSmallMaxT = 16;

template <bool XBF, bool WBF>
__global__ void __launch_bounds__(kSmallWarps * 32)
route_logits_small_kernel(const void *x, int64_t ld_x, const void *wr, int T, int H, int E, float *logits,
                          unsigned *status) {
  extern __shared__ __align__(128) uint8_t rsm[];
  __shared__ __align__(8) uint64_t bar;
  constexpr uint32_t xsz = XBF ? 2 : 4, wsz = WBF ? 2 : 4;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int e0 = blockIdx.x * kSmallE, t0 = blockIdx.y * kSmallT;
  const int ne = min(kSmallE, E - e0), nt = min(kSmallT, T - t0);
  const uint32_t wrow_bytes = (uint32_t)H * wsz, xrow_bytes = (uint32_t)H * xsz;
  const uint32_t wbase = smem_addr(rsm), xbase = wbase + kSmallE * wrow_bytes;
  const uint32_t fb = smem_addr(&bar);
  if (tid == 0) {
    mbar_init(fb, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    mbar_arrive_expect_tx(fb, (uint32_t)ne * wrow_bytes + (uint32_t)nt * xrow_bytes);
    const uint64_t wpol = policy_evict_first(), xpol = policy_evict_last();  // x is read by every CTA
    for (int i = 0; i < ne; ++i)
      bulk_g2s(wbase + (uint32_t)i * wrow_bytes, static_cast<const uint8_t *>(wr) + (int64_t)(e0 + i) * wrow_bytes,
               wrow_bytes, fb, wpol);
    for (int j = 0; j < nt; ++j)
      bulk_g2s(xbase + (uint32_t)j * xrow_bytes, static_cast<const uint8_t *>(x) + (int64_t)(t0 + j) * ld_x * xsz,
               xrow_bytes, fb, xpol);
  }
  if (!mbar_wait(fb, 0, status)) {
    mbar_wait(fb, 0, nullptr);  // once more (bounded) before leaving with copies in flight
    return;
  }
  const int el = warp >> 1, tl0 = 4 * (warp & 1);
  if (el >= ne || tl0 >= nt) return;
  const int nj = min(4, nt - tl0);
  const uint32_t wrow = wbase + (uint32_t)el * wrow_bytes, xrow = xbase + (uint32_t)tl0 * xrow_bytes;
  float p[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  const int nch = H / 8;
#pragma unroll 1
  for (int c = lane; c < nch; c += 32) {
    float wv[8];
    load8_smem(wrow + (uint32_t)c * 8 * wsz, WBF, wv);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (j < nj) {
        float xv[8];
        load8_smem(xrow + (uint32_t)j * xrow_bytes + (uint32_t)c * 8 * xsz, XBF, xv);
#pragma unroll
        for (int q = 0; q < 8; ++q) p[j] = __fmaf_rn(xv[q], wv[q], p[j]);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) p[j] = __fadd_rn(p[j], __shfl_xor_sync(0xffffffffu, p[j], s));
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (lane == j && j < nj) logits[(int64_t)(t0 + tl0 + j) * E + e0 + el] = p[j];
}

// The small-batch kernel when T and its shared memory allow (else false).
bool launch_route_logits_small(bool xbf, bool wbf, const void *x, int64_t ld_x, const void *wr, int T, int H, int E,
                               float *logits, cudaStream_t s, cudaError_t *err) {
  if (T > kSmallMaxT) return false;
  const size_t smem = (size_t)kSmallE * H * (wbf ? 2 : 4) + (size_t)kSmallT * H * (xbf ? 2 : 4);
  if (smem > 200 * 1024) return false;
  void (*kern)(const void *, int64_t, const void *, int, int, int, float *, unsigned *) =
      xbf ? (wbf ? route_logits_small_kernel<true, true> : route_logits_small_kernel<true, false>)
          : (wbf ? route_logits_small_kernel<false, true> : route_logits_small_kernel<false, false>);
  if (smem > 48 * 1024 &&
      ensure_smem_attr(reinterpret_cast<const void *>(kern), (int)smem, "moe_route_topk") != MOE_OK) {
    *err = cudaErrorInvalidValue;
    return true;
  }
  const dim3 grid((E + kSmallE - 1) / kSmallE, (T + kSmallT - 1) / kSmallT);
  kern<<<grid, kSmallWarps * 32, smem, s>>>(x, ld_x, wr, T, H, E, logits, device_status_word());
  *err = cudaGetLastError();
  return true;
}

template <int EW, bool XBF, bool WBF>
cudaError_t launch_route_logits(const void *x, int64_t ld_x, const void *wr, int T, int H, int E, float *logits,
                                cudaStream_t s) {
  constexpr uint32_t smem = 2u * (kRouteWarps * EW * kRouteSlab * 8 * (WBF ? 2 : 4) +
                                  kRouteTokens * kRouteSlab * 8 * (XBF ? 2 : 4));
  static_assert(smem <= 227 * 1024, "slabs fit shared memory");
  if (smem > 48 * 1024 &&
      ensure_smem_attr(reinterpret_cast<const void *>(route_logits_kernel<EW, XBF, WBF>), (int)smem,
                       "moe_route_topk") != MOE_OK)
    return cudaErrorInvalidValue;
  dim3 grid((E + kRouteWarps * EW - 1) / (kRouteWarps * EW), (T + kRouteTokens - 1) / kRouteTokens);
  route_logits_kernel<EW, XBF, WBF><<<grid, kRouteWarps * 32, smem, s>>>(x, ld_x, wr, T, H, E, logits);
  return cudaGetLastError();
}

template <int EW>
cudaError_t launch_route_logits_dt(bool xbf, bool wbf, const void *x, int64_t ld_x, const void *wr, int T, int H,
                                   int E, float *logits, cudaStream_t s) {
  if (xbf && wbf) return launch_route_logits<EW, true, true>(x, ld_x, wr, T, H, E, logits, s);
  if (xbf) return launch_route_logits<EW, true, false>(x, ld_x, wr, T, H, E, logits, s);
  if (wbf) return launch_route_logits<EW, false, true>(x, ld_x, wr, T, H, E, logits, s);
  return launch_route_logits<EW, false, false>(x, ld_x, wr, T, H, E, logits, s);
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
  if ((T + kRouteTokens - 1) / kRouteTokens > 65535) return fail(MOE_ERR_UNSUPPORTED, "moe_route_topk: T=%d too large", T);
  // experts per warp: more CTAs for small batches, more reuse of each staged input for large ones
  const bool xbf = x_dtype == MOE_BF16, wbf = w_dtype == MOE_BF16;
  cudaError_t err = cudaSuccess;
  if (!launch_route_logits_small(xbf, wbf, x, ld_x, w_router, T, H, E, logits, s, &err))
    err = T <= 8    ? launch_route_logits_dt<1>(xbf, wbf, x, ld_x, w_router, T, H, E, logits, s)
          : T <= 64 ? launch_route_logits_dt<2>(xbf, wbf, x, ld_x, w_router, T, H, E, logits, s)
                    : launch_route_logits_dt<4>(xbf, wbf, x, ld_x, w_router, T, H, E, logits, s);
  if (err != cudaSuccess) return cuda_fail(err, "moe_route_topk: logits launch");
  topk_kernel<<<(T + 3) / 4, 128, 0, s>>>(logits, bias, T, E, k, ids, weights);
  err = cudaGetLastError();
  if (err != cudaSuccess) return cuda_fail(err, "moe_route_topk: top-k launch");
  return MOE_OK;
}
