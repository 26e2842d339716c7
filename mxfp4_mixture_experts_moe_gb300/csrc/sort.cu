// Expert sorter: stable counting sort of the token->expert assignments.
//
// "DeepSeek-V4-Flash on AMD gfx90a", §7.1 item 8 (expert sorter grouping
// assignments into row blocks), and the lucebox PR "feat(ds4): add concurrent
// serving on Strix Halo and R9700 + Strix", "Reduce expert-route overhead"
// (negative sentinels for rows an expert does not own).  Integer work only:
// the result is unique and matches the oracle bit for bit.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kSortThreads = 1024;

// One CTA.  Phase 1 counts per expert (shared-memory integer atomics; counts
// do not depend on their order).  Phase 2 scans the padded counts into
// offsets.  Phase 3 places assignments tile by tile in increasing a: inside a
// warp, lanes with the same expert rank themselves with match_any; across
// the warps of a tile, a per-warp count table gives each warp its base.
__global__ void __launch_bounds__(kSortThreads)
sort_kernel(const int32_t *ids, int A, int E, int tile_rows, int32_t *offsets, int32_t *sorted, int32_t *inv,
            unsigned *status) {
  extern __shared__ int sm[];
  int *count = sm;               // [E]
  int *base = count + E;         // [E] segment start
  int *running = base + E;       // [E] assignments placed so far
  int *wcnt = running + E;       // [32][E] per-warp counts of the current tile
  __shared__ int warp_tot[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  for (int i = tid; i < E; i += kSortThreads) {
    count[i] = 0;
    running[i] = 0;
  }
  for (int i = tid; i < 32 * E; i += kSortThreads) wcnt[i] = 0;
  __syncthreads();
  for (int a = tid; a < A; a += kSortThreads) {
    const int e = ids[a];
    if (e >= 0 && e < E) atomicAdd(&count[e], 1);
    else if (status) atomicOr(status, MOE_DEV_BAD_EXPERT_ID);
  }
  __syncthreads();

  // exclusive scan of padded counts (E <= 1024: one value per thread)
  int v = 0;
  if (tid < E) v = (count[tid] + tile_rows - 1) / tile_rows * tile_rows;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    warp_tot[lane] = w;  // inclusive
  }
  __syncthreads();
  const int excl = incl - v + (warp > 0 ? warp_tot[warp - 1] : 0);
  if (tid < E) {
    base[tid] = excl;
    offsets[tid] = excl;
    for (int p = excl + count[tid]; p < excl + v; ++p) sorted[p] = -1;
  }
  if (tid == kSortThreads - 1) offsets[E] = warp_tot[31];
  __syncthreads();

  const unsigned lt_mask = (1u << lane) - 1u;
  for (int tile = 0; tile < A; tile += kSortThreads) {
    const int a = tile + tid;
    int e = a < A ? ids[a] : -1;
    const bool ok = e >= 0 && e < E;
    if (!ok) e = -1 - (a < A ? 0 : 1);  // invalid / past-the-end lanes group apart
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt_mask);
    if (ok && rank == 0) wcnt[warp * E + e] = __popc(peers);
    __syncthreads();
    if (ok) {
      int pre = 0;
      for (int w = 0; w < warp; ++w) pre += wcnt[w * E + e];
      const int pos = base[e] + running[e] + pre + rank;
      sorted[pos] = a;
      inv[a] = pos;
    } else if (a < A) {
      inv[a] = -1;
    }
    __syncthreads();
    for (int i = tid; i < E; i += kSortThreads) {
      int tot = 0;
      for (int w = 0; w < 32; ++w) {
        tot += wcnt[w * E + i];
        wcnt[w * E + i] = 0;
      }
      running[i] += tot;
    }
    __syncthreads();
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int64_t moe_sort_tokens_capacity(int T, int k, int E, int tile_rows) {
  if (T < 0 || k < 0 || E < 0 || tile_rows < 1) return -1;
  return (int64_t)T * k + (int64_t)E * (tile_rows - 1);
}

extern "C" moe_status moe_sort_tokens(const int32_t *ids, int T, int k, int E, int tile_rows, int32_t *offsets,
                                      int32_t *sorted, int64_t cap, int32_t *inv, void *stream) {
  if (T < 0 || k <= 0 || E <= 0 || tile_rows < 1) return fail(MOE_ERR_INVALID_ARG, "moe_sort_tokens: T=%d k=%d E=%d tile_rows=%d", T, k, E, tile_rows);
  if (E > 1024) return fail(MOE_ERR_UNSUPPORTED, "moe_sort_tokens: E=%d > 1024", E);
  const int64_t A = (int64_t)T * k;
  const int64_t need = A + (int64_t)E * (tile_rows - 1);
  if (need > 0x7fffffff) return fail(MOE_ERR_UNSUPPORTED, "moe_sort_tokens: too many assignments");
  if (!offsets) return fail(MOE_ERR_INVALID_ARG, "moe_sort_tokens: null offsets");
  if (A > 0 && (!ids || !inv)) return fail(MOE_ERR_INVALID_ARG, "moe_sort_tokens: null pointer");
  if (cap < need || (need > 0 && !sorted)) return fail(MOE_ERR_INVALID_ARG, "moe_sort_tokens: cap=%lld < %lld", (long long)cap, (long long)need);
  const size_t smem = sizeof(int) * (size_t)E * 35;
  const moe_status ast = ensure_smem_attr(reinterpret_cast<const void *>(sort_kernel), 35 * 1024 * 4,
                                         "moe_sort_tokens: smem attribute");
  if (ast != MOE_OK) return ast;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  sort_kernel<<<1, kSortThreads, smem, s>>>(ids, (int)A, E, tile_rows, offsets, sorted, inv, device_status_word());
  cudaError_t err = cudaGetLastError();
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_sort_tokens: launch");
}
