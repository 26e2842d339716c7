// Tensor-core (tcgen05) path of the MXFP4 expert projections, used by the
// stage calls for the experts with more than 4 rows in batches of more than
// 16 rows (prefill and large decode batches; the 1-16-row decode regime and
// the light experts keep the CUDA-core kernels).
//
// The layer's projections as grouped GEMMs over the rows routed to each
// expert: "DeepSeek-V4-Flash on AMD gfx90a", §6.1 (packed FP4 weights with
// E8M0 block scales against INT8 per-32 activations, the block terms
// I_b * xs_b * 2^(u_b - 128)) and "Optimizing DeepSeek V4 Flash Inference on a
// Strix Halo Pair", "MXFP4 routed-expert kernels" (prefill tiles over the
// tokens of one expert).  An output is  sum_k v_k 2^(u_b - 127) y_k  with v_k
// the E2M1 weight values, u_b their E8M0 byte and y_k = q_k xs_b the Q8
// activation (code times block scale).
//
// The tensor core takes the weights as stored (kind::mxf4, K = 64 per MMA,
// the E8M0 byte as A's block scale).  y is not an MMA type, so a pre-pass
// (plane_kernel) writes the activation row of every sorted position (the
// rows of an expert's tile are then consecutive) as six E2M1 "planes" with
// E8M0 block scales of their own, y ~ sum_p d_p 2^(e_pb - 127), built
// greedily per 32-block: plane p's scale is the smallest power of two that
// puts the block's remaining values within E2M1's range (+-6), its digits
// are those values rounded to E2M1, and the rounding error is left to plane
// p + 1.  Each plane gains about two bits; six leave an error near 1e-5 of
// the projection's RMS (the layer's tolerance is 1e-3; five planes left
// 2e-4, enough to move one Q8(h) code in two thousand across a rounding
// boundary) and give every integer of a unit-scale block exactly.  The
// planes are 6 x 16 rows of one MMA operand (N = 96): one MMA per matrix and
// K-step covers 16 activation rows, and the accumulator takes the whole
// reduction, read once per tile.
//
// Edge cases take an exact fallback in the epilogue (the CUDA-core block
// arithmetic, acc = fma(I_b, xs_b * 2^(u_b - 128), acc) block by block):
// weight rows with an E8M0 byte outside [64, 192] (the MMA is given such a
// byte clamped into that range) and activation rows whose plane scales would
// leave E8M0's range or whose values are not finite.  No real checkpoint or
// activation reaches either; the tests do.
//
// Tiles: 128 weight rows (MMA M) x up to 16 activation rows of one expert,
// K in stages of 256 (4 K-steps).  One persistent CTA per SM walks the tiles
// it derives from the expert offsets:
//   warps 0-7   epilogue: tensor-memory lane quadrant warp % 4, 8 activation
//               rows each: sums the planes' columns, SwiGLU, stores (and
//               the exact fallback where a tile needs it)
//   warps 8-11  per stage: A block scales (clamped, the quadrant's rows) and
//               B block scales (all 96 operand rows, in every quadrant) into
//               tensor memory
//   warp 12     tensor copies (TMA, 128-byte swizzled boxes) of the weights
//               and of the tile's activation planes
//   warp 13     MMA issue
//   warp 14     column tables of the next tile
// Tensor memory: per stage slot the A and B scales, two K-steps per 32-bit
// word (the instruction descriptor's scale-factor IDs pick the half); two
// accumulator buffers of 96 columns per matrix, so the epilogue of one tile
// overlaps the MMAs of the next.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <map>
#include <mutex>

#include "mx_device.cuh"
#include "tc_device.cuh"

namespace moe {
namespace {

constexpr int kRows = 128;                       // weight rows per tile (MMA M)
constexpr int kNTMax = 32;                       // activation rows per tile, at most (NT = 16 or 32)
constexpr int kPlanes = 6;                       // E2M1 planes per activation row
constexpr int kStageK = 256;                     // reduction elements per stage (8 MX blocks)
constexpr int kSteps = kStageK / 64;             // MMA K-steps per stage
constexpr uint32_t kAMat = kRows * kStageK / 2;  // one matrix's packed weights per stage (16 KB)
constexpr int kDrainWarps = 8;
constexpr int kPrepWarps = 4;
constexpr int kWarpTma = kDrainWarps + kPrepWarps;
constexpr int kWarpMma = kWarpTma + 1;
constexpr int kWarpTab = kWarpMma + 1;
constexpr int kThreads = 32 * (kWarpTab + 1);
constexpr int kMaxStages = 8;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kUcLo = 0x40404040u;  // E8M0 bytes given to the MMA: clamped to [64, 192]
constexpr uint32_t kUcHi = 0xC0C0C0C0u;

// Four E8M0 bytes clamped to the MMA's range.
MOE_DEVFN uint32_t clamp_e8m0x4(uint32_t w) { return __vmaxu4(__vminu4(w, kUcHi), kUcLo); }
// Non-zero when one of four E8M0 bytes lies outside the MMA's range.
MOE_DEVFN uint32_t outside_e8m0x4(uint32_t w) { return __vcmpltu4(w, kUcLo) | __vcmpgtu4(w, kUcHi); }

enum Mode { kSwiglu = 0, kRaw = 1, kDownMode = 2 };

struct TcArgs {
  const int8_t *aq;  // Q8 activation codes: x rows (gate/up, by token) or h rows (down, by assignment)
  int64_t ld_aq;
  const float *as;
  int64_t ld_as;
  const uint8_t *w0, *w1;  // packed weights [E*N][K/2] (the exact fallback reads them)
  const uint8_t *s0, *s1;  // E8M0 bytes of the weight rows, [E*N][K/32]
  const int32_t *offsets, *sorted;
  int64_t cap;
  int A, k, E, K, N;  // K reduction length, N output rows per expert
  int bytoken;        // activation row of assignment a: a / k (1) or a (0)
  int min_rows;       // experts with at most this many rows are left to the CUDA-core kernel
  uint32_t kdiv;
  int npos;                // sorted positions (of the planes)
  const uint8_t *bsc;      // [npos][kPlanes][K/32] E8M0 bytes of the planes
  const int *bflag;        // [npos] != 0: the position takes the exact fallback
  float *out0, *out1;
  int64_t ld_out;
  unsigned *status;
  int nstage;
  uint32_t off_a, off_b, off_misc;  // shared memory (from the 1024-aligned base)
};

struct TcMaps {  // 2-D tensor maps (TMA): the packed weights, the activation planes
  CUtensorMap w[2];
  CUtensorMap b;
};

struct TcShared {
  uint64_t a_full[kMaxStages], b_full[kMaxStages], slot_free[kMaxStages];
  uint64_t d_full[2], d_free[2];
  uint64_t tab_full[2], tab_empty[2], ext_full[2];
  uint32_t tmem_slot;
  int ncols[2];
  int mrow[2];         // first output row of the tile within its expert
  int64_t wrow[2];     // first weight row of the tile (expert * N + mrow)
  int col0[2];         // first sorted position of the tile
  int colrow[2][kNTMax];  // activation row of each column (row 0 for a column without one)
  int colasg[2][kNTMax];  // output row (assignment) of each column (-1: none)
  int colext[2][kNTMax];  // the column's activation row takes the exact fallback
  int ext[2][4];       // per table buffer and quadrant: a weight byte outside the clamp range
  int prefix[1];       // [E + 1] tiles before expert e
};

uint32_t tc_shared_bytes(int E) { return (uint32_t)(sizeof(TcShared) + 4u * (uint32_t)E); }

MOE_DEVFN void tmem_ld8_nowait(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}
MOE_DEVFN void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Bounded mbarrier wait without back-off sleeps, for the short hand-offs of
// the MMA thread and the epilogue; gives up as mbar_wait does.
MOE_DEVFN bool mbar_wait_spin(uint32_t bar, uint32_t parity, unsigned *status) {
  uint64_t t0 = 0;
  for (uint32_t i = 0; i < kWaitMaxPolls; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (i == 64) t0 = gtimer_ns();
    else if (i > kWaitMinPolls && (i & 255u) == 0 && gtimer_ns() - t0 > kWaitLimitNs) break;
  }
  if (status) atomicOr(status, MOE_DEV_WAIT_TIMEOUT);
  return false;
}

// Bounded mbarrier wait taken by a whole warp, with one answer for all lanes.
MOE_DEVFN bool warp_wait(uint32_t bar, uint32_t parity, unsigned *status) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, status));
}

// 2-D tensor copy of one box into shared memory, completing on bar, with an
// L2 cache policy for the lines it reads.
MOE_DEVFN void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// Eight floats rounded to E2M1 (round to nearest, ties to even, saturating
// at +-6), element i in nibble i of the result (the weights' packing).
MOE_DEVFN uint32_t e2m1x8_from_f32(const float (&t)[8]) {
  uint32_t w;
  asm("{\n .reg .b8 b0, b1, b2, b3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      " mov.b32 %0, {b0, b1, b2, b3};\n}"
      : "=r"(w)
      : "f"(t[0]), "f"(t[1]), "f"(t[2]), "f"(t[3]), "f"(t[4]), "f"(t[5]), "f"(t[6]), "f"(t[7]));
  return w;
}

// The eight E2M1 values of a word (element i in nibble i), exactly.
MOE_DEVFN void e2m1x8_to_f32(uint32_t w, float (&v)[8]) {
  uint32_t h[4];
  asm("{\n .reg .b8 b0, b1, b2, b3;\n"
      " mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n"
      " cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n"
      " cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
#pragma unroll
  for (int i = 0; i < 4; ++i)
    asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %2;\n cvt.f32.f16 %0, lo;\n cvt.f32.f16 %1, hi;\n}"
        : "=f"(v[2 * i]), "=f"(v[2 * i + 1])
        : "r"(h[i]));
}

// The activation planes, by sorted position (so that the 16 positions of a
// tile are 16 consecutive rows of each plane): one thread per (position,
// 32-block), of the activation row of the position's assignment.  y = q * xs,
// then for each plane: m = max |remaining|, scale s = 2^e the smallest power
// of two with m / s <= 6, digits = E2M1(remaining / s), remaining -= digits
// * s.  A block of zeros (and a position without an assignment) gets scale
// byte 127 and zero digits.  bflag[pos] is set when a scale leaves
// [2^-126, 2^126] or y is not finite (the caller zeroes bflag first).
// planes[p][pos][K/2] (element k of a row in nibble k % 2 of byte k / 2, as
// the weights), bsc[pos][p][nb].
__global__ void __launch_bounds__(256) plane_kernel(const int8_t *aq, int64_t ld_aq, const float *as, int64_t ld_as,
                                                     const int32_t *sorted, int npos, int A, int bytoken,
                                                     uint32_t kdiv, int K, uint8_t *planes, uint8_t *bsc,
                                                     int *bflag) {
  const int nb = K / 32;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)npos * nb) return;
  const int pos = (int)(i / nb), b = (int)(i - (int64_t)pos * nb);
  const int a = sorted[pos];
  float r[32];
  bool bad = false;
  if (a >= 0 && a < A) {
    const int row = bytoken ? token_of(a, kdiv) : a;
    const int8_t *src = aq + (int64_t)row * ld_aq + 32 * b;
    const uint4 lo = ldg_nc(src), hi = ldg_nc(src + 16);
    const float xs = as[(int64_t)row * ld_as + b];
    const uint32_t cw[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int t = 0; t < 4; ++t) r[4 * j + t] = __fmul_rn((float)(int)(int8_t)(cw[j] >> (8 * t)), xs);
    bad = !(fabsf(xs) <= 1.0e36f);  // NaN, infinity, or values that could overflow
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) r[j] = 0.0f;
  }
  const int64_t pstride = (int64_t)npos * (K / 2);
  uint8_t *dst = planes + (int64_t)pos * (K / 2) + 16 * b;
  uint8_t *sdst = bsc + (int64_t)pos * kPlanes * nb + b;
#pragma unroll 1
  for (int pl = 0; pl < kPlanes; ++pl) {
    float m = 0.0f;
#pragma unroll
    for (int j = 0; j < 32; ++j) m = fmaxf(m, fabsf(r[j]));
    uint4 word = make_uint4(0, 0, 0, 0);
    uint32_t ebyte = 127u;
    if (m > 0.0f) {
      const uint32_t mb = __float_as_uint(m);
      const int ef = (int)(mb >> 23);
      if (ef == 0) bad = true;  // a subnormal maximum: the scales would leave E8M0's normal range
      // m in [2^E, 2^(E+1)): s = 2^(E-2) when m <= 1.5 * 2^E, else 2^(E-1)
      int se = ef - 127 - 2 + ((mb & 0x7FFFFFu) > 0x400000u ? 1 : 0);
      if (se < -126 || se > 126) bad = true;
      se = se < -126 ? -126 : (se > 126 ? 126 : se);
      ebyte = (uint32_t)(se + 127);
      const float s = __uint_as_float((uint32_t)(se + 127) << 23);
      const float inv = __uint_as_float((uint32_t)(127 - se) << 23);
      uint32_t wv[4];
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        float t[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) t[e] = __fmul_rn(r[8 * w + e], inv);
        wv[w] = e2m1x8_from_f32(t);
        float d[8];
        e2m1x8_to_f32(wv[w], d);
#pragma unroll
        for (int e = 0; e < 8; ++e) r[8 * w + e] = __fmaf_rn(-d[e], s, r[8 * w + e]);
      }
      word = make_uint4(wv[0], wv[1], wv[2], wv[3]);
    }
    *reinterpret_cast<uint4 *>(dst + pl * pstride) = word;
    sdst[pl * nb] = (uint8_t)ebyte;
  }
  if (bad) atomicOr(bflag + pos, 1);
}

// The layer's exact value of one output (weight row wr of matrix m, activation
// row xr): acc = fma(I_b, xs_b * 2^(u_b - 128), acc) over the blocks in order.
MOE_DEVFN float exact_output(const TcArgs &p, int m, int64_t wr, int xr) {
  const int nb = p.K / 32;
  const uint8_t *w = (m == 0 ? p.w0 : p.w1) + wr * (p.K / 2);
  const uint8_t *sc = (m == 0 ? p.s0 : p.s1) + wr * nb;
  const int8_t *x = p.aq + (int64_t)xr * p.ld_aq;
  const float *xs = p.as + (int64_t)xr * p.ld_as;
  float acc = 0.0f;
#pragma unroll 1
  for (int b = 0; b < nb; ++b) {
    const uint4 wb = ldg_stream(w + 16 * b);
    const uint4 lo = ldg_nc(x + 32 * b), hi = ldg_nc(x + 32 * b + 16);
    const uint32_t ww[4] = {wb.x, wb.y, wb.z, wb.w};
    const uint32_t xw[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    int d = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t q0, q1;
      e2m1x8_to_off12(ww[j], q0, q1);
      d = __dp4a((int)xw[2 * j], (int)q0, d);
      d = __dp4a((int)xw[2 * j + 1], (int)q1, d);
    }
    const int I = d - 12 * block_sum8(lo, hi);
    acc = __fmaf_rn(__int2float_rn(I), __fmul_rn(xs[b], e8m0_half(sc[b])), acc);
  }
  return acc;
}

struct Tile {
  int e, mtile, ncols;
  int col0;  // first sorted position of the tile
};

template <int NT>
MOE_DEVFN Tile tile_of(const TcShared &S, const TcArgs &p, int t, int mt) {
  // expert: last e with prefix[e] <= t (binary search over E+1 entries)
  int lo = 0, hi = p.E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (S.prefix[mid] <= t) lo = mid;
    else hi = mid;
  }
  Tile tl;
  tl.e = lo;
  const int local = t - S.prefix[lo];
  tl.mtile = local % mt;
  const int ntile = local / mt;
  const int b = p.offsets[lo], n_e = p.offsets[lo + 1] - b;
  tl.col0 = b + ntile * NT;
  tl.ncols = min(NT, n_e - ntile * NT);
  return tl;
}

// Assignment of column c of a tile (-1: none; an entry past A is skipped and
// flagged), and its activation row (row 0 when there is none: a valid row
// whose results are never stored).
MOE_DEVFN int column_assignment(const TcArgs &p, const Tile &tl, int c, bool flag) {
  int a = -1;
  if (c < tl.ncols) {
    a = p.sorted[tl.col0 + c];
    if (a >= p.A) {
      if (flag && p.status) atomicOr(p.status, MOE_DEV_BAD_ROW);
      a = -1;
    }
  }
  return a;
}
MOE_DEVFN int column_row(const TcArgs &p, int a) { return a < 0 ? 0 : (p.bytoken ? token_of(a, p.kdiv) : a); }

template <int MODE, int NT>
__global__ void __launch_bounds__(kThreads, 1) tc_expert_kernel(const TcArgs p, const __grid_constant__ TcMaps maps) {
  constexpr int NM = MODE == kDownMode ? 1 : 2;
  constexpr int kN = kPlanes * NT;                      // MMA N: plane p's rows at [NT p, NT p + NT)
  constexpr uint32_t kBStage = kN * kStageK / 2;        // the planes of a stage
  constexpr int ND = (NM == 2 && NT == 32) ? 1 : 2;     // accumulator buffers
  constexpr int kSfbGroups = kN / 32;                   // 32-row groups of B (its scale columns)
  // per slot: A scales (4 columns per matrix and K-step pair), B scales (4
  // or 8 per pair: one per 32-row group of B)
  constexpr uint32_t kSfbCols = (kSfbGroups + 3) & ~3;
  constexpr uint32_t kSlotCols = 4u * (kSteps / 2) * NM + kSfbCols * (kSteps / 2);
  constexpr uint32_t kDBase = kTmemCols - (uint32_t)(ND * NM * kN);
  extern __shared__ __align__(1024) uint8_t smem_dyn[];
  const uint32_t dyn = smem_addr(smem_dyn);
  const uint32_t pad = ((dyn + 1023u) & ~1023u) - dyn;
  uint8_t *smem = smem_dyn + pad;
  const uint32_t sb = dyn + pad;
  TcShared &S = *reinterpret_cast<TcShared *>(smem + p.off_misc);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  const int K = p.K, nstg = K / kStageK, mt = p.N / kRows;
  const int NS = p.nstage;
  const uint32_t s_a = sb + p.off_a, s_b = sb + p.off_b;
  // K-step s's scales: bytes 2 (s & 1), + 1 of the pair's column
  auto sfa_col = [&](int slot, int s, int m) { return (uint32_t)slot * kSlotCols + 4u * (uint32_t)((s >> 1) * NM + m); };
  auto sfb_col = [&](int slot, int s) {
    return (uint32_t)slot * kSlotCols + 4u * (kSteps / 2) * NM + kSfbCols * (uint32_t)(s >> 1);
  };
  auto d_col = [&](int buf, int m) { return kDBase + (uint32_t)(buf * NM + m) * kN; };

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_addr(&S.a_full[s]), 1);
      mbar_init(smem_addr(&S.b_full[s]), kPrepWarps);
      mbar_init(smem_addr(&S.slot_free[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_addr(&S.d_full[b]), 1);
      mbar_init(smem_addr(&S.d_free[b]), kDrainWarps);
      mbar_init(smem_addr(&S.tab_full[b]), 1);
      mbar_init(smem_addr(&S.tab_empty[b]), kPrepWarps + kDrainWarps);
      mbar_init(smem_addr(&S.ext_full[b]), kPrepWarps);
    }
    fence_mbar_init();
  }
  if (warp == kWarpTab) {
    // tiles per expert, prefix-summed (every CTA derives the same list)
    int carry = 0;
    if (lane == 0) S.prefix[0] = 0;
    for (int e0 = 0; e0 < p.E; e0 += 32) {
      const int e = e0 + lane;
      int nt = 0;
      if (e < p.E) {
        const int b = p.offsets[e], en = p.offsets[e + 1];
        const bool bad = b < 0 || en < b || en > p.cap;
        if (bad && p.status) atomicOr(p.status, MOE_DEV_BAD_ROW);
        if (!bad && en - b > p.min_rows) nt = ((en - b + NT - 1) / NT) * mt;
      }
      int incl = nt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (e < p.E) S.prefix[e + 1] = carry + incl;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  if (warp == 0) tmem_alloc(smem_addr(&S.tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(&S.tmem_slot);
  const int ntiles = S.prefix[p.E];
  const int my_tiles = cta < ntiles ? (ntiles - cta + G - 1) / G : 0;

  if (warp < kDrainWarps) {
    // ------------------------------------------------ epilogue
    constexpr int kHalf = NT / 2;  // activation rows (columns) per epilogue warp
    const int q = warp & 3, h = warp >> 2;
    const uint32_t lanes = (uint32_t)(32 * q) << 16;
    const int r = 32 * q + lane;  // weight row of the tile = tensor-memory lane
    bool ok = true;
    for (int lt = 0; lt < my_tiles && ok; ++lt) {
      const int tb = lt & 1, ph = (lt >> 1) & 1;
      const int buf = lt % ND, bph = (lt / ND) & 1;
      ok = warp_wait(smem_addr(&S.tab_full[tb]), ph, p.status) &&
           __all_sync(0xffffffffu, mbar_wait_spin(smem_addr(&S.d_full[buf]), bph, p.status));
      if (!ok) break;
      tc_fence_after();
      const int ncols = S.ncols[tb];
      const int c0 = kHalf * h;  // this warp's first column
      float v[NM][kHalf];
      if (c0 < ncols) {
#pragma unroll
        for (int m = 0; m < NM; ++m) {
#pragma unroll
          for (int c8 = 0; c8 < kHalf; c8 += 8) {
            uint32_t d[kPlanes][8];
#pragma unroll
            for (int pl = 0; pl < kPlanes; ++pl)
              tmem_ld8_nowait(tmem + lanes + d_col(buf, m) + (uint32_t)(NT * pl + c0 + c8), d[pl]);
            tmem_ld_wait();
            // the planes' partial sums, smallest first
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              float s = __uint_as_float(d[kPlanes - 1][j]);
#pragma unroll
              for (int pl = kPlanes - 2; pl >= 0; --pl) s = __fadd_rn(s, __uint_as_float(d[pl][j]));
              v[m][c8 + j] = s;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&S.d_free[buf]));
      // the tile's weight-byte flags (complete once every stage was prepared)
      ok = warp_wait(smem_addr(&S.ext_full[tb]), ph, p.status);
      if (!ok) break;
      if (c0 < ncols) {
        const bool exta = S.ext[tb][q] != 0;
        const int64_t orow = (int64_t)S.mrow[tb] + r;
#pragma unroll
        for (int j = 0; j < kHalf; ++j) {
          const int c = c0 + j;
          const int a = c < ncols ? S.colasg[tb][c] : -1;
          if (a < 0) continue;
          float o[NM];
#pragma unroll
          for (int m = 0; m < NM; ++m) o[m] = v[m][j];
          if (exta || S.colext[tb][c] != 0) {
#pragma unroll 1
            for (int m = 0; m < NM; ++m) o[m] = exact_output(p, m, S.wrow[tb] + r, S.colrow[tb][c]);
          }
          if (MODE == kSwiglu) {
            p.out0[(int64_t)a * p.ld_out + orow] = __fmul_rn(silu(o[0]), o[NM - 1]);
          } else if (MODE == kRaw) {
            p.out0[(int64_t)a * p.ld_out + orow] = o[0];
            p.out1[(int64_t)a * p.ld_out + orow] = o[NM - 1];
          } else {
            p.out0[(int64_t)a * p.ld_out + orow] = o[0];
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&S.tab_empty[tb]));
    }
  } else if (warp < kWarpTma) {
    // ------------------------------------------------ A and B block scales
    const int q = warp & 3;
    const uint32_t lanes = (uint32_t)(32 * q) << 16;
    const int nbk = K / 32;
    bool ok = true;
    for (int lt = 0; lt < my_tiles && ok; ++lt) {
      const int tb = lt & 1;
      ok = warp_wait(smem_addr(&S.tab_full[tb]), (lt >> 1) & 1, p.status);
      if (!ok) break;
      const int64_t wrow = S.wrow[tb] + 32 * q + lane;  // this lane's weight row (A scales)
      // operand rows n = 32 c + lane of B (plane n / NT, column n % NT): their
      // scale bytes, in column group c of every quadrant
      const uint8_t *brow[kSfbGroups];
#pragma unroll
      for (int c = 0; c < kSfbGroups; ++c) {
        const int n = 32 * c + lane;
        brow[c] = p.bsc + ((int64_t)min(S.col0[tb] + n % NT, p.npos - 1) * kPlanes + n / NT) * nbk;
      }
      uint32_t outside = 0;
      // the scale bytes of a stage are requested kAhead stages before they
      // are stored, so their load latency overlaps the stages between
      constexpr int kAhead = NT == 16 ? 3 : 2;
      uint2 ra[kAhead][NM], rb[kAhead][kSfbGroups];
      auto load_scales = [&](int st, uint2 (&a)[NM], uint2 (&b)[kSfbGroups]) {
        if (st < nstg) {
#pragma unroll
          for (int m = 0; m < NM; ++m)
            a[m] = __ldg(reinterpret_cast<const uint2 *>((m == 0 ? p.s0 : p.s1) + wrow * nbk + st * 8));
#pragma unroll
          for (int c = 0; c < kSfbGroups; ++c) b[c] = __ldg(reinterpret_cast<const uint2 *>(brow[c] + st * 8));
        }
      };
#pragma unroll
      for (int i = 0; i < kAhead; ++i) load_scales(i, ra[i], rb[i]);
      for (int st = 0; st < nstg && ok; ++st) {
        const int g = lt * nstg + st, slot = g % NS;
        uint2 sfw[NM], bfw[kSfbGroups];
#pragma unroll
        for (int m = 0; m < NM; ++m) sfw[m] = ra[0][m];
#pragma unroll
        for (int c = 0; c < kSfbGroups; ++c) bfw[c] = rb[0][c];
#pragma unroll
        for (int i = 0; i + 1 < kAhead; ++i) {
#pragma unroll
          for (int m = 0; m < NM; ++m) ra[i][m] = ra[i + 1][m];
#pragma unroll
          for (int c = 0; c < kSfbGroups; ++c) rb[i][c] = rb[i + 1][c];
        }
        load_scales(st + kAhead, ra[kAhead - 1], rb[kAhead - 1]);
        if (g >= NS) {
          ok = warp_wait(smem_addr(&S.slot_free[slot]), ((g / NS) - 1) & 1, p.status);
          if (!ok) break;
        }
        tc_fence_after();
        // a word of four E8M0 bytes = the two blocks of K-steps 2 i and 2 i + 1
#pragma unroll
        for (int m = 0; m < NM; ++m) {
          outside |= outside_e8m0x4(sfw[m].x) | outside_e8m0x4(sfw[m].y);
          tmem_st1(tmem + lanes + sfa_col(slot, 0, m) + (uint32_t)q, clamp_e8m0x4(sfw[m].x));
          tmem_st1(tmem + lanes + sfa_col(slot, 2, m) + (uint32_t)q, clamp_e8m0x4(sfw[m].y));
        }
#pragma unroll
        for (int c = 0; c < kSfbGroups; ++c) {
          tmem_st1(tmem + lanes + sfb_col(slot, 0) + (uint32_t)c, bfw[c].x);
          tmem_st1(tmem + lanes + sfb_col(slot, 2) + (uint32_t)c, bfw[c].y);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&S.b_full[slot]));
      }
      if (!ok) break;
      const int any = __any_sync(0xffffffffu, outside != 0);
      if (lane == 0) {
        S.ext[tb][q] = any;
        mbar_arrive(smem_addr(&S.ext_full[tb]));
        mbar_arrive(smem_addr(&S.tab_empty[tb]));
      }
      __syncwarp();
    }
  } else if (warp == kWarpTma) {
    // ------------------------------------------------ tensor copies of the weights and planes
    if (lane == 0) {
      // weights are read once; the planes by every M-tile of their expert
      const uint64_t pol = policy_evict_first(), keep = policy_evict_last();
      bool ok = true;
      for (int lt = 0; lt < my_tiles && ok; ++lt) {
        const Tile tl = tile_of<NT>(S, p, cta + lt * G, mt);
        const int row0 = tl.e * p.N + tl.mtile * kRows;
        for (int st = 0; st < nstg; ++st) {
          const int g = lt * nstg + st, slot = g % NS;
          if (g >= NS && !mbar_wait(smem_addr(&S.slot_free[slot]), ((g / NS) - 1) & 1, p.status)) {
            ok = false;
            break;
          }
          const uint32_t bar = smem_addr(&S.a_full[slot]);
          mbar_arrive_expect_tx(bar, (uint32_t)NM * kAMat + kBStage);
#pragma unroll
          for (int m = 0; m < NM; ++m)
            tma_load_2d(s_a + (uint32_t)(slot * NM + m) * kAMat, &maps.w[m], st * (kStageK / 2), row0, bar, pol);
          // the tile's 16 sorted positions of each plane: operand rows 16 pl ..
#pragma unroll
          for (int pl = 0; pl < kPlanes; ++pl)
            tma_load_2d(s_b + (uint32_t)slot * kBStage + (uint32_t)pl * (NT * kStageK / 2), &maps.b,
                        st * (kStageK / 2), pl * p.npos + tl.col0, bar, keep);
        }
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ------------------------------------------------ MMA issue
    if (lane == 0) {
      const uint32_t idesc = idesc_mxf4(kRows, kN);
      const uint64_t adesc0 = smem_desc_sw128(s_a), bdesc0 = smem_desc_sw128(s_b);
      bool ok = true;
      for (int lt = 0; lt < my_tiles && ok; ++lt) {
        const int buf = lt % ND;
        if (lt >= ND && !mbar_wait_spin(smem_addr(&S.d_free[buf]), ((lt / ND) - 1) & 1, p.status)) break;
        tc_fence_after();
        for (int st = 0; st < nstg && ok; ++st) {
          const int g = lt * nstg + st, slot = g % NS;
          ok = mbar_wait_spin(smem_addr(&S.a_full[slot]), (g / NS) & 1, p.status) &&
               mbar_wait_spin(smem_addr(&S.b_full[slot]), (g / NS) & 1, p.status);
          if (!ok) break;
          // the planes arrived by cp.async (generic proxy): visible to the
          // tensor core's reads from here on
          fence_proxy_async();
          tc_fence_after();
          const uint64_t ad0 = adesc0 + (uint64_t)(((uint32_t)slot * NM * kAMat) >> 4);
          const uint64_t bd0 = bdesc0 + (uint64_t)(((uint32_t)slot * kBStage) >> 4);
#pragma unroll
          for (int s = 0; s < kSteps; ++s)
#pragma unroll
            for (int m = 0; m < NM; ++m)
              mma_mxf4(tmem + d_col(buf, m), ad0 + (uint64_t)((m * kAMat + 32u * s) >> 4), bd0 + (uint64_t)((32u * s) >> 4),
                       idesc_sf_ids(idesc, 2u * (s & 1), 2u * (s & 1)), tmem + sfa_col(slot, s, m),
                       tmem + sfb_col(slot, s), st > 0 || s > 0);
          mma_commit(smem_addr(&S.slot_free[slot]));
        }
        if (ok) mma_commit(smem_addr(&S.d_full[buf]));
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ column tables, one tile ahead
    for (int lt = 0; lt < my_tiles; ++lt) {
      const Tile tl = tile_of<NT>(S, p, cta + lt * G, mt);
      const int tb = lt & 1;
      if (lt >= 2 && !warp_wait(smem_addr(&S.tab_empty[tb]), ((lt >> 1) - 1) & 1, p.status)) break;
      if (lane < NT) {
        const int a = column_assignment(p, tl, lane, true);
        const int row = column_row(p, a);
        S.colasg[tb][lane] = a;
        S.colrow[tb][lane] = row;
        S.colext[tb][lane] = a >= 0 ? p.bflag[tl.col0 + lane] : 0;
      }
      if (lane == 0) {
        S.ncols[tb] = tl.ncols;
        S.mrow[tb] = tl.mtile * kRows;
        S.wrow[tb] = (int64_t)tl.e * p.N + tl.mtile * kRows;
        S.col0[tb] = tl.col0;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&S.tab_full[tb]));
    }
  }
  // every MMA of this CTA has completed (the epilogue waited for the last one)
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// Packed weights [rows][cols bytes] as a 2-D tensor map with boxes of 128
// bytes x 128 rows, 128-byte swizzled.
bool encode_rows(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {128u, (cuuint32_t)kRows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The activation planes [rows][cols bytes] as a 2-D tensor map with boxes of
// 128 bytes x nt rows (one plane's rows of a tile), 128-byte swizzled.
bool encode_planes(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, int nt) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {128u, (cuuint32_t)nt};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Stream-ordered scratch for the activation planes: one memory pool per
// device that keeps its memory between calls (a call allocates and frees on
// its stream, so calls on different streams never share a buffer).
cudaMemPool_t scratch_pool(int dev) {
  static std::mutex mu;
  static std::map<int, cudaMemPool_t> pools;
  std::lock_guard<std::mutex> lock(mu);
  auto it = pools.find(dev);
  if (it != pools.end()) return it->second;
  cudaMemPoolProps props{};
  props.allocType = cudaMemAllocationTypePinned;
  props.location.type = cudaMemLocationTypeDevice;
  props.location.id = dev;
  cudaMemPool_t pool = nullptr;
  if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) return nullptr;
  uint64_t keep = ~0ull;
  cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
  pools[dev] = pool;
  return pool;
}

}  // namespace

bool tc_expert_supported(int K, int N) { return K % kStageK == 0 && K <= 8192 && N % kRows == 0; }

// Launch of the tensor-core path (moe_mxfp4_gateup_swiglu, moe_mxfp4_gateup
// and moe_mxfp4_down for T > 16) over the experts with more than min_rows
// rows.  mode 0: gate and up with SwiGLU into out0; 1: gate into out0, up
// into out1; 2: down into out0.
moe_status launch_tc_expert(int mode, const int8_t *aq, int64_t ld_aq, const float *as, int64_t ld_as,
                            const uint8_t *w0, const uint8_t *s0, const uint8_t *w1, const uint8_t *s1,
                            const int32_t *offsets, const int32_t *sorted, int64_t cap, int A, int k, int E, int K,
                            int N, int bytoken, int min_rows, float *out0, float *out1, int64_t ld_out,
                            cudaStream_t stream, const char *name) {
  if (!tc_expert_supported(K, N))
    return fail(MOE_ERR_UNSUPPORTED, "%s: tensor path needs K %% 256 == 0 (<= 8192) and rows %% 128 == 0", name);
  if (E > 4096) return fail(MOE_ERR_UNSUPPORTED, "%s: E=%d", name, E);
  if ((uintptr_t)s0 % 8 || (mode != kDownMode && (uintptr_t)s1 % 8))
    return fail(MOE_ERR_INVALID_ARG, "%s: the tensor path needs 8-byte aligned scale bytes", name);
  const int nm = mode == kDownMode ? 1 : 2;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_fail(err, name);
  int optin = 0;
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  const int npos = (int)cap;  // sorted positions (the planes are written by position)
  const int nb = K / 32;
  TcArgs p{};
  p.aq = aq; p.ld_aq = ld_aq; p.as = as; p.ld_as = ld_as;
  p.w0 = w0; p.w1 = w1; p.s0 = s0; p.s1 = s1;
  p.offsets = offsets; p.sorted = sorted; p.cap = cap;
  p.A = A; p.k = k; p.E = E; p.K = K; p.N = N; p.bytoken = bytoken; p.min_rows = min_rows < 0 ? 0 : min_rows;
  p.kdiv = kdiv_of(k);
  p.npos = npos;
  p.out0 = out0; p.out1 = out1; p.ld_out = ld_out;
  p.status = device_status_word();
  TcMaps maps{};
  const uint64_t wrows = (uint64_t)E * N;
  for (int m = 0; m < nm; ++m) {
    if (!encode_rows(&maps.w[m], m == 0 ? w0 : w1, wrows, (uint64_t)K / 2))
      return fail(MOE_ERR_UNSUPPORTED, "%s: tensor maps of the weights could not be built (16-byte aligned weights are required)", name);
  }
  // token tiles of 32 rows when the experts average many rows (fewer weight
  // reads from shared memory per row; gate/up then has one accumulator
  // buffer), else of 16 rows
  const int nt = (int64_t)A >= 48ll * E ? 32 : 16;
  const int kn = kPlanes * nt;
  const int nd = (nm == 2 && nt == 32) ? 1 : 2;
  const uint32_t bstage = (uint32_t)kn * kStageK / 2;
  // tensor memory: per stage slot 4 columns per matrix and K-step pair (A
  // scales) and 4 or 8 per pair (B scales); the accumulator buffers at the top
  const uint32_t slot_cols = 4u * (kSteps / 2) * (uint32_t)nm + ((uint32_t)(kn / 32 + 3) & ~3u) * (kSteps / 2);
  const int ns_tmem = (int)((kTmemCols - (uint32_t)(nd * nm * kn)) / slot_cols);
  // shared memory: the stage ring (packed weights, planes), then the small state
  const uint32_t stage = (uint32_t)nm * kAMat + bstage;
  const size_t fixed = (size_t)tc_shared_bytes(E) + 1024u + 64u;
  int ns = (int)(((size_t)optin - fixed) / stage);
  if (ns > kMaxStages) ns = kMaxStages;
  if (ns > ns_tmem) ns = ns_tmem;
  if (ns < 2) return fail(MOE_ERR_UNSUPPORTED, "%s: tensor path does not fit shared memory", name);
  p.nstage = ns;
  p.off_a = 0;  // 1024-aligned (swizzled copies)
  p.off_b = (uint32_t)ns * nm * kAMat;
  p.off_misc = (p.off_b + (uint32_t)ns * bstage + 63u) & ~63u;
  const size_t smem = (size_t)p.off_misc + tc_shared_bytes(E) + 1024u;  // + alignment of the base
  if (smem > (size_t)optin) return fail(MOE_ERR_UNSUPPORTED, "%s: tensor path needs %zu bytes of shared memory", name, smem);
  auto kern = nt == 32 ? (mode == kSwiglu ? tc_expert_kernel<kSwiglu, 32>
                                           : mode == kRaw ? tc_expert_kernel<kRaw, 32> : tc_expert_kernel<kDownMode, 32>)
                       : (mode == kSwiglu ? tc_expert_kernel<kSwiglu, 16>
                                          : mode == kRaw ? tc_expert_kernel<kRaw, 16> : tc_expert_kernel<kDownMode, 16>);
  const moe_status ast = ensure_smem_attr(reinterpret_cast<const void *>(kern), optin, name);
  if (ast != MOE_OK) return ast;

  // the planes of every sorted position (stream-ordered scratch)
  const size_t plane_bytes = (size_t)kPlanes * npos * (K / 2);
  const size_t bsc_bytes = ((size_t)npos * kPlanes * nb + 255) & ~(size_t)255;
  const size_t scratch = plane_bytes + bsc_bytes + (size_t)npos * 4;
  cudaMemPool_t pool = scratch_pool(dev);
  if (!pool) return fail(MOE_ERR_CUDA, "%s: no memory pool for the activation planes", name);
  void *buf = nullptr;
  err = cudaMallocFromPoolAsync(&buf, scratch, pool, stream);
  if (err != cudaSuccess) return cuda_fail(err, name);
  uint8_t *planes = static_cast<uint8_t *>(buf);
  p.bsc = planes + plane_bytes;
  p.bflag = reinterpret_cast<const int *>(planes + plane_bytes + bsc_bytes);
  if (!encode_planes(&maps.b, planes, (uint64_t)kPlanes * npos, (uint64_t)K / 2, nt)) {
    cudaFreeAsync(buf, stream);
    return fail(MOE_ERR_UNSUPPORTED, "%s: tensor map of the activation planes could not be built", name);
  }
  err = cudaMemsetAsync(planes + plane_bytes + bsc_bytes, 0, (size_t)npos * 4, stream);
  if (err == cudaSuccess) {
    const int64_t nthreads = (int64_t)npos * nb;
    plane_kernel<<<(unsigned)((nthreads + 255) / 256), 256, 0, stream>>>(
        aq, ld_aq, as, ld_as, sorted, npos, A, bytoken, p.kdiv, K, planes, planes + plane_bytes,
        const_cast<int *>(p.bflag));
    err = cudaGetLastError();
  }
  if (err == cudaSuccess) {
    kern<<<sm_count(), kThreads, smem, stream>>>(p, maps);
    err = cudaGetLastError();
  }
  const cudaError_t ferr = cudaFreeAsync(buf, stream);
  if (err != cudaSuccess) return cuda_fail(err, name);
  return ferr == cudaSuccess ? MOE_OK : cuda_fail(ferr, name);
}

}  // namespace moe
