// Tensor-core (tcgen05) path of the MXFP4 expert projections, used by the
// stage calls for the experts with more than 4 rows in batches of more than
// 16 rows (prefill and large decode batches; the 1-16-row decode regime and
// the light experts keep the CUDA-core kernels).
//
// The layer's projections as grouped GEMMs over the rows routed to each
// expert: "DeepSeek-V4-Flash on AMD gfx90a", §6.1 (packed FP4 weights with
// E8M0 block scales against INT8 per-32 activations: an exact integer dot
// per block of 32, then activation and E8M0 scaling) and "Optimizing
// DeepSeek V4 Flash Inference on a Strix Halo Pair", "MXFP4 routed-expert
// kernels" (prefill tiles over the tokens of one expert).
//
// Every block dot is exact, as in the CUDA-core kernels.  The tensor core
// takes the weights as they are stored: E2M1 nibbles (kind::mxf4, K = 64 per
// MMA = two MX blocks) with the weight's E8M0 byte u as the block scale of A,
// clamped to uc = min(max(u, 64), 192) so that every partial sum of the MMA
// is an exact normal fp32 number; the drain multiplies the activation scale
// by the remainder 2^(u - uc) (NaN for byte 255) when a byte lies outside
// that range (no real checkpoint has one; the multiply is skipped when all 32
// rows of a warp are inside it).
// The Q8 codes q of the activations are not an MMA type, so each is written
// as three signed base-8 digits q = d0 + 8 d1 + 64 d2, d0, d1 in {-4..3} and
// d2 in {-2..2} (every q in [-128, 127] has this form), each an exact E2M1
// value; plane i is an MMA operand with block scale 8^i.  The three plane
// MMAs sum into one fp32 accumulator:  D = 2^(u-127) * sum_k v_k q_k =
// I_b 2^(u-128) with I_b the integer block dot of twice the E2M1 values;
// every partial sum is a multiple of 2^(uc-128) below 2^(uc-110), exact in
// fp32 (uc = u inside the clamp range).  Every MMA accumulates (a block-scaled MMA that overwrites its
// accumulator costs several times one that adds to it); the drain sets each
// accumulator buffer back to zero after reading it.  To keep the
// two blocks of a K-step apart, the B operand has two rows per activation
// row: rows [0, 32) carry the even block of each K-step (zeros in the odd
// one), rows [32, 64) the odd block.  The epilogue of each K-step ("drain")
// then forms  acc = fma(D, xs_b * 2^(u-uc), acc)  per (weight row,
// activation row, block), which equals the CUDA-core term
// fma(I_b, xs_b * 2^(u-128), acc): the same exact product, one rounding
// (both scale products are exact whenever they are normal numbers).  Blocks are accumulated in
// increasing order; the CUDA-core kernels add per-lane partial sums in a
// butterfly instead, so the two paths agree within fp32 rounding, not bit
// for bit.
//
// Tiles: 128 weight rows (MMA M) x up to 32 activation rows of one expert
// (MMA N = 64), K in stages of 256 (8 blocks, 4 K-steps).  One persistent CTA
// per SM walks the tiles it derives from the expert offsets:
//   warps 0-7   drain: TMEM lane quadrant warp % 4, 16 activation rows each;
//               fp32 accumulators in registers, epilogue (SwiGLU) and store
//   warps 8-11  per stage: the digit planes of the stage's activation codes
//               into shared memory (a 256-entry table per nibble position),
//               the stage's activation scales, and the A block scales
//               (E8M0 bytes of the weight rows) into tensor memory
//   warp 12     tensor copies (TMA) of the packed weights, 128-byte swizzled
//   warp 13     MMA issue
//   warp 14     column tables of the next tile
// Tensor memory: B scales (3 planes), a ring of A scales per stage slot, and
// 3 (gate/up) or 6 (down) K-step accumulator buffers of 64 columns per matrix.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "mx_device.cuh"
#include "tc_device.cuh"

namespace moe {
namespace {

constexpr int kRows = 128;                     // weight rows per tile (MMA M)
constexpr int kNT = 32;                        // activation rows per tile, at most
constexpr int kN = 2 * kNT;                    // MMA N: even-block rows, then odd-block rows
constexpr int kStageK = 256;                   // reduction elements per stage (8 MX blocks)
constexpr int kSteps = kStageK / 64;           // MMA K-steps per stage
constexpr int kPlanes = 3;                     // base-8 digit planes of the Q8 codes
constexpr uint32_t kAMat = kRows * kStageK / 2;  // one matrix's packed weights per stage (16 KB)
constexpr uint32_t kBPlane = kN * kStageK / 2;   // one digit plane per stage (8 KB)
constexpr uint32_t kBStage = kPlanes * kBPlane;  // 24 KB
constexpr uint32_t kXsStage = kNT * 8 * 4;       // activation scales of a stage (1 KB)
constexpr int kDrainWarps = 8;
constexpr int kPrepWarps = 4;
constexpr int kWarpTma = kDrainWarps + kPrepWarps;
constexpr int kWarpMma = kWarpTma + 1;
constexpr int kWarpTab = kWarpMma + 1;
constexpr int kThreads = 32 * (kWarpTab + 1);
constexpr int kMaxStages = 4;
constexpr int kMaxDBuf = 8;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfaBase = 16;   // columns [0, 12): B scales, plane i at 4 i
constexpr uint32_t kDBase = 128;    // first accumulator column
constexpr uint32_t kUcLo = 0x40404040u;  // E8M0 bytes given to the MMA: clamped to [64, 192]
constexpr uint32_t kUcHi = 0xC0C0C0C0u;

// Four E8M0 bytes clamped to the MMA's range.
MOE_DEVFN uint32_t clamp_e8m0x4(uint32_t w) { return __vmaxu4(__vminu4(w, kUcHi), kUcLo); }
// Non-zero when one of four E8M0 bytes lies outside the MMA's range.
MOE_DEVFN uint32_t outside_e8m0x4(uint32_t w) { return __vcmpltu4(w, kUcLo) | __vcmpgtu4(w, kUcHi); }
// 2^(u - uc) for an E8M0 byte u and its clamped value uc (exact; NaN for 255).
MOE_DEVFN float e8m0_remainder(uint32_t u) {
  const uint32_t uc = u < 64u ? 64u : (u > 192u ? 192u : u);
  return u == 255u ? __uint_as_float(0x7FC00000u) : __uint_as_float((127u + u - uc) << 23);
}

enum Mode { kSwiglu = 0, kRaw = 1, kDownMode = 2 };

struct TcArgs {
  const int8_t *aq;  // Q8 activation codes: x rows (gate/up, by token) or h rows (down, by assignment)
  int64_t ld_aq;
  const float *as;
  int64_t ld_as;
  const uint8_t *s0, *s1;  // E8M0 bytes of the weight rows, [E*N][K/32]
  const int32_t *offsets, *sorted;
  int64_t cap;
  int A, k, E, K, N;  // K reduction length, N output rows per expert
  int bytoken;        // activation row of assignment a: a / k (1) or a (0)
  int min_rows;       // experts with at most this many rows are left to the CUDA-core kernel
  uint32_t kdiv;
  float *out0, *out1;
  int64_t ld_out;
  unsigned *status;
  int nstage, ndbuf;
  uint32_t off_a, off_b, off_xs, off_misc;  // shared memory (from the 1024-aligned base)
};

struct TcMaps {  // 2-D tensor maps (TMA) of the packed weights
  CUtensorMap w[2];
};

struct TcShared {
  uint64_t a_full[kMaxStages], b_full[kMaxStages], slot_free[kMaxStages];
  uint64_t d_full[kMaxDBuf], d_free[kMaxDBuf];
  uint64_t tab_full[2], tab_empty[2];
  uint32_t tmem_slot;
  int ncols[2];
  int mrow[2];        // first output row of the tile within its expert
  int64_t wrow[2];    // first weight row of the tile (expert * N + mrow)
  int colrow[2][kNT]; // activation row of each column (-1: none)
  int colasg[2][kNT]; // output row (assignment) of each column (-1: none)
  uint32_t lut[2][256];  // Q8 code -> its four digit codes, low / high nibble of byte i = plane i
  int ext[kMaxStages][4];  // per stage slot and lane quadrant: an E8M0 byte outside the MMA's clamp range
  int prefix[1];         // [E + 1] tiles before expert e
};

uint32_t tc_shared_bytes(int E) { return (uint32_t)(sizeof(TcShared) + 4u * (uint32_t)E); }

MOE_DEVFN void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

MOE_DEVFN void tmem_ld16_nowait(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
MOE_DEVFN void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Bounded mbarrier wait without back-off sleeps, for the short hand-offs of
// the MMA thread and the drain (try_wait itself suspends the thread for a
// while); gives up after 2^22 polls.
MOE_DEVFN bool mbar_wait_spin(uint32_t bar, uint32_t parity, unsigned *status) {
  for (uint32_t i = 0; i < (1u << 22); ++i)
    if (mbar_try_wait(bar, parity)) return true;
  if (status) atomicOr(status, MOE_DEV_WAIT_TIMEOUT);
  return false;
}

// Bounded mbarrier wait taken by a whole warp, with one answer for all lanes.
MOE_DEVFN bool warp_wait(uint32_t bar, uint32_t parity, unsigned *status) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, status));
}

// 2-D tensor copy of one box into shared memory, completing on bar.
MOE_DEVFN void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Base-8 digits of a Q8 code (as its byte): q = d0 + 8 d1 + 64 d2 with d0,
// d1 in {-4..3} and d2 in {-2..2}; digit codes are E2M1 (0 -> 0, 1 -> 0x2,
// 2 -> 0x4, 3 -> 0x5, 4 -> 0x6, sign bit 0x8).  Returns the three codes,
// plane i in nibble i.
MOE_DEVFN uint32_t digit_codes(int q) {
  uint32_t codes = 0;
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    const int d = i < 2 ? ((q + 4) & 7) - 4 : q;  // q is in [-2, 2] for the last digit
    const int a = d < 0 ? -d : d;
    const uint32_t mag = a == 0 ? 0u : a == 1 ? 2u : a == 2 ? 4u : a == 3 ? 5u : 6u;
    codes |= (mag | (d < 0 ? 8u : 0u)) << (4 * i);
    q = (q - d) >> 3;  // exact: q - d is a multiple of 8
  }
  return codes;
}

// Byte offset of (row r, byte j) of a no-swizzle K-major operand with 128-byte
// rows: core matrices of 8 rows x 16 bytes, 128 bytes apart along K, 8-row
// groups 1024 bytes apart.
MOE_DEVFN uint32_t bofs(int r, int j) {
  return (uint32_t)(r >> 3) * 1024u + (uint32_t)(j >> 4) * 128u + (uint32_t)(r & 7) * 16u + (uint32_t)(j & 15);
}

struct Tile {
  int e, mtile, ncols;
  int col0;  // first sorted position of the tile
};

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
  tl.col0 = b + ntile * kNT;
  tl.ncols = min(kNT, n_e - ntile * kNT);
  return tl;
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) tc_expert_kernel(const TcArgs p, const __grid_constant__ TcMaps maps) {
  constexpr int NM = MODE == kDownMode ? 1 : 2;
  extern __shared__ __align__(1024) uint8_t smem_dyn[];
  const uint32_t dyn = smem_addr(smem_dyn);
  const uint32_t pad = ((dyn + 1023u) & ~1023u) - dyn;
  uint8_t *smem = smem_dyn + pad;
  const uint32_t sb = dyn + pad;
  TcShared &S = *reinterpret_cast<TcShared *>(smem + p.off_misc);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  const int K = p.K, nstg = K / kStageK, mt = p.N / kRows;
  const int NS = p.nstage, ND = p.ndbuf;
  const uint32_t s_a = sb + p.off_a, s_b = sb + p.off_b, s_xs = sb + p.off_xs;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_addr(&S.a_full[s]), 1);
      mbar_init(smem_addr(&S.b_full[s]), kPrepWarps);
      mbar_init(smem_addr(&S.slot_free[s]), 1 + kDrainWarps);
    }
    for (int b = 0; b < ND; ++b) {
      mbar_init(smem_addr(&S.d_full[b]), 1);
      mbar_init(smem_addr(&S.d_free[b]), kDrainWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_addr(&S.tab_full[b]), 1);
      mbar_init(smem_addr(&S.tab_empty[b]), kPrepWarps + kDrainWarps);
    }
    fence_mbar_init();
  }
  // digit tables, and zeros in the operand halves that no stage ever writes
  for (int i = tid; i < 256; i += kThreads) {
    const uint32_t c = digit_codes((int)(int8_t)i);
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int pl = 0; pl < kPlanes; ++pl) {
      const uint32_t d = (c >> (4 * pl)) & 0xFu;
      lo |= d << (8 * pl);
      hi |= d << (8 * pl + 4);
    }
    S.lut[0][i] = lo;
    S.lut[1][i] = hi;
  }
  for (uint32_t o = 16u * tid; o < (uint32_t)NS * kBStage; o += 16u * kThreads) sts128(s_b + o, make_uint4(0, 0, 0, 0));
  fence_proxy_async();
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
        if (!bad && en - b > p.min_rows) nt = ((en - b + kNT - 1) / kNT) * mt;
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
  if (warp < 4) {
    // B block scales: plane i = 8^i for both blocks of a K-step, every lane
    const uint32_t lanes = (uint32_t)(32 * warp) << 16;
#pragma unroll
    for (int pl = 0; pl < kPlanes; ++pl)
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_st1(tmem + lanes + 4u * pl + c, 0x01010101u * (127u + 3u * pl));
    // every accumulator column starts at zero (the MMAs only add)
    const uint32_t zero[32] = {};
    for (uint32_t c = kDBase; c < kTmemCols; c += 32) tmem_st32(tmem + lanes + c, zero);
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int ntiles = S.prefix[p.E];
  const int my_tiles = cta < ntiles ? (ntiles - cta + G - 1) / G : 0;

  if (warp < kDrainWarps) {
    // ------------------------------------------------ drain + epilogue
    const int q = warp & 3, h = warp >> 2;
    const uint32_t lanes = (uint32_t)(32 * q) << 16;
    const int r = 32 * q + lane;  // weight row of the tile = TMEM lane
    bool ok = true;
    for (int lt = 0; lt < my_tiles && ok; ++lt) {
      const int tb = lt & 1;
      ok = warp_wait(smem_addr(&S.tab_full[tb]), (lt >> 1) & 1, p.status);
      if (!ok) break;
      const int ncols = S.ncols[tb];
      const bool active = 16 * h < ncols;
      float acc[NM][16];
#pragma unroll
      for (int m = 0; m < NM; ++m)
#pragma unroll
        for (int c = 0; c < 16; ++c) acc[m][c] = 0.0f;
      for (int st = 0; st < nstg && ok; ++st) {
        const int g = lt * nstg + st, slot = g % NS;
        const uint32_t xsb = s_xs + (uint32_t)slot * kXsStage;
        // the stage's activation scales are in place (the phase cannot move
        // on before this warp releases the slot)
        ok = warp_wait(smem_addr(&S.b_full[slot]), (g / NS) & 1, p.status);
        if (!ok) break;
        // the MMA saw the E8M0 bytes of this quadrant's rows clamped; if one
        // lay outside the clamp range, the remainders are applied (the two
        // bytes of each K-step are read again for that)
        const bool ext = S.ext[slot][q] != 0;
        for (int s = 0; s < kSteps; ++s) {
          const int j = g * kSteps + s, db = j % ND;
          ok = __all_sync(0xffffffffu, mbar_wait_spin(smem_addr(&S.d_full[db]), (j / ND) & 1, p.status));
          if (!ok) break;
          tc_fence_after();
          if (active) {
            const uint32_t dcol = tmem + lanes + kDBase + (uint32_t)db * NM * kN + 16u * h;
            if (!ext) {
              uint32_t de[NM][16], dd[NM][16];
#pragma unroll
              for (int m = 0; m < NM; ++m) {
                tmem_ld16_nowait(dcol + (uint32_t)m * kN, de[m]);
                tmem_ld16_nowait(dcol + (uint32_t)m * kN + kNT, dd[m]);
              }
              // scales of blocks 8 st + 2 s and + 1 of columns 16 h .. 16 h + 15
              float x0[16], x1[16];
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                const uint4 a = lds128(xsb + (uint32_t)((2 * s) * kNT + 16 * h + 4 * v) * 4u);
                const uint4 b = lds128(xsb + (uint32_t)((2 * s + 1) * kNT + 16 * h + 4 * v) * 4u);
                x0[4 * v] = __uint_as_float(a.x); x0[4 * v + 1] = __uint_as_float(a.y);
                x0[4 * v + 2] = __uint_as_float(a.z); x0[4 * v + 3] = __uint_as_float(a.w);
                x1[4 * v] = __uint_as_float(b.x); x1[4 * v + 1] = __uint_as_float(b.y);
                x1[4 * v + 2] = __uint_as_float(b.z); x1[4 * v + 3] = __uint_as_float(b.w);
              }
              tmem_ld_wait();
#pragma unroll
              for (int c = 0; c < 16; ++c) {
#pragma unroll
                for (int m = 0; m < NM; ++m) {
                  acc[m][c] = __fmaf_rn(__uint_as_float(de[m][c]), x0[c], acc[m][c]);
                  acc[m][c] = __fmaf_rn(__uint_as_float(dd[m][c]), x1[c], acc[m][c]);
                }
              }
            } else {
              // a byte of this quadrant's rows lay outside the MMA's clamp
              // range: D = I_b 2^(uc-128) times xs 2^(u-uc), one matrix and
              // one block at a time (the activation scales read again from
              // shared memory, so this rare path needs few registers)
#pragma unroll
              for (int m = 0; m < NM; ++m) {
                const int64_t sb = (S.wrow[tb] + r) * (int64_t)(K / 32) + st * 8 + 2 * s;
                const uint32_t w2 = __ldg(reinterpret_cast<const unsigned short *>((m == 0 ? p.s0 : p.s1) + sb));
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                  const float f = e8m0_remainder((w2 >> (8 * half)) & 0xFFu);
                  uint32_t d[16];
                  tmem_ld16_nowait(dcol + (uint32_t)(m * kN + half * kNT), d);
                  tmem_ld_wait();
                  const uint32_t xrow = xsb + (uint32_t)((2 * s + half) * kNT + 16 * h) * 4u;
#pragma unroll
                  for (int c = 0; c < 16; ++c)
                    acc[m][c] = __fmaf_rn(__uint_as_float(d[c]), __fmul_rn(lds_f32(xrow + 4u * c), f), acc[m][c]);
                }
              }
            }
          }
          {
            // back to zero for the MMAs that add into this buffer next
            const uint32_t zero[16] = {};
            const uint32_t dz = tmem + lanes + kDBase + (uint32_t)db * NM * kN + 16u * h;
#pragma unroll
            for (int m = 0; m < NM; ++m) {
              tmem_st16(dz + (uint32_t)m * kN, zero);
              tmem_st16(dz + (uint32_t)m * kN + kNT, zero);
            }
            tmem_st_wait();
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(&S.d_free[db]));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&S.slot_free[slot]));
      }
      if (ok && active) {
        const int64_t orow = (int64_t)S.mrow[tb] + r;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int col = 16 * h + c;
          const int a = col < ncols ? S.colasg[tb][col] : -1;
          if (a >= 0) {
            if (MODE == kSwiglu) p.out0[(int64_t)a * p.ld_out + orow] = __fmul_rn(silu(acc[0][c]), acc[NM - 1][c]);
            else if (MODE == kRaw) {
              p.out0[(int64_t)a * p.ld_out + orow] = acc[0][c];
              p.out1[(int64_t)a * p.ld_out + orow] = acc[NM - 1][c];
            } else {
              p.out0[(int64_t)a * p.ld_out + orow] = acc[0][c];
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&S.tab_empty[tb]));
    }
  } else if (warp < kWarpTma) {
    // ------------------------------------------------ digit planes, activation scales, A scales
    const int q = warp & 3;
    const uint32_t lanes = (uint32_t)(32 * q) << 16;
    const int tp = tid - 32 * kDrainWarps;  // 0 .. 127
    const int jb = tp >> 4;                 // block of the stage this thread converts
    // (lanes of an 8-lane phase take 8 consecutive rows of one block: their
    // 16-byte plane stores fall in 8 distinct bank groups)
    const int nbk = K / 32;
    bool ok = true;
    for (int lt = 0; lt < my_tiles && ok; ++lt) {
      const int tb = lt & 1;
      ok = warp_wait(smem_addr(&S.tab_full[tb]), (lt >> 1) & 1, p.status);
      if (!ok) break;
      const int ncols = S.ncols[tb];
      const int64_t wrow = S.wrow[tb] + 32 * q + lane;  // this lane's weight row (A scales)
      int crow[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int c = (tp & 15) + 16 * u;
        crow[u] = c < ncols ? S.colrow[tb][c] : -1;
      }
      // a stage's codes and scales are loaded one stage ahead, so their
      // latency overlaps the conversion of the stage before
      uint4 code[2][2];
      float xsv[2];
      uint2 sfw[NM];
      auto load_stage = [&](int st, uint4 (&cd)[2][2], float (&xv)[2], uint2 (&sf)[NM]) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          if (crow[u] >= 0 && st < nstg) {
            const int8_t *src = p.aq + (int64_t)crow[u] * p.ld_aq + st * kStageK + 32 * jb;
            cd[u][0] = ldg_nc(src);
            cd[u][1] = ldg_nc(src + 16);
            xv[u] = __ldg(p.as + (int64_t)crow[u] * p.ld_as + st * 8 + jb);
          } else {
            cd[u][0] = cd[u][1] = make_uint4(0, 0, 0, 0);
            xv[u] = 0.0f;
          }
        }
#pragma unroll
        for (int m = 0; m < NM; ++m)
          sf[m] = st < nstg ? __ldg(reinterpret_cast<const uint2 *>((m == 0 ? p.s0 : p.s1) + wrow * nbk + st * 8))
                            : make_uint2(0, 0);
      };
      load_stage(0, code, xsv, sfw);
      for (int st = 0; st < nstg && ok; ++st) {
        const int g = lt * nstg + st, slot = g % NS;
        uint4 ncode[2][2];
        float nxsv[2];
        uint2 nsfw[NM];
        load_stage(st + 1, ncode, nxsv, nsfw);
        if (g >= NS) {
          ok = warp_wait(smem_addr(&S.slot_free[slot]), ((g / NS) - 1) & 1, p.status);
          if (!ok) break;
        }
        tc_fence_after();
        const uint32_t bst = s_b + (uint32_t)slot * kBStage;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int c = (tp & 15) + 16 * u;
          if (crow[u] < 0) continue;
          // 16 code pairs -> 16 words, byte i = plane i's byte of the pair
          const uint32_t cw[8] = {code[u][0].x, code[u][0].y, code[u][0].z, code[u][0].w,
                                  code[u][1].x, code[u][1].y, code[u][1].z, code[u][1].w};
          uint32_t pw[4][4];  // [plane][word of 4 pairs]
#pragma unroll
          for (int g4 = 0; g4 < 4; ++g4) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t v = cw[2 * g4 + (i >> 1)];
              const int sh = 16 * (i & 1);
              w[i] = S.lut[0][(v >> sh) & 0xFFu] | S.lut[1][(v >> (sh + 8)) & 0xFFu];
            }
            const uint32_t t0 = prmt(w[0], w[1], 0x5140u), t1 = prmt(w[0], w[1], 0x7362u);
            const uint32_t t2 = prmt(w[2], w[3], 0x5140u), t3 = prmt(w[2], w[3], 0x7362u);
            pw[0][g4] = prmt(t0, t2, 0x5410u);
            pw[1][g4] = prmt(t0, t2, 0x7632u);
            pw[2][g4] = prmt(t1, t3, 0x5410u);
            pw[3][g4] = prmt(t1, t3, 0x7632u);
          }
          const int brow = (jb & 1) ? kNT + c : c;  // odd blocks go to the second half of the rows
          const uint32_t off = bofs(brow, 16 * jb);
#pragma unroll
          for (int pl = 0; pl < kPlanes; ++pl)
            sts128(bst + (uint32_t)pl * kBPlane + off, make_uint4(pw[pl][0], pw[pl][1], pw[pl][2], pw[pl][3]));
          sts32(s_xs + (uint32_t)slot * kXsStage + (uint32_t)(jb * kNT + c) * 4u, __float_as_uint(xsv[u]));
        }
        // does one of this quadrant's rows hold an E8M0 byte outside the
        // MMA's clamp range in this stage?
        {
          uint32_t outside = 0;
#pragma unroll
          for (int m = 0; m < NM; ++m) outside |= outside_e8m0x4(sfw[m].x) | outside_e8m0x4(sfw[m].y);
          const int any = __any_sync(0xffffffffu, outside != 0);
          if (lane == 0) S.ext[slot][q] = any;
        }
        // A block scales of the stage: K-step s of matrix m at columns
        // kSfaBase + 4 (slot-local index) + quadrant, bytes 0 / 1 = its two blocks
#pragma unroll
        for (int m = 0; m < NM; ++m) {
#pragma unroll
          for (int s = 0; s < kSteps; ++s) {
            const uint32_t w2 = clamp_e8m0x4(s < 2 ? sfw[m].x : sfw[m].y) >> (16 * (s & 1));
            const uint32_t col = kSfaBase + 4u * (uint32_t)((slot * kSteps + s) * NM + m) + (uint32_t)q;
            tmem_st1(tmem + lanes + col, w2 & 0xFFFFu);
          }
        }
        tmem_st_wait();
        fence_proxy_async();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&S.b_full[slot]));
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          code[u][0] = ncode[u][0];
          code[u][1] = ncode[u][1];
          xsv[u] = nxsv[u];
        }
#pragma unroll
        for (int m = 0; m < NM; ++m) sfw[m] = nsfw[m];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&S.tab_empty[tb]));
    }
  } else if (warp == kWarpTma) {
    // ------------------------------------------------ tensor copies of the weights
    if (lane == 0) {
      for (int lt = 0; lt < my_tiles; ++lt) {
        const Tile tl = tile_of(S, p, cta + lt * G, mt);
        const int row0 = tl.e * p.N + tl.mtile * kRows;
        bool ok = true;
        for (int st = 0; st < nstg; ++st) {
          const int g = lt * nstg + st, slot = g % NS;
          if (g >= NS && !mbar_wait(smem_addr(&S.slot_free[slot]), ((g / NS) - 1) & 1, p.status)) {
            ok = false;
            break;
          }
          const uint32_t bar = smem_addr(&S.a_full[slot]);
          mbar_arrive_expect_tx(bar, (uint32_t)NM * kAMat);
#pragma unroll
          for (int m = 0; m < NM; ++m)
            tma_load_2d(s_a + (uint32_t)(slot * NM + m) * kAMat, &maps.w[m], st * (kStageK / 2), row0, bar);
        }
        if (!ok) break;
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ------------------------------------------------ MMA issue
    if (lane == 0) {
      const uint32_t idesc = idesc_mxf4(kRows, kN);
      const uint64_t adesc0 = smem_desc_sw128(s_a), bdesc0 = smem_desc(s_b, 128u, 1024u);
      bool ok = true;
      for (int lt = 0; lt < my_tiles && ok; ++lt) {
        for (int st = 0; st < nstg && ok; ++st) {
          const int g = lt * nstg + st, slot = g % NS;
          ok = mbar_wait_spin(smem_addr(&S.a_full[slot]), (g / NS) & 1, p.status) &&
               mbar_wait_spin(smem_addr(&S.b_full[slot]), (g / NS) & 1, p.status);
          if (!ok) break;
          tc_fence_after();
          // descriptors of this stage; the MMAs below only add constant offsets
          const uint64_t ad0 = adesc0 + (uint64_t)(((uint32_t)slot * NM * kAMat) >> 4);
          const uint64_t bd0 = bdesc0 + (uint64_t)(((uint32_t)slot * kBStage) >> 4);
          const uint32_t sfa0 = tmem + kSfaBase + 4u * (uint32_t)(slot * kSteps * NM);
#pragma unroll
          for (int s = 0; s < kSteps; ++s) {
            const int j = g * kSteps + s, db = j % ND;
            if (j >= ND && !mbar_wait_spin(smem_addr(&S.d_free[db]), ((j / ND) - 1) & 1, p.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t d0 = tmem + kDBase + (uint32_t)db * (NM * kN);
#pragma unroll
            for (int pl = 0; pl < kPlanes; ++pl)
#pragma unroll
              for (int m = 0; m < NM; ++m)
                mma_mxf4(d0 + (uint32_t)m * kN, ad0 + (uint64_t)((m * kAMat + 32u * s) >> 4),
                         bd0 + (uint64_t)((pl * kBPlane + 256u * s) >> 4), idesc, sfa0 + 4u * (uint32_t)(s * NM + m),
                         tmem + 4u * pl, true);
            mma_commit(smem_addr(&S.d_full[db]));
          }
          if (ok) mma_commit(smem_addr(&S.slot_free[slot]));
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ column tables, one tile ahead
    for (int lt = 0; lt < my_tiles; ++lt) {
      const Tile tl = tile_of(S, p, cta + lt * G, mt);
      const int tb = lt & 1;
      if (lt >= 2 && !warp_wait(smem_addr(&S.tab_empty[tb]), ((lt >> 1) - 1) & 1, p.status)) break;
      const int c = lane;
      int a = -1;
      if (c < tl.ncols) {
        a = p.sorted[tl.col0 + c];  // -1: padding of the expert's segment
        if (a >= p.A) {
          if (p.status) atomicOr(p.status, MOE_DEV_BAD_ROW);
          a = -1;
        }
      }
      S.colasg[tb][c] = a;
      S.colrow[tb][c] = a < 0 ? -1 : (p.bytoken ? token_of(a, p.kdiv) : a);
      if (lane == 0) {
        S.ncols[tb] = tl.ncols;
        S.mrow[tb] = tl.mtile * kRows;
        S.wrow[tb] = (int64_t)tl.e * p.N + tl.mtile * kRows;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&S.tab_full[tb]));
    }
  }
  // every MMA of this CTA has completed (the drain waited for the last one)
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
  TcArgs p{};
  p.aq = aq; p.ld_aq = ld_aq; p.as = as; p.ld_as = ld_as;
  p.s0 = s0; p.s1 = s1;
  p.offsets = offsets; p.sorted = sorted; p.cap = cap;
  p.A = A; p.k = k; p.E = E; p.K = K; p.N = N; p.bytoken = bytoken; p.min_rows = min_rows < 0 ? 0 : min_rows;
  p.kdiv = kdiv_of(k);
  p.out0 = out0; p.out1 = out1; p.ld_out = ld_out;
  p.status = device_status_word();
  TcMaps maps{};
  const uint64_t rows = (uint64_t)E * N;
  for (int m = 0; m < nm; ++m) {
    if (!encode_rows(&maps.w[m], m == 0 ? w0 : w1, rows, (uint64_t)K / 2))
      return fail(MOE_ERR_UNSUPPORTED, "%s: tensor maps of the weights could not be built (16-byte aligned weights are required)", name);
  }
  // tensor memory: B scales [0, 16), A scales (4 columns per matrix and K-step
  // of each stage slot) from 16, accumulators (64 columns per matrix) from 128
  const int ns_tmem = (int)((kDBase - kSfaBase) / (4u * kSteps * (uint32_t)nm));
  p.ndbuf = (int)((kTmemCols - kDBase) / (uint32_t)(nm * kN));
  if (p.ndbuf > kMaxDBuf) p.ndbuf = kMaxDBuf;
  // shared memory: the stage ring (packed weights, digit planes, activation
  // scales), then the small state
  const uint32_t stage = (uint32_t)nm * kAMat + kBStage + kXsStage;
  const size_t fixed = (size_t)tc_shared_bytes(E) + 1024u + 64u;
  int ns = (int)(((size_t)optin - fixed) / stage);
  if (ns > kMaxStages) ns = kMaxStages;
  if (ns > ns_tmem) ns = ns_tmem;
  if (ns < 2) return fail(MOE_ERR_UNSUPPORTED, "%s: tensor path does not fit shared memory", name);
  p.nstage = ns;
  p.off_a = 0;  // 1024-aligned (swizzled copies)
  p.off_b = (uint32_t)ns * nm * kAMat;
  p.off_xs = p.off_b + (uint32_t)ns * kBStage;
  p.off_misc = (p.off_xs + (uint32_t)ns * kXsStage + 63u) & ~63u;
  const size_t smem = (size_t)p.off_misc + tc_shared_bytes(E) + 1024u;  // + alignment of the base
  if (smem > (size_t)optin) return fail(MOE_ERR_UNSUPPORTED, "%s: tensor path needs %zu bytes of shared memory", name, smem);
  auto kern = mode == kSwiglu ? tc_expert_kernel<kSwiglu> : mode == kRaw ? tc_expert_kernel<kRaw> : tc_expert_kernel<kDownMode>;
  const moe_status ast = ensure_smem_attr(reinterpret_cast<const void *>(kern), optin, name);
  if (ast != MOE_OK) return ast;
  kern<<<sm_count(), kThreads, smem, stream>>>(p, maps);
  err = cudaGetLastError();
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, name);
}

}  // namespace moe
