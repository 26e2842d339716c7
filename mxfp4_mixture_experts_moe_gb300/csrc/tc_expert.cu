// Tensor-core (tcgen05) path of the MXFP4 expert projections, used by the
// stage calls for batches of more than 16 rows (prefill and large decode
// batches; the 1-16-row exact-rows regime never takes it).
//
// The layer's projections as grouped GEMMs, "DeepSeek-V4-Flash on AMD gfx90a",
// §6.1 (packed FP4 weights with E8M0 block scales, INT8 per-32 activations)
// and "Optimizing DeepSeek V4 Flash Inference on a Strix Halo Pair", "MXFP4
// routed-expert kernels" (prefill tiles over the tokens of one expert).
// Per expert e with n_e rows, out[row i][token t] = sum_k W[i][k] X[t][k]
// with W the dequantised MXFP4 weights and X the dequantised Q8 activations.
//
// Operands (f16, tensor-core kind::f16, fp32 accumulation in tensor memory
// over the whole reduction):
//   A = E2M1 value * 2^(u - umax_i)   exact in f16 (umax_i = largest scale
//       byte of weight row i in the tile; factors below 2^-24 flush to 0)
//   B = Bhi + Blo, two f16 operands: v = q * sx / S_t (q the Q8 code, sx its
//       block scale, S_t a power of two per token column with |v| <= 2^15),
//       Bhi = f16(v), Blo = f16(v - Bhi): about 22 significant bits
// and the epilogue multiplies by 2^(umax_i - 127) * S_t.  Unlike the
// CUDA-core path there is no per-block integer dot here; the result differs
// from the exact one by the tensor core's fp32 accumulation (relative
// ~1e-5 on a 4096-term reduction) and B's residual.
//
// Tiles: 128 weight rows x up to 32 token columns of one expert, K in chunks
// of 64 (two MX blocks); two MMAs (Bhi, Blo) per matrix and K step, A read
// from tensor memory.  One persistent CTA per SM walks the tile list it
// derives from the expert offsets, with warp-specialised roles:
//   warps 0-15  widen the packed weights of one row and 64 K to f16 in
//               registers and store them into a tensor-memory operand stage
//               (tcgen05.st), one lane per weight row, in groups that take
//               alternate chunks;
//   warps 16-19 copy the token rows ahead (cp.async ring), write Bhi / Blo
//               into a shared-memory operand stage, and drain the previous
//               tile's accumulators (one TMEM lane quadrant each);
//   warp 20     issues the tensor copies (TMA): 128 weight rows x 128 bytes
//               (256 K) per copy, 128-byte swizzled, and the tile's scale
//               bytes into a double buffer;
//   warp 21     issues the MMAs;
//   warp 22     builds the next tile's column tables (assignment, activation
//               row, S_t) ahead of time.
// Tensor memory holds two accumulator buffers (the epilogue of one tile
// overlaps the next) and the A operand stages.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "mx_device.cuh"
#include "tc_device.cuh"

namespace moe {
namespace {

constexpr int kTcRows = 128;    // weight rows per tile (MMA M)
constexpr int kTcCols = 32;     // token columns per tile, at most (MMA N)
constexpr int kTcK = 64;        // reduction elements per chunk (one operand stage)
constexpr int kTcSlice = 256;   // reduction elements per packed-weight copy (128-byte rows)
constexpr int kAWarps = 16;     // weight converters
constexpr int kBWarps = 4;      // token side and epilogue
constexpr int kWarpProd = kAWarps + kBWarps;
constexpr int kWarpMma = kWarpProd + 1;
constexpr int kWarpTab = kWarpMma + 1;
constexpr int kTcThreads = 32 * (kWarpTab + 1);
constexpr int kBThreads = 32 * kBWarps;
constexpr int kBAhead = 6;      // token-row chunks in flight per token-side thread
constexpr int kMaxA = 8;        // operand stages, at most
constexpr int kMaxRaw = 8;      // packed-weight stages, at most
constexpr uint32_t kRawMat = 128u * 128u;                     // one matrix's packed slice, 16 KB
constexpr uint32_t kBStage = 2u * kTcCols * kTcK * 2u;        // Bhi + Blo of one chunk, 8 KB
constexpr uint32_t kBRawSlot = (uint32_t)kBThreads * 20u;      // 16 code bytes + 1 scale per thread
constexpr uint32_t kAccCols = 128;  // TMEM columns [0, 128): two accumulator buffers of 64
constexpr uint32_t kTmemCols = 512;

static_assert(kBThreads == 4 * kTcCols, "one token-side thread per (column, 16-element piece)");

struct TcArgs {
  const int8_t *aq;  // Q8 activation codes: x rows (gate/up, by token) or h rows (down, by assignment)
  int64_t ld_aq;
  const float *as;
  int64_t ld_as;
  const int32_t *offsets, *sorted;
  int64_t cap;
  int A, k, E, K, N;  // K reduction length, N output rows per expert
  int bytoken;        // activation row of assignment a: a / k (1) or a (0)
  uint32_t kdiv;
  float *out;
  int64_t ld_out;
  unsigned *status;
  int as16;  // activation scale rows are 16-byte aligned
  int nA;    // operand stages
  int nraw;  // packed-weight stages
  // shared memory (bytes from the 1024-aligned base)
  uint32_t scale_buf;  // one tile's scale bytes (NM x 128 rows x K/32)
  uint32_t off_scale, off_raw, off_b, off_braw, off_misc;
};

struct TcMaps {  // 2-D tensor maps (TMA) of the packed weights and their scale bytes
  CUtensorMap w[2], s[2];
};

struct TcShared {
  uint64_t raw_full[kMaxRaw], raw_empty[kMaxRaw];
  uint64_t full[kMaxA], a_empty[kMaxA];
  uint64_t acc_full[2], acc_empty[2], scale_full[2], scale_empty[2], tab_full[2], tab_empty[2], umax_full[3];
  uint32_t tmem_slot;
  int ncols[2], mtile[2];
  int colrow[2][kTcCols], colasg[2][kTcCols];
  float colS[2][kTcCols], colInv[2][kTcCols];
  int umax[3][2 * kTcRows];  // largest scale byte of each weight row (matrix-major)
  int prefix[1];             // [E + 1] tiles before expert e
};

uint32_t tc_shared_bytes(int E) { return (uint32_t)(sizeof(TcShared) + 4u * (uint32_t)E); }

// f16 bits of 2^-d (d >= 0): normal down to 2^-14, subnormal to 2^-24, else 0.
MOE_DEVFN uint32_t f16_pow2_neg(int d) {
  if (d <= 14) return (uint32_t)(15 - d) << 10;
  if (d <= 24) return 1u << (24 - d);
  return 0u;
}

// 2^(u - 127) as fp32 (u = 255: NaN).
MOE_DEVFN float e8m0_value(int u) {
  if (u >= 255) return __uint_as_float(0x7FC00000u);
  if (u >= 1) return __uint_as_float((uint32_t)u << 23);
  return __uint_as_float(0x00400000u);
}

// Smallest power of two >= v for finite v > 0; 1 otherwise.
MOE_DEVFN float pow2_ceil(float v) {
  if (!(v > 0.0f) || !(v < 3.0e38f)) return 1.0f;
  const uint32_t b = __float_as_uint(v);
  const uint32_t e = b >> 23, man = b & 0x7FFFFFu;
  if (e == 0) return __uint_as_float(0x00800000u);  // below the normal range: 2^-126
  return __uint_as_float((e + (man != 0)) << 23);
}

MOE_DEVFN uint32_t lds_u16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

// A box of 128 rows x nb bytes lands in shared memory with the tensor-copy
// swizzle that matches its row length (nb = 128 / 64 / 32 bytes: 128B / 64B /
// 32B swizzle, 16: none): the 16-byte chunk j of row r sits at chunk j ^ x(r).
MOE_DEVFN uint32_t swz_of(int r, int nb) {
  return nb == 128 ? (uint32_t)(r & 7) : nb == 64 ? (uint32_t)((r >> 1) & 3) : nb == 32 ? (uint32_t)((r >> 2) & 1) : 0u;
}
MOE_DEVFN uint32_t swz_addr(uint32_t base, int r, int byte, int nb, uint32_t x) {
  return base + (uint32_t)r * (uint32_t)nb + ((((uint32_t)byte >> 4) ^ x) << 4) + ((uint32_t)byte & 15u);
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

struct Tile {
  int e, mtile, ncols, ncol16;
  int64_t row0;  // first weight row of the tile (expert e)
  int col0;      // first sorted position of the tile
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
  tl.col0 = b + ntile * kTcCols;
  tl.ncols = min(kTcCols, n_e - ntile * kTcCols);
  tl.ncol16 = (tl.ncols + 15) & ~15;
  tl.row0 = (int64_t)lo * p.N + (int64_t)tl.mtile * kTcRows;
  return tl;
}

// Four packed bytes (8 weights) -> four f16x2 pairs scaled by f2.
MOE_DEVFN void widen8(uint32_t w, uint32_t f2, uint32_t *o) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}\n"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w));
#pragma unroll
  for (int i = 0; i < 4; ++i) asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(o[i]) : "r"(f2));
}

template <int NM>
__global__ void __launch_bounds__(kTcThreads, 1) tc_expert_kernel(const TcArgs p, const __grid_constant__ TcMaps maps) {
  extern __shared__ __align__(1024) uint8_t smem_dyn[];
  const uint32_t dyn = smem_addr(smem_dyn);
  const uint32_t pad = ((dyn + 1023u) & ~1023u) - dyn;
  uint8_t *smem = smem_dyn + pad;
  const uint32_t sb = dyn + pad;
  TcShared &S = *reinterpret_cast<TcShared *>(smem + p.off_misc);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  const int K = p.K, nb = K / 32, nchunk = K / kTcK, nslice = K / kTcSlice, mt = p.N / kTcRows;
  const int nA = p.nA, nraw = p.nraw;
  constexpr int NG = 4 / NM;  // converter groups (chunks c = group mod NG)

  if (tid == 0) {
    for (int s = 0; s < nraw; ++s) {
      mbar_init(smem_addr(&S.raw_full[s]), 1);
      mbar_init(smem_addr(&S.raw_empty[s]), kAWarps);
    }
    for (int s = 0; s < nA; ++s) {
      mbar_init(smem_addr(&S.full[s]), 4 * NM + kBWarps);
      mbar_init(smem_addr(&S.a_empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_addr(&S.acc_full[b]), 1);
      mbar_init(smem_addr(&S.acc_empty[b]), kBWarps);
      mbar_init(smem_addr(&S.scale_full[b]), 1);
      mbar_init(smem_addr(&S.scale_empty[b]), kAWarps);
      mbar_init(smem_addr(&S.tab_full[b]), 1);
      mbar_init(smem_addr(&S.tab_empty[b]), kBWarps);
    }
    for (int b = 0; b < 3; ++b) mbar_init(smem_addr(&S.umax_full[b]), 4 * NM);
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
        if (!bad && en > b) nt = ((en - b + kTcCols - 1) / kTcCols) * mt;
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
  const uint32_t s_scale = sb + p.off_scale, s_raw = sb + p.off_raw, s_b = sb + p.off_b, s_braw = sb + p.off_braw;

  if (warp < kAWarps) {
    // ------------------------------------------------ weights -> tensor memory
    const int grp = warp / (4 * NM), mm = NM == 2 ? (warp >> 2) & 1 : 0, q = warp & 3;
    const int r = 32 * q + lane;  // weight row of the tile = TMEM lane
    const uint32_t lanes = (uint32_t)(32 * q) << 16;
    const uint32_t xs = swz_of(r, nb), xr = (uint32_t)(r & 7);
    for (int lt = 0; lt < my_tiles; ++lt) {
      const int sbuf = lt & 1;
      const uint32_t scl = s_scale + (uint32_t)sbuf * p.scale_buf + (uint32_t)mm * kTcRows * nb;
      if (!warp_wait(smem_addr(&S.scale_full[sbuf]), (lt >> 1) & 1, p.status)) break;
      uint32_t m4 = 0;
      for (int j = 0; j < nb / 16; ++j) {
        const uint4 v = lds128(swz_addr(scl, r, 16 * j, nb, xs));
        m4 = __vmaxu4(__vmaxu4(m4, v.x), __vmaxu4(__vmaxu4(v.y, v.z), v.w));
      }
      const int umax = (int)max(max(m4 & 0xFFu, (m4 >> 8) & 0xFFu), max((m4 >> 16) & 0xFFu, m4 >> 24));
      if (grp == 0) {
        S.umax[lt % 3][mm * kTcRows + r] = umax;
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&S.umax_full[lt % 3]));
      }
      bool dead = false;
      for (int c = grp; c < nchunk; c += NG) {
        const int g = lt * nchunk + c, s = g % nA;
        const int J = lt * nslice + (c >> 2), rs = J % nraw;
        if (!warp_wait(smem_addr(&S.raw_full[rs]), (J / nraw) & 1, p.status)) { dead = true; break; }
        if (g >= nA && !warp_wait(smem_addr(&S.a_empty[s]), ((g / nA) - 1) & 1, p.status)) { dead = true; break; }
        tc_fence_after();
        const uint32_t row = s_raw + (uint32_t)rs * NM * kRawMat + (uint32_t)mm * kRawMat + (uint32_t)r * 128u;
        const uint32_t j0 = 2u * (uint32_t)(c & 3);
        const uint4 pa = lds128(row + ((j0 ^ xr) << 4));
        const uint4 pb = lds128(row + (((j0 + 1u) ^ xr) << 4));
        const uint32_t u2 = lds_u16(swz_addr(scl, r, 2 * c, nb, xs));
        const uint32_t fa = f16_pow2_neg(umax - (int)(u2 & 0xFFu)), fb = f16_pow2_neg(umax - (int)(u2 >> 8));
        const uint32_t fa2 = fa | (fa << 16), fb2 = fb | (fb << 16);
        uint32_t o[32];
        widen8(pa.x, fa2, o + 0);
        widen8(pa.y, fa2, o + 4);
        widen8(pa.z, fa2, o + 8);
        widen8(pa.w, fa2, o + 12);
        widen8(pb.x, fb2, o + 16);
        widen8(pb.y, fb2, o + 20);
        widen8(pb.z, fb2, o + 24);
        widen8(pb.w, fb2, o + 28);
        tmem_st32(tmem + lanes + kAccCols + (uint32_t)(s * NM + mm) * 32u, o);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_addr(&S.full[s]));
          if ((c & 3) + NG >= 4) mbar_arrive(smem_addr(&S.raw_empty[rs]));  // this group's last chunk of the slice
        }
      }
      if (dead) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&S.scale_empty[sbuf]));
    }
  } else if (warp < kWarpProd) {
    // ------------------------------------------------ token side + epilogue
    const int bt = tid - 32 * kAWarps, q = warp & 3;
    const int cc = bt >> 2, pc = bt & 3;  // token column, 16-element piece of the chunk
    const int total = my_tiles * nchunk;
    bool dead = false;
    auto issue = [&](int pos) {
      if (pos < total) {
        const int lt = pos / nchunk, c = pos - lt * nchunk, tb = lt & 1;
        if (c == 0 && !warp_wait(smem_addr(&S.tab_full[tb]), (lt >> 1) & 1, p.status)) dead = true;
        const int row = dead ? -1 : S.colrow[tb][cc];
        if (row >= 0) {
          const uint32_t slot = s_braw + (uint32_t)(pos % kBAhead) * kBRawSlot;
          cp_async16(slot + 16u * bt, p.aq + (int64_t)row * p.ld_aq + c * kTcK + 16 * pc);
          cp_async4(slot + 16u * kBThreads + 4u * bt, p.as + (int64_t)row * p.ld_as + 2 * c + (pc >> 1));
        }
      }
      cp_async_commit();
    };
    auto epilogue = [&](int lt) {
      const int ab = lt & 1, tb = lt & 1, u3 = lt % 3;
      bool ok = warp_wait(smem_addr(&S.acc_full[ab]), (lt >> 1) & 1, p.status) &&
                warp_wait(smem_addr(&S.umax_full[u3]), (lt / 3) & 1, p.status);
      tc_fence_after();
      const int i = 32 * q + lane;
      const float rs0 = e8m0_value(S.umax[u3][i]);
      const float rs1 = NM == 2 ? e8m0_value(S.umax[u3][kTcRows + i]) : 0.0f;
      const int ncols = S.ncols[tb], ncol16 = (ncols + 15) & ~15;
      const int64_t orow = (int64_t)S.mtile[tb] * kTcRows + i;
      const uint32_t acc = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)ab * 64u;
      for (int cb = 0; ok && cb < ncol16; cb += 16) {
        float d0[16];
        tmem_ld16(acc + (uint32_t)cb, d0);
        if (NM == 2) {
          float d1[16];
          tmem_ld16(acc + 32u + (uint32_t)cb, d1);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int col = cb + j;
            const int a = col < ncols ? S.colasg[tb][col] : -1;
            if (a >= 0) {
              const float Sc = S.colS[tb][col];
              const float gv = __fmul_rn(__fmul_rn(d0[j], rs0), Sc), uv = __fmul_rn(__fmul_rn(d1[j], rs1), Sc);
              p.out[(int64_t)a * p.ld_out + orow] = __fmul_rn(silu(gv), uv);
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int col = cb + j;
            const int a = col < ncols ? S.colasg[tb][col] : -1;
            if (a >= 0) p.out[(int64_t)a * p.ld_out + orow] = __fmul_rn(__fmul_rn(d0[j], rs0), S.colS[tb][col]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_addr(&S.acc_empty[ab]));
        mbar_arrive(smem_addr(&S.tab_empty[tb]));
      }
      return ok;
    };
    for (int j = 0; j < kBAhead - 1; ++j) issue(j);
    for (int pos = 0; pos < total && !dead; ++pos) {
      issue(pos + kBAhead - 1);
      cp_async_wait<kBAhead - 1>();
      const int lt = pos / nchunk, c = pos - lt * nchunk, tb = lt & 1;
      const int s = pos % nA;
      if (pos >= nA && !warp_wait(smem_addr(&S.a_empty[s]), ((pos / nA) - 1) & 1, p.status)) break;
      const int ncols = S.ncols[tb], ncol16 = (ncols + 15) & ~15;
      if (cc < ncol16) {
        uint32_t hi[8], lo[8];
        const int row = S.colrow[tb][cc];
        if (cc < ncols && row >= 0) {
          const uint32_t slot = s_braw + (uint32_t)(pos % kBAhead) * kBRawSlot;
          const uint4 codes = lds128(slot + 16u * bt);
          const float fac = __fmul_rn(lds_f32(slot + 16u * kBThreads + 4u * bt), S.colInv[tb][cc]);
          const uint32_t cw[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint32_t wv = cw[i >> 1];
            const int sh = 16 * (i & 1);
            const float v0 = __fmul_rn((float)(int8_t)(wv >> sh), fac);
            const float v1 = __fmul_rn((float)(int8_t)(wv >> (sh + 8)), fac);
            asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(hi[i]) : "f"(v1), "f"(v0));
            float h0, h1;
            asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n cvt.f32.f16 %0, l;\n cvt.f32.f16 %1, h;\n}\n"
                : "=f"(h0), "=f"(h1) : "r"(hi[i]));
            asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(lo[i]) : "f"(__fsub_rn(v1, h1)), "f"(__fsub_rn(v0, h0)));
          }
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) hi[i] = lo[i] = 0u;
        }
        const uint32_t st = s_b + (uint32_t)s * kBStage;
        const uint32_t o0 = tile_offset(cc, 16 * pc), o1 = tile_offset(cc, 16 * pc + 8);
        sts128(st + o0, make_uint4(hi[0], hi[1], hi[2], hi[3]));
        sts128(st + o1, make_uint4(hi[4], hi[5], hi[6], hi[7]));
        sts128(st + kBStage / 2 + o0, make_uint4(lo[0], lo[1], lo[2], lo[3]));
        sts128(st + kBStage / 2 + o1, make_uint4(lo[4], lo[5], lo[6], lo[7]));
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&S.full[s]));
      // the previous tile's accumulators, once this tile's first chunks are on their way
      if (lt >= 1 && c == min(1, nchunk - 1) && !epilogue(lt - 1)) dead = true;
    }
    cp_async_wait<0>();
    if (!dead && my_tiles > 0) epilogue(my_tiles - 1);
  } else if (warp == kWarpProd) {
    // ------------------------------------------------ tensor copies
    if (lane == 0) {
      int J = 0;
      for (int lt = 0; lt < my_tiles; ++lt) {
        const Tile tl = tile_of(S, p, cta + lt * G, mt);
        const int sbuf = lt & 1;
        if (lt >= 2 && !mbar_wait(smem_addr(&S.scale_empty[sbuf]), ((lt >> 1) - 1) & 1, p.status)) break;
        const uint32_t sbar = smem_addr(&S.scale_full[sbuf]);
        mbar_arrive_expect_tx(sbar, (uint32_t)NM * kTcRows * nb);
#pragma unroll
        for (int mm = 0; mm < NM; ++mm)
          tma_load_2d(s_scale + (uint32_t)sbuf * p.scale_buf + (uint32_t)mm * kTcRows * nb, &maps.s[mm], 0,
                      (int)tl.row0, sbar);
        bool dead = false;
        for (int sl = 0; sl < nslice; ++sl, ++J) {
          const int rs = J % nraw;
          if (J >= nraw && !mbar_wait(smem_addr(&S.raw_empty[rs]), ((J / nraw) - 1) & 1, p.status)) {
            dead = true;
            break;
          }
          const uint32_t bar = smem_addr(&S.raw_full[rs]);
          mbar_arrive_expect_tx(bar, (uint32_t)NM * kRawMat);
#pragma unroll
          for (int mm = 0; mm < NM; ++mm)
            tma_load_2d(s_raw + (uint32_t)(rs * NM + mm) * kRawMat, &maps.w[mm], sl * 128, (int)tl.row0, bar);
        }
        if (dead) break;
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ------------------------------------------------ MMA issue
    if (lane == 0) {
      for (int lt = 0; lt < my_tiles; ++lt) {
        const Tile tl = tile_of(S, p, cta + lt * G, mt);
        const int ab = lt & 1;
        if (lt >= 2 && !mbar_wait(smem_addr(&S.acc_empty[ab]), ((lt >> 1) - 1) & 1, p.status)) break;
        tc_fence_after();
        const uint32_t idesc = idesc_f16(kTcRows, tl.ncol16);
        bool ok = true;
        for (int c = 0; c < nchunk; ++c) {
          const int g = lt * nchunk + c, s = g % nA;
          if (!mbar_wait(smem_addr(&S.full[s]), (g / nA) & 1, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t bh = s_b + (uint32_t)s * kBStage, bl = bh + kBStage / 2;
#pragma unroll
          for (int mm = 0; mm < NM; ++mm) {
            const uint32_t d = tmem + (uint32_t)ab * 64u + (uint32_t)mm * 32u;
            const uint32_t a = tmem + kAccCols + (uint32_t)(s * NM + mm) * 32u;
#pragma unroll
            for (int ks = 0; ks < kTcK / 16; ++ks) {
              mma_f16_ts(d, a + 8u * ks, smem_desc(bh + 256u * ks, kCoreLbo, kCoreSbo), idesc, c > 0 || ks > 0);
              mma_f16_ts(d, a + 8u * ks, smem_desc(bl + 256u * ks, kCoreLbo, kCoreSbo), idesc, true);
            }
          }
          mma_commit(smem_addr(&S.a_empty[s]));
        }
        if (!ok) break;
        mma_commit(smem_addr(&S.acc_full[ab]));
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
      const int row = a < 0 ? -1 : (p.bytoken ? token_of(a, p.kdiv) : a);
      // the column's scale S_t: |q * sx| <= 127 * max sx; S_t scales the
      // column into [-2^15, 2^15], the top of the f16 normal range, so that
      // blocks far below the column's largest stay normal (full 11-bit
      // precision in Bhi and Blo)
      float mx = 0.0f;
      if (row >= 0) {
        const float *sp = p.as + (int64_t)row * p.ld_as;
        if (p.as16) {
          const float4 *s4 = reinterpret_cast<const float4 *>(sp);
          for (int w = 0; w < nb / 4; ++w) {
            const float4 v = __ldg(s4 + w);
            mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
          }
        } else {
          for (int w = 0; w < nb; ++w) mx = fmaxf(mx, fabsf(__ldg(sp + w)));
        }
      }
      const float Sc = __fmul_rn(pow2_ceil(127.0f * mx), 1.0f / 32768.0f);
      S.colasg[tb][c] = a;
      S.colrow[tb][c] = row;
      S.colS[tb][c] = Sc;
      S.colInv[tb][c] = 1.0f / Sc;
      if (lane == 0) {
        S.ncols[tb] = tl.ncols;
        S.mtile[tb] = tl.mtile;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&S.tab_full[tb]));
    }
  }
  // every MMA of this CTA has completed (the last epilogue waited for it)
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

// Row-major u8 matrix [rows][cols] (cols bytes per row) as a 2-D tensor map
// with boxes of box_cols bytes x 128 rows, swizzled to match box_cols.
bool encode_rows(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint32_t box_cols) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {box_cols, (cuuint32_t)kTcRows};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle swz = box_cols == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                 : box_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                 : box_cols == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                  : CU_TENSOR_MAP_SWIZZLE_NONE;
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tc_expert_supported(int K, int N) { return K % 512 == 0 && K <= 4096 && N % kTcRows == 0; }

// Launch of the tensor-core path (moe_mxfp4_gateup_swiglu / moe_mxfp4_down for
// T > 16).  nm = 2: gate and up with SwiGLU; nm = 1: down.
moe_status launch_tc_expert(int nm, const int8_t *aq, int64_t ld_aq, const float *as, int64_t ld_as,
                            const uint8_t *w0, const uint8_t *s0, const uint8_t *w1, const uint8_t *s1,
                            const int32_t *offsets, const int32_t *sorted, int64_t cap, int A, int k, int E,
                            int K, int N, int bytoken, float *out, int64_t ld_out, cudaStream_t stream,
                            const char *name) {
  if (!tc_expert_supported(K, N))
    return fail(MOE_ERR_UNSUPPORTED, "%s: tensor path needs K %% 512 == 0 (<= 4096) and rows %% 128 == 0", name);
  if (E > 4096) return fail(MOE_ERR_UNSUPPORTED, "%s: E=%d", name, E);
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_fail(err, name);
  int optin = 0;
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  TcArgs p{};
  p.aq = aq; p.ld_aq = ld_aq; p.as = as; p.ld_as = ld_as;
  p.offsets = offsets; p.sorted = sorted; p.cap = cap;
  p.A = A; p.k = k; p.E = E; p.K = K; p.N = N; p.bytoken = bytoken;
  p.kdiv = kdiv_of(k);
  p.out = out; p.ld_out = ld_out;
  p.status = device_status_word();
  p.as16 = ((uintptr_t)as % 16 == 0 && ld_as % 4 == 0) ? 1 : 0;
  TcMaps maps{};
  const uint64_t rows = (uint64_t)E * N;
  for (int mm = 0; mm < nm; ++mm) {
    if (!encode_rows(&maps.w[mm], mm == 0 ? w0 : w1, rows, (uint64_t)K / 2, 128u) ||
        !encode_rows(&maps.s[mm], mm == 0 ? s0 : s1, rows, (uint64_t)K / 32, (uint32_t)(K / 32)))
      return fail(MOE_ERR_UNSUPPORTED, "%s: tensor maps of the weights could not be built (16-byte aligned weights and scales are required)", name);
  }
  // shared memory: two tile-scale buffers, the packed-weight ring, the
  // operand (Bhi / Blo) ring, the token-row ring, small state.  Operand
  // stages also take tensor memory (nm x 32 columns each, after the two
  // accumulator buffers); packed-weight stages get what shared memory is left.
  const uint32_t nb = (uint32_t)K / 32;
  p.scale_buf = (uint32_t)nm * kTcRows * nb;
  const int na_tmem = (int)((kTmemCols - kAccCols) / (32u * (uint32_t)nm));
  const size_t fixed0 = 2u * (size_t)p.scale_buf + (size_t)kBAhead * kBRawSlot + tc_shared_bytes(E) + 1024u + 64u;
  int nA = na_tmem < kMaxA ? na_tmem : kMaxA, nraw = 0;
  const int min_a = 4 / nm + 1;
  for (; nA >= min_a; --nA) {
    const size_t fixed = fixed0 + (size_t)nA * kBStage;
    nraw = fixed < (size_t)optin ? (int)(((size_t)optin - fixed) / ((size_t)nm * kRawMat)) : 0;
    if (nraw >= 3) break;
  }
  if (nA < min_a) nA = min_a;
  if (nraw > kMaxRaw) nraw = kMaxRaw;
  if (nraw < 2) return fail(MOE_ERR_UNSUPPORTED, "%s: tensor path does not fit shared memory", name);
  p.nA = nA;
  p.nraw = nraw;
  p.off_scale = 0;
  p.off_raw = 2u * p.scale_buf;  // a multiple of 1024 (swizzled copies land 1024-aligned)
  p.off_b = p.off_raw + (uint32_t)nraw * nm * kRawMat;
  p.off_braw = p.off_b + (uint32_t)nA * kBStage;
  p.off_misc = (p.off_braw + (uint32_t)kBAhead * kBRawSlot + 63u) & ~63u;
  const size_t smem = (size_t)p.off_misc + tc_shared_bytes(E) + 1024u;  // + alignment of the base
  if (smem > (size_t)optin) return fail(MOE_ERR_UNSUPPORTED, "%s: tensor path needs %zu bytes of shared memory", name, smem);
  auto kern = nm == 2 ? tc_expert_kernel<2> : tc_expert_kernel<1>;
  static bool configured[2][64] = {};
  if (dev < 64 && !configured[nm - 1][dev]) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
    if (err != cudaSuccess) return cuda_fail(err, name);
    configured[nm - 1][dev] = true;
  }
  kern<<<sm_count(), kTcThreads, smem, stream>>>(p, maps);
  err = cudaGetLastError();
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, name);
}

}  // namespace moe
