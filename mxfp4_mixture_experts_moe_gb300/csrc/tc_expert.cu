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
// Tiles: 128 weight rows x up to 64 token columns of one expert, K in chunks
// of 64 (two MX blocks); two MMAs (Bhi, Blo) per matrix and K step.  One
// persistent CTA per SM walks the tile list it derives from the expert
// offsets.  The packed weights of a chunk arrive by one 2-D tensor copy
// (TMA) per matrix, the tile's scale bytes by one per matrix, the token rows
// by cp.async, all into a deep raw ring; warps 0-7 widen them to f16 into an
// operand ring in the tensor core's K-major core-matrix layout; warp 8
// issues the MMAs; warps 0-3 also drain the accumulators (one TMEM lane
// quadrant each).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "mx_device.cuh"
#include "tc_device.cuh"

namespace moe {
namespace {

constexpr int kTcRows = 128;   // weight rows per tile (MMA M)
constexpr int kTcCols = 64;    // token columns per tile, at most (MMA N)
constexpr int kTcK = 64;       // reduction elements per chunk
constexpr int kTcRawMax = 12;  // packed-input stages, at most (as many as shared memory holds)
constexpr int kTcF16Max = 4;   // f16 operand stages, at most
constexpr int kTcConv = 8;     // converter warps
constexpr int kTcThreads = (kTcConv + 1) * 32;
constexpr int kConvThreads = kTcConv * 32;
constexpr uint32_t kRawArow = 32;  // packed A row of a chunk (TMA box row)
constexpr uint32_t kRawBrow = 80;  // B code row: 64 bytes, padded (conflict-free 8-byte reads)
constexpr uint32_t kF16Mat = (uint32_t)kTcRows * kTcK * 2;  // one f16 A matrix tile, 16 KB
constexpr uint32_t kF16B = (uint32_t)kTcCols * kTcK * 2;    // one f16 B tile (hi or lo), 8 KB

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
  // shared memory (bytes from the dynamic base)
  uint32_t raw_stage, raw_b, raw_bs;  // raw stage size; B codes / B scales offsets in a stage
  uint32_t f16_stage;                 // operand stage size (NM A tiles, then Bhi, Blo)
  int nraw;                           // packed-input stages
  int nf16;                           // operand stages
  uint32_t off_raw, off_f16, off_scale, off_misc;
};

struct TcMaps {  // 2-D tensor maps (TMA) of the packed weights and their scale bytes
  CUtensorMap w[2], s[2];
};

struct TcMisc {  // small shared state
  uint64_t *raw_full, *f16_full, *f16_empty, *acc_full, *acc_empty, *scale_full;
  uint32_t *tmem_slot;
  int *prefix;   // [E+1] tiles before expert e
  int *colrow;   // [64] activation row of each token column (-1: padding)
  int *colasg;   // [64] assignment of each column (-1: padding)
  int *umax;     // [2][128] largest scale byte of each weight row
  float *colS;   // [64] token scale S_t (a power of two)
  float *colInv; // [64] 1 / S_t
};

MOE_DEVFN TcMisc tc_misc(uint8_t *base) {
  TcMisc m;
  uint64_t *b = reinterpret_cast<uint64_t *>(base);
  m.raw_full = b; b += kTcRawMax;
  m.f16_full = b; b += kTcF16Max;
  m.f16_empty = b; b += kTcF16Max;
  m.acc_full = b; b += 1;
  m.acc_empty = b; b += 1;
  m.scale_full = b; b += 1;
  uint32_t *w = reinterpret_cast<uint32_t *>(b);
  m.tmem_slot = w; w += 4;
  m.colrow = reinterpret_cast<int *>(w); w += kTcCols;
  m.colasg = reinterpret_cast<int *>(w); w += kTcCols;
  m.umax = reinterpret_cast<int *>(w); w += 2 * kTcRows;
  m.colS = reinterpret_cast<float *>(w); w += kTcCols;
  m.colInv = reinterpret_cast<float *>(w); w += kTcCols;
  m.prefix = reinterpret_cast<int *>(w);
  return m;
}

uint32_t tc_misc_bytes(int E) {
  return 8u * (kTcRawMax + 2 * kTcF16Max + 3) + 4u * (4 + 4 * kTcCols + 2 * kTcRows) + 4u * (E + 1);
}

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

MOE_DEVFN Tile tile_of(const TcMisc &m, const TcArgs &p, int t, int mt) {
  // expert: last e with prefix[e] <= t (binary search over E+1 entries)
  int lo = 0, hi = p.E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (m.prefix[mid] <= t) lo = mid;
    else hi = mid;
  }
  Tile tl;
  tl.e = lo;
  const int local = t - m.prefix[lo];
  tl.mtile = local % mt;
  const int ntile = local / mt;
  const int b = p.offsets[lo], n_e = p.offsets[lo + 1] - b;
  tl.col0 = b + ntile * kTcCols;
  tl.ncols = min(kTcCols, n_e - ntile * kTcCols);
  tl.ncol16 = (tl.ncols + 15) & ~15;
  tl.row0 = (int64_t)lo * p.N + (int64_t)tl.mtile * kTcRows;
  return tl;
}

// One chunk of the packed inputs into a raw stage: the weights by tensor copy
// (thread 0, expect_tx on the stage barrier), the token rows by cp.async from
// every converter thread (each then arrives on the barrier when its copies land).
template <int NM>
MOE_DEVFN void issue_raw(const TcArgs &p, const TcMaps &maps, const TcMisc &m, const Tile &tl, uint32_t raw,
                         uint32_t bar, int chunk, int ct) {
  const int k0 = chunk * kTcK;
  if (ct == 0) {
    mbar_arrive_expect_tx(bar, (uint32_t)NM * kTcRows * kRawArow);
#pragma unroll
    for (int mm = 0; mm < NM; ++mm)
      tma_load_2d(raw + (uint32_t)mm * kTcRows * kRawArow, &maps.w[mm], k0 / 2, (int)tl.row0, bar);
  }
  for (int q = ct; q < tl.ncol16 * 4; q += kConvThreads) {
    const int c = q >> 2, part = q & 3;
    const uint32_t dst = raw + p.raw_b + (uint32_t)c * kRawBrow + 16u * part;
    const int row = m.colrow[c];
    if (row >= 0) cp_async16(dst, p.aq + (int64_t)row * p.ld_aq + k0 + 16 * part);
    else sts128(dst, make_uint4(0, 0, 0, 0));
  }
  for (int q = ct; q < tl.ncol16 * 2; q += kConvThreads) {
    const int c = q >> 1, j = q & 1;
    const uint32_t dst = raw + p.raw_bs + (uint32_t)c * 8u + 4u * j;
    const int row = m.colrow[c];
    if (row >= 0) cp_async4(dst, p.as + (int64_t)row * p.ld_as + k0 / 32 + j);
    else sts32(dst, 0u);
  }
  cp_async_mbar_arrive_noinc(bar);
}

template <int NM>
__global__ void __launch_bounds__(kTcThreads, 1) tc_expert_kernel(const TcArgs p, const __grid_constant__ TcMaps maps) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  const int K = p.K, nb = K / 32, nchunk = K / kTcK, mt = p.N / kTcRows;
  const TcMisc m = tc_misc(smem + p.off_misc);
  const uint32_t sraw = smem_addr(smem + p.off_raw), sf16 = smem_addr(smem + p.off_f16);
  const uint32_t sscale = smem_addr(smem + p.off_scale);

  if (tid == 0) {
    for (int s = 0; s < p.nraw; ++s) mbar_init(smem_addr(&m.raw_full[s]), kConvThreads + 1);
    for (int s = 0; s < p.nf16; ++s) {
      mbar_init(smem_addr(&m.f16_full[s]), kConvThreads);
      mbar_init(smem_addr(&m.f16_empty[s]), 1);
    }
    mbar_init(smem_addr(m.acc_full), 1);
    mbar_init(smem_addr(m.acc_empty), 4);
    mbar_init(smem_addr(m.scale_full), 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_addr(m.tmem_slot), NM * kTcRows);
    // tiles per expert, prefix-summed (every CTA derives the same list)
    int carry = 0;
    if (lane == 0) m.prefix[0] = 0;
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
      if (e < p.E) m.prefix[e + 1] = carry + incl;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(m.tmem_slot);
  const int ntiles = m.prefix[p.E];

  if (warp == kTcConv) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      const int nf16 = p.nf16;
      int g = 0, done = 0;
      for (int t = cta; t < ntiles; t += G) {
        const Tile tl = tile_of(m, p, t, mt);
        const uint32_t idesc = idesc_f16(kTcRows, tl.ncol16);
        if (done > 0 && !mbar_wait(smem_addr(m.acc_empty), (done - 1) & 1, p.status)) break;
        tc_fence_after();
        bool ok = true;
        for (int c = 0; c < nchunk; ++c, ++g) {
          const int s = g % nf16;
          if (!mbar_wait(smem_addr(&m.f16_full[s]), (g / nf16) & 1, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = sf16 + (uint32_t)s * p.f16_stage;
#pragma unroll
          for (int mm = 0; mm < NM; ++mm) {
#pragma unroll
            for (int ks = 0; ks < kTcK / 16; ++ks) {
              const uint64_t ad = smem_desc(st + mm * kF16Mat + 256u * ks, kCoreLbo, kCoreSbo);
              mma_f16(tmem + (uint32_t)mm * kTcRows, ad, smem_desc(st + NM * kF16Mat + 256u * ks, kCoreLbo, kCoreSbo),
                      idesc, c > 0 || ks > 0);
              mma_f16(tmem + (uint32_t)mm * kTcRows, ad,
                      smem_desc(st + NM * kF16Mat + kF16B + 256u * ks, kCoreLbo, kCoreSbo), idesc, true);
            }
          }
          mma_commit(smem_addr(&m.f16_empty[s]));
        }
        if (!ok) break;
        mma_commit(smem_addr(m.acc_full));
        ++done;
      }
    }
    return;
  }

  // ------------------------------------------------------------ converters
  const int ct = tid;  // 0 .. kConvThreads-1
  const int nraw = p.nraw, nf16 = p.nf16;
  int g = 0, done = 0;
  bool dead = false;
  for (int t = cta; t < ntiles && !dead; t += G) {
    const Tile tl = tile_of(m, p, t, mt);
    // the tile's scale bytes (NM x 128 rows x nb) by tensor copy
    if (ct == 0) {
      mbar_arrive_expect_tx(smem_addr(m.scale_full), (uint32_t)NM * kTcRows * nb);
#pragma unroll
      for (int mm = 0; mm < NM; ++mm)
        tma_load_2d(sscale + (uint32_t)mm * kTcRows * nb, &maps.s[mm], 0, (int)tl.row0, smem_addr(m.scale_full));
    }
    // columns: activation row and assignment of each token column
    for (int c = ct; c < kTcCols; c += kConvThreads) {
      int a = -1;
      if (c < tl.ncols) {
        a = p.sorted[tl.col0 + c];
        if (a >= p.A) {
          if (p.status) atomicOr(p.status, MOE_DEV_BAD_ROW);
          a = -1;
        }
      }
      m.colasg[c] = a;
      m.colrow[c] = a < 0 ? -1 : (p.bytoken ? token_of(a, p.kdiv) : a);
    }
    bar_sync_named(1, kConvThreads);  // the column tables are read by other threads below
    // prologue: the first raw chunks (the scale copy is already on its way)
    for (int j = 0; j < nraw && j < nchunk; ++j)
      issue_raw<NM>(p, maps, m, tl, sraw + (uint32_t)((g + j) % nraw) * p.raw_stage,
                    smem_addr(&m.raw_full[(g + j) % nraw]), j, ct);
    // each token column's scale S_t: two threads per column, half the row's block scales each
    if (ct < 2 * kTcCols) {
      const int c = ct >> 1, half = ct & 1;
      const int row = m.colrow[c];
      float mx = 0.0f;
      if (row >= 0) {
        const float *sp = p.as + (int64_t)row * p.ld_as + half * (nb / 2);
        if (p.as16) {
          const float4 *s4 = reinterpret_cast<const float4 *>(sp);
          for (int w = 0; w < nb / 8; ++w) {
            const float4 v = __ldg(s4 + w);
            mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
          }
        } else {
          for (int w = 0; w < nb / 2; ++w) mx = fmaxf(mx, fabsf(__ldg(sp + w)));
        }
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      if (half == 0) {
        // |q * sx| <= 127 * max sx; S_t scales the column into [-2^15, 2^15],
        // the top of the f16 normal range, so that blocks far below the
        // column's largest stay normal (full 11-bit precision in Bhi and Blo)
        const float S = __fmul_rn(pow2_ceil(127.0f * mx), 1.0f / 32768.0f);
        m.colS[c] = S;
        m.colInv[c] = 1.0f / S;
      }
    }
    // each weight row's largest scale byte
    if (!mbar_wait(smem_addr(m.scale_full), done & 1, p.status)) dead = true;
    if (ct < NM * kTcRows) {
      uint32_t m4 = 0;
      for (int w = 0; w < nb / 16; ++w) {
        const uint4 v = lds128(sscale + (uint32_t)ct * nb + 16u * w);
        m4 = __vmaxu4(__vmaxu4(m4, v.x), __vmaxu4(__vmaxu4(v.y, v.z), v.w));
      }
      m.umax[ct] = (int)max(max(m4 & 0xFFu, (m4 >> 8) & 0xFFu), max((m4 >> 16) & 0xFFu, m4 >> 24));
    }
    bar_sync_named(1, kConvThreads);
    for (int c = 0; c < nchunk; ++c, ++g) {
      const int rs = g % nraw, s = g % nf16;
      const uint32_t raw = sraw + (uint32_t)rs * p.raw_stage;
      const uint32_t st = sf16 + (uint32_t)s * p.f16_stage;
      if (!mbar_wait(smem_addr(&m.raw_full[rs]), (g / nraw) & 1, p.status)) dead = true;
      if (g >= nf16 && !mbar_wait(smem_addr(&m.f16_empty[s]), ((g / nf16) - 1) & 1, p.status)) dead = true;
      if (!dead) {
        // A: (matrix, row, half) -> 32 weights of one MX block, scaled by 2^(u - umax)
#pragma unroll
        for (int j = 0; j < NM; ++j) {
          const int q = ct + kConvThreads * j;
          const int mm = q >> 8, r = q & 127, h = (q >> 7) & 1;
          const uint4 pk = lds128(raw + (uint32_t)mm * kTcRows * kRawArow + (uint32_t)r * kRawArow + 16u * h);
          const int u = (int)lds_u8(sscale + (uint32_t)(mm * kTcRows + r) * nb + 2 * c + h);
          const uint32_t f1 = f16_pow2_neg(m.umax[mm * kTcRows + r] - u);
          const uint32_t f2 = f1 | (f1 << 16);
          const uint32_t pw[4] = {pk.x, pk.y, pk.z, pk.w};
#pragma unroll
          for (int wd = 0; wd < 4; ++wd) {
            uint32_t o[4];
            asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
                " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
                " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}\n"
                : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
                : "r"(pw[wd]));
#pragma unroll
            for (int i = 0; i < 4; ++i) asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(o[i]) : "r"(f2));
            sts128(st + (uint32_t)mm * kF16Mat + tile_offset(r, 32 * h + 8 * wd), make_uint4(o[0], o[1], o[2], o[3]));
          }
        }
        // B: (column, group of 8) -> v = q * sx / S_t as f16 hi + lo
        for (int q = ct; q < tl.ncol16 * 8; q += kConvThreads) {
          const int cc = q % tl.ncol16, grp = q / tl.ncol16;
          uint2 codes;
          asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(codes.x), "=r"(codes.y)
                       : "r"(raw + p.raw_b + (uint32_t)cc * kRawBrow + 8u * grp));
          const float fac = __fmul_rn(lds_f32(raw + p.raw_bs + (uint32_t)cc * 8u + 4u * (grp >> 2)), m.colInv[cc]);
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t wv = i < 2 ? codes.x : codes.y;
            const int sh = 16 * (i & 1);
            const float v0 = __fmul_rn((float)(int8_t)(wv >> sh), fac);
            const float v1 = __fmul_rn((float)(int8_t)(wv >> (sh + 8)), fac);
            asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(hi[i]) : "f"(v1), "f"(v0));
            float h0, h1;
            asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n cvt.f32.f16 %0, l;\n cvt.f32.f16 %1, h;\n}\n"
                : "=f"(h0), "=f"(h1) : "r"(hi[i]));
            asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(lo[i]) : "f"(__fsub_rn(v1, h1)), "f"(__fsub_rn(v0, h0)));
          }
          const uint32_t off = tile_offset(cc, 8 * grp);
          sts128(st + NM * kF16Mat + off, make_uint4(hi[0], hi[1], hi[2], hi[3]));
          sts128(st + NM * kF16Mat + kF16B + off, make_uint4(lo[0], lo[1], lo[2], lo[3]));
        }
      }
      fence_proxy_async();
      mbar_arrive(smem_addr(&m.f16_full[s]));
      bar_sync_named(1, kConvThreads);  // every converter is done with raw stage rs
      if (c + nraw < nchunk) issue_raw<NM>(p, maps, m, tl, raw, smem_addr(&m.raw_full[rs]), c + nraw, ct);
    }
    // ---------------------------------------------------------- epilogue
    if (warp < 4) {
      const bool ok = !dead && mbar_wait(smem_addr(m.acc_full), done & 1, p.status);
      tc_fence_after();
      const int i = 32 * warp + lane;  // weight row in the tile = TMEM lane
      const float rs0 = e8m0_value(m.umax[i]);
      const float rs1 = NM == 2 ? e8m0_value(m.umax[kTcRows + i]) : 0.0f;
      const int64_t orow = (int64_t)tl.mtile * kTcRows + i;
      for (int cb = 0; ok && cb < tl.ncol16; cb += 32) {
        float d0[32];
        tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)cb, d0);
        if (NM == 2) {
          float d1[32];
          tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)(kTcRows + cb), d1);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int col = cb + j;
            const int a = col < tl.ncols ? m.colasg[col] : -1;
            if (a >= 0) {
              const float S = m.colS[col];
              const float gv = __fmul_rn(__fmul_rn(d0[j], rs0), S), uv = __fmul_rn(__fmul_rn(d1[j], rs1), S);
              p.out[(int64_t)a * p.ld_out + orow] = __fmul_rn(silu(gv), uv);
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int col = cb + j;
            const int a = col < tl.ncols ? m.colasg[col] : -1;
            if (a >= 0) p.out[(int64_t)a * p.ld_out + orow] = __fmul_rn(__fmul_rn(d0[j], rs0), m.colS[col]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(m.acc_empty));
    }
    ++done;
    bar_sync_named(1, kConvThreads);  // the epilogue is done with this tile's tables
  }
  // all MMAs of this CTA have completed (the last epilogue waited for them)
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, NM * kTcRows);
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
// with boxes of box_cols bytes x 128 rows.
bool encode_rows(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint32_t box_cols) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {box_cols, (cuuint32_t)kTcRows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tc_expert_supported(int K, int N) { return K % 512 == 0 && K <= 8192 && N % kTcRows == 0; }

// Launch of the tensor-core path (moe_mxfp4_gateup_swiglu / moe_mxfp4_down for
// T > 16).  nm = 2: gate and up with SwiGLU; nm = 1: down.
moe_status launch_tc_expert(int nm, const int8_t *aq, int64_t ld_aq, const float *as, int64_t ld_as,
                            const uint8_t *w0, const uint8_t *s0, const uint8_t *w1, const uint8_t *s1,
                            const int32_t *offsets, const int32_t *sorted, int64_t cap, int A, int k, int E,
                            int K, int N, int bytoken, float *out, int64_t ld_out, cudaStream_t stream,
                            const char *name) {
  if (!tc_expert_supported(K, N))
    return fail(MOE_ERR_UNSUPPORTED, "%s: tensor path needs K %% 512 == 0 (<= 8192) and rows %% 128 == 0", name);
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
    if (!encode_rows(&maps.w[mm], mm == 0 ? w0 : w1, rows, (uint64_t)K / 2, kRawArow) ||
        !encode_rows(&maps.s[mm], mm == 0 ? s0 : s1, rows, (uint64_t)K / 32, (uint32_t)(K / 32)))
      return fail(MOE_ERR_UNSUPPORTED, "%s: tensor maps of the weights could not be built (16-byte aligned weights and scales are required)", name);
  }
  p.raw_b = (uint32_t)nm * kTcRows * kRawArow;
  p.raw_bs = p.raw_b + (uint32_t)kTcCols * kRawBrow;
  p.raw_stage = (p.raw_bs + (uint32_t)kTcCols * 8u + 127u) & ~127u;
  p.f16_stage = (uint32_t)nm * kF16Mat + 2 * kF16B;
  // operand stages first (deep enough to cover the MMA round trip), then the
  // tile's scales, then as many packed-input stages as shared memory holds
  const uint32_t scale_bytes = ((uint32_t)nm * kTcRows * (K / 32) + 127u) & ~127u;
  const size_t misc = tc_misc_bytes(E) + 128;
  int nf16 = kTcF16Max, nraw = 0;
  for (; nf16 >= 2; --nf16) {
    const size_t fixed = (size_t)nf16 * p.f16_stage + scale_bytes + misc;
    nraw = fixed < (size_t)optin ? (int)(((size_t)optin - fixed) / p.raw_stage) : 0;
    if (nraw >= 3) break;
  }
  if (nraw > kTcRawMax) nraw = kTcRawMax;
  if (nf16 < 2 || nraw < 2) return fail(MOE_ERR_UNSUPPORTED, "%s: tensor path does not fit shared memory", name);
  p.nf16 = nf16;
  p.nraw = nraw;
  p.off_f16 = 0;
  p.off_scale = (uint32_t)nf16 * p.f16_stage;
  p.off_raw = p.off_scale + scale_bytes;
  p.off_misc = p.off_raw + (uint32_t)nraw * p.raw_stage;
  const size_t smem = p.off_misc + tc_misc_bytes(E);
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
