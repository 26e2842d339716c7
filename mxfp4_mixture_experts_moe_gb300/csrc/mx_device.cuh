// Device arithmetic shared by every kernel of the layer.  Each step of the
// layer has exactly one implementation here, so the stand-alone stage kernels
// and the fused decode kernel compute the same bits for every row.
#pragma once

#include <math_constants.h>

#include "common.cuh"

namespace moe {

// ------------------------------------------------------------------ misc

MOE_DEVFN void bar_sync_named(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
MOE_DEVFN float lds_f32(uint32_t addr) {
  float r;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(r) : "r"(addr));
  return r;
}
MOE_DEVFN uint32_t lds_u32(uint32_t addr) {
  uint32_t r;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(r) : "r"(addr));
  return r;
}
MOE_DEVFN int lds_s32(uint32_t addr) {
  int r;
  asm volatile("ld.shared.s32 %0, [%1];" : "=r"(r) : "r"(addr));
  return r;
}
MOE_DEVFN void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
MOE_DEVFN void sts32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

MOE_DEVFN float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
MOE_DEVFN float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ------------------------------------------------------------------ router

// 8 consecutive bf16 / fp32 values from shared memory, widened exactly.
MOE_DEVFN void load8_smem(uint32_t addr, bool bf16, float (&v)[8]) {
  if (bf16) {
    const uint4 r = lds128(addr);
    v[0] = bf16_lo(r.x); v[1] = bf16_hi(r.x); v[2] = bf16_lo(r.y); v[3] = bf16_hi(r.y);
    v[4] = bf16_lo(r.z); v[5] = bf16_hi(r.z); v[6] = bf16_lo(r.w); v[7] = bf16_hi(r.w);
  } else {
    const uint4 a = lds128(addr), b = lds128(addr + 16);
    v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y); v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
    v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y); v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
  }
}


// Top-k of one token, one warp.  score = logit (+ bias); the k largest
// scores are taken in descending order, equal scores by lower expert id, and
// a NaN score is never taken (an id of 0x7fffffff marks a slot that only NaN
// scores were left for).  Weights: sigmoid of the selected scores over their
// sum, added in slot order.  Every lane returns the same ids/weights.
MOE_DEVFN float topk_score(const float *logits_row, const float *bias, int e) {
  const float v = logits_row[e];
  return bias ? __fadd_rn(v, bias[e]) : v;
}

// Order-preserving key of a float score (larger score -> larger key, every
// real score > 0); -0 is first turned into +0 so that the keys tie exactly
// where the scores compare equal.  NaN gets key 0, "absent".
MOE_DEVFN uint32_t score_key(float v) {
  if (v != v) return 0u;
  const uint32_t u = __float_as_uint(__fadd_rn(v, 0.0f));
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
MOE_DEVFN float key_score(uint32_t key) {  // inverse of score_key on real scores
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// S = scores per lane (expert lane + 32 s); E <= 32 * S.  Each lane reads its
// scores once, then every round is register work: the lane's best key (the
// first of equal keys has the lower id), the warp's largest key, and the
// lowest id holding it.  Used for large S.
template <int S>
MOE_DEVFN void topk_warp_scan(const float *logits_row, const float *bias, int E, int k, int (&ids)[8], float (&w)[8]) {
  const int lane = threadIdx.x & 31;
  uint32_t key[S];
#pragma unroll
  for (int s = 0; s < S; ++s) {
    const int e = lane + 32 * s;
    key[s] = e < E ? score_key(topk_score(logits_row, bias, e)) : 0u;
  }
  float sel[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    ids[j] = 0;
    sel[j] = 0.0f;
  }
#pragma unroll 1
  for (int j = 0; j < k; ++j) {
    uint32_t bk = 0u;
    int bi = 0x7fffffff;
#pragma unroll
    for (int s = 0; s < S; ++s) {
      if (key[s] > bk) {
        bk = key[s];
        bi = lane + 32 * s;
      }
    }
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, bk);
    const int win = (int)__reduce_min_sync(0xffffffffu, bk == kmax ? (uint32_t)bi : 0xffffffffu);
#pragma unroll
    for (int s = 0; s < S; ++s)
      if (lane + 32 * s == win) key[s] = 0u;
    const float ws = kmax ? key_score(kmax) : -CUDART_INF_F;
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      if (jj == j) {
        ids[jj] = win;
        sel[jj] = ws;
      }
    }
  }
  float total = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < k) {
      sel[j] = __frcp_rn(__fadd_rn(1.0f, expf(-sel[j])));
      total = __fadd_rn(total, sel[j]);
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) w[j] = j < k ? __fdiv_rn(sel[j], total) : 0.0f;
}

// The same selection for small S: each lane first sorts its S entries by
// (key desc, id asc) with a stable odd-even transposition sort, so a round
// only reads the lane's head entry, and the winning lane pops it.  Slot j's
// id and score stay in lane j; the weights are formed there (the sum over
// the slots is taken in slot order, as in topk_warp_scan) and broadcast.
template <int S>
MOE_DEVFN void topk_warp_sorted(const float *logits_row, const float *bias, int E, int k, int (&ids)[8],
                                float (&w)[8]) {
  const int lane = threadIdx.x & 31;
  uint32_t key[S];
  int kid[S];
#pragma unroll
  for (int s = 0; s < S; ++s) {
    const int e = lane + 32 * s;
    key[s] = e < E ? score_key(topk_score(logits_row, bias, e)) : 0u;
    kid[s] = e;
  }
#pragma unroll
  for (int pass = 0; pass < S; ++pass) {
#pragma unroll
    for (int s = pass & 1; s + 1 < S; s += 2) {
      if (key[s + 1] > key[s]) {  // strict: equal keys keep their id order
        const uint32_t tk = key[s];
        key[s] = key[s + 1];
        key[s + 1] = tk;
        const int ti = kid[s];
        kid[s] = kid[s + 1];
        kid[s + 1] = ti;
      }
    }
  }
  int my_id = 0;
  float my_sel = 0.0f;
#pragma unroll 1
  for (int j = 0; j < k; ++j) {
    const uint32_t bk = key[0];
    const int bi = bk ? kid[0] : 0x7fffffff;
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, bk);
    const int win = (int)__reduce_min_sync(0xffffffffu, bk == kmax ? (uint32_t)bi : 0xffffffffu);
    if (bk == kmax && bi == win) {
#pragma unroll
      for (int s = 0; s + 1 < S; ++s) {
        key[s] = key[s + 1];
        kid[s] = kid[s + 1];
      }
      key[S - 1] = 0u;
    }
    if (lane == j) {
      my_id = win;
      my_sel = kmax ? key_score(kmax) : -CUDART_INF_F;
    }
  }
  const float sg = __frcp_rn(__fadd_rn(1.0f, expf(-my_sel)));
  float total = 0.0f;
#pragma unroll 1
  for (int j = 0; j < k; ++j) total = __fadd_rn(total, __shfl_sync(0xffffffffu, sg, j));
  const float my_w = __fdiv_rn(sg, total);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    ids[j] = j < k ? __shfl_sync(0xffffffffu, my_id, j) : 0;
    w[j] = j < k ? __shfl_sync(0xffffffffu, my_w, j) : 0.0f;
  }
}

// Top-k in two stages for latency: stage 1, one warp per 32 consecutive
// experts, takes that group's k best (score desc, id asc) by k rounds of warp
// max; stage 2, one warp per token, merges the groups' lists the same way.
// The selection order, the ids (0x7fffffff for a slot only NaN scores were
// left for) and the weights are those of topk_warp_sorted: the best entry of
// the union is the best entry of the group that holds it.
// Stage 1 of expert group g (32 g .. 32 g + 31) of one token: writes k
// (key, id) pairs to ck/ci.
MOE_DEVFN void topk_group_stage(const float *logits_row, const float *bias, int E, int k, int g, uint32_t *ck,
                                int *ci) {
  const int lane = threadIdx.x & 31;
  const int e = 32 * g + lane;
  uint32_t key = e < E ? score_key(topk_score(logits_row, bias, e)) : 0u;
#pragma unroll 1
  for (int j = 0; j < k; ++j) {
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
    const int wl = __ffs(__ballot_sync(0xffffffffu, key == kmax)) - 1;  // lowest id holding it
    if (lane == 0) {
      ck[j] = kmax;
      ci[j] = kmax ? 32 * g + wl : 0x7fffffff;
    }
    if (lane == wl) key = 0u;
  }
}

struct NoPick {
  MOE_DEVFN void operator()(int, int) const {}
};

// Stage 2: merge of n <= 64 (key, id) pairs into the k slots and weights
// (every lane returns them).  on_pick(j, id) is called by every lane as soon
// as slot j is decided (id 0x7fffffff: only NaN scores were left).
template <class Pick = NoPick>
MOE_DEVFN void topk_merge_stage(const uint32_t *ck, const int *ci, int n, int k, int (&ids)[8], float (&w)[8],
                                Pick on_pick = Pick()) {
  const int lane = threadIdx.x & 31;
  uint32_t ka = lane < n ? ck[lane] : 0u, kb = lane + 32 < n ? ck[lane + 32] : 0u;
  int ia = lane < n ? ci[lane] : 0x7fffffff, ib = lane + 32 < n ? ci[lane + 32] : 0x7fffffff;
  int my_id = 0;
  float my_sel = 0.0f;
#pragma unroll 1
  for (int j = 0; j < k; ++j) {
    const bool a_first = ka > kb || (ka == kb && ia < ib);
    const uint32_t bk = a_first ? ka : kb;
    const int bi = a_first ? ia : ib;
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, bk);
    const int win = (int)__reduce_min_sync(0xffffffffu, bk == kmax ? (uint32_t)bi : 0xffffffffu);
    if (ka == kmax && ia == win) {
      ka = 0u;
      ia = 0x7fffffff;
    } else if (kb == kmax && ib == win) {
      kb = 0u;
      ib = 0x7fffffff;
    }
    if (lane == j) {
      my_id = kmax ? win : 0x7fffffff;
      my_sel = kmax ? key_score(kmax) : -CUDART_INF_F;
    }
    on_pick(j, kmax ? win : 0x7fffffff);
  }
  const float sg = __frcp_rn(__fadd_rn(1.0f, expf(-my_sel)));
  float total = 0.0f;
#pragma unroll 1
  for (int j = 0; j < k; ++j) total = __fadd_rn(total, __shfl_sync(0xffffffffu, sg, j));
  const float my_w = __fdiv_rn(sg, total);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    ids[j] = j < k ? __shfl_sync(0xffffffffu, my_id, j) : 0;
    w[j] = j < k ? __shfl_sync(0xffffffffu, my_w, j) : 0.0f;
  }
}

MOE_DEVFN void topk_warp(const float *logits_row, const float *bias, int E, int k, int (&ids)[8], float (&w)[8]) {
  if (E <= 64) topk_warp_sorted<2>(logits_row, bias, E, k, ids, w);
  else if (E <= 256) topk_warp_sorted<8>(logits_row, bias, E, k, ids, w);
  else topk_warp_scan<32>(logits_row, bias, E, k, ids, w);
}

// ------------------------------------------------------------------ Q8

// Q8 of one block of 32 values: scale = amax/127 (IEEE), q = rne(v * (1/scale))
// clamped to +-127.  Returns the scale; codes packed 4 per word, element 0 in
// the low byte; *sum = the exact sum of the 32 codes.
MOE_DEVFN float q8_block(const float (&v)[32], uint32_t (&packed)[8], int *sum) {
  float amax = 0.0f;
#pragma unroll
  for (int l = 0; l < 32; ++l) amax = fmaxf(amax, fabsf(v[l]));
  const float d = __fdiv_rn(amax, 127.0f);
  const float inv = d > 0.0f ? __frcp_rn(d) : 0.0f;
  int s = 0;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int qi = __float2int_rn(__fmul_rn(v[4 * c + j], inv));
      qi = max(-127, min(127, qi));
      s += qi;
      word |= (uint32_t)(qi & 0xFF) << (8 * j);
    }
    packed[c] = word;
  }
  if (sum) *sum = s;
  return d;
}

// ------------------------------------------------------------------ MXFP4 dots

// silu(g) = g / (1 + exp(-g)) with the fast exp and divide (for g < -87 the
// divide returns 0, the limit of silu).
MOE_DEVFN float silu(float g) { return __fdividef(g, __fadd_rn(1.0f, __expf(-g))); }

MOE_DEVFN int block_sum8(const uint4 &lo, const uint4 &hi) {
  int s = 0;
  s = __dp4a((int)lo.x, 0x01010101, s);
  s = __dp4a((int)lo.y, 0x01010101, s);
  s = __dp4a((int)lo.z, 0x01010101, s);
  s = __dp4a((int)lo.w, 0x01010101, s);
  s = __dp4a((int)hi.x, 0x01010101, s);
  s = __dp4a((int)hi.y, 0x01010101, s);
  s = __dp4a((int)hi.z, 0x01010101, s);
  s = __dp4a((int)hi.w, 0x01010101, s);
  return s;
}

// The blocks b = lane + 32 s of one output row of NM matrices, taken from a
// shared-memory stage (matrix m's rows start at wbase + m*wstride, its E8M0
// bytes at sbase + m*sstride), converted once: wq = 12 + 2*E2M1 value per
// byte, ws = 2^(u-128).
template <int NM, int S>
MOE_DEVFN void load_weights(uint32_t wbase, uint32_t wstride, uint32_t sbase, uint32_t sstride, int r, int K,
                            uint32_t (&wq)[NM][S][8], float (&ws)[NM][S]) {
  const int lane = threadIdx.x & 31;
  const int nb = K / 32;
#pragma unroll
  for (int m = 0; m < NM; ++m) {
#pragma unroll
    for (int s = 0; s < S; ++s) {
      const int b = lane + 32 * s;
      if (b < nb) {
        const uint4 raw = lds128(wbase + m * wstride + (uint32_t)r * (K / 2) + 16u * b);
        e2m1x8_to_off12(raw.x, wq[m][s][0], wq[m][s][1]);
        e2m1x8_to_off12(raw.y, wq[m][s][2], wq[m][s][3]);
        e2m1x8_to_off12(raw.z, wq[m][s][4], wq[m][s][5]);
        e2m1x8_to_off12(raw.w, wq[m][s][6], wq[m][s][7]);
        ws[m][s] = e8m0_half(lds_u8(sbase + m * sstride + (uint32_t)r * nb + b));
      }
    }
  }
}

// Block term of one activation block against the converted weights:
// acc[m] = fma(float(I_b), sx * ws, acc[m]), I_b = dot(x, 12 + 2v) - 12*sum(x).
template <int NM, int S>
MOE_DEVFN void block_terms(int s, const uint4 &lo, const uint4 &hi, float sx, int xsum,
                           const uint32_t (&wq)[NM][S][8], const float (&ws)[NM][S], float (&acc)[NM]) {
  const uint32_t xw[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
  for (int m = 0; m < NM; ++m) {
    int d = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) d = __dp4a((int)xw[j], (int)wq[m][s][j], d);
    const int I = d - 12 * xsum;
    acc[m] = __fmaf_rn(__int2float_rn(I), __fmul_rn(sx, ws[m][s]), acc[m]);
  }
}

// An activation row staged in shared memory: the K codes as two planes of
// 16-byte half blocks (first halves of all blocks, then second halves), then
// nb fp32 scales, then nb int32 block sums.  Row size K + 8*nb bytes.
template <int NM, int S>
MOE_DEVFN void row_dot_smem(uint32_t row, int K, const uint32_t (&wq)[NM][S][8], const float (&ws)[NM][S],
                            float (&acc)[NM]) {
  const int lane = threadIdx.x & 31;
  const int nb = K / 32;
#pragma unroll
  for (int m = 0; m < NM; ++m) acc[m] = 0.0f;
#pragma unroll
  for (int s = 0; s < S; ++s) {
    const int b = lane + 32 * s;
    if (b < nb) {
      const uint4 lo = lds128(row + 16u * b), hi = lds128(row + 16u * (nb + b));
      const float sx = lds_f32(row + (uint32_t)K + 4u * b);
      const int xsum = lds_s32(row + (uint32_t)K + 4u * (nb + b));
      block_terms<NM, S>(s, lo, hi, sx, xsum, wq, ws, acc);
    }
  }
}

// 8 E2M1 codes -> twice their magnitudes, split by sign: pos holds 2|v| for
// positive codes and 0 for negative ones, neg the reverse, so that
// dot(x, 2v) = dot(x, pos) - dot(x, neg).  One byte-permute lookup per 4
// codes and sign (a set selector top bit replicates the table byte's zero sign
// bit); the high halves come down with shifts on the integer-logic pipe (the
// multiply pipe is already the busier one: it carries the dp4a).  For weights
// used by one row.
MOE_DEVFN void e2m1x8_pos_neg(uint32_t w, uint32_t &p_lo, uint32_t &p_hi, uint32_t &n_lo, uint32_t &n_hi) {
  const uint32_t T0 = 0x03020100u, T1 = 0x0C080604u;  // {0,1,2,3 | 4,6,8,12}
  const uint32_t wx = w ^ 0x88888888u;
  p_lo = prmt(T0, T1, w);
  p_hi = prmt(T0, T1, w >> 16);
  n_lo = prmt(T0, T1, wx);
  n_hi = prmt(T0, T1, wx >> 16);
}

// row_dot_smem with packed weights decoded by sign (no block sums needed).
// The integer block dots, and so every result, equal row_dot_smem's.
template <int NM, int S>
MOE_DEVFN void row_dot_smem_pn(uint32_t row, int K, const uint4 (&wr)[NM][S], const float (&ws)[NM][S],
                               float (&acc)[NM]) {
  const int lane = threadIdx.x & 31;
  const int nb = K / 32;
#pragma unroll
  for (int m = 0; m < NM; ++m) acc[m] = 0.0f;
#pragma unroll
  for (int s = 0; s < S; ++s) {
    const int b = lane + 32 * s;
    if (b < nb) {
      const uint4 lo = lds128(row + 16u * b), hi = lds128(row + 16u * (nb + b));
      const float sx = lds_f32(row + (uint32_t)K + 4u * b);
      const uint32_t xw[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
      for (int m = 0; m < NM; ++m) {
        const uint32_t wv[4] = {wr[m][s].x, wr[m][s].y, wr[m][s].z, wr[m][s].w};
        int dp = 0, dn = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t pl, ph, nl, nh;
          e2m1x8_pos_neg(wv[j], pl, ph, nl, nh);
          dp = __dp4a((int)xw[2 * j], (int)pl, dp);
          dp = __dp4a((int)xw[2 * j + 1], (int)ph, dp);
          dn = __dp4a((int)xw[2 * j], (int)nl, dn);
          dn = __dp4a((int)xw[2 * j + 1], (int)nh, dn);
        }
        acc[m] = __fmaf_rn(__int2float_rn(dp - dn), __fmul_rn(sx, ws[m][s]), acc[m]);
      }
    }
  }
}

// The same from a row of codes and scales in global memory.
template <int NM, int S>
MOE_DEVFN void row_dot_global(const int8_t *xr, const float *sr, int K, const uint32_t (&wq)[NM][S][8],
                              const float (&ws)[NM][S], float (&acc)[NM]) {
  const int lane = threadIdx.x & 31;
  const int nb = K / 32;
#pragma unroll
  for (int m = 0; m < NM; ++m) acc[m] = 0.0f;
#pragma unroll
  for (int s = 0; s < S; ++s) {
    const int b = lane + 32 * s;
    if (b < nb) {
      const uint4 lo = ldg_nc(xr + 32 * b), hi = ldg_nc(xr + 32 * b + 16);
      block_terms<NM, S>(s, lo, hi, sr[b], block_sum8(lo, hi), wq, ws, acc);
    }
  }
}

// The 256 values e8m0_half(u) as a table in shared memory (1 KB at tab), so
// that the hot loops turn a scale byte into its factor with one load instead
// of the integer decode.  The block's threads write the entries; the caller
// synchronises before the first use.
MOE_DEVFN void fill_e8m0_table(uint32_t tab) {
  for (uint32_t u = threadIdx.x; u < 256u; u += blockDim.x) sts32(tab + 4u * u, __float_as_uint(e8m0_half(u)));
}

// NM weight rows read block by block from shared memory (not preloaded into
// registers) against one staged activation row: the form for weights that
// are used by one activation row only.  wrow[m] / srow[m]: shared addresses of
// row m's packed codes and scale bytes; tab: the e8m0_half table (TAB), or
// unused (the scale bytes decoded in registers, for instantiations where the
// table's extra loads would cost register spills).  Same terms, same order
// per lane as row_dot_smem_pn.
template <int NM, int S, bool TAB = true>
MOE_DEVFN void row_dot_stage_pn(uint32_t xrow, int K, const uint32_t (&wrow)[NM], const uint32_t (&srow)[NM],
                                uint32_t tab, float (&acc)[NM]) {
  const int lane = threadIdx.x & 31;
  const int nb = K / 32;
#pragma unroll
  for (int m = 0; m < NM; ++m) acc[m] = 0.0f;
#pragma unroll
  for (int s = 0; s < S; ++s) {
    const int b = lane + 32 * s;
    if (b < nb) {
      const uint4 lo = lds128(xrow + 16u * b), hi = lds128(xrow + 16u * (nb + b));
      const float sx = lds_f32(xrow + (uint32_t)K + 4u * b);
      const uint32_t xw[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
      for (int m = 0; m < NM; ++m) {
        const uint4 w = lds128(wrow[m] + 16u * b);
        const uint32_t u = lds_u8(srow[m] + b);
        const float ws = TAB ? lds_f32(tab + 4u * u) : e8m0_half(u);
        const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
        int dp = 0, dn = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t pl, ph, nl, nh;
          e2m1x8_pos_neg(wv[j], pl, ph, nl, nh);
          dp = __dp4a((int)xw[2 * j], (int)pl, dp);
          dp = __dp4a((int)xw[2 * j + 1], (int)ph, dp);
          dn = __dp4a((int)xw[2 * j], (int)nl, dn);
          dn = __dp4a((int)xw[2 * j + 1], (int)nh, dn);
        }
        acc[m] = __fmaf_rn(__int2float_rn(dp - dn), __fmul_rn(sx, ws), acc[m]);
      }
    }
  }
}

// Butterfly of two per-lane sums at once: lanes 0-15 finish the first, 16-31
// the second, each with exactly the pairs and association of its own full
// xor butterfly (so the bits equal two separate butterflies).  Lane 0 returns
// (first, second).
MOE_DEVFN void reduce_pair(float a, float b, float &first, float &second) {
  const int lane = threadIdx.x & 31;
  const bool upper = (lane & 16) != 0;
  float keep = upper ? b : a;
  const float send = upper ? a : b;
  keep = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, 16));
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) keep = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, keep, o));
  first = keep;
  second = __shfl_xor_sync(0xffffffffu, keep, 16);
}

MOE_DEVFN float reduce_one(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Loads that bypass L1 (data written by other CTAs of the same grid).
MOE_DEVFN float ldcg_f32(const float *p) {
  float r;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(r) : "l"(p));
  return r;
}
MOE_DEVFN uint4 ldcg_v4(const void *p) {
  uint4 r;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// Stage one activation row from global Q8 codes + scales into the shared
// layout above, computing the block sums.  Lanes of the calling threads take
// blocks idx0, idx0+stride, ...
MOE_DEVFN void stage_q8_block(uint32_t row, int K, int b, const int8_t *src_codes, float scale) {
  const int nb = K / 32;
  const uint4 lo = ldg_nc(src_codes + 32 * b), hi = ldg_nc(src_codes + 32 * b + 16);
  sts128(row + 16u * b, lo);
  sts128(row + 16u * (nb + b), hi);
  sts32(row + (uint32_t)K + 4u * b, __float_as_uint(scale));
  sts32(row + (uint32_t)K + 4u * (nb + b), (uint32_t)block_sum8(lo, hi));
}

}  // namespace moe
