// MXFP4 expert projections of calls of 1-16 rows (the exact-rows regime of
// "Optimizing DeepSeek V4 Flash Inference on a Strix Halo Pair", "The exact-
// rows contract"), and of the light experts of larger calls: gate/up
// (+SwiGLU) and down (+ the slot-ordered combine).
//
// The arithmetic per row and output is the layer's one-row arithmetic ("DeepSeek-
// V4-Flash on AMD gfx90a", §6.1): lane l takes the 32-element blocks l, l+32,
// ... of the output row, forms each exact integer block dot I_b from the
// E2M1 nibbles split by sign (dp4a against the Q8 codes), adds
// fma(I_b, xs_b * 2^(u_b-128), acc) in increasing block order, and the 32 lane
// sums meet in a fixed xor butterfly: the bits of the single-launch decode
// kernel and of the one-row call, whatever the number of rows.
//
// Work split (GB300-first): one persistent CTA per SM owns the same slice of
// output rows of every active expert.  A producer warp streams ring items
// through shared memory with cp.async.bulk (TMA): an item is half of an
// expert's slice (gate/up: both matrices) or the whole slice (down), with the
// first rows of the expert's activations staged beside it.  Four groups of
// seven consumer warps take every fourth item, so four items are computed at
// once; a warp takes one output row (gate/up) or two (down) at a time and
// reads the weights straight from the stage for each activation row.
#include "mx_device.cuh"

namespace moe {
namespace {

constexpr int kGroups = 4;
constexpr int kGroupWarps = 7;
constexpr int kConsWarps = kGroups * kGroupWarps;
constexpr int kKrowThreads = 32 * (kConsWarps + 1);  // + the producer warp
constexpr int kKrowMaxStages = 8;
// Staged activation rows are traded for ring stages until this many fit (four
// items computed, three loading): measured against five stages, the light
// experts of zipf-32 / zipf-64 gain 3%, 1-16-row calls are unchanged.
constexpr int kKrowStagesWanted = 7;
constexpr int kKrowMaxAct = 4;  // activation rows staged with an item, at most


enum KrowMode { kKGateUp = 0, kKGateUpRaw = 1, kKDown = 2 };

struct KrowArgs {
  const int8_t *aq;  // Q8 codes: x rows (gate/up, by token) or h rows (down, by assignment)
  int64_t ld_aq;
  const float *as;   // Q8 scales
  int64_t ld_as;
  const uint8_t *w0, *s0, *w1, *s1;  // [E][N][K/2] weights, [E][N][K/32] E8M0 bytes (w1/s1: up)
  const int32_t *offsets, *sorted;
  int64_t cap;
  int A, k, E, K, N;
  uint32_t kdiv;
  int max_rows;       // experts with more rows are left to the tensor-core kernel
  float *out0, *out1;
  int64_t ld_out;
  const float *wts;   // fused combine (down): [T][k] routing weights
  float *cout;        //   layer output [T][ld_cout]
  int64_t ld_cout;
  int T;
  int R;              // output rows per CTA (max)
  int nstage;
  uint32_t stage_bytes;
  uint32_t wreg, sreg;  // one matrix's weight / scale region in a stage
  uint32_t act_off;     // activation rows in a stage, from here
  uint32_t act_row;     // bytes of a staged activation row: K codes, then nb fp32 scales
  int armax;            // activation rows staged per item
  int s16, as16;        // weight scales / activation scales copyable in 16-byte pieces
  unsigned *status;
};

// Sign-split block dot of one 32-element block: dp - dn with the codes of the
// activation block (lo: elements 0..15, hi: 16..31) and 16 bytes of packed
// weights (the same terms as row_dot_stage_pn).
MOE_DEVFN int pn_block(const uint4 &lo, const uint4 &hi, const uint4 &w) {
  const uint32_t xw[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
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
  return dp - dn;
}

// NM weight rows (packed codes at wrow[m], E8M0 bytes at srow[m], shared
// memory) against one activation row, staged (codes in element order at
// xrow, then the block scales) or in global memory (xg, sg).
template <int NM, int S, bool STAGED>
MOE_DEVFN void krow_dot(uint32_t xrow, const int8_t *xg, const float *sg, int K, const uint32_t (&wrow)[NM],
                        const uint32_t (&srow)[NM], uint32_t tab, float (&acc)[NM]) {
  const int lane = threadIdx.x & 31;
  const int nb = K / 32;
#pragma unroll
  for (int m = 0; m < NM; ++m) acc[m] = 0.0f;
#pragma unroll
  for (int s = 0; s < S; ++s) {
    const int b = lane + 32 * s;
    if (b < nb) {
      uint4 lo, hi;
      float sx;
      if (STAGED) {
        lo = lds128(xrow + 32u * b);
        hi = lds128(xrow + 32u * b + 16u);
        sx = lds_f32(xrow + (uint32_t)K + 4u * b);
      } else {
        lo = ldg_nc(xg + 32 * b);
        hi = ldg_nc(xg + 32 * b + 16);
        sx = sg[b];
      }
#pragma unroll
      for (int m = 0; m < NM; ++m) {
        const int I = pn_block(lo, hi, lds128(wrow[m] + 16u * b));
        acc[m] = __fmaf_rn(__int2float_rn(I), __fmul_rn(sx, lds_f32(tab + 4u * lds_u8(srow[m] + b))), acc[m]);
      }
    }
  }
}

template <int MODE, int S, bool CMB>
__global__ void __launch_bounds__(kKrowThreads, 1) krow_kernel(const KrowArgs p) {
  constexpr int NM = MODE == kKDown ? 1 : 2;
  constexpr int NH = MODE == kKDown ? 1 : 2;  // items per expert (halves of the slice)
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int n_active;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n0 = (int)((int64_t)blockIdx.x * p.N / gridDim.x);
  const int n1 = (int)((int64_t)(blockIdx.x + 1) * p.N / gridDim.x);
  const int R = n1 - n0;
  const int K = p.K, nb = K / 32;
  const int NS = p.nstage;

  uint8_t *stages = smem;
  // A full barrier per (stage, group): the groups take every kGroups-th item
  // and the stages cycle with another period, so on one stage-wide barrier a
  // group could come to its phase while an earlier item of another group on
  // that stage has not landed, which a parity wait cannot tell apart.  Each
  // group waits on its own barriers in order; item it arms barrier
  // (it % NS, it % kGroups), phase it / lcm(NS, kGroups).
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)NS * p.stage_bytes);
  uint64_t *empty = full + NS * kGroups;
  const uint32_t stab = smem_addr(empty + NS);  // [256] e8m0_half table
  const int L = NS % kGroups == 0 ? NS : NS % 2 == 0 ? 2 * NS : kGroups * NS;  // lcm(NS, kGroups = 4)
  int *active = reinterpret_cast<int *>(empty + NS) + 256;  // [E]
  int *offs = active + p.E;                           // [E+1]
  float *ys = reinterpret_cast<float *>((reinterpret_cast<uintptr_t>(offs + p.E + 1) + 15) & ~uintptr_t(15));  // [A][R] (CMB)

  for (int i = tid; i <= p.E; i += blockDim.x) offs[i] = p.offsets[i];
  fill_e8m0_table(stab);
  if (tid == 0) {
    for (int s = 0; s < NS * kGroups; ++s) mbar_init(smem_addr(&full[s]), 33);  // 1 expect_tx + 32 cp.async arrives
    for (int s = 0; s < NS; ++s) mbar_init(smem_addr(&empty[s]), kGroupWarps);
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == 0) {
    // the experts with rows (and at most max_rows of them), increasing id
    int cnt = 0;
    const unsigned lt = (1u << lane) - 1u;
    for (int e0 = 0; e0 < p.E; e0 += 32) {
      const int e = e0 + lane;
      bool act_e = false;
      if (e < p.E) {
        const int64_t b = offs[e], en = offs[e + 1];
        const bool bad = b < 0 || en < b || en > p.cap;
        if (bad && p.status) atomicOr(p.status, MOE_DEV_BAD_ROW);
        act_e = !bad && en > b && en - b <= p.max_rows;
      }
      const unsigned m = __ballot_sync(0xffffffffu, act_e);
      if (act_e) active[cnt + __popc(m & lt)] = e;
      cnt += __popc(m);
    }
    if (lane == 0) n_active = cnt;
  }
  __syncthreads();
  const int nitem = n_active * NH;
  // rows [r0, r1) of the CTA slice that item it covers
  auto item_rows = [&](int it, int &r0, int &r1) {
    const int h = it % NH;
    r0 = h * R / NH;
    r1 = (h + 1) * R / NH;
  };
  // assignment and activation row of sorted position q (false: none)
  auto resolve = [&](int q, int &a, int &arow) -> bool {
    a = p.sorted[q];
    if (a < 0) return false;
    if (a >= p.A) {
      if (lane == 0 && p.status) atomicOr(p.status, MOE_DEV_BAD_ROW);
      return false;
    }
    arow = MODE == kKDown ? a : token_of(a, p.kdiv);
    return true;
  };

  if (warp == kConsWarps) {
    // ------------------------------------------------------------ producer
    const uint64_t wpol = policy_evict_first(), apol = policy_evict_last();
    int issued = 0;
    for (int it = 0; it < nitem; ++it) {
      const int st = it % NS;
      if (it >= NS && !mbar_wait(smem_addr(&empty[st]), ((it / NS) - 1) & 1, p.status)) break;
      const int e = active[it / NH];
      int r0, r1;
      item_rows(it, r0, r1);
      const uint32_t wbytes = (uint32_t)(r1 - r0) * (K / 2), sbytes = (uint32_t)(r1 - r0) * nb;
      const int64_t row0 = (int64_t)e * p.N + n0 + r0;
      const uint32_t sbase = smem_addr(stages + (size_t)st * p.stage_bytes);
      const uint32_t fb = smem_addr(&full[st * kGroups + it % kGroups]);
      const int seg_b = offs[e], nq = min(offs[e + 1] - seg_b, p.armax);
      // the staged activation rows: positions seg_b .. seg_b + nq - 1 (slot j
      // = position seg_b + j; a position without a valid assignment is skipped)
      int arow_l = -1;  // lane j < nq: the activation row of slot j, or -1
      if (lane < nq) {
        const int a = p.sorted[seg_b + lane];
        arow_l = (a >= 0 && a < p.A) ? (MODE == kKDown ? a : token_of(a, p.kdiv)) : -1;
      }
      const int nvalid = __popc(__ballot_sync(0xffffffffu, arow_l >= 0));
      if (lane == 0) {
        mbar_arrive_expect_tx(fb, NM * wbytes + (p.s16 ? NM * sbytes : 0u) +
                                      (uint32_t)nvalid * ((uint32_t)K + (p.as16 ? 4u * (uint32_t)nb : 0u)));
        bulk_g2s(sbase, p.w0 + row0 * (K / 2), wbytes, fb, wpol);
        if (NM == 2) bulk_g2s(sbase + p.wreg, p.w1 + row0 * (K / 2), wbytes, fb, wpol);
        if (p.s16) {
          bulk_g2s(sbase + NM * p.wreg, p.s0 + row0 * nb, sbytes, fb, wpol);
          if (NM == 2) bulk_g2s(sbase + NM * p.wreg + p.sreg, p.s1 + row0 * nb, sbytes, fb, wpol);
        }
      }
      for (int j = 0; j < nq; ++j) {
        const int ar = __shfl_sync(0xffffffffu, arow_l, j);
        if (ar < 0) continue;
        const uint32_t dst = sbase + p.act_off + (uint32_t)j * p.act_row;
        if (lane == 0) {
          bulk_g2s(dst, p.aq + (int64_t)ar * p.ld_aq, (uint32_t)K, fb, apol);
          if (p.as16) bulk_g2s(dst + (uint32_t)K, p.as + (int64_t)ar * p.ld_as, 4u * (uint32_t)nb, fb, apol);
        }
        if (!p.as16)
          for (int c = lane; c < nb; c += 32) cp_async4(dst + (uint32_t)K + 4u * c, p.as + (int64_t)ar * p.ld_as + c);
      }
      if (!p.s16) {
#pragma unroll
        for (int m = 0; m < NM; ++m) {
          const uint8_t *src = (m == 0 ? p.s0 : p.s1) + row0 * nb;
          const uint32_t dst = sbase + NM * p.wreg + m * p.sreg;
          for (uint32_t c = lane; c < sbytes / 4; c += 32) cp_async4(dst + 4 * c, src + 4 * c);
        }
      }
      cp_async_mbar_arrive_noinc(fb);
      issued = it + 1;
    }
    // never leave with copies in flight into this CTA's shared memory
    for (int it = issued > NS ? issued - NS : 0; it < issued; ++it)
      mbar_wait(smem_addr(&full[(it % NS) * kGroups + it % kGroups]), (it / L) & 1, p.status);
    return;
  }

  // -------------------------------------------------------------- consumers
  const int grp = warp / kGroupWarps, wig = warp - grp * kGroupWarps;
  auto put_down = [&](int a, int r, float v) {
    if (CMB) {
      ys[(int64_t)a * p.R + r] = v;
      if (p.out0) p.out0[(int64_t)a * p.ld_out + n0 + r] = v;
    } else {
      p.out0[(int64_t)a * p.ld_out + n0 + r] = v;
    }
  };
  for (int it = grp; it < nitem; it += kGroups) {
    const int st = it % NS;
    if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&full[st * kGroups + grp]), (it / L) & 1, p.status))) break;
    const int e = active[it / NH];
    int r0, r1;
    item_rows(it, r0, r1);
    const int nrow = r1 - r0;
    const int seg_b = offs[e], seg_e = offs[e + 1];
    const uint32_t sbase = smem_addr(stages + (size_t)st * p.stage_bytes);
    const uint32_t abase = sbase + p.act_off;
    if constexpr (MODE == kKDown) {
      // four output rows per warp, u + j nu (j < 4; each keeps its own
      // arithmetic, the activation loads serve all four); a row past the
      // slice repeats row u and is not written
      const int nu = (nrow + 3) >> 2;
      for (int u = wig; u < nu; u += kGroupWarps) {
        int rr[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) rr[j] = u + j * nu < nrow ? u + j * nu : u;
        uint32_t wrow[4], srow[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          wrow[j] = sbase + (uint32_t)rr[j] * (K / 2);
          srow[j] = sbase + p.wreg + (uint32_t)rr[j] * nb;
        }
#pragma unroll 1
        for (int q = seg_b; q < seg_e; ++q) {
          int a, arow;
          if (!resolve(q, a, arow)) continue;
          float acc[4];
          if (q - seg_b < p.armax)
            krow_dot<4, S, true>(abase + (uint32_t)(q - seg_b) * p.act_row, nullptr, nullptr, K, wrow, srow, stab, acc);
          else
            krow_dot<4, S, false>(0, p.aq + (int64_t)arow * p.ld_aq, p.as + (int64_t)arow * p.ld_as, K, wrow, srow, stab, acc);
          float y[4];
          reduce_pair(acc[0], acc[1], y[0], y[1]);
          reduce_pair(acc[2], acc[3], y[2], y[3]);
          if (lane == 0) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (j == 0 || rr[j] != u) put_down(a, r0 + rr[j], y[j]);
          }
        }
      }
    } else {
      for (int r = wig; r < nrow; r += kGroupWarps) {
        const uint32_t wrow[2] = {sbase + (uint32_t)r * (K / 2), sbase + p.wreg + (uint32_t)r * (K / 2)};
        const uint32_t srow[2] = {sbase + 2 * p.wreg + (uint32_t)r * nb, sbase + 2 * p.wreg + p.sreg + (uint32_t)r * nb};
#pragma unroll 1
        for (int q = seg_b; q < seg_e; ++q) {
          int a, arow;
          if (!resolve(q, a, arow)) continue;
          float acc[2];
          if (q - seg_b < p.armax)
            krow_dot<2, S, true>(abase + (uint32_t)(q - seg_b) * p.act_row, nullptr, nullptr, K, wrow, srow, stab, acc);
          else
            krow_dot<2, S, false>(0, p.aq + (int64_t)arow * p.ld_aq, p.as + (int64_t)arow * p.ld_as, K, wrow, srow, stab, acc);
          float g, u;
          reduce_pair(acc[0], acc[1], g, u);
          if (lane == 0) {
            const int64_t o = (int64_t)a * p.ld_out + n0 + r0 + r;
            if (MODE == kKGateUp) {
              p.out0[o] = __fmul_rn(silu(g), u);
            } else {
              p.out0[o] = g;
              p.out1[o] = u;
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&empty[st]));
  }
  if constexpr (CMB) {
    // every expert's y rows of this CTA's output rows are in shared memory:
    // out[t, n0 + r] = the slot-ordered combine (fma chain over the slots; a
    // slot of weight exactly 0 adds nothing), as the stand-alone combine
    bar_sync_named(1, kConsWarps * 32);
    for (int idx = tid; idx < p.T * p.R; idx += kConsWarps * 32) {
      const int t = idx / p.R, r = idx - t * p.R;
      if (r >= R) continue;
      const float *wt = p.wts + (int64_t)t * p.k;
      const float *yt = ys + (int64_t)t * p.k * p.R + r;
      float acc = wt[0] != 0.0f ? __fmul_rn(wt[0], yt[0]) : 0.0f;
      for (int j = 1; j < p.k; ++j)
        if (wt[j] != 0.0f) acc = __fmaf_rn(wt[j], yt[(int64_t)j * p.R], acc);
      p.cout[(int64_t)t * p.ld_cout + n0 + r] = acc;
    }
  }
}

}  // namespace

// Launch of the 1-16-row kernel (mode 0 gate/up + SwiGLU into out0, 1 gate
// into out0 and up into out1, 2 down into out0, with the combine into cout
// when cout is given).  Returns MOE_ERR_UNSUPPORTED, with nothing enqueued,
// when the shape does not fit its shared-memory plan.
moe_status launch_krow(int mode, const int8_t *aq, int64_t ld_aq, const float *as, int64_t ld_as, const uint8_t *w0,
                       const uint8_t *s0, const uint8_t *w1, const uint8_t *s1, const int32_t *offsets,
                       const int32_t *sorted, int64_t cap, int T, int k, int E, int K, int N, int max_rows,
                       float *out0, float *out1, int64_t ld_out, const float *wts, float *cout, int64_t ld_cout,
                       cudaStream_t stream, const char *name) {
  const int nm = mode == kKDown ? 1 : 2, nh = mode == kKDown ? 1 : 2;
  const int nb = K / 32;
  const int S = (nb + 31) / 32;
  if (S > 4) return fail(MOE_ERR_UNSUPPORTED, "%s: K=%d", name, K);
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_fail(err, name);
  int optin = 0;
  err = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (err != cudaSuccess) return cuda_fail(err, name);
  const int G = N < sm_count() ? N : sm_count();
  KrowArgs p{};
  p.aq = aq; p.ld_aq = ld_aq; p.as = as; p.ld_as = ld_as;
  p.w0 = w0; p.s0 = s0; p.w1 = w1; p.s1 = s1;
  p.offsets = offsets; p.sorted = sorted; p.cap = cap;
  p.A = T * k; p.k = k; p.E = E; p.K = K; p.N = N;
  p.kdiv = kdiv_of(k);
  p.max_rows = max_rows;
  p.out0 = out0; p.out1 = out1; p.ld_out = ld_out;
  p.wts = wts; p.cout = cout; p.ld_cout = ld_cout; p.T = T;
  p.status = device_status_word();
  p.R = (N + G - 1) / G;
  const int ritem = (p.R + nh - 1) / nh;
  p.wreg = (uint32_t)ritem * (K / 2);
  p.sreg = ((uint32_t)ritem * nb + 15u) & ~15u;
  p.act_off = nm * (p.wreg + p.sreg);
  p.act_row = (uint32_t)K + 4u * nb;
  p.s16 = (nb % 16) == 0 && (uintptr_t)s0 % 16 == 0 && (s1 == nullptr || (uintptr_t)s1 % 16 == 0);
  p.as16 = (uintptr_t)as % 16 == 0 && ld_as % 4 == 0;
  const bool cmb = mode == kKDown && cout != nullptr;
  const size_t fixed = (kGroups + 1) * 8 * kKrowMaxStages + 1024 + 4 * (size_t)(2 * E + 1) + 16 +
                       (cmb ? (size_t)p.A * p.R * 4 + 16 : 0) + 64;
  const size_t budget = (size_t)optin - 1024;
  if (budget < fixed) return fail(MOE_ERR_UNSUPPORTED, "%s: no shared-memory plan", name);
  // as many staged activation rows per item as leave kKrowStagesWanted
  // stages; else the plan with the most stages
  int best_ns = 0, best_ar = 0;
  uint32_t best_stage = 0;
  for (int ar = kKrowMaxAct; ar >= 1; --ar) {
    const uint32_t stage = (p.act_off + (uint32_t)ar * p.act_row + 127u) & ~127u;
    int ns = (int)((budget - fixed) / stage);
    if (ns > kKrowMaxStages) ns = kKrowMaxStages;
    if (ns > best_ns) {
      best_ns = ns;
      best_ar = ar;
      best_stage = stage;
    }
    if (ns >= kKrowStagesWanted) break;
  }
  if (best_ns < 2) return fail(MOE_ERR_UNSUPPORTED, "%s: no shared-memory plan", name);
  p.nstage = best_ns;
  p.armax = best_ar;
  p.stage_bytes = best_stage;
  const size_t smem = (size_t)best_ns * best_stage + fixed;
  if (smem > budget) return fail(MOE_ERR_UNSUPPORTED, "%s: no shared-memory plan (%zu bytes)", name, smem);
  void (*kern)(KrowArgs) = nullptr;
  if (mode == kKGateUp) kern = S == 1 ? krow_kernel<kKGateUp, 1, false> : S == 2 ? krow_kernel<kKGateUp, 2, false> : krow_kernel<kKGateUp, 4, false>;
  else if (mode == kKGateUpRaw) kern = S == 1 ? krow_kernel<kKGateUpRaw, 1, false> : S == 2 ? krow_kernel<kKGateUpRaw, 2, false> : krow_kernel<kKGateUpRaw, 4, false>;
  else if (cmb) kern = S == 1 ? krow_kernel<kKDown, 1, true> : S == 2 ? krow_kernel<kKDown, 2, true> : krow_kernel<kKDown, 4, true>;
  else kern = S == 1 ? krow_kernel<kKDown, 1, false> : S == 2 ? krow_kernel<kKDown, 2, false> : krow_kernel<kKDown, 4, false>;
  const moe_status ast = ensure_smem_attr(reinterpret_cast<const void *>(kern), (int)budget, name);
  if (ast != MOE_OK) return ast;
  kern<<<G, kKrowThreads, smem, stream>>>(p);
  err = cudaGetLastError();
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, name);
}

}  // namespace moe
