// MXFP4 expert projections against Q8 activations: gate/up (+SwiGLU) and down.
//
// Follows the decode route of "DeepSeek-V4-Flash on AMD gfx90a", §6.1: packed
// 4-bit weights read without any offline expansion, E2M1 nibbles turned into
// the small integers 0, ±1, ±2, ±3, ±4, ±6, ±8, ±12, an exact integer dot per
// block of 32, then activation and E8M0 scaling; and "Optimizing DeepSeek V4
// Flash Inference on a Strix Halo Pair", "MXFP4 routed-expert kernels" and
// "The exact-rows contract": one weight pass serves every resident row of an
// expert and every row keeps the one-row arithmetic.
//
// Work split (GB300-first): the grid is one persistent CTA per SM.  CTA c owns
// the same contiguous slice of output rows [n0, n1) of EVERY expert that has
// assignments, so the bytes each SM streams are equal whatever the routing.
// A producer warp streams the CTA's slice of each active expert, one expert
// per stage, into a ring of shared-memory stages with cp.async.bulk (TMA) for
// the packed weights and cp.async for the E8M0 bytes, completing on mbarriers.
// Consumer warps take one output row at a time: lane l owns the 16-byte
// blocks l, l+32, ... of the row (exactly one MX block each), converts the
// nibbles once, then loops over the expert's rows.
//
// Per row and output, the arithmetic is fixed: lane l accumulates its blocks
// in increasing order, acc = fma(float(I_b), xs_b * 2^(u_b-128), acc); the 32
// lane sums are combined by a fixed xor butterfly.  Nothing depends on how
// many rows the call has, so a T-row call reproduces T one-row calls bit for
// bit.
#include "mx_device.cuh"

namespace moe {
namespace {

enum Mode { kGateUpSwiglu = 0, kGateUpRaw = 1, kDown = 2 };

struct MxArgs {
  const int8_t *aq;  // Q8 activation codes: x rows (gate/up, by token) or h rows (down, by assignment)
  int64_t ld_aq;
  const float *as;   // Q8 scales
  int64_t ld_as;
  const uint8_t *w0, *s0;  // gate (or down) weights / E8M0 bytes, [E][N][K/2] / [E][N][K/32]
  const uint8_t *w1, *s1;  // up weights / bytes (gate/up only)
  const int32_t *offsets;  // [E+1]
  const int32_t *sorted;   // [cap]
  int64_t cap;
  int A, k, E;
  int K;  // reduction length
  int N;  // output rows per expert
  int n_act;          // activation rows: T (gate/up) or A (down)
  uint32_t kdiv;      // kdiv_of(k): token of assignment a = token_of(a, kdiv)
  float *out0, *out1;
  int64_t ld_out;
  // fused combine (down only): out[t] = slot-ordered combine of the y rows,
  // which stay in shared memory (out0, the y rows in global memory, optional)
  const float *wts;   // [T][k] routing weights
  float *cout;        // [T][ld_cout] layer output
  int64_t ld_cout;
  int T;
  int R;              // output rows per CTA (max)
  int nstage;
  uint32_t stage_bytes;
  uint32_t wreg;      // bytes of one matrix's weight slice region in a stage
  uint32_t sreg;      // bytes of one matrix's scale slice region (16-aligned)
  int scale16;        // scale rows are whole 16-byte chunks at 16-byte aligned addresses
  int rowtab;         // sorted positions (< cap <= kRowTab) get their activation row from shared memory
  int act_smem;       // all activation rows are staged in shared memory
  int win_rows;       // else (if > 0): the rows of each expert are staged in passes of this many (two buffers)
  int max_rows;       // experts with more rows than this are left to the tensor-core kernel
  uint32_t act_row_bytes;  // K codes (two half-block planes) + nb scales + nb block sums
  unsigned *status;
};

constexpr int kRowTab = 4096;
// Activation rows per pass when not every row fits shared memory (two
// buffers of this many rows; what is left of shared memory goes to the ring).
#ifndef MOE_WIN_ROWS
#define MOE_WIN_ROWS 8
#endif
constexpr int kWinRows = MOE_WIN_ROWS;

// Shared-memory layout (dynamic):
//   [nstage weight stages][full bars][empty bars][active: E][offs: E+1]
//   [rowtab: cap ints, if used][activation rows: all of them, or a window]
// An activation row holds the K Q8 codes as two planes of 16-byte half
// blocks (first halves of all blocks, then second halves: lanes reading
// consecutive blocks hit consecutive 16-byte bank groups), then nb fp32
// scales, then nb int32 block sums.  When not every activation row fits,
// the rows of each expert are taken in passes of at most win_rows rows, in
// two window buffers: the rows of pass i+1 are copied (cp.async) while pass
// i is computed, and each thread adds the block sums of the blocks it
// copied once its copies have landed; one barrier per pass hands both
// buffers over.
// WIN: the activation rows of each expert are staged in window passes; CMB
// (down only): the CTA keeps its y rows in shared memory and ends with the
// slot-ordered combine of its output rows ("DeepSeek-V4-Flash on AMD
// gfx90a", §8.2 down consumer: FP32 top-k partials and a fixed reduction).
// Each is a separate instantiation, so the kernel of the other cases keeps
// its own tight loop.
template <int MODE, int S, bool WIN, bool CMB = false>
__global__ void __launch_bounds__(512, 1) mx_expert_kernel(const MxArgs p) {
  constexpr int NM = (MODE == kDown) ? 1 : 2;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int n_active;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ncons = (blockDim.x >> 5) - 1;
  const int n0 = (int)((int64_t)blockIdx.x * p.N / gridDim.x);
  const int n1 = (int)((int64_t)(blockIdx.x + 1) * p.N / gridDim.x);
  const int R = n1 - n0;
  const int nb = p.K / 32;
  const int nstage = p.nstage;

  uint8_t *stages = smem;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)nstage * p.stage_bytes);
  uint64_t *empty = full + nstage;
  const uint32_t stab = smem_addr(empty + nstage);        // [256] e8m0_half table
  int *active = reinterpret_cast<int *>(empty + nstage) + 256;  // [E] active experts, in id order
  int *offs = active + p.E;                               // [E+1] copy of offsets
  int *rowtab = offs + p.E + 1;                           // [cap] activation row per sorted position
  uint8_t *act = reinterpret_cast<uint8_t *>(rowtab + (p.rowtab ? p.cap : 0));
  act = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(act) + 15) & ~uintptr_t(15));
  const uint32_t act_base = smem_addr(act);
  float *ys = reinterpret_cast<float *>(act + (p.act_smem ? (size_t)p.n_act * p.act_row_bytes : 0));  // [A][R] (CMB)

  // Stage the expert offsets in one parallel pass, then list the experts
  // that own rows (ballot compaction keeps increasing id order).
  for (int i = tid; i <= p.E; i += blockDim.x) offs[i] = p.offsets[i];
  fill_e8m0_table(stab);
  if (tid == 0) {
    for (int s = 0; s < nstage; ++s) {
      mbar_init(smem_addr(&full[s]), 33);  // 1 expect_tx arrive + 32 cp.async arrives
      mbar_init(smem_addr(&empty[s]), ncons);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == 0) {
    int cnt = 0;
    const unsigned lt = (1u << lane) - 1u;
    for (int e0 = 0; e0 < p.E; e0 += 32) {
      const int e = e0 + lane;
      bool act_e = false;
      if (e < p.E) {
        const int64_t b = offs[e], en = offs[e + 1];
        const bool bad = b < 0 || en < b || en > p.cap;
        if (bad && p.status) atomicOr(p.status, MOE_DEV_BAD_ROW);
        act_e = !bad && en > b && en - b <= p.max_rows;  // heavier experts: the tensor-core kernel
      }
      const unsigned m = __ballot_sync(0xffffffffu, act_e);
      if (act_e) active[cnt + __popc(m & lt)] = e;
      cnt += __popc(m);
    }
    if (lane == 0) n_active = cnt;
  }
  __syncthreads();
  const int nact = n_active;

  if (warp == ncons) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = policy_evict_first();
    const uint32_t wbytes = (uint32_t)R * (p.K / 2);
    const uint32_t sbytes = (uint32_t)R * nb;
    const bool s16 = p.scale16 != 0;
    int issued = 0;
    for (int it = 0; it < nact; ++it) {
      const int st = it % nstage;
      if (it >= nstage && !mbar_wait(smem_addr(&empty[st]), ((it / nstage) - 1) & 1, p.status)) break;
      const int e = active[it];
      const uint32_t sbase = smem_addr(stages + (size_t)st * p.stage_bytes);
      const uint32_t fb = smem_addr(&full[st]);
      const int64_t row0 = (int64_t)e * p.N + n0;
      if (lane == 0) {
        mbar_arrive_expect_tx(fb, NM * wbytes);
        bulk_g2s(sbase, p.w0 + row0 * (p.K / 2), wbytes, fb, pol);
        if (NM == 2) bulk_g2s(sbase + p.wreg, p.w1 + row0 * (p.K / 2), wbytes, fb, pol);
      }
#pragma unroll
      for (int m = 0; m < NM; ++m) {
        const uint8_t *src = (m == 0 ? p.s0 : p.s1) + row0 * nb;
        const uint32_t dst = sbase + NM * p.wreg + m * p.sreg;
        if (s16) {
          for (uint32_t c = lane; c < sbytes / 16; c += 32) cp_async16(dst + 16 * c, src + 16 * c);
        } else {
          for (uint32_t c = lane; c < sbytes / 4; c += 32) cp_async4(dst + 4 * c, src + 4 * c);
        }
      }
      cp_async_mbar_arrive_noinc(fb);
      issued = it + 1;
    }
    // Never leave with copies in flight into this CTA's shared memory.
    for (int it = issued > nstage ? issued - nstage : 0; it < issued; ++it)
      mbar_wait(smem_addr(&full[it % nstage]), (it / nstage) & 1, p.status);
    return;
  }

  // -------------------------------------------------------------- consumers
  // Activation row of each sorted position (-1: padding, -2: out of range).
  const int nsorted = offs[p.E] < 0 ? 0 : (offs[p.E] > p.cap ? (int)p.cap : offs[p.E]);
  // (positions past offsets[E] hold no entry: -2, so that malformed offsets
  // can never turn an unwritten entry into a row index)
  if (p.rowtab) {
    for (int q = tid; q < p.cap; q += ncons * 32) {
      const int a = q < nsorted ? p.sorted[q] : p.A;
      rowtab[q] = a < 0 ? -1 : (a >= p.A ? -2 : (MODE == kDown ? a : token_of(a, p.kdiv)));
    }
  }
  // Stage every activation row once: codes in two half-block planes, the
  // scales, and the exact block sums sum(q) used by the offset encoding.
  if (p.act_smem) {
    for (int idx = tid; idx < p.n_act * nb; idx += ncons * 32) {
      const int r = idx / nb, b = idx - r * nb;
      stage_q8_block(act_base + (uint32_t)r * p.act_row_bytes, p.K, b, p.aq + (int64_t)r * p.ld_aq,
                     p.as[(int64_t)r * p.ld_as + b]);
    }
  }
  bar_sync_named(1, ncons * 32);

  // lane 0: the down output of row r for assignment a (CMB: into the CTA's
  // y rows in shared memory, and to out0 when given)
  auto put_down = [&](int a, int r, float v) {
    if (CMB) {
      ys[(int64_t)a * p.R + r] = v;
      if (p.out0) p.out0[(int64_t)a * p.ld_out + n0 + r] = v;
    } else {
      p.out0[(int64_t)a * p.ld_out + n0 + r] = v;
    }
  };
  // CMB: every expert's y rows of this CTA's output rows are in shared
  // memory: out[t, n0 + r] = slot-ordered combine, as the stand-alone combine
  // (fma chain over the slots, a slot of weight exactly 0 adds nothing)
  auto combine = [&]() {
    bar_sync_named(1, ncons * 32);
    for (int idx = tid; idx < p.T * p.R; idx += ncons * 32) {
      const int t = idx / p.R, r = idx - t * p.R;
      if (r >= R) continue;
      const float *wt = p.wts + (int64_t)t * p.k;
      const float *yt = ys + (int64_t)t * p.k * p.R + r;
      float acc = wt[0] != 0.0f ? __fmul_rn(wt[0], yt[0]) : 0.0f;
      for (int j = 1; j < p.k; ++j)
        if (wt[j] != 0.0f) acc = __fmaf_rn(wt[j], yt[(int64_t)j * p.R], acc);
      p.cout[(int64_t)t * p.ld_cout + n0 + r] = acc;
    }
  };

  if constexpr (!WIN) {
    // assignment and activation row of sorted position q (false: nothing to do)
    auto resolve = [&](int q, int &a, int &arow) -> bool {
      if (p.rowtab) {
        arow = rowtab[q];
        if (arow < 0) {
          if (arow == -2 && lane == 0 && p.status) atomicOr(p.status, MOE_DEV_BAD_ROW);
          return false;
        }
        a = p.sorted[q];
        return true;
      }
      a = p.sorted[q];
      if (a < 0) return false;
      if (a >= p.A) {
        if (lane == 0 && p.status) atomicOr(p.status, MOE_DEV_BAD_ROW);
        return false;
      }
      arow = MODE == kDown ? a : token_of(a, p.kdiv);
      return true;
    };
    // lane 0: the gate/up outputs of row r for assignment a
    auto put_gateup = [&](int a, int r, float g, float u) {
      const int64_t o = (int64_t)a * p.ld_out + n0 + r;
      if (MODE == kGateUpSwiglu) {
        p.out0[o] = __fmul_rn(silu(g), u);
      } else {
        p.out0[o] = g;
        p.out1[o] = u;
      }
    };
    for (int it = 0; it < nact; ++it) {
      const int st = it % nstage;
      if (!mbar_wait(smem_addr(&full[st]), (it / nstage) & 1, p.status)) break;
      const int e = active[it];
      const int seg_b = offs[e], seg_e = offs[e + 1];
      const uint32_t sbase = smem_addr(stages + (size_t)st * p.stage_bytes);

      if constexpr (MODE == kDown) {
        // more rows than warps: two output rows per warp, u and u + nu, so
        // that each activation row's loads serve both and one butterfly
        // reduces both (each row keeps its own arithmetic); not with four
        // blocks per lane, whose two converted rows would not fit registers
        const int nu = (S <= 2 && R > ncons) ? (R + 1) >> 1 : 0;
        for (int r = warp; nu == 0 && r < R; r += ncons) {
          uint32_t wq[1][S][8];
          float ws[1][S];
          load_weights<1, S>(sbase, 0, sbase + p.wreg, 0, r, p.K, wq, ws);
#pragma unroll 1
          for (int q = seg_b; q < seg_e; ++q) {
            int a, arow;
            if (!resolve(q, a, arow)) continue;
            float acc[1];
            if (p.act_smem) row_dot_smem<1, S>(act_base + (uint32_t)arow * p.act_row_bytes, p.K, wq, ws, acc);
            else row_dot_global<1, S>(p.aq + (int64_t)arow * p.ld_aq, p.as + (int64_t)arow * p.ld_as, p.K, wq, ws, acc);
            const float v = reduce_one(acc[0]);
            if (lane == 0) put_down(a, r, v);
          }
        }
        for (int u = warp; u < nu; u += ncons) {
          const int r2 = u + nu < R ? u + nu : u;
          const uint32_t dw = (uint32_t)(r2 - u) * (p.K / 2), dsc = (uint32_t)(r2 - u) * nb;
          uint32_t wq[2][S][8];
          float ws[2][S];
          load_weights<2, S>(sbase, dw, sbase + p.wreg, dsc, u, p.K, wq, ws);
#pragma unroll 1
          for (int q = seg_b; q < seg_e; ++q) {
            int a, arow;
            if (!resolve(q, a, arow)) continue;
            float acc[2];
            if (p.act_smem) row_dot_smem<2, S>(act_base + (uint32_t)arow * p.act_row_bytes, p.K, wq, ws, acc);
            else row_dot_global<2, S>(p.aq + (int64_t)arow * p.ld_aq, p.as + (int64_t)arow * p.ld_as, p.K, wq, ws, acc);
            float v0, v1;
            reduce_pair(acc[0], acc[1], v0, v1);
            if (lane == 0) {
              put_down(a, u, v0);
              if (r2 != u) put_down(a, r2, v1);
            }
          }
        }
      } else if (p.act_smem && seg_e - seg_b == 1) {
        // an expert with one row: the weights are read from the stage and
        // decoded by sign for that row alone (fewer integer operations than
        // converting them once for several rows); the same block dots
        int a, arow;
        if (resolve(seg_b, a, arow)) {
          for (int r = warp; r < R; r += ncons) {
            const uint32_t wrow[2] = {sbase + (uint32_t)r * (p.K / 2), sbase + p.wreg + (uint32_t)r * (p.K / 2)};
            const uint32_t srow[2] = {sbase + 2 * p.wreg + (uint32_t)r * nb, sbase + 2 * p.wreg + p.sreg + (uint32_t)r * nb};
            float acc[2];
            row_dot_stage_pn<2, S>(act_base + (uint32_t)arow * p.act_row_bytes, p.K, wrow, srow, stab, acc);
            float g, u;
            reduce_pair(acc[0], acc[1], g, u);
            if (lane == 0) put_gateup(a, r, g, u);
          }
        }
      } else {
        for (int r = warp; r < R; r += ncons) {
          uint32_t wq[NM][S][8];
          float ws[NM][S];
          load_weights<NM, S>(sbase, p.wreg, sbase + NM * p.wreg, p.sreg, r, p.K, wq, ws);
#pragma unroll 1
          for (int q = seg_b; q < seg_e; ++q) {
            int a, arow;
            if (!resolve(q, a, arow)) continue;
            float acc[NM];
            if (p.act_smem) row_dot_smem<NM, S>(act_base + (uint32_t)arow * p.act_row_bytes, p.K, wq, ws, acc);
            else row_dot_global<NM, S>(p.aq + (int64_t)arow * p.ld_aq, p.as + (int64_t)arow * p.ld_as, p.K, wq, ws, acc);
            float g, u;
            reduce_pair(acc[0], acc[NM - 1], g, u);
            if (lane == 0) put_gateup(a, r, g, u);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&empty[st]));
    }
    if constexpr (CMB) combine();
    return;
  } else {
  // activation row of sorted position q (-1: padding, -2: out of range)
  auto row_of = [&](int q) -> int {
    if (p.rowtab) return rowtab[q];
    const int a = p.sorted[q];
    return a < 0 ? -1 : (a >= p.A ? -2 : (MODE == kDown ? a : token_of(a, p.kdiv)));
  };
  const int W = p.win_rows;
  const uint32_t wbuf = (uint32_t)W * p.act_row_bytes;  // bytes of one window buffer
  // the passes, in ring order: pass (it, c0) takes rows [c0, min(c0 + W, seg_e)) of item it
  auto next_pass = [&](int &it, int &c0) {
    const int e = active[it];
    c0 += W;
    if (c0 >= offs[e + 1]) {
      ++it;
      c0 = it < nact ? offs[active[it]] : 0;
    }
  };
  // copies of the rows of pass (it, c0) into window buffer `buf` (no wait)
  auto copy_pass = [&](int it, int c0, int buf) {
    const int c1 = min(offs[active[it] + 1], c0 + W);
    const uint32_t base = act_base + (uint32_t)buf * wbuf;
    for (int idx = tid; idx < (c1 - c0) * nb; idx += ncons * 32) {
      const int qq = idx / nb, b = idx - qq * nb;
      const int arow = row_of(c0 + qq);
      if (arow < 0) continue;
      const uint32_t row = base + (uint32_t)qq * p.act_row_bytes;
      const int8_t *src = p.aq + (int64_t)arow * p.ld_aq + 32 * b;
      cp_async16(row + 16u * b, src);
      cp_async16(row + 16u * (nb + b), src + 16);
      cp_async4(row + (uint32_t)p.K + 4u * b, p.as + (int64_t)arow * p.ld_as + b);
    }
    cp_async_commit();
  };
  // block sums of the blocks this thread copied for pass (it, c0)
  auto sum_pass = [&](int it, int c0, int buf) {
    const int c1 = min(offs[active[it] + 1], c0 + W);
    const uint32_t base = act_base + (uint32_t)buf * wbuf;
    for (int idx = tid; idx < (c1 - c0) * nb; idx += ncons * 32) {
      const int qq = idx / nb, b = idx - qq * nb;
      if (row_of(c0 + qq) < 0) continue;
      const uint32_t row = base + (uint32_t)qq * p.act_row_bytes;
      sts32(row + (uint32_t)p.K + 4u * (nb + b), (uint32_t)block_sum8(lds128(row + 16u * b), lds128(row + 16u * (nb + b))));
    }
  };
  int pit = 0, pc0 = nact > 0 ? offs[active[0]] : 0, pbuf = 0;  // the pass whose rows are being copied
  if (nact > 0) copy_pass(pit, pc0, pbuf);

  // A warp whose wait on a stage gave up stops computing, but keeps arriving
  // on the ring and on the named barriers, so no other warp waits on it.
  bool dead = false;
  for (int it = 0; it < nact; ++it) {
    const int st = it % nstage;
    if (!dead) dead = !__all_sync(0xffffffffu, mbar_wait(smem_addr(&full[st]), (it / nstage) & 1, p.status));
    const int e = active[it];
    const int seg_b = offs[e], seg_e = offs[e + 1];
    const uint32_t sbase = smem_addr(stages + (size_t)st * p.stage_bytes);
    for (int c0 = seg_b; c0 < seg_e; c0 += W) {  // passes over the expert's rows
      const int c1 = min(seg_e, c0 + W);
      // this pass's rows (pit, pc0 == it, c0): wait for this thread's
      // copies, add their block sums, then one barrier: every row of the
      // pass is ready and every warp is done with the other buffer
      cp_async_wait<0>();
      sum_pass(pit, pc0, pbuf);
      const uint32_t wrows = act_base + (uint32_t)pbuf * wbuf;
      bar_sync_named(1, ncons * 32);
      next_pass(pit, pc0);
      pbuf ^= 1;
      if (pit < nact) copy_pass(pit, pc0, pbuf);  // the next pass's rows, while this one is computed
      if (dead) continue;
      // the down projection: two output rows per warp when there are more
      // rows than warps (as in the loop above)
      const int nu = (MODE == kDown && S <= 2 && R > ncons) ? (R + 1) >> 1 : 0;
      if constexpr (MODE == kDown) {
        for (int u = warp; u < nu; u += ncons) {
          const int r2 = u + nu < R ? u + nu : u;
          uint32_t wq[2][S][8];
          float ws[2][S];
          load_weights<2, S>(sbase, (uint32_t)(r2 - u) * (p.K / 2), sbase + p.wreg, (uint32_t)(r2 - u) * nb, u, p.K,
                             wq, ws);
#pragma unroll 1
          for (int q = c0; q < c1; ++q) {
            const int arow = row_of(q);
            if (arow < 0) {
              if (arow == -2 && lane == 0 && p.status) atomicOr(p.status, MOE_DEV_BAD_ROW);
              continue;
            }
            const int a = p.sorted[q];
            float acc[2];
            row_dot_smem<2, S>(wrows + (uint32_t)(q - c0) * p.act_row_bytes, p.K, wq, ws, acc);
            float v0, v1;
            reduce_pair(acc[0], acc[1], v0, v1);
            if (lane == 0) {
              put_down(a, u, v0);
              if (r2 != u) put_down(a, r2, v1);
            }
          }
        }
      }
      for (int r = warp; nu == 0 && r < R; r += ncons) {
        uint32_t wq[NM][S][8];
        float ws[NM][S];
        load_weights<NM, S>(sbase, p.wreg, sbase + NM * p.wreg, p.sreg, r, p.K, wq, ws);
        const int n = n0 + r;
#pragma unroll 1
        for (int q = c0; q < c1; ++q) {
          const int arow = row_of(q);
          if (arow < 0) {
            if (arow == -2 && lane == 0 && p.status) atomicOr(p.status, MOE_DEV_BAD_ROW);
            continue;
          }
          const int a = p.sorted[q];
          float acc[NM];
          row_dot_smem<NM, S>(wrows + (uint32_t)(q - c0) * p.act_row_bytes, p.K, wq, ws, acc);
          if (NM == 2) {
            float g, u;
            reduce_pair(acc[0], acc[NM - 1], g, u);
            if (lane == 0) {
              if (MODE == kGateUpSwiglu) {
                p.out0[(int64_t)a * p.ld_out + n] = __fmul_rn(silu(g), u);
              } else {
                p.out0[(int64_t)a * p.ld_out + n] = g;
                p.out1[(int64_t)a * p.ld_out + n] = u;
              }
            }
          } else {
            const float v = reduce_one(acc[0]);
            if (lane == 0) put_down(a, r, v);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&empty[st]));
  }
  cp_async_wait<0>();  // nothing of this thread's in flight at exit
  }
}

template <int MODE>
moe_status launch_mx(MxArgs p, cudaStream_t stream, const char *name) {
  constexpr int NM = (MODE == kDown) ? 1 : 2;
  const int nb = p.K / 32;
  const int S = (nb + 31) / 32;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_fail(err, name);
  int smem_optin = 0;
  err = cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (err != cudaSuccess) return cuda_fail(err, name);
  const size_t budget = (size_t)smem_optin - 1024;
  const int sms = sm_count();
  p.rowtab = p.cap <= kRowTab ? 1 : 0;
  p.act_row_bytes = (uint32_t)p.K + 8u * nb;
  const size_t fixed = (size_t)p.E * 8 + 4 + 16 * 8 + 32 + 1024 + (p.rowtab ? 4 * (size_t)p.cap : 0) + 16;
  int G = p.N < sms ? p.N : sms;
  for (;;) {
    p.R = (p.N + G - 1) / G;
    p.wreg = (uint32_t)p.R * (p.K / 2);
    p.sreg = ((uint32_t)p.R * nb + 15u) & ~15u;
    p.stage_bytes = (NM * (p.wreg + p.sreg) + 127u) & ~127u;
    if (budget >= fixed + 2 * (size_t)p.stage_bytes || G >= p.N) break;
    G = (2 * G < p.N) ? 2 * G : p.N;
  }
  // the fused combine keeps the y rows of this CTA's output rows ([A][R])
  const bool cmb = MODE == kDown && p.cout != nullptr;
  const size_t ys_bytes = cmb ? (((size_t)p.A * p.R * 4 + 15) & ~size_t(15)) : 0;
  if (budget < fixed + ys_bytes + 2 * (size_t)p.stage_bytes)
    return fail(MOE_ERR_UNSUPPORTED, "%s: K=%d too large for the shared-memory ring", name, p.K);
  // every activation row in shared memory if they fit beside a two-stage
  // ring; else, for the light experts of a large batch (the tile policy),
  // two window buffers of up to kWinRows rows each; else rows from global
  // memory (the 1-16-row calls: an expert has one or two rows there, and a
  // barrier per window pass costs more than the L2 reads it saves)
  const size_t room = budget - fixed - ys_bytes - 2 * (size_t)p.stage_bytes;  // >= 0: checked above
  const size_t all_rows = (size_t)p.n_act * p.act_row_bytes;
  size_t act_bytes = 0;  // never more than room
  p.act_smem = all_rows <= room ? 1 : 0;
  p.win_rows = 0;
  if (p.act_smem) {
    act_bytes = all_rows;
  } else if (p.max_rows != 0x7fffffff) {
    const size_t w = room / (2 * (size_t)p.act_row_bytes);
    p.win_rows = (int)(w < (size_t)kWinRows ? w : (size_t)kWinRows);
    act_bytes = 2 * (size_t)p.win_rows * p.act_row_bytes;
  }
  const size_t ns = (budget - fixed - ys_bytes - act_bytes) / p.stage_bytes;
  p.nstage = ns > 6 ? 6 : (int)ns;
  p.scale16 = (nb % 16) == 0 && (uintptr_t)p.s0 % 16 == 0 && (p.s1 == nullptr || (uintptr_t)p.s1 % 16 == 0);
  const int per_warp = (p.R + 14) / 15;
  const int ncons = (p.R + per_warp - 1) / per_warp;
  const size_t smem = (size_t)p.nstage * p.stage_bytes + fixed + act_bytes + ys_bytes;
  if (p.nstage < 2 || smem > budget || act_bytes > room)
    return fail(MOE_ERR_UNSUPPORTED, "%s: no shared-memory plan (stages %d, %zu bytes)", name, p.nstage, smem);
  const dim3 block((ncons + 1) * 32);

  const bool win = !p.act_smem && p.win_rows > 0;
  if (cmb && win) return fail(MOE_ERR_UNSUPPORTED, "%s: fused combine with activation windows", name);
  void (*kern)(MxArgs) = win ? (S == 1 ? mx_expert_kernel<MODE, 1, true>
                                      : (S == 2 ? mx_expert_kernel<MODE, 2, true> : mx_expert_kernel<MODE, 4, true>))
                             : (S == 1 ? mx_expert_kernel<MODE, 1, false>
                                      : (S == 2 ? mx_expert_kernel<MODE, 2, false> : mx_expert_kernel<MODE, 4, false>));
  if constexpr (MODE == kDown) {
    if (cmb)
      kern = S == 1 ? mx_expert_kernel<MODE, 1, false, true>
                    : (S == 2 ? mx_expert_kernel<MODE, 2, false, true> : mx_expert_kernel<MODE, 4, false, true>);
  }
  const moe_status ast = ensure_smem_attr(reinterpret_cast<const void *>(kern), (int)budget, name);
  if (ast != MOE_OK) return ast;
  kern<<<G, block, smem, stream>>>(p);
  err = cudaGetLastError();
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, name);
}

moe_status check_common(const char *name, const int8_t *aq, int64_t ld_aq, const float *as, int64_t ld_as,
                        const void *w0, const void *s0, const void *w1, const void *s1, const int32_t *offsets,
                        const int32_t *sorted, int64_t cap, int T, int k, int E, int H, int I, const void *out,
                        int64_t ld_out, int Kred, int rows_act) {
  if (T < 0 || k <= 0 || E <= 0 || H <= 0 || I <= 0) return fail(MOE_ERR_INVALID_ARG, "%s: T=%d k=%d E=%d H=%d I=%d", name, T, k, E, H, I);
  if (H % 128 || I % 128) return fail(MOE_ERR_INVALID_ARG, "%s: H=%d and I=%d must be multiples of 128", name, H, I);
  if (Kred > 4096) return fail(MOE_ERR_UNSUPPORTED, "%s: reduction length %d > 4096", name, Kred);
  if (E > 4096) return fail(MOE_ERR_UNSUPPORTED, "%s: E=%d > 4096", name, E);
  if ((int64_t)T * k > 0x7fffffff) return fail(MOE_ERR_UNSUPPORTED, "%s: too many assignments", name);
  if (T == 0) return MOE_OK;
  if (!aq || !as || !w0 || !s0 || (w1 == nullptr) != (s1 == nullptr) || !offsets || !sorted || !out)
    return fail(MOE_ERR_INVALID_ARG, "%s: null pointer", name);
  if ((uintptr_t)aq % 16 || ld_aq % 16 || ld_aq < Kred) return fail(MOE_ERR_INVALID_ARG, "%s: Q8 codes must be 16-byte aligned with ld a multiple of 16 >= %d (ld=%lld)", name, Kred, (long long)ld_aq);
  if ((uintptr_t)as % 4 || ld_as < Kred / 32) return fail(MOE_ERR_INVALID_ARG, "%s: bad Q8 scale stride %lld", name, (long long)ld_as);
  if ((uintptr_t)w0 % 16 || (w1 && (uintptr_t)w1 % 16)) return fail(MOE_ERR_INVALID_ARG, "%s: weights must be 16-byte aligned", name);
  if ((uintptr_t)s0 % 4 || (s1 && (uintptr_t)s1 % 4)) return fail(MOE_ERR_INVALID_ARG, "%s: scale bytes must be 4-byte aligned", name);
  if (cap < 0) return fail(MOE_ERR_INVALID_ARG, "%s: cap=%lld", name, (long long)cap);
  if ((uintptr_t)out % 4) return fail(MOE_ERR_INVALID_ARG, "%s: output must be 4-byte aligned", name);
  (void)rows_act;
  (void)ld_out;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

static moe_status gateup_impl(int mode, const int8_t *xq, int64_t ld_xq, const float *xs, int64_t ld_xs,
                              const uint8_t *wg, const uint8_t *sg, const uint8_t *wu, const uint8_t *su,
                              const int32_t *offsets, const int32_t *sorted, int64_t cap, int T, int k, int E,
                              int H, int I, float *o0, float *o1, int64_t ld, void *stream, const char *name) {
  moe_status st = check_common(name, xq, ld_xq, xs, ld_xs, wg, sg, wu, su, offsets, sorted, cap, T, k, E, H, I, o0,
                               ld, H, T);
  if (st != MOE_OK || T == 0) return st;
  if (!wu) return fail(MOE_ERR_INVALID_ARG, "%s: null up weights", name);
  if (ld < I) return fail(MOE_ERR_INVALID_ARG, "%s: output ld=%lld < I=%d", name, (long long)ld, I);
  if (mode == kGateUpRaw && (!o1 || (uintptr_t)o1 % 4)) return fail(MOE_ERR_INVALID_ARG, "%s: bad up output", name);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // tile policy: from kTensorMinRows rows on, experts with more than
  // kLightExpertRows rows take the tensor-core kernel, the rest this one
  const bool split = T >= kTensorMinRows && tc_expert_supported(H, I);
  if (split) {
    st = launch_tc_expert(mode == kGateUpSwiglu ? 0 : 1, xq, ld_xq, xs, ld_xs, wg, sg, wu, su, offsets, sorted, cap,
                          T * k, k, E, H, I, 1, kLightExpertRows, o0, mode == kGateUpSwiglu ? nullptr : o1, ld, s,
                          name);
    if (st != MOE_OK) return st;
  }
  if (split) {
    // the light experts of a 17+-row call: the four-group kernel (krow.cu)
    // when its plan fits (for 1-16-row calls the kernel below is faster: it
    // converts the weights of an expert with several rows once)
    st = launch_krow(mode == kGateUpSwiglu ? 0 : 1, xq, ld_xq, xs, ld_xs, wg, sg, wu, su, offsets, sorted, cap, T, k,
                     E, H, I, kLightExpertRows, o0, o1, ld, nullptr, nullptr, 0, s, name);
    if (st != MOE_ERR_UNSUPPORTED) return st;
  }
  MxArgs p{};
  p.max_rows = split ? kLightExpertRows : 0x7fffffff;
  p.aq = xq; p.ld_aq = ld_xq; p.as = xs; p.ld_as = ld_xs;
  p.w0 = wg; p.s0 = sg; p.w1 = wu; p.s1 = su;
  p.offsets = offsets; p.sorted = sorted; p.cap = cap;
  p.A = T * k; p.k = k; p.E = E; p.K = H; p.N = I;
  p.n_act = T;
  p.kdiv = kdiv_of(k);
  p.out0 = o0; p.out1 = o1; p.ld_out = ld;
  p.status = device_status_word();
  return mode == kGateUpSwiglu ? launch_mx<kGateUpSwiglu>(p, s, name) : launch_mx<kGateUpRaw>(p, s, name);
}

extern "C" moe_status moe_mxfp4_gateup_swiglu(const int8_t *xq, int64_t ld_xq, const float *xs, int64_t ld_xs,
                                              const uint8_t *wg, const uint8_t *sg, const uint8_t *wu,
                                              const uint8_t *su, const int32_t *offsets, const int32_t *sorted,
                                              int64_t cap, int T, int k, int E, int H, int I, float *h,
                                              int64_t ld_h, void *stream) {
  return gateup_impl(kGateUpSwiglu, xq, ld_xq, xs, ld_xs, wg, sg, wu, su, offsets, sorted, cap, T, k, E, H, I, h,
                     nullptr, ld_h, stream, "moe_mxfp4_gateup_swiglu");
}

extern "C" moe_status moe_mxfp4_gateup(const int8_t *xq, int64_t ld_xq, const float *xs, int64_t ld_xs,
                                       const uint8_t *wg, const uint8_t *sg, const uint8_t *wu, const uint8_t *su,
                                       const int32_t *offsets, const int32_t *sorted, int64_t cap, int T, int k,
                                       int E, int H, int I, float *g, float *u, int64_t ld_gu, void *stream) {
  return gateup_impl(kGateUpRaw, xq, ld_xq, xs, ld_xs, wg, sg, wu, su, offsets, sorted, cap, T, k, E, H, I, g, u,
                     ld_gu, stream, "moe_mxfp4_gateup");
}

extern "C" moe_status moe_mxfp4_down(const int8_t *hq, int64_t ld_hq, const float *hs, int64_t ld_hs,
                                     const uint8_t *wd, const uint8_t *sd, const int32_t *offsets,
                                     const int32_t *sorted, int64_t cap, int T, int k, int E, int H, int I, float *y,
                                     int64_t ld_y, void *stream) {
  const char *name = "moe_mxfp4_down";
  moe_status st = check_common(name, hq, ld_hq, hs, ld_hs, wd, sd, nullptr, nullptr, offsets, sorted, cap, T, k, E,
                               H, I, y, ld_y, I, T * k);
  if (st != MOE_OK || T == 0) return st;
  if (ld_y < H) return fail(MOE_ERR_INVALID_ARG, "%s: ld_y=%lld < H=%d", name, (long long)ld_y, H);
  const bool split = T >= kTensorMinRows && tc_expert_supported(I, H);  // tile policy, as for gate/up
  if (split) {
    st = launch_tc_expert(2, hq, ld_hq, hs, ld_hs, wd, sd, nullptr, nullptr, offsets, sorted, cap, T * k, k, E, I, H,
                          0, kLightExpertRows, y, nullptr, ld_y, static_cast<cudaStream_t>(stream), name);
    if (st != MOE_OK) return st;
  }
  // the four-group kernel (krow.cu) for every expert of a 1-16-row call, or
  // the light experts of a larger one, when its shared-memory plan fits the
  // shape; the kernel below otherwise
  st = launch_krow(2, hq, ld_hq, hs, ld_hs, wd, sd, nullptr, nullptr, offsets, sorted, cap, T, k, E, I, H,
                   split ? kLightExpertRows : 0x7fffffff, y, nullptr, ld_y, nullptr, nullptr, 0,
                   static_cast<cudaStream_t>(stream), name);
  if (st != MOE_ERR_UNSUPPORTED) return st;
  MxArgs p{};
  p.max_rows = split ? kLightExpertRows : 0x7fffffff;
  p.aq = hq; p.ld_aq = ld_hq; p.as = hs; p.ld_as = ld_hs;
  p.w0 = wd; p.s0 = sd;
  p.offsets = offsets; p.sorted = sorted; p.cap = cap;
  p.A = T * k; p.k = k; p.E = E; p.K = I; p.N = H;
  p.n_act = T * k;
  p.kdiv = kdiv_of(k);
  p.out0 = y; p.ld_out = ld_y;
  p.status = device_status_word();
  return launch_mx<kDown>(p, static_cast<cudaStream_t>(stream), name);
}

extern "C" moe_status moe_mxfp4_down_combine(const int8_t *hq, int64_t ld_hq, const float *hs, int64_t ld_hs,
                                             const uint8_t *wd, const uint8_t *sd, const int32_t *offsets,
                                             const int32_t *sorted, int64_t cap, const float *w, int T, int k, int E,
                                             int H, int I, float *out, int64_t ld_out, float *y, int64_t ld_y,
                                             void *stream) {
  const char *name = "moe_mxfp4_down_combine";
  moe_status st = check_common(name, hq, ld_hq, hs, ld_hs, wd, sd, nullptr, nullptr, offsets, sorted, cap, T, k, E,
                               H, I, out, ld_out, I, T * k);
  if (st != MOE_OK || T == 0) return st;
  if (!w || (uintptr_t)w % 4) return fail(MOE_ERR_INVALID_ARG, "%s: bad routing weights", name);
  if (ld_out < H) return fail(MOE_ERR_INVALID_ARG, "%s: ld_out=%lld < H=%d", name, (long long)ld_out, H);
  if (y && (ld_y < H || (uintptr_t)y % 4)) return fail(MOE_ERR_INVALID_ARG, "%s: bad y output", name);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // one launch while the batch keeps the CUDA-core path and a CTA's y rows
  // fit its shared memory beside the ring
  const bool split = T >= kTensorMinRows && tc_expert_supported(I, H);
  if (!split) {
    st = launch_krow(2, hq, ld_hq, hs, ld_hs, wd, sd, nullptr, nullptr, offsets, sorted, cap, T, k, E, I, H,
                     0x7fffffff, y, nullptr, y ? ld_y : 0, w, out, ld_out, s, name);
    if (st != MOE_ERR_UNSUPPORTED) return st;
    MxArgs p{};
    p.max_rows = 0x7fffffff;
    p.aq = hq; p.ld_aq = ld_hq; p.as = hs; p.ld_as = ld_hs;
    p.w0 = wd; p.s0 = sd;
    p.offsets = offsets; p.sorted = sorted; p.cap = cap;
    p.A = T * k; p.k = k; p.E = E; p.K = I; p.N = H;
    p.n_act = T * k;
    p.kdiv = kdiv_of(k);
    p.out0 = y; p.ld_out = y ? ld_y : 0;
    p.wts = w; p.cout = out; p.ld_cout = ld_out; p.T = T;
    p.status = device_status_word();
    st = launch_mx<kDown>(p, s, name);
    if (st != MOE_ERR_UNSUPPORTED) return st;
  }
  // otherwise the down projection into y, then the combine
  if (!y) return fail(MOE_ERR_UNSUPPORTED, "%s: T=%d takes two launches and needs the y buffer", name, T);
  st = moe_mxfp4_down(hq, ld_hq, hs, ld_hs, wd, sd, offsets, sorted, cap, T, k, E, H, I, y, ld_y, stream);
  if (st != MOE_OK) return st;
  return moe_combine(y, ld_y, w, T, k, H, out, ld_out, stream);
}
