// Fused single-launch forward of the MoE layer for small decode batches.
//
// The same layer as the six stage calls ("DeepSeek-V4-Flash on AMD gfx90a",
// Fig. 1 and §6.1; "Optimizing DeepSeek V4 Flash Inference on a Strix Halo
// Pair", "MXFP4 routed-expert kernels": "MoE decode is pure bandwidth"), with
// the same arithmetic (every step comes from mx_device.cuh), so it gives the
// same bits as the stage calls, row for row.  What changes is the schedule:
// one cooperative launch of one CTA per SM instead of eight kernels.
//
//   A   router logits (a warp per expert, experts spread over all CTAs) and,
//       in every CTA, Q8 of the T activation rows into shared memory
//   --- grid barrier
//   A'  every CTA: top-k of every token, stable sort of the assignments
//   B   one TMA ring per CTA streams the CTA's output slice of every active
//       expert: first the gate/up slices (h -> global), then the down slices
//       (prefetched into L2 while gate/up runs)
//   --- grid barrier (consumer warps only; the producer keeps streaming)
//   C   Q8 of every h row into shared memory, down projection of the CTA's
//       slice, then the slot-ordered combine of that slice -> out
//
// Waits are bounded: a grid barrier or an mbarrier that does not complete in
// about a second sets MOE_DEV_WAIT_TIMEOUT and the kernel returns.
#include <algorithm>
#include <atomic>

#include "mx_device.cuh"

namespace moe {
namespace {

constexpr int kWarps = 29;
constexpr int kThreads = kWarps * 32;
constexpr int kCons = kWarps - 1;  // warps 0..27 consume (<= 64 registers each); warp 28 produces
constexpr int kGroup = kCons / 2;  // consumer warps per ring item (two items in flight)
constexpr int kMaxA = 64;          // assignments T*k handled by the fused path
constexpr int kSlotWord = 8;       // first per-expert readiness word of the workspace
constexpr int kSharedWord = kSlotWord + kMaxA - 1;  // the shared expert's (T*k <= kMaxA - 1 with one)

struct DecodeArgs {
  const void *x;
  int64_t ld_x;
  int xbf;
  const void *wr;
  int wbf;
  const float *bias;
  const uint8_t *wg, *sg, *wu, *su, *wd, *sd;
  int T, H, E, k, I, A;
  uint32_t kdiv;  // kdiv_of(k): token of assignment a = token_of(a, kdiv)
  float *out;
  int64_t ld_out;
  float *logits;
  int32_t *ids;
  float *weights;
  float *h;
  int64_t ld_h;
  float *y;  // optional
  int64_t ld_y;
  unsigned long long *bar;  // [0] arrival counter, [1] barrier hold (0), [2] readiness hold (0),
                            // [kSlotWord + j] h of expert slot j done
  unsigned *status;
  // geometry (host-computed)
  int nstage;
  uint32_t stage_bytes;
  uint32_t gwreg, gsreg;  // gate/up stage: weight / scale region per matrix
  uint32_t dwreg;         // down slice: weight region (scale bytes follow)
  uint32_t dslot;         // bytes of one down slice in a stage (128-aligned)
  int dpp;                // down slices per ring stage
  uint32_t xrow, hrow;    // staged activation row bytes
  uint32_t off_bars, off_act, off_hq, off_y, off_logit, off_cand, off_misc;
  int Rd;                 // max down rows per CTA (row stride of the y slice)
  int Rg;                 // max gate/up rows per CTA (row stride of the gate/up sums)
  int g16, d16;           // scale bytes copyable in 16-byte pieces
  int hqr;                // Q8(h) in the last ring stage during the down phase (down items skip that stage)
  // optional shared expert: one more expert of the routed experts' format,
  // run on every token with weight 1 and added after the routed combine
  int shared;
  const uint8_t *swg, *ssg, *swu, *ssu, *swd, *ssd;
  float *sh_h;            // [T][ld_sh_h] its SwiGLU activations (exchange buffer)
  int64_t ld_sh_h;
  float *sh_y;            // [T][ld_sh_y] its down output, or null
  int64_t ld_sh_y;
};

struct Misc {  // views into the small shared-memory region (A = T*k <= 64)
  int *ids;     // [A] expert of assignment a
  float *w;     // [A] routing weight of assignment a
  int *srt;     // [R] assignment at sorted position p (R = A, + T shared-expert rows A + t)
  int *skey;    // [A] expert at sorted position p
  int *segb;    // [A+2] start of the j-th expert segment (segb[nact]: the routed rows; segb[nact+1]: + the shared expert's)
  int *active;  // [A] expert of the j-th segment, increasing id
  int *scalars; // [0] number of segments, [1] barrier flag, [2 + g] wait result of group g
};

MOE_DEVFN Misc misc_view(uint8_t *base, int A, int R) {
  Misc m;
  int *p = reinterpret_cast<int *>(base);
  m.ids = p; p += A;
  m.w = reinterpret_cast<float *>(p); p += A;
  m.srt = p; p += R;
  m.skey = p; p += A;
  m.segb = p; p += A + 2;
  m.active = p; p += A;
  m.scalars = p;
  return m;
}

constexpr uint64_t kBarrierTimeoutNs = 250ull * 1000 * 1000;  // 0.25 s
// The time limit counts only after this many polls (several milliseconds of
// polling), so that a step of the global timer (it can be re-synchronised)
// never ends a wait of normal length.
constexpr uint32_t kMinPolls = 1u << 14;

// Programmatic dependent launch: wait until the kernels this launch depends
// on have completed and their writes are visible (returns at once when the
// launch was not programmatic); allow the kernel after this one to launch.
MOE_DEVFN void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
MOE_DEVFN void grid_dependents_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

MOE_DEVFN uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Grid-wide barrier for the `nthreads` threads of every CTA that reach it
// (named barrier `bar_id` inside the CTA).  The workspace holds a 64-bit
// arrival counter that only grows: each call adds G per barrier, so the
// counter is a multiple of G between calls; a CTA reads it at kernel start
// and rounds down (no CTA can pass barrier 1 before every CTA has started),
// and barrier i completes when the counter reaches base + i*G + hold, where
// `hold` is workspace word 1 (0 in use; a test sets it to make the wait run
// out).  Arrival is a fire-and-forget release add; waiting polls with acquire
// loads for at most kBarrierTimeoutNs.  Returns false on timeout.
MOE_DEVFN bool grid_barrier(unsigned long long *ctr, unsigned long long target, int bar_id, int nthreads, int *flag,
                            unsigned *status) {
  bar_sync_named(bar_id, nthreads);
  if (threadIdx.x == 0) {
    asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(ctr), "l"(1ull) : "memory");
    const uint64_t t0 = globaltimer_ns();
    int ok = 1;
    for (uint32_t i = 0;; ++i) {
      unsigned long long v;
      asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(ctr) : "memory");
      if (v >= target) break;
      if (i > (1u << 26) || (i > kMinPolls && globaltimer_ns() - t0 > kBarrierTimeoutNs)) {
        ok = 0;
        break;
      }
      if (i >= 8) __nanosleep(32);
    }
    if (!ok && status) atomicOr(status, MOE_DEV_WAIT_TIMEOUT);
    *reinterpret_cast<volatile int *>(flag) = ok;
  }
  bar_sync_named(bar_id, nthreads);
  return *reinterpret_cast<volatile int *>(flag) != 0;
}

// Wait (one thread) until *ctr >= target: acquire loads for at most
// kBarrierTimeoutNs.  Returns false on timeout.
MOE_DEVFN bool wait_count(unsigned long long *ctr, unsigned long long target, unsigned *status) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0;; ++i) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(ctr) : "memory");
    if (v >= target) return true;
    if (i > (1u << 26) || (i > kMinPolls && globaltimer_ns() - t0 > kBarrierTimeoutNs)) {
      if (status) atomicOr(status, MOE_DEV_WAIT_TIMEOUT);
      return false;
    }
    if (i >= 8) __nanosleep(32);
  }
}

MOE_DEVFN void load32_smem(uint32_t addr, bool bf16, float (&v)[32]) {
  const uint32_t step = bf16 ? 16u : 32u;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    float w8[8];
    load8_smem(addr + c * step, bf16, w8);
#pragma unroll
    for (int j = 0; j < 8; ++j) v[8 * c + j] = w8[j];
  }
}

// One router logit (one expert row, one token) from shared memory, one warp,
// in the order of the router kernels: lane l accumulates the chunks l, l+32,
// ... of 8 consecutive inputs in increasing order with one fma per element,
// then the 32 partial sums meet in an xor butterfly.  The chunk loads of four
// consecutive passes are issued together; the fma order is unchanged.
MOE_DEVFN float router_dot_smem(uint32_t wrow, bool wbf, uint32_t xrow, bool xbf, int H) {
  const int lane = threadIdx.x & 31;
  const int nch = H / 8;
  float p = 0.0f;
  if (wbf && xbf) {
    // bf16 rows: the raw 16-byte chunks of four passes in flight, widened on use
#pragma unroll 1
    for (int c0 = lane; c0 < nch; c0 += 128) {
      uint4 wr[4], xr[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (c0 + 32 * i < nch) {
          wr[i] = lds128(wrow + 16u * (uint32_t)(c0 + 32 * i));
          xr[i] = lds128(xrow + 16u * (uint32_t)(c0 + 32 * i));
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (c0 + 32 * i < nch) {
          const uint32_t wv[4] = {wr[i].x, wr[i].y, wr[i].z, wr[i].w};
          const uint32_t xv[4] = {xr[i].x, xr[i].y, xr[i].z, xr[i].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            p = __fmaf_rn(bf16_lo(xv[q]), bf16_lo(wv[q]), p);
            p = __fmaf_rn(bf16_hi(xv[q]), bf16_hi(wv[q]), p);
          }
        }
      }
    }
  } else {
    const uint32_t wstep = wbf ? 16u : 32u, xstep = xbf ? 16u : 32u;
#pragma unroll 1
    for (int c = lane; c < nch; c += 32) {
      float wv[8], xv[8];
      load8_smem(wrow + (uint32_t)c * wstep, wbf, wv);
      load8_smem(xrow + (uint32_t)c * xstep, xbf, xv);
#pragma unroll
      for (int q = 0; q < 8; ++q) p = __fmaf_rn(xv[q], wv[q], p);
    }
  }
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) p = __fadd_rn(p, __shfl_xor_sync(0xffffffffu, p, s));
  return p;
}

// Q8 of one 32-value block into a staged row: codes in the split-half layout
// (elements 0..15 of block b at 16 b, 16..31 at 16 (nb + b)), then the
// block scales.
MOE_DEVFN void q8_to_row(const float (&v)[32], uint32_t row, int K, int b) {
  const int nb = K / 32;
  uint32_t pk[8];
  int sum;
  const float d = q8_block(v, pk, &sum);
  sts128(row + 16u * b, make_uint4(pk[0], pk[1], pk[2], pk[3]));
  sts128(row + 16u * (nb + b), make_uint4(pk[4], pk[5], pk[6], pk[7]));
  sts32(row + (uint32_t)K + 4u * b, __float_as_uint(d));
}

// Q8 of one 32-value block by a lane pair (lanes 2i, 2i+1; the whole warp
// must call): each lane holds 16 values (half 0: elements 0..15, half 1:
// 16..31).  amax is combined across the pair; every other step is
// q8_block's, element by element, so the codes and the scale are q8_block's.
// Half 0 writes the first half-block plane and the scale, half 1 the second
// plane.
MOE_DEVFN void q8_pair_to_row(const float (&v)[16], int half, bool store, uint32_t row, int K, int b) {
  const int nb = K / 32;
  float amax = 0.0f;
#pragma unroll
  for (int l = 0; l < 16; ++l) amax = fmaxf(amax, fabsf(v[l]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  const float d = __fdiv_rn(amax, 127.0f);
  const float inv = d > 0.0f ? __frcp_rn(d) : 0.0f;
  uint32_t pk[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int qi = __float2int_rn(__fmul_rn(v[4 * c + j], inv));
      qi = max(-127, min(127, qi));
      word |= (uint32_t)(qi & 0xFF) << (8 * j);
    }
    pk[c] = word;
  }
  if (store) {
    sts128(row + 16u * (half ? nb + b : b), make_uint4(pk[0], pk[1], pk[2], pk[3]));
    if (half == 0) sts32(row + (uint32_t)K + 4u * b, __float_as_uint(d));
  }
}

// Stable sort of the A assignments by expert (ties by assignment index), the
// order of the stand-alone sorter: assignment a lands at position
// #{b : (id_b, b) < (id_a, a)}.  One thread per assignment, then one warp
// cuts the sorted keys into expert segments (increasing expert id).
// An expert id outside [0, E) (top-k of NaN scores) sorts last as E, is left
// out of every segment and raises MOE_DEV_BAD_EXPERT_ID: no weight address is
// ever formed from it.
MOE_DEVFN void rank_sort(const Misc &m, int A, int E, unsigned *status) {
  const int tid = threadIdx.x;
  if (tid < A) {
    int e = m.ids[tid];
    if (e < 0 || e >= E) {
      e = E;
      if (status) atomicOr(status, MOE_DEV_BAD_EXPERT_ID);
    }
    int rank = 0;
    for (int b = 0; b < A; ++b) {
      int eb = m.ids[b];
      if (eb < 0 || eb >= E) eb = E;
      rank += (eb < e) || (eb == e && b < tid);
    }
    m.srt[rank] = tid;
    m.skey[rank] = e;
  }
  __syncthreads();
  if (tid < 32) {
    const int lane = tid;
    const unsigned lt = (1u << lane) - 1u;
    int cnt = 0;
    for (int p0 = 0; p0 < A; p0 += 32) {
      const int q = p0 + lane;
      const bool st = q < A && m.skey[q] < E && (q == 0 || m.skey[q] != m.skey[q - 1]);
      const unsigned bal = __ballot_sync(0xffffffffu, st);
      if (st) {
        const int j = cnt + __popc(bal & lt);
        m.segb[j] = q;
        m.active[j] = m.skey[q];
      }
      cnt += __popc(bal);
    }
    // the last valid segment ends where the invalid ids (if any) begin
    int nvalid = 0;
    for (int q = lane; q < A; q += 32) nvalid += m.skey[q] < E;
    nvalid = __reduce_add_sync(0xffffffffu, (unsigned)nvalid);
    if (lane == 0) {
      m.segb[cnt] = nvalid;
      m.scalars[0] = cnt;
    }
  }
  __syncthreads();
}

// SG, SD: 32-block groups per lane for the gate/up (K = H) and down (K = I)
// rows.  FULL: H = 1024 SG and I = 1024 SD exactly, so every size below is a
// compile-time constant.
// rank_sort by one warp (the whole warp calls it) for A <= 32 assignments:
// the same ranks, segments and flags, with the ranks counted over shuffled
// ids and the segments cut with one ballot.
MOE_DEVFN void rank_sort_warp(const Misc &m, int A, int E, unsigned *status) {
  const int lane = threadIdx.x & 31;
  int e = E;
  if (lane < A) {
    e = m.ids[lane];
    if (e < 0 || e >= E) {
      e = E;
      if (status) atomicOr(status, MOE_DEV_BAD_EXPERT_ID);
    }
  }
  int rank = 0;
#pragma unroll 1
  for (int b = 0; b < A; ++b) {
    const int eb = __shfl_sync(0xffffffffu, e, b);
    rank += (eb < e) || (eb == e && b < lane);
  }
  if (lane < A) {
    m.srt[rank] = lane;
    m.skey[rank] = e;
  }
  __syncwarp();
  const int kq = lane < A ? m.skey[lane] : E;
  const int kp = (lane > 0 && lane < A) ? m.skey[lane - 1] : -1;
  const bool st = lane < A && kq < E && (lane == 0 || kq != kp);
  const unsigned bal = __ballot_sync(0xffffffffu, st);
  if (st) {
    const int j = __popc(bal & ((1u << lane) - 1u));
    m.segb[j] = lane;
    m.active[j] = kq;
  }
  const int nvalid = __popc(__ballot_sync(0xffffffffu, lane < A && kq < E));
  if (lane == 0) {
    m.segb[__popc(bal)] = nvalid;
    m.scalars[0] = __popc(bal);
  }
}

// Ring stage of item it, and how many earlier items used that stage (the
// phase parity of its barriers).  Gate/up items cycle through the NS stages;
// with hqr the down items cycle through the first NS - 1, the last one
// holding Q8(h) during the down phase.
MOE_DEVFN void ring_slot(int it, int nslot, int NS, bool hqr, int &st, int &use) {
  if (!hqr || it < nslot) {
    st = it % NS;
    use = it / NS;
    return;
  }
  const int d = it - nslot, NSd = NS - 1;
  st = d % NSd;
  use = (nslot - st + NS - 1) / NS + d / NSd;  // gate/up items on stage st, then earlier down items
}

// Full barrier (index into the kernel's full barriers) and phase parity of
// ring item it.  The routed gate/up items alternate between the two consumer
// groups, and each group waits only on barriers of its own, one per (stage,
// group) at 2 st + g, in order.  The items every consumer warp waits for
// (the shared expert's gate/up item, then the down items) have a third
// barrier per stage, at 2 NS + st.  With one barrier per stage for both
// groups, an odd number of stages would let a group reach its item's phase
// while the other group's item before it on that stage has not landed, and
// a parity wait cannot tell those phases apart.
MOE_DEVFN void ring_full(int it, int s0, int nslot, int NS, bool hqr, int &bar, uint32_t &parity) {
  int st, use;
  ring_slot(it, nslot, NS, hqr, st, use);
  if (it >= s0 && it < nslot) {
    const int j = it - s0, L = (NS & 1) ? 2 * NS : NS;  // items (stage, group) repeat every lcm(NS, 2)
    bar = 2 * st + (j & 1);
    parity = (uint32_t)(j / L) & 1u;
  } else {
    int n = 0;  // earlier all-warp items on stage st
    if (it >= nslot) {
      const int d = it - nslot;
      n = (hqr ? d / (NS - 1) : d / NS) + ((s0 && st == 0) ? 1 : 0);
    }
    bar = 2 * NS + st;
    parity = (uint32_t)n & 1u;
  }
}
// The barrier of ring item it on stage st (ring_full's index without its
// divisions; the hot loops track the phase parities themselves).
MOE_DEVFN int ring_full_bar(int it, int st, int s0, int nslot, int NS) {
  return (it >= s0 && it < nslot) ? 2 * st + ((it - s0) & 1) : 2 * NS + st;
}

// The producer warp's copies of one gate/up slice (rows row0 .. of both
// matrices, Rg rows each) into the ring stage at sbase, completing on the
// stage's full barrier fb (the whole warp calls it: the scale bytes may need
// per-lane copies).
MOE_DEVFN void gateup_copies(uint32_t sbase, uint32_t fb, const uint8_t *wg, const uint8_t *wu, const uint8_t *sg,
                             const uint8_t *su, int64_t row0, uint32_t gwb, uint32_t gsb, const DecodeArgs &p, int H,
                             int nbH, uint64_t pol) {
  const int lane = threadIdx.x & 31;
  if (lane == 0) {
    mbar_arrive_expect_tx(fb, 2 * gwb + (p.g16 ? 2 * gsb : 0u));
    if (gwb > 0) {  // a CTA may own no gate/up rows when I < #SMs
      bulk_g2s(sbase, wg + row0 * (H / 2), gwb, fb, pol);
      bulk_g2s(sbase + p.gwreg, wu + row0 * (H / 2), gwb, fb, pol);
      if (p.g16) {  // the slice's scale bytes are one contiguous 16-byte-aligned run
        bulk_g2s(sbase + 2 * p.gwreg, sg + row0 * nbH, gsb, fb, pol);
        bulk_g2s(sbase + 2 * p.gwreg + p.gsreg, su + row0 * nbH, gsb, fb, pol);
      }
    }
  }
  if (!p.g16) {
#pragma unroll
    for (int mm = 0; mm < 2; ++mm) {
      const uint8_t *src = (mm == 0 ? sg : su) + row0 * nbH;
      const uint32_t dst = sbase + 2 * p.gwreg + mm * p.gsreg;
      for (uint32_t c = lane; c < gsb / 4; c += 32) cp_async4(dst + 4 * c, src + 4 * c);
    }
  }
  cp_async_mbar_arrive_noinc(fb);
}

template <int SG, int SD, bool FULL, bool SHARED>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const DecodeArgs p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = gridDim.x, cta = blockIdx.x;
  const int H = FULL ? 1024 * SG : p.H, I = FULL ? 1024 * SD : p.I;
  const int E = p.E, k = p.k, T = p.T, A = p.A;
  const int nbH = H / 32, nbI = I / 32;
  const int nstage = p.nstage;
  // this CTA's output slices (G * 4096 fits 32 bits)
  const int n0g = (int)((unsigned)(cta * I) / (unsigned)G), Rg = (int)((unsigned)((cta + 1) * I) / (unsigned)G) - n0g;
  const int n0d = (int)((unsigned)(cta * H) / (unsigned)G), Rd = (int)((unsigned)((cta + 1) * H) / (unsigned)G) - n0d;

  // the next kernel on the stream may be launched now; its CTAs start on SMs
  // as this launch's CTAs leave them, and wait for this launch to complete
  // before they touch anything it uses (programmatic dependent launch)
  grid_dependents_launch();
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + p.off_bars);
  uint64_t *empty = full + 3 * nstage;  // full: 2 per stage (one per consumer group), then 1 per stage for all warps
  const uint32_t act = smem_addr(smem + p.off_act);
  float *yslice = reinterpret_cast<float *>(smem + p.off_y);
  float *logit_s = reinterpret_cast<float *>(smem + p.off_logit);
  const Misc m = misc_view(smem + p.off_misc, A, A + (SHARED ? T : 0));
  // the scale-factor table (not for H = 2048 full-shape builds, where its
  // extra loads spill registers)
  constexpr bool kTab = !(FULL && SG == 2);
  __shared__ __align__(16) uint32_t e8m0_tab[256];  // static: its address is a constant, not a register
  const uint32_t stab = smem_addr(e8m0_tab);
  fill_e8m0_table(stab);  // published by the first barrier below

  const int nrw = (E + G - 1) / G;  // router warps in this kernel (host ensures <= 8)
  const uint32_t wsz = p.wbf ? 2u : 4u, xsz = p.xbf ? 2u : 4u;
  // router rows, then x rows, in ring stages not yet in use (stage 0 takes
  // the shared expert's gate/up slice from the start)
  constexpr int s0 = SHARED ? 1 : 0;  // gate/up ring items before the routed slots (the shared expert's)
  const uint32_t front = smem_addr(smem) + (s0 ? p.stage_bytes : 0u);
  const uint32_t xs_smem = front + (uint32_t)nrw * H * wsz;
  uint64_t *fbar = full + 4 * nstage;
  if (tid == 0) {
    for (int s = 0; s < 3 * nstage; ++s) mbar_init(smem_addr(&full[s]), 33);  // 1 expect_tx + 32 cp.async arrives
    for (int s = 0; s < nstage; ++s) mbar_init(smem_addr(&empty[s]), kGroup);
    mbar_init(smem_addr(fbar), 1);
    fence_mbar_init();
    m.scalars[4] = 0;
    m.scalars[5] = 0;
    // stage this CTA's router rows and the T activation rows with bulk copies
    int nrows = 0;
    for (int w = 0; w < nrw; ++w) nrows += (cta + G * w) < E;
    mbar_arrive_expect_tx(smem_addr(fbar), (uint32_t)nrows * H * wsz + (uint32_t)T * H * xsz);
    const uint64_t pol = policy_evict_first();
    for (int w = 0; w < nrw; ++w) {
      const int e = cta + G * w;
      if (e < E)
        bulk_g2s(front + (uint32_t)w * H * wsz, static_cast<const uint8_t *>(p.wr) + (int64_t)e * H * wsz, H * wsz,
                 smem_addr(fbar), pol);
    }
  }
  // Everything above reads only this launch's weights.  From here on the
  // kernel reads x and the workspace and writes its outputs, which the kernel
  // before it on the stream may still be using when this one was launched
  // early (programmatic dependent launch): wait for that kernel to complete.
  grid_dependency_wait();
  if (tid == 0) {
    const uint64_t pol = policy_evict_first();
    for (int t = 0; t < T; ++t)
      bulk_g2s(xs_smem + (uint32_t)t * H * xsz, static_cast<const uint8_t *>(p.x) + (int64_t)t * p.ld_x * xsz, H * xsz,
               smem_addr(fbar), pol);
  }
  __shared__ unsigned long long bar_base, ready_hold;
  if (tid == 32) {
    unsigned long long v, hold, rhold;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p.bar) : "memory");
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(hold) : "l"(p.bar + 1) : "memory");
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(rhold) : "l"(p.bar + 2) : "memory");
    bar_base = v / (unsigned long long)G * (unsigned long long)G + hold;
    ready_hold = rhold;  // 0 in use; a test sets it to make the readiness waits run out
  }
  __syncthreads();
  // the shared expert does not depend on the routing: its gate/up slice is
  // requested at once, into stage 0
  if constexpr (SHARED) {
    if (warp == kCons)
      gateup_copies(smem_addr(smem), smem_addr(&full[2 * nstage]), p.swg, p.swu, p.ssg, p.ssu, n0g, (uint32_t)Rg * (H / 2),
                    (uint32_t)Rg * nbH, p, H, nbH, policy_evict_first());
  }
  // a CTA that gives up before the ring runs first lets that copy land
  // (bounded), so no copy is still writing its shared memory when it exits
  auto settle_shared = [&]() {
    if (s0 && warp == kCons) mbar_wait(smem_addr(&full[2 * nstage]), 0, p.status);
  };
  if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(fbar), 0, p.status))) {
    settle_shared();
    return;
  }
  const unsigned long long base = bar_base;

  // ---------------------------------------------------------------- A
  // router: one warp per (router row of this CTA, token); Q8(x) on the rest
  int nrows_here = 0;
  for (int w = 0; w < nrw; ++w) nrows_here += (cta + G * w) < E;
  const int nunits = nrows_here * T;
  const int rwarps = min(nunits, kWarps / 2);
  if (warp < rwarps) {
#pragma unroll 1
    for (int u = warp; u < nunits; u += rwarps) {
      const int w = u / T, t = u - w * T;
      const float v = router_dot_smem(front + (uint32_t)w * H * wsz, p.wbf != 0, xs_smem + (uint32_t)t * H * xsz,
                                      p.xbf != 0, H);
      if (lane == 0) p.logits[(int64_t)t * E + cta + G * w] = v;
    }
  } else {
    const int q0 = tid - rwarps * 32, qn = kThreads - rwarps * 32;
    for (int idx = q0; idx < T * nbH; idx += qn) {
      const int t = idx / nbH, b = idx - t * nbH;
      float v[32];
      load32_smem(xs_smem + (uint32_t)t * H * xsz + 32u * b * xsz, p.xbf != 0, v);
      q8_to_row(v, act + (uint32_t)t * p.xrow, H, b);
    }
  }
  // CTA 0 clears the per-expert readiness words; barrier 1 publishes that
  // before any CTA can count on them
  if (cta == 0 && tid < kMaxA) p.bar[kSlotWord + tid] = 0ull;
  if (!grid_barrier(p.bar, base + (unsigned long long)G, 0, kThreads, &m.scalars[1], p.status)) {
    settle_shared();
    return;
  }

  // ---------------------------------------------------------------- A'
  for (int i = tid; i < T * E; i += kThreads) logit_s[i] = ldcg_f32(p.logits + i);
  __syncthreads();
  // top-k in two stages: a warp per (token, group of 32 experts), then a
  // warp per token merges the groups' candidates
  const int ngrp = (E + 31) >> 5;  // <= 8 on this path
  uint32_t *cand_key = reinterpret_cast<uint32_t *>(smem + p.off_cand);
  int *cand_id = reinterpret_cast<int *>(smem + p.off_cand) + T * 8 * 8;
  for (int u = warp; u < T * ngrp; u += kWarps) {
    const int t = u / ngrp, g = u - t * ngrp;
    topk_group_stage(logit_s + t * E, p.bias, E, k, g, cand_key + u * k, cand_id + u * k);
  }
  __syncthreads();
  // the producer's copies of one gate/up slice into ring stage st (the whole
  // producer warp calls it: the scale bytes may need per-lane copies)
  const uint64_t pol = policy_evict_first();
  const uint32_t gwb = (uint32_t)Rg * (H / 2), gsb = (uint32_t)Rg * nbH;
  auto issue_gateup = [&](int it, int expert) {
    const int st = it % nstage;
    gateup_copies(smem_addr(smem + (size_t)st * p.stage_bytes), smem_addr(&full[2 * st + ((it - s0) & 1)]), p.wg, p.wu,
                  p.sg, p.su, (int64_t)expert * I + n0g, gwb, gsb, p, H, nbH, pol);
  };
  int early = s0;  // gate/up ring items the producer already requested
  if (T == 1) {
    // one token: the producer warp merges, and requests slot j's gate/up slice
    // as soon as slot j is decided; the ring takes the slots in score order
    // (each expert has exactly one row, so no sort is needed)
    if (warp == kCons) {
      int id[8];
      float wv[8];
      auto pick = [&](int j, int e) {
        if (j + s0 < nstage && e >= 0 && e < E) issue_gateup(j + s0, e);
      };
      topk_merge_stage(cand_key, cand_id, ngrp * k, k, id, wv, pick);
      bool valid = false;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j < k && lane == j) {
          m.ids[j] = id[j];
          m.w[j] = wv[j];
          valid = id[j] >= 0 && id[j] < E;
          if (valid) {
            m.srt[j] = j;
            m.skey[j] = id[j];
            m.segb[j] = j;
            m.active[j] = id[j];
          } else if (cta == 0 && p.status) {
            atomicOr(p.status, MOE_DEV_BAD_EXPERT_ID);
          }
          if (cta == 0) {
            p.ids[j] = id[j];
            p.weights[j] = wv[j];
          }
        }
      }
      // invalid slots (NaN scores) come last in score order
      const int nv = __popc(__ballot_sync(0xffffffffu, valid));
      if (lane == 0) {
        m.segb[nv] = nv;
        m.scalars[0] = nv;
      }
    }
    __syncthreads();
    early = min(nstage, s0 + m.scalars[0]);
  } else {
    if (warp < T) {
      int id[8];
      float wv[8];
      topk_merge_stage(cand_key + warp * ngrp * k, cand_id + warp * ngrp * k, ngrp * k, k, id, wv);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j < k && lane == j) {
          m.ids[warp * k + j] = id[j];
          m.w[warp * k + j] = wv[j];
          if (cta == 0) {
            p.ids[(int64_t)warp * k + j] = id[j];
            p.weights[(int64_t)warp * k + j] = wv[j];
          }
        }
      }
    }
    __syncthreads();
    if (A <= 32) {
      if (warp == 0) rank_sort_warp(m, A, E, cta == 0 ? p.status : nullptr);
      __syncthreads();
    } else {
      rank_sort(m, A, E, cta == 0 ? p.status : nullptr);
    }
  }
  const int nact = m.scalars[0];
  // ring items: the shared expert's gate/up (if any), the routed slots'
  // gate/up, then the down items, dpp down slices each (the routed slots',
  // then the shared expert's)
  const int nslot = nact + s0;
  const int ndi = p.dpp == 2 ? (nslot + 1) >> 1 : (nslot + p.dpp - 1) / p.dpp;
  if (warp == kCons) {
    // ------------------------------------------------------------ producer
    // streams this CTA's gate/up slice of every active expert through the
    // ring, then its down slices, dpp slots per stage; once the first stages
    // are requested it asks for the down slices to be pulled into L2, so the
    // down copies (issued when gate/up stages free up) read from L2
    const uint32_t dw = (uint32_t)Rd * (I / 2), ds = (uint32_t)Rd * nbI;
    const int first = nslot < nstage ? nslot : nstage;
    // down slice j: a routed slot's expert (j < nact) or the shared expert
    auto dsrc = [&](int j, const uint8_t *&w, const uint8_t *&sc) {
      const bool shd = SHARED && j >= nact;
      const int64_t drow0 = (int64_t)(shd ? 0 : m.active[j]) * H + n0d;
      w = (shd ? p.swd : p.wd) + drow0 * (I / 2);
      sc = (shd ? p.ssd : p.sd) + drow0 * nbI;
    };
    // once the first stages are requested, pull the down slices into L2
    auto prefetch_down = [&]() {
      if (dw > 0) {
        for (int j = lane; j < nslot; j += 32) {
          const uint8_t *w, *sc;
          dsrc(j, w, sc);
          asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(w), "r"(dw) : "memory");
          if (p.d16) asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(sc), "r"(ds) : "memory");
        }
      }
    };
    if (early >= first) prefetch_down();
    int issued = early;
    for (int it = early; it < nslot + ndi; ++it) {
      int st, use;
      ring_slot(it, nslot, nstage, p.hqr, st, use);
      if (use >= 1 && !mbar_wait(smem_addr(&empty[st]), (use - 1) & 1, p.status)) break;
      const uint32_t sbase = smem_addr(smem + (size_t)st * p.stage_bytes);
      const uint32_t fb = smem_addr(&full[ring_full_bar(it, st, s0, nslot, nstage)]);
      if (it < nslot) {
        issue_gateup(it, m.active[it - s0]);  // it >= early >= s0: the shared item went out at the start
      } else {
        const int j0 = (it - nslot) * p.dpp, j1 = min(nslot, j0 + p.dpp);
        if (lane == 0) {
          mbar_arrive_expect_tx(fb, (uint32_t)(j1 - j0) * (dw + (p.d16 ? ds : 0u)));
          if (dw > 0) {
            for (int j = j0; j < j1; ++j) {
              const uint8_t *w, *sc;
              dsrc(j, w, sc);
              const uint32_t dst = sbase + (uint32_t)(j - j0) * p.dslot;
              bulk_g2s(dst, w, dw, fb, pol);
              if (p.d16) bulk_g2s(dst + p.dwreg, sc, ds, fb, pol);
            }
          }
        }
        if (!p.d16) {
          for (int j = j0; j < j1; ++j) {
            const uint8_t *w, *src;
            dsrc(j, w, src);
            const uint32_t dst = sbase + (uint32_t)(j - j0) * p.dslot + p.dwreg;
            for (uint32_t c = lane; c < ds / 4; c += 32) cp_async4(dst + 4 * c, src + 4 * c);
          }
        }
        cp_async_mbar_arrive_noinc(fb);
      }
      issued = it + 1;
      if (it == first - 1) prefetch_down();
    }
    // before exiting, the latest copy into every stage has landed: the last
    // item issued into each stage (1 + its index, 16 bits per stage; with hqr
    // the down items skip the last stage, so its latest copy can be a gate/up
    // item long before the end)
    uint64_t last = 0;
    for (int it = 0; it < issued; ++it) {
      int st, use;
      ring_slot(it, nslot, nstage, p.hqr, st, use);
      last = (last & ~(0xFFFFull << (16 * st))) | ((uint64_t)(it + 1) << (16 * st));
    }
    for (int st = 0; st < nstage; ++st) {
      const int i1 = (int)((last >> (16 * st)) & 0xFFFFu);
      if (i1) {
        int fbi;
        uint32_t par;
        ring_full(i1 - 1, s0, nslot, nstage, p.hqr, fbi, par);
        mbar_wait(smem_addr(&full[fbi]), par, p.status);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  // Gate/up: two groups of kGroup warps take alternate ring items (group g:
  // items g, g+2, ...), so two items are computed at once.  A unit is one
  // output row of the expert, both matrices in one warp, SwiGLU in the warp;
  // when a group has written its h slice of expert slot j it counts that in
  // the workspace word of slot j.
  // Down: once every slot is counted by all CTAs, all consumer warps
  // quantise every h row into shared memory at once (the region of Q8(x),
  // no longer read), then the groups take the down ring items (dpp slots
  // each, their slices already pulled into L2) in units of two rows of one
  // slot, and leave y in shared memory for the combine.  A warp whose wait
  // gave up stops computing but keeps arriving on the ring and on the named
  // barriers, so no other warp waits on it.  It still waits (bounded) for
  // each ring copy to land before it releases the stage, so the producer
  // never re-arms a stage with a copy in flight, unless a copy itself never
  // landed ("broken"): then it stops waiting on the ring.
  const int grp = warp / kGroup, gw = warp - grp * kGroup;
  const int gbar = 3 + grp;  // named barrier of this group
  bool dead = false;
  // the shared expert's item (ring item 0, landed long before the routed
  // ones): every consumer warp, units of (row, token); its rows extend the
  // sorted positions after the routed ones (srt = A + t), so the Q8(h) and
  // down passes below treat it as one more segment
  if (s0) {
    if (warp == 0) {
      const int nq0 = m.segb[nact];
      for (int t = lane; t < T; t += 32) m.srt[nq0 + t] = A + t;
      if (lane == 0) m.segb[nact + 1] = nq0 + T;
    }
    if (!dead) dead = !__all_sync(0xffffffffu, mbar_wait(smem_addr(&full[2 * nstage]), 0, p.status));
    if (!dead) {
      const uint32_t sbase = smem_addr(smem);
#pragma unroll 1
      for (int u = warp; u < Rg * T; u += kCons) {
        const int r = u / T, t = u - r * T;
        const uint32_t wrow[2] = {sbase + (uint32_t)r * (H / 2), sbase + p.gwreg + (uint32_t)r * (H / 2)};
        const uint32_t srow[2] = {sbase + 2 * p.gwreg + (uint32_t)r * nbH,
                                  sbase + 2 * p.gwreg + p.gsreg + (uint32_t)r * nbH};
        float acc[2];
        row_dot_stage_pn<2, SG, kTab>(act + (uint32_t)t * p.xrow, H, wrow, srow, stab, acc);
        float g, u2;
        reduce_pair(acc[0], acc[1], g, u2);
        if (lane == 0) p.sh_h[(int64_t)t * p.ld_sh_h + n0g + r] = __fmul_rn(silu(g), u2);
      }
    }
    bar_sync_named(1, kCons * 32);
    if (warp == 0 && lane == 0)
      asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p.bar + kSharedWord), "l"(1ull) : "memory");
    if (grp == 0 && lane == 0) mbar_arrive(smem_addr(&empty[0]));
  }
  // this group's next phase parity on its barrier of each stage (bit st)
  uint32_t gpar = 0;
  for (int it = s0 + grp, st = (s0 + grp) % nstage; it < nslot;
       it += 2, st = st + 2 >= nstage ? st + 2 - nstage : st + 2) {  // st: stage of item it
    const int js = it - s0;  // routed slot
    if (!dead)
      dead = !__all_sync(0xffffffffu, mbar_wait(smem_addr(&full[2 * st + grp]), (gpar >> st) & 1u, p.status));
    gpar ^= 1u << st;
    const uint32_t sbase = smem_addr(smem + (size_t)st * p.stage_bytes);
    if (!dead) {
      const int sb = m.segb[js], se = m.segb[js + 1];
#pragma unroll 1
      for (int r = gw; r < Rg; r += kGroup) {
        const uint32_t wrow[2] = {sbase + (uint32_t)r * (H / 2), sbase + p.gwreg + (uint32_t)r * (H / 2)};
        const uint32_t srow[2] = {sbase + 2 * p.gwreg + (uint32_t)r * nbH,
                                  sbase + 2 * p.gwreg + p.gsreg + (uint32_t)r * nbH};
#pragma unroll 1
        for (int q = sb; q < se; ++q) {
          const int a = m.srt[q];
          const int t = token_of(a, p.kdiv);
          float acc[2];
          row_dot_stage_pn<2, SG, kTab>(act + (uint32_t)t * p.xrow, H, wrow, srow, stab, acc);
          float g, u;
          reduce_pair(acc[0], acc[1], g, u);
          if (lane == 0) p.h[(int64_t)a * p.ld_h + n0g + r] = __fmul_rn(silu(g), u);
        }
      }
    }
    // this CTA's h slice of expert slot js is written: count it (release)
    bar_sync_named(gbar, kGroup * 32);
    if (gw == 0 && lane == 0)
      asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p.bar + kSlotWord + js), "l"(1ull) : "memory");
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&empty[st]));
  }

  // ---- down phase
  // once every slot is complete in every CTA (one warp polls the readiness
  // words), all consumer warps quantise every h row into shared memory
  if (dead && lane == 0) {  // in the gate/up phase only a ring copy that never landed makes a warp give up
    m.scalars[4] = 1;
    m.scalars[5] = 1;
  }
  bar_sync_named(1, kCons * 32);
  if (warp == 0) {
    bool ok = m.scalars[4] == 0;
    const unsigned long long ready = (unsigned long long)G + ready_hold;
    for (int j = lane; j < nact; j += 32) ok = ok && wait_count(p.bar + kSlotWord + j, ready, p.status);
    if (s0 && lane == 0) ok = ok && wait_count(p.bar + kSharedWord, ready, p.status);
    ok = __all_sync(0xffffffffu, ok);
    if (lane == 0 && !ok) m.scalars[4] = 1;
  }
  bar_sync_named(1, kCons * 32);
  dead = m.scalars[4] != 0;  // one answer for the whole CTA from here on
  bool broken = m.scalars[5] != 0;
  // Q8(h) rows by sorted position: the last ring stage (idle once every
  // gate/up item is consumed; the down items skip it) or the region of Q8(x)
  const uint32_t hq = smem_addr(smem + (p.hqr ? (size_t)(nstage - 1) * p.stage_bytes : (size_t)p.off_hq));
  const int nq = m.segb[nact];  // routed rows; the shared expert's T rows follow
  if (!dead) {
    const int ntask = 2 * (nq + s0 * T) * nbI;  // (row, block, half), one per lane
#pragma unroll 1
    for (int c = warp; 32 * c < ntask; c += kCons) {
      const int idx = 32 * c + lane;
      const bool valid = idx < ntask;
      const int blk = valid ? idx >> 1 : 0;
      const int ql = blk / nbI, b = blk - ql * nbI;
      const float *src = ((SHARED && ql >= nq) ? p.sh_h + (int64_t)(ql - nq) * p.ld_sh_h
                                               : p.h + (int64_t)m.srt[ql] * p.ld_h) + 32 * b + 16 * (idx & 1);
      float v[16];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const uint4 r = valid ? ldcg_v4(src + 4 * q4) : make_uint4(0, 0, 0, 0);
        v[4 * q4] = __uint_as_float(r.x);
        v[4 * q4 + 1] = __uint_as_float(r.y);
        v[4 * q4 + 2] = __uint_as_float(r.z);
        v[4 * q4 + 3] = __uint_as_float(r.w);
      }
      q8_pair_to_row(v, lane & 1, valid, hq + (uint32_t)ql * p.hrow, I, b);
    }
  }
  bar_sync_named(1, kCons * 32);
  // down ring items: every consumer warp takes every item; group g computes
  // the item's slices g, g + 2, ... (a unit is two rows of one slice sharing
  // the activation loads), then group 0 releases the stage.  Slice j < nact
  // is routed slot j; slice nact the shared expert (its y rows follow the
  // A routed ones in the slice buffer)
  uint32_t apar = s0 ? 1u : 0u;  // next phase parity of the all-warp barrier of each stage (bit st)
  for (int it = nslot; it < nslot + ndi; ++it) {
    int st, use;
    ring_slot(it, nslot, nstage, p.hqr, st, use);
    if (!broken && !__all_sync(0xffffffffu, mbar_wait(smem_addr(&full[2 * nstage + st]), (apar >> st) & 1u, p.status)))
      broken = dead = true;
    apar ^= 1u << st;
    if (!dead) {
      const int j0 = (it - nslot) * p.dpp, j1 = min(nslot, j0 + p.dpp);
      for (int j = j0 + grp; j < j1; j += 2) {
        const uint32_t sbase = smem_addr(smem + (size_t)st * p.stage_bytes) + (uint32_t)(j - j0) * p.dslot;
        const int sb = m.segb[j], se = m.segb[j + 1];
#pragma unroll 1
        for (int r = gw; r < Rd; r += 2 * kGroup) {
          const bool two = r + kGroup < Rd;
          const int r2 = two ? r + kGroup : r;  // one row left: both halves read row r
          const uint32_t wrow[2] = {sbase + (uint32_t)r * (I / 2), sbase + (uint32_t)r2 * (I / 2)};
          const uint32_t srow[2] = {sbase + p.dwreg + (uint32_t)r * nbI, sbase + p.dwreg + (uint32_t)r2 * nbI};
#pragma unroll 1
          for (int q = sb; q < se; ++q) {
            const int a = m.srt[q];
            float acc[2];
            row_dot_stage_pn<2, SD, kTab>(hq + (uint32_t)q * p.hrow, I, wrow, srow, stab, acc);
            float v0, v1;
            reduce_pair(acc[0], acc[1], v0, v1);
            if (lane == 0) {
              const bool ys = SHARED && a >= A;  // the shared expert's row
              float *yo = ys ? p.sh_y : p.y;      // optional global copies
              const int64_t yrow = ys ? (int64_t)(a - A) * p.ld_sh_y : (int64_t)a * p.ld_y;
              yslice[a * p.Rd + r] = v0;
              if (yo) yo[yrow + n0d + r] = v0;
              if (two) {
                yslice[a * p.Rd + r2] = v1;
                if (yo) yo[yrow + n0d + r2] = v1;
              }
            }
          }
        }
      }
    }
    bar_sync_named(1, kCons * 32);
    if (grp == 0 && lane == 0) mbar_arrive(smem_addr(&empty[st]));
  }
  bar_sync_named(1, kCons * 32);
  // combine of this CTA's output slice, slot order
  for (int idx = tid; idx < T * Rd; idx += kCons * 32) {
    const int t = idx / Rd, r = idx - t * Rd;
    const float *wt = m.w + t * k;
    // (as the stand-alone combine: a slot of weight exactly 0 adds nothing)
    float acc = wt[0] != 0.0f ? __fmul_rn(wt[0], yslice[(t * k) * p.Rd + r]) : 0.0f;
    for (int j = 1; j < k; ++j)
      if (wt[j] != 0.0f) acc = __fmaf_rn(wt[j], yslice[(t * k + j) * p.Rd + r], acc);
    if (s0) acc = __fadd_rn(acc, yslice[(A + t) * p.Rd + r]);  // the shared expert's join
    p.out[(int64_t)t * p.ld_out + n0d + r] = acc;
  }
}

using DecodeKernel = void (*)(DecodeArgs);

// The single-launch kernel for a shape.  With a shared expert, only the
// DeepSeek-size shapes and the smallest one are instantiated (null otherwise).
DecodeKernel pick(int sg, int sd, bool full, bool shared) {
  if (shared) {
    if (full && sg == 4 && sd == 2) return decode_kernel<4, 2, true, true>;
    if (full && sg == 4 && sd == 4) return decode_kernel<4, 4, true, true>;
    if (full && sg == 2 && sd == 4) return decode_kernel<2, 4, true, true>;
    if (full && sg == 2 && sd == 2) return decode_kernel<2, 2, true, true>;
    if (!full && sg == 1 && sd == 1) return decode_kernel<1, 1, false, true>;
    return nullptr;
  }
  if (full) {
    if (sg == 4 && sd == 2) return decode_kernel<4, 2, true, false>;
    if (sg == 4 && sd == 4) return decode_kernel<4, 4, true, false>;
    if (sg == 2 && sd == 4) return decode_kernel<2, 4, true, false>;
    if (sg == 2 && sd == 2) return decode_kernel<2, 2, true, false>;
  }
  if (sg == 1 && sd == 1) return decode_kernel<1, 1, false, false>;
  if (sg == 2 && sd == 1) return decode_kernel<2, 1, false, false>;
  if (sg == 2 && sd == 2) return decode_kernel<2, 2, false, false>;
  if (sg == 4 && sd == 2) return decode_kernel<4, 2, false, false>;
  if (sg == 4 && sd == 4) return decode_kernel<4, 4, false, false>;
  if (sg == 1 && sd == 2) return decode_kernel<1, 2, false, false>;
  if (sg == 2 && sd == 4) return decode_kernel<2, 4, false, false>;
  if (sg == 4 && sd == 1) return decode_kernel<4, 1, false, false>;
  if (sg == 1 && sd == 4) return decode_kernel<1, 4, false, false>;
  return nullptr;
}

// The kernel instantiation for H, I (K blocks per lane rounded up to 1, 2 or
// 4), or null.
DecodeKernel kernel_for(int H, int I, bool shared, int &SGp, int &SDp, bool &full) {
  const int SG = (H / 32 + 31) / 32, SD = (I / 32 + 31) / 32;
  SGp = SG == 3 ? 4 : SG;
  SDp = SD == 3 ? 4 : SD;
  full = H == 1024 * SGp && I == 1024 * SDp;
  return pick(SGp, SDp, full, shared);
}

uint32_t align16(uint64_t v) { return (uint32_t)((v + 15) & ~uint64_t(15)); }

// Shared-memory plan of the fused kernel for p.T/H/E/k/I on a device with
// `optin` bytes per CTA and G SMs.  Returns false when it does not fit.
bool plan_smem(DecodeArgs &p, int G, int optin, size_t *smem_out) {
  const int H = p.H, I = p.I, E = p.E, T = p.T, A = p.A;
  const int nbH = H / 32, nbI = I / 32;
  const int Rg = (I + G - 1) / G, Rd = (H + G - 1) / G;
  p.Rd = Rd;
  p.Rg = Rg;
  p.gwreg = (uint32_t)Rg * (H / 2);
  p.gsreg = align16((uint64_t)Rg * nbH);
  p.dwreg = (uint32_t)Rd * (I / 2);
  const uint32_t gstage = 2 * (p.gwreg + p.gsreg), dstage = p.dwreg + align16((uint64_t)Rd * nbI);
  p.dslot = (dstage + 127u) & ~127u;
  p.stage_bytes = ((gstage > p.dslot ? gstage : p.dslot) + 127u) & ~127u;
  p.dpp = (int)(p.stage_bytes / p.dslot);
  p.xrow = (uint32_t)H + 4u * nbH;  // codes, then the block scales
  p.hrow = (uint32_t)I + 4u * nbI;
  const uint64_t act_bytes = align16((uint64_t)T * p.xrow);
  // Q8(h) of every assignment, in the region of Q8(x): the down phase
  // starts after every gate/up unit has read its activations
  const int rows = A + (p.shared ? T : 0);  // h / y rows: the assignments, then the shared expert's tokens
  const uint64_t hq_bytes = align16((uint64_t)rows * p.hrow);
  const uint64_t y_bytes = align16((uint64_t)rows * Rd * 4);
  const uint64_t logit_bytes = align16((uint64_t)T * E * 4);
  const uint64_t cand_bytes = (uint64_t)T * 8 * 8 * 8;  // top-k candidates: T x 8 groups x 8 (key, id)
  const uint64_t misc_bytes = align16(4ull * (5 * A + rows + 2 + 8));  // ids w srt skey segb active + 8 scalars
  // (+ 1 KB: the kernel's static e8m0 table comes out of the same per-block budget)
  const uint64_t small = 32ull * 8 + y_bytes + logit_bytes + cand_bytes + misc_bytes + 1024;
  const uint64_t budget = (uint64_t)optin - 1024;
  auto stages = [&](uint64_t tail) { return tail >= budget ? 0 : std::min<int>(4, (int)((budget - tail) / p.stage_bytes)); };
  // Q8(h) in the region of Q8(x) (both outside the ring), or in the last
  // ring stage during the down phase when that gives the ring one more stage
  // (the down items then cycle through one stage fewer)
  const int ns_apart = stages(small + std::max(act_bytes, hq_bytes)), ns_in = stages(small + act_bytes);
  p.hqr = hq_bytes <= p.stage_bytes && ns_in >= 3 && ns_in > ns_apart;
  const uint64_t tail = small + (p.hqr ? act_bytes : std::max(act_bytes, hq_bytes));
  const int ns = p.hqr ? ns_in : ns_apart;
  if (ns < 2) return false;
  p.nstage = ns;
  // the ring area first holds the CTA's router rows and the activation rows
  const uint64_t front = (uint64_t)((E + G - 1) / G) * H * (p.wbf ? 2 : 4) + (uint64_t)T * H * (p.xbf ? 2 : 4);
  const uint64_t ring = std::max<uint64_t>((uint64_t)ns * p.stage_bytes,
                                          (p.shared ? p.stage_bytes : 0) + align16(front));
  if (ring + tail > budget) return false;
  p.off_bars = (uint32_t)ring;
  p.off_act = p.off_bars + 32 * 8;  // 4 NS + 1 <= 17 mbarriers; the activation rows stay 128-byte aligned
  p.off_hq = p.off_act;
  p.off_y = p.off_act + (uint32_t)(p.hqr ? act_bytes : std::max(act_bytes, hq_bytes));
  p.off_logit = p.off_y + (uint32_t)y_bytes;
  p.off_cand = p.off_logit + (uint32_t)logit_bytes;
  p.off_misc = p.off_cand + (uint32_t)cand_bytes;
  *smem_out = p.off_misc + misc_bytes;
  return true;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" size_t moe_decode_workspace_bytes(void) { return 8 * (kSlotWord + kMaxA); }

namespace {

int max_tokens(int H, int E, int k, int I, bool shared) {
  if (H <= 0 || E <= 0 || k <= 0 || k > 8 || I <= 0 || H % 128 || I % 128 || H > 4096 || I > 4096 || E > 256) return 0;
  int dev = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
  const int G = sm_count();
  if ((E + G - 1) / G > 8) return 0;
  int sgp = 0, sdp = 0;
  bool full = false;
  if (!kernel_for(H, I, shared, sgp, sdp, full)) return 0;
  int best = 0;
  for (int T = 1; T <= kCons && T * k <= kMaxA - (shared ? 1 : 0); ++T) {
    DecodeArgs p{};
    p.T = T; p.H = H; p.E = E; p.k = k; p.I = I; p.A = T * k;
    p.wbf = 0; p.xbf = 0;  // fp32 router and activations: the larger staging
    p.shared = shared;
    size_t smem = 0;
    if (plan_smem(p, G, optin, &smem)) best = T;
    else break;
  }
  return best;
}

}  // namespace

extern "C" int moe_decode_max_tokens(int H, int E, int k, int I) { return max_tokens(H, E, k, I, false); }

extern "C" int moe_decode_max_tokens_shared(int H, int E, int k, int I) { return max_tokens(H, E, k, I, true); }

namespace moe {

moe_status decode_forward(const char *name, const void *x, moe_dtype x_dtype, int64_t ld_x, const void *w_router,
                          moe_dtype w_dtype, const float *bias, const uint8_t *wg, const uint8_t *sg, const uint8_t *wu,
                          const uint8_t *su, const uint8_t *wd, const uint8_t *sd, int T, int H, int E, int k, int I,
                          float *out, int64_t ld_out, float *logits, int32_t *ids, float *weights, float *h,
                          int64_t ld_h, float *y, int64_t ld_y, void *workspace, size_t ws_bytes,
                          const SharedArgs *sh, bool clear_ws, void *stream) {
  if (T < 0 || H <= 0 || E <= 0 || k <= 0 || I <= 0) return fail(MOE_ERR_INVALID_ARG, "%s: T=%d H=%d E=%d k=%d I=%d", name, T, H, E, k, I);
  if (x_dtype != MOE_F32 && x_dtype != MOE_BF16) return fail(MOE_ERR_INVALID_ARG, "%s: bad x dtype", name);
  if (w_dtype != MOE_F32 && w_dtype != MOE_BF16) return fail(MOE_ERR_INVALID_ARG, "%s: bad router dtype", name);
  if (H % 128 || I % 128) return fail(MOE_ERR_INVALID_ARG, "%s: H=%d and I=%d must be multiples of 128", name, H, I);
  if (H > 4096 || I > 4096) return fail(MOE_ERR_UNSUPPORTED, "%s: H, I <= 4096", name);
  if (E > 256) return fail(MOE_ERR_UNSUPPORTED, "%s: E=%d > 256 (use the stage calls)", name, E);
  if (k > 8 || k > E) return fail(MOE_ERR_INVALID_ARG, "%s: k=%d must be <= min(E, 8)", name, k);
  if (T == 0) return MOE_OK;
  const int A = T * k;
  if (A > kMaxA || T > kCons) return fail(MOE_ERR_UNSUPPORTED, "%s: T*k=%d beyond the fused decode path (<= %d)", name, A, kMaxA);
  if (sh) {  // the shared expert's readiness word is the last one
    if (A > kMaxA - 1) return fail(MOE_ERR_UNSUPPORTED, "%s: T*k=%d beyond the fused path with a shared expert (<= %d)", name, A, kMaxA - 1);
    if (!sh->wg || !sh->sg || !sh->wu || !sh->su || !sh->wd || !sh->sd || !sh->h)
      return fail(MOE_ERR_INVALID_ARG, "%s: null shared-expert pointer", name);
    if ((uintptr_t)sh->wg % 16 || (uintptr_t)sh->wu % 16 || (uintptr_t)sh->wd % 16 || (uintptr_t)sh->sg % 4 ||
        (uintptr_t)sh->su % 4 || (uintptr_t)sh->sd % 4)
      return fail(MOE_ERR_INVALID_ARG, "%s: shared-expert weights must be 16-byte aligned, scale bytes 4-byte aligned", name);
    if (sh->ld_h < I || sh->ld_h % 4 || (uintptr_t)sh->h % 16 || (sh->y && sh->ld_y < H))
      return fail(MOE_ERR_INVALID_ARG, "%s: bad shared-expert output strides", name);
  }
  if (!x || !w_router || !wg || !sg || !wu || !su || !wd || !sd || !out || !logits || !ids || !weights || !h || !workspace)
    return fail(MOE_ERR_INVALID_ARG, "%s: null pointer", name);
  if (ws_bytes < moe_decode_workspace_bytes() || (uintptr_t)workspace % 8) return fail(MOE_ERR_INVALID_ARG, "%s: workspace too small", name);
  const int xes = x_dtype == MOE_BF16 ? 2 : 4;
  if (ld_x < H || (ld_x * xes) % 16 || (uintptr_t)x % 16 || (uintptr_t)w_router % 16) return fail(MOE_ERR_INVALID_ARG, "%s: x / router must be 16-byte aligned with 16-byte row strides", name);
  if ((uintptr_t)wg % 16 || (uintptr_t)wu % 16 || (uintptr_t)wd % 16) return fail(MOE_ERR_INVALID_ARG, "%s: weights must be 16-byte aligned", name);
  if ((uintptr_t)sg % 4 || (uintptr_t)su % 4 || (uintptr_t)sd % 4) return fail(MOE_ERR_INVALID_ARG, "%s: scale bytes must be 4-byte aligned", name);
  if (ld_out < H || ld_h < I || (ld_h % 4) || (uintptr_t)h % 16 || (y && ld_y < H)) return fail(MOE_ERR_INVALID_ARG, "%s: bad output strides", name);

  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_fail(err, name);
  int optin = 0, coop = 0;
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
  if (!coop) return fail(MOE_ERR_UNSUPPORTED, "%s: device has no cooperative launch", name);
  const int G = sm_count();
  if ((E + G - 1) / G > 8) return fail(MOE_ERR_UNSUPPORTED, "%s: too many experts per SM", name);
  const int nbH = H / 32, nbI = I / 32;
  int SGp = 0, SDp = 0;
  bool full = false;
  DecodeKernel kern = kernel_for(H, I, sh != nullptr, SGp, SDp, full);
  if (!kern) return fail(MOE_ERR_UNSUPPORTED, "%s: shape", name);

  DecodeArgs p{};
  p.x = x; p.ld_x = ld_x; p.xbf = x_dtype == MOE_BF16;
  p.wr = w_router; p.wbf = w_dtype == MOE_BF16; p.bias = bias;
  p.wg = wg; p.sg = sg; p.wu = wu; p.su = su; p.wd = wd; p.sd = sd;
  p.T = T; p.H = H; p.E = E; p.k = k; p.I = I; p.A = A;
  p.kdiv = kdiv_of(k);
  p.out = out; p.ld_out = ld_out; p.logits = logits; p.ids = ids; p.weights = weights;
  p.h = h; p.ld_h = ld_h; p.y = y; p.ld_y = ld_y;
  p.bar = static_cast<unsigned long long *>(workspace);
  p.status = device_status_word();
  if (sh) {
    p.shared = 1;
    p.swg = sh->wg; p.ssg = sh->sg; p.swu = sh->wu; p.ssu = sh->su; p.swd = sh->wd; p.ssd = sh->sd;
    p.sh_h = sh->h; p.ld_sh_h = sh->ld_h; p.sh_y = sh->y; p.ld_sh_y = sh->ld_y;
  }

  size_t smem = 0;
  if (!plan_smem(p, G, optin, &smem)) return fail(MOE_ERR_UNSUPPORTED, "%s: T=%d does not fit the fused path's shared memory", name, T);

  p.g16 = nbH % 16 == 0 && (uintptr_t)sg % 16 == 0 && (uintptr_t)su % 16 == 0 &&
          (!sh || ((uintptr_t)sh->sg % 16 == 0 && (uintptr_t)sh->su % 16 == 0));
  p.d16 = nbI % 16 == 0 && (uintptr_t)sd % 16 == 0 && (!sh || (uintptr_t)sh->sd % 16 == 0);

  // the dynamic limit leaves room for the static shared memory (the e8m0 table and a few words)
  const moe_status ast = ensure_smem_attr(reinterpret_cast<const void *>(kern), optin - 2048, name);
  if (ast != MOE_OK) return ast;
  if (clear_ws) {  // every check has passed: only now is anything enqueued
    err = cudaMemsetAsync(workspace, 0, moe_decode_workspace_bytes(), static_cast<cudaStream_t>(stream));
    if (err != cudaSuccess) return cuda_fail(err, name);
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(G);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  // cooperative (every CTA resident: the grid barrier) and programmatic
  // (this launch may begin while the kernel before it finishes; it waits for
  // it before reading x or the workspace).  Without programmatic launches the
  // kernel runs unchanged: its wait then returns at once.
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  static std::atomic<int> pdl{1};  // cleared if the runtime refuses the pair
  cfg.numAttrs = pdl.load() ? 2 : 1;
  err = cudaLaunchKernelEx(&cfg, kern, p);
  if (err != cudaSuccess && cfg.numAttrs == 2) {
    (void)cudaGetLastError();
    pdl.store(0);
    cfg.numAttrs = 1;
    err = cudaLaunchKernelEx(&cfg, kern, p);
  }
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, name);
}

}  // namespace moe

extern "C" moe_status moe_decode_forward(const void *x, moe_dtype x_dtype, int64_t ld_x, const void *w_router,
                                         moe_dtype w_dtype, const float *bias, const uint8_t *wg, const uint8_t *sg,
                                         const uint8_t *wu, const uint8_t *su, const uint8_t *wd, const uint8_t *sd,
                                         int T, int H, int E, int k, int I, float *out, int64_t ld_out,
                                         float *logits, int32_t *ids, float *weights, float *h, int64_t ld_h,
                                         float *y, int64_t ld_y, void *workspace, size_t ws_bytes, void *stream) {
  return decode_forward("moe_decode_forward", x, x_dtype, ld_x, w_router, w_dtype, bias, wg, sg, wu, su, wd, sd, T, H,
                        E, k, I, out, ld_out, logits, ids, weights, h, ld_h, y, ld_y, workspace, ws_bytes, nullptr,
                        false, stream);
}

extern "C" moe_status moe_decode_forward_shared(const void *x, moe_dtype x_dtype, int64_t ld_x, const void *w_router,
                                                moe_dtype w_dtype, const float *bias, const uint8_t *wg,
                                                const uint8_t *sg, const uint8_t *wu, const uint8_t *su,
                                                const uint8_t *wd, const uint8_t *sd, const uint8_t *shared_wg,
                                                const uint8_t *shared_sg, const uint8_t *shared_wu,
                                                const uint8_t *shared_su, const uint8_t *shared_wd,
                                                const uint8_t *shared_sd, int T, int H, int E, int k, int I,
                                                float *out, int64_t ld_out, float *logits, int32_t *ids,
                                                float *weights, float *h, int64_t ld_h, float *y, int64_t ld_y,
                                                float *shared_h, int64_t ld_shared_h, float *shared_y,
                                                int64_t ld_shared_y, void *workspace, size_t ws_bytes, void *stream) {
  const SharedArgs sh{shared_wg, shared_sg, shared_wu, shared_su, shared_wd, shared_sd,
                      shared_h, ld_shared_h, shared_y, ld_shared_y};
  return decode_forward("moe_decode_forward_shared", x, x_dtype, ld_x, w_router, w_dtype, bias, wg, sg, wu, su, wd, sd,
                        T, H, E, k, I, out, ld_out, logits, ids, weights, h, ld_h, y, ld_y, workspace, ws_bytes, &sh,
                        false, stream);
}
