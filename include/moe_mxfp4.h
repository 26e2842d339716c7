/*
 * moe_mxfp4.h -- C ABI of the GB300 (sm_103a) MXFP4 routed-expert MoE layer.
 *
 * One MoE layer forward is six stream-ordered calls:
 *
 *   moe_route_topk           router logits + top-k + routing weights
 *   moe_sort_tokens          group the token->expert assignments by expert
 *   act_quant_q8             Q8 (int8 per 32 + fp32 scale) of the activations
 *   moe_mxfp4_gateup_swiglu  h = silu(Wg x) * (Wu x) per assignment (MXFP4 weights)
 *   act_quant_q8             Q8 of h
 *   moe_mxfp4_down           y = Wd h per assignment
 *   moe_combine              out[t] = sum_j w[t,j] * y[t*k+j], slot order
 *
 * and, for a layer with a shared expert, the stage calls on its one-expert
 * weight set followed by moe_join_add (out += ys).
 *
 * It follows the layer as the DeepSeek-V4-Flash pages describe it:
 *  - "DeepSeek-V4-Flash on AMD gfx90a: Correctness Recovery and Inference
 *    Performance Engineering": Fig. 1 (router top-6 -> routed experts gate/up ->
 *    down -> add partials), §6.1 (packed 4-bit FP4 weights, online INT8 per-32
 *    activation quantisation, E2M1 nibbles as 0,±1,..,±12, integer dot then
 *    activation and E8M0 scaling), §7.1 item 8 (expert sorter), §8.2 (FP32 top-k
 *    partials and a fixed reduction), §5.3 (deterministic top-k ties by logical id);
 *  - "Optimizing DeepSeek V4 Flash Inference on a Strix Halo Pair": "MXFP4
 *    routed-expert kernels" and "The exact-rows contract" (one weight pass
 *    serves K resident rows; every row keeps the one-row arithmetic; explicit
 *    output strides);
 *  - "feat(ds4): add concurrent serving on Strix Halo and R9700 + Strix":
 *    "Reduce expert-route overhead" (negative sentinels for unowned slots).
 *
 * Conventions shared by every call
 *  - All pointers are DEVICE pointers owned by the caller; the library never
 *    allocates, frees or retains them, and never synchronises the stream.
 *    Its own scratch: the tensor-core path of the expert projections (calls
 *    of 17 rows or more) writes the activations' E2M1 planes to a buffer it
 *    allocates and frees on the call's stream (stream-ordered, from a memory
 *    pool of the library's that keeps its memory between calls; about
 *    6 * (K / 2) + 6 * K / 32 + 4 bytes per sorted position); the single-
 *    launch decode calls need the workspace they are given and nothing else.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *    enqueue work; results are ready when the stream reaches them.
 *  - Matrices are row-major; ld_* are row strides in ELEMENTS of that array.
 *  - Validation of sizes, strides, alignment and null pointers happens on the
 *    host before any launch; a failing call enqueues nothing and returns
 *    MOE_ERR_INVALID_ARG (or MOE_ERR_UNSUPPORTED), with the reason in
 *    moe_last_error().  Launch failures return MOE_ERR_CUDA.
 *  - Values the host cannot see (expert ids, sort offsets) are bounds-checked
 *    on the device; an out-of-range value is skipped and raises a bit in the
 *    device status word, read by moe_device_status().
 *  - Deterministic: no floating-point atomics; the same call on the same
 *    inputs gives the same bits.
 *  - Exact rows ("The exact-rows contract" of the Strix Halo record): for
 *    T <= 16 rows every row's result is computed by the arithmetic of the
 *    one-row call, so a T-row call gives, row by row, the bits of T one-row
 *    calls (stage calls and the single-launch decode path alike).  Routing,
 *    the sorter, Q8 and the combine keep that for every T.  From 17 rows on,
 *    the expert projections of experts with more than 4 rows run on the
 *    tensor cores, which take each activation value as six E2M1 planes with
 *    their own E8M0 scales (about 1e-5 of the output's RMS, exact for unit
 *    scales) and accumulate the whole reduction in fp32: those rows agree
 *    with the one-row call within the layer's tolerance, not bit for bit.
 *  - Requires an sm_103a device (GB300); MOE_ERR_UNSUPPORTED otherwise.
 *
 * Weight layout (one layer; E experts; all contiguous, 16-byte aligned):
 *  - wg, wu: uint8 [E][I][H/2]; byte c of a row holds element 2c in its low
 *    nibble and 2c+1 in its high nibble; a nibble is an E2M1 code (OCP MX).
 *  - sg, su: uint8 [E][I][H/32]; one E8M0 byte (2^(u-127); 255 = NaN) per 32
 *    consecutive elements of a row.  Every byte 0..255 is accepted; a block
 *    term is I_b * (xs_b * 2^(u-128)) in fp32, so results match the exact
 *    value within fp32 rounding wherever that scale product and the sums
 *    are finite fp32 numbers (byte 255 makes the outputs it reaches NaN).
 *  - wd: uint8 [E][H][I/2], sd: uint8 [E][H][I/32], same conventions.
 */
#ifndef MOE_MXFP4_H
#define MOE_MXFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exported from libmoe_mxfp4.so (everything else in it is hidden). */
#ifndef MOE_API
#define MOE_API __attribute__((visibility("default")))
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1, /* bad size, stride, alignment or null pointer; nothing enqueued */
    MOE_ERR_UNSUPPORTED = 2, /* shape or device outside what this build handles */
    MOE_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
    MOE_ERR_DEVICE = 4       /* moe_device_status: the device status word was non-zero */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

/* Device status bits (moe_device_status). */
#define MOE_DEV_BAD_EXPERT_ID 0x1u  /* an expert id outside [0, E) was skipped */
#define MOE_DEV_BAD_ROW 0x2u        /* a sorted entry or offset outside its range was skipped */
#define MOE_DEV_WAIT_TIMEOUT 0x4u   /* a bounded wait on a copy gave up; outputs are incomplete */

/* Message for the last non-OK status returned on this host thread. */
MOE_API const char *moe_last_error(void);

/* ABI version of this header (bumped on any signature change or addition;
 * 2 adds moe_join_add, moe_decode_max_tokens_shared and
 * moe_decode_forward_shared; 3 adds moe_mxf4_mma_probe; 4 adds
 * moe_mxfp4_down_combine). */
MOE_API int moe_abi_version(void);
#define MOE_ABI_VERSION 4

/* Synchronises `stream`, then reads and clears the device status word of the
 * current device into *flags (may be NULL).  Returns MOE_ERR_DEVICE when the
 * word was non-zero.  Test and debugging aid; not for the hot path. */
MOE_API moe_status moe_device_status(void *stream, uint32_t *flags);

/* ---------------------------------------------------------------- routing */

/* Router and top-k.  Fig. 1 of the gfx90a report ("Router Top-6"), with §5.3's
 * deterministic selection.
 *  x        [T][ld_x] activations (MOE_F32 or MOE_BF16), first H columns used.
 *  w_router [E][H] router weights (MOE_F32 or MOE_BF16).
 *  bias     [E] fp32 logit bias, or NULL.
 *  logits   [T][E] fp32 output: the router logits (no bias), each the fp32
 *           result of one fixed summation order -- H is cut into chunks of 8
 *           consecutive elements, chunk c feeds partial sum c mod 32 (chunks in
 *           increasing order, one fused multiply-add per element), then the 32
 *           partials are added pairwise p[l] += p[l+s], s = 16, 8, 4, 2, 1.
 *  ids      [T][k] int32 output: the k experts of largest score = logit + bias,
 *           ties to the lower id, in descending score order.  A NaN score
 *           is never taken; a slot for which only NaN scores are left gets
 *           the id 0x7fffffff (no expert) and weight 0.
 *  weights  [T][k] fp32 output: sigmoid(score) renormalised over the k slots.
 * Requires H % 8 == 0, 1 <= k <= min(E, 8), E <= 1024; x and w_router
 * 16-byte aligned, ld_x * element size a multiple of 16 bytes. */
MOE_API moe_status moe_route_topk(const void *x, moe_dtype x_dtype, int64_t ld_x,
                          const void *w_router, moe_dtype w_dtype, const float *bias,
                          int T, int H, int E, int k,
                          float *logits, int32_t *ids, float *weights, void *stream);

/* ---------------------------------------------------------------- sorter */

/* Length the `sorted` array needs: T*k + E*(tile_rows-1). */
MOE_API int64_t moe_sort_tokens_capacity(int T, int k, int E, int tile_rows);

/* Stable counting sort of the A = T*k assignments a = t*k + j by expert (the
 * expert sorter of the gfx90a report, §7.1 item 8).
 *  ids      [T][k] expert ids.
 *  offsets  [E+1] output: expert e owns sorted[offsets[e] .. offsets[e+1]).
 *  sorted   [cap] output: assignment ids, increasing within each expert; each
 *           expert's segment is padded to a multiple of tile_rows with -1
 *           (the negative sentinel of the lucebox PR, "Reduce expert-route
 *           overhead").  Entries past offsets[E] are not written.
 *  inv      [T*k] output: position of assignment a in `sorted` (-1 if its id
 *           was out of range).
 * Requires E <= 1024, tile_rows >= 1, cap >= moe_sort_tokens_capacity(). */
MOE_API moe_status moe_sort_tokens(const int32_t *ids, int T, int k, int E, int tile_rows,
                           int32_t *offsets, int32_t *sorted, int64_t cap, int32_t *inv,
                           void *stream);

/* ---------------------------------------------------------------- Q8 */

/* Q8 quantisation, per row and per block of 32 columns (the gfx90a report,
 * §6.1 "online BF16 activation quantization to INT8 per 32 elements"):
 * amax = max|x|, scale = amax/127 (IEEE fp32 division), q = round-to-nearest-
 * even(x * (1/scale)) clamped to [-127, 127]; amax = 0 gives scale 0, q = 0.
 *  x      [rows][ld_x] MOE_F32 or MOE_BF16 (finite values).
 *  q      [rows][ld_q] int8 output;  scale [rows][ld_s] fp32 output.
 * Requires cols % 32 == 0; x and q 16-byte aligned with row strides that are
 * multiples of 16 bytes. */
MOE_API moe_status act_quant_q8(const void *x, moe_dtype x_dtype, int rows, int cols, int64_t ld_x,
                        int8_t *q, int64_t ld_q, float *scale, int64_t ld_s, void *stream);

/* ---------------------------------------------------------------- experts */

/* Gate/up MXFP4 projections with SwiGLU (the Strix Halo record, "MXFP4
 * routed-expert kernels": register-resident gate/up reductions; the lucebox PR
 * folds SwiGLU into the gate/up pass).  For every assignment a in `sorted`
 * (entries < 0 skipped) with expert e = the segment it sits in, token t = a/k:
 *   G[i] = sum_b I_b * xs[t,b] * 2^(sg[e,i,b]-128), U[i] likewise,
 *   I_b  = exact integer sum over the 32 elements of block b of
 *          xq[t,.] * (2 * E2M1 value)  (twice the E2M1 value is an integer),
 *   h[a, i] = silu(G[i]) * U[i],   silu(g) = g / (1 + exp(-g)).
 * Scaled block terms are accumulated in fp32 in a fixed order; for T <= 16
 * that order does not depend on the number of rows (see "Exact rows" above).
 * One pass over an expert's weights serves all its rows.
 *  xq [T][ld_xq] int8, xs [T][ld_xs] fp32  (Q8 of the activations).
 *  offsets [E+1], sorted [cap] from moe_sort_tokens.
 *  h [T*k][ld_h] fp32 output; rows of assignments not in `sorted` untouched.
 * Requires H % 128 == 0, H <= 4096, I % 128 == 0; xq 16-byte aligned, ld_xq a
 * multiple of 16; weights 16-byte aligned. */
MOE_API moe_status moe_mxfp4_gateup_swiglu(const int8_t *xq, int64_t ld_xq, const float *xs, int64_t ld_xs,
                                   const uint8_t *wg, const uint8_t *sg,
                                   const uint8_t *wu, const uint8_t *su,
                                   const int32_t *offsets, const int32_t *sorted, int64_t cap,
                                   int T, int k, int E, int H, int I,
                                   float *h, int64_t ld_h, void *stream);

/* The same projections without the activation: g[a,i] = G[i], u[a,i] = U[i]
 * (same arithmetic, same bits as the values silu() is applied to above).
 * g and u are [T*k][ld_gu] fp32 outputs. */
MOE_API moe_status moe_mxfp4_gateup(const int8_t *xq, int64_t ld_xq, const float *xs, int64_t ld_xs,
                            const uint8_t *wg, const uint8_t *sg,
                            const uint8_t *wu, const uint8_t *su,
                            const int32_t *offsets, const int32_t *sorted, int64_t cap,
                            int T, int k, int E, int H, int I,
                            float *g, float *u, int64_t ld_gu, void *stream);

/* Down MXFP4 projection (the gfx90a report, §6.1 "top-6 slots in the down
 * projection", §8.2 FP32 top-k partials): for every assignment a in `sorted`
 * with expert e, y[a, n] = sum_b I_b * hs[a,b] * 2^(sd[e,n,b]-128), n < H,
 * same block dot and fixed fp32 order as above.
 *  hq [T*k][ld_hq] int8, hs [T*k][ld_hs] fp32 (Q8 of h).
 *  y  [T*k][ld_y] fp32 output.
 * Requires I % 128 == 0, I <= 4096, H % 128 == 0; hq 16-byte aligned, ld_hq a
 * multiple of 16; weights 16-byte aligned. */
MOE_API moe_status moe_mxfp4_down(const int8_t *hq, int64_t ld_hq, const float *hs, int64_t ld_hs,
                          const uint8_t *wd, const uint8_t *sd,
                          const int32_t *offsets, const int32_t *sorted, int64_t cap,
                          int T, int k, int E, int H, int I,
                          float *y, int64_t ld_y, void *stream);

/* Down projection and routing-weighted combine in one pass (the down
 * consumer of "DeepSeek-V4-Flash on AMD gfx90a", §8.2: the down outputs stay
 * FP32 top-k partials and meet in a fixed reduction, without a round trip of
 * y through memory).  out is bit-identical to moe_mxfp4_down followed by
 * moe_combine on the same inputs: the same block dots and fixed fp32 order
 * per output, then the same slot-ordered fma chain (a slot of weight exactly
 * 0 adds nothing).
 *  hq, hs, wd, sd, offsets, sorted, cap: as moe_mxfp4_down.
 *  w    [T][k] fp32 routing weights (moe_route_topk's).
 *  out  [T][ld_out] fp32 output: the layer output.
 *  y    [T*k][ld_y] fp32: the per-slot down outputs as well, or NULL.
 * One launch when T <= 16 and a CTA's y rows fit its shared memory; otherwise
 * moe_mxfp4_down into y, then moe_combine (y is then required, else
 * MOE_ERR_UNSUPPORTED).  Other requirements and errors as moe_mxfp4_down. */
MOE_API moe_status moe_mxfp4_down_combine(const int8_t *hq, int64_t ld_hq, const float *hs, int64_t ld_hs,
                                  const uint8_t *wd, const uint8_t *sd,
                                  const int32_t *offsets, const int32_t *sorted, int64_t cap,
                                  const float *w, int T, int k, int E, int H, int I,
                                  float *out, int64_t ld_out, float *y, int64_t ld_y, void *stream);

/* ---------------------------------------------------------------- combine */

/* Routing-weighted combine in slot order (the gfx90a report, §8.2 "FP32 top-k
 * partial and fixed reduction"): out[t,n] = fma(w[t,k-1], y[t*k+k-1,n], ...
 * fma(w[t,1], y[t*k+1,n], w[t,0]*y[t*k,n])), fp32.  A slot of weight exactly
 * 0 adds nothing and its y row is not read (top-k gives that weight to a slot
 * with no expert, whose y row no projection writes).
 *  y [T*k][ld_y], w [T][k] fp32; out [T][ld_out] fp32 output. */
MOE_API moe_status moe_combine(const float *y, int64_t ld_y, const float *w, int T, int k, int H,
                       float *out, int64_t ld_out, void *stream);

/* ---------------------------------------------------------------- shared expert */

/* The join of the shared expert ("DeepSeek-V4-Flash on AMD gfx90a", Execution
 * structure and Fig. 1: a shared expert beside the routed experts, both
 * feeding a join that adds their partials): out[t,n] = out[t,n] + ys[t,n],
 * fp32, one rounding.  The shared expert itself is the stage calls above on
 * a one-expert weight set (E = 1, k = 1, offsets {0, T}, sorted 0..T-1):
 * the layer's Q8(x) rows -> moe_mxfp4_gateup_swiglu -> act_quant_q8 ->
 * moe_mxfp4_down -> ys; the pages give neither the shared expert's weight
 * format nor the join's arithmetic, and this is the plainest reading that
 * keeps the routed experts' arithmetic.
 *  ys  [T][ld_ys] fp32 (device, read); out [T][ld_out] fp32 (device, read and
 *      written; the routed output on entry).
 * Errors: MOE_ERR_INVALID_ARG for T < 0, H <= 0, null pointers or ld < H
 * (nothing is launched); T = 0 is a no-op. */
MOE_API moe_status moe_join_add(const float *ys, int64_t ld_ys, int T, int H, float *out, int64_t ld_out,
                                void *stream);

/* ---------------------------------------------------------------- fused decode */

/* Bytes of the workspace moe_decode_forward needs (a grid-barrier counter
 * and one readiness counter per active expert). */
MOE_API size_t moe_decode_workspace_bytes(void);

/* Largest T that moe_decode_forward accepts for this layer shape on the
 * current device (0: none; needs the CUDA device to be set). */
MOE_API int moe_decode_max_tokens(int H, int E, int k, int I);

/* The whole layer for a small decode batch in ONE launch: router + top-k +
 * sort + Q8(x) + gate/up + SwiGLU + Q8(h) + down + combine, with the same
 * arithmetic as the stage calls above, so every output is bit-identical to
 * running them in sequence (the Strix Halo record's exact-rows contract:
 * batching never changes a row's bits).  A cooperative launch of one CTA per
 * SM; each SM streams its share of every selected expert's weights through a
 * TMA ring, gate/up slices first, then down slices (prefetched into L2).
 *  x, w_router, bias, weights: as for the stage calls (x [T][ld_x]).
 *  out      [T][ld_out] fp32 output (the layer output).
 *  logits   [T][E], ids [T][k], weights [T][k]: outputs, as moe_route_topk.
 *  h        [T*k][ld_h] fp32: the SwiGLU activations (output; also the
 *           exchange buffer between the two projections; 16-byte aligned,
 *           ld_h a multiple of 4).
 *  y        [T*k][ld_y] fp32 per-slot down outputs, or NULL.
 *  workspace  >= moe_decode_workspace_bytes(), 8-byte aligned, zero-filled
 *           before its first use; each call leaves it ready for the next.
 *           Calls that share a workspace must not run concurrently.
 * Requires T <= moe_decode_max_tokens(H, E, k, I) (T*k <= 64, T <= 14, and the
 * activation rows must fit shared memory; else MOE_ERR_UNSUPPORTED: use the
 * stage calls), E <= 256, plus the stage calls' shape rules (H, I multiples
 * of 128, <= 4096).
 * A wait that does not complete (a device fault elsewhere) sets
 * MOE_DEV_WAIT_TIMEOUT and the launch returns with outputs incomplete; the
 * workspace must then be zero-filled again. */
MOE_API moe_status moe_decode_forward(const void *x, moe_dtype x_dtype, int64_t ld_x,
                                      const void *w_router, moe_dtype w_dtype, const float *bias,
                                      const uint8_t *wg, const uint8_t *sg, const uint8_t *wu, const uint8_t *su,
                                      const uint8_t *wd, const uint8_t *sd,
                                      int T, int H, int E, int k, int I,
                                      float *out, int64_t ld_out,
                                      float *logits, int32_t *ids, float *weights,
                                      float *h, int64_t ld_h, float *y, int64_t ld_y,
                                      void *workspace, size_t ws_bytes, void *stream);

/* Largest T that moe_decode_forward_shared accepts (its shared expert adds T
 * rows to the single launch's shared memory and needs T*k <= 63). */
MOE_API int moe_decode_max_tokens_shared(int H, int E, int k, int I);

/* moe_decode_forward for a layer with a shared expert ("DeepSeek-V4-Flash on
 * AMD gfx90a", Execution structure and Fig. 1), in the same single launch:
 * the shared expert's gate/up slice is requested at the start (it does not
 * depend on the routing) and computed while the router and top-k run; its
 * down slice follows the routed ones; the combine then adds its output,
 * out[t] = (routed combine)[t] + ys[t], fp32, so every output is bit-identical
 * to moe_decode_forward followed by the shared expert's stage calls and
 * moe_join_add.
 *  shared_wg .. shared_sd  the shared expert's weights: one expert in the
 *           routed experts' layout ([I][H/2], [I][H/32], [H][I/2], [H][I/32]);
 *           16-byte aligned nibbles, 4-byte aligned scale bytes.
 *  shared_h [T][ld_shared_h] fp32: its SwiGLU activations (output and
 *           exchange buffer; 16-byte aligned, ld a multiple of 4).
 *  shared_y [T][ld_shared_y] fp32: its down output, or NULL.
 * Other arguments, requirements and errors as moe_decode_forward, with
 * T <= moe_decode_max_tokens_shared(H, E, k, I). */
MOE_API moe_status moe_decode_forward_shared(const void *x, moe_dtype x_dtype, int64_t ld_x,
                                             const void *w_router, moe_dtype w_dtype, const float *bias,
                                             const uint8_t *wg, const uint8_t *sg, const uint8_t *wu,
                                             const uint8_t *su, const uint8_t *wd, const uint8_t *sd,
                                             const uint8_t *shared_wg, const uint8_t *shared_sg,
                                             const uint8_t *shared_wu, const uint8_t *shared_su,
                                             const uint8_t *shared_wd, const uint8_t *shared_sd,
                                             int T, int H, int E, int k, int I,
                                             float *out, int64_t ld_out,
                                             float *logits, int32_t *ids, float *weights,
                                             float *h, int64_t ld_h, float *y, int64_t ld_y,
                                             float *shared_h, int64_t ld_shared_h,
                                             float *shared_y, int64_t ld_shared_y,
                                             void *workspace, size_t ws_bytes, void *stream);

/* moe_decode_forward for callers that cannot allocate device memory when they
 * run the layer (serving loops that cannot afford the device-wide
 * synchronisation an allocation can cause, runtimes that own all device
 * memory, embedders that forbid allocation after start-up).  The papers have no counterpart to this call;
 * it exists for such callers only.
 * Same inputs, rules and output `out` as moe_decode_forward, computed by the
 * same kernel with the same bits.  Every intermediate (barrier counters,
 * logits, ids, weights, h) lives in one fixed array of device memory owned by
 * the library (about 1.1 MiB per device, held from library load until process
 * exit); nothing is allocated and the intermediates are not returned.
 * Limits of that array: T*k <= 64, T*E <= 32768, I <= 4096; beyond them the
 * call returns MOE_ERR_UNSUPPORTED (use moe_decode_forward with your own
 * buffers).
 * Every call looks up the array's device address on the current device (a
 * host-side query); the first call on a device also loads the library's
 * module there, so make that first call before any stream capture.  Each call
 * checks every argument first and, only then, clears the barrier words on
 * `stream` before its launch (a rejected call enqueues nothing).  All calls
 * on one device share the array: calls that may overlap on the GPU
 * (different streams without ordering between them) race and give wrong
 * results. */
MOE_API moe_status moe_decode_forward_noalloc(const void *x, moe_dtype x_dtype, int64_t ld_x,
                                              const void *w_router, moe_dtype w_dtype, const float *bias,
                                              const uint8_t *wg, const uint8_t *sg, const uint8_t *wu,
                                              const uint8_t *su, const uint8_t *wd, const uint8_t *sd,
                                              int T, int H, int E, int k, int I,
                                              float *out, int64_t ld_out, void *stream);

/* ---------------------------------------------------------------- measurement */

/* Throughput probe of the tensor-core instruction the prefill projections
 * run on (a measurement aid beside the layer; the pages have no counterpart:
 * it measures the roofline the tensor-core expert path is reported against).
 * One CTA per SM issues `iters` accumulating block-scaled FP4 MMAs (kind::mxf4
 * with E8M0 block scales, M = 128, N = n, K = 64) on zeroed shared-memory
 * operands, in the operand and scale layout of the tensor-core expert kernel.
 * *flops receives the launch's floating-point operations,
 * 2 * 128 * n * 64 * iters * (number of SMs); the caller times the launch
 * (events on `stream`).  n: 64, 128 or 256; 1 <= iters <= 2^20 (else
 * MOE_ERR_INVALID_ARG, nothing launched).  A wait that runs out raises
 * MOE_DEV_WAIT_TIMEOUT. */
MOE_API moe_status moe_mxf4_mma_probe(int n, int iters, double *flops, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_MXFP4_H */
