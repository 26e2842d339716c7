"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test fixes one part of the oracle with something independent: the
pages' printed value set, closed forms, hand-worked special cases, library
routines (numpy stable sort, fp64 dense matmul, scipy's expit) or brute force
on small inputs.  They are chosen so that a plausible slip (a dropped block,
a flipped sign, the other nibble first, a transposed weight, a factor of two
in the scale, the wrong rounding) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

# OCP MX E2M1: sign, 2-bit exponent (bias 1), 1-bit mantissa; written out by hand.
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
              -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def _dequant_weights(w_packed, s_bytes):
    """Dense fp64 weights from packed nibbles and E8M0 bytes, via the hand table."""
    rows, half = w_packed.shape
    codes = np.empty((rows, 2 * half), dtype=np.int64)
    codes[:, 0::2] = w_packed & 0x0F
    codes[:, 1::2] = w_packed >> 4
    vals = np.array(E2M1_TABLE)[codes]
    scale = np.array([math.ldexp(1.0, int(u) - 127) for u in range(255)])[s_bytes.astype(np.int64)]
    return vals * np.repeat(scale, 32, axis=1)


def _dequant_q8(q, d):
    return q.astype(np.float64) * np.repeat(d.astype(np.float64), 32, axis=1)


# --------------------------------------------------------------- formats

def test_e2m1_matches_hand_table():
    for c in range(16):
        v = oracle.e2m1(c)
        assert v == E2M1_TABLE[c], c
        assert math.copysign(1.0, v) == math.copysign(1.0, E2M1_TABLE[c])


def test_e2m1_doubled_set_is_the_pages_set():
    with open(os.path.join(GOLDEN, "e2m1_doubled_values.txt")) as f:
        vals = [int(t) for line in f if not line.startswith("#") for t in line.split()]
    doubled = {int(round(2 * oracle.e2m1(c))) for c in range(16)}
    assert doubled == set(vals)


def test_e8m0_powers_of_two():
    for u in range(255):
        assert oracle.e8m0(u) == math.ldexp(1.0, u - 127)
    assert math.isnan(oracle.e8m0(255))


# --------------------------------------------------------------- block dot

def test_block_dot_nibble_order_special_cases():
    nib = np.zeros(16, np.uint8)
    nib[3] = 0x7 | (0xC << 4)         # element 6: code 7 (=6.0), element 7: code 12 (=-2.0)
    q = np.zeros(32, np.int8)
    q[6] = 5
    assert oracle.block_dot(q, nib) == 5 * 12    # 2 * 6.0
    q[:] = 0
    q[7] = 5
    assert oracle.block_dot(q, nib) == 5 * -4    # 2 * -2.0
    # -0 (code 8) contributes nothing
    nib[:] = 0x88
    q[:] = 127
    assert oracle.block_dot(q, nib) == 0


def test_block_dot_extremes():
    nib = np.full(16, 0x77, np.uint8)   # all +6.0
    q = np.full(32, 127, np.int8)
    assert oracle.block_dot(q, nib) == 32 * 127 * 12
    q[:] = -127
    assert oracle.block_dot(q, nib) == -32 * 127 * 12


def test_block_dot_bruteforce_random():
    rng_bytes = synth.random_bytes(7, 100, 16 * 200).reshape(200, 16)
    qs = synth.int8_codes(7, 101, 200, 32)
    tab = np.array(E2M1_TABLE)
    for nib, q in zip(rng_bytes, qs):
        codes = np.empty(32, np.int64)
        codes[0::2] = nib & 15
        codes[1::2] = nib >> 4
        ref = sum(int(qq) * int(round(2 * tab[c])) for qq, c in zip(q, codes))
        assert oracle.block_dot(q, nib) == ref


# --------------------------------------------------------------- Q8

def test_q8_zero_block():
    x = np.zeros((1, 64), np.float32)
    x[0, 40] = 3.0
    q, d = oracle.quant_q8(x)
    assert d[0, 0] == 0.0 and np.all(q[0, :32] == 0)
    assert d[0, 1] == np.float32(3.0) / np.float32(127.0)


def test_q8_amax_maps_to_127_and_ties_go_even():
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = 127.0      # amax 127 -> d = 1, 1/d = 1
    x[0, 1] = 2.5
    x[0, 2] = 3.5
    x[0, 3] = -2.5
    x[0, 4] = -127.0
    x[0, 5] = 0.5
    x[0, 6] = 1.5
    q, d = oracle.quant_q8(x)
    assert d[0, 0] == 1.0
    assert list(q[0, :7]) == [127, 2, 4, -2, -127, 0, 2]


def test_q8_reconstruction_bound_and_range():
    x = synth.normal(3, 200, 0, 64 * 512).astype(np.float32).reshape(64, 512)
    x *= np.repeat(synth.positive_scales(3, 201, 64, 16, 1e-3, 1e3), 32, axis=1)
    q, d = oracle.quant_q8(x)
    assert np.abs(q.astype(np.int32)).max() <= 127
    xb = x.reshape(64, 16, 32)
    amax = np.abs(xb).max(axis=2)
    assert np.array_equal(d, (amax / np.float32(127.0)).astype(np.float32))
    # the largest element of each block maps to +-127
    qb = q.reshape(64, 16, 32).astype(np.int32)
    idx = np.abs(xb).argmax(axis=2)
    assert np.all(np.abs(np.take_along_axis(qb, idx[..., None], 2)) == 127)
    err = np.abs(xb.astype(np.float64) - qb * d[..., None].astype(np.float64))
    assert np.all(err <= 0.5 * d[..., None] * (1 + 2.0 ** -20))


def test_q8_monotone():
    x = np.linspace(-5, 5, 32 * 8, dtype=np.float32).reshape(1, -1)
    x[0, ::32] = 5.0  # same amax in every block
    q, _ = oracle.quant_q8(x)
    for b in range(8):
        blk = q[0, 32 * b + 1: 32 * b + 32].astype(int)
        assert np.all(np.diff(blk) >= 0)


def test_q8_bf16_input_is_exact_widening():
    x = synth.normal(4, 202, 0, 4 * 256).astype(np.float32).reshape(4, 256)
    xb = synth.f32_to_bf16_bits(x)
    q1, d1 = oracle.quant_q8(xb)
    q2, d2 = oracle.quant_q8(synth.bf16_bits_to_f32(xb).reshape(4, 256))
    assert np.array_equal(q1, q2) and np.array_equal(d1, d2)


# --------------------------------------------------------------- projections

@pytest.mark.parametrize("H,I", [(256, 128), (512, 96)])
def test_gateup_equals_dense_dequantised_matvec(H, I):
    wg = synth.random_bytes(5, 300, I * H // 2).reshape(I, H // 2)
    wu = synth.random_bytes(5, 301, I * H // 2).reshape(I, H // 2)
    sg = synth.e8m0_bytes(5, 302, I * H // 32, -6, 2).reshape(I, H // 32)
    su = synth.e8m0_bytes(5, 303, I * H // 32, -6, 2).reshape(I, H // 32)
    xq = synth.int8_codes(5, 304, 1, H)[0]
    xs = synth.positive_scales(5, 305, 1, H // 32)[0]
    G, U = oracle.expert_gateup(xq, xs, wg, sg, wu, su)
    xd = _dequant_q8(xq[None], xs[None])[0]
    Wg, Wu = _dequant_weights(wg, sg), _dequant_weights(wu, su)
    for got, W in ((G, Wg), (U, Wu)):
        ref = W @ xd
        bound = 1e-13 * (np.abs(W) @ np.abs(xd))
        assert np.all(np.abs(got - ref) <= bound)


def test_down_equals_dense_dequantised_matvec():
    H, I = 192, 256
    wd = synth.random_bytes(6, 310, H * I // 2).reshape(H, I // 2)
    sd = synth.e8m0_bytes(6, 311, H * I // 32, -8, 3).reshape(H, I // 32)
    hq = synth.int8_codes(6, 312, 1, I)[0]
    hs = synth.positive_scales(6, 313, 1, I // 32)[0]
    y = oracle.expert_down(hq, hs, wd, sd)
    W = _dequant_weights(wd, sd)
    xd = _dequant_q8(hq[None], hs[None])[0]
    assert np.all(np.abs(y - W @ xd) <= 1e-13 * (np.abs(W) @ np.abs(xd)))


def test_silu():
    from scipy.special import expit
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(40.0) - 40.0) < 1e-12
    assert abs(oracle.silu(-40.0)) < 1e-15
    for g in np.linspace(-20, 20, 81):
        assert abs(oracle.silu(g) - g * expit(g)) <= 1e-15 * max(1.0, abs(g))


# --------------------------------------------------------------- router

def test_router_logits_within_fp32_bound_of_fp64():
    spec = synth.LayerSpec(H=512, E=16, k=4, I=64, x_dtype="bf16", wr_dtype="bf16", seed=11)
    x = synth.activations(spec, 5)
    wr = synth.router_weights(spec)
    got = oracle.router_logits(x, wr)
    xf = synth.bf16_bits_to_f32(x).reshape(5, -1).astype(np.float64)
    wf = synth.bf16_bits_to_f32(wr).reshape(16, -1).astype(np.float64)
    ref = xf @ wf.T
    bound = 512 * 2.0 ** -24 * (np.abs(xf) @ np.abs(wf).T)
    assert np.all(np.abs(got - ref) <= bound)


def test_router_logit_summation_order():
    # x.w = 1 at element 0 (partial sum 0) and 2^-24 at elements 8..15 (partial
    # sum 1).  The stated order sums 8 * 2^-24 = 2^-21 in partial 1 before
    # adding it to 1.0: 1 + 2^-21.  A plain left-to-right fp32 sum would give
    # exactly 1.0 (each 2^-24 is half an ulp of 1 and ties to even).
    H = 256
    x = np.zeros((1, H), np.float32)
    w = np.zeros((1, H), np.float32)
    x[0, 0], w[0, 0] = 1.0, 1.0
    x[0, 8:16], w[0, 8:16] = 2.0 ** -12, 2.0 ** -12
    got = oracle.router_logits(x, w)[0, 0]
    assert got == np.float32(1.0 + 2.0 ** -21)
    # chunks 0 and 32 share partial sum 0, so they are added in sequence there
    x[0, 8:16] = 0
    x[0, 256 - 8:] = 0
    x2 = np.zeros((1, 512), np.float32)
    w2 = np.zeros((1, 512), np.float32)
    x2[0, 0], w2[0, 0] = 1.0, 1.0
    x2[0, 256:264], w2[0, 256:264] = 2.0 ** -12, 2.0 ** -12    # chunk 32 -> partial 0
    assert oracle.router_logits(x2, w2)[0, 0] == np.float32(1.0)


def test_topk_matches_stable_argsort_and_weights():
    from scipy.special import expit
    spec = synth.DSV4
    logits = synth.normal(1, 400, 0, 20 * 256).astype(np.float32).reshape(20, 256)
    bias = synth.router_bias(synth.DSV4_ZIPF)
    for b in (None, bias):
        ids, w = oracle.topk(logits, 6, b)
        score = logits if b is None else (logits + b[None, :]).astype(np.float32)
        ref = np.argsort(-score, axis=1, kind="stable")[:, :6]
        assert np.array_equal(ids, ref)
        s = expit(np.take_along_axis(score, ids, 1).astype(np.float64))
        assert np.allclose(w, s / s.sum(1, keepdims=True), rtol=1e-14, atol=0)
        assert np.allclose(w.sum(1), 1.0, rtol=0, atol=1e-14)
    del spec


def test_topk_ties_go_to_lower_id():
    logits = np.zeros((2, 8), np.float32)
    logits[0, [2, 5, 6]] = 1.0
    logits[1, :] = 0.5
    ids, _ = oracle.topk(logits, 3)
    assert list(ids[0]) == [2, 5, 6]
    assert list(ids[1]) == [0, 1, 2]


NO_EXPERT = 0x7FFFFFFF


def test_topk_nan_scores_are_never_taken():
    """Brute force over rows with NaN scores sprinkled in (some rows keep
    fewer than k real scores, one has none): the k best real scores by
    (score desc, id asc), then slots with no expert (id 0x7fffffff, weight
    0); weights are expit of the taken scores over their sum.  Infinite
    scores are ordinary scores (+inf first, -inf last with weight 0)."""
    from scipy.special import expit
    T, E, k = 12, 16, 6
    logits = synth.normal(3, 410, 0, T * E).astype(np.float32).reshape(T, E)
    nan_mask = synth.uniform01(3, 411, 0, T * E).reshape(T, E) < 0.4
    logits[nan_mask] = np.nan
    logits[3, 12:] = np.nan          # row 3: only 12 real scores at most
    logits[4, :] = np.nan            # row 4: none
    logits[5, :E - 3] = np.nan       # row 5: 3 real scores < k
    logits[6, 2], logits[6, 7] = np.inf, -np.inf
    logits[7, :] = np.nan            # row 7: a real score and -inf, nothing else
    logits[7, 1], logits[7, 5] = -np.inf, 0.3
    ids, w = oracle.topk(logits, k)
    for t in range(T):
        real = [(-float(logits[t, e]), e) for e in range(E) if not np.isnan(logits[t, e])]
        take = [e for _, e in sorted(real)[:k]]
        ref_ids = take + [NO_EXPERT] * (k - len(take))
        assert list(ids[t]) == ref_ids, t
        sig = np.array([expit(float(logits[t, e])) for e in take] + [0.0] * (k - len(take)))
        total = sig.sum()
        if total > 0:
            assert np.allclose(w[t], sig / total, rtol=1e-14, atol=0), t
        else:
            assert np.isnan(w[t]).all(), t
    assert list(ids[4]) == [NO_EXPERT] * k
    assert ids[6, 0] == 2
    assert list(ids[7]) == [5, 1] + [NO_EXPERT] * (k - 2) and list(w[7]) == [1.0] + [0.0] * (k - 1)


def test_layer_slot_without_expert_contributes_nothing():
    """Every router row but expert 3's is NaN, so with k = 2 each token's
    second slot has no expert: its id is 0x7fffffff, its weight 0, its h and
    y rows 0, and the layer output equals the k = 1 layer's (expert 3 with
    weight 1) exactly."""
    spec = synth.TINY
    x = synth.activations(spec, 3)
    wr = synth.router_weights(spec).copy()
    wr[[e for e in range(spec.E) if e != 3]] = np.nan
    experts = {3: synth.expert(spec, 3)}
    r2 = oracle.layer(x, wr, None, 2, experts)
    r1 = oracle.layer(x, wr, None, 1, experts)
    assert (r2["ids"][:, 0] == 3).all() and (r2["ids"][:, 1] == NO_EXPERT).all()
    assert (r2["w"][:, 0] == 1.0).all() and (r2["w"][:, 1] == 0.0).all()
    assert not r2["h"][1::2].any() and not r2["y"][1::2].any()
    assert np.array_equal(r2["out"], r1["out"])
    assert np.isfinite(r2["out"]).all()


# --------------------------------------------------------------- sorter

@pytest.mark.parametrize("T,k,E", [(1, 6, 256), (16, 6, 256), (37, 2, 8), (64, 6, 256)])
def test_sort_matches_numpy_stable_argsort(T, k, E):
    ids = (synth.raw_u64(2, 500 + T, 0, T * k) % np.uint64(E)).astype(np.int32).reshape(T, k)
    offsets, srt, inv = oracle.sort(ids, E, 1)
    flat = ids.ravel()
    assert np.array_equal(srt, np.argsort(flat, kind="stable"))
    assert np.array_equal(np.diff(offsets), np.bincount(flat, minlength=E))
    assert np.array_equal(srt[inv], np.arange(T * k))


def test_sort_padding():
    ids = np.array([[3, 1], [3, 0], [1, 3]], np.int32)
    offsets, srt, inv = oracle.sort(ids, 4, 4)
    assert list(offsets) == [0, 4, 8, 8, 12]
    assert list(srt) == [3, -1, -1, -1, 1, 4, -1, -1, 0, 2, 5, -1]
    assert np.array_equal(srt[inv], np.arange(6))


def test_combine_matches_weighted_sum():
    y = synth.normal(8, 700, 0, 12 * 64).reshape(12, 64)
    w = synth.uniform01(8, 701, 0, 4 * 3).reshape(4, 3)
    out = oracle.combine(y, w)
    ref = np.einsum("tj,tjn->tn", w, y.reshape(4, 3, 64))
    assert np.allclose(out, ref, rtol=1e-14, atol=1e-14)
    # slot j of token t is row t*k + j
    w1 = np.zeros((4, 3))
    w1[2, 1] = 1.0
    assert np.array_equal(oracle.combine(y, w1)[2], y[2 * 3 + 1])


# --------------------------------------------------------------- layer

def _textbook_layer(x_f32, wr_f32, bias, k, experts, E):
    """Dense fp64 statement of the layer (dequantise, matmul, silu, combine),
    reusing only the separately pinned Q8 step."""
    from scipy.special import expit
    T, H = x_f32.shape
    logits = x_f32.astype(np.float64) @ wr_f32.astype(np.float64).T
    score = logits + (0 if bias is None else bias[None, :])
    ids = np.argsort(-score, axis=1, kind="stable")[:, :k]
    sel = np.take_along_axis(score, ids, 1)
    w = expit(sel) / expit(sel).sum(1, keepdims=True)
    xq, xs = oracle.quant_q8(x_f32)
    xd = _dequant_q8(xq, xs)
    out = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            ew = experts[ids[t, j]]
            G = _dequant_weights(ew.wg, ew.sg) @ xd[t]
            U = _dequant_weights(ew.wu, ew.su) @ xd[t]
            h = G * expit(G) * U
            hq, hs = oracle.quant_q8(h.astype(np.float32)[None])
            y = _dequant_weights(ew.wd, ew.sd) @ _dequant_q8(hq, hs)[0]
            out[t] += w[t, j] * y
    return ids, out


def test_layer_matches_textbook_dense_layer():
    spec = synth.TINY
    x = synth.activations(spec, 3)
    wr = synth.router_weights(spec)
    experts = {e: synth.expert(spec, e) for e in range(spec.E)}
    r = oracle.layer(x, wr, None, spec.k, experts)
    ids, out = _textbook_layer(x, wr, None, spec.k, experts, spec.E)
    assert np.array_equal(r["ids"], ids)
    # the oracle takes the sigmoid of the fp32 logit (its reading of the
    # router), the textbook the fp64 one: routing weights differ by ~1e-8
    rms = np.sqrt(np.mean(out ** 2))
    assert np.max(np.abs(r["out"] - out)) <= 1e-6 * rms


def test_layer_single_expert_all_ones():
    # E = k = 1, every weight code 2 (= 1.0), E8M0 127 (= 1): each gate/up
    # output is the sum of the dequantised activations; w = 1.
    H, I = 256, 64
    ew = synth.ExpertWeights(
        wg=np.full((I, H // 2), 0x22, np.uint8), sg=np.full((I, H // 32), 127, np.uint8),
        wu=np.full((I, H // 2), 0x22, np.uint8), su=np.full((I, H // 32), 127, np.uint8),
        wd=np.full((H, I // 2), 0x22, np.uint8), sd=np.full((H, I // 32), 127, np.uint8))
    x = synth.normal(9, 600, 0, 2 * H).astype(np.float32).reshape(2, H)
    wr = np.ones((1, H), np.float32)
    r = oracle.layer(x, wr, None, 1, {0: ew})
    assert np.all(r["w"] == 1.0)
    for t in range(2):
        q, d = oracle.quant_q8(x[t:t + 1])
        g = float(np.sum(_dequant_q8(q, d)))
        h = g * g / (1.0 + math.exp(-g))
        hq, hs = oracle.quant_q8(np.full((1, I), h, np.float32))
        y = float(np.sum(_dequant_q8(hq, hs)))
        assert np.allclose(r["out"][t], y, rtol=1e-12, atol=0)


def test_layer_zero_weights_give_zero():
    spec = synth.TINY
    x = synth.activations(spec, 2)
    wr = synth.router_weights(spec)
    z = synth.ExpertWeights(
        wg=np.zeros((spec.I, spec.H // 2), np.uint8), sg=np.full((spec.I, spec.H // 32), 127, np.uint8),
        wu=np.zeros((spec.I, spec.H // 2), np.uint8), su=np.full((spec.I, spec.H // 32), 127, np.uint8),
        wd=np.zeros((spec.H, spec.I // 2), np.uint8), sd=np.full((spec.H, spec.I // 32), 127, np.uint8))
    r = oracle.layer(x, wr, None, spec.k, {e: z for e in range(spec.E)})
    assert np.all(r["out"] == 0.0)


def test_layer_token_permutation_is_exact():
    spec = synth.TINY
    x = synth.activations(spec, 5)
    wr = synth.router_weights(spec)
    experts = {e: synth.expert(spec, e) for e in range(spec.E)}
    r = oracle.layer(x, wr, None, spec.k, experts)
    perm = np.array([3, 0, 4, 1, 2])
    rp = oracle.layer(x[perm], wr, None, spec.k, experts)
    assert np.array_equal(rp["out"], r["out"][perm])
    assert np.array_equal(rp["ids"], r["ids"][perm])
    aperm = (perm[:, None] * spec.k + np.arange(spec.k)[None]).ravel()
    assert np.array_equal(rp["hq"], r["hq"][aperm])


# --------------------------------------------------------------- shared expert

def test_shared_expert_matches_textbook_dense_expert():
    # the shared expert written out with dense fp64 matrices: G, U = W x,
    # h = silu(G) U, y = Wd Q8(h), joined onto the routed output
    from scipy.special import expit
    spec = synth.TINY
    x = synth.activations(spec, 3)
    wr = synth.router_weights(spec)
    experts = {e: synth.expert(spec, e) for e in range(spec.E)}
    sh = synth.shared_expert(spec)
    r = oracle.layer(x, wr, None, spec.k, experts, shared=sh)
    xd = _dequant_q8(*oracle.quant_q8(x))
    ys = np.empty((3, spec.H))
    for t in range(3):
        G = _dequant_weights(sh.wg, sh.sg) @ xd[t]
        U = _dequant_weights(sh.wu, sh.su) @ xd[t]
        h = G * expit(G) * U
        hq, hs = oracle.quant_q8(h.astype(np.float32)[None])
        ys[t] = _dequant_weights(sh.wd, sh.sd) @ _dequant_q8(hq, hs)[0]
    rms = np.sqrt(np.mean(ys ** 2))
    assert np.max(np.abs(r["ys"] - ys)) <= 1e-6 * rms
    assert np.array_equal(r["out"], r["out_routed"] + r["ys"])
    assert not np.array_equal(r["out"], r["out_routed"])


def test_shared_expert_is_a_one_expert_routed_layer():
    # a routed layer with one expert and k = 1 gives that expert weight
    # sigmoid(l) / sigmoid(l) = 1, so its output is the shared expert's
    spec = synth.TINY
    x = synth.activations(spec, 4)
    sh = synth.shared_expert(spec)
    r1 = oracle.layer(x, np.ones((1, spec.H), np.float32), None, 1, {0: sh})
    assert np.all(r1["w"] == 1.0)
    s = oracle.shared_expert(r1["xq"], r1["xs"], sh)
    assert np.array_equal(s["ys"], r1["out"])
    assert np.array_equal(s["hq"], r1["hq"]) and np.array_equal(s["hs"], r1["hs"])


def test_shared_expert_zero_down_weights_leave_the_routed_output():
    spec = synth.TINY
    x = synth.activations(spec, 2)
    wr = synth.router_weights(spec)
    experts = {e: synth.expert(spec, e) for e in range(spec.E)}
    sh = synth.shared_expert(spec)
    sh.wd[...] = 0
    r = oracle.layer(x, wr, None, spec.k, experts, shared=sh)
    assert np.all(r["ys"] == 0.0)
    assert np.array_equal(r["out"], r["out_routed"])


def test_shared_expert_down_sign_flip_negates_exactly():
    # flipping the sign bit of every down nibble negates every block dot
    spec = synth.TINY
    x = synth.activations(spec, 2)
    xq, xs = oracle.quant_q8(x)
    sh = synth.shared_expert(spec)
    a = oracle.shared_expert(xq, xs, sh)
    sh.wd ^= 0x88
    b = oracle.shared_expert(xq, xs, sh)
    assert np.array_equal(b["ys"], -a["ys"])
    assert np.array_equal(b["hq"], a["hq"])
