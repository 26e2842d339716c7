"""The per-expert tile policy of the expert projections (batches of more than
16 rows) against the oracle and against one-row calls.

"Optimizing DeepSeek V4 Flash Inference on a Strix Halo Pair", "MXFP4
routed-expert kernels": small batches take a direct route instead of
partially filled expert tiles; "DeepSeek-V4-Flash on AMD gfx90a", §7.1 item 8:
the expert sorter decides the tiles.  From 17 rows on, the stage calls split
the experts on the device by their row counts in `offsets`: an expert with at
most 4 rows is computed by the CUDA-core k-row kernel (its rows staged in
passes of a few rows when the batch's rows do not all fit shared memory), an
expert with more by the tensor-core kernel.

The batch here has one expert in every token (64 rows), one in every fourth
token (16 rows), one in every sixteenth (4 rows: the largest light expert)
and many with one or two rows.  Every output is checked against the oracle within
the layer's tolerance, and every row of a light expert must carry the bits of
the one-row call of its token.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import TOL, bits_equal, dev, ensure_built, host, max_err_over_rms, upload_layer

pytestmark = pytest.mark.gpu

T, K = 64, 6
HOT, WARM, EDGE = 7, 11, 12  # 64, 16 and 4 rows
LIGHT = 4  # largest light expert


@pytest.fixture(scope="module")
def moe():
    return ensure_built()


@pytest.fixture(scope="module")
def layer(moe):
    return upload_layer(synth.DSV4)


def _ids():
    """Top-k ids of the 64 tokens (distinct within a token)."""
    ids = np.empty((T, K), np.int32)
    spread = [e for e in range(synth.DSV4.E) if e not in (HOT, WARM, EDGE)]
    nxt = 0
    for t in range(T):
        row = [HOT]
        if t % 4 == 0:
            row.append(WARM)
        if t % 16 == 1:
            row.append(EDGE)
        while len(row) < K:  # each of the rest appears once or twice in the batch
            row.append(spread[nxt % len(spread)])
            nxt += 1
        ids[t] = row
    return ids


def _rows_per_expert(ids):
    return np.bincount(ids.ravel(), minlength=synth.DSV4.E)


def _stack(lw, names):
    return [getattr(lw, n) for n in names]


def test_batch_has_the_intended_row_counts():
    c = _rows_per_expert(_ids())
    assert c[HOT] == 64 and c[WARM] == 16 and c[EDGE] == LIGHT
    assert set(np.unique(c[c > 0])) <= {1, 2, LIGHT, 16, 64}


def test_gateup_tile_policy_vs_oracle_and_one_row_calls(moe, layer):
    spec = synth.DSV4
    ids = _ids()
    xq = synth.int8_codes(71, 7000, T, spec.H)
    xs = synth.positive_scales(71, 7001, T, spec.H // 32)
    offsets, srt, _ = oracle.sort(ids, spec.E, 1)
    wg, sg, wu, su = _stack(layer, ("wg", "sg", "wu", "su"))
    g = torch.empty(T * K, spec.I, device="cuda")
    u = torch.empty(T * K, spec.I, device="cuda")
    moe.moe_mxfp4_gateup(dev(xq), dev(xs), wg, sg, wu, su, dev(offsets), dev(srt), K, g, u)
    h = torch.empty(T * K, spec.I, device="cuda")
    moe.moe_mxfp4_gateup_swiglu(dev(xq), dev(xs), wg, sg, wu, su, dev(offsets), dev(srt), K, h)
    gg, uu, hh = host(g), host(u), host(h)
    assert moe.moe_device_status() == 0
    counts = _rows_per_expert(ids)
    # against the oracle: every heavy and light kind of expert, several tokens
    for t in (0, 1, 9, 33, 62, 63):
        for j in range(K):
            a, e = t * K + j, int(ids[t, j])
            ew = synth.expert(spec, e)
            go, uo = oracle.expert_gateup(xq[t], xs[t], ew.wg, ew.sg, ew.wu, ew.su)
            assert max_err_over_rms(gg[a], go) <= TOL, (t, j, e)
            assert max_err_over_rms(uu[a], uo) <= TOL, (t, j, e)
    # light experts (<= 4 rows): the bits of the one-row call of the token
    for t in (1, 2, 17, 40, 63):
        o1, s1, _ = oracle.sort(ids[t:t + 1], spec.E, 1)
        g1 = torch.empty(K, spec.I, device="cuda")
        u1 = torch.empty(K, spec.I, device="cuda")
        h1 = torch.empty(K, spec.I, device="cuda")
        moe.moe_mxfp4_gateup(dev(xq[t:t + 1]), dev(xs[t:t + 1]), wg, sg, wu, su, dev(o1), dev(s1), K, g1, u1)
        moe.moe_mxfp4_gateup_swiglu(dev(xq[t:t + 1]), dev(xs[t:t + 1]), wg, sg, wu, su, dev(o1), dev(s1), K, h1)
        g1, u1, h1 = host(g1), host(u1), host(h1)
        for j in range(K):
            a = t * K + j
            if counts[ids[t, j]] <= LIGHT:
                assert bits_equal(gg[a], g1[j]) and bits_equal(uu[a], u1[j]) and bits_equal(hh[a], h1[j]), (t, j)
            else:
                assert max_err_over_rms(gg[a], g1[j]) <= 2 * TOL
    assert moe.moe_device_status() == 0


def test_down_tile_policy_vs_oracle_and_one_row_calls(moe, layer):
    spec = synth.DSV4
    ids = _ids()
    A = T * K
    hq = synth.int8_codes(72, 7100, A, spec.I)
    hs = synth.positive_scales(72, 7101, A, spec.I // 32)
    offsets, srt, _ = oracle.sort(ids, spec.E, 1)
    y = torch.empty(A, spec.H, device="cuda")
    moe.moe_mxfp4_down(dev(hq), dev(hs), layer.wd, layer.sd, dev(offsets), dev(srt), T, K, y)
    yy = host(y)
    assert moe.moe_device_status() == 0
    counts = _rows_per_expert(ids)
    for t in (0, 1, 9, 62):
        for j in range(K):
            a, e = t * K + j, int(ids[t, j])
            ew = synth.expert(spec, e)
            assert max_err_over_rms(yy[a], oracle.expert_down(hq[a], hs[a], ew.wd, ew.sd)) <= TOL, (t, j, e)
    for t in (1, 2, 17, 40):
        o1, s1, _ = oracle.sort(ids[t:t + 1], spec.E, 1)
        y1 = torch.empty(K, spec.H, device="cuda")
        moe.moe_mxfp4_down(dev(hq[t * K:(t + 1) * K]), dev(hs[t * K:(t + 1) * K]), layer.wd, layer.sd, dev(o1),
                           dev(s1), 1, K, y1)
        y1 = host(y1)
        for j in range(K):
            if counts[ids[t, j]] <= LIGHT:
                assert bits_equal(yy[t * K + j], y1[j]), (t, j)
    assert moe.moe_device_status() == 0


def test_padded_segments_on_both_kernels(moe, layer):
    """Sorter tiles of 4 rows pad every segment with -1 (the light threshold
    counts the padded length): outputs of the real rows are unchanged."""
    spec = synth.DSV4
    ids = _ids()
    xq = synth.int8_codes(73, 7200, T, spec.H)
    xs = synth.positive_scales(73, 7201, T, spec.H // 32)
    wg, sg, wu, su = _stack(layer, ("wg", "sg", "wu", "su"))
    outs = []
    for tile in (1, 4):
        offsets, srt, _ = oracle.sort(ids, spec.E, tile)
        cap = moe.moe_sort_tokens_capacity(T, K, spec.E, tile)
        srt_full = np.concatenate([srt, np.full(cap - srt.size, -1, np.int32)])
        h = torch.full((T * K, spec.I), float("nan"), device="cuda")
        moe.moe_mxfp4_gateup_swiglu(dev(xq), dev(xs), wg, sg, wu, su, dev(offsets), dev(srt_full), K, h)
        outs.append(host(h))
    assert np.isfinite(outs[1]).all()
    assert max_err_over_rms(outs[1], outs[0]) <= 2 * TOL
    assert moe.moe_device_status() == 0
