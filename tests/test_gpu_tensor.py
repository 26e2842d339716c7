"""The tensor-core (tcgen05) expert projections, taken by the stage calls for
batches of more than 16 rows, against the oracle.

The tensor path gives the MMA the E2M1 weights with their E8M0 byte as the
block scale, and each activation value q * xs as six E2M1 planes with E8M0
block scales of their own (a greedy expansion, about two bits per plane);
the accumulator takes the whole reduction in fp32.  With unit scales (xs =
1, E8M0 bytes 128) the planes hold every Q8 code exactly and every output is
a sum of integer block dots, so those cases are compared bit for bit with
the oracle; with the layer's scales the bar is the layer's tolerance,
max|err| <= 1e-3 * RMS.  Cases span several 128-row weight tiles, experts
with more than 16 rows (several token tiles), experts with a handful of
rows, padded segments, and reduction lengths from 256 to 4096 (the tensor
path needs a multiple of 256; other shapes keep the CUDA-core path).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import TOL, dev, ensure_built, host, max_err_over_rms

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    return ensure_built()


def _skewed_rows(T, k, E, seed, hot):
    """Top-k ids per token: expert `hot` in every row, the rest spread."""
    ids = np.empty((T, k), np.int32)
    for t in range(T):
        r = synth.raw_u64(seed, 3000 + t, 0, E)
        order = [e for e in np.argsort(r, kind="stable").tolist() if e != hot]
        ids[t] = np.array([hot] + order[: k - 1], np.int32)
    return ids


def _stack(experts, E, name):
    return torch.from_numpy(np.stack([getattr(experts[e], name) for e in range(E)])).cuda()


@pytest.mark.parametrize("H,I,E,k,T,tile", [(4096, 256, 5, 2, 300, 1), (512, 384, 7, 3, 41, 4),
                                            (1024, 128, 3, 2, 17, 1)])
def test_tensor_gateup_swiglu(moe, H, I, E, k, T, tile):
    spec = synth.LayerSpec(H=H, E=E, k=k, I=I, seed=31)
    ex = {e: synth.expert(spec, e) for e in range(E)}
    xs = synth.positive_scales(31, 2101, T, H // 32)
    xq = synth.int8_codes(31, 2100, T, H)
    ids = _skewed_rows(T, k, E, 31, hot=E - 1)  # one expert takes every row: > 128 when T > 128
    offsets, srt, _ = oracle.sort(ids, E, tile)
    cap = moe.moe_sort_tokens_capacity(T, k, E, tile)
    srt_full = np.concatenate([srt, np.full(cap - srt.size, -1, np.int32)])
    W = {n: _stack(ex, E, n) for n in ("wg", "sg", "wu", "su")}
    h = torch.full((T * k, I + 8), float("nan"), device="cuda")[:, :I]
    moe.moe_mxfp4_gateup_swiglu(dev(xq, 16), dev(xs), W["wg"], W["sg"], W["wu"], W["su"], dev(offsets),
                                dev(srt_full), k, h)
    ho = np.empty((T * k, I))
    for a in range(T * k):
        e = ex[ids.ravel()[a]]
        g, u = oracle.expert_gateup(xq[a // k], xs[a // k], e.wg, e.sg, e.wu, e.su)
        ho[a] = np.vectorize(oracle.silu)(g) * u
    hg = host(h)
    assert np.isfinite(hg).all()
    assert max_err_over_rms(hg, ho) <= TOL
    assert moe.moe_device_status() == 0


@pytest.mark.parametrize("H,I,E,k,T,tile", [(4096, 2048, 3, 2, 150, 4), (384, 1024, 6, 3, 20, 1)])
def test_tensor_down(moe, H, I, E, k, T, tile):
    spec = synth.LayerSpec(H=H, E=E, k=k, I=I, seed=32)
    ex = {e: synth.expert(spec, e) for e in range(E)}
    A = T * k
    hs = synth.positive_scales(32, 2201, A, I // 32)
    hq = synth.int8_codes(32, 2200, A, I)
    ids = _skewed_rows(T, k, E, 32, hot=0)
    offsets, srt, _ = oracle.sort(ids, E, tile)
    cap = moe.moe_sort_tokens_capacity(T, k, E, tile)
    srt_full = np.concatenate([srt, np.full(cap - srt.size, -1, np.int32)])
    y = torch.full((A, H + 4), float("nan"), device="cuda")[:, :H]
    moe.moe_mxfp4_down(dev(hq, 32), dev(hs), _stack(ex, E, "wd"), _stack(ex, E, "sd"), dev(offsets),
                       dev(srt_full), T, k, y)
    yo = np.empty((A, H))
    for a in range(A):
        e = ex[ids.ravel()[a]]
        yo[a] = oracle.expert_down(hq[a], hs[a], e.wd, e.sd)
    yg = host(y)
    assert np.isfinite(yg).all()
    assert max_err_over_rms(yg, yo) <= TOL
    assert moe.moe_device_status() == 0


def test_tensor_path_large_activations(moe):
    """Activation scales far from 1 (|x| ~ 1.3e5) are applied in fp32 after
    the exact block dots, so the result is still the oracle's."""
    spec = synth.LayerSpec(H=512, E=2, k=1, I=128, seed=33)
    ex = {e: synth.expert(spec, e) for e in range(2)}
    T = 20
    xq = synth.int8_codes(33, 2300, T, 512)
    xs = synth.positive_scales(33, 2301, T, 16, lo=200.0, hi=1000.0)
    ids = np.zeros((T, 1), np.int32)
    offsets, srt, _ = oracle.sort(ids, 2, 1)
    W = {n: _stack(ex, 2, n) for n in ("wg", "sg", "wu", "su")}
    h = torch.empty(T, 128, device="cuda")
    moe.moe_mxfp4_gateup_swiglu(dev(xq), dev(xs), W["wg"], W["sg"], W["wu"], W["su"], dev(offsets), dev(srt), 1, h)
    ho = np.empty((T, 128))
    for t in range(T):
        g, u = oracle.expert_gateup(xq[t], xs[t], ex[0].wg, ex[0].sg, ex[0].wu, ex[0].su)
        ho[t] = np.vectorize(oracle.silu)(g) * u
    hg = host(h)
    assert np.isfinite(hg).all()
    assert max_err_over_rms(hg, ho) <= TOL
    assert moe.moe_device_status() == 0


def test_sixteen_rows_keep_the_exact_path(moe):
    """16 rows take the CUDA-core path, 17 rows of the same data the tensor
    path: on the 16 shared rows the two agree within the tolerance."""
    H, I, E, k = 512, 256, 3, 2
    spec = synth.LayerSpec(H=H, E=E, k=k, I=I, seed=34)
    ex = {e: synth.expert(spec, e) for e in range(E)}
    xq = synth.int8_codes(34, 2400, 17, H)
    xs = synth.positive_scales(34, 2401, 17, H // 32)
    ids = _skewed_rows(17, k, E, 34, hot=1)
    W = {n: _stack(ex, E, n) for n in ("wg", "sg", "wu", "su")}
    outs = {}
    for T in (16, 17):
        offsets, srt, _ = oracle.sort(ids[:T], E, 1)
        h = torch.empty(T * k, I, device="cuda")
        moe.moe_mxfp4_gateup_swiglu(dev(xq[:T]), dev(xs[:T]), W["wg"], W["sg"], W["wu"], W["su"], dev(offsets),
                                    dev(srt), k, h)
        outs[T] = host(h)
    assert max_err_over_rms(outs[17][: 16 * k], outs[16]) <= 2 * TOL
    assert moe.moe_device_status() == 0


def _unit_scale_expert(spec, e):
    """An expert of the spec with every E8M0 byte 128: each block term of the
    projections is then the integer block dot itself."""
    ex = synth.expert(spec, e)
    for n in ("sg", "su", "sd"):
        getattr(ex, n)[...] = 128
    return ex


@pytest.mark.parametrize("H,I,E,k,T", [(4096, 256, 3, 2, 70), (256, 128, 4, 3, 33)])
def test_tensor_block_dots_exact(moe, H, I, E, k, T):
    """Unit scales: gate/up (moe_mxfp4_gateup) and down outputs are sums of
    exact integer block dots, equal to the oracle's bit for bit."""
    spec = synth.LayerSpec(H=H, E=E, k=k, I=I, seed=35)
    ex = {e: _unit_scale_expert(spec, e) for e in range(E)}
    A = T * k
    xq = synth.int8_codes(35, 2500, T, H)
    xs = np.ones((T, H // 32), np.float32)
    ids = _skewed_rows(T, k, E, 35, hot=1)
    offsets, srt, _ = oracle.sort(ids, E, 1)
    W = {n: _stack(ex, E, n) for n in ("wg", "sg", "wu", "su", "wd", "sd")}
    g = torch.empty(A, I, device="cuda")
    u = torch.empty(A, I, device="cuda")
    moe.moe_mxfp4_gateup(dev(xq), dev(xs), W["wg"], W["sg"], W["wu"], W["su"], dev(offsets), dev(srt), k, g, u)
    hq = synth.int8_codes(35, 2501, A, I)
    hs = np.ones((A, I // 32), np.float32)
    y = torch.empty(A, H, device="cuda")
    moe.moe_mxfp4_down(dev(hq), dev(hs), W["wd"], W["sd"], dev(offsets), dev(srt), T, k, y)
    gg, uu, yy = host(g), host(u), host(y)
    for a in range(A):
        e = ex[ids.ravel()[a]]
        go, uo = oracle.expert_gateup(xq[a // k], xs[a // k], e.wg, e.sg, e.wu, e.su)
        assert np.array_equal(gg[a], go.astype(np.float32)), a
        assert np.array_equal(uu[a], uo.astype(np.float32)), a
        yo = oracle.expert_down(hq[a], hs[a], e.wd, e.sd)
        assert np.array_equal(yy[a], yo.astype(np.float32)), a
    assert moe.moe_device_status() == 0
