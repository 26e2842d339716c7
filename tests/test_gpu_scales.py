"""E8M0 scale bytes over their whole range, through both expert paths, against
the oracle.

The E8M0 byte u of a block scales its exact integer dot by 2^(u-128) (the
E8M0 factor 2^(u-127), halved because the dots count twice the E2M1 values);
byte 255 is NaN ("DeepSeek-V4-Flash on AMD gfx90a", §6.1 "E8M0 scaling";
OCP MX).  The CUDA-core kernels (1-16 rows) form each block term as
I_b * (xs_b * 2^(u-128)); the tensor path (experts with many rows) gives the
MMA the byte clamped to [64, 192] and applies the remaining power of two to
the activation scale.  Both must match the oracle's fp64 value for bytes
0, 1, 2 (subnormal factors), 126-128, 240-254 (factors up to 2^126) and 255
(NaN), mixed within rows.

Every case keeps the scale products xs_b * 2^(u-128) and the outputs finite
normal fp32 numbers, the range in which the layer's arithmetic is exact up to
fp32 rounding: per 32-block column b the activation scale is chosen for the
class of bytes that column holds, so that every class contributes visibly to
every output.  Outputs a byte 255 reaches must be NaN on both sides; every
other output must be within the layer's tolerance of the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import TOL, dev, ensure_built, host

pytestmark = pytest.mark.gpu

LOW, MID, HIGH = (0, 1, 2), (126, 127, 128), (240, 250, 253, 254)
CLASSES = (LOW, MID, HIGH)
# activation scale per class: xs * 2^(u - 128) lands near 2^-20 .. 2^-14
# (the high class needs a subnormal fp32 activation scale for that)
XS_EXP = {0: 107, 1: -19, 2: -140}


@pytest.fixture(scope="module")
def moe():
    return ensure_built()


def _scale_bytes(seed, stream, rows, nb, nan_rows):
    """E8M0 bytes [rows, nb]: block column b holds bytes of class b % 3, drawn
    at random from it; rows in nan_rows get byte 255 in block 1."""
    r = synth.raw_u64(seed, stream, 0, rows * nb).reshape(rows, nb)
    out = np.empty((rows, nb), np.uint8)
    for b in range(nb):
        cls = CLASSES[b % 3]
        out[:, b] = np.array(cls, np.uint8)[(r[:, b] % np.uint64(len(cls))).astype(np.int64)]
    out[list(nan_rows), 1] = 255
    return out


def _act_scales(seed, stream, rows, nb):
    """Activation scales [rows, nb] for the block classes: 2^XS_EXP[class]
    times a factor in [1, 2)."""
    f = 1.0 + synth.uniform01(seed, stream, 0, rows * nb).reshape(rows, nb)
    e = np.array([XS_EXP[b % 3] for b in range(nb)], np.float64)[None, :]
    return (f * np.exp2(e)).astype(np.float32)


def _experts(spec, seed):
    ex = {}
    for e in range(spec.E):
        w = synth.expert(spec, e)
        nan_g = {i for i in range(spec.I) if i % 37 == 5}
        nan_d = {n for n in range(spec.H) if n % 41 == 7}
        w.sg[...] = _scale_bytes(seed, 100 + 8 * e, spec.I, spec.H // 32, nan_g)
        w.su[...] = _scale_bytes(seed, 101 + 8 * e, spec.I, spec.H // 32, set())
        w.sd[...] = _scale_bytes(seed, 102 + 8 * e, spec.H, spec.I // 32, nan_d)
        ex[e] = w
    return ex


def _ids(T, k, E, seed):
    """Expert 0 takes every token (many rows: the tensor path when T is
    large); the other k-1 slots are spread over the rest."""
    ids = np.empty((T, k), np.int32)
    for t in range(T):
        r = synth.raw_u64(seed, 5000 + t, 0, E)
        rest = [e for e in np.argsort(r, kind="stable").tolist() if e != 0]
        ids[t] = np.array([0] + rest[: k - 1], np.int32)
    return ids


def _stack(ex, E, name):
    return torch.from_numpy(np.stack([getattr(ex[e], name) for e in range(E)])).cuda()


def _check(got, ref):
    """NaN exactly where the oracle has NaN; elsewhere max|err| <= TOL * RMS."""
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.isfinite(got[fin]).all()
    rms = float(np.sqrt(np.mean(ref[fin] ** 2)))
    err = float(np.max(np.abs(got[fin] - ref[fin]))) / rms
    assert err <= TOL, err


@pytest.mark.parametrize("T", [5, 150])
def test_gateup_scale_bytes_whole_range(moe, T):
    H, I, E, k = 512, 256, 3, 2
    spec = synth.LayerSpec(H=H, E=E, k=k, I=I, seed=61)
    ex = _experts(spec, 61)
    xq = synth.int8_codes(61, 6000, T, H)
    xs = _act_scales(61, 6001, T, H // 32)
    ids = _ids(T, k, E, 61)
    offsets, srt, _ = oracle.sort(ids, E, 1)
    W = {n: _stack(ex, E, n) for n in ("wg", "sg", "wu", "su")}
    g = torch.empty(T * k, I, device="cuda")
    u = torch.empty(T * k, I, device="cuda")
    moe.moe_mxfp4_gateup(dev(xq), dev(xs), W["wg"], W["sg"], W["wu"], W["su"], dev(offsets), dev(srt), k, g, u)
    h = torch.empty(T * k, I, device="cuda")
    moe.moe_mxfp4_gateup_swiglu(dev(xq), dev(xs), W["wg"], W["sg"], W["wu"], W["su"], dev(offsets), dev(srt), k, h)
    go, uo, ho = (np.empty((T * k, I)) for _ in range(3))
    for a in range(T * k):
        e = ex[ids.ravel()[a]]
        go[a], uo[a] = oracle.expert_gateup(xq[a // k], xs[a // k], e.wg, e.sg, e.wu, e.su)
        with np.errstate(invalid="ignore", over="ignore"):
            ho[a] = np.array([oracle.silu(v) for v in go[a]]) * uo[a]
    assert np.isnan(go).any() and not np.isnan(uo).any()
    _check(host(g), go)
    _check(host(u), uo)
    _check(host(h), ho)
    assert moe.moe_device_status() == 0


@pytest.mark.parametrize("T", [5, 150])
def test_down_scale_bytes_whole_range(moe, T):
    H, I, E, k = 512, 256, 3, 2
    spec = synth.LayerSpec(H=H, E=E, k=k, I=I, seed=62)
    ex = _experts(spec, 62)
    A = T * k
    hq = synth.int8_codes(62, 6100, A, I)
    hs = _act_scales(62, 6101, A, I // 32)
    ids = _ids(T, k, E, 62)
    offsets, srt, _ = oracle.sort(ids, E, 1)
    y = torch.empty(A, H, device="cuda")
    moe.moe_mxfp4_down(dev(hq), dev(hs), _stack(ex, E, "wd"), _stack(ex, E, "sd"), dev(offsets), dev(srt), T, k, y)
    yo = np.empty((A, H))
    for a in range(A):
        e = ex[ids.ravel()[a]]
        yo[a] = oracle.expert_down(hq[a], hs[a], e.wd, e.sd)
    assert np.isnan(yo).any()
    _check(host(y), yo)
    assert moe.moe_device_status() == 0


def test_both_paths_agree_on_extreme_bytes(moe):
    """The 5 rows of the 1-16-row call are the first 5 rows of the 150-row
    call (expert 0 holds every token): the tensor path's rows of expert 0
    agree with the CUDA-core path's within the tolerance, NaN for NaN."""
    H, I, E, k = 512, 256, 3, 2
    spec = synth.LayerSpec(H=H, E=E, k=k, I=I, seed=63)
    ex = _experts(spec, 63)
    xq = synth.int8_codes(63, 6200, 150, H)
    xs = _act_scales(63, 6201, 150, H // 32)
    W = {n: _stack(ex, E, n) for n in ("wg", "sg", "wu", "su")}
    ids = _ids(150, k, E, 63)
    outs = {}
    for T in (5, 150):
        offsets, srt, _ = oracle.sort(ids[:T], E, 1)
        g = torch.empty(T * k, I, device="cuda")
        u = torch.empty(T * k, I, device="cuda")
        moe.moe_mxfp4_gateup(dev(xq[:T]), dev(xs[:T]), W["wg"], W["sg"], W["wu"], W["su"], dev(offsets), dev(srt),
                             k, g, u)
        outs[T] = (host(g), host(u))
    rows = np.arange(0, 5 * k, k)  # slot 0 of each token: expert 0
    for i in range(2):
        _check(outs[150][i][rows], outs[5][i][rows].astype(np.float64))
    assert moe.moe_device_status() == 0
