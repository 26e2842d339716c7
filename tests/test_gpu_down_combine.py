"""The fused down projection + combine (moe_mxfp4_down_combine) against the
two stage calls it replaces, and against the oracle.

"DeepSeek-V4-Flash on AMD gfx90a", §8.2 (down consumer): the down outputs
stay fp32 top-k partials and meet in a fixed reduction.  The fused call must
give the bits of moe_mxfp4_down followed by moe_combine: the same block dots
and fp32 order per output, then the same slot-ordered fma chain, for every
batch size it runs in one launch (1-16 rows) and in the two-launch fallback
beyond.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import TOL, bits_equal, dev, ensure_built, host, max_err_over_rms

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    return ensure_built()


SPEC = synth.LayerSpec(H=1024, E=16, k=4, I=512, seed=81)


@pytest.fixture(scope="module")
def weights(moe):
    ex = {e: synth.expert(SPEC, e) for e in range(SPEC.E)}
    wd = torch.from_numpy(np.stack([ex[e].wd for e in range(SPEC.E)])).cuda()
    sd = torch.from_numpy(np.stack([ex[e].sd for e in range(SPEC.E)])).cuda()
    return ex, wd, sd


def _inputs(T, seed):
    k, E, I = SPEC.k, SPEC.E, SPEC.I
    ids = np.empty((T, k), np.int32)
    for t in range(T):
        r = synth.raw_u64(seed, 8000 + t, 0, E)
        ids[t] = np.argsort(r, kind="stable")[:k]
    hq = synth.int8_codes(seed, 8100, T * k, I)
    hs = synth.positive_scales(seed, 8101, T * k, I // 32)
    w = synth.uniform01(seed, 8102, 0, T * k).reshape(T, k).astype(np.float32)
    w /= w.sum(axis=1, keepdims=True)
    return ids, hq, hs, w


def _two_calls(moe, wd, sd, offsets, srt, hq_d, hs_d, w_d, T):
    y = torch.empty(T * SPEC.k, SPEC.H, device="cuda")
    out = torch.empty(T, SPEC.H, device="cuda")
    moe.moe_mxfp4_down(hq_d, hs_d, wd, sd, offsets, srt, T, SPEC.k, y)
    moe.moe_combine(y, w_d, out)
    return host(y), host(out)


@pytest.mark.parametrize("T,pad", [(1, 0), (3, 16), (8, 0), (16, 32), (20, 0)])
def test_fused_equals_down_then_combine(moe, weights, T, pad):
    ex, wd, sd = weights
    ids, hq, hs, w = _inputs(T, 82 + T)
    offsets, srt, _ = oracle.sort(ids, SPEC.E, 1)
    o_d, s_d = dev(offsets), dev(srt)
    hq_d, hs_d, w_d = dev(hq, 16), dev(hs), dev(w)
    y_ref, out_ref = _two_calls(moe, wd, sd, o_d, s_d, hq_d, hs_d, w_d, T)
    out = torch.full((T, SPEC.H + pad), float("nan"), device="cuda")[:, :SPEC.H]
    y = torch.full((T * SPEC.k, SPEC.H + pad), float("nan"), device="cuda")[:, :SPEC.H]
    moe.moe_mxfp4_down_combine(hq_d, hs_d, wd, sd, o_d, s_d, w_d, T, SPEC.k, out, y)
    assert bits_equal(host(out), out_ref)
    assert bits_equal(host(y), y_ref)
    if T < 17:  # one launch: the y buffer is optional
        out2 = torch.empty(T, SPEC.H, device="cuda")
        moe.moe_mxfp4_down_combine(hq_d, hs_d, wd, sd, o_d, s_d, w_d, T, SPEC.k, out2)
        assert bits_equal(host(out2), out_ref)
    # against the oracle: per slot down outputs, then the weighted sum
    yo = np.empty((T * SPEC.k, SPEC.H))
    for a in range(T * SPEC.k):
        e = ex[ids.ravel()[a]]
        yo[a] = oracle.expert_down(hq[a], hs[a], e.wd, e.sd)
    oo = oracle.combine(yo, w.astype(np.float64))
    assert max_err_over_rms(host(out), oo) <= TOL
    assert moe.moe_device_status() == 0


def test_zero_weight_slot_reads_no_y(moe, weights):
    """A slot of weight exactly 0 (top-k's slot with no expert) adds nothing:
    its unwritten y row, here NaN, never reaches the output."""
    _, wd, sd = weights
    T = 4
    ids, hq, hs, w = _inputs(T, 90)
    ids[:, -1] = 0x7FFFFFFF - 0  # the last slot of every token has no expert
    w[:, -1] = 0.0
    flat = ids.ravel()
    valid = flat != 0x7FFFFFFF
    order = np.argsort(np.where(valid, flat, SPEC.E), kind="stable")
    srt = order[: valid.sum()].astype(np.int32)
    counts = np.bincount(flat[valid], minlength=SPEC.E)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    out = torch.empty(T, SPEC.H, device="cuda")
    moe.moe_mxfp4_down_combine(dev(hq), dev(hs), wd, sd, dev(offsets), dev(srt), dev(w), T, SPEC.k, out)
    assert np.isfinite(host(out)).all()
    y = torch.full((T * SPEC.k, SPEC.H), float("nan"), device="cuda")
    moe.moe_mxfp4_down(dev(hq), dev(hs), wd, sd, dev(offsets), dev(srt), T, SPEC.k, y)
    ref = torch.empty(T, SPEC.H, device="cuda")
    moe.moe_combine(y, dev(w), ref)
    assert bits_equal(host(out), host(ref))
    assert moe.moe_device_status() == 0


def test_two_launch_fallback_needs_y(moe, weights):
    _, wd, sd = weights
    T = 20
    ids, hq, hs, w = _inputs(T, 91)
    offsets, srt, _ = oracle.sort(ids, SPEC.E, 1)
    out = torch.empty(T, SPEC.H, device="cuda")
    with pytest.raises(moe.MoeError) as err:
        moe.moe_mxfp4_down_combine(dev(hq), dev(hs), wd, sd, dev(offsets), dev(srt), dev(w), T, SPEC.k, out)
    assert err.value.status == moe.MOE_ERR_UNSUPPORTED
