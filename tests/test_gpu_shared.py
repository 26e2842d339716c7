"""The shared expert ("DeepSeek-V4-Flash on AMD gfx90a", Execution structure
and Fig. 1: a shared expert beside the routed experts, both feeding the join
that adds their partials) against the oracle.

The layer runs it as the stage calls on a one-expert weight set (every token,
weight 1) followed by moe_join_add, after either the single-launch routed
path or the routed stage calls.  Checked here:

* the join: the joined output equals, bit for bit, the fp32 sum of the
  routed-only output and the shared expert's output;
* the shared expert's output against the oracle's, max|err| <= 1e-3 * RMS,
  plus the one-step Q8(h) allowance of the layer tests (a code of the
  GPU's h may sit one step from the oracle's where h * (1/scale) lies near a
  .5 boundary; codes never differ by more than one step);
* exact rows: for 1-16 rows (the CUDA-core kernels) every row of the shared
  expert's output equals the one-row call's bits.
"""
import dataclasses

import numpy as np
import pytest

import oracle
import synth
from gpu_util import TOL, bits_equal, dev, ensure_built, host, upload_layer

pytestmark = pytest.mark.gpu

_NAMES = ("wg", "sg", "wu", "su", "wd", "sd")


@pytest.fixture(scope="module")
def moe():
    return ensure_built()


def _with_shared(lw, spec):
    from mxfp4_mixture_experts_moe_gb300 import SharedExpertWeights
    sh = synth.shared_expert(spec)
    shd = SharedExpertWeights(**{n: dev(getattr(sh, n)[None]) for n in _NAMES})
    return sh, dataclasses.replace(lw, shared=shd)


def _check_shared_output(ws, r):
    """ws.sh_y against the oracle's ys, with the Q8(h) flip allowance."""
    hq_g = host(ws.sh_hq).astype(np.int32)
    hq_o = r["hq"].astype(np.int32)
    hs_o = r["hs"].astype(np.float64)
    assert np.allclose(host(ws.sh_hs), hs_o, rtol=1e-4, atol=0)
    flip = hq_g != hq_o
    assert np.all(np.abs(hq_g - hq_o) <= 1)
    allow = (np.repeat(hs_o, 32, axis=1) * flip * 6.0).sum(axis=1)  # |w| <= 6 (E8M0 <= 127)
    yg, yo = host(ws.sh_y).astype(np.float64), r["ys"]
    assert np.isfinite(yg).all()
    rms = np.sqrt(np.mean(yo ** 2))
    assert np.all(np.abs(yg - yo).max(axis=1) <= TOL * rms + allow)


def _run(moe, lw, x, T, fused):
    """Routed-only and joined forwards of the same tokens; returns the joined
    workspace and the routed-only output."""
    routed = dataclasses.replace(lw, shared=None)
    ws_r = moe.Workspace(T, routed, "cuda")
    out_r = host(moe.MoeLayer(routed, fused=fused).forward(x, ws_r)).copy()
    ws = moe.Workspace(T, lw, "cuda")
    out = host(moe.MoeLayer(lw, fused=fused).forward(x, ws)).copy()
    assert moe.moe_device_status() == 0
    assert bits_equal(out, (out_r + host(ws.sh_y)).astype(np.float32))
    return ws, out


@pytest.mark.parametrize("T,fused", [(1, True), (3, True), (3, False), (16, False), (20, False)])
def test_shared_expert_tiny(moe, T, fused):
    spec = synth.TINY
    sh, lw = _with_shared(upload_layer(spec), spec)
    x = synth.activations(spec, T)
    ws, out = _run(moe, lw, dev(x), T, fused)
    xq, xs = oracle.quant_q8(x)
    _check_shared_output(ws, oracle.shared_expert(xq, xs, sh))


@pytest.mark.parametrize("T,fused", [(1, True), (8, False), (24, False)])
def test_shared_expert_dsv4(moe, T, fused):
    spec = synth.DSV4
    x = synth.activations(spec, T, token0=40)
    _, ids, _ = oracle.route(x, synth.router_weights(spec), spec.k)
    sh, lw = _with_shared(upload_layer(spec, only=set(ids.ravel().tolist())), spec)
    ws, out = _run(moe, lw, dev(x), T, fused)
    xq, xs = oracle.quant_q8(x)
    _check_shared_output(ws, oracle.shared_expert(xq, xs, sh))


def test_shared_expert_rows_are_exact_across_batch_sizes(moe):
    spec = synth.TINY
    sh, lw = _with_shared(upload_layer(spec), spec)
    x = synth.activations(spec, 16, token0=7)
    one = []
    for t in range(16):
        ws = moe.Workspace(1, lw, "cuda")
        moe.MoeLayer(lw, fused=False).forward(dev(x[t:t + 1]), ws)
        one.append(host(ws.sh_y)[0].copy())
    for T in (2, 5, 16):
        ws = moe.Workspace(T, lw, "cuda")
        moe.MoeLayer(lw, fused=False).forward(dev(x[:T]), ws)
        yg = host(ws.sh_y)
        for t in range(T):
            assert bits_equal(yg[t], one[t]), (T, t)
    assert moe.moe_device_status() == 0
