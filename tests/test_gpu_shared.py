"""The shared expert ("DeepSeek-V4-Flash on AMD gfx90a", Execution structure
and Fig. 1: a shared expert beside the routed experts, both feeding the join
that adds their partials) against the oracle.

The layer runs it as the stage calls on a one-expert weight set (every token,
weight 1) followed by moe_join_add after the routed stage calls, or inside
the single launch (moe_decode_forward_shared) for small batches.  Checked
here:

* the join: the joined output equals, bit for bit, the fp32 sum of the
  routed-only output and the shared expert's output;
* the single launch against the stage calls: the same bits for the output,
  the shared expert's h and its down output;
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
    # the scales carry h's error: fp32 rounding up to 16 rows; beyond, the
    # tensor path's h is held to the layer's tolerance (max|err| <= TOL * RMS)
    assert np.allclose(host(ws.sh_hs), hs_o, rtol=TOL, atol=0)
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


def _check_fused_equals_stages(moe, lw, x, T):
    """The single launch with the shared expert gives the stage calls' bits."""
    assert moe.MoeLayer(lw).shared_in_one_launch(T)
    ws_f = moe.Workspace(T, lw, "cuda")
    out_f = host(moe.MoeLayer(lw, fused=True).forward(x, ws_f)).copy()
    ws_s, out_s = _run(moe, lw, x, T, False)
    assert bits_equal(out_f, out_s)
    assert bits_equal(host(ws_f.sh_y), host(ws_s.sh_y))
    assert bits_equal(host(ws_f.sh_h), host(ws_s.sh_h))
    assert moe.moe_device_status() == 0
    return ws_s


def _run_mode(moe, lw, x, T, mode):
    """mode "one": the single launch with the shared expert (checked against
    the stage calls bit for bit); "mixed": the routed single launch, then the
    shared expert's stage calls; "stages": stage calls for both."""
    layer = moe.MoeLayer(lw)
    if mode == "one":
        return _check_fused_equals_stages(moe, lw, x, T)
    if mode == "mixed":
        if not layer.use_fused(T) or layer.shared_in_one_launch(T):
            pytest.skip("this batch is not between the two single-launch limits")
        return _run(moe, lw, x, T, True)[0]
    return _run(moe, lw, x, T, False)[0]


@pytest.mark.parametrize("T,mode", [(1, "one"), (3, "one"), (3, "stages"), (16, "stages"), (20, "stages")])
def test_shared_expert_tiny(moe, T, mode):
    spec = synth.TINY
    sh, lw = _with_shared(upload_layer(spec), spec)
    x = synth.activations(spec, T)
    ws = _run_mode(moe, lw, dev(x), T, mode)
    xq, xs = oracle.quant_q8(x)
    _check_shared_output(ws, oracle.shared_expert(xq, xs, sh))


@pytest.mark.parametrize("T,mode", [(1, "one"), (3, "one"), (4, "mixed"), (8, "stages"), (24, "stages")])
def test_shared_expert_dsv4(moe, T, mode):
    spec = synth.DSV4
    x = synth.activations(spec, T, token0=40)
    _, ids, _ = oracle.route(x, synth.router_weights(spec), spec.k)
    sh, lw = _with_shared(upload_layer(spec, only=set(ids.ravel().tolist())), spec)
    ws = _run_mode(moe, lw, dev(x), T, mode)
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
