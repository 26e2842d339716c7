"""The single-launch decode path (moe_decode_forward) against the six stage
calls and the oracle.

The fused kernel uses the same device arithmetic as the stage kernels, so its
outputs must be bit-identical to running the stages in sequence, at every
batch size it accepts (the exact-rows contract of "Optimizing DeepSeek V4
Flash Inference on a Strix Halo Pair": a row's bits never depend on the
batch or on the code path that computed them).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import TOL, bits_equal, dev, ensure_built, host, max_err_over_rms, upload_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    return ensure_built()


@pytest.fixture(scope="module")
def dsv4(moe):
    return upload_layer(synth.DSV4)


def _forward(moe, lw, x, fused, pad=0):
    ws = moe.Workspace(x.shape[0], lw, "cuda", pad=pad)
    layer = moe.MoeLayer(lw, fused=fused)
    assert layer.use_fused(x.shape[0]) == bool(fused), (x.shape[0], layer._max_t if fused else None)
    layer.forward(x, ws)
    torch.cuda.synchronize()
    return ws


def _same(a, b, fields=("out", "ids", "logits", "w", "h", "y")):
    for f in fields:
        assert bits_equal(host(getattr(a, f)), host(getattr(b, f))), f


def test_fused_limit(moe, dsv4):
    tmax = moe.moe_decode_max_tokens(4096, 256, 6, 2048)
    assert tmax >= 4
    x_ok = dev(synth.activations(synth.DSV4, tmax))
    ws = moe.Workspace(tmax, dsv4, "cuda")
    moe.moe_decode_forward(x_ok, dsv4.wr, None, dsv4.wg, dsv4.sg, dsv4.wu, dsv4.su, dsv4.wd, dsv4.sd, 6, ws.out,
                           ws.logits, ws.ids, ws.w, ws.h, ws.y, ws.decode_ws)
    # the bound holds for fp32 activations and router; bf16 staging is smaller
    x = dev(synth.activations(synth.DSV4, 12))
    ws = moe.Workspace(12, dsv4, "cuda")  # T*k = 72 > 64: always beyond the fused path
    with pytest.raises(moe.MoeError):
        moe.moe_decode_forward(x, dsv4.wr, None, dsv4.wg, dsv4.sg, dsv4.wu, dsv4.su, dsv4.wd, dsv4.sd, 6, ws.out,
                               ws.logits, ws.ids, ws.w, ws.h, ws.y, ws.decode_ws)


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5])
def test_fused_equals_stage_calls(moe, dsv4, T):
    x = dev(synth.activations(synth.DSV4, T, token0=4000 + T))
    _same(_forward(moe, dsv4, x, True), _forward(moe, dsv4, x, False))
    assert moe.moe_device_status() == 0


def test_fused_one_token_sweep(moe, dsv4):
    """Many one-token calls, each against the stage calls bit for bit.  The
    two consumer groups of the single launch share its three ring stages, so
    this also checks that no group reads a stage before its own item landed
    (a parity wait that met a barrier one phase behind gave wrong h rows in a
    few calls of a sweep like this one)."""
    x = synth.activations(synth.DSV4, 24, token0=900)
    for t in range(x.shape[0]):
        xt = dev(x[t:t + 1])
        _same(_forward(moe, dsv4, xt, True), _forward(moe, dsv4, xt, False))
    assert moe.moe_device_status() == 0


def test_fused_tiny_layer_and_padding(moe):
    spec = synth.TINY  # I = 128 < 152 SMs: some CTAs own no gate/up rows
    lw = upload_layer(spec)
    for T in (1, 5, 14):
        x = dev(synth.activations(spec, T), 24)
        a = _forward(moe, lw, x, True, pad=40)
        _same(a, _forward(moe, lw, x, False))
    assert moe.moe_device_status() == 0


def test_fused_skewed_routing(moe, dsv4):
    from mxfp4_mixture_experts_moe_gb300 import LayerWeights
    lw = LayerWeights(wr=dsv4.wr, bias=dev(synth.router_bias(synth.DSV4_ZIPF)), wg=dsv4.wg, sg=dsv4.sg,
                      wu=dsv4.wu, su=dsv4.su, wd=dsv4.wd, sd=dsv4.sd, k=dsv4.k)
    x = dev(synth.activations(synth.DSV4_ZIPF, 5, token0=77))
    a, b = _forward(moe, lw, x, True), _forward(moe, lw, x, False)
    _same(a, b)
    assert len(np.unique(host(a.ids))) < 30  # several tokens share experts


def test_fused_vs_oracle(moe, dsv4):
    spec = synth.DSV4
    x = synth.activations(spec, 3, token0=808)
    ws = _forward(moe, dsv4, dev(x), True)
    _, ids, _ = oracle.route(x, synth.router_weights(spec), spec.k)
    r = oracle.layer(x, synth.router_weights(spec), None, spec.k,
                     {int(e): synth.expert(spec, int(e)) for e in np.unique(ids)})
    assert np.array_equal(host(ws.ids), r["ids"])
    assert bits_equal(host(ws.logits), r["logits"])
    assert max_err_over_rms(host(ws.h), r["h"]) <= TOL
    assert max_err_over_rms(host(ws.out), r["out"]) <= TOL


def test_fused_graph_replay(moe, dsv4):
    x = dev(synth.activations(synth.DSV4, 1, token0=9))
    ws = moe.Workspace(1, dsv4, "cuda")
    layer = moe.MoeLayer(dsv4, fused=True)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()  # buffers were filled on the default stream
    with torch.cuda.stream(s):
        layer.forward(x, ws, s)
    torch.cuda.synchronize()
    ref = host(ws.out).copy()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        layer.forward(x, ws, s)
    for i in range(300):
        ws.out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert bits_equal(host(ws.out), ref), i


@pytest.mark.parametrize("T", [1, 4])
def test_fused_barrier_timeout_is_reported(moe, dsv4, T):
    """A grid barrier that can never complete (the workspace's hold word
    raises every barrier's target above the number of CTAs) must give up
    within its time bound, raise MOE_DEV_WAIT_TIMEOUT and return; with the
    hold cleared the next call works again.  T = 4 is a shape whose Q8(h)
    rows take the ring's last stage in the down phase, so the producer's
    exit drain must find that stage's last copy among the gate/up items."""
    x = dev(synth.activations(synth.DSV4, T, token0=10))
    ws = moe.Workspace(T, dsv4, "cuda")
    layer = moe.MoeLayer(dsv4, fused=True)
    layer.forward(x, ws)
    assert moe.moe_device_status() == 0
    ref = host(ws.out).copy()
    ws.decode_ws[1] = 1
    layer.forward(x, ws)
    assert moe.moe_device_status() & moe.MOE_DEV_WAIT_TIMEOUT
    ws.decode_ws[1] = 0
    ws.out.zero_()
    layer.forward(x, ws)
    assert moe.moe_device_status() == 0
    assert bits_equal(host(ws.out), ref)


@pytest.mark.parametrize("T", [1, 4])
def test_fused_readiness_timeout_is_reported(moe, dsv4, T):
    """The wait for every CTA's h slices (the per-expert readiness words) runs
    out when the workspace's readiness hold raises its target above the
    number of CTAs.  The kernel must raise MOE_DEV_WAIT_TIMEOUT and return;
    its consumer warps still wait (bounded) for each ring copy before they
    release its stage, so the producer never re-arms a stage with a copy in
    flight and leaves none behind.  With the hold cleared the next call gives
    the bits of the call before."""
    x = dev(synth.activations(synth.DSV4, T, token0=11))
    ws = moe.Workspace(T, dsv4, "cuda")
    layer = moe.MoeLayer(dsv4, fused=True)
    layer.forward(x, ws)
    assert moe.moe_device_status() == 0
    ref = host(ws.out).copy()
    ws.decode_ws[2] = 1
    layer.forward(x, ws)
    assert moe.moe_device_status() & moe.MOE_DEV_WAIT_TIMEOUT
    ws.decode_ws[2] = 0
    ws.out.zero_()
    layer.forward(x, ws)
    assert moe.moe_device_status() == 0
    assert bits_equal(host(ws.out), ref)


def test_fused_nan_scores_are_flagged_not_followed(moe, dsv4):
    """NaN activations make every router score NaN, so top-k has no valid
    expert: every slot gets the oracle's "no expert" id 0x7fffffff.  The
    fused kernel must flag the ids and read no weights for them (and not
    fault); the stage path's sorter does the same."""
    x = torch.full((1, 4096), float("nan"), dtype=torch.bfloat16, device="cuda")
    for fused in (True, False):
        ws = moe.Workspace(1, dsv4, "cuda")
        moe.MoeLayer(dsv4, fused=fused).forward(x, ws)
        assert moe.moe_device_status() & moe.MOE_DEV_BAD_EXPERT_ID
        ref_ids, _ = oracle.topk(host(ws.logits), dsv4.k)
        assert np.array_equal(host(ws.ids), ref_ids)
        assert (ref_ids == 0x7FFFFFFF).all()


@pytest.mark.parametrize("T", [1, 3])
def test_nan_router_rows_match_the_oracle(moe, T):
    """Every router row but expert 3's is NaN, so each token's second slot has
    no expert.  On the single launch and on the stage calls alike, the ids
    (0x7fffffff for that slot), the weights (1 and 0) and the layer output
    (the empty slot adds nothing) match the oracle, and the device status
    flags the missing expert."""
    spec = synth.TINY
    wr = synth.router_weights(spec).copy()
    wr[[e for e in range(spec.E) if e != 3]] = np.nan
    lw = upload_layer(spec)
    lw.wr = dev(wr)
    xh = synth.activations(spec, T, token0=60)
    r = oracle.layer(xh, wr, None, spec.k, {3: synth.expert(spec, 3)})
    assert (r["ids"][:, 1] == 0x7FFFFFFF).all()
    outs = []
    for fused in (True, False):
        ws = moe.Workspace(T, lw, "cuda")
        ws.y.fill_(float("nan"))  # rows no projection writes must not be read
        moe.MoeLayer(lw, fused=fused).forward(dev(xh), ws)
        assert moe.moe_device_status() & moe.MOE_DEV_BAD_EXPERT_ID
        assert np.array_equal(host(ws.ids), r["ids"])
        assert np.allclose(host(ws.w), r["w"], rtol=1e-6, atol=0)
        assert max_err_over_rms(host(ws.out), r["out"]) <= TOL
        outs.append(host(ws.out))
    assert bits_equal(outs[0], outs[1])


def test_fused_single_expert_per_token(moe):
    """k = 1 (one expert per token): the assignment is the token itself, in the
    fused kernel and in the stage calls alike."""
    spec = synth.LayerSpec(H=256, E=8, k=1, I=128, x_dtype="f32", wr_dtype="f32", seed=41)
    lw = upload_layer(spec)
    for T in (1, 4):
        x = dev(synth.activations(spec, T, token0=50))
        a, b = _forward(moe, lw, x, True), _forward(moe, lw, x, False)
        _same(a, b)
        xs = synth.activations(spec, T, token0=50)
        _, ids, _ = oracle.route(xs, synth.router_weights(spec), spec.k)
        r = oracle.layer(xs, synth.router_weights(spec), None, spec.k,
                         {e: synth.expert(spec, e) for e in np.unique(ids).tolist()})
        assert max_err_over_rms(host(a.out), r["out"]) <= TOL
    assert moe.moe_device_status() == 0
