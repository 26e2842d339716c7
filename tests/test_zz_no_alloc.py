"""moe_decode_forward_noalloc: the decode layer for callers that cannot
allocate device memory when they run it (a runtime that owns all device
memory, an embedder that forbids allocation after start-up).

The entry point keeps its intermediates in a fixed device array owned by the
library, so its only output is the layer output.  These tests call it through
the C ABI twice in a row (the second call reuses what the first left in the
array) and compare each result with moe_decode_forward, which takes its
buffers from the caller.  This file is collected last on purpose: it must
pass both alone in a fresh process and after every other GPU test.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import TOL, bits_equal, dev, ensure_built, host, max_err_over_rms, upload_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    return ensure_built()


@pytest.fixture(scope="module")
def dsv4(moe):
    return upload_layer(synth.DSV4)


def _with_caller_buffers(moe, lw, x):
    ws = moe.Workspace(x.shape[0], lw, "cuda")
    moe.moe_decode_forward(x, lw.wr, lw.bias, lw.wg, lw.sg, lw.wu, lw.su, lw.wd, lw.sd, lw.k, ws.out, ws.logits,
                           ws.ids, ws.w, ws.h, ws.y, ws.decode_ws)
    torch.cuda.synchronize()
    return host(ws.out)


def _no_alloc(moe, lw, x):
    out = torch.full((x.shape[0], lw.H), float("nan"), dtype=torch.float32, device="cuda")
    moe.moe_decode_forward_noalloc(x, lw.wr, lw.bias, lw.wg, lw.sg, lw.wu, lw.su, lw.wd, lw.sd, lw.k, out)
    torch.cuda.synchronize()
    return host(out)


def test_no_alloc_matches_caller_buffers_twice(moe, dsv4):
    tmax = moe.moe_decode_max_tokens(dsv4.H, dsv4.E, dsv4.k, dsv4.I)
    batches = [dev(synth.activations(synth.DSV4, tmax, token0=9100)),
               dev(synth.activations(synth.DSV4, 1, token0=9200))]
    got = [_no_alloc(moe, dsv4, x) for x in batches]  # two calls in a row
    for x, g in zip(batches, got):
        ref = _with_caller_buffers(moe, dsv4, x)
        assert np.isfinite(g).all()
        assert max_err_over_rms(g, ref) <= TOL
        assert bits_equal(g, ref)  # same kernel, same arithmetic
    assert moe.moe_device_status() == 0


def test_no_alloc_rejects_sizes_beyond_its_array(moe, dsv4):
    x = dev(synth.activations(synth.DSV4, 11))  # T*k = 66 > 64 slots
    out = torch.zeros(11, dsv4.H, dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoeError, match="scratch limit"):
        moe.moe_decode_forward_noalloc(x, dsv4.wr, dsv4.bias, dsv4.wg, dsv4.sg, dsv4.wu, dsv4.su, dsv4.wd, dsv4.sd,
                                       dsv4.k, out)
