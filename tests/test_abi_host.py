"""Host-side checks of the C ABI that need no GPU: the library builds for
sm_103a, exports exactly what include/moe_mxfp4.h declares, and rejects bad
arguments on the host before touching CUDA."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from mxfp4_mixture_experts_moe_gb300 import build
    build.build()
    import mxfp4_mixture_experts_moe_gb300 as moe
    return moe.load()


def _declared():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            src = open(os.path.join(inc, f)).read()
            names |= set(re.findall(r"^MOE_API\s+[\w\s\*]*?\b(\w+)\s*\(", src, re.M))
    return names


def test_header_declares_the_abi():
    d = _declared()
    for n in ("moe_route_topk", "moe_sort_tokens", "act_quant_q8", "moe_mxfp4_gateup_swiglu", "moe_mxfp4_down",
              "moe_combine"):
        assert n in d


def test_library_exports_every_declared_symbol(lib):
    import mxfp4_mixture_experts_moe_gb300 as moe
    for n in _declared():
        assert hasattr(lib, n), n
    assert set(moe.EXPORTS) == _declared()
    assert lib.moe_abi_version() == 4


def test_library_exports_nothing_else():
    import subprocess
    from mxfp4_mixture_experts_moe_gb300 import build
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True).stdout
    syms = {l.split()[-1] for l in out.splitlines() if l.split()[1] in ("T", "W")}
    ours = {s for s in syms if s.startswith(("moe_", "act_"))}
    assert ours == _declared()


def test_host_validation_rejects_bad_arguments(lib):
    import mxfp4_mixture_experts_moe_gb300 as moe
    p = C.c_void_p(16)
    # H not a multiple of 8
    st = lib.moe_route_topk(p, 1, 16, p, 1, None, 1, 12, 8, 2, p, p, p, None)
    assert st == moe.MOE_ERR_INVALID_ARG and "multiple of 8" in lib.moe_last_error().decode()
    # k > 8
    assert lib.moe_route_topk(p, 1, 256, p, 1, None, 1, 256, 16, 9, p, p, p, None) == moe.MOE_ERR_INVALID_ARG
    # E > 1024 unsupported
    assert lib.moe_route_topk(p, 1, 256, p, 1, None, 1, 256, 2048, 2, p, p, p, None) == moe.MOE_ERR_UNSUPPORTED
    # misaligned x
    assert lib.moe_route_topk(C.c_void_p(18), 1, 256, p, 1, None, 1, 256, 8, 2, p, p, p, None) == \
        moe.MOE_ERR_INVALID_ARG
    # Q8: cols not a multiple of 32; q stride not a multiple of 16
    assert lib.act_quant_q8(p, 0, 1, 40, 40, p, 48, p, 2, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.act_quant_q8(p, 0, 2, 64, 64, p, 72, p, 2, None) == moe.MOE_ERR_INVALID_ARG
    # sort: cap too small
    assert lib.moe_sort_tokens(p, 4, 6, 256, 64, p, p, 24, p, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_sort_tokens_capacity(4, 6, 256, 64) == 24 + 256 * 63
    # projections: H not a multiple of 128, reduction length too long, null pointer
    assert lib.moe_mxfp4_gateup_swiglu(p, 16, p, 1, p, p, p, p, p, p, 8, 1, 1, 1, 96, 128, p, 128, None) == \
        moe.MOE_ERR_INVALID_ARG
    assert lib.moe_mxfp4_gateup_swiglu(p, 8192, p, 256, p, p, p, p, p, p, 8, 1, 1, 1, 8192, 128, p, 128,
                                       None) == moe.MOE_ERR_UNSUPPORTED
    assert lib.moe_mxfp4_down(None, 16, p, 1, p, p, p, p, 8, 1, 1, 1, 128, 128, p, 128, None) == \
        moe.MOE_ERR_INVALID_ARG
    # combine: output stride shorter than H
    assert lib.moe_combine(p, 64, p, 1, 2, 64, p, 32, None) == moe.MOE_ERR_INVALID_ARG
    # shared-expert join: stride shorter than H, null output, negative T
    assert lib.moe_join_add(p, 32, 1, 64, p, 64, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_join_add(p, 64, 1, 64, None, 64, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_join_add(p, 64, -1, 64, p, 64, None) == moe.MOE_ERR_INVALID_ARG
    # fused down + combine: null routing weights; T = 0 is a no-op
    assert lib.moe_mxfp4_down_combine(p, 16, p, 1, p, p, p, p, 8, None, 1, 1, 1, 128, 128, p, 128, None, 0,
                                      None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_mxfp4_down_combine(None, 16, None, 1, None, None, None, None, 0, None, 0, 6, 256, 4096, 2048,
                                      None, 4096, None, 0, None) == moe.MOE_OK
    # tensor-core probe: unsupported n, iteration count out of range (nothing launched)
    f = C.c_double(0.0)
    assert lib.moe_mxf4_mma_probe(96, 16, C.byref(f), None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_mxf4_mma_probe(64, 0, C.byref(f), None) == moe.MOE_ERR_INVALID_ARG


def test_empty_batch_is_a_host_noop(lib):
    import mxfp4_mixture_experts_moe_gb300 as moe
    # T = 0 returns before any CUDA call (works without a GPU)
    assert lib.moe_route_topk(None, 1, 256, None, 1, None, 0, 256, 8, 2, None, None, None, None) == moe.MOE_OK
    assert lib.act_quant_q8(None, 0, 0, 64, 64, None, 64, None, 2, None) == moe.MOE_OK
    assert lib.moe_combine(None, 64, None, 0, 2, 64, None, 64, None) == moe.MOE_OK
    assert lib.moe_join_add(None, 64, 0, 64, None, 64, None) == moe.MOE_OK
    assert lib.moe_mxfp4_down(None, 16, None, 1, None, None, None, None, 0, 0, 6, 256, 4096, 2048, None, 4096,
                              None) == moe.MOE_OK
