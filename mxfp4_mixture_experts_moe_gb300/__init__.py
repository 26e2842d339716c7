"""GB300 (sm_103a) MXFP4 routed-expert MoE layer: thin Python binding.

Every function here only marshals torch tensors into the C ABI of
``libmoe_mxfp4.so`` (declared in ``include/moe_mxfp4.h``) and raises on a
non-OK status.  All arithmetic runs in the library's CUDA kernels; there is no
CPU or PyTorch fallback: the first call fails loudly when the library has not
been built (``python -m mxfp4_mixture_experts_moe_gb300.build``).

The functions keep the C names and argument order, minus the sizes, which are
read from the tensors' shapes, and with the stream defaulting to PyTorch's
current stream.  The library is loaded on first use (so that the build
module can be imported before it exists); a missing library raises there.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

from .build import LIB as _LIB_PATH


MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_DEVICE = range(5)
MOE_F32, MOE_BF16 = 0, 1
MOE_DEV_BAD_EXPERT_ID, MOE_DEV_BAD_ROW, MOE_DEV_WAIT_TIMEOUT = 0x1, 0x2, 0x4

EXPORTS = ["moe_last_error", "moe_abi_version", "moe_device_status", "moe_route_topk",
           "moe_sort_tokens_capacity", "moe_sort_tokens", "act_quant_q8", "moe_mxfp4_gateup_swiglu",
           "moe_mxfp4_gateup", "moe_mxfp4_down", "moe_mxfp4_down_combine", "moe_combine", "moe_join_add",
           "moe_decode_workspace_bytes",
           "moe_decode_max_tokens", "moe_decode_forward", "moe_decode_forward_noalloc",
           "moe_decode_max_tokens_shared", "moe_decode_forward_shared", "moe_mxf4_mma_probe"]

_P, _I, _L = C.c_void_p, C.c_int, C.c_int64
_SIG = {
    "moe_last_error": (C.c_char_p, []),
    "moe_abi_version": (_I, []),
    "moe_device_status": (_I, [_P, C.POINTER(C.c_uint32)]),
    "moe_route_topk": (_I, [_P, _I, _L, _P, _I, _P, _I, _I, _I, _I, _P, _P, _P, _P]),
    "moe_sort_tokens_capacity": (_L, [_I, _I, _I, _I]),
    "moe_sort_tokens": (_I, [_P, _I, _I, _I, _I, _P, _P, _L, _P, _P]),
    "act_quant_q8": (_I, [_P, _I, _I, _I, _L, _P, _L, _P, _L, _P]),
    "moe_mxfp4_gateup_swiglu": (_I, [_P, _L, _P, _L, _P, _P, _P, _P, _P, _P, _L, _I, _I, _I, _I, _I, _P, _L, _P]),
    "moe_mxfp4_gateup": (_I, [_P, _L, _P, _L, _P, _P, _P, _P, _P, _P, _L, _I, _I, _I, _I, _I, _P, _P, _L, _P]),
    "moe_mxfp4_down": (_I, [_P, _L, _P, _L, _P, _P, _P, _P, _L, _I, _I, _I, _I, _I, _P, _L, _P]),
    "moe_combine": (_I, [_P, _L, _P, _I, _I, _I, _P, _L, _P]),
    "moe_mxfp4_down_combine": (_I, [_P, _L, _P, _L, _P, _P, _P, _P, _L, _P, _I, _I, _I, _I, _I, _P, _L, _P, _L, _P]),
    "moe_join_add": (_I, [_P, _L, _I, _I, _P, _L, _P]),
    "moe_decode_workspace_bytes": (C.c_size_t, []),
    "moe_decode_max_tokens": (_I, [_I, _I, _I, _I]),
    "moe_decode_forward": (_I, [_P, _I, _L, _P, _I, _P] + [_P] * 6 + [_I] * 5 + [_P, _L] + [_P] * 3
                           + [_P, _L, _P, _L, _P, C.c_size_t, _P]),
    "moe_decode_forward_noalloc": (_I, [_P, _I, _L, _P, _I, _P] + [_P] * 6 + [_I] * 5 + [_P, _L, _P]),
    "moe_decode_max_tokens_shared": (_I, [_I, _I, _I, _I]),
    "moe_mxf4_mma_probe": (_I, [_I, _I, C.POINTER(C.c_double), _P]),
    "moe_decode_forward_shared": (_I, [_P, _I, _L, _P, _I, _P] + [_P] * 12 + [_I] * 5 + [_P, _L] + [_P] * 3
                                  + [_P, _L, _P, _L, _P, _L, _P, _L, _P, C.c_size_t, _P]),
}
library_path = _LIB_PATH


class _Native:
    """The loaded C library; loads on first attribute access, raises if absent.
    Each entry point gets its C signature when it is first used."""
    _cdll = None
    _bound = set()

    def __getattr__(self, name):
        if _Native._cdll is None:
            if not os.path.exists(_LIB_PATH):
                raise ImportError(f"{_LIB_PATH} is missing: build it with "
                                  "`python -m mxfp4_mixture_experts_moe_gb300.build` (there is no fallback path)")
            _Native._cdll = C.CDLL(_LIB_PATH)
        f = getattr(_Native._cdll, name)
        if name not in _Native._bound and name in _SIG:
            f.restype, f.argtypes = _SIG[name]
            _Native._bound.add(name)
        return f


_lib = _Native()


def load():
    """Load the library now (raises ImportError if it has not been built) and
    give every entry point it exports its C signature."""
    _lib.moe_abi_version
    for name in _SIG:
        if hasattr(_Native._cdll, name):
            getattr(_lib, name)
    return _Native._cdll


class MoeError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"status {status}: {msg}")
        self.status = status


def _check(status: int):
    if status != MOE_OK:
        raise MoeError(status, _lib.moe_last_error().decode(errors="replace"))


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dt(t):
    if t.dtype == torch.float32:
        return MOE_F32
    if t.dtype == torch.bfloat16:
        return MOE_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ld(t):
    assert t.dim() == 2 and t.stride(1) == 1, "expected a 2-D tensor with unit column stride"
    return t.stride(0)


def moe_abi_version() -> int:
    return _lib.moe_abi_version()


def moe_last_error() -> str:
    return _lib.moe_last_error().decode(errors="replace")


def moe_device_status(stream=None) -> int:
    """Synchronise the stream; return (and clear) the device status bits."""
    flags = C.c_uint32(0)
    st = _lib.moe_device_status(_stream(stream), C.byref(flags))
    if st not in (MOE_OK, MOE_ERR_DEVICE):
        _check(st)
    return flags.value


def moe_route_topk(x, w_router, bias, k, logits, ids, weights, stream=None):
    T, H = x.shape[0], w_router.shape[1]
    E = w_router.shape[0]
    _check(_lib.moe_route_topk(_ptr(x), _dt(x), _ld(x), _ptr(w_router), _dt(w_router), _ptr(bias),
                               T, H, E, k, _ptr(logits), _ptr(ids), _ptr(weights), _stream(stream)))


def moe_sort_tokens_capacity(T, k, E, tile_rows=1) -> int:
    return _lib.moe_sort_tokens_capacity(T, k, E, tile_rows)


def moe_sort_tokens(ids, E, tile_rows, offsets, sorted_, inv, stream=None):
    T, k = ids.shape
    _check(_lib.moe_sort_tokens(_ptr(ids), T, k, E, tile_rows, _ptr(offsets), _ptr(sorted_),
                                sorted_.numel(), _ptr(inv), _stream(stream)))


def act_quant_q8(x, q, scale, stream=None):
    rows, cols = x.shape
    _check(_lib.act_quant_q8(_ptr(x), _dt(x), rows, cols, _ld(x), _ptr(q), _ld(q), _ptr(scale), _ld(scale),
                             _stream(stream)))


def moe_mxfp4_gateup_swiglu(xq, xs, wg, sg, wu, su, offsets, sorted_, k, h, stream=None):
    T, H = xq.shape[0], wg.shape[2] * 2
    E, I = wg.shape[0], wg.shape[1]
    _check(_lib.moe_mxfp4_gateup_swiglu(_ptr(xq), _ld(xq), _ptr(xs), _ld(xs), _ptr(wg), _ptr(sg), _ptr(wu),
                                        _ptr(su), _ptr(offsets), _ptr(sorted_), sorted_.numel(), T, k, E, H, I,
                                        _ptr(h), _ld(h), _stream(stream)))


def moe_mxfp4_gateup(xq, xs, wg, sg, wu, su, offsets, sorted_, k, g, u, stream=None):
    T, H = xq.shape[0], wg.shape[2] * 2
    E, I = wg.shape[0], wg.shape[1]
    assert g.stride() == u.stride()
    _check(_lib.moe_mxfp4_gateup(_ptr(xq), _ld(xq), _ptr(xs), _ld(xs), _ptr(wg), _ptr(sg), _ptr(wu), _ptr(su),
                                 _ptr(offsets), _ptr(sorted_), sorted_.numel(), T, k, E, H, I, _ptr(g), _ptr(u),
                                 _ld(g), _stream(stream)))


def moe_mxfp4_down(hq, hs, wd, sd, offsets, sorted_, T, k, y, stream=None):
    E, H, I = wd.shape[0], wd.shape[1], wd.shape[2] * 2
    _check(_lib.moe_mxfp4_down(_ptr(hq), _ld(hq), _ptr(hs), _ld(hs), _ptr(wd), _ptr(sd), _ptr(offsets),
                               _ptr(sorted_), sorted_.numel(), T, k, E, H, I, _ptr(y), _ld(y), _stream(stream)))


def moe_mxfp4_down_combine(hq, hs, wd, sd, offsets, sorted_, w, T, k, out, y=None, stream=None):
    E, H, I = wd.shape[0], wd.shape[1], wd.shape[2] * 2
    _check(_lib.moe_mxfp4_down_combine(_ptr(hq), _ld(hq), _ptr(hs), _ld(hs), _ptr(wd), _ptr(sd), _ptr(offsets),
                                       _ptr(sorted_), sorted_.numel(), _ptr(w), T, k, E, H, I, _ptr(out), _ld(out),
                                       _ptr(y), 0 if y is None else _ld(y), _stream(stream)))


def moe_combine(y, w, out, stream=None):
    T, k = w.shape
    H = out.shape[1]
    _check(_lib.moe_combine(_ptr(y), _ld(y), _ptr(w), T, k, H, _ptr(out), _ld(out), _stream(stream)))


def moe_join_add(ys, out, stream=None):
    """out += ys (the shared expert's join onto the routed output)."""
    T, H = out.shape
    _check(_lib.moe_join_add(_ptr(ys), _ld(ys), T, H, _ptr(out), _ld(out), _stream(stream)))


def moe_decode_workspace_bytes() -> int:
    return _lib.moe_decode_workspace_bytes()


def moe_decode_max_tokens(H, E, k, I) -> int:
    return _lib.moe_decode_max_tokens(H, E, k, I)


def moe_decode_forward(x, w_router, bias, wg, sg, wu, su, wd, sd, k, out, logits, ids, weights, h, y, workspace,
                       stream=None):
    T, H = x.shape[0], w_router.shape[1]
    E, I = w_router.shape[0], wg.shape[1]
    _check(_lib.moe_decode_forward(_ptr(x), _dt(x), _ld(x), _ptr(w_router), _dt(w_router), _ptr(bias),
                                   _ptr(wg), _ptr(sg), _ptr(wu), _ptr(su), _ptr(wd), _ptr(sd), T, H, E, k, I,
                                   _ptr(out), _ld(out), _ptr(logits), _ptr(ids), _ptr(weights), _ptr(h), _ld(h),
                                   _ptr(y), _ld(y) if y is not None else 0, _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_decode_max_tokens_shared(H, E, k, I) -> int:
    return _lib.moe_decode_max_tokens_shared(H, E, k, I)


def moe_decode_forward_shared(x, w_router, bias, wg, sg, wu, su, wd, sd, shared, k, out, logits, ids, weights, h, y,
                              shared_h, shared_y, workspace, stream=None):
    """moe_decode_forward with the layer's shared expert (``shared`` has its
    wg .. sd, one expert each) in the same launch."""
    T, H = x.shape[0], w_router.shape[1]
    E, I = w_router.shape[0], wg.shape[1]
    _check(_lib.moe_decode_forward_shared(
        _ptr(x), _dt(x), _ld(x), _ptr(w_router), _dt(w_router), _ptr(bias),
        _ptr(wg), _ptr(sg), _ptr(wu), _ptr(su), _ptr(wd), _ptr(sd),
        _ptr(shared.wg), _ptr(shared.sg), _ptr(shared.wu), _ptr(shared.su), _ptr(shared.wd), _ptr(shared.sd),
        T, H, E, k, I, _ptr(out), _ld(out), _ptr(logits), _ptr(ids), _ptr(weights), _ptr(h), _ld(h),
        _ptr(y), _ld(y) if y is not None else 0, _ptr(shared_h), _ld(shared_h),
        _ptr(shared_y), _ld(shared_y) if shared_y is not None else 0, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_decode_forward_noalloc(x, w_router, bias, wg, sg, wu, su, wd, sd, k, out, stream=None):
    """moe_decode_forward for callers that cannot allocate device memory when
    they run the layer (a runtime that owns all device memory, an embedder
    that forbids allocation after start-up): the intermediates live in a
    fixed device array owned by the library (T*k <= 64, T*E <= 32768,
    I <= 4096) and only ``out`` is written.  The first call on a device looks
    up that array; make it before any stream capture.  Calls that overlap on
    the GPU share the array and race."""
    T, H = x.shape[0], w_router.shape[1]
    E, I = w_router.shape[0], wg.shape[1]
    _check(_lib.moe_decode_forward_noalloc(_ptr(x), _dt(x), _ld(x), _ptr(w_router), _dt(w_router), _ptr(bias),
                                           _ptr(wg), _ptr(sg), _ptr(wu), _ptr(su), _ptr(wd), _ptr(sd), T, H, E, k,
                                           I, _ptr(out), _ld(out), _stream(stream)))


from .layer import MoeLayer, LayerWeights, SharedExpertWeights, Workspace  # noqa: E402


def moe_mxf4_mma_probe(n: int, iters: int, stream=None) -> float:
    """Launch the FP4 tensor-core throughput probe (one CTA per SM, `iters`
    M=128 x N=n x K=64 block-scaled MMAs each); returns the launch's flops.
    The caller times the launch (events on the same stream)."""
    flops = C.c_double(0.0)
    _check(_lib.moe_mxf4_mma_probe(int(n), int(iters), C.byref(flops), _stream(stream)))
    return flops.value
