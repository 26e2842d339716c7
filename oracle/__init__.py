"""CPU oracle of the MXFP4 routed-expert MoE layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline /
``--impl reference`` leg may import this package.  The product path (the
``mxfp4_mixture_experts_moe_gb300`` package and its CUDA library) never
imports, loads or calls it, and shares no code with it.

This module only marshals numpy arrays into the plain C oracle in
``moe_oracle.c`` (built on demand with gcc into ``oracle/_build``); every step
of the arithmetic lives there, each function citing the passage it follows.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11, no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            P = C.c_void_p
            i64 = C.c_int64
            L.moe_oracle_e2m1.argtypes = [C.c_int]
            L.moe_oracle_e2m1.restype = C.c_double
            L.moe_oracle_e8m0.argtypes = [C.c_int]
            L.moe_oracle_e8m0.restype = C.c_double
            L.moe_oracle_silu.argtypes = [C.c_double]
            L.moe_oracle_silu.restype = C.c_double
            L.moe_oracle_router_logits.argtypes = [P, C.c_int, i64, P, C.c_int, C.c_int, C.c_int, C.c_int, P]
            L.moe_oracle_topk.argtypes = [P, P, C.c_int, C.c_int, C.c_int, P, P]
            L.moe_oracle_sort.argtypes = [P, C.c_int, C.c_int, C.c_int, C.c_int, P, P, i64, P]
            L.moe_oracle_sort.restype = i64
            L.moe_oracle_quant_q8.argtypes = [P, C.c_int, C.c_int, C.c_int, i64, P, i64, P, i64]
            L.moe_oracle_block_dot.argtypes = [P, P]
            L.moe_oracle_block_dot.restype = C.c_int32
            L.moe_oracle_expert_gateup.argtypes = [P, P, P, P, P, P, C.c_int, C.c_int, P, P]
            L.moe_oracle_expert_down.argtypes = [P, P, P, P, C.c_int, C.c_int, P]
            L.moe_oracle_combine.argtypes = [P, P, C.c_int, C.c_int, C.c_int, P]
            L.moe_oracle_layer.argtypes = ([P, C.c_int, C.c_int, C.c_int, P, C.c_int, P, C.c_int, C.c_int, C.c_int]
                                           + [P] * 6 + [P] * 10)
            L.moe_oracle_layer.restype = C.c_int
            L.moe_oracle_shared_expert.argtypes = [P, P, C.c_int, C.c_int, C.c_int] + [P] * 6 + [P] * 5
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _is_bf16(a: np.ndarray) -> int:
    if a.dtype == np.uint16:
        return 1
    if a.dtype == np.float32:
        return 0
    raise TypeError(f"expected float32 or bf16 bits (uint16), got {a.dtype}")


def e2m1(code: int) -> float:
    return lib().moe_oracle_e2m1(int(code))


def e8m0(u: int) -> float:
    return lib().moe_oracle_e8m0(int(u))


def silu(g: float) -> float:
    return lib().moe_oracle_silu(float(g))


def router_logits(x: np.ndarray, wr: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x)
    wr = np.ascontiguousarray(wr)
    T, H = x.shape
    E = wr.shape[0]
    out = np.empty((T, E), dtype=np.float32)
    lib().moe_oracle_router_logits(_p(x), _is_bf16(x), H, _p(wr), _is_bf16(wr), T, H, E, _p(out))
    return out


def topk(logits: np.ndarray, k: int, bias: np.ndarray | None = None):
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = logits.shape
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    lib().moe_oracle_topk(_p(logits), _p(b), T, E, k, _p(ids), _p(w))
    return ids, w


def sort(ids: np.ndarray, E: int, tile_rows: int = 1):
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = ids.shape
    A = T * k
    cap = A + E * (tile_rows - 1)
    offsets = np.empty(E + 1, dtype=np.int32)
    srt = np.empty(max(cap, 1), dtype=np.int32)
    inv = np.empty(max(A, 1), dtype=np.int32)
    n = lib().moe_oracle_sort(_p(ids), T, k, E, tile_rows, _p(offsets), _p(srt), cap, _p(inv))
    if n < 0:
        raise ValueError(f"oracle sort failed ({n})")
    return offsets, srt[:n], inv[:A]


def quant_q8(x: np.ndarray):
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    q = np.empty((rows, cols), dtype=np.int8)
    d = np.empty((rows, cols // 32), dtype=np.float32)
    lib().moe_oracle_quant_q8(_p(x), _is_bf16(x), rows, cols, cols, _p(q), cols, _p(d), cols // 32)
    return q, d


def block_dot(q32: np.ndarray, nib16: np.ndarray) -> int:
    q32 = np.ascontiguousarray(q32, dtype=np.int8)
    nib16 = np.ascontiguousarray(nib16, dtype=np.uint8)
    assert q32.size == 32 and nib16.size == 16
    return int(lib().moe_oracle_block_dot(_p(q32), _p(nib16)))


def expert_gateup(xq, xs, wg, sg, wu, su):
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    xs = np.ascontiguousarray(xs, dtype=np.float32)
    I, Hh = wg.shape
    H = 2 * Hh
    G = np.empty(I, dtype=np.float64)
    U = np.empty(I, dtype=np.float64)
    arrs = [np.ascontiguousarray(a, dtype=np.uint8) for a in (wg, sg, wu, su)]
    lib().moe_oracle_expert_gateup(_p(xq), _p(xs), *[_p(a) for a in arrs], H, I, _p(G), _p(U))
    return G, U


def expert_down(hq, hs, wd, sd):
    hq = np.ascontiguousarray(hq, dtype=np.int8)
    hs = np.ascontiguousarray(hs, dtype=np.float32)
    H, Ih = wd.shape
    I = 2 * Ih
    y = np.empty(H, dtype=np.float64)
    wd = np.ascontiguousarray(wd, dtype=np.uint8)
    sd = np.ascontiguousarray(sd, dtype=np.uint8)
    lib().moe_oracle_expert_down(_p(hq), _p(hs), _p(wd), _p(sd), H, I, _p(y))
    return y


def combine(y: np.ndarray, w: np.ndarray) -> np.ndarray:
    y = np.ascontiguousarray(y, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    T, k = w.shape
    H = y.shape[1]
    out = np.empty((T, H), dtype=np.float64)
    lib().moe_oracle_combine(_p(y), _p(w), T, k, H, _p(out))
    return out


def shared_expert(xq, xs, ew, out=None):
    """The shared expert on the Q8 rows xq [T, H] / xs [T, H/32]: ``ew`` has
    wg, sg, wu, su, wd, sd arrays of one expert.  Returns a dict with h, hq,
    hs and ys [T, H] (f64) and, when ``out`` (the routed output [T, H]) is
    given, the joined output routed + ys."""
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    xs = np.ascontiguousarray(xs, dtype=np.float32)
    T, H = xq.shape
    I = ew.wg.shape[0]
    arrs = [np.ascontiguousarray(getattr(ew, n), dtype=np.uint8) for n in ("wg", "sg", "wu", "su", "wd", "sd")]
    r = dict(h=np.empty((T, I), np.float64), hq=np.empty((T, I), np.int8), hs=np.empty((T, I // 32), np.float32),
             ys=np.empty((T, H), np.float64))
    joined = None if out is None else np.array(out, dtype=np.float64, copy=True, order="C")
    lib().moe_oracle_shared_expert(_p(xq), _p(xs), T, H, I, *[_p(a) for a in arrs], _p(r["h"]), _p(r["hq"]),
                                   _p(r["hs"]), _p(r["ys"]), None if joined is None else _p(joined))
    if joined is not None:
        r["out"] = joined
    return r


def layer(x: np.ndarray, wr: np.ndarray, bias, k: int, experts: dict, shared=None):
    """Full layer for the T tokens of x.  ``experts`` maps an expert id to an
    object with wg, sg, wu, su, wd, sd arrays (only the selected experts are
    needed; use :func:`route` first to know which).  Returns a dict of every
    stage: logits, ids, w, xq, xs, h, hq, hs, y, out.  With ``shared`` (one
    expert's arrays) the shared expert joins: out is then routed + shared,
    out_routed the routed part, and shared_h / shared_hq / shared_hs / ys the
    shared expert's stages."""
    x = np.ascontiguousarray(x)
    wr = np.ascontiguousarray(wr)
    T, H = x.shape
    E = wr.shape[0]
    any_e = next(iter(experts.values()))
    I = any_e.wg.shape[0]
    A = T * k
    keep = []

    def ptrs(name):
        arr = (C.c_void_p * E)()
        for e, ew in experts.items():
            a = np.ascontiguousarray(getattr(ew, name), dtype=np.uint8)
            keep.append(a)
            arr[e] = a.ctypes.data
        return arr

    tables = [ptrs(n) for n in ("wg", "sg", "wu", "su", "wd", "sd")]
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    r = dict(
        logits=np.empty((T, E), np.float32), ids=np.empty((T, k), np.int32), w=np.empty((T, k), np.float64),
        xq=np.empty((T, H), np.int8), xs=np.empty((T, H // 32), np.float32),
        h=np.empty((A, I), np.float64), hq=np.empty((A, I), np.int8), hs=np.empty((A, I // 32), np.float32),
        y=np.empty((A, H), np.float64), out=np.empty((T, H), np.float64))
    rc = lib().moe_oracle_layer(
        _p(x), _is_bf16(x), T, H, _p(wr), _is_bf16(wr), _p(b), E, k, I,
        *[C.cast(t, C.c_void_p) for t in tables],
        _p(r["logits"]), _p(r["ids"]), _p(r["w"]), _p(r["xq"]), _p(r["xs"]),
        _p(r["h"]), _p(r["hq"]), _p(r["hs"]), _p(r["y"]), _p(r["out"]))
    if rc != 0:
        raise KeyError("a selected expert's weights were not provided")
    if shared is not None:
        sr = shared_expert(r["xq"], r["xs"], shared, out=r["out"])
        r["out_routed"] = r["out"]
        r["out"] = sr["out"]
        r.update(shared_h=sr["h"], shared_hq=sr["hq"], shared_hs=sr["hs"], ys=sr["ys"])
    return r


def route(x: np.ndarray, wr: np.ndarray, k: int, bias=None):
    """Router logits and top-k only (to learn which experts a batch needs)."""
    logits = router_logits(x, wr)
    ids, w = topk(logits, k, bias)
    return logits, ids, w
