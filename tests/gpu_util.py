"""Helpers shared by the GPU tests: device copies of the seeded synthetic
layer, and the tolerance rule of the parity contract."""
from __future__ import annotations

import numpy as np
import torch

import synth


def ensure_built():
    from mxfp4_mixture_experts_moe_gb300 import build
    build.build()
    import mxfp4_mixture_experts_moe_gb300 as moe
    moe.load()
    return moe


def dev(a: np.ndarray, pad_cols: int = 0) -> torch.Tensor:
    """numpy -> cuda; uint16 arrays are bf16 bit patterns.  With pad_cols the
    result is a view with a padded (still 16-byte aligned) row stride."""
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a))
    if pad_cols and t.dim() == 2:
        full = torch.zeros(t.shape[0], t.shape[1] + pad_cols, dtype=t.dtype)
        full[:, :t.shape[1]] = t
        return full.cuda()[:, :t.shape[1]]
    return t.cuda()


def host(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def bits_equal(a, b) -> bool:
    a = np.ascontiguousarray(a)
    b = np.ascontiguousarray(b)
    return a.shape == b.shape and a.dtype == b.dtype and a.tobytes() == b.tobytes()


def max_err_over_rms(got, ref) -> float:
    """max|got - ref| / RMS(ref); the parity contract asks for <= 1e-3."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    return float(np.max(np.abs(got - ref))) / (rms if rms > 0 else 1.0)


TOL = 1e-3  # max |err| <= 1e-3 * RMS(output) for fp32 outputs


def upload_layer(spec: synth.LayerSpec, experts: dict | None = None, only: set | None = None):
    """Device LayerWeights for spec.  With ``only``, experts outside the set
    are left as zeros (they must never be read)."""
    from mxfp4_mixture_experts_moe_gb300 import LayerWeights
    H, E, I = spec.H, spec.E, spec.I
    wr = dev(synth.router_weights(spec))
    b = synth.router_bias(spec)
    bias = None if b is None else dev(b)
    shapes = dict(wg=(E, I, H // 2), sg=(E, I, H // 32), wu=(E, I, H // 2), su=(E, I, H // 32),
                  wd=(E, H, I // 2), sd=(E, H, I // 32))
    t = {n: torch.zeros(s, dtype=torch.uint8, device="cuda") for n, s in shapes.items()}
    for e in range(E):
        if only is not None and e not in only:
            continue
        ew = experts[e] if experts and e in experts else synth.expert(spec, e)
        for n in shapes:
            t[n][e].copy_(torch.from_numpy(getattr(ew, n)))
    return LayerWeights(wr=wr, bias=bias, k=spec.k, **t)
