"""One MoE layer forward as the sequence of C-ABI calls.

The layer of the DeepSeek-V4-Flash pages ("DeepSeek-V4-Flash on AMD gfx90a",
Fig. 1): route top-k -> sort -> Q8(x) -> gate/up + SwiGLU -> Q8(h) -> down ->
slot-ordered combine, and, when the layer has a shared expert, that expert on
every token (weight 1) joined onto the routed output.  This module only
allocates device buffers (through PyTorch) and issues the calls; it computes
nothing itself.
"""
from __future__ import annotations

import dataclasses

import torch

from . import (act_quant_q8, moe_combine, moe_decode_forward, moe_decode_forward_shared, moe_decode_max_tokens,
               moe_decode_max_tokens_shared, moe_decode_workspace_bytes, moe_join_add, moe_mxfp4_down,
               moe_mxfp4_down_combine, moe_mxfp4_gateup_swiglu, moe_route_topk, moe_sort_tokens,
               moe_sort_tokens_capacity)


@dataclasses.dataclass
class SharedExpertWeights:
    """The layer's shared expert as a one-expert weight set in the boundary
    layout of the routed experts, run on every token with weight 1."""
    wg: torch.Tensor  # [1, I, H/2] uint8
    sg: torch.Tensor  # [1, I, H/32] uint8
    wu: torch.Tensor
    su: torch.Tensor
    wd: torch.Tensor  # [1, H, I/2] uint8
    sd: torch.Tensor  # [1, H, I/32] uint8


@dataclasses.dataclass
class LayerWeights:
    """Device weights of one layer in the boundary layout (see moe_mxfp4.h)."""
    wr: torch.Tensor            # [E, H] router, float32 or bfloat16
    bias: torch.Tensor | None   # [E] float32 logit bias or None
    wg: torch.Tensor            # [E, I, H/2] uint8
    sg: torch.Tensor            # [E, I, H/32] uint8
    wu: torch.Tensor
    su: torch.Tensor
    wd: torch.Tensor            # [E, H, I/2] uint8
    sd: torch.Tensor            # [E, H, I/32] uint8
    k: int
    shared: SharedExpertWeights | None = None

    @property
    def E(self):
        return self.wr.shape[0]

    @property
    def H(self):
        return self.wr.shape[1]

    @property
    def I(self):
        return self.wg.shape[1]

    @property
    def nbytes(self) -> int:
        ts = [self.wr, self.wg, self.sg, self.wu, self.su, self.wd, self.sd]
        if self.shared is not None:
            sh = self.shared
            ts += [sh.wg, sh.sg, sh.wu, sh.su, sh.wd, sh.sd]
        return sum(t.numel() * t.element_size() for t in ts)


class Workspace:
    """Every intermediate of one forward over T tokens (device tensors).

    ``pad`` adds that many extra columns to every 2-D buffer (rounded to keep
    16-byte row alignment), so the calls run on padded row strides.
    """

    def __init__(self, T: int, lw: LayerWeights, device, pad: int = 0, tile_rows: int = 1):
        H, E, k, I = lw.H, lw.E, lw.k, lw.I
        A = T * k
        p16 = (pad + 15) // 16 * 16

        def buf(rows, cols, dtype, align_cols=1):
            extra = p16 if pad else 0
            extra = (extra + align_cols - 1) // align_cols * align_cols
            full = torch.empty(rows, cols + extra, dtype=dtype, device=device)
            return full[:, :cols]

        self.T, self.A, self.tile_rows = T, A, tile_rows
        self.logits = torch.empty(T, E, dtype=torch.float32, device=device)  # [T][E], no row stride in the ABI
        self.ids = torch.empty(T, k, dtype=torch.int32, device=device)
        self.w = torch.empty(T, k, dtype=torch.float32, device=device)
        self.offsets = torch.empty(E + 1, dtype=torch.int32, device=device)
        cap = moe_sort_tokens_capacity(T, k, E, tile_rows)
        self.sorted = torch.empty(max(cap, 1), dtype=torch.int32, device=device)
        self.inv = torch.empty(max(A, 1), dtype=torch.int32, device=device)
        self.xq = buf(T, H, torch.int8, 16)
        self.xs = buf(T, H // 32, torch.float32)
        self.h = buf(A, I, torch.float32)
        self.hq = buf(A, I, torch.int8, 16)
        self.hs = buf(A, I // 32, torch.float32)
        self.y = buf(A, H, torch.float32)
        self.out = buf(T, H, torch.float32)
        # grid-barrier counters of the fused decode path (zero-filled once)
        nws = (moe_decode_workspace_bytes() + 7) // 8
        self.decode_ws = torch.zeros(nws, dtype=torch.int64, device=device)
        if lw.shared is not None:
            # the shared expert's stages: one expert holding every token in order
            self.sh_offsets = torch.tensor([0, T], dtype=torch.int32, device=device)
            self.sh_sorted = torch.arange(max(T, 1), dtype=torch.int32, device=device)
            self.sh_h = buf(T, I, torch.float32)
            self.sh_hq = buf(T, I, torch.int8, 16)
            self.sh_hs = buf(T, I // 32, torch.float32)
            self.sh_y = buf(T, H, torch.float32)


class MoeLayer:
    def __init__(self, weights: LayerWeights, fused: bool | None = None):
        """fused: None = use the single-launch decode path when the batch
        allows it; True / False force it on / off."""
        self.lw = weights
        self.fused = fused

    def use_fused(self, T: int) -> bool:
        """The single-launch path takes batches up to moe_decode_max_tokens()
        (activation rows must fit its shared memory); larger ones use the
        stage calls."""
        if self.fused is False:
            return False
        self._limits()
        return 0 < T <= self._max_t

    def shared_in_one_launch(self, T: int) -> bool:
        """A layer with a shared expert runs it inside the single launch for
        batches up to moe_decode_max_tokens_shared(); between that and the
        routed limit the shared expert follows as stage calls."""
        return self.lw.shared is not None and self.use_fused(T) and T <= self._max_ts

    def _limits(self):
        if not hasattr(self, "_max_t"):
            lw = self.lw
            self._max_t = moe_decode_max_tokens(lw.H, lw.E, lw.k, lw.I)
            self._max_ts = 0 if lw.shared is None else moe_decode_max_tokens_shared(lw.H, lw.E, lw.k, lw.I)

    def forward(self, x: torch.Tensor, ws: Workspace, stream=None, events: dict | None = None) -> torch.Tensor:
        """out = MoE(x) for the T rows of x ([T, H] bf16/f32, unit column stride).

        ``events`` optionally maps a stage name ("decode" for the single launch,
        with the shared expert when it fits; "route", "sort", "quant_x",
        "gateup", "quant_h", "down", "combine" for the stage calls (below
        17 rows "down" is the fused down projection and combine);
        "shared_quant_x" (after the single launch only), "shared_gateup",
        "shared_quant_h", "shared_down", "join" for the shared expert's stage
        calls) to a (start, end) pair of torch.cuda.Event recorded around that
        stage on ``stream``."""
        lw = self.lw
        s = torch.cuda.current_stream() if stream is None else stream
        ev = events or {}

        def stage(name, fn, *args):
            if name in ev:
                ev[name][0].record(s)
            fn(*args, stream=s)
            if name in ev:
                ev[name][1].record(s)

        sh = lw.shared
        if self.use_fused(ws.T):
            # one launch: the routed layer, and the shared expert when it fits
            one = self.shared_in_one_launch(ws.T)
            if "decode" in ev:
                ev["decode"][0].record(s)
            if one:
                moe_decode_forward_shared(x, lw.wr, lw.bias, lw.wg, lw.sg, lw.wu, lw.su, lw.wd, lw.sd, sh, lw.k,
                                          ws.out, ws.logits, ws.ids, ws.w, ws.h, ws.y, ws.sh_h, ws.sh_y,
                                          ws.decode_ws, stream=s)
            else:
                moe_decode_forward(x, lw.wr, lw.bias, lw.wg, lw.sg, lw.wu, lw.su, lw.wd, lw.sd, lw.k, ws.out,
                                   ws.logits, ws.ids, ws.w, ws.h, ws.y, ws.decode_ws, stream=s)
            if "decode" in ev:
                ev["decode"][1].record(s)
            if one or sh is None:
                return ws.out
            stage("shared_quant_x", act_quant_q8, x, ws.xq, ws.xs)  # the single launch keeps Q8(x) on chip
        else:
            stage("route", moe_route_topk, x, lw.wr, lw.bias, lw.k, ws.logits, ws.ids, ws.w)
            stage("sort", moe_sort_tokens, ws.ids, lw.E, ws.tile_rows, ws.offsets, ws.sorted, ws.inv)
            stage("quant_x", act_quant_q8, x, ws.xq, ws.xs)
            stage("gateup", moe_mxfp4_gateup_swiglu, ws.xq, ws.xs, lw.wg, lw.sg, lw.wu, lw.su, ws.offsets, ws.sorted,
                  lw.k, ws.h)
            stage("quant_h", act_quant_q8, ws.h, ws.hq, ws.hs)
            if ws.T < 17:
                # down projection and combine in one launch (y kept as well)
                stage("down", moe_mxfp4_down_combine, ws.hq, ws.hs, lw.wd, lw.sd, ws.offsets, ws.sorted, ws.w, ws.T,
                      lw.k, ws.out, ws.y)
            else:
                stage("down", moe_mxfp4_down, ws.hq, ws.hs, lw.wd, lw.sd, ws.offsets, ws.sorted, ws.T, lw.k, ws.y)
                stage("combine", moe_combine, ws.y, ws.w, ws.out)
        if sh is not None:
            # the shared expert: the stage calls on its one-expert weight set
            # (every token, weight 1), then its join onto the routed output
            stage("shared_gateup", moe_mxfp4_gateup_swiglu, ws.xq, ws.xs, sh.wg, sh.sg, sh.wu, sh.su, ws.sh_offsets,
                  ws.sh_sorted, 1, ws.sh_h)
            stage("shared_quant_h", act_quant_q8, ws.sh_h, ws.sh_hq, ws.sh_hs)
            stage("shared_down", moe_mxfp4_down, ws.sh_hq, ws.sh_hs, sh.wd, sh.sd, ws.sh_offsets, ws.sh_sorted, ws.T,
                  1, ws.sh_y)
            stage("join", moe_join_add, ws.sh_y, ws.out)
        return ws.out

    def kernels_per_forward(self, T: int) -> int:
        """Launches of this library's kernels per forward."""
        if self.use_fused(T):
            if self.lw.shared is None or self.shared_in_one_launch(T):
                return 1
            return 1 + 5  # the shared expert's quant x, gate/up, quant h, down, join
        n = 8 if T >= 17 else 7  # logits, top-k, sort, quant x, gate/up, quant h, down (+ combine)
        lw = self.lw
        if T >= 17:  # tile policy: light experts on the CUDA-core kernel, the rest on the tensor-core kernel
            n += (lw.H % 256 == 0 and lw.I % 128 == 0) + (lw.I % 256 == 0 and lw.H % 128 == 0)
        if lw.shared is not None:
            n += 4  # the shared expert's gate/up, quant h, down, join
            if T >= 17:
                n += (lw.H % 256 == 0 and lw.I % 128 == 0) + (lw.I % 256 == 0 and lw.H % 128 == 0)
        return n
