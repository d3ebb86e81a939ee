"""Device-side buffers for one MoE layer, and a call of moe_forward on them.

PyTorch provides the device memory and the stream; the arithmetic is all in
libmoe_b300.so.  Used by the tests, the benchmark and the smoke entry point.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

from . import moe
from .inputs import MoEInputs


def _bf16(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


def _u8(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


@dataclasses.dataclass
class DeviceMoE:
    """All arguments of moe_forward resident on one device."""

    T: int
    d: int
    W: int
    E: int
    k: int
    limit: float
    alpha: float
    x: torch.Tensor
    router_w: torch.Tensor
    router_b: torch.Tensor
    w_gu: torch.Tensor
    w_gu_scale: torch.Tensor
    b_gu: torch.Tensor
    w_dn: torch.Tensor
    w_dn_scale: torch.Tensor
    b_dn: torch.Tensor
    out: torch.Tensor
    workspace: torch.Tensor
    norm_w: torch.Tensor | None = None     # RMSNorm weight of the pre-norm block
    eps: float = 1e-5

    @classmethod
    def upload(cls, inp: MoEInputs, device="cuda") -> "DeviceMoE":
        wl = inp.wl
        ws_bytes = moe.moe_workspace_bytes(wl.T, wl.d, wl.W, wl.E, wl.k)
        return cls(
            T=wl.T, d=wl.d, W=wl.W, E=wl.E, k=wl.k, limit=inp.limit, alpha=inp.alpha,
            x=_bf16(inp.x, device),
            router_w=torch.from_numpy(inp.router_w).to(device),
            router_b=torch.from_numpy(inp.router_b).to(device),
            w_gu=_u8(inp.w_gu, device), w_gu_scale=_u8(inp.w_gu_scale, device),
            b_gu=_bf16(inp.b_gu, device),
            w_dn=_u8(inp.w_dn, device), w_dn_scale=_u8(inp.w_dn_scale, device),
            b_dn=_bf16(inp.b_dn, device),
            out=torch.empty((wl.T, wl.d), dtype=torch.bfloat16, device=device),
            workspace=torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=device),
            norm_w=None if inp.norm_w is None else torch.from_numpy(inp.norm_w).to(device),
            eps=inp.eps,
        )

    def forward(self, x=None, out=None, stream=None) -> torch.Tensor:
        """moe_forward, or moe_block_forward when the layer carries a norm weight."""
        x = self.x if x is None else x
        out = self.out if out is None else out
        if self.norm_w is not None:
            moe.moe_block_forward(x, self.T, self.d, self.W, self.norm_w, self.eps,
                                  self.router_w, self.router_b, self.w_gu, self.w_gu_scale,
                                  self.b_gu, self.w_dn, self.w_dn_scale, self.b_dn, self.E,
                                  self.k, self.limit, self.alpha, out, self.workspace,
                                  self.workspace.numel(), stream)
            return out
        moe.moe_forward(x, self.T, self.d, self.W, self.router_w, self.router_b,
                        self.w_gu, self.w_gu_scale, self.b_gu, self.w_dn, self.w_dn_scale,
                        self.b_dn, self.E, self.k, self.limit, self.alpha, out,
                        self.workspace, self.workspace.numel(), stream)
        return out

    def capture_graph(self) -> "torch.cuda.CUDAGraph":
        """A CUDA graph of one moe_forward on this layer's buffers: replaying it
        reads self.x and writes self.out with a single launch from the host.

        moe_forward neither synchronises nor allocates, so it can be captured;
        its kernels' programmatic launches become graph edges.  One eager call
        first sets the kernels' launch attributes outside the capture.
        """
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self.forward()
        torch.cuda.current_stream().wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            self.forward()
        return graph

    def route(self, stream=None):
        T, k, E = self.T, self.k, self.E
        dev = self.x.device
        idx = torch.empty((T, k), dtype=torch.int32, device=dev)
        w = torch.empty((T, k), dtype=torch.float32, device=dev)
        off = torch.empty(E + 1, dtype=torch.int32, device=dev)
        perm = torch.empty(T * k, dtype=torch.int32, device=dev)
        inv = torch.empty((T, k), dtype=torch.int32, device=dev)
        moe.moe_route(self.x, T, self.d, self.router_w, self.router_b, E, k, idx, w, off, perm,
                      inv, self.workspace, self.workspace.numel(), stream)
        return idx, w, off, perm, inv

    def hidden_format(self) -> tuple:
        """(format, exponent) of h on this shape and clamp (moe.HIDDEN_*)."""
        return moe.moe_hidden_format(self.T, self.d, self.W, self.E, self.k, self.limit)

    def hidden_dtype(self) -> torch.dtype:
        """The element type of the h_hi / h_lo tables on this shape and clamp."""
        fmt, _ = self.hidden_format()
        return {moe.HIDDEN_F16_PAIR: torch.float16, moe.HIDDEN_BF16_PAIR: torch.bfloat16,
                moe.HIDDEN_E4M3_TERMS: torch.float8_e4m3fn}[fmt]

    def hidden(self) -> torch.Tensor:
        """h of every permuted row as fp32 [T*k, W], rebuilt from its stored terms."""
        fmt, ex = self.hidden_format()
        R = self.T * self.k
        if fmt == moe.HIDDEN_E4M3_TERMS:
            off, _ = moe.moe_workspace_region(self.T, self.d, self.W, self.E, self.k, "h_hi")
            q = self.workspace[off:off + 4 * R * self.W].view(torch.float8_e4m3fn).view(4, R, self.W)
            h = torch.zeros((R, self.W), dtype=torch.float64, device=q.device)
            for t in range(4):
                h += q[t].double() / 16.0 ** t
            return (h * 2.0 ** ex).float()
        return self.region("h_hi").float() + self.region("h_lo").float()

    def region(self, which: str) -> torch.Tensor:
        """A view of an intermediate table inside the workspace (after forward)."""
        off, nb = moe.moe_workspace_region(self.T, self.d, self.W, self.E, self.k, which)
        raw = self.workspace[off:off + nb]
        R = self.T * self.k
        dtype, shape = {
            "topk_idx": (torch.int32, (self.T, self.k)), "topk_w": (torch.float32, (self.T, self.k)),
            "offsets": (torch.int32, (self.E + 1,)), "perm": (torch.int32, (R,)),
            "inv": (torch.int32, (self.T, self.k)), "x_perm": (torch.float16, (R, self.d)),
            "h_hi": (self.hidden_dtype(), (R, self.W)), "h_lo": (self.hidden_dtype(), (R, self.W)),
            # (in the E4M3 terms format the four tables start at h_hi; see hidden())
            "y": (torch.float32, (R, self.d)),
        }[which]
        return raw.view(dtype).view(shape)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)
