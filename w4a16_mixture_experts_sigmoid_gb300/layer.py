"""One routed-expert W4A16 MoE layer resident on the GPU.

Holds the layer's device weights and a workspace; every call goes through
the C ABI (moe_forward / moe_forward_host). PyTorch only provides device
memory and the stream.
"""
from __future__ import annotations

import torch

from . import binding as B


class MoeW4A16Layer:
    def __init__(self, E: int, top_k: int, H: int, I: int, w13, s13, w2, s2, shared_wgu=None, shared_wd=None,
                 device="cuda"):
        def dev(a, dtype):
            if a is None:
                return None
            t = torch.as_tensor(a) if not isinstance(a, torch.Tensor) else a
            return t.to(device=device, dtype=dtype).contiguous()

        self.E, self.top_k, self.H, self.I = E, top_k, H, I
        self.w13 = dev(w13, torch.int32)
        self.s13 = dev(s13, torch.int16)   # bf16 bit patterns
        self.w2 = dev(w2, torch.int32)
        self.s2 = dev(s2, torch.int16)
        self.sh_gu = dev(shared_wgu, torch.int16)
        self.sh_d = dev(shared_wd, torch.int16)
        self.dims = B.dims(E, top_k, H, I)
        self.weights = B.weights(self.w13, self.s13, self.w2, self.s2, self.sh_gu, self.sh_d)
        self.shared_I = 0 if self.sh_d is None else int(self.sh_d.shape[1])
        self._ws = None
        self._ws_T = -1
        self.device = device

    @classmethod
    def from_arrays(cls, shape, arrays: dict, device="cuda"):
        import numpy as np

        def t(key):
            a = arrays.get(key)
            if a is None:
                return None
            a = np.ascontiguousarray(a)
            if a.dtype == np.uint16:
                a = a.view(np.int16)
            return torch.from_numpy(a)

        return cls(shape.E, shape.top_k, shape.H, shape.I, t("w13"), t("s13"), t("w2"), t("s2"), t("sh_gu"),
                   t("sh_d"), device=device)

    def workspace(self, T: int, host_staging: bool = False) -> torch.Tensor:
        need = B.moe_workspace_size(self.dims, T, self.shared_I)
        if host_staging:
            need += B.moe_host_staging_size(self.dims, T)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.zeros(need, dtype=torch.uint8, device=self.device)
        return self._ws

    def forward(self, x: torch.Tensor, logits: torch.Tensor, out: torch.Tensor | None = None, flags: int = 0,
                stream=None) -> torch.Tensor:
        T = int(x.shape[0])
        if out is None:
            out = torch.empty((T, self.H), dtype=torch.int16, device=self.device)
        ws = self.workspace(T)
        B.moe_forward(self.dims, self.weights, x, logits, T, out, ws, flags, stream)
        return out

    def forward_host(self, x_host, logits_host, out_host, flags: int = 0, stream=None):
        T = int(x_host.shape[0])
        ws = self.workspace(T, host_staging=True)
        B.moe_forward_host(self.dims, self.weights, x_host, logits_host, T, out_host, ws, flags, stream)
        return out_host

    def check_status(self, stream=None) -> int:
        return 0 if self._ws is None else B.moe_check_status(self._ws, stream)


class MoeW4A16Stack:
    """Layers chained as pre-norm residual blocks, x <- x + MoE_l(RMSNorm(x)), in one C call
    (moe_stack_forward). Every layer's weights stay resident; the router logits of each layer
    are inputs."""

    def __init__(self, layers: list, eps: float = 1e-6):
        if not layers:
            raise ValueError("a stack needs at least one layer")
        first = layers[0]
        for lay in layers:
            if (lay.E, lay.top_k, lay.H, lay.I, lay.shared_I) != (first.E, first.top_k, first.H, first.I,
                                                                   first.shared_I):
                raise ValueError("all layers of a stack must have the same shape")
        self.layers = layers
        self.eps = float(eps)
        self.dims = first.dims
        self.H = first.H
        self.shared_I = first.shared_I
        self.device = first.device
        self._ws = None

    def workspace(self, T: int) -> torch.Tensor:
        need = B.moe_stack_workspace_size(self.dims, T, self.shared_I)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.zeros(need, dtype=torch.uint8, device=self.device)
        return self._ws

    def forward(self, x: torch.Tensor, logits: list, out: torch.Tensor | None = None, flags: int = 0,
                stream=None) -> torch.Tensor:
        T = int(x.shape[0])
        if out is None:
            out = torch.empty((T, self.H), dtype=torch.int16, device=self.device)
        B.moe_stack_forward(self.dims, [lay.weights for lay in self.layers], logits, x, T, self.eps, out,
                            self.workspace(T), flags, stream)
        return out

    def check_status(self, stream=None) -> int:
        return 0 if self._ws is None else B.moe_check_status(self._ws, stream)


class MoeFp4Layer:
    """One routed-expert layer with 4-bit float weights (E2M1 codes, an E4M3 scale per 16 inputs,
    an fp32 scale per matrix and expert; optional bf16 shared expert), resident on the GPU; every
    call goes through the C ABI (moe_forward_fp4)."""

    def __init__(self, E: int, top_k: int, H: int, I: int, w13, s13, g13, w2, s2, g2, shared_wgu=None,
                 shared_wd=None, device="cuda"):
        def dev(a, dtype):
            if a is None:
                return None
            t = torch.as_tensor(a) if not isinstance(a, torch.Tensor) else a
            return t.to(device=device, dtype=dtype).contiguous()

        self.E, self.top_k, self.H, self.I = E, top_k, H, I
        self.w13, self.s13, self.g13 = dev(w13, torch.int32), dev(s13, torch.uint8), dev(g13, torch.float32)
        self.w2, self.s2, self.g2 = dev(w2, torch.int32), dev(s2, torch.uint8), dev(g2, torch.float32)
        self.sh_gu = dev(shared_wgu, torch.int16)
        self.sh_d = dev(shared_wd, torch.int16)
        self.dims = B.dims(E, top_k, H, I, group=16)
        self.weights = B.weights_fp4(self.w13, self.s13, self.g13, self.w2, self.s2, self.g2, self.sh_gu, self.sh_d)
        self.shared_I = 0 if self.sh_d is None else int(self.sh_d.shape[1])
        self._ws = None
        self.device = device

    @classmethod
    def from_arrays(cls, shape, arrays: dict, device="cuda"):
        import numpy as np

        def t(key):
            a = arrays.get(key)
            if a is None:
                return None
            a = np.ascontiguousarray(a)
            if a.dtype == np.uint16:
                a = a.view(np.int16)
            return torch.from_numpy(a)

        return cls(shape.E, shape.top_k, shape.H, shape.I, t("w13"), t("s13"), t("g13"), t("w2"), t("s2"), t("g2"),
                   t("sh_gu"), t("sh_d"), device=device)

    def workspace(self, T: int) -> torch.Tensor:
        need = B.moe_workspace_size(self.dims, T, self.shared_I)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.zeros(need, dtype=torch.uint8, device=self.device)
        return self._ws

    def forward(self, x: torch.Tensor, logits: torch.Tensor, out: torch.Tensor | None = None, flags: int = 0,
                stream=None) -> torch.Tensor:
        T = int(x.shape[0])
        if out is None:
            out = torch.empty((T, self.H), dtype=torch.int16, device=self.device)
        B.moe_forward_fp4(self.dims, self.weights, x, logits, T, out, self.workspace(T), flags, stream)
        return out

    def check_status(self, stream=None) -> int:
        return 0 if self._ws is None else B.moe_check_status(self._ws, stream)
