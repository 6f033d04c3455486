"""Device-resident block state: weights, fp32 gradients, workspace, two streams.

PyTorch only allocates memory and streams here; every operation of the block
runs in liboases.so through the C ABI.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

from . import (PARAM_NAMES, desc_from_shape, grads_struct, oases_block_fwd,
               oases_block_recompute_bwd, oases_stack_step, oases_workspace_bytes,
               weights_struct)

# storage type per block dtype (MX-FP8 blocks store bf16 and quantise per GEMM)
TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16, "mxfp8": torch.bfloat16}


class DeviceBlock:
    """One block / layer / stack of ``shape`` with the given per-layer parameters.

    layers: list (one entry per layer) of {name: array-like} in the C-ABI names.
    """

    def __init__(self, shape, layers: Sequence[Dict], recompute: str = "fine",
                 sub_batches: Optional[int] = None, device: str = "cuda:0",
                 streams: Optional[tuple] = None, reduce: str = "fused"):
        self.shape = shape
        self.device = torch.device(device)
        self.dtype = TORCH_DTYPE[shape.dtype]
        self.n_layers = len(layers)
        self.desc = desc_from_shape(shape, recompute, sub_batches, reduce)
        self.params: List[Dict[str, torch.Tensor]] = []
        self.grads: List[Dict[str, torch.Tensor]] = []
        for p in layers:
            self.params.append({k: torch.as_tensor(np.asarray(v, np.float32)).to(
                self.device, self.dtype).contiguous() for k, v in p.items()})
            self.grads.append({k: torch.zeros(np.shape(v), dtype=torch.float32, device=self.device)
                               for k, v in p.items()})
        self.wstructs = [weights_struct(p) for p in self.params]
        self.gstructs = [grads_struct(g) for g in self.grads]
        nbytes = oases_workspace_bytes(self.desc, self.n_layers)
        if nbytes == 0:
            raise ValueError("invalid block shape for the library: %r" % (shape,))
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        if streams is None:
            streams = (torch.cuda.Stream(self.device), torch.cuda.Stream(self.device))
        self.s0, self.s1 = streams

    # -- helpers --------------------------------------------------------------
    def tensor(self, a) -> torch.Tensor:
        return torch.as_tensor(np.asarray(a, np.float32)).to(self.device, self.dtype).contiguous()

    def empty_like_io(self) -> torch.Tensor:
        return torch.empty((self.shape.rows, self.shape.hidden), dtype=self.dtype,
                           device=self.device)

    def zero_grads(self) -> None:
        for g in self.grads:
            for t in g.values():
                t.zero_()

    def _enter(self):
        cur = torch.cuda.current_stream(self.device)
        self.s0.wait_stream(cur)

    def _leave(self):
        torch.cuda.current_stream(self.device).wait_stream(self.s0)

    # -- the three C entry points ----------------------------------------------
    def step(self, x: torch.Tensor, g: torch.Tensor, y: Optional[torch.Tensor] = None,
             dx: Optional[torch.Tensor] = None):
        """oases_stack_step: forward + recompute + backward; grads accumulate."""
        y = self.empty_like_io() if y is None else y
        dx = self.empty_like_io() if dx is None else dx
        self._enter()
        oases_stack_step(self.desc, self.wstructs, x, g, y, dx, self.gstructs, self.workspace,
                         s0=self.s0, s1=self.s1)
        self._leave()
        return y, dx

    def fwd(self, x: torch.Tensor, y: Optional[torch.Tensor] = None) -> torch.Tensor:
        assert self.n_layers == 1, "the block API takes one layer"
        y = self.empty_like_io() if y is None else y
        self._enter()
        oases_block_fwd(self.desc, self.wstructs[0], x, y, self.workspace, s0=self.s0, s1=self.s1)
        self._leave()
        return y

    def recompute_bwd(self, x: torch.Tensor, dy: torch.Tensor,
                      dx: Optional[torch.Tensor] = None) -> torch.Tensor:
        assert self.n_layers == 1, "the block API takes one layer"
        dx = self.empty_like_io() if dx is None else dx
        self._enter()
        oases_block_recompute_bwd(self.desc, self.wstructs[0], x, dy, dx, self.gstructs[0],
                                  self.workspace, s0=self.s0, s1=self.s1)
        self._leave()
        return dx

    def grads_numpy(self) -> List[Dict[str, np.ndarray]]:
        return [{k: v.double().cpu().numpy() for k, v in g.items()} for g in self.grads]


def to_numpy(t: torch.Tensor) -> np.ndarray:
    return t.detach().double().cpu().numpy()
