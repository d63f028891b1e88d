"""``torch.optim.Optimizer`` front end of the fused HiMuon step.

HiMuon ("Hierarchical Muon: Tiled Newton-Schulz Updates for Efficient Muon
Optimization", abstract) turns each 2-D weight's momentum-gradient matrix into
an update direction with the tiled Newton-Schulz map. This class keeps the
momentum buffers and the step counter, and per parameter group issues ONE
``himuon_step`` call over all of the group's matrices (cross-layer batching,
memory-bounded chunks, the tile size of the current step from a runtime
schedule: abstract, sentence 6). All arithmetic runs in libhimuon's kernels;
this module only collects tensors and arguments.

Only 2-D parameters are accepted: biases, norms and embeddings (or anything
else the method does not apply to) stay with another optimizer of the
caller's choice, e.g. ``torch.optim.AdamW`` on the remaining parameters.
"""

from __future__ import annotations

import torch

from . import QUINTIC, HimuonError, TSchedule, step as _himuon_step

__all__ = ["HiMuon"]


class HiMuon(torch.optim.Optimizer):
    """HiMuon over 2-D CUDA parameters (bf16 or fp32, row-major).

    Arguments (per parameter group):
      lr, momentum (mu), nesterov, weight_decay (decoupled), scale_mode
        ("sqrt_aspect": s = sqrt(max(1, H / W)); "none"),
      T: tile size, an int or a schedule ``[(start_step, T), ...]`` /
        ``TSchedule`` evaluated at the optimizer's step count,
      K: NS steps; coeffs: one (a, b, c) triple or K per-step triples;
      norm ("tile", "matrix", "none"), eps, path ("auto", "tensor", "fp32"),
      chunk_bytes: memory bound of one launch (0: unbounded),
      momentum_dtype: dtype of the momentum buffers (float32 or bfloat16).
    Gradients must have the parameter's shape, be row-major and live on the
    parameter's device. Parameters without a gradient are skipped that step.
    """

    def __init__(self, params, lr: float = 0.02, momentum: float = 0.95, nesterov: bool = True,
                 weight_decay: float = 0.0, T=128, K: int = 5, coeffs=QUINTIC,
                 norm: str = "tile", eps: float = 1e-7, scale_mode: str = "sqrt_aspect",
                 path: str = "auto", chunk_bytes: int = 0, momentum_dtype=torch.float32):
        if lr < 0 or momentum < 0 or weight_decay < 0:
            raise ValueError("lr, momentum and weight_decay must be >= 0")
        if momentum_dtype not in (torch.float32, torch.bfloat16):
            raise ValueError("momentum_dtype must be torch.float32 or torch.bfloat16")
        defaults = dict(lr=lr, momentum=momentum, nesterov=nesterov, weight_decay=weight_decay,
                        T=T, K=K, coeffs=coeffs, norm=norm, eps=eps, scale_mode=scale_mode,
                        path=path, chunk_bytes=chunk_bytes, momentum_dtype=momentum_dtype)
        super().__init__(params, defaults)
        for group in self.param_groups:
            for p in group["params"]:
                if p.dim() != 2:
                    raise ValueError(
                        f"HiMuon takes 2-D weight matrices only; got a parameter of shape "
                        f"{tuple(p.shape)}: give it to another optimizer")
                if p.dtype not in (torch.float32, torch.bfloat16):
                    raise ValueError("HiMuon parameters must be float32 or bfloat16")
            group.setdefault("step_count", 0)   # kept in the group: saved by state_dict()
            self.tile_size(group)                # validates the schedule

    @staticmethod
    def tile_size(group) -> int:
        """The tile size this group uses at its current step (runtime schedule)."""
        T = group["T"]
        if isinstance(T, int):
            return T
        sched = T if isinstance(T, TSchedule) else TSchedule(T)
        return sched(group["step_count"])

    @torch.no_grad()
    def step(self, closure=None):
        loss = None
        if closure is not None:
            with torch.enable_grad():
                loss = closure()
        for group in self.param_groups:
            Ws, Gs, Ms = [], [], []
            for p in group["params"]:
                if p.grad is None:
                    continue
                if p.grad.is_sparse:
                    raise HimuonError(1, "sparse gradients are not supported")
                state = self.state[p]
                if "momentum_buffer" not in state:
                    state["momentum_buffer"] = torch.zeros_like(p, dtype=group["momentum_dtype"],
                                                                memory_format=torch.contiguous_format)
                Ws.append(p)
                Gs.append(p.grad)
                Ms.append(state["momentum_buffer"])
            if not Ws:
                continue
            devices = {w.device for w in Ws}
            if len(devices) != 1:
                raise HimuonError(1, "all parameters of a group must be on one device")
            _himuon_step(Ws, Gs, Ms, self.tile_size(group), group["K"], lr=group["lr"],
                         mu=group["momentum"], nesterov=group["nesterov"],
                         weight_decay=group["weight_decay"], scale_mode=group["scale_mode"],
                         coeffs=group["coeffs"], norm=group["norm"], eps=group["eps"],
                         path=group["path"], chunk_bytes=group["chunk_bytes"])
        for group in self.param_groups:
            group["step_count"] += 1
        return loss
