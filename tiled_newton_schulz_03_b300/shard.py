"""HiMuon step sharded over the ranks of a data-parallel job.

Tiles, and so whole matrices, are independent ("Hierarchical Muon: Tiled
Newton-Schulz Updates for Efficient Muon Optimization", abstract, sentences
3-4), so in data-parallel training, where every rank holds the same gradients
after their all-reduce, the matrices can be split across ranks: each rank runs
the fused step (``himuon_step``) on the matrices it owns, and the new weights
then go from each owner to every rank. Only the owner keeps a matrix's
momentum buffer. The exchange is the one collective of the path: one
broadcast per matrix from its owner (``torch.distributed``; NCCL on GPUs, gloo
on CPU).

The assignment balances the NS work 6 H W min(T, max(H, W)) K across ranks
(longest first onto the least loaded rank, ties to the lower rank), so it is
the same on every rank without communication.
"""

from __future__ import annotations

import torch

__all__ = ["assign", "ShardedStep"]


def assign(shapes, world: int, T: int, K: int = 5):
    """Owner rank of each (H, W) matrix: greedy balance of the NS flops."""
    if world < 1:
        raise ValueError("world must be >= 1")
    work = [6.0 * H * W * min(T, max(H, W)) * max(K, 1) for H, W in shapes]
    order = sorted(range(len(shapes)), key=lambda i: (-work[i], i))
    load = [0.0] * world
    owner = [0] * len(shapes)
    for i in order:
        r = min(range(world), key=lambda q: (load[q], q))
        owner[i] = r
        load[r] += work[i]
    return owner


class ShardedStep:
    """A HiMuon step split across the ranks of ``group``.

    ``step_fn(Ws, Gs, Ms)`` runs the fused step on the given lists (normally
    ``functools.partial(tiled_newton_schulz_03_b300.step, T=..., K=..., ...)``);
    it is called once per step with this rank's matrices only. ``Ms`` holds the
    momentum buffers of the owned matrices (None elsewhere).
    """

    def __init__(self, shapes, T: int, K: int, step_fn, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.rank = dist.get_rank(group) if dist.is_initialized() else 0
        self.world = dist.get_world_size(group) if dist.is_initialized() else 1
        self.owner = assign(shapes, self.world, T, K)
        self.step_fn = step_fn

    def mine(self):
        return [i for i, r in enumerate(self.owner) if r == self.rank]

    @torch.no_grad()
    def __call__(self, Ws, Gs, Ms):
        idx = self.mine()
        if idx:
            self.step_fn([Ws[i] for i in idx], [Gs[i] for i in idx], [Ms[i] for i in idx])
        if self.world > 1:
            for i, W in enumerate(Ws):
                src = self.dist.get_global_rank(self.group, self.owner[i]) if self.group is not None \
                    else self.owner[i]
                self.dist.broadcast(W, src=src, group=self.group)
        return Ws
