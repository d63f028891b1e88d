"""Seeded synthetic inputs shaped like the momentum-gradient matrices of the workloads.

This module holds no arithmetic of the method: it only draws random matrices.
Both the CUDA path and the fp64 oracle consume what it returns, so the two see
the same bytes.

Recipes (every draw is seeded; seed = base + matrix index):

* ``gaussian``: i.i.d. N(0, std^2) entries.
* ``lowrank_noise``: ``scale / sqrt(r) * P @ Q^T + noise_std * N`` with P (H x r),
  Q (W x r) and N (H x W) i.i.d. N(0, 1), so the low-rank part has entry
  standard deviation ``scale``; defaults r = 8, scale = 1e-2, noise_std = 1e-3.
* Weights: N(0, 0.02^2); momentum starts at zero.

Generation runs on the device the caller names (CPU for small parity cases, the
GPU for the multi-GB layer sets), with a ``torch.Generator`` seeded per matrix.
"""

from __future__ import annotations

import torch

# Matrix shapes, (H, W) = (out_features, in_features) as in torch.nn.Linear.
GPT2_SMALL_LAYER = [(768, 768)] * 4 + [(3072, 768), (768, 3072)]
LLAMA3_8B_LAYER = [(4096, 4096), (4096, 4096), (1024, 4096), (1024, 4096),
                   (14336, 4096), (14336, 4096), (4096, 14336)]
RAGGED_SET = [(1000, 3000), (5120, 13824), (2048, 50257)]


def gpt2_small_shapes(layers: int = 12):
    """GPT-2-small 2-D weights: 4 attention 768x768 + MLP 3072x768 and 768x3072."""
    return [s for _ in range(layers) for s in GPT2_SMALL_LAYER]


def llama3_8b_shapes(layers: int = 32):
    """Llama-3-8B 2-D weights: Q, O 4096^2; K, V 1024x4096 (GQA); gate, up
    14336x4096; down 4096x14336."""
    return [s for _ in range(layers) for s in LLAMA3_8B_LAYER]


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def gaussian(H: int, W: int, seed: int, std: float = 1.0, dtype=torch.float32,
             device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    x = torch.randn((H, W), generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def lowrank_noise(H: int, W: int, seed: int, rank: int = 8, scale: float = 1e-2,
                  noise_std: float = 1e-3, dtype=torch.bfloat16,
                  device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    P = torch.randn((H, rank), generator=g, device=device, dtype=torch.float32)
    Q = torch.randn((W, rank), generator=g, device=device, dtype=torch.float32)
    N = torch.randn((H, W), generator=g, device=device, dtype=torch.float32)
    out = torch.addmm(N.mul_(noise_std), P, Q.t(), alpha=scale / rank ** 0.5)
    return out.to(dtype)


def gradient_set(shapes, seed: int, rank: int = 8, dtype=torch.bfloat16,
                 device="cpu", out=None):
    """One low-rank-plus-noise gradient per shape; matrix i uses seed + i.

    ``out`` (a list of preallocated tensors) is filled in place when given.
    """
    res = []
    for i, (H, W) in enumerate(shapes):
        t = lowrank_noise(H, W, seed + i, rank=rank, dtype=dtype, device=device)
        if out is not None:
            out[i].copy_(t)
            t = out[i]
        res.append(t)
    return res


def weight_set(shapes, seed: int, dtype=torch.bfloat16, device="cpu"):
    return [gaussian(H, W, seed + i, std=0.02, dtype=dtype, device=device)
            for i, (H, W) in enumerate(shapes)]
