"""Tiled-versus-full matrix-function diagnostics of the HiMuon map.

HiMuon ("Hierarchical Muon: Tiled Newton-Schulz Updates for Efficient Muon
Optimization", abstract) replaces Muon's full-matrix Newton-Schulz map by the
same map on T x T tiles. The abstract mentions controlled matrix-function
diagnostics but defines no metric, so this tool reports, for each tile size T
on a synthetic gradient-shaped matrix G:

* ``rel_dist_full``: ||O_T - O_full||_F / ||O_full||_F, the distance of the
  tiled output from the full-matrix output (T >= max(H, W) gives exactly 0);
* ``cos_full``: <O_T, O_full> / (||O_T|| ||O_full||), the alignment of the two
  update directions;
* ``rel_dist_polar``: ||O_T - U V^T||_F / ||U V^T||_F, where G = U S V^T: how far
  each output is from the orthogonal polar factor that an exact
  orthogonalisation would give;
* the singular values of O_T (min, median, max, max/min of the nonzero ones and
  the fraction inside [0.5, 1.5]): the spectrum flattening the map achieves;
* ``flops_ratio``: the NS work of the tiled map relative to the full map
  (6 H W T K against K (4 r^2 s + 2 r^3), r = min(H, W), s = max(H, W));
* ``ms``: the time of the library call (CUDA events).

Every O_T comes from the library's public API (``tiled_ns``). The analysis
itself (singular values, polar factor) uses torch.linalg in float64; it is a
diagnostic, not part of the optimizer path.

Run: ``python -m tiled_newton_schulz_03_b300.diagnostics [--H 4096 --W 4096]``
(one JSON line per T).
"""

from __future__ import annotations

import argparse
import json

import torch

from . import QUINTIC, tiled_ns
from . import synth

__all__ = ["spectrum_stats", "polar_factor", "rel_dist", "cosine", "ns_work", "compare", "main"]


def rel_dist(X: torch.Tensor, Y: torch.Tensor) -> float:
    """||X - Y||_F / ||Y||_F in float64."""
    X, Y = X.double(), Y.double()
    return float(torch.linalg.norm(X - Y) / torch.linalg.norm(Y))


def cosine(X: torch.Tensor, Y: torch.Tensor) -> float:
    X, Y = X.double(), Y.double()
    return float((X * Y).sum() / (torch.linalg.norm(X) * torch.linalg.norm(Y)))


def polar_factor(G: torch.Tensor) -> torch.Tensor:
    """U V^T from the reduced SVD G = U S V^T (float64)."""
    U, _, Vh = torch.linalg.svd(G.double(), full_matrices=False)
    return U @ Vh


def spectrum_stats(O: torch.Tensor, tol: float = 1e-6) -> dict:
    """Summary of the singular values of O (float64); values below tol times
    the largest count as zero (rank deficiency, e.g. zero tiles)."""
    s = torch.linalg.svdvals(O.double())
    smax = float(s.max()) if s.numel() else 0.0
    nz = s[s > tol * max(smax, 1e-300)]
    return {"sv_min": float(s.min()), "sv_median": float(s.median()), "sv_max": smax,
            "sv_spread_nonzero": float(nz.max() / nz.min()) if nz.numel() else float("nan"),
            "sv_frac_in_0.5_1.5": float(((s >= 0.5) & (s <= 1.5)).double().mean()),
            "rank": int(nz.numel())}


def ns_work(H: int, W: int, T: int, K: int) -> float:
    """NS flops: 6 H W T K for tiles of T (T < max(H, W)), else the full map's
    K (4 r^2 s + 2 r^3) in the short-side Gram form."""
    r, s = min(H, W), max(H, W)
    if T >= s:
        return float(K * (4 * r * r * s + 2 * r ** 3))
    return 6.0 * H * W * T * K


def compare(G: torch.Tensor, Ts, K: int = 5, coeffs=QUINTIC, norm: str = "tile",
            path: str = "auto", reps: int = 3) -> list:
    """Diagnostics of the tiled map at every T in ``Ts`` against the full map."""
    H, W = G.shape
    full = tiled_ns(G, max(H, W), K, coeffs=coeffs, norm=norm, path=path, out_dtype=torch.float32)
    P = polar_factor(G)
    w_full = ns_work(H, W, max(H, W), K)
    rows = []
    for T in Ts:
        out = torch.empty(H, W, dtype=torch.float32, device=G.device)
        tiled_ns(G, T, K, coeffs=coeffs, norm=norm, path=path, out=out)      # warm-up
        times = []
        for _ in range(reps):
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            tiled_ns(G, T, K, coeffs=coeffs, norm=norm, path=path, out=out)
            e.record()
            torch.cuda.synchronize()
            times.append(s.elapsed_time(e))
        row = {"H": H, "W": W, "T": int(T), "K": K, "full": T >= max(H, W),
               "rel_dist_full": rel_dist(out, full), "cos_full": cosine(out, full),
               "rel_dist_polar": rel_dist(out, P),
               "flops_ratio": ns_work(H, W, T, K) / w_full, "ms": sorted(times)[len(times) // 2]}
        row.update(spectrum_stats(out))
        rows.append(row)
    return rows


def main(argv=None):
    ap = argparse.ArgumentParser(description="tiled-vs-full diagnostics of the HiMuon map")
    ap.add_argument("--H", type=int, default=4096)
    ap.add_argument("--W", type=int, default=4096)
    ap.add_argument("--rank", type=int, default=8, help="rank of the synthetic low-rank part")
    ap.add_argument("--seed", type=int, default=3)
    ap.add_argument("--K", type=int, default=5)
    ap.add_argument("--T", type=int, nargs="*", default=[32, 64, 128, 256, 512, 1024])
    ap.add_argument("--path", default="auto")
    args = ap.parse_args(argv)
    G = synth.lowrank_noise(args.H, args.W, seed=args.seed, rank=args.rank, device="cuda")
    Ts = sorted(set(args.T) | {max(args.H, args.W)})
    for row in compare(G, Ts, args.K, path=args.path):
        print(json.dumps({k: (round(v, 6) if isinstance(v, float) else v) for k, v in row.items()}))


if __name__ == "__main__":
    main()
