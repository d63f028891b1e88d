"""fp64 CPU oracle of the HiMuon tiled Newton-Schulz map and of one HiMuon step.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this module. The product path (the CUDA
library and its Python binding) never imports, links or calls it, and it shares
no code with that path.

Source: "Hierarchical Muon: Tiled Newton-Schulz Updates for Efficient Muon
Optimization" (abstract). What the abstract fixes:

* Muon-type optimizers build an update direction for a dense weight by applying a
  finite Newton-Schulz (NS) map to the momentum-gradient matrix (abstract,
  sentence 1).
* HiMuon cuts each H x W momentum-gradient matrix into T x T tiles, applies the
  same finite NS map to every tile on its own, and puts the results back in place
  (abstract, sentence 3).
* For T below the matrix sizes this is a local map: interactions inside a tile
  are kept, those across tile borders are dropped (abstract, sentence 4).
* The leading NS work is O(H W T K) for fixed T (abstract, sentence 5).

What the abstract leaves open, and the reading taken here (each one is also a
parameter):

* NS step: A = X X^T, B = b A + c A^2, X <- a X + B X, repeated K times, with the
  quintic coefficients (a, b, c) = (3.4445, -4.7750, 2.0315) as default. The
  coefficients may also change from step to step (a per-step schedule of K
  triples); a triple with c = 0 is a cubic step.
* Normalisation before the first step: X <- X / (||X||_F + eps), eps = 1e-7, per
  tile by default ("tile"); "matrix" uses the norm of the whole matrix for every
  tile of it; "none" skips it.
* Edge tiles: where T does not divide H or W the last tiles are smaller
  rectangles h x w, h = min(T, H - iT), w = min(T, W - jT).
* Tall tiles (h > w) still use the h x h Gram X X^T here.
* Momentum: M <- mu M + G; the NS input is U = G + mu M (Nesterov) or U = M.
* Update: W <- W - lr * wd * W - lr * s * O with O the tiled NS output and
  s = sqrt(max(1, H / W)) ("sqrt_aspect") or s = 1 ("none").

Everything is computed in float64 from the exact values of the inputs it is
given (bf16 or fp32 inputs convert to float64 without rounding).

Pinned by tests/test_oracle.py: SVD closed form, diagonal and rotated tiles,
full-matrix equivalence at T >= max(H, W), tile independence, the classical
polar limit, the work count, identity and zero-padding cases, step identities.
"""

from __future__ import annotations

import math

import numpy as np

QUINTIC = (3.4445, -4.7750, 2.0315)
DEFAULT_EPS = 1e-7
NORM_MODES = ("tile", "matrix", "none")
SCALE_MODES = ("sqrt_aspect", "none")


def tile_grid(H: int, W: int, T: int):
    """Tiles of an H x W matrix cut at multiples of T (abstract, sentence 3).

    Yields (i0, j0, h, w) in row-major tile order; edge tiles are the smaller
    rectangles left over where T does not divide H or W.
    """
    if H < 0 or W < 0 or T < 1:
        raise ValueError("need H, W >= 0 and T >= 1")
    for i0 in range(0, H, T):
        for j0 in range(0, W, T):
            yield i0, j0, min(T, H - i0), min(T, W - j0)


def num_tiles(H: int, W: int, T: int) -> int:
    return (-(-H // T)) * (-(-W // T))


def frobenius_normalise(X: np.ndarray, eps: float) -> np.ndarray:
    """X / (||X||_F + eps) over the last two axes."""
    n = np.sqrt(np.sum(X * X, axis=(-2, -1), keepdims=True))
    return X / (n + eps)


def step_coefficients(coeffs, K: int):
    """The (a, b, c) of each of the K steps.

    ``coeffs`` is one triple (the same map at every step) or a sequence of K
    triples (a per-step schedule: step k uses the k-th triple).
    """
    items = list(coeffs)
    if len(items) == 3 and all(np.ndim(v) == 0 for v in items):
        return [tuple(float(v) for v in items)] * K
    if len(items) != K or any(len(t) != 3 for t in items):
        raise ValueError(f"coeffs: one (a, b, c) triple or exactly K = {K} triples")
    return [tuple(float(v) for v in t) for t in items]


def ns_steps(X: np.ndarray, K: int, coeffs=QUINTIC) -> np.ndarray:
    """K steps of the finite NS map on an already normalised X.

    Step k forms the Gram matrix A = X X^T, the polynomial B = b_k A + c_k A^2
    and the new iterate a_k X + B X, with (a_k, b_k, c_k) from
    ``step_coefficients``. Works on one matrix (h, w) or a stack (n, h, w).
    """
    X = np.asarray(X, dtype=np.float64)
    for a, b, c in step_coefficients(coeffs, K):
        A = X @ np.swapaxes(X, -1, -2)
        B = b * A + c * (A @ A)
        X = a * X + B @ X
    return X


def ns_map(X: np.ndarray, K: int, coeffs=QUINTIC, norm: str = "tile",
           eps: float = DEFAULT_EPS, scale: float | None = None) -> np.ndarray:
    """Normalise one matrix (or a stack), then run K NS steps.

    ``scale`` overrides the normalising factor (used for the per-matrix mode, where
    the factor comes from the whole matrix rather than the tile).
    """
    X = np.asarray(X, dtype=np.float64)
    if scale is not None:
        X = X * scale
    elif norm == "tile":
        X = frobenius_normalise(X, eps)
    elif norm == "none":
        pass
    else:
        raise ValueError(f"ns_map: norm {norm!r} needs an explicit scale")
    return ns_steps(X, K, coeffs)


def tiled_ns(G: np.ndarray, T: int, K: int, coeffs=QUINTIC, norm: str = "tile",
             eps: float = DEFAULT_EPS) -> np.ndarray:
    """HiMuon tiled NS map of one H x W matrix (abstract, sentences 3-5).

    Every tile is normalised and iterated on its own; the outputs are written back
    at the tile's place. Tiles of the same shape are stacked so that numpy runs
    them as one batched product; each tile's arithmetic is unchanged by that.
    """
    if norm not in NORM_MODES:
        raise ValueError(f"unknown norm mode {norm!r}")
    G = np.asarray(G, dtype=np.float64)
    H, W = G.shape
    out = np.zeros((H, W), dtype=np.float64)
    if H == 0 or W == 0:
        return out
    scale = None
    if norm == "matrix":
        scale = 1.0 / (math.sqrt(float(np.sum(G * G))) + eps)
    by_shape: dict[tuple[int, int], list[tuple[int, int]]] = {}
    for i0, j0, h, w in tile_grid(H, W, T):
        by_shape.setdefault((h, w), []).append((i0, j0))
    for (h, w), places in by_shape.items():
        stack = np.stack([G[i0:i0 + h, j0:j0 + w] for i0, j0 in places])
        res = ns_map(stack, K, coeffs, norm, eps, scale)
        for (i0, j0), r in zip(places, res):
            out[i0:i0 + h, j0:j0 + w] = r
    return out


def tiled_ns_tiles(G: np.ndarray, T: int, K: int, tiles, coeffs=QUINTIC,
                   norm: str = "tile", eps: float = DEFAULT_EPS,
                   matrix_norm: float | None = None):
    """The tiled map evaluated on a chosen subset of tiles only.

    ``tiles`` is a list of (ti, tj) tile indices. Because tiles are independent
    (abstract, sentence 4) each output tile equals the one ``tiled_ns`` would give;
    this is how outputs of large matrices are checked a sample at a time. For the
    "matrix" norm mode the whole-matrix norm must be passed in (or is computed).
    Returns a list of (i0, j0, out_tile).
    """
    G = np.asarray(G)
    H, W = G.shape
    scale = None
    if norm == "matrix":
        if matrix_norm is None:
            g = np.asarray(G, dtype=np.float64)
            matrix_norm = math.sqrt(float(np.sum(g * g)))
        scale = 1.0 / (matrix_norm + eps)
    res = []
    for ti, tj in tiles:
        i0, j0 = ti * T, tj * T
        h, w = min(T, H - i0), min(T, W - j0)
        X = np.asarray(G[i0:i0 + h, j0:j0 + w], dtype=np.float64)
        res.append((i0, j0, ns_map(X, K, coeffs, norm, eps, scale)))
    return res


def full_ns(G: np.ndarray, K: int, coeffs=QUINTIC, norm: str = "tile",
            eps: float = DEFAULT_EPS) -> np.ndarray:
    """Full-matrix NS map of Muon (abstract, sentences 1-2): no tiling at all.

    Normalisation is over the whole matrix ("tile" and "matrix" coincide here).
    """
    G = np.asarray(G, dtype=np.float64)
    X = G if norm == "none" else frobenius_normalise(G, eps)
    return ns_steps(X, K, coeffs)


def momentum(M: np.ndarray, G: np.ndarray, mu: float, nesterov: bool = True):
    """Momentum-gradient of Muon: M <- mu M + G; U = G + mu M (Nesterov) or M."""
    M_new = mu * np.asarray(M, dtype=np.float64) + np.asarray(G, dtype=np.float64)
    U = np.asarray(G, dtype=np.float64) + mu * M_new if nesterov else M_new
    return M_new, U


def update_scale(H: int, W: int, mode: str = "sqrt_aspect") -> float:
    """Per-matrix update scale: sqrt(max(1, H / W)) or 1."""
    if mode == "sqrt_aspect":
        return math.sqrt(max(1.0, H / W))
    if mode == "none":
        return 1.0
    raise ValueError(f"unknown scale mode {mode!r}")


def himuon_step(Wt: np.ndarray, G: np.ndarray, M: np.ndarray, T: int, K: int,
                lr: float, mu: float, nesterov: bool = True,
                weight_decay: float = 0.0, scale_mode: str = "sqrt_aspect",
                coeffs=QUINTIC, norm: str = "tile", eps: float = DEFAULT_EPS):
    """One HiMuon optimizer step on one weight matrix.

    Momentum (M, U), the tiled NS map of U, then the scaled, decoupled update
    W <- W - lr * wd * W - lr * s * O. Returns (W_new, M_new, O) in float64.
    """
    Wt = np.asarray(Wt, dtype=np.float64)
    H, Wd = Wt.shape
    M_new, U = momentum(M, G, mu, nesterov)
    O = tiled_ns(U, T, K, coeffs, norm, eps)
    s = update_scale(H, Wd, scale_mode)
    W_new = Wt - lr * weight_decay * Wt - lr * s * O
    return W_new, M_new, O


def ns_mac_count(H: int, W: int, T: int, K: int) -> int:
    """Multiply-adds of the tiled map as this oracle forms it (X X^T form).

    Per step and h x w tile: X X^T costs h*h*w, A A costs h^3, B X costs h*h*w.
    For T dividing H and W this is 3 H W T K, i.e. O(H W T K) (abstract,
    sentence 5).
    """
    total = 0
    for _, _, h, w in tile_grid(H, W, T):
        total += 2 * h * h * w + h ** 3
    return K * total


def full_mac_count(H: int, W: int, K: int) -> int:
    """Multiply-adds of full-matrix NS in the min-side Gram form: O(r^2 s K)."""
    r, s = min(H, W), max(H, W)
    return K * (2 * r * r * s + r ** 3)


def quintic_scalar(sigma: float, K: int, coeffs=QUINTIC) -> float:
    """The scalar polynomials p_k(x) = a_k x + b_k x^3 + c_k x^5, k = 0..K-1,
    applied in turn."""
    x = float(sigma)
    for a, b, c in step_coefficients(coeffs, K):
        x = a * x + b * x ** 3 + c * x ** 5
    return x
