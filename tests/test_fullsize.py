"""GPU parity at the workloads' full sizes, in the launch configuration of the
benchmark, checked against the fp64 oracle.

Tiles are independent (the method's abstract, sentence 4), so on the large
workloads the oracle recomputes a sample of tiles (or aligned regions that hold
whole tiles for every T used) from the same input values and compares them one
by one. Where the whole output is affordable on the host (the GPT-2-small set,
the 4096 x 4096 full-matrix map) it is compared in full.

Tolerances as in test_parity.py: relative Frobenius error <= 2e-2 against the
oracle for the bf16 tensor path, on the NS output and on the update W_new - W0;
momentum (one fp32 FMA) to 1e-6. The bf16 weights start at zero, so the stored
W_new = bf16(-lr s O) carries only bf16's own relative rounding (at most 2^-8
per element, its unit roundoff), and the update is checked at 2e-2 with no
allowance for the rounding of a non-zero W.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import tiled_newton_schulz_03_b300 as hm
from tiled_newton_schulz_03_b300 import synth

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2
QUINTIC = (3.4445, -4.7750, 2.0315)


def f64(t):
    return t.detach().float().cpu().double().numpy()


def rel_fro(got, want):
    return float(np.linalg.norm(np.asarray(got) - np.asarray(want)) / np.linalg.norm(want))


def step_region(W0, G, M0, T, K, lr, mu, s):
    """Oracle step on a region that is a union of whole tiles: momentum, tiled
    NS of the region (tile grid anchored at its corner), update with the
    matrix's own scale s."""
    M_new, U = oracle.momentum(M0, G, mu, True)
    O = oracle.tiled_ns(U, T, K)
    return W0 - lr * s * O, M_new


def check_update(W_gpu, W0, W_ref, tol=TOL_BF16):
    d_gpu, d_ref = W_gpu - W0, W_ref - W0
    assert np.linalg.norm(d_gpu - d_ref) <= tol * np.linalg.norm(d_ref)


def chunk_edge_tiles(shapes, T, per_tile_bytes, chunk_bytes):
    """(matrix, ti, tj) of the first and last tile of every launch of a step.

    The work list is every tile of every matrix in order (row-major within a
    matrix), cut into launches that each hold at most chunk_bytes of operand
    bytes. With all tiles full (T divides every side) each launch holds
    chunk_bytes // per_tile_bytes tiles."""
    per = chunk_bytes // per_tile_bytes
    starts, n = [], 0
    for i, (H, W) in enumerate(shapes):
        starts.append(n)
        n += (H // T) * (W // T)
    edges = set()
    for c0 in range(0, n, per):
        for t in (c0, min(n, c0 + per) - 1):
            i = max(k for k in range(len(shapes)) if starts[k] <= t)
            lt, tw = t - starts[i], shapes[i][1] // T
            edges.add((i, lt // tw, lt % tw))
    return sorted(edges), -(-n // per)


@pytest.fixture(scope="module", autouse=True)
def built():
    from tiled_newton_schulz_03_b300 import build
    build.build()
    hm.load_library()
    yield
    torch.cuda.synchronize()
    assert hm.device_error() == 0


def test_llama3_8b_step_full_size_sampled():
    """The benchmark's workload: 224 matrices (6.98 G parameters), bf16 G, fp32 M,
    bf16 W, T = 128, K = 5, Nesterov, chunks of <= 8 GB, one fused step. Checked
    tiles: the first and last tile of every launch (a chunk edge is where an
    off-by-one in the work split would land) and 2 random tiles of every matrix
    of 3 layers. M starts non-zero, so momentum and the Nesterov input matter."""
    dev = torch.device("cuda", 0)
    shapes = synth.llama3_8b_shapes()
    T, chunk = 128, 8 << 30
    Gs = [synth.lowrank_noise(H, W, seed=1000 + i, rank=16, device=dev) for i, (H, W) in enumerate(shapes)]
    Ws = [torch.zeros(H, W, dtype=torch.bfloat16, device=dev) for H, W in shapes]
    Ms = [synth.gaussian(H, W, seed=700000 + i, std=1e-3, device=dev) for i, (H, W) in enumerate(shapes)]
    # bf16 G + fp32 M + bf16 W per element of a 128 x 128 tile
    edges, nlaunch = chunk_edge_tiles(shapes, T, T * T * (2 + 4 + 2), chunk)
    assert nlaunch == 7
    rng = np.random.default_rng(7)
    picks = set(edges)
    for i, (H, W) in enumerate(shapes):
        if i // 7 in (0, 15, 31):
            for _ in range(2):
                picks.add((i, int(rng.integers(0, H // T)), int(rng.integers(0, W // T))))
    saved = []
    for i, ti, tj in sorted(picks):
        sl = (slice(T * ti, T * ti + T), slice(T * tj, T * tj + T))
        saved.append((i, sl, f64(Gs[i][sl]), f64(Ms[i][sl])))
    l0 = hm.default_handle().launch_count()
    hm.step(Ws, Gs, Ms, T, 5, lr=0.02, mu=0.95, nesterov=True, chunk_bytes=chunk)
    torch.cuda.synchronize()
    assert hm.default_handle().launch_count() - l0 == nlaunch
    for i, sl, G, M0 in saved:
        H, W = shapes[i]
        W_ref, M_ref = step_region(np.zeros_like(G), G, M0, T, 5, 0.02, 0.95, math.sqrt(max(1.0, H / W)))
        assert rel_fro(f64(Ms[i][sl]), M_ref) <= 1e-6
        check_update(f64(Ws[i][sl]), np.zeros_like(G), W_ref)
    del Gs, Ws, Ms
    torch.cuda.empty_cache()


def test_gpt2_small_three_steps_full_set():
    """12 layers x {4 x 768^2, 768 x 3072, 3072 x 768}, T = 128, K = 5, three
    successive fused steps with fresh gradients (seeds 1..3); layer 0 is tracked
    by the oracle through all three steps, every matrix after the first."""
    dev = torch.device("cuda", 0)
    shapes = synth.gpt2_small_shapes()
    Ws = [torch.zeros(H, W, dtype=torch.bfloat16, device=dev) for H, W in shapes]
    Ms = [torch.zeros(H, W, device=dev) for H, W in shapes]
    Wr = [f64(w) for w in Ws[:6]]
    Winit = [w.copy() for w in Wr]
    Mr = [np.zeros(s) for s in shapes[:6]]
    for step in range(3):
        Gs = [synth.lowrank_noise(H, W, seed=1 + step + 100 * i, rank=8, device=dev) for i, (H, W) in enumerate(shapes)]
        if step == 0:
            W0 = [f64(w) for w in Ws]
            G0 = [f64(g) for g in Gs]
        hm.step(Ws, Gs, Ms, 128, 5, lr=0.02, mu=0.95, nesterov=True)
        for i in range(6):
            H, W = shapes[i]
            Wr[i], Mr[i] = step_region(Wr[i], f64(Gs[i]), Mr[i], 128, 5, 0.02, 0.95,
                                       math.sqrt(max(1.0, H / W)))
        if step == 0:
            torch.cuda.synchronize()
            for i, (H, W) in enumerate(shapes):
                W_ref, _ = step_region(W0[i], G0[i], np.zeros((H, W)), 128, 5, 0.02, 0.95,
                                       math.sqrt(max(1.0, H / W)))
                check_update(f64(Ws[i]), W0[i], W_ref)
    torch.cuda.synchronize()
    for i in range(6):
        check_update(f64(Ws[i]), Winit[i], Wr[i])          # three steps' total update
        assert rel_fro(f64(Ms[i]), Mr[i]) <= 1e-5


@pytest.mark.parametrize("T", [32, 64, 128, 256])
def test_sweep_4096_tiled_sampled(T):
    """One 4096 x 4096 bf16 matrix (rank 8 + noise), K = 5: 8 sampled tiles."""
    G = synth.lowrank_noise(4096, 4096, seed=3, rank=8, device="cuda")
    out = hm.tiled_ns(G, T, 5, path="tensor", out_dtype=torch.float32)
    n = 4096 // T
    rng = np.random.default_rng(T)
    for ti, tj in rng.integers(0, n, size=(8, 2)):
        sl = (slice(T * ti, T * ti + T), slice(T * tj, T * tj + T))
        assert rel_fro(f64(out[sl]), oracle.tiled_ns(f64(G[sl]), T, 5)) <= TOL_BF16


def test_sweep_4096_full_matrix():
    """T = 4096 on the 4096 x 4096 matrix: the full-matrix map, checked whole."""
    G = synth.lowrank_noise(4096, 4096, seed=3, rank=8, device="cuda")
    out = hm.tiled_ns(G, 4096, 5, path="tensor", out_dtype=torch.float32)
    want = oracle.full_ns(f64(G), 5)
    assert rel_fro(f64(out), want) <= TOL_BF16


@pytest.mark.parametrize("K", [3, 5])
def test_ragged_shapes_tile_schedule(K):
    """1000 x 3000, 5120 x 13824, 2048 x 50257 bf16 (rank 8 + noise), three fused
    steps with T = 64, 128, 256. Regions of 256 x 256 (whole tiles for every T)
    at the matrices' corners and ragged edges are tracked by the oracle; the
    2048 x 50257 matrix has rows that are not 16-byte aligned."""
    dev = torch.device("cuda", 0)
    shapes = [(1000, 3000), (5120, 13824), (2048, 50257)]
    Ws = [torch.zeros(H, W, dtype=torch.bfloat16, device=dev) for H, W in shapes]
    Ms = [torch.zeros(H, W, device=dev) for H, W in shapes]
    regions = []
    for i, (H, W) in enumerate(shapes):
        for r0, c0 in ((0, 0), ((H - 1) // 256 * 256, (W - 1) // 256 * 256), (256, (W - 1) // 256 * 256)):
            sl = (slice(r0, min(H, r0 + 256)), slice(c0, min(W, c0 + 256)))
            w0 = f64(Ws[i][sl])
            regions.append([i, sl, w0, np.zeros((sl[0].stop - r0, sl[1].stop - c0)), w0.copy()])
    sched = hm.TSchedule([(0, 64), (1, 128), (2, 256)])
    for step in range(3):
        T = sched(step)
        Gs = [synth.lowrank_noise(H, W, seed=300 + 10 * step + i, rank=8, device=dev) for i, (H, W) in enumerate(shapes)]
        for reg in regions:
            i, sl = reg[0], reg[1]
            H, W = shapes[i]
            reg[2], reg[3] = step_region(reg[2], f64(Gs[i][sl]), reg[3], T, K, 0.02, 0.95,
                                         math.sqrt(max(1.0, H / W)))
        hm.step(Ws, Gs, Ms, T, K, lr=0.02, mu=0.95, nesterov=True)
    torch.cuda.synchronize()
    for i, sl, W_ref, M_ref, W_init in regions:
        assert rel_fro(f64(Ms[i][sl]), M_ref) <= 1e-5
        check_update(f64(Ws[i][sl]), W_init, W_ref)         # three steps' total update


@pytest.mark.parametrize("T", [64, 128, 256])
def test_unaligned_rows_bit_identical_to_aligned_full_size(T):
    """The ragged set's 2048 x 50257 matrix, two fused steps, stored once with its
    own leading dimension (rows not 16-byte aligned: loaded and converted row by
    row) and once inside a 2048 x 50264 buffer (16-byte aligned rows: TMA-staged,
    or 16-byte row loads at T = 256). Both do the same arithmetic in the same
    order, so every element of W and M must agree bit for bit: a stage that
    reached its slot before it was complete, or a row taken from the wrong
    place, would not."""
    dev = torch.device("cuda", 0)
    H, W = 2048, 50257
    G0 = synth.lowrank_noise(H, W, seed=61, rank=8, device=dev)
    W0 = synth.gaussian(H, W, seed=62, std=0.02, dtype=torch.bfloat16, device=dev)
    M0 = synth.gaussian(H, W, seed=63, std=1e-3, device=dev)
    res = []
    for ld in (W, 50264):
        def place(x):
            buf = torch.zeros(H, ld, dtype=x.dtype, device=dev)
            v = buf[:, :W]
            v.copy_(x)
            return v
        G, Wt, M = place(G0), place(W0), place(M0)
        for _ in range(2):
            hm.step([Wt], [G], [M], T, 5, lr=0.02, mu=0.95, nesterov=True)
        torch.cuda.synchronize()
        res.append((Wt.clone(), M.clone()))
    assert torch.equal(res[0][0], res[1][0])
    assert torch.equal(res[0][1], res[1][1])
