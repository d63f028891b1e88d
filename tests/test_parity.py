"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances (per matrix, relative Frobenius error against the oracle's fp64
result on the same input values): 2e-2 for the bf16 tensor-core path, 1e-5 for
the fp32 validation path. Indexing and reassembly are checked bit-exactly with
maps whose result is exactly representable (identity coefficients, K = 0 with
no normalisation), and tile independence by perturbing one tile.
"""

import numpy as np
import pytest
import torch

import oracle
import tiled_newton_schulz_03_b300 as hm
from tiled_newton_schulz_03_b300 import synth

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2
TOL_FP32 = 1e-5


def rel_fro(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    return float(np.linalg.norm(got - want) / np.linalg.norm(want))


def f64(t):
    return t.detach().float().cpu().double().numpy()


@pytest.fixture(scope="module", autouse=True)
def built():
    from tiled_newton_schulz_03_b300 import build
    build.build()
    hm.load_library()
    yield
    torch.cuda.synchronize()
    assert hm.device_error() == 0


# ---------------------------------------------------------------- one matrix

@pytest.mark.parametrize("T,path,tol", [(128, "tensor", TOL_BF16), (64, "tensor", TOL_BF16),
                                        (32, "tensor", TOL_BF16),
                                        (64, "fp32", TOL_FP32), (128, "fp32", TOL_FP32),
                                        (32, "fp32", TOL_FP32)])
def test_gaussian_fp32_256x512(T, path, tol):
    G = synth.gaussian(256, 512, seed=0)            # fp32, N(0, 1)
    out = hm.tiled_ns(G.cuda(), T, 5, path=path, out_dtype=torch.float32)
    want = oracle.tiled_ns(f64(G), T, 5)
    assert rel_fro(f64(out), want) <= tol


@pytest.mark.parametrize("H,W", [(300, 530), (128, 128), (1, 1), (1, 300), (257, 3),
                                 (129, 255), (768, 3072)])
@pytest.mark.parametrize("path", ["tensor", "fp32"])
@pytest.mark.parametrize("T", [128, 64, 32])
def test_lowrank_bf16_ragged(H, W, path, T):
    G = synth.lowrank_noise(H, W, seed=H * 7 + W)
    out = hm.tiled_ns(G.cuda(), T, 5, path=path, out_dtype=torch.float32)
    want = oracle.tiled_ns(f64(G), T, 5)
    assert rel_fro(f64(out), want) <= (TOL_BF16 if path == "tensor" else TOL_FP32)


@pytest.mark.parametrize("T", [128, 64, 32])
@pytest.mark.parametrize("K", [0, 1, 3])
@pytest.mark.parametrize("path", ["tensor", "fp32"])
def test_small_K(K, path, T):
    G = synth.lowrank_noise(200, 300, seed=K + 40)
    out = hm.tiled_ns(G.cuda(), T, K, path=path, out_dtype=torch.float32)
    want = oracle.tiled_ns(f64(G), T, K)
    tol = TOL_BF16 if (path == "tensor" and K > 0) else TOL_FP32
    assert rel_fro(f64(out), want) <= tol


@pytest.mark.parametrize("T", [128, 64, 32])
@pytest.mark.parametrize("norm", ["matrix", "none"])
@pytest.mark.parametrize("path", ["tensor", "fp32"])
def test_norm_modes(norm, path, T):
    G = synth.lowrank_noise(256, 384, seed=5)
    if norm == "none":
        G = (G.float() / G.float().norm() * 0.5).to(torch.bfloat16)   # keep the map stable
    out = hm.tiled_ns(G.cuda(), T, 5, norm=norm, path=path, out_dtype=torch.float32)
    want = oracle.tiled_ns(f64(G), T, 5, norm=norm)
    assert rel_fro(f64(out), want) <= (TOL_BF16 if path == "tensor" else TOL_FP32)


@pytest.mark.parametrize("T", [128, 32])
def test_other_coefficients(T):
    G = synth.lowrank_noise(256, 256, seed=8)
    coeffs = (1.5, -0.5, 0.0)
    out = hm.tiled_ns(G.cuda(), T, 8, coeffs=coeffs, out_dtype=torch.float32)
    want = oracle.tiled_ns(f64(G), T, 8, coeffs)
    assert rel_fro(f64(out), want) <= TOL_BF16


# ---------------------------------------------------------------- per-step coefficient schedules

# three quintic steps, a quintic with p(1) = 1 and p'(1) = 0, then a cubic
# (c = 0: two products instead of three) polishing step
SCHED = [(3.4445, -4.7750, 2.0315)] * 3 + [(2.0, -1.5, 0.5), (1.5, -0.5, 0.0)]


@pytest.mark.parametrize("T,path", [(32, "tensor"), (64, "tensor"), (128, "tensor"), (256, "tensor"),
                                    (100, "tensor"), (1024, "tensor"), (16, "tensor"),
                                    (128, "fp32"), (64, "fp32")])
def test_per_step_schedule_matches_oracle(T, path):
    G = synth.lowrank_noise(300, 530, seed=T + 7)
    out = hm.tiled_ns(G.cuda(), T, 5, coeffs=SCHED, path=path, out_dtype=torch.float32)
    want = oracle.tiled_ns(f64(G), T, 5, SCHED)
    assert rel_fro(f64(out), want) <= (TOL_BF16 if path == "tensor" else TOL_FP32)
    # a wrong step order would give another map: the check can tell them apart
    assert rel_fro(oracle.tiled_ns(f64(G), T, 5, SCHED[::-1]), want) > 4 * TOL_BF16


@pytest.mark.parametrize("T", [32, 64, 128, 256])
def test_constant_schedule_equals_single_triple_bit_exact(T):
    G = synth.lowrank_noise(384, 520, seed=T).cuda()
    one = hm.tiled_ns(G, T, 5, path="tensor")
    many = hm.tiled_ns(G, T, 5, coeffs=[hm.QUINTIC] * 5, path="tensor")
    assert torch.equal(one, many)


@pytest.mark.parametrize("T", [128, 64, 32])
def test_step_with_schedule_matches_oracle(T):
    shapes = [(768, 768), (300, 530)]
    Ws, Gs, Ms = _step_case(shapes, 120)
    W0, M0 = [f64(w) for w in Ws], [f64(m) for m in Ms]
    hm.step(Ws, Gs, Ms, T, 5, lr=0.02, mu=0.95, coeffs=SCHED, path="tensor")
    for i in range(len(shapes)):
        Wn, Mn, _ = oracle.himuon_step(W0[i], f64(Gs[i]), M0[i], T, 5, lr=0.02, mu=0.95,
                                       coeffs=SCHED)
        assert rel_fro(f64(Ms[i]), Mn) <= 1e-6
        check_update(f64(Ws[i]), W0[i], Wn, TOL_BF16)


def test_schedule_errors():
    G = synth.lowrank_noise(64, 64, seed=1).cuda()
    with pytest.raises(hm.HimuonError):                   # K triples needed
        hm.tiled_ns(G, 64, 5, coeffs=SCHED[:4])
    bad = list(SCHED)
    bad[2] = (float("nan"), 0.0, 0.0)
    with pytest.raises(hm.HimuonError) as e:              # checked on the host, nothing launched
        hm.tiled_ns(G, 64, 5, coeffs=bad)
    assert e.value.status_name == "INVALID_ARG" and "step 2" in str(e.value)
    tiny_c = list(SCHED)
    tiny_c[1] = (3.0, -1.0, 1e-35)                        # b / c beyond 1e30
    with pytest.raises(hm.HimuonError) as e:
        hm.tiled_ns(G, 64, 5, coeffs=tiny_c)
    assert e.value.status_name == "INVALID_ARG" and "step 1" in str(e.value)


@pytest.mark.parametrize("T", [64, 128, 256])
def test_small_c_step_matches_oracle(T):
    # b / c = -12500 and e / c = 1250: the on-chip kernels' A A accumulator
    # starts at those multiples of A_bf and I, and c scales the sum back
    sched = [hm.QUINTIC] * 2 + [(1.625, -1.0, 8e-5)] + [hm.QUINTIC] * 2
    G = synth.lowrank_noise(320, 448, seed=T + 11)
    out = hm.tiled_ns(G.cuda(), T, 5, coeffs=sched, out_dtype=torch.float32)
    want = oracle.tiled_ns(f64(G), T, 5, sched)
    assert rel_fro(f64(out), want) <= TOL_BF16


# ---------------------------------------------------------------- bit-exact structure

@pytest.mark.parametrize("T", [128, 64, 32, 256])   # on-chip (two), warp-tile and GEMM kernels
@pytest.mark.parametrize("H,W", [(300, 530), (129, 1), (1000, 3000)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_identity_map_is_bit_exact(H, W, dtype, T):
    G = synth.gaussian(H, W, seed=3, dtype=dtype).cuda()
    for K, coeffs in ((0, hm.QUINTIC), (3, (1.0, 0.0, 0.0))):
        out = hm.tiled_ns(G, T, K, coeffs=coeffs, norm="none", out_dtype=dtype)
        assert torch.equal(out, G)


def test_fp32_in_bf16_out_rounds_once():
    G = synth.gaussian(130, 260, seed=4).cuda()
    out = hm.tiled_ns(G, 128, 0, norm="none", out_dtype=torch.bfloat16)
    assert torch.equal(out, G.to(torch.bfloat16))


@pytest.mark.parametrize("path,T,H,W", [("tensor", 128, 384, 512), ("fp32", 128, 384, 512),
                                        ("tensor", 32, 384, 512), ("tensor", 256, 384, 512),
                                        ("tensor", 64, 384, 512), ("tensor", 64, 320, 448)])
def test_perturbing_one_tile_leaves_others_bit_identical(path, T, H, W):
    # T = 64 stacks two tiles into one 128-row tensor-core operand; 320 x 448
    # has 35 tiles, so the last stage holds one valid tile and an empty slot.
    G = synth.lowrank_noise(H, W, seed=9).cuda()
    base = hm.tiled_ns(G, T, 5, path=path)
    G2 = G.clone()
    G2[130:140, 260:300] += 0.01          # inside the tiles that hold rows 130-139, cols 260-299
    pert = hm.tiled_ns(G2, T, 5, path=path)
    mask = torch.ones_like(G, dtype=torch.bool)
    r0, r1 = 130 // T * T, -(-140 // T) * T
    c0, c1 = 260 // T * T, -(-300 // T) * T
    mask[r0:r1, c0:c1] = False
    assert torch.equal(base[mask], pert[mask])
    assert not torch.equal(base[~mask], pert[~mask])


@pytest.mark.parametrize("T", [128, 64, 32, 256])
def test_in_place_equals_out_of_place(T):
    G = synth.lowrank_noise(300, 400, seed=10).cuda()
    ref = hm.tiled_ns(G, T, 5)
    X = G.clone()
    hm.tiled_ns(X, T, 5, out=X)
    assert torch.equal(X, ref)


def test_unaligned_leading_dimension():
    # ld = 50257 bf16 elements: rows are not 16-byte aligned (scalar-load path).
    base = synth.lowrank_noise(256, 50257, seed=11).cuda()
    view = base[:, 1000:1300]               # 256 x 300, ld 50257, odd offset
    out = hm.tiled_ns(view, 128, 5, out_dtype=torch.float32)
    want = oracle.tiled_ns(f64(view), 128, 5)
    assert rel_fro(f64(out), want) <= TOL_BF16
    ref = hm.tiled_ns(view.contiguous(), 128, 5, out_dtype=torch.float32)
    assert torch.equal(out, ref)


# ---------------------------------------------------------------- batching, chunking

def test_batched_equals_single_calls_and_oracle():
    shapes = [(768, 768), (3072, 768), (768, 3072), (200, 130), (1, 5)]
    Gs = [synth.lowrank_noise(H, W, seed=20 + i).cuda() for i, (H, W) in enumerate(shapes)]
    outs = hm.tiled_ns_batched(Gs, 128, 5, out_dtype=torch.float32)
    for G, O in zip(Gs, outs):
        single = hm.tiled_ns(G, 128, 5, out_dtype=torch.float32)
        assert torch.equal(O, single)
        assert rel_fro(f64(O), oracle.tiled_ns(f64(G), 128, 5)) <= TOL_BF16


@pytest.mark.parametrize("T", [64, 128])
def test_batched_stages_straddle_matrices_bit_exact(T):
    """Odd tile counts per matrix: at T = 64 a stage (two stacked tiles) then
    holds the last tile of one matrix and the first of the next; each output
    must equal the single-matrix call bit for bit, and every chunk budget must
    give the same bits."""
    shapes = [(192, 320), (64, 64), (300, 130), (128, 200)]   # 15, 1, 15, 8 tiles at T = 64
    Gs = [synth.lowrank_noise(H, W, seed=60 + i).cuda() for i, (H, W) in enumerate(shapes)]
    outs = hm.tiled_ns_batched(Gs, T, 5, path="tensor", out_dtype=torch.float32)
    for G, O in zip(Gs, outs):
        assert torch.equal(O, hm.tiled_ns(G, T, 5, path="tensor", out_dtype=torch.float32))
        assert rel_fro(f64(O), oracle.tiled_ns(f64(G), T, 5)) <= TOL_BF16
    for chunk in (1, 3 * T * T * 2 + 1, 16 * T * T * 2):
        again = hm.tiled_ns_batched(Gs, T, 5, path="tensor", out_dtype=torch.float32,
                                    chunk_bytes=chunk)
        for a, b in zip(outs, again):
            assert torch.equal(a, b)


@pytest.mark.parametrize("path", ["tensor", "fp32"])
def test_chunking_does_not_change_result(path):
    shapes = [(512, 512), (256, 768), (384, 130)]
    Gs = [synth.lowrank_noise(H, W, seed=30 + i).cuda() for i, (H, W) in enumerate(shapes)]
    ref = hm.tiled_ns_batched(Gs, 128, 5, path=path)
    for chunk in (1, 128 * 128 * 2, 5 * 128 * 128 * 2 + 7, 10 ** 9):
        outs = hm.tiled_ns_batched(Gs, 128, 5, path=path, chunk_bytes=chunk)
        for a, b in zip(ref, outs):
            assert torch.equal(a, b)


# ---------------------------------------------------------------- fused step

def _step_case(shapes, seed, mdtype=torch.float32, wdtype=torch.bfloat16, w0="auto"):
    """Weights, gradients and a non-zero momentum buffer for a step test.

    Weights in bf16 start at zero (w0 "auto"): then W_new = bf16(-lr s O) and
    the update is measured to bf16's own relative rounding (at most 2^-8 per
    element, its unit roundoff), far inside 2e-2, instead of being buried
    under the rounding of |W| ~ 0.02 (about 5 % of an update of lr * 0.08).
    fp32 weights start at N(0, 0.02^2).
    """
    zero = w0 == "zero" or (w0 == "auto" and wdtype == torch.bfloat16)
    Ws = [(torch.zeros(H, W, dtype=wdtype) if zero else
           synth.gaussian(H, W, seed + i, std=0.02, dtype=wdtype)).cuda() for i, (H, W) in enumerate(shapes)]
    Gs = [synth.lowrank_noise(H, W, seed=seed + 100 + i).cuda() for i, (H, W) in enumerate(shapes)]
    Ms = [synth.gaussian(H, W, seed + 200 + i, std=1e-3, dtype=mdtype).cuda() for i, (H, W) in enumerate(shapes)]
    return Ws, Gs, Ms


def check_update(W_gpu, W0, W_ref, tol):
    """The update W_new - W0 against the oracle's, relative Frobenius error <= tol."""
    d_gpu, d_ref = W_gpu - W0, W_ref - W0
    assert np.linalg.norm(d_gpu - d_ref) <= tol * np.linalg.norm(d_ref)


@pytest.mark.parametrize("path,wdtype,T", [("tensor", torch.bfloat16, 128), ("tensor", torch.float32, 128),
                                           ("tensor", torch.bfloat16, 64), ("tensor", torch.float32, 64),
                                           ("fp32", torch.float32, 128)])
def test_step_matches_oracle(path, wdtype, T):
    shapes = [(768, 768), (3072, 768), (300, 530)]
    Ws, Gs, Ms = _step_case(shapes, 50, wdtype=wdtype)
    W0 = [f64(w) for w in Ws]
    M0 = [f64(m) for m in Ms]
    hm.step(Ws, Gs, Ms, T, 5, lr=0.02, mu=0.95, nesterov=True, path=path)
    for i, (H, W) in enumerate(shapes):
        Wn, Mn, O = oracle.himuon_step(W0[i], f64(Gs[i]), M0[i], T, 5, lr=0.02, mu=0.95)
        # momentum: one fp32 FMA per element
        assert rel_fro(f64(Ms[i]), Mn) <= 1e-6
        check_update(f64(Ws[i]), W0[i], Wn, TOL_BF16 if path == "tensor" else TOL_FP32)


@pytest.mark.parametrize("T,H,W", [(128, 384, 256), (128, 256, 520), (64, 320, 200), (64, 192, 448)])
def test_step_weight_reduce_add_is_one_rounding_of_w_plus_update(T, H, W):
    """bf16 weights with 16-byte aligned rows and no weight decay take their
    update by a TMA reduce-add of D = bf16(-lr s O) onto W. From W0 = 0 the step
    stores D itself; from any W0 (same G and M) it must store bf16_rne(W0 + D),
    element for element. Shapes with aligned rows and tall or full tiles only
    (unaligned rows are the next test's; wide edge tiles take the
    read-modify-write, one rounding of W0 + fp32 update); right-edge tiles
    narrower than a 64-column box (8 and 8 columns at 520 and 200) check the box
    clipping."""
    G = synth.lowrank_noise(H, W, seed=T + H).cuda()
    M0 = synth.gaussian(H, W, 3, std=1e-3).cuda()
    W0 = synth.gaussian(H, W, 4, std=0.02, dtype=torch.bfloat16).cuda()
    Wz, Mz = torch.zeros_like(W0), M0.clone()
    hm.step([Wz], [G], [Mz], T, 5, lr=0.02, mu=0.95, path="tensor")
    Wa, Ma = W0.clone(), M0.clone()
    hm.step([Wa], [G], [Ma], T, 5, lr=0.02, mu=0.95, path="tensor")
    assert torch.equal(Ma, Mz)
    want = (W0.float() + Wz.float()).to(torch.bfloat16)
    assert torch.equal(Wa, want)
    Wn, _, _ = oracle.himuon_step(np.zeros((H, W)), f64(G), f64(M0), T, 5, lr=0.02, mu=0.95)
    check_update(f64(Wz), np.zeros((H, W)), Wn, TOL_BF16)


@pytest.mark.parametrize("T,H,W", [(128, 256, 521), (128, 128, 515), (64, 192, 203), (64, 128, 131),
                                   (256, 256, 521), (256, 512, 520), (200, 400, 411)])
def test_step_unaligned_bf16_rows_one_rounding(T, H, W):
    """bf16 weights without weight decay whose rows TMA does not take (odd
    widths; at 128 < T <= 256 every width): each row's 16-byte aligned interior
    gets D = bf16(-lr s O) by one bulk reduce-add and the elements outside it by
    single atomic adds. From W0 = 0 the step stores D; from any W0 (same G and
    M) it must store bf16_rne(W0 + D), element for element. H is a multiple of
    T, so no tile runs transposed; some right-edge tiles (9, 3, 11 and 3
    columns) are narrower than one 16-byte chunk plus a phase, so some rows
    have no interior at all."""
    G = synth.lowrank_noise(H, W, seed=T + W).cuda()
    M0 = synth.gaussian(H, W, 5, std=1e-3).cuda()
    W0 = synth.gaussian(H, W, 6, std=0.02, dtype=torch.bfloat16).cuda()
    Wz, Mz = torch.zeros_like(W0), M0.clone()
    hm.step([Wz], [G], [Mz], T, 5, lr=0.02, mu=0.95, path="tensor")
    Wa, Ma = W0.clone(), M0.clone()
    hm.step([Wa], [G], [Ma], T, 5, lr=0.02, mu=0.95, path="tensor")
    assert torch.equal(Ma, Mz)
    want = (W0.float() + Wz.float()).to(torch.bfloat16)
    assert torch.equal(Wa, want)
    Wn, _, _ = oracle.himuon_step(np.zeros((H, W)), f64(G), f64(M0), T, 5, lr=0.02, mu=0.95)
    check_update(f64(Wz), np.zeros((H, W)), Wn, TOL_BF16)


@pytest.mark.parametrize("T", [64, 128])
def test_step_mixed_weight_update_paths(T):
    """Weights updated four ways in one call: aligned bf16 rows by TMA
    reduce-add, unaligned bf16 rows (odd widths) by bulk reduce-adds of their
    aligned interiors, fp32 weights by the row pass, wide edge tiles by the
    epilogue threads. Odd tile counts at T = 64 put tiles
    of different paths into one stacked stage."""
    shapes = [(192, 320), (130, 203), (64, 64), (200, 530), (70, 300)]
    dtypes = [torch.bfloat16, torch.bfloat16, torch.float32, torch.bfloat16, torch.float32]
    Ws = [torch.zeros(H, W, dtype=dt).cuda() if dt == torch.bfloat16 else
          synth.gaussian(H, W, 7 + i, std=0.02).cuda() for i, ((H, W), dt) in enumerate(zip(shapes, dtypes))]
    Gs = [synth.lowrank_noise(H, W, seed=150 + i).cuda() for i, (H, W) in enumerate(shapes)]
    Ms = [synth.gaussian(H, W, 160 + i, std=1e-3).cuda() for i, (H, W) in enumerate(shapes)]
    W0, M0 = [f64(w) for w in Ws], [f64(m) for m in Ms]
    hm.step(Ws, Gs, Ms, T, 5, lr=0.02, mu=0.95, path="tensor")
    for i in range(len(shapes)):
        Wn, Mn, _ = oracle.himuon_step(W0[i], f64(Gs[i]), M0[i], T, 5, lr=0.02, mu=0.95)
        assert rel_fro(f64(Ms[i]), Mn) <= 1e-6
        check_update(f64(Ws[i]), W0[i], Wn, TOL_BF16)


def test_step_zero_lr_keeps_weights_and_updates_momentum():
    Ws, Gs, Ms = _step_case([(256, 384)], 60)
    W0 = Ws[0].clone()
    M0 = f64(Ms[0])
    hm.step(Ws, Gs, Ms, 128, 5, lr=0.0, mu=0.9)
    assert torch.equal(Ws[0], W0)
    assert rel_fro(f64(Ms[0]), 0.9 * M0 + f64(Gs[0])) <= 1e-6


def test_t32_step_and_chunking():
    shapes = [(300, 200), (96, 500)]
    Ws, Gs, Ms = _step_case(shapes, 95)
    W0, M0 = [f64(w) for w in Ws], [f64(m) for m in Ms]
    hm.step(Ws, Gs, Ms, 32, 5, lr=0.02, mu=0.95, path="tensor")
    for i in range(len(shapes)):
        Wn, Mn, _ = oracle.himuon_step(W0[i], f64(Gs[i]), M0[i], 32, 5, lr=0.02, mu=0.95)
        assert rel_fro(f64(Ms[i]), Mn) <= 1e-6
        check_update(f64(Ws[i]), W0[i], Wn, TOL_BF16)
    ref = hm.tiled_ns_batched(Gs, 32, 5, path="tensor")
    outs = hm.tiled_ns_batched(Gs, 32, 5, path="tensor", chunk_bytes=3 * 32 * 32 * 2 + 1)
    for a, b in zip(ref, outs):
        assert torch.equal(a, b)


@pytest.mark.parametrize("T", [8, 16, 24])
@pytest.mark.parametrize("H,W", [(256, 512), (300, 530), (37, 9)])
def test_tensor_tiles_below_32(H, W, T):
    """T <= 32 runs one warp per tile, zero-padded to 32 x 32."""
    G = synth.gaussian(H, W, seed=T + H)
    out = hm.tiled_ns(G.cuda(), T, 5, path="tensor", out_dtype=torch.float32)
    want = oracle.tiled_ns(f64(G), T, 5)
    assert rel_fro(f64(out), want) <= TOL_BF16


@pytest.mark.parametrize("T", [1, 5])
def test_auto_path_sends_tiny_tiles_to_fp32(T):
    """Tiles of fewer than 64 elements: the AUTO path takes the fp32 kernels (a
    1 x 1 tile on bf16 operands is off by about 2 %)."""
    G = synth.gaussian(256, 512, seed=T)
    out = hm.tiled_ns(G.cuda(), T, 5, path="auto", out_dtype=torch.float32)
    want = oracle.tiled_ns(f64(G), T, 5)
    assert rel_fro(f64(out), want) <= TOL_FP32


def test_t16_step_fp32_weights_bf16_momentum():
    Ws, Gs, Ms = _step_case([(200, 130), (64, 96)], 97, mdtype=torch.bfloat16, wdtype=torch.float32)
    W0, M0 = [f64(w) for w in Ws], [f64(m) for m in Ms]
    hm.step(Ws, Gs, Ms, 16, 5, lr=0.02, mu=0.95, weight_decay=0.01, path="tensor")
    for i in range(2):
        Wn, Mn, _ = oracle.himuon_step(W0[i], f64(Gs[i]), M0[i], 16, 5, lr=0.02, mu=0.95,
                                       weight_decay=0.01)
        assert rel_fro(f64(Ms[i]), Mn) <= 2.0 ** -8       # bf16 momentum buffer: unit roundoff
        check_update(f64(Ws[i]), W0[i], Wn, TOL_BF16)


def test_step_three_successive_steps_with_tile_schedule():
    shapes = [(1000, 3000 // 4), (2048, 503)]
    Ws, _, Ms = _step_case(shapes, 70)
    Wr = [f64(w) for w in Ws]
    Mr = [f64(m) for m in Ms]
    sched = hm.TSchedule([(0, 128), (1, 128), (2, 128)])
    for s in range(3):
        Gs = [synth.lowrank_noise(H, W, seed=1000 * s + i).cuda() for i, (H, W) in enumerate(shapes)]
        T = sched(s)
        hm.step(Ws, Gs, Ms, T, 5, lr=0.02, mu=0.95)
        for i in range(len(shapes)):
            Wr[i], Mr[i], _ = oracle.himuon_step(Wr[i], f64(Gs[i]), Mr[i], T, 5, lr=0.02, mu=0.95)
    for i, (H, W) in enumerate(shapes):
        check_update(f64(Ws[i]), np.zeros((H, W)), Wr[i], TOL_BF16)   # W starts at zero
        assert rel_fro(f64(Ms[i]), Mr[i]) <= 1e-5


def test_step_weight_decay_and_fp32_weights():
    Ws, Gs, Ms = _step_case([(256, 256)], 80, wdtype=torch.float32)
    W0, M0 = f64(Ws[0]), f64(Ms[0])
    hm.step(Ws, Gs, Ms, 128, 5, lr=0.01, mu=0.9, weight_decay=0.1, nesterov=False,
            scale_mode="none")
    Wn, _, _ = oracle.himuon_step(W0, f64(Gs[0]), M0, 128, 5, lr=0.01, mu=0.9, nesterov=False,
                                  weight_decay=0.1, scale_mode="none")
    check_update(f64(Ws[0]), W0, Wn, TOL_BF16)


# ---------------------------------------------------------------- 128 < T <= 256: one tile on a pair of SMs

@pytest.mark.parametrize("T,H,W", [(256, 300, 530), (256, 1000, 300), (256, 512, 512), (200, 450, 700),
                                   (160, 330, 170), (129, 260, 390), (256, 44, 600), (256, 600, 81)])
def test_pair_kernel_matches_oracle(T, H, W):
    """Tiles zero-padded to 256 x 256, held on two SMs. Wide edge tiles (fewer
    rows than columns, e.g. 44 x 256) run transposed, tall ones (600 x 81) as
    they are; T = 129 and 200 give tile origins that are not 16-byte aligned."""
    G = synth.lowrank_noise(H, W, seed=H + 3 * W + T)
    out = hm.tiled_ns(G.cuda(), T, 5, path="tensor", out_dtype=torch.float32)
    want = oracle.tiled_ns(f64(G), T, 5)
    assert rel_fro(f64(out), want) <= TOL_BF16


@pytest.mark.parametrize("K", [1, 2, 3])
def test_pair_kernel_small_K_and_fp32_input(K):
    G = synth.gaussian(384, 520, seed=K)                  # fp32 input
    out = hm.tiled_ns(G.cuda(), 256, K, path="tensor", out_dtype=torch.float32)
    assert rel_fro(f64(out), oracle.tiled_ns(f64(G), 256, K)) <= TOL_BF16
    o16 = hm.tiled_ns(G.cuda(), 256, K, path="tensor", out_dtype=torch.bfloat16)
    assert torch.equal(o16, out.to(torch.bfloat16))      # one rounding of the same fp32 result


@pytest.mark.parametrize("K,coeffs", [(5, SCHED), (3, (1.5, -0.5, 0.0)), (1, hm.QUINTIC)])
def test_pair_kernel_many_tiles_per_cluster(K, coeffs):
    """120 tiles of 256 x 256 on at most 74 clusters, so clusters run several
    tiles back to back. Each step's arrival of the peer block (armed, copied,
    waited on before C X, also on steps without A A) repeats across tiles."""
    G = synth.lowrank_noise(3072, 2560, seed=9 + K)
    out = hm.tiled_ns(G.cuda(), 256, K, coeffs=coeffs, path="tensor", out_dtype=torch.float32)
    want = oracle.tiled_ns(f64(G), 256, K, coeffs)
    assert rel_fro(f64(out), want) <= TOL_BF16


@pytest.mark.parametrize("T", [256, 200])
def test_pair_kernel_step_matches_oracle(T):
    shapes = [(768, 768), (300, 530), (1000, 300), (520, 1030)]
    Ws, Gs, Ms = _step_case(shapes, 130 + T)
    W0, M0 = [f64(w) for w in Ws], [f64(m) for m in Ms]
    hm.step(Ws, Gs, Ms, T, 5, lr=0.02, mu=0.95, nesterov=True, path="tensor")
    for i in range(len(shapes)):
        Wn, Mn, _ = oracle.himuon_step(W0[i], f64(Gs[i]), M0[i], T, 5, lr=0.02, mu=0.95)
        assert rel_fro(f64(Ms[i]), Mn) <= 1e-6
        check_update(f64(Ws[i]), W0[i], Wn, TOL_BF16)


def test_pair_kernel_step_weight_decay_fp32_weights_bf16_momentum():
    shapes = [(512, 300), (260, 700)]
    Ws, Gs, Ms = _step_case(shapes, 140, mdtype=torch.bfloat16, wdtype=torch.float32)
    W0, M0 = [f64(w) for w in Ws], [f64(m) for m in Ms]
    hm.step(Ws, Gs, Ms, 256, 5, lr=0.01, mu=0.9, weight_decay=0.05, nesterov=False, path="tensor")
    for i in range(len(shapes)):
        Wn, Mn, _ = oracle.himuon_step(W0[i], f64(Gs[i]), M0[i], 256, 5, lr=0.01, mu=0.9,
                                       weight_decay=0.05, nesterov=False)
        assert rel_fro(f64(Ms[i]), Mn) <= 2.0 ** -8       # bf16 momentum buffer: unit roundoff
        check_update(f64(Ws[i]), W0[i], Wn, TOL_BF16)


# ---------------------------------------------------------------- other large tiles and the full matrix

@pytest.mark.parametrize("H,W,T", [(300, 530, 256), (1000, 300, 256), (513, 200, 384),
                                   (600, 640, 4096), (1024, 1024, 1024), (130, 700, 96),
                                   (300, 410, 100)])
def test_gemm_path_matches_oracle(H, W, T):
    G = synth.lowrank_noise(H, W, seed=H + 3 * W + T)
    out = hm.tiled_ns(G.cuda(), T, 5, path="tensor", out_dtype=torch.float32)
    want = oracle.tiled_ns(f64(G), T, 5)
    assert rel_fro(f64(out), want) <= TOL_BF16


def test_full_matrix_equals_one_tile_and_differs_from_tiled():
    G = synth.lowrank_noise(512, 768, seed=77).cuda()
    full = hm.tiled_ns(G, 768, 5, path="tensor", out_dtype=torch.float32)
    full2 = hm.tiled_ns(G, 4096, 5, path="tensor", out_dtype=torch.float32)
    assert torch.equal(full, full2)                       # any T >= max(H, W): one tile
    want = oracle.full_ns(f64(G), 5)
    assert rel_fro(f64(full), want) <= TOL_BF16
    tiled = hm.tiled_ns(G, 128, 5, out_dtype=torch.float32)
    assert rel_fro(f64(tiled), want) > 0.05               # a local map, not the full one


def test_gemm_path_4096_t256_sampled_tiles():
    # 4096 x 4096 at T = 256: 256 independent tiles; the oracle checks a sample
    G = synth.lowrank_noise(4096, 4096, seed=5, device="cuda")
    out = hm.tiled_ns(G, 256, 5, path="tensor", out_dtype=torch.float32)
    rng = np.random.default_rng(0)
    for ti, tj in rng.integers(0, 16, size=(6, 2)):
        sl = (slice(256 * ti, 256 * ti + 256), slice(256 * tj, 256 * tj + 256))
        want = oracle.tiled_ns(f64(G[sl]), 256, 5)
        assert rel_fro(f64(out[sl]), want) <= TOL_BF16


@pytest.mark.parametrize("T", [256, 100])
def test_gemm_path_step_matches_oracle(T):
    shapes = [(768, 768), (300, 530), (1000, 300)]
    Ws, Gs, Ms = _step_case(shapes, 90)
    W0 = [f64(w) for w in Ws]
    M0 = [f64(m) for m in Ms]
    hm.step(Ws, Gs, Ms, T, 5, lr=0.02, mu=0.95, nesterov=True, path="tensor")
    for i in range(len(shapes)):
        Wn, Mn, _ = oracle.himuon_step(W0[i], f64(Gs[i]), M0[i], T, 5, lr=0.02, mu=0.95)
        assert rel_fro(f64(Ms[i]), Mn) <= 1e-6
        check_update(f64(Ws[i]), W0[i], Wn, TOL_BF16)


def test_gemm_path_chunking_and_batching_bit_exact():
    shapes = [(600, 520), (300, 1030), (257, 257)]
    Gs = [synth.lowrank_noise(H, W, seed=40 + i).cuda() for i, (H, W) in enumerate(shapes)]
    ref = hm.tiled_ns_batched(Gs, 256, 5, path="tensor")
    for chunk in (1, 256 * 256 * 2 * 3 + 5):
        outs = hm.tiled_ns_batched(Gs, 256, 5, path="tensor", chunk_bytes=chunk)
        for a, b in zip(ref, outs):
            assert torch.equal(a, b)
    for G, O in zip(Gs, ref):
        assert torch.equal(hm.tiled_ns(G, 256, 5, path="tensor"), O)


# ---------------------------------------------------------------- errors

def test_bad_arguments_raise_without_launch():
    G = torch.zeros(4, 4, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(hm.HimuonError) as e:
        hm.tiled_ns(G, 0, 5)
    assert e.value.status_name == "INVALID_ARG"
    with pytest.raises(hm.HimuonError):
        hm.tiled_ns(G, 128, 65)
    with pytest.raises(hm.HimuonError):
        hm.tiled_ns(G, 128, 5, out=G[:, :3])
    with pytest.raises(hm.HimuonError) as e:
        hm.tiled_ns(G, 48, 5, path="tensor")         # no tensor kernel for 32 < T < 64
    assert e.value.status_name == "UNSUPPORTED"
    big = torch.zeros(8, 8, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(hm.HimuonError):               # partial overlap of out and G
        hm.tiled_ns(big[:, :4], 128, 5, out=big[:, 2:6])


def test_bounded_wait_times_out_and_context_survives():
    h = hm.Handle()
    hm.set_wait_limit(1_000_000, handle=h)           # 1 ms
    hm.wait_selftest(handle=h)
    assert hm.device_error(handle=h) == 4            # HIMUON_ERR_TIMEOUT
    assert hm.device_error(handle=h) == 0            # cleared
    G = synth.lowrank_noise(128, 128, seed=1).cuda()
    out = hm.tiled_ns(G, 128, 5, handle=h, out_dtype=torch.float32)
    assert rel_fro(f64(out), oracle.tiled_ns(f64(G), 128, 5)) <= TOL_BF16
    h.close()
