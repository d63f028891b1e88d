"""Pins of the fp64 oracle against mathematics that does not come from the oracle.

Source of the method: "Hierarchical Muon: Tiled Newton-Schulz Updates for
Efficient Muon Optimization", abstract. Each test names the property it pins and
the kind of mistake in the oracle it would catch.
"""

from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import QUINTIC

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def rng(seed):
    return np.random.default_rng(seed)


def p_exact(x: Fraction, K: int, coeffs) -> Fraction:
    """The odd scalar polynomial a x + b x^3 + c x^5, K times, in exact rationals."""
    a, b, c = (Fraction(v) for v in coeffs)
    for _ in range(K):
        x = a * x + b * x ** 3 + c * x ** 5
    return x


def svd_closed_form(X, K, coeffs, eps):
    """U diag(p^K(sigma / (||sigma||_2 + eps))) V^T from numpy's SVD.

    The NS step maps X = U S V^T to U (a S + b S^3 + c S^5) V^T, so the iterate
    stays in the singular basis and only the singular values move. The Frobenius
    norm equals ||sigma||_2.
    """
    U, S, Vt = np.linalg.svd(X, full_matrices=False)
    s = S / (np.linalg.norm(S) + eps)
    f = np.array([float(p_exact(Fraction(float(v)), K, coeffs)) for v in s])
    return (U * f) @ Vt


# -- the map on one tile: SVD closed form (catches wrong sign, dropped term,
#    transposed operand, wrong normalisation) ----------------------------------

@pytest.mark.parametrize("h,w", [(1, 1), (1, 5), (5, 1), (3, 3), (4, 7), (8, 5), (8, 8)])
@pytest.mark.parametrize("K", [0, 1, 2, 5])
def test_single_tile_matches_svd_closed_form(h, w, K):
    X = rng(100 * h + w + K).standard_normal((h, w))
    got = oracle.ns_map(X, K, QUINTIC, "tile", 1e-7)
    want = svd_closed_form(X, K, QUINTIC, 1e-7)
    assert np.max(np.abs(got - want)) <= 1e-11 * max(1.0, np.max(np.abs(want)))


@pytest.mark.parametrize("coeffs", [(3.4445, -4.7750, 2.0315), (1.5, -0.5, 0.0),
                                    (2.0, -1.5, 0.5), (1.0, 0.3, -0.2)])
def test_other_coefficients_match_svd_closed_form(coeffs):
    X = rng(7).standard_normal((6, 4))
    got = oracle.ns_map(X, 3, coeffs, "tile", 1e-7)
    want = svd_closed_form(X, 3, coeffs, 1e-7)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-11)


def test_tiled_map_equals_closed_form_on_every_ragged_tile():
    # 11 x 13 with T = 4: tiles 4x4, 4x1, 3x4, 3x1 at the edges.
    G = rng(3).standard_normal((11, 13))
    out = oracle.tiled_ns(G, 4, 5)
    n = 0
    for i0, j0, h, w in oracle.tile_grid(11, 13, 4):
        want = svd_closed_form(G[i0:i0 + h, j0:j0 + w], 5, QUINTIC, 1e-7)
        np.testing.assert_allclose(out[i0:i0 + h, j0:j0 + w], want, rtol=0, atol=1e-11)
        n += 1
    assert n == oracle.num_tiles(11, 13, 4) == 12


# -- diagonal and rotated tiles: scalar polynomial on the singular values -------

@pytest.mark.parametrize("K", [1, 3, 5])
def test_diagonal_tile_is_scalar_polynomial_with_sign(K):
    d = [Fraction(3), Fraction(-1), Fraction(1, 2), Fraction(-2, 5)]
    X = np.zeros((4, 6))
    for i, v in enumerate(d):
        X[i, i] = float(v)
    out = oracle.ns_map(X, K, QUINTIC, "tile", 0.0)
    norm = np.sqrt(float(sum(v * v for v in d)))
    want = np.zeros_like(X)
    for i, v in enumerate(d):
        sv = float(v) / norm
        # p is odd: the sign rides along, magnitude from the exact polynomial.
        want[i, i] = float(p_exact(Fraction(abs(sv)), K, QUINTIC)) * np.sign(sv)
    np.testing.assert_allclose(out, want, rtol=0, atol=1e-13)


def test_rotated_diagonal_tile():
    r = rng(11)
    Q1, _ = np.linalg.qr(r.standard_normal((7, 7)))
    Q2, _ = np.linalg.qr(r.standard_normal((5, 5)))
    d = np.array([2.0, 1.0, 0.5, 0.25, 0.125])
    D = np.zeros((7, 5))
    D[:5, :5] = np.diag(d)
    X = Q1 @ D @ Q2.T
    out = oracle.ns_map(X, 5, QUINTIC, "tile", 0.0)
    f = np.array([float(p_exact(Fraction(v / np.linalg.norm(d)), 5, QUINTIC)) for v in d])
    F = np.zeros((7, 5))
    F[:5, :5] = np.diag(f)
    np.testing.assert_allclose(out, Q1 @ F @ Q2.T, rtol=0, atol=1e-12)


def test_one_by_one_tile_hand_value():
    # x = 2: normalised to 2 / (2 + eps); one quintic step at 1 gives
    # a + b + c = 3.4445 - 4.7750 + 2.0315 = 0.7010.
    out = oracle.ns_map(np.array([[2.0]]), 1, QUINTIC, "tile", 0.0)
    assert abs(out[0, 0] - 0.7010) < 1e-12
    out = oracle.ns_map(np.array([[-2.0]]), 1, QUINTIC, "tile", 0.0)
    assert abs(out[0, 0] + 0.7010) < 1e-12


# -- full-matrix special case (abstract, sentences 1-2 and 4) --------------------

@pytest.mark.parametrize("H,W,T", [(6, 9, 9), (9, 6, 16), (8, 8, 8)])
def test_tile_covering_matrix_is_full_matrix_ns(H, W, T):
    G = rng(H * W).standard_normal((H, W))
    tiled = oracle.tiled_ns(G, T, 5)
    full = oracle.full_ns(G, 5)
    np.testing.assert_allclose(tiled, full, rtol=0, atol=1e-12)
    np.testing.assert_allclose(full, svd_closed_form(G, 5, QUINTIC, 1e-7), rtol=0, atol=1e-11)


def test_tiled_differs_from_full_below_matrix_size():
    # A local map, not an approximation of the full one (abstract, sentence 4).
    G = rng(5).standard_normal((8, 8))
    assert np.max(np.abs(oracle.tiled_ns(G, 4, 5) - oracle.full_ns(G, 5))) > 1e-2


# -- classical polar limit (Bjorck-Bowie cubic iteration) -----------------------

def test_cubic_coefficients_converge_to_polar_factor():
    r = rng(21)
    U, _ = np.linalg.qr(r.standard_normal((8, 6)))
    V, _ = np.linalg.qr(r.standard_normal((6, 6)))
    X = U @ np.diag(np.linspace(1.0, 3.0, 6)) @ V.T
    out = oracle.ns_map(X, 60, (1.5, -0.5, 0.0), "tile", 1e-7)
    np.testing.assert_allclose(out, U @ V.T, rtol=0, atol=1e-10)


# -- tile independence (abstract, sentence 4) -------------------------------------

def test_perturbing_one_tile_leaves_all_other_tiles_bit_identical():
    G = rng(9).standard_normal((20, 30))
    base = oracle.tiled_ns(G, 8, 5)
    G2 = G.copy()
    G2[9:12, 17:20] += 0.5          # inside tile (1, 2): rows 8..15, cols 16..23
    pert = oracle.tiled_ns(G2, 8, 5)
    changed = np.zeros_like(G, dtype=bool)
    changed[8:16, 16:24] = True
    assert np.array_equal(base[~changed], pert[~changed])
    assert not np.allclose(base[changed], pert[changed])


def test_sampled_tiles_equal_full_tiled_output():
    G = rng(12).standard_normal((37, 50))
    full = oracle.tiled_ns(G, 16, 5)
    for i0, j0, t in oracle.tiled_ns_tiles(G, 16, 5, [(0, 0), (2, 3), (1, 1)]):
        h, w = t.shape
        np.testing.assert_allclose(full[i0:i0 + h, j0:j0 + w], t, rtol=0, atol=1e-13)


# -- identity, zero, normalisation, zero padding ---------------------------------

def test_identity_coefficients_without_normalisation_is_exact_copy():
    G = rng(1).standard_normal((13, 7))
    assert np.array_equal(oracle.tiled_ns(G, 4, 5, (1.0, 0.0, 0.0), "none"), G)
    assert np.array_equal(oracle.tiled_ns(G, 4, 0, QUINTIC, "none"), G)


def test_k0_gives_unit_frobenius_tiles():
    G = rng(2).standard_normal((10, 10)) * 7.0
    out = oracle.tiled_ns(G, 4, 0)
    for i0, j0, h, w in oracle.tile_grid(10, 10, 4):
        n = np.linalg.norm(G[i0:i0 + h, j0:j0 + w])
        assert abs(np.linalg.norm(out[i0:i0 + h, j0:j0 + w]) - n / (n + 1e-7)) < 1e-14


def test_zero_tile_maps_to_zero():
    G = rng(4).standard_normal((8, 8))
    G[:4, 4:] = 0.0
    out = oracle.tiled_ns(G, 4, 5)
    assert np.array_equal(out[:4, 4:], np.zeros((4, 4)))
    assert np.all(np.isfinite(out))


def test_zero_padding_to_full_tiles_changes_nothing():
    # Zero rows/columns stay zero through the polynomial and leave the Frobenius
    # norm alone, so a ragged tile equals the valid block of its padded tile.
    G = rng(6).standard_normal((10, 13))
    P = np.zeros((12, 16))
    P[:10, :13] = G
    np.testing.assert_allclose(oracle.tiled_ns(P, 4, 5)[:10, :13],
                               oracle.tiled_ns(G, 4, 5), rtol=0, atol=1e-13)


def test_scale_invariance_up_to_eps():
    G = rng(8).standard_normal((12, 12))
    np.testing.assert_allclose(oracle.tiled_ns(1e3 * G, 4, 5, eps=0.0),
                               oracle.tiled_ns(G, 4, 5, eps=0.0), rtol=0, atol=1e-10)


def test_matrix_norm_mode_uses_one_factor_for_all_tiles():
    G = rng(10).standard_normal((8, 12))
    n = np.linalg.norm(G)
    out = oracle.tiled_ns(G, 4, 2, norm="matrix", eps=1e-7)
    for i0, j0, h, w in oracle.tile_grid(8, 12, 4):
        # Every tile is scaled by the whole-matrix norm, then the polynomial acts
        # on its singular values.
        Ut, S, Vt = np.linalg.svd(G[i0:i0 + h, j0:j0 + w], full_matrices=False)
        f = [float(p_exact(Fraction(float(v / (n + 1e-7))), 2, QUINTIC)) for v in S]
        want = (Ut * np.array(f)) @ Vt
        np.testing.assert_allclose(out[i0:i0 + h, j0:j0 + w], want, rtol=0, atol=1e-12)


# -- work count (abstract, sentence 5) --------------------------------------------

def _brute_force_macs(H, W, T, K):
    """Count multiply-adds by walking the loops of each product on each tile."""
    n = 0
    for _, _, h, w in oracle.tile_grid(H, W, T):
        for _ in range(K):
            for i in range(h):            # A = X X^T
                for j in range(h):
                    n += w
            for i in range(h):            # A A
                for j in range(h):
                    n += h
            for i in range(h):            # B X
                for j in range(w):
                    n += h
    return n


@pytest.mark.parametrize("H,W,T,K", [(5, 7, 3, 2), (8, 8, 4, 1), (9, 4, 5, 3), (1, 1, 1, 1)])
def test_mac_count_brute_force(H, W, T, K):
    assert oracle.ns_mac_count(H, W, T, K) == _brute_force_macs(H, W, T, K)


@pytest.mark.parametrize("H,W,T,K", [(4096, 4096, 128, 5), (14336, 4096, 128, 5),
                                     (1024, 4096, 64, 3), (768, 3072, 256, 5)])
def test_mac_count_is_3HWTK_for_divisible_shapes(H, W, T, K):
    assert oracle.ns_mac_count(H, W, T, K) == 3 * H * W * T * K


def test_full_tile_work_is_r2sK():
    # One tile covering a wide matrix is the min-side Gram form: O(r^2 s K).
    assert oracle.ns_mac_count(64, 256, 256, 5) == oracle.full_mac_count(64, 256, 5)


def test_tiled_work_grows_linearly_in_T():
    w = [oracle.ns_mac_count(1024, 1024, T, 5) for T in (32, 64, 128, 256)]
    assert w[1] == 2 * w[0] and w[2] == 2 * w[1] and w[3] == 2 * w[2]


# -- one optimizer step ----------------------------------------------------------

def test_momentum_hand_values():
    M, U = oracle.momentum(np.array([[1.0]]), np.array([[1.0]]), 0.5, nesterov=True)
    assert M[0, 0] == 1.5 and U[0, 0] == 1.75
    M, U = oracle.momentum(np.array([[1.0]]), np.array([[1.0]]), 0.5, nesterov=False)
    assert M[0, 0] == 1.5 and U[0, 0] == 1.5


def test_step_with_zero_lr_keeps_weights():
    r = rng(13)
    Wt, G = r.standard_normal((6, 10)), r.standard_normal((6, 10))
    W1, M1, _ = oracle.himuon_step(Wt, G, np.zeros_like(G), 4, 5, lr=0.0, mu=0.95)
    assert np.array_equal(W1, Wt)
    np.testing.assert_array_equal(M1, G)


def test_step_with_zero_momentum_is_plain_tiled_map():
    r = rng(14)
    Wt, G = r.standard_normal((12, 6)), r.standard_normal((12, 6))
    M0 = r.standard_normal((12, 6))
    W1, _, _ = oracle.himuon_step(Wt, G, M0, 4, 5, lr=0.1, mu=0.0)
    s = np.sqrt(2.0)                      # sqrt(max(1, 12 / 6))
    np.testing.assert_allclose(W1, Wt - 0.1 * s * oracle.tiled_ns(G, 4, 5), rtol=0, atol=1e-14)


def test_update_scale():
    assert oracle.update_scale(14336, 4096) == np.sqrt(14336 / 4096)
    assert oracle.update_scale(1024, 4096) == 1.0
    assert oracle.update_scale(1024, 4096, "none") == 1.0


def test_weight_decay_is_decoupled():
    r = rng(15)
    Wt, G = r.standard_normal((4, 4)), r.standard_normal((4, 4))
    Wa, _, O = oracle.himuon_step(Wt, G, np.zeros_like(G), 4, 5, lr=0.1, mu=0.9, weight_decay=0.5)
    Wb, _, _ = oracle.himuon_step(Wt, G, np.zeros_like(G), 4, 5, lr=0.1, mu=0.9, weight_decay=0.0)
    np.testing.assert_allclose(Wa, Wb - 0.1 * 0.5 * Wt, rtol=0, atol=1e-15)


def test_ema_momentum_gives_same_direction_up_to_eps():
    # U and (1 - mu) U normalise to the same tile, so the direction agrees.
    r = rng(16)
    G = r.standard_normal((8, 8))
    O1 = oracle.tiled_ns(G, 4, 5, eps=0.0)
    O2 = oracle.tiled_ns(0.05 * G, 4, 5, eps=0.0)
    np.testing.assert_allclose(O1, O2, rtol=0, atol=1e-11)


# -- which quantity the step hands to the NS map ----------------------------------
# With mu != 0, M0 != 0 and no normalisation, the Nesterov input U = G + mu M_new
# and the plain-momentum input M_new differ, so passing the wrong one (or G, or
# M0) to the NS map changes O. All values below are exact rationals.

def _p1(x: Fraction) -> Fraction:
    return p_exact(x, 1, QUINTIC)


@pytest.mark.parametrize("nesterov,u", [(True, Fraction(7, 4)), (False, Fraction(3, 2))])
def test_step_ns_input_hand_value_1x1(nesterov, u):
    # G = 1, M0 = 1, mu = 1/2: M_new = 3/2; U = 1 + 3/4 = 7/4 (Nesterov) or 3/2.
    W0, lr = 0.25, 0.125
    W1, M1, O = oracle.himuon_step(np.array([[W0]]), np.array([[1.0]]), np.array([[1.0]]), 1, 1,
                                   lr=lr, mu=0.5, nesterov=nesterov, norm="none")
    assert M1[0, 0] == 1.5
    want_o = _p1(u)
    assert abs(O[0, 0] - float(want_o)) <= 1e-12 * abs(float(want_o))
    want_w = Fraction(W0) - Fraction(lr) * want_o          # s = sqrt(max(1, 1/1)) = 1
    assert abs(W1[0, 0] - float(want_w)) <= 1e-12 * abs(float(want_w))
    # the other readings give other values: the pin separates them
    for wrong in (Fraction(3, 2) if nesterov else Fraction(7, 4), Fraction(1)):
        assert abs(float(_p1(wrong)) - float(want_o)) > 0.1


def test_step_ns_input_scale_and_decay_hand_value_2x1():
    # A 2 x 1 matrix (H / W = 2, so s = sqrt(2)) with U = [7/4, 0]^T: the
    # Gram is diag(49/16, 0), so one step maps 7/4 to p(7/4) and 0 to 0.
    W0 = np.array([[0.5], [-0.25]])
    G = np.array([[1.0], [0.0]])
    M0 = np.array([[1.0], [0.0]])
    lr, wd = 0.125, 0.5
    W1, M1, O = oracle.himuon_step(W0, G, M0, 2, 1, lr=lr, mu=0.5, nesterov=True,
                                   weight_decay=wd, norm="none")
    po = float(_p1(Fraction(7, 4)))
    np.testing.assert_allclose(O[:, 0], [po, 0.0], rtol=1e-12, atol=0)
    np.testing.assert_array_equal(M1[:, 0], [1.5, 0.0])
    s = np.sqrt(2.0)
    want = W0[:, 0] - lr * wd * W0[:, 0] - lr * s * np.array([po, 0.0])
    np.testing.assert_allclose(W1[:, 0], want, rtol=1e-13, atol=0)


def test_step_ns_input_with_tile_norm_is_direction_of_u():
    # Per-tile normalisation removes the length of U but not its direction:
    # on a 1 x 2 tile U = G + mu (mu M0 + G) with G = [1, 0], M0 = [0, 4],
    # mu = 1/2 gives M_new = [1, 2] and U = [1, 0] + [1/2, 1] = [3/2, 1].
    G = np.array([[1.0, 0.0]])
    M0 = np.array([[0.0, 4.0]])
    _, M1, O = oracle.himuon_step(np.zeros((1, 2)), G, M0, 2, 1, lr=0.0, mu=0.5, eps=0.0)
    np.testing.assert_array_equal(M1, [[1.0, 2.0]])
    u = np.array([1.5, 1.0])
    n = np.linalg.norm(u)
    # a rank-1 row: the NS step acts on its one singular value 1 after normalising
    np.testing.assert_allclose(O[0], u / n * float(_p1(Fraction(1))), rtol=1e-12, atol=0)


# -- per-step coefficient schedules --------------------------------------------
# Step k applies p_k(s) = a_k s + b_k s^3 + c_k s^5 to the singular values, so K
# steps are the composition p_{K-1} o ... o p_0 (first triple first).

MIXED = [(3.4445, -4.7750, 2.0315), (2.0, -1.5, 0.5), (1.5, -0.5, 0.0), (1.875, -1.25, 0.375)]


def p_sched(x: Fraction, sched) -> Fraction:
    for a, b, c in sched:
        a, b, c = Fraction(a), Fraction(b), Fraction(c)
        x = a * x + b * x ** 3 + c * x ** 5
    return x


@pytest.mark.parametrize("h,w", [(1, 1), (3, 5), (6, 4), (8, 8)])
def test_schedule_matches_svd_closed_form(h, w):
    X = rng(200 + 10 * h + w).standard_normal((h, w))
    got = oracle.ns_map(X, len(MIXED), MIXED, "tile", 1e-7)
    U, S, Vt = np.linalg.svd(X, full_matrices=False)
    s = S / (np.linalg.norm(S) + 1e-7)
    f = np.array([float(p_sched(Fraction(float(v)), MIXED)) for v in s])
    np.testing.assert_allclose(got, (U * f) @ Vt, rtol=0, atol=1e-11)


def test_schedule_order_is_first_triple_first():
    X = rng(31).standard_normal((5, 7))
    fwd = oracle.ns_map(X, 4, MIXED, "tile", 0.0)
    rev = oracle.ns_map(X, 4, MIXED[::-1], "tile", 0.0)
    assert np.max(np.abs(fwd - rev)) > 1e-3
    # 1 x 1 hand value: x = 1 after normalisation; p_0(1) = a+b+c = 0.701,
    # then the cubic 2 - 1.5 + 0.5 at 0.701, ...
    x = oracle.ns_map(np.array([[3.0]]), 2, MIXED[:2], "tile", 0.0)[0, 0]
    y = Fraction(7010, 10000)
    want = 2 * y - Fraction(3, 2) * y ** 3 + Fraction(1, 2) * y ** 5
    assert abs(x - float(want)) < 1e-13


def test_constant_schedule_equals_single_triple_exactly():
    G = rng(32).standard_normal((20, 13))
    one = oracle.tiled_ns(G, 8, 5, QUINTIC)
    many = oracle.tiled_ns(G, 8, 5, [QUINTIC] * 5)
    assert np.array_equal(one, many)


def test_quintic_then_cubic_schedule_reaches_polar_factor():
    # the quintic leaves singular values in a band around 1; cubic Newton-Schulz
    # steps (Bjorck-Bowie) then converge them to exactly 1: the polar factor
    r = rng(33)
    U, _ = np.linalg.qr(r.standard_normal((9, 6)))
    V, _ = np.linalg.qr(r.standard_normal((6, 6)))
    X = U @ np.diag(np.geomspace(1.0, 0.05, 6)) @ V.T
    sched = [QUINTIC] * 5 + [(1.5, -0.5, 0.0)] * 25
    out = oracle.ns_map(X, len(sched), sched, "tile", 1e-7)
    np.testing.assert_allclose(out, U @ V.T, rtol=0, atol=1e-10)
    # the quintic alone does not: its fixed band is not {1}
    q = oracle.ns_map(X, 30, QUINTIC, "tile", 1e-7)
    assert np.max(np.abs(q - U @ V.T)) > 1e-2


def test_schedule_length_must_be_K():
    with pytest.raises(ValueError):
        oracle.ns_map(np.eye(3), 3, MIXED, "tile", 0.0)
