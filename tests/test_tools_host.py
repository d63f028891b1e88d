"""Host-side parts of the optimizer wrapper and the diagnostics tool (no GPU):
argument checks, the runtime tile schedule of the optimizer, and the
diagnostics' analysis helpers against closed forms."""

import numpy as np
import pytest
import torch

import oracle
from tiled_newton_schulz_03_b300 import diagnostics
from tiled_newton_schulz_03_b300.optim import HiMuon


def test_optimizer_rejects_non_2d_parameters():
    w = torch.nn.Parameter(torch.zeros(4, 4))
    b = torch.nn.Parameter(torch.zeros(4))
    with pytest.raises(ValueError, match="2-D"):
        HiMuon([w, b])
    with pytest.raises(ValueError):
        HiMuon([torch.nn.Parameter(torch.zeros(4, 4, dtype=torch.float16))])
    HiMuon([w])                                   # 2-D alone is fine


def test_optimizer_tile_schedule_follows_step_count():
    w = torch.nn.Parameter(torch.zeros(8, 8))
    opt = HiMuon([w], T=[(0, 64), (1, 128), (3, 256)])
    g = opt.param_groups[0]
    seen = []
    for s in range(5):
        g["step_count"] = s
        seen.append(HiMuon.tile_size(g))
    assert seen == [64, 128, 128, 256, 256]
    assert "step_count" in opt.state_dict()["param_groups"][0]


def test_polar_factor_and_spectrum_closed_form():
    r = np.random.default_rng(0)
    U, _ = np.linalg.qr(r.standard_normal((9, 5)))
    V, _ = np.linalg.qr(r.standard_normal((5, 5)))
    G = torch.tensor(U @ np.diag([3.0, 2.0, 1.0, 0.5, 0.1]) @ V.T)
    P = diagnostics.polar_factor(G)
    np.testing.assert_allclose(P.numpy(), U @ V.T, atol=1e-12)
    st = diagnostics.spectrum_stats(P)
    assert abs(st["sv_min"] - 1) < 1e-12 and abs(st["sv_max"] - 1) < 1e-12
    assert st["sv_frac_in_0.5_1.5"] == 1.0 and st["rank"] == 5
    st = diagnostics.spectrum_stats(G)
    assert abs(st["sv_spread_nonzero"] - 30.0) < 1e-9 and abs(st["sv_median"] - 1.0) < 1e-12


def test_distance_and_cosine():
    X = torch.tensor([[3.0, 4.0]])
    assert diagnostics.rel_dist(X, X) == 0.0
    assert abs(diagnostics.rel_dist(2 * X, X) - 1.0) < 1e-15
    assert abs(diagnostics.cosine(X, torch.tensor([[4.0, -3.0]]))) < 1e-15
    assert abs(diagnostics.cosine(X, 5 * X) - 1.0) < 1e-15


@pytest.mark.parametrize("H,W,T,K", [(512, 768, 128, 5), (4096, 4096, 32, 3), (768, 3072, 256, 5)])
def test_ns_work_matches_oracle_count(H, W, T, K):
    # tiled: 2 flops per multiply-add of the oracle's count (divisible shapes)
    assert diagnostics.ns_work(H, W, T, K) == 2 * oracle.ns_mac_count(H, W, T, K)
    # full map, short-side Gram form
    assert diagnostics.ns_work(H, W, max(H, W), K) == 2 * oracle.full_mac_count(H, W, K)
