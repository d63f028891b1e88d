"""The optimizer wrapper and the diagnostics tool on the GPU: the wrapper is
bit-identical to direct himuon_step calls (it only marshals arguments), the
diagnostics agree with the fp64 oracle's tiled and full maps."""

import numpy as np
import pytest
import torch

import oracle
import tiled_newton_schulz_03_b300 as hm
from tiled_newton_schulz_03_b300 import diagnostics, synth
from tiled_newton_schulz_03_b300.optim import HiMuon

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from tiled_newton_schulz_03_b300 import build
    build.build()
    hm.load_library()


def test_optimizer_equals_direct_steps_with_schedule():
    shapes = [(768, 768), (3072, 768), (300, 530)]
    params = [torch.nn.Parameter(synth.gaussian(H, W, 5 + i, std=0.02, dtype=torch.bfloat16).cuda())
              for i, (H, W) in enumerate(shapes)]
    Ws = [p.detach().clone() for p in params]
    Ms = [torch.zeros(H, W, device="cuda") for H, W in shapes]
    sched = [(0, 64), (1, 128), (2, 256)]
    opt = HiMuon(params, lr=0.02, momentum=0.95, T=sched, K=5, weight_decay=0.01)
    for s in range(3):
        grads = [synth.lowrank_noise(H, W, seed=40 + 10 * s + i).cuda() for i, (H, W) in enumerate(shapes)]
        for p, g in zip(params, grads):
            p.grad = g
        params[2].grad = None if s == 1 else params[2].grad    # skipped on step 1
        opt.step()
        T = hm.TSchedule(sched)(s)
        idx = [0, 1] if s == 1 else [0, 1, 2]
        hm.step([Ws[i] for i in idx], [grads[i] for i in idx], [Ms[i] for i in idx], T, 5,
                lr=0.02, mu=0.95, weight_decay=0.01)
    for p, w, m in zip(params, Ws, Ms):
        assert torch.equal(p.detach(), w)
        assert torch.equal(opt.state[p]["momentum_buffer"], m)
    assert opt.param_groups[0]["step_count"] == 3


def test_optimizer_state_dict_round_trip():
    p = torch.nn.Parameter(torch.zeros(256, 256, dtype=torch.bfloat16, device="cuda"))
    opt = HiMuon([p], T=[(0, 64), (1, 128)])
    p.grad = synth.lowrank_noise(256, 256, seed=1).cuda()
    opt.step()
    sd = opt.state_dict()
    q = torch.nn.Parameter(p.detach().clone())
    opt2 = HiMuon([q], T=[(0, 64), (1, 128)])
    opt2.load_state_dict(sd)
    assert opt2.param_groups[0]["step_count"] == 1 and HiMuon.tile_size(opt2.param_groups[0]) == 128
    for o, x in ((opt, p), (opt2, q)):
        x.grad = synth.lowrank_noise(256, 256, seed=2).cuda()
        o.step()
    assert torch.equal(p.detach(), q.detach())


def test_diagnostics_against_oracle():
    G = synth.lowrank_noise(384, 640, seed=11).cuda()
    rows = diagnostics.compare(G, [64, 128, 640], K=5)
    g = G.double().cpu().numpy()
    full = oracle.full_ns(g, 5)
    for r in rows:
        if r["full"]:
            assert r["rel_dist_full"] == 0.0 and abs(r["cos_full"] - 1.0) < 1e-12
            continue
        want = np.linalg.norm(oracle.tiled_ns(g, r["T"], 5) - full) / np.linalg.norm(full)
        assert abs(r["rel_dist_full"] - want) <= 0.02 * max(want, 0.1)
        assert r["flops_ratio"] < 1.0 and np.isfinite(r["sv_spread_nonzero"])
    assert rows[0]["flops_ratio"] < rows[1]["flops_ratio"]
