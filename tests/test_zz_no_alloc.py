"""The allocation-free entry point himuon_tiled_ns_fp32_noalloc, called
through the C ABI, against the fp64 oracle and the handle-based fp32 path.

That entry point serves callers that cannot call cudaMalloc (their device
memory is all reserved by another allocator, or they must not risk the device
synchronisation cudaMalloc can cause): it keeps its scratch in a fixed device
array of the library. This file is named so that pytest collects it last.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import tiled_newton_schulz_03_b300 as hm
from tiled_newton_schulz_03_b300 import synth

pytestmark = pytest.mark.gpu

TOL_FP32 = 1e-5


def f64(t):
    return t.detach().float().cpu().double().numpy()


def rel_fro(got, want):
    got, want = np.asarray(got, dtype=np.float64), np.asarray(want, dtype=np.float64)
    return float(np.linalg.norm(got - want) / np.linalg.norm(want))


@pytest.fixture(scope="module")
def lib():
    from tiled_newton_schulz_03_b300 import build
    build.build()
    return hm.load_library()


def _call_noalloc(lib, G, out, T, K, norm="tile"):
    p = hm.NSParams()
    lib.himuon_default_ns_params(ctypes.byref(p))
    p.norm = {"tile": 0, "matrix": 1, "none": 2}[norm]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    dt = {torch.bfloat16: 0, torch.float32: 1}
    return lib.himuon_tiled_ns_fp32_noalloc(
        ctypes.c_void_p(G.data_ptr()), G.size(0), G.size(1), G.stride(0), dt[G.dtype], T, K,
        ctypes.byref(p), ctypes.c_void_p(out.data_ptr()), out.stride(0), dt[out.dtype], stream)


@pytest.mark.parametrize("H,W,T,norm", [(300, 530, 128, "tile"), (2000, 1500, 256, "matrix"),
                                        (257, 129, 64, "none")])
def test_noalloc_matches_oracle_and_handle_path_twice(lib, H, W, T, norm):
    G = synth.lowrank_noise(H, W, seed=H + W).cuda()
    if norm == "none":
        G = (G.float() / G.float().norm() * 0.5).to(torch.bfloat16)
    want = oracle.tiled_ns(f64(G), T, 5, norm=norm)
    ref = hm.tiled_ns(G, T, 5, norm=norm, path="fp32", out_dtype=torch.float32)
    for _ in range(2):                          # the array keeps the last call's contents
        out = torch.full((H, W), float("nan"), device="cuda")
        assert _call_noalloc(lib, G, out, T, 5, norm) == 0
        torch.cuda.synchronize()
        assert rel_fro(f64(out), want) <= TOL_FP32
        assert rel_fro(f64(out), f64(ref)) <= TOL_FP32


def test_noalloc_in_place_and_fp32_in_bf16_out(lib):
    G = synth.gaussian(300, 200, seed=5)                 # fp32 input
    want = oracle.tiled_ns(f64(G), 64, 5)
    G = G.cuda()
    X = G.clone()
    assert _call_noalloc(lib, X, X, 64, 5) == 0          # in place
    torch.cuda.synchronize()
    assert rel_fro(f64(X), want) <= TOL_FP32
    ref16 = hm.tiled_ns(G, 64, 5, path="fp32", out_dtype=torch.bfloat16)
    for _ in range(2):
        o16 = torch.zeros(300, 200, dtype=torch.bfloat16, device="cuda")
        assert _call_noalloc(lib, G, o16, 64, 5) == 0    # fp32 in, bf16 out
        torch.cuda.synchronize()
        assert torch.equal(o16, ref16)                   # same per-tile arithmetic, one rounding


def test_noalloc_leaves_device_memory_unchanged(lib):
    G = synth.lowrank_noise(1000, 700, seed=9).cuda()
    out = torch.empty(1000, 700, device="cuda")
    assert _call_noalloc(lib, G, out, 128, 5) == 0       # first call: set-up done
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert _call_noalloc(lib, G, out, 128, 5) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_noalloc_rejects_oversized_tiles(lib):
    G = torch.zeros(2048, 2048, device="cuda", dtype=torch.bfloat16)
    out = torch.empty(2048, 2048, device="cuda")
    assert _call_noalloc(lib, G, out, 2048, 5) == 1           # HIMUON_ERR_INVALID_ARG
    assert b"fixed scratch" in lib.himuon_last_error_string()
