"""Host logic of bench.py that needs no GPU: the roofline arithmetic and the
multi-rank launch command."""

import bench


PEAKS = {"bf16_tflops": 1747.0, "hbm_gbs": 6494.3}


def test_roofline_takes_the_slower_bound():
    # Llama-3-8B set, T = 128, K = 5: 26.80 TFLOP and 14 B/param of the fused step
    params = 6979321856
    flops = 6.0 * 128 * 5 * params
    nbytes = 14.0 * params
    r = bench.roofline(flops, nbytes, 43.116e-3, PEAKS, "measured")
    t_tc, t_hbm = flops / 1747e12, nbytes / 6494.3e9
    assert r["bound"] == "tensor" and t_tc > t_hbm
    assert abs(r["frac"] - max(t_tc, t_hbm) / 43.116e-3) < 1e-3
    assert abs(r["roofline_ms"] - 1e3 * t_tc) < 1e-3
    # same work with more bytes: HBM bound, frac in GB/s terms
    r = bench.roofline(flops, 4 * nbytes, 0.1, PEAKS, "measured")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["frac"] - 4 * nbytes / 6494.3e9 / 0.1) < 1e-3


def test_roofline_frac_is_one_at_the_bound():
    r = bench.roofline(1747e12, 1.0, 1.0, PEAKS, "measured")
    assert r["frac"] == 1.0


def test_relaunch_command_starts_n_local_ranks():
    cmd = bench.relaunch_command(["--gpus", "4", "--steps", "3"], 4, 29500)
    assert "torch.distributed.run" in cmd and "--nproc-per-node=4" in cmd
    assert "--master-addr=127.0.0.1" in cmd and "--master-port=29500" in cmd
    assert cmd[-4:] == ["--gpus", "4", "--steps", "3"]
