"""The multi-GPU (replicas) path of bench.py on CPU ranks: two gloo processes
build the JSON line from per-rank results the way the GPU ranks do, and the
reference arm's extra ranks exit without work.  No GPU is touched."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _fake_results(rank):
    """What bench_prefill / bench_decode return, with rank-dependent times."""
    import synth
    pre = {"wl": synth.BY_NAME["glm_prefill"], "T": 4096, "step_ms": [3.0 + rank] * 4,
           "stage": {"w13": 2.0 + 0.5 * rank, "w2": 1.0}, "launches": 70, "regime": 2,
           "counts": np.arange(1, 257, dtype=np.int32), "clocks": {"sm_mhz": 2070.0},
           "e2e_s": 0.004 + 0.001 * rank, "h2d": 100, "d2h": 200}
    dec = {"wl": synth.BY_NAME["glm_decode"], "T": 1, "step_ms": [0.6 + 0.2 * rank] * 4,
           "layers": 8, "n_active": [9] * 8, "stage": {"w13": 0.03}, "launches": 400,
           "clocks": {"sm_mhz": 2070.0}, "e2e_s": 0.001, "h2d": 1, "d2h": 1}
    return pre, dec


def _rank_main(rank, world, port, out_path):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)

    def reduce_max(v):
        t = torch.tensor([float(v)])
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    pre, dec = _fake_results(rank)
    pk = {"hbm_gbs": 6792.4, "bf16_tflops": 1898.0, "bf16_tflops_sustained": 1707.1}
    line = bench.make_line(pre, dec, world, reduce_max, pk, "measured", 4, 3)
    dist.barrier()
    dist.destroy_process_group()
    if rank == 0:
        with open(out_path, "w") as f:
            json.dump(line, f)


def test_two_gloo_ranks_take_the_slowest_rank(tmp_path):
    import torch.multiprocessing as mp
    out = str(tmp_path / "line.json")
    mp.start_processes(_rank_main, args=(2, _free_port(), out), nprocs=2, start_method="spawn")
    line = json.load(open(out))
    assert line["n_gpus"] == 2 and line["scaling"] == "weak"
    assert line["config"]["parallelism"] == "replicas"
    assert line["ms_per_step"] == pytest.approx(4.0)                 # max over ranks
    assert line["value"] == pytest.approx(2 * 4096 / 4.0e-3)         # tokens of all ranks
    assert line["e2e"]["value"] == pytest.approx(2 * 4096 / 0.005)
    assert line["decode"]["ms_per_step"] == pytest.approx(0.8)
    assert line["decode"]["tokens_per_s"] == pytest.approx(2 / 0.8e-3)
    assert line["decode"]["e2e"]["value"] == pytest.approx(2 / 0.001)   # host buffers, every step
    assert line["roofline"]["unit"] == "TFLOP/s"
    for key in ("metric", "unit", "higher_is_better", "dtype", "data", "config", "gpu_launches",
                "clocks", "e2e", "roofline", "vs_baseline", "steps", "warmup"):
        assert key in line


def test_reference_arm_extra_rank_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "1"],
                       capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_decode_roofline_names_the_kernel_of_its_path():
    """The decode roofline entry names the kernel the automatic choice ran:
    the GEMV at one token, the decode tensor-core kernel at 2-8 (whose DRAM
    traffic the committed capture does not cover)."""
    sys.path.insert(0, ROOT)
    import bench
    import synth
    pk = {"hbm_gbs": 6792.4, "bf16_tflops": 1898.0, "bf16_tflops_sustained": 1707.1}
    base = {"wl": synth.BY_NAME["glm_decode"], "stage": {"w13": 0.1}, "n_active": [30]}
    tc = bench.roofline_gemv(dict(base, T=4, regime=3), pk, "measured")
    assert tc["kernel"] == "decode_tc_w13" and tc["traffic"] is None and tc["bound"] == "hbm"
    gv = bench.roofline_gemv(dict(base, T=1, regime=1), pk, "measured")
    assert gv["kernel"] == "gemv_w13"
    assert gv["achieved"] == pytest.approx((30 * 2 * 6144 * 2048 * 9 // 16 + 6144 * 2) / 0.1e-3 / 1e9,
                                           rel=1e-3)
    assert "w2" not in gv   # no W2 stage time, no W2 entry


def test_decode_roofline_reports_the_w2_pass_of_its_path():
    """Beside W13, the W2 entry counts the activated experts' down-projection
    rows and scales plus h's two bf16 planes, and names the kernel that the
    path and shape select: the K-split MMA kernel for K = 1024 / 2048 shared
    by routed and shared experts, the tiled one up to K = 4096, the SIMT
    kernel beyond, the decode tensor-core kernel at 2-8 tokens."""
    sys.path.insert(0, ROOT)
    import bench
    import synth
    pk = {"hbm_gbs": 6792.4, "bf16_tflops": 1898.0, "bf16_tflops_sustained": 1707.1}
    st = {"w13": 0.1, "w2": 0.05}
    glm = {"wl": synth.BY_NAME["glm_decode"], "stage": st, "n_active": [9]}
    w2 = bench.roofline_gemv(dict(glm, T=1, regime=1), pk, "measured")["w2"]
    assert w2["kernel"] == "gemv_w2_ks"
    by = 9 * 6144 * 2048 * 9 // 16 + 9 * 2 * 2048 * 2
    assert w2["achieved"] == pytest.approx(by / 0.05e-3 / 1e9, rel=1e-3)
    assert w2["frac"] == pytest.approx(w2["achieved"] / 6792.4, rel=1e-3)
    assert bench.roofline_gemv(dict(glm, T=4, regime=3), pk, "measured")["w2"]["kernel"] == \
        "decode_tc_w2"
    mix = {"wl": synth.BY_NAME["mixtral"], "stage": st, "n_active": [2]}
    assert bench.roofline_gemv(dict(mix, T=1, regime=1), pk, "measured")["w2"]["kernel"] == \
        "gemv_w2_simt"
    olm = {"wl": synth.BY_NAME["olmoe"], "stage": st, "n_active": [8]}
    assert bench.roofline_gemv(dict(olm, T=1, regime=1), pk, "measured")["w2"]["kernel"] == \
        "gemv_w2_ks"


def test_algorithmic_units_match_the_published_per_layer_figures():
    """bench.py's bytes and FLOPs of a layer reproduce the per-layer workload
    table of the scope: a GLM-shaped decode layer with 9 activated experts
    (8 routed + shared) at T = 1 moves 197.4 MB; the prefill layer at T = 4096
    does 2.80 TFLOP (routed 2.47 + shared 0.31 + router 0.013)."""
    sys.path.insert(0, ROOT)
    import bench
    import synth
    dec = synth.BY_NAME["glm_decode"]
    assert bench.layer_bytes(dec, 9, 1) / 1e6 == pytest.approx(197.4, abs=0.05)
    pre = synth.BY_NAME["glm_prefill"]
    fl = bench.layer_flops(pre, 4096)
    assert fl / 1e12 == pytest.approx(2.80, abs=0.005)
    routed = 2 * 4096 * 8 * 3 * 6144 * 2048
    shared = 2 * 4096 * 1 * 3 * 6144 * 2048
    router = 2 * 4096 * 6144 * 256
    assert (routed / 1e12, shared / 1e12, router / 1e12) == (
        pytest.approx(2.47, abs=0.005), pytest.approx(0.31, abs=0.005),
        pytest.approx(0.013, abs=0.0005))
    assert fl == routed + shared + router


def test_clock_records_are_checked_and_a_bad_region_is_measured_once_more():
    """A timed region that saw a hardware or thermal slowdown, or sat well
    below the maximum SM clock with no reason given, is measured once more
    (single process); sw_power_cap is kept.  The second record is the one
    reported, the rejected one beside it."""
    sys.path.insert(0, ROOT)
    import bench
    ok = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 10}
    assert bench.clocks_ok(ok)
    assert bench.clocks_ok(dict(ok, sm_mhz=1455.0, reasons=["sw_power_cap"]))
    assert not bench.clocks_ok(dict(ok, reasons=["hw_slowdown"]))
    assert not bench.clocks_ok(dict(ok, reasons=["sw_thermal_slowdown", "sw_power_cap"]))
    assert not bench.clocks_ok(dict(ok, sm_mhz=1200.0))          # a leftover clock lock

    records = [dict(ok, reasons=["hw_thermal_slowdown"]), ok]

    class FakeSampler:
        def __init__(self, dev):
            self.rec = records.pop(0)

        def __enter__(self):
            return self

        def __exit__(self, *a):
            return False

        def summary(self):
            return dict(self.rec)

    runs = []
    out, c = bench.timed_region(None, lambda: runs.append(1) or len(runs), sampler=FakeSampler)
    assert len(runs) == 2 and out == 2
    assert c["remeasured"] and c["rejected"]["reasons"] == ["hw_thermal_slowdown"]
    assert c["reasons"] == []

    records[:] = [ok]
    runs.clear()
    out, c = bench.timed_region(None, lambda: runs.append(1) or len(runs), sampler=FakeSampler)
    assert len(runs) == 1 and "remeasured" not in c

    records[:] = [dict(ok, reasons=["hw_slowdown"])]    # several ranks: no retry, reported as is
    runs.clear()
    out, c = bench.timed_region(None, lambda: runs.append(1) or len(runs), retry=False,
                                sampler=FakeSampler)
    assert len(runs) == 1 and c["reasons"] == ["hw_slowdown"]
