"""Host logic of bench.py without a GPU: the multi-rank timing reduction
(2 gloo ranks on CPU), the workload table and the JSON contract of the
reference arm."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_q):
    # CPU ranks (gloo) wherever the test runs, also on a machine with fewer
    # GPUs than ranks: no device is visible to them
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    r, ws = bench.dist_setup()
    assert (r, ws) == (rank, world) and dist.get_backend() == "gloo"
    elapsed = 10.0 + rank  # rank 1 is the slow one
    bench.barrier(ws)
    out_q.put((rank, bench.max_over_ranks(elapsed, ws)))
    # the reference arm runs on rank 0 only
    class A:
        pass
    if rank != 0:
        out_q.put((rank, bench.run_reference(A(), rank, ws)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_timing_takes_the_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in range(3)]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    maxes = sorted(v for r, v in got if isinstance(v, float))
    assert maxes == [11.0, 11.0]
    assert (1, None) in got


def test_reference_arm_prints_the_contract_line():
    res = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "3", "--warmup", "3",
                          "--ref-streams", "32"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    line = json.loads(res.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert "workload" in line["config"]


def test_workload_table_matches_the_sparsity_rule():
    from ar_image_gen_gb300.synth import WORKLOADS, n_att_for

    assert WORKLOADS["janus-b96"].N_att == 29 and WORKLOADS["janus-b96"].streams == 3072
    assert [WORKLOADS[f"sweep512-s{s}"].N_att for s in (0, 50, 75, 90, 95)] == [512, 512, 256, 102, 51]
    assert (WORKLOADS["lumina-s90-b16"].N_att, WORKLOADS["lumina-s95-b16"].N_att) == (410, 205)
    # Lumina-mGPT-shaped: 90 % and 95 % sparsity at batch 16, 32 and 54
    for s, n in ((90, 410), (95, 205)):
        for b in (16, 32, 54):
            wl = WORKLOADS[f"lumina-s{s}-b{b}"]
            assert (wl.N_att, wl.batch, wl.N_r, wl.L_dec, wl.layers) == (n, b, 2048, 4096, 32)
    assert WORKLOADS["stress-s95"].N_att == 405 and WORKLOADS["stress-s95"].L_dec == 8100
    assert n_att_for(1000, 0, 2000) == 1000
    d = WORKLOADS["janus-b96"].dense()
    assert d.N_r == d.N_att == d.L_dec == 576


def test_clock_records_that_disqualify_a_run():
    import bench

    ok = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    assert bench.clocks_rejected(ok) is None
    assert bench.clocks_rejected(dict(ok, reasons=["sw_power_cap"])) is None  # kept and noted
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        assert r in bench.clocks_rejected(dict(ok, reasons=[r]))
    assert "no throttle reason" in bench.clocks_rejected(dict(ok, sm_mhz=1400.0))
    assert bench.clocks_rejected(dict(ok, sm_mhz=1400.0, reasons=["sw_power_cap"])) is None
    assert bench.clocks_rejected({"sm_mhz": None, "sm_max_mhz": None, "reasons": []}) is None


def test_clock_sampler_parses_nvidia_smi_lines():
    import bench

    c = bench.ClockSampler(None)
    c.lines = ["2070, 2070, 900.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
               "1980, 2070, 1300.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
               "garbage"]
    s = c.summary()
    assert s["samples"] == 2 and s["sm_max_mhz"] == 2070.0 and s["reasons"] == ["sw_power_cap"]
    assert s["sm_mhz"] == (2070 + 1980) / 2


def test_step_ranges_names_runs_of_steps():
    import bench

    assert bench.step_ranges([5, 6, 7, 2, 3, 9]) == "5..7, 2..3, 9..9"
    assert bench.step_ranges([]) == ""


def test_oracle_sample_stays_inside_the_trace():
    """The CPU baseline times phase-3 steps only and never steps past the
    trace's last step: once the sample reaches L_dec it is prefilled again
    and brought back to N_r (untimed)."""
    import re

    import bench
    from ar_image_gen_gb300.synth import WORKLOADS

    wl = WORKLOADS["tiny"]
    res = bench.oracle_baseline(wl, n_streams=4, budget_s=0.3, device="cpu")
    runs = re.search(r"phase-3 steps (.*) of the 64-step trace", res["sample"]).group(1).split(", ")
    assert len(runs) >= 2  # the sample wrapped around at least once
    for r in runs:
        a, b = (int(x) for x in r.split(".."))
        assert wl.N_r <= a <= b <= wl.L_dec - 1
    assert res["value"] > 0 and res["cores"] >= 1


def test_cpu_sample_is_bounded():
    import bench
    from ar_image_gen_gb300.synth import WORKLOADS

    assert bench.cpu_sample_streams(WORKLOADS["janus-b96"]) == 3072
    assert 32 <= bench.cpu_sample_streams(WORKLOADS["stress-s95"]) <= 128
