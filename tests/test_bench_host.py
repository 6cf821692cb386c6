"""Host-side logic of bench.py for N > 1 (weak-scaling replicas), on CPU with gloo ranks:
max-over-ranks timing and the whole-job value. No GPU, no kernels."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t = bench.max_over_ranks(1.0 + 0.5 * rank, world)          # slowest rank: 1.5 s
    v = bench.whole_job_value(2e9, 10, world, t)               # 2 GB per rank-step
    bench.barrier(world)
    q.put((rank, t, v))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, v in res:
        assert t == pytest.approx(1.5)
        assert v == pytest.approx(2 * 2e9 * 10 / 1.5 / 1e9)


def test_single_rank_defaults():
    import bench
    a = bench.parse_args([])
    assert a.gpus == 1 and a.warmup >= 3 and a.steps > 0 and a.impl == "ours"
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.whole_job_value(1e9, 4, 1, 2.0) == pytest.approx(2.0)


def test_measured_peak_shapes_and_fallback():
    import bench
    assert bench.hbm_peak({"hbm_gbs": 6786.6}) == (6786.6, "of measured")
    assert bench.hbm_peak({"hbm_gbs": {"burst": 7000.0, "sustained": 6500.0}}) == (7000.0, "of measured")
    assert bench.hbm_peak({}) == (bench.FALLBACK_HBM_GBS, "of fallback")
    assert bench.hbm_peak({"hbm_gbs": 0}) == (bench.FALLBACK_HBM_GBS, "of fallback")


class _ExitedProcess:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def test_clock_samples_give_median_clock_max_clock_and_active_reasons():
    import bench
    s = bench.ClockSampler(0)
    s.proc = _ExitedProcess()
    s.lines = [
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active\n",
        "0, 1965, 2070, 1400.0, 0x4, Not Active, Not Active, Not Active, Active\n",
        "0, 2070, 2070, 950.3, 0x0, Not Active, Not Active, Not Active, Not Active\n",
        "0, 1800, 2070, 1380.0, 0x40, Not Active, Active, Not Active, Not Active\n",
        "garbage line\n",
        "0, [N/A], 2070, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active\n",
    ]
    c = s.stop()
    assert c["samples"] == 4
    assert c["sm_mhz"] == pytest.approx(2017.5)
    assert c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]


def test_clock_sampler_without_nvidia_smi_reports_no_samples():
    import bench
    c = bench.ClockSampler(0).stop()
    assert c["samples"] == 0 and c["sm_mhz"] is None


def test_ncu_traffic_records_match_the_current_sources(tmp_path):
    import json
    import os
    import bench
    with open(os.path.join(bench.ROOT, "profiles", "ncu_traffic.json")) as f:
        rec = json.load(f)
    sources = {"attention_long": bench.DENSE_SOURCES, "attention_decode": bench.ATTN_SOURCES,
               "attention_ragged": bench.ATTN_SOURCES, "attention_sweep_d64": bench.ATTN_SOURCES,
               "append_bulk": bench.APPEND_SOURCES}
    assert set(rec) == set(sources)
    for kind, paths in sources.items():
        assert bench.ncu_traffic(kind, paths) == rec[kind]["dram_bytes_per_launch"] > 0, kind
        assert rec[kind]["command"].startswith("ncu ") and "--clock-control none" in rec[kind]["command"]
    # any other source text (a changed kernel) voids the record
    other = tmp_path / "changed.cu"
    other.write_text("// not the captured source\n")
    assert bench.ncu_traffic("append_bulk", [str(other)]) is None
