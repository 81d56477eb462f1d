"""Host logic of bench.py on CPU: the max-over-ranks timing and whole-job
throughput with two gloo ranks, and the reference arm's line format."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    bench.dist_init("gloo")
    el = 1.0 + rank          # rank 1 is the slowest
    m = bench.max_over_ranks(el)
    res = bench.aggregate(bytes_per_step=1000, steps=10, world=world, seconds_max=m)
    bench.barrier()
    torch.distributed.destroy_process_group()
    q.put((rank, m, res))


def test_max_over_ranks_and_aggregate_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, m, res in got:
        assert m == 2.0
        assert res["value"] == pytest.approx(1000 * 10 * 2 / 2.0 / 1e9)
        assert res["us_per_call"] == pytest.approx(2.0 / 10 * 1e6)


def test_reference_arm_line_format():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3", "--ref-seconds", "1",
                        "--workload", "m1_nkv1_n1152"],
                       capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_roofline_bytes_formula():
    from kv_insert_gb300 import workloads as wl
    w = wl.WORKLOADS["m8_nkv8_n9216"]
    assert w.roofline_bytes() == 151_289_856
    assert wl.WORKLOADS["m1_nkv1_n1152"].roofline_bytes() == 18_893_312
    assert wl.WORKLOADS["m8_nkv16_n18432"].roofline_bytes() == 302_448_640


def test_all_cores_baseline_shards_reproduce_the_whole_call():
    """The all-cores CPU baseline runs each call as KV-head shards; the
    shards' columns and cache rows must be bit-identical to the whole call."""
    import numpy as np
    import bench
    import oracle
    from kv_insert_gb300 import workloads as wl
    w = wl.Workload("shard_check_m3_nkv2", M=3, num_kv_heads=2, max_pos=64, num_pages=4, seed=77)
    inp = wl.make_inputs(w)
    xb, Wb = wl.bits(inp["x"]), wl.bits(inp["W"])
    pos, cs = inp["positions"].numpy(), inp["cos_sin"].numpy()
    cache = wl.bits(inp["kv_cache"]).copy()
    slots = inp["slots"].numpy()
    whole, err = oracle.qkv_front(xb, Wb, pos, slots, cs, cache, w.num_kv_heads)
    assert err == 0
    for g in range(w.num_kv_heads):
        rows = bench.shard_rows(w.num_kv_heads, g)
        shard_cache = np.zeros((1, 1, 16, 128), np.uint16)
        part = bench.oracle_shard_call(xb, np.ascontiguousarray(Wb[rows]), pos, cs, shard_cache)
        assert np.array_equal(part, whole[:, rows]), g
        for t, slot in enumerate(slots):
            page, off = divmod(int(slot), 16)
            assert np.array_equal(shard_cache[0, 0, t], cache[page, g, off]), (g, t)


def test_all_cores_baseline_line():
    """The all-cores oracle baseline reports whole calls per second in the
    metric's unit, the threads it used and what it ran."""
    import bench
    from kv_insert_gb300 import workloads as wl
    w = wl.WORKLOADS["m1_nkv1_n1152"]
    line = bench.cpu_baseline_all_cores(wl.make_inputs(w), w, 0.01)
    assert line["kind"] == "oracle" and line["unit"] == bench.UNIT
    assert line["value"] > 0 and 1 <= line["cores"] <= (os.cpu_count() or 1)
    assert "KV-head shards" in line["sample"]


def test_clock_samples_are_kept_only_inside_the_timed_window():
    import bench
    """The sampler keeps nvidia-smi's own timestamps; a summary over a window
    uses only the samples taken while the timed work ran."""
    import datetime
    text = "\n".join([
        "2026/12/03 05:29:31.000, 0, 1980, 2070, 180.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/12/03 05:29:31.500, 0, 1410, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
        "2026/12/03 05:29:31.550, 0, 1430, 2070, 1395.0, 0x4, Not Active, Not Active, Not Active, Active",
        "2026/12/03 05:29:31.600, 0, 1450, 2070, 1380.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/12/03 05:29:32.500, 0, 1995, 2070, 170.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ])
    s = bench.ClockSampler(0)
    s.rows = s.parse(text)
    assert len(s.rows) == 5
    t0 = datetime.datetime(2026, 12, 3, 5, 29, 31, 400000)
    t1 = datetime.datetime(2026, 12, 3, 5, 29, 31, 700000)
    w = s.summary(t0, t1)
    assert w["samples"] == 3 and w["sm_mhz"] == 1430 and w["sm_mhz_min"] == 1410
    assert w["reasons"] == ["sw_power_cap"] and w["sm_max_mhz"] == 2070
    assert s.summary()["samples"] == 5
    assert s.summary(t1, t1) is None


def test_region_stats_per_call():
    import bench
    st = bench.region_stats([0.002, 0.001, 0.003, 0.001, 0.002], 100)
    assert st["regions"] == 5 and abs(st["us_per_call_median"] - 20.0) < 1e-9
    assert st["us_per_call_p10"] <= st["us_per_call_median"] <= st["us_per_call_p90"]
    assert abs(st["timed_seconds"] - 0.009) < 1e-12
