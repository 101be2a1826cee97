"""Host logic of bench.py without a GPU: the cross-rank aggregation (two gloo
ranks on the CPU), the clock-record parser and the roofline inputs."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms, units = bench.aggregate(1.0 + rank, 100 * (rank + 1), world)
    q.put((rank, ms, units))
    dist.destroy_process_group()


def test_aggregate_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(2))
    assert all(ms == 2.0 and units == 300 for _, ms, units in res)


def test_aggregate_single_rank_identity():
    assert bench.aggregate(3.5, 7, 1) == (3.5, 7)


def test_clock_summary_parser(tmp_path):
    c = bench.ClockSampler(0)
    f = tmp_path / "c.csv"
    f.write_text("0, 1900, 2070, 900.1, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n"
                 "0, 1950, 2070, 910.0, 0x0, Not Active, Not Active, Not Active, Not Active\n"
                 "0, 1850, 2070, 920.0, 0x0, Not Active, Not Active, Not Active, Not Active\n")

    class F:
        name = str(f)
    c.file = F()
    s = c.summary()
    assert s["sm_mhz"] == 1900 and s["sm_max_mhz"] == 2070 and s["reasons"] == ["sw_power_cap"]


def test_traffic_note_requires_matching_source(tmp_path, monkeypatch):
    note = tmp_path / "t.md"
    note.write_text(f"kernel_source_sha256_16: {bench.kernel_source_hash()}\ndram_bytes_per_launch: 1.5e8\n")
    monkeypatch.setattr(bench, "TRAFFIC_NOTE", str(note))
    assert bench.recorded_traffic() == 1.5e8
    note.write_text("kernel_source_sha256_16: 0000\ndram_bytes_per_launch: 1.5e8\n")
    assert bench.recorded_traffic() is None


def test_warmup_floor():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "1"])


def test_reference_arm_line(capsys):
    # the oracle arm prints one JSON line with the contract's keys (one layer,
    # one timed step: a few seconds on the host cores)
    import json
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3", "--ref-layers", "1"])
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    r = json.loads(lines[0])
    assert r["impl"] == "reference" and r["metric"] == bench.METRIC and r["unit"] == bench.UNIT
    assert r["higher_is_better"] is True and r["value"] > 0 and r["steps"] == 1 and r["warmup"] == 3
    assert r["config"]["workload"] == "stack69_n64_h48_pool96_pad4"
    assert r["cpu_baseline"]["kind"] == "oracle" and r["cpu_baseline"]["value"] == r["value"]
    assert r["e2e"] == {"value": r["value"], "unit": r["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_print_nothing(capsys, monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3", "--ref-layers", "1"])
    assert capsys.readouterr().out.strip() == ""
