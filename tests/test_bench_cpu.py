"""bench.py host logic on the CPU: accounting, peaks, and the multi-rank path
(world size 2 over gloo: max-over-ranks timing and rank-0-only reporting)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_accounting_matches_the_workload():
    s = bench.SCAN
    assert (s.batch, s.dim, s.seqlen, s.dstate) == (1, 5120, 131072, 16)
    assert bench.scan_elements() == 1 * 5120 * 131072 * 16
    btd = 5120 * 131072
    # u, delta, z in + out, bf16; B, C; A, D, bias; final state
    assert bench.scan_bytes() == 8 * btd + 4 * 16 * 131072 + 5120 * 16 * 4 + 2 * 5120 * 4 + 5120 * 16 * 4
    # SFU work in the roofline's unit: N + 4 exp2-equivalents per (b, t, d)
    assert bench.scan_sfu_units() == btd * 20
    # what the kernel issues: N + 1 exp2 and one tanh per (b, t, d), at per-op rates
    rates = {"ex2": 2.0, "tanh": 0.5}
    assert bench.scan_sfu_issued_seconds(rates) == pytest.approx(btd * (17 / 2.0 + 1 / 0.5))
    assert bench.decode_bytes() == (2 * 256 * 5120 * 16 * 4 + 4 * 256 * 5120 * 2 + 2 * 256 * 16 * 2
                                    + 5120 * 16 * 4 + 2 * 5120 * 4)


def test_peaks_fall_back_when_file_missing(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.load_peaks()
    assert p["source"] == "fallback" and p["hbm_gbs"] == 6400.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6500.0, "sm_max_mhz": 2000}))
    p = bench.load_peaks()
    assert p == {"hbm_gbs": 6500.0, "sm_max_mhz": 2000.0, "source": "measured"}


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    r, w, lr = bench.dist_env()
    bench.dist_init(w, "gloo")
    m = bench.max_over_ranks(10.0 + r, w)
    bench.barrier(w)
    q.put((r, w, lr, m))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_rank_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [x[0] for x in res] == [0, 1] and all(x[1] == 2 for x in res)
    assert all(x[3] == 11.0 for x in res), res


def test_reference_arm_nonzero_rank_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_clock_summary_takes_the_median_under_load_and_every_reason():
    rows = [
        "0, 1200, 2032, 90.5, 0x0, Not Active, Not Active, Not Active, Not Active",       # before the region
        "0, 2032, 2032, 700.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2032, 900.0, 0x4, Not Active, Not Active, Not Active, Active",          # power cap
        "0, 2010, 2032, [N/A], 0x0, Not Active, Not Active, Not Active, Not Active",      # power unreadable
        "0, 2020, 2032, 880.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1150, 2032, 95.0, 0x0, Not Active, Not Active, Not Active, Not Active",       # after the region
        "garbage line",
    ]
    s = bench.summarize_clock_samples(rows)
    assert s["samples"] == 6 and s["samples_under_load"] == 3
    assert s["sm_mhz"] == 2020.0 and s["sm_max_mhz"] == 2032.0 and s["power_w_max"] == 900.0
    assert s["reasons"] == ["sw_power_cap"]
    hot = rows[:1] + ["0, 1700, 2032, 800.0, 0x40, Not Active, Active, Not Active, Not Active"]
    assert bench.summarize_clock_samples(hot)["reasons"] == ["hw_thermal_slowdown"]
    # no power readings at all: every sample counts
    nopw = [r.replace("700.0", "[N/A]").replace("900.0", "[N/A]").replace("880.0", "[N/A]")
            .replace("90.5", "[N/A]").replace("95.0", "[N/A]") for r in rows]
    s = bench.summarize_clock_samples(nopw)
    assert s["samples_under_load"] == 6 and s["power_w_max"] is None and s["sm_mhz"] == 1995.0
    assert bench.summarize_clock_samples([])["reasons"] == ["no samples"]
