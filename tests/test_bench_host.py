"""bench.py host logic: flop and byte accounting, the traffic record's source check, and
the multi-rank barrier / max-over-ranks path on CPU (gloo, world size 2)."""

import json
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_numbers.txt")


def _golden():
    out = []
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].split()
        if line:
            out.append((line[0], [int(x) for x in line[1:]]))
    return out


def test_headline_flops_follow_the_page_convention():
    # 4 * B * H * N^2 * d, halved for causal.
    assert bench.workload_flops(1, 12, 8192, 64, True) == 4 * 12 * 8192 ** 2 * 64 / 2
    assert bench.workload_flops(1, 1, 256, 64, False) == 4 * 256 ** 2 * 64


def test_row_flops_sum_to_the_exact_causal_count():
    N, d = 97, 64
    exact = bench.row_flops(np.arange(N), d, N, True)
    assert exact == 4 * d * N * (N + 1) / 2
    assert bench.row_flops(np.arange(N), d, N, False) == 4 * d * N * N


@pytest.mark.parametrize("kind,args", _golden())
def test_page_numbers(kind, args):
    if kind == "scores_per_head":
        T, stated = args
        assert abs(T * T - stated) / stated < 0.05
    elif kind == "naive_bytes":
        n, b = args
        assert 5 * 4 * n * n == b
    elif kind == "online_floor_bytes":
        n, d, b = args
        assert 4 * 4 * n * d == b


def test_recorded_traffic_requires_matching_source(tmp_path, monkeypatch):
    prof = tmp_path / "p.md"
    prof.write_text(f"traffic_bytes_per_launch: 123456\nsource_sha256: {bench.source_sha256()}\n")
    monkeypatch.setattr(bench, "TRAFFIC_PROFILE", str(prof))
    assert bench.recorded_traffic() == (123456, "ncu capture of this source")
    prof.write_text("traffic_bytes_per_launch: 123456\nsource_sha256: " + "0" * 64 + "\n")
    assert bench.recorded_traffic()[0] is None


def test_peaks_fall_back_when_file_missing(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, src = bench.load_peaks()
    assert src == "fallback" and peaks["bf16_tflops"] == 1900.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"bf16_tflops": 1941.2, "hbm_gbs": 6772.5}))
    peaks, src = bench.load_peaks()
    assert src == "measured" and peaks["bf16_tflops"] == 1941.2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    r, w, _ = bench.dist_env()
    g = bench.Group(w)
    g.barrier()
    m = g.max(float(10 + r * 5))
    g.barrier()
    g.close()
    q.put((r, w, m))


def test_two_rank_barrier_and_max_over_ranks():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 2, 15.0), (1, 2, 15.0)]


def test_reference_arm_prints_one_line(capsys, monkeypatch):
    # A tiny stand-in workload keeps this a CPU test of the arm's logic.
    monkeypatch.setattr(bench, "WORKLOAD", {**bench.WORKLOAD, "H": 2, "N": 256})
    bench.main(["--impl", "reference", "--steps", "3", "--warmup", "3", "--reference-seconds", "2"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "TFLOP/s"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_decode_bytes_count_k_v_once_and_q_o():
    # bf16: K and V (Nk x d each) read once per head, q read and o written (Nq x d each).
    assert bench.decode_bytes(16, 12, 1, 8192, 64) == 2 * 16 * 12 * (2 * 8192 * 64 + 2 * 64)
    assert bench.decode_bytes(1, 1, 4, 100, 64, esz=4) == 4 * (2 * 100 * 64 + 2 * 4 * 64)


def test_decode_traffic_record_is_keyed_to_the_decode_source(tmp_path):
    prof = tmp_path / "d.md"
    prof.write_text(f"traffic_bytes_per_launch: 777\nsource_sha256: {bench.source_sha256(bench.DECODE_SOURCE)}\n")
    assert bench.recorded_traffic(str(prof), bench.DECODE_SOURCE) == (777, "ncu capture of this source")
    assert bench.recorded_traffic(str(prof), bench.TC_SOURCE)[0] is None
