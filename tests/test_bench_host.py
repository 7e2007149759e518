"""Host-side logic of bench.py: FLOP accounting, the CPU-baseline sample, and
the multi-rank aggregation (max time over ranks, work of all ranks) run as two
gloo ranks on the CPU."""
import os
import socket

import numpy as np
import pytest

import bench
import seeded_inputs as si


def test_headline_flops():
    # 4 * B * h * d * T^2 / 2 for the causal T = 8192 workload
    assert bench.attention_flops(si.WORKLOADS[4]) == pytest.approx(2.749e11, rel=1e-3)
    w = si.WORKLOADS[4].replace(mask=si.MASK_NONE, T_q=10, T_k=20, B=1, h=1)
    assert bench.attention_flops(w) == 4 * 64 * 10 * 20


def test_row_flops_sum_to_the_causal_triangle():
    w = si.WORKLOADS[4].replace(T_q=64, T_k=64)
    t = np.arange(64)
    assert bench.row_flops(w, t) == 2 * 128 * 64 * 65 / 2


def test_oracle_sample_rows_cover_every_head():
    w = si.WORKLOADS[4]
    rows, t = bench.oracle_sample_rows(w, 1024, 3)
    assert len(rows) == w.B * w.h * len(t)
    assert set(rows // w.T_q) == set(range(w.B * w.h))
    assert np.all(rows % w.T_q == np.tile(t, w.B * w.h))


def test_reference_line_fields(capsys, monkeypatch):
    # tiny stand-in workload so the test stays fast
    monkeypatch.setattr(bench, "WORKLOAD", si.WORKLOADS[4].replace(B=1, h=2, T_q=256, T_k=256))
    args = bench.parse(["--impl", "reference", "--steps", "2", "--warmup", "3",
                        "--oracle-stride", "8"])
    assert bench.run_reference(args, 0, 1) == 0
    import json
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["value"] > 0


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [2.0, 3.0][rank]
    ms_max = bench.max_over_ranks(ms, dist, "cpu")
    q.put((rank, ms_max, bench.whole_job_value(1e12, world, ms_max)))
    dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for _, ms_max, value in res:
        assert ms_max == 3.0
        assert value == pytest.approx(2 * 1e12 / 3e-3 / 1e12)


def test_visible_pairs_and_mha_flops():
    w = si.WORKLOADS[2].replace(B=1, h=1, T_q=4, T_k=4, d_model=64)
    assert bench.visible_pairs(w, None) == 1 + 2 + 3 + 4          # causal triangle
    w2 = si.WORKLOADS[1].replace(B=2, h=3, T_q=5, T_k=7, d_model=64)
    lens = np.array([7, 2], dtype=np.int32)
    assert bench.visible_pairs(w2, lens) == 3 * 5 * (7 + 2)
    # projections 2MKN each: Q and O with M = B*T_q, K and V with M = B*T_k
    hd = w2.h * 64
    proj = 2 * 10 * 64 * hd + 2 * 2 * 14 * 64 * hd + 2 * 10 * hd * 64
    assert bench.mha_flops(w2, lens) == pytest.approx(proj + 256 * 3 * 5 * 9)


def test_decode_bytes_counts_visible_rows():
    w = si.WORKLOADS[5].replace(B=2, h=3, T_q=2, T_k=100)
    # rows of 64 bf16 = 128 bytes; K and V of every visible key, q and o rows
    assert bench.decode_bytes(w, np.array([10, 200], dtype=np.int32)) == 3 * (
        (10 + 100) * 2 * 128 + 2 * 2 * 2 * 128)
    assert bench.decode_bytes(w.replace(mask=si.MASK_NONE), None) == 3 * (
        200 * 2 * 128 + 2 * 2 * 2 * 128)
