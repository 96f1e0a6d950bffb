"""bench.py host logic without a GPU: the max/sum aggregation over ranks (gloo,
world size 2), the reference arm's JSON line, peaks and traffic bookkeeping."""
import json
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, bench.aggregate(float(rank + 1), 100.0 * (rank + 1), world)))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_aggregate_two_ranks_gloo():
    """Replicas: the step time is the max over ranks, the work the sum."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert results[0] == (2.0, 300.0) and results[1] == (2.0, 300.0)


def test_aggregate_single_rank_is_identity():
    assert bench.aggregate(3.5, 7.0, 1) == (3.5, 7.0)


def test_reference_arm_json(capsys, monkeypatch):
    monkeypatch.delenv("RANK", raising=False)
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3",
                       "--ref-rows", "1"]) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["metric"] == bench.METRIC
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["config"]["workload"].startswith("dense SiTU-GLU FFN")


def test_reference_arm_other_ranks_do_nothing(capsys, monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--gpus", "2", "--impl", "reference", "--steps", "1", "--warmup", "3"]) == 0
    assert capsys.readouterr().out == ""


def test_warmup_floor():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_peaks_and_traffic(tmp_path, monkeypatch):
    peaks, src = bench.load_peaks()
    assert src in ("measured", "fallback") and peaks["hbm_gbs"] > 0
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_peaks() == (bench.FALLBACK_PEAKS, "fallback")
    assert bench.profiled_traffic("ffn_gate_up_situ", "x", 10) is None
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.txt").write_text("# c\nk abc 2.5 row f.md\n")
    assert bench.profiled_traffic("k", "abc", 4) == 10.0
    assert bench.profiled_traffic("k", "old", 4) is None  # kernel changed since the capture


def test_gpus_must_match_the_rank_count(monkeypatch):
    """--gpus N needs N ranks (one process per GPU); a single process asked for more
    GPUs refuses instead of quietly measuring one."""
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    with pytest.raises(SystemExit) as e:
        bench.main(["--gpus", "2", "--impl", "reference", "--steps", "1", "--warmup", "3"])
    assert e.value.code == 2
    monkeypatch.setenv("WORLD_SIZE", "2")
    with pytest.raises(SystemExit):
        bench.main(["--gpus", "1", "--impl", "reference", "--steps", "1", "--warmup", "3"])


def test_route_sample_covers_every_expert():
    """The grouped CPU baseline's sample: n distinct routes, seeded, holding the first and
    the last row of every non-empty expert's group (expert order, ties by flat index)."""
    import numpy as np
    import torch

    g = torch.Generator().manual_seed(3)
    ids = torch.randint(0, 50, (300, 4), generator=g, dtype=torch.int32)
    ids[ids == 7] = 8  # expert 7 without routes
    s = bench.route_sample(ids, 160, seed=0)
    flat = ids.view(-1).numpy()
    assert s.size == 160 and np.unique(s).size == 160 and (np.diff(s) > 0).all()
    assert set(np.unique(flat[s])) == set(np.unique(flat))
    assert np.array_equal(s, bench.route_sample(ids, 160, seed=0))
    for e in np.unique(flat):
        where = np.nonzero(flat == e)[0]
        assert where[0] in s and where[-1] in s
    # Fewer routes asked than the group ends: every group's first and last row is kept.
    ends = {int(i) for e in np.unique(flat) for i in np.nonzero(flat == e)[0][[0, -1]]}
    assert set(bench.route_sample(ids, 10, seed=0).tolist()) == ends


def test_accuracy_and_ulp_stats():
    """The bench's accuracy figures: error over the FFN bound 2e-2 (1 + |ref|), and bf16
    ulps of the FP64 value (2^(floor(log2 |ref|) - 7), 2^-133 below 2^-126)."""
    import math

    import numpy as np
    import torch

    ref = np.array([1.0, 2.0])
    a = bench.accuracy_stats(torch.tensor([1.0, 2.0625]), ref)
    assert math.isclose(a["max_abs_err"], 0.0625)
    assert math.isclose(a["max_err_over_bound"], 0.0625 / 0.06)
    assert math.isclose(a["rms_rel_err"], math.sqrt(0.0625 ** 2 / 5.0))
    u = bench.ulp_stats(torch.tensor([1.0 + 2.0 ** -7, 3.0, 0.0, 2.0 ** -130]),
                        np.array([1.0, 3.0, 0.0, 0.0]))
    assert math.isclose(u["max_ulp_err"], 2.0 ** 3)  # 2^-130 off a zero: 2^-130 / 2^-133
    assert math.isclose(u["frac_within_half_ulp"], 0.5)  # 3.0 and 0.0 exact
    u2 = bench.ulp_stats(torch.tensor([1.0 + 2.0 ** -7]), np.array([1.0]))
    assert math.isclose(u2["max_ulp_err"], 1.0)
