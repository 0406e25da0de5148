"""Multi-rank host logic of bench.py on CPU: two gloo ranks.

The bench runs one replica of the prefill per GPU (the path has no exchange
step); the job's throughput counts every rank's tokens over the slowest
rank's time, and the reference arm runs on rank 0 only."""
import io
import json
import os
import socket
import sys
import contextlib

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank, world, port):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)


def _aggregate_worker(rank, world, port, q):
    _env(rank, world, port)
    import bench
    import torch.distributed as dist
    w, r, _, pg = bench.dist_setup()
    assert (w, r) == (world, rank) and pg is not None
    seconds = [1.0, 2.5][rank]
    q.put((rank, bench.aggregate(pg, seconds, tokens_per_rank=1000, steps=4, device="cpu")))
    dist.destroy_process_group()


def _reference_worker(rank, world, port, q):
    _env(rank, world, port)
    import bench
    import torch.distributed as dist
    args = bench.parse(["--impl", "reference", "--steps", "1", "--warmup", "0", "--gpus", str(world)])
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(args)
    q.put((rank, buf.getvalue()))
    if dist.is_initialized():
        dist.destroy_process_group()


def _run(target, world=2):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=target, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=600) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    return out


def test_aggregate_counts_all_ranks_over_slowest():
    out = _run(_aggregate_worker)
    for rank in (0, 1):
        value, ms_per_step, t_max = out[rank]
        assert t_max == 2.5
        assert value == pytest.approx(2 * 1000 * 4 / 2.5)
        assert ms_per_step == pytest.approx(2500.0 / 4)


def test_reference_arm_runs_on_rank_zero_only():
    out = _run(_reference_worker)
    assert out[1] == ""
    line = json.loads(out[0].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_cpu_baseline_reports_all_cores_and_one_core():
    """The CPU-baseline leg on a small layer: both runs time the oracle as it
    stands, the one-core figure comes from one unit scaled to all of them."""
    sys.path.insert(0, ROOT)
    import bench
    from linear_attention_linearization_gb300 import inputs
    w = inputs.Workload("case", 2, 4, 2, 16, 96, 8, 16, 8 + 2 * 6, 6, 16)
    q, k, v, Wf = inputs.make_inputs(w, seed=1)
    r, keep, thr = bench.cpu_baseline(q, k, v, Wf, w, 64)
    assert keep["y"].shape == (w.B, w.Hq, 64, w.d) and thr == r["cores"]
    assert r["kind"] == "oracle" and r["unit"] == "tokens/s" and r["value"] > 0
    assert 1 <= r["cores"] <= w.B * w.Hkv and r["seconds"] > 0
    one = r["one_core"]
    assert one["cores"] == 1 and one["value"] > 0 and one["unit"] == "tokens/s"
    json.dumps(r)


def test_cpu_decode_baseline_runs_the_oracle_decode_step():
    sys.path.insert(0, ROOT)
    import bench
    from linear_attention_linearization_gb300 import inputs
    w = inputs.Workload("case", 16, 4, 2, 16, 200, 8, 16, 8 + 2 * 6, 6, 16)
    r = bench.cpu_decode_baseline(w, seed=3, steps=4)
    assert r["kind"] == "oracle" and r["unit"] == "tokens/s" and r["value"] > 0 and r["ms_per_step"] > 0
    assert 1 <= r["cores"] <= w.Hkv
    json.dumps(r)


def test_parity_object_of_the_bench_line():
    """The bench's parity check on the host: the oracle's own output rounded to
    bf16 and its own selection pass; a selection changed outside a near tie is
    flagged, and a perturbed output shows its relative error."""
    sys.path.insert(0, ROOT)
    import numpy as np
    import torch
    import bench
    from linear_attention_linearization_gb300 import inputs
    from oracle import brute
    w = inputs.Workload("case", 1, 4, 2, 16, 96, 8, 16, 8 + 2 * 6, 6, 16)
    q, k, v, Wf = inputs.make_inputs(w, seed=2)
    keep = {}
    bench.oracle_sample(q, k, v, Wf, w, w.N, 1, keep)
    out = torch.from_numpy(keep["y"]).to(torch.bfloat16)
    sel = torch.from_numpy(np.stack([brute.select(keep["scores"][b], w.C, w.lam, w.T_max)
                                     for b in range(w.B)]).astype(np.int32))
    p = bench.parity_vs_oracle(out, sel, w, w.N, keep, 1)
    assert p["within_tolerance"] and p["max_err_rel"] < 2 ** -8 and p["sel_exact_outside_ties"]
    assert p["sel_differs_in_near_ties"] == 0
    bad = sel.clone()
    bad[0, 0, 0, 0] = next(x for x in range(w.C) if x not in sel[0, 0, 0].tolist())
    p = bench.parity_vs_oracle(out, bad, w, w.N, keep, 1)
    assert not p["sel_exact_outside_ties"]
    out2 = out.clone()
    out2[0, 1, 50, 3] += 0.5 * float(np.abs(keep["y"]).max())
    p = bench.parity_vs_oracle(out2, sel, w, w.N, keep, 1)
    assert 0.45 < p["max_err_rel"] < 0.55 and not p["within_tolerance"]
