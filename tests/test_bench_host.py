"""Host-side logic of bench.py that runs without a GPU: tensor chunking of the
end-to-end leg, the N > 1 replica reduction (two gloo ranks on CPU), and the
reference arm's behaviour on non-zero ranks."""
import json
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def test_chunks_cover_all_tensors_in_order():
    sizes = [5, 1, 1, 100, 3, 3, 50, 7]
    for n in (1, 2, 3, 5, 16):
        ch = bench._chunks(sizes, n)
        flat = [i for c in ch for i in c]
        assert flat == list(range(len(sizes)))
        assert 1 <= len(ch) <= n


def test_job_throughput():
    assert bench.job_throughput(1, 1000, 10, 1000.0) == 10_000
    # weak scaling: the job processes every rank's parameters in the slowest time
    assert bench.job_throughput(4, 1000, 10, 2000.0) == 20_000


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, ws, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    elapsed = [10.0, 25.0][rank]
    launches = [100, 100][rank]
    mx = bench.reduce_scalar(elapsed, "max", ws)
    sm = bench.reduce_scalar(float(launches), "sum", ws)
    out[rank] = (mx, sm, bench.job_throughput(ws, 8, 100, mx))
    dist.destroy_process_group()


def test_replica_reduction_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        mx, sm, thr = out[r]
        assert mx == 25.0          # the slowest rank's time
        assert sm == 200.0         # launches of both ranks
        assert thr == 2 * 8 * 100 / 25e-3


def test_reference_arm_nonzero_rank_does_nothing(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"]) == 0
    assert capsys.readouterr().out == ""


@pytest.mark.slow
def test_reference_arm_line(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"]) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "params/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["config"]["params"] == 8_030_261_248


def test_algorithmic_bytes_per_param():
    """Each state byte read and written once, the gradient read once: AdamW with
    8-bit rho moves 2+2+1+1+1 + 2*2/32 read and 2+1+1+1 + 2*2/32 written."""
    from quantized_optimizer_state_gb300 import workloads as wl
    adamw = wl.workload("flat_1m")
    lion = wl.workload("llama31_8b_lion")
    assert bench._algo_bytes(adamw, 8) == 12.25
    assert bench._algo_bytes(adamw, 16) == 14.25
    assert bench._algo_bytes(adamw, 8, "f32") == 14.25
    assert bench._algo_bytes(lion, 8) == 2 + 2 * (2 + 1 + 1 + 2 / 32)
    assert bench._algo_bytes(lion, 16, "f32") == 4 + 2 * (2 + 2 + 1 + 2 / 32)


def test_flat_offsets_are_aligned_and_disjoint():
    sizes = [1, 4096, 33, 0, 65537, 8]
    offs, total = bench.flat_offsets(sizes)
    assert offs[0] == 0 and all(o % 64 == 0 for o in offs)
    ends = [o + n for o, n in zip(offs, sizes)]
    assert all(e <= o2 for e, o2 in zip(ends, offs[1:])) and ends[-1] <= total
    assert total - sum(sizes) < 64 * len(sizes)
