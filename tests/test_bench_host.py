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


_NCU_CSV = '''==PROF== Connected to process 1
"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"
"0","1","python","h","void fo::split_kernel<8>(const float *, unsigned short *, void *, long)","1","7","(256, 1, 1)","(456, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","Mbyte","999.00"
"1","1","python","h","void fo::<unnamed>::fo_fused_step_kernel<(fo::Opt)0, 8, 16, false, 8>(fo::StepParams)","1","7","(256, 1, 1)","(456, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","Gbyte","1.10"
"1","1","python","h","void fo::<unnamed>::fo_fused_step_kernel<(fo::Opt)0, 8, 16, false, 8>(fo::StepParams)","1","7","(256, 1, 1)","(456, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_write.sum","Mbyte","550.50"
'''


def test_traffic_record_is_per_parameter_and_keyed_to_the_sources(tmp_path, monkeypatch):
    """An ncu capture of one step-kernel launch on a small case becomes DRAM
    bytes per parameter; bench scales it to a table and drops it once the
    kernel sources change."""
    csv_path = tmp_path / "traffic.csv"
    csv_path.write_text(_NCU_CSV)
    monkeypatch.setattr(bench, "TRAFFIC", str(tmp_path / "traffic.json"))
    assert bench._ncu_bytes(str(csv_path)) == 1.10e9 + 550.5e6
    assert bench.main(["--record-traffic", f"{csv_path}:flat_256m", "--traffic-command", "ncu ..."]) == 0
    rec = json.load(open(tmp_path / "traffic.json"))["adamw_rho8_bf16"]
    assert rec["dram_bytes_per_param"] == (1.10e9 + 550.5e6) / (1 << 28)
    # two sizes: the slope, which cancels a constant (lines still in L2 at the end)
    small = tmp_path / "small.csv"
    small.write_text(_NCU_CSV.replace('"1.10"', '"0.50"'))
    assert bench.main(["--record-traffic", f"{csv_path}:flat_256m,{small}:flat_128m"]) == 0
    rec = json.load(open(tmp_path / "traffic.json"))["adamw_rho8_bf16"]
    assert rec["dram_bytes_per_param"] == (1.10e9 - 0.50e9) / ((1 << 28) - (1 << 27))
    assert bench._profiled_traffic("adamw", 8, "bf16", 1000) == rec["dram_bytes_per_param"] * 1000
    assert bench._profiled_traffic("lion", 8, "bf16", 1000) is None
    monkeypatch.setattr(bench, "_kernel_source_hash", lambda: "0" * 16)
    assert bench._profiled_traffic("adamw", 8, "bf16", 1000) is None


def test_per_config_covers_the_other_configurations():
    keys = {k for k, *_ in bench.PER_CONFIG}
    assert {"flat_1m", "gpt2_small", "resnet50", "llama31_8b_lion", "stress_64m_rho8",
            "stress_64m_rho16", "gpt2_small_sparse_wte"} <= keys
    flush = {k: f for k, _, _, _, f in bench.PER_CONFIG}
    assert flush["flat_1m"] and not flush["gpt2_small"]        # only the L2-sized step is flushed
    assert bench.L2_FLUSH_BYTES > 129e6
