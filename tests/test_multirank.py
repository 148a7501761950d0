"""The multi-rank path of bench.py on CPU: two processes over gloo (127.0.0.1).
Each rank runs its own replica of the layer (token-parallel, no exchange), so
the only collective is the max over ranks of the step time, and the whole-job
throughput is world x tokens per rank / slowest step time."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, step_ms, out_q):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(step_ms[rank], dist, "cpu")
        value = bench.whole_job_tokens_per_s(world, 8192, slowest / 1e3)
        dist.barrier()
        out_q.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("step_ms", [(15.5, 16.25), (20.0, 12.0)])
def test_two_gloo_ranks_agree_on_slowest_step(step_ms):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, step_ms, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    slowest = max(step_ms)
    for rank, got, value in res:
        assert got == pytest.approx(slowest)
        assert value == pytest.approx(2 * 8192 / (slowest / 1e3))


def test_single_process_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_tokens_per_s(1, 8, 0.001) == pytest.approx(8000.0)


def _run_bench(args, env_extra):
    import json
    import subprocess
    env = dict(os.environ, **env_extra)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                       env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    return [json.loads(l) for l in lines]


def test_reference_arm_runs_on_rank0_only():
    """--impl reference under a 2-rank launch: rank 1 exits 0 without work and
    prints nothing; rank 0 times the oracle and prints one reference line."""
    assert _run_bench(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3"],
                      {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}) == []
    out = _run_bench(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3"],
                     {"RANK": "0", "WORLD_SIZE": "1", "LOCAL_RANK": "0"})
    assert len(out) == 1
    line = out[0]
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "tokens/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


def test_attention_reference_arm_line():
    """--impl reference for the attention workload (tiny shape, CPU only): one
    line with the attention metric, the oracle's rate and zero copy bytes."""
    out = _run_bench(["--impl", "reference", "--workload", "attn_tiny", "--steps", "1", "--warmup", "3"],
                     {"RANK": "0", "WORLD_SIZE": "1", "LOCAL_RANK": "0"})
    assert len(out) == 1
    line = out[0]
    assert line["impl"] == "reference" and line["value"] > 0 and "attention" in line["metric"]
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_attention_work_counts():
    """The bench's algorithmic work for the attention block: causal pairs
    T(T+1)/2 per head counted by brute force, projection flops from the shapes."""
    import bench
    import synth
    inp = synth.make_attn_inputs(37, 256, 4, 2, 1, Dh=128)
    w = bench.attn_work(inp)
    pairs = sum(1 for q in range(inp.T) for k in range(inp.T) if k <= q)
    assert w["attn"] == ("tensor", 4.0 * 128 * 4 * pairs)
    assert w["qkv"] == ("tensor", 2.0 * 37 * 256 * (4 + 2 * 2) * 128)
    assert w["oproj"] == ("tensor", 2.0 * 37 * 4 * 128 * 256)
    assert bench.attn_compulsory_bytes(inp) == 4 * 37 * 128 * 2 + 2 * 2 * 37 * 128 * 2 + 37 * 4 * 128 * 2


def test_bench_names_the_kernel_of_each_path():
    """The kernel the bench's roofline names for each path of the layer: the
    int8 GEMV kernels up to 16 tokens (grouped scales as the second template
    argument), the bf16 weight-streaming kernels up to 16, the paired grouped
    GEMMs from F = 16384 and T = 2048, and the same names ncu prints."""
    import bench
    import synth
    i8 = synth.make_inputs(16, 256, 512, 3, name="n", weight_dtype="int8")
    assert bench.kernel_function("up_geglu", i8)[0] == "gemv_i8_kernel<0, 0>"
    assert bench.kernel_function("down", i8)[0] == "gemv_i8_kernel<1, 0>"
    g8 = synth.make_inputs(8, 1024, 1024, 3, name="n", weight_dtype="int8", int8_scale_shape=(8, 8))
    assert bench.kernel_function("down", g8)[0] == "gemv_i8_kernel<1, 1>"
    assert bench.kernel_function("up_geglu", synth.make_inputs(17, 256, 512, 3, name="n", weight_dtype="int8"))[0] \
        == "grouped_gemm_kernel<0, 1, 1>"
    assert bench.kernel_function("up_geglu", synth.make_inputs(8, 256, 512, 3, name="n"))[0] == "decode_gemm_kernel<0>"
    big = synth.MoeInputs(**{**synth.make_inputs(16, 256, 512, 3, name="n").__dict__, "T": 2048, "F": 16384})
    assert bench.kernel_function("down", big)[0] == "grouped_gemm_kernel<1, 0, 2>"
    for role in ("up_geglu", "down"):  # every named source file exists (the traffic record's hash)
        for inp in (i8, g8, big):
            bench.source_hash(bench.kernel_function(role, inp)[1])
    assert bench.INT8_BAND_TOKENS == tuple(sorted(bench.INT8_BAND_TOKENS))
    assert max(bench.INT8_BAND_TOKENS) <= bench.GEMV_I8_MAX_T == bench.DECODE_MAX_T
