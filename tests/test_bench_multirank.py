"""The benchmark's multi-rank bookkeeping on CPU: two gloo ranks, max-over-ranks
timing and the whole-job weak-scaling rate (no GPU, no data-path collective)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 10.0 + 5.0 * rank                      # the slower rank sets the job time
    got = bench.reduce_max(ms)
    rate = bench.job_throughput(1000.0, world, got)
    q.put((rank, got, rate))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_max_and_weak_scaling():
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
    for rank, got, rate in res:
        assert got == 15.0
        assert rate == pytest.approx(2 * 1000.0 / 0.015)


def test_single_process_without_group():
    import bench
    assert bench.reduce_max(3.5) == 3.5
    assert bench.job_throughput(100.0, 1, 1000.0) == 100.0


def test_workload_options_set_query_heads_and_sizes():
    """bench.py's workload options: --q-heads changes only the query heads (64 over the
    8 kv heads of the Llama-3-8B shape is query group 8) and must be a multiple of the kv
    heads; --batch / --context set the shape."""
    import argparse
    import bench
    args = argparse.Namespace(workload=2, batch=16, context=0, bits=0, group=0, residual=0, q_heads=64)
    wl = bench.workload_spec(args)
    assert (wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.lengths) == (16, 64, 8, (32768,) * 16)
    with pytest.raises(SystemExit):
        bench.workload_spec(argparse.Namespace(**{**vars(args), "q_heads": 12}))


def test_oracle_parts_times_quantization_and_attention_apart(oracle_lib):
    """The cpu_baseline's two parts on the tiny workload: positive median times, the
    quantized token count and the attention context it reports."""
    import bench
    import synth
    wl = synth.workload(0)
    q_s, nq, a_s, L = bench.oracle_parts(wl, 2, 2, runs=3, quant_tokens=256)
    assert q_s > 0 and a_s > 0
    assert nq == 256 and L == wl.lengths[0] == 1024
