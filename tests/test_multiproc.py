"""Multi-process (world size 2, gloo on CPU) checks of the N > 1 logic.

* The row-parallel reduce: each rank computes its own pre-reduce partials (with its weight
  shard), an all-reduce sums them, and the result is the unsharded layer ("Megatron-LM
  深度学习与源码分析文档", Part 2 §2 Row Parallel: Y = sum_i Y_i).
* bench.py's aggregation: the slowest rank's time and the whole-job throughput.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _tp_reduce_worker(rank, world, port, q):
    try:
        _init(rank, world, port)
        import synth
        from oracle import layer as ol
        cfg = synth.LayerConfig("mp", batch=2, seq=16, hidden=64, heads=4, groups=2, head_dim=16, ffn=96,
                                norm="layer", act="swiglu", rope_base=1e4, bias=True)
        inp = synth.make_inputs(cfg, seed=17, affine="random", biases="random")
        sh = synth.shard_weights(cfg, inp, world, rank)
        x = ol._tokens(inp["x"], cfg)
        ya = torch.from_numpy(ol.attn_partial(cfg, world, x, sh))
        dist.all_reduce(ya)                                   # the all-reduce after the row-parallel linear
        h = x + ya.numpy() + ol.bf16_to_f64(inp["b_o"])
        ym = torch.from_numpy(ol.mlp_partial(cfg, world, h, sh))
        dist.all_reduce(ym)
        y = h + ym.numpy() + ol.bf16_to_f64(inp["b_fc2"])
        want = ol.layer_forward(cfg, inp)["y"]
        q.put((rank, float(np.max(np.abs(y - want)))))
        dist.destroy_process_group()
    except Exception as e:  # report instead of hanging the parent
        q.put((rank, repr(e)))


def _bench_agg_worker(rank, world, port, q):
    try:
        _init(rank, world, port)
        import bench
        local = [10.0 + 10.0 * rank, 5.0 * (2 - rank)]        # rank 0: (10, 10) ms, rank 1: (20, 5) ms
        mx = bench.max_over_ranks(local, dist)
        q.put((rank, mx, bench.job_throughput(world, 1e12, 4, mx[0])))
        dist.destroy_process_group()
    except Exception as e:
        q.put((rank, repr(e), None))


def _run(worker, world=2):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(out, key=lambda t: t[0])


def test_row_parallel_allreduce_of_partials_reproduces_the_layer():
    out = _run(_tp_reduce_worker)
    for rank, err in out:
        assert isinstance(err, float), err
        assert err < 1e-10


def test_bench_takes_the_slowest_rank_and_whole_job_work():
    out = _run(_bench_agg_worker)
    for rank, mx, thr in out:
        assert mx == [20.0, 10.0], mx
        assert thr == pytest.approx(2 * 1e12 * 4 / 20e-3 / 1e12)
