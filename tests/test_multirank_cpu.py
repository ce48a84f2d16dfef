"""The multi-rank side of the path on the CPU, with 2 gloo ranks.

Tokens are independent, so N GPUs each take a token shard (or, in bench.py's weak
scaling, a full per-GPU batch) and nothing is exchanged in the forward. The one
cross-token quantity is the RMSNorm weight gradient: summed over the shards it
must equal the gradient over all tokens. The rank bookkeeping of
rope_qkv_prologue_gb300.replicas (token shards, the gradient sum, the max of
the per-rank times, total bytes over ranks) is checked here as well.
"""

import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch
    import torch.distributed as dist

    import oracle.prologue as P
    from rope_qkv_prologue_gb300 import replicas
    import workloads
    from workloads import bits_u16 as u16

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = workloads.gqa_inputs(24, 8, 2, 64, seed=77, rope_base=5e5, pos_high=131072, with_grads=True)
        L = P.PackedLayout("interleaved", 8, 2, 64)
        xq, xk, _ = P.split_heads(L, u16(wl.packed_rows()))
        sl = slice(*replicas.token_shard(wl.T, rank, world))           # this rank's token shard
        r = P.prologue_bwd(L, u16(wl.dq)[sl], u16(wl.dk)[sl], u16(wl.dv)[sl], xq[sl], xk[sl], wl.pos.numpy()[sl],
                           wl.w_q.numpy(), wl.w_k.numpy(), wl.eps, wl.rope_base)
        dw = torch.from_numpy(np.concatenate([r["dw_q"], r["dw_k"]]))
        replicas.sum_over_ranks(dw)  # the data-parallel gradient all-reduce
        shard_dp = torch.from_numpy(r["dpacked"])
        gathered = [torch.empty_like(shard_dp) for _ in range(world)]
        dist.all_gather(gathered, shard_dp)
        ms = replicas.max_over_ranks([1.0 + rank, 10.0 - rank], "cpu")
        if rank == 0:
            out.put({"dw": dw.numpy(), "dpacked": torch.cat(gathered).numpy(), "ms": ms})
    finally:
        dist.destroy_process_group()


def test_token_shards_and_dw_allreduce_match_the_whole_batch():
    import oracle.prologue as P
    import workloads
    from workloads import bits_u16 as u16

    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    wl = workloads.gqa_inputs(24, 8, 2, 64, seed=77, rope_base=5e5, pos_high=131072, with_grads=True)
    L = P.PackedLayout("interleaved", 8, 2, 64)
    xq, xk, _ = P.split_heads(L, u16(wl.packed_rows()))
    full = P.prologue_bwd(L, u16(wl.dq), u16(wl.dk), u16(wl.dv), xq, xk, wl.pos.numpy(), wl.w_q.numpy(),
                          wl.w_k.numpy(), wl.eps, wl.rope_base)
    want = np.concatenate([full["dw_q"], full["dw_k"]])
    assert np.allclose(res["dw"], want, rtol=1e-12, atol=1e-12 * np.abs(want).max())
    assert np.array_equal(res["dpacked"], full["dpacked"])   # per-token results do not depend on sharding
    assert res["ms"] == [2.0, 10.0]                          # max over ranks, element-wise


def test_whole_job_throughput_counts_every_rank():
    from rope_qkv_prologue_gb300 import replicas

    assert replicas.whole_job_gbs(1e9, 1, 1.0) == pytest.approx(1000.0)
    assert replicas.whole_job_gbs(1e9, 4, 2.0) == pytest.approx(2000.0)


def test_token_shards_cover_the_batch_once():
    from rope_qkv_prologue_gb300 import replicas

    for T in (0, 1, 7, 16384, 16385):
        for world in (1, 2, 3, 8):
            spans = [replicas.token_shard(T, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == T
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            assert max(b - a for a, b in spans) - min(b - a for a, b in spans) <= 1
    with pytest.raises(ValueError):
        replicas.token_shard(10, 2, 2)
