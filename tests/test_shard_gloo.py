"""Multi-rank path on CPU: two gloo ranks each take half of the KV heads, run the
forward and backward on their shard (the oracle stands in for the device), and
the gathered shards equal the single-process result exactly: the path shards
over KV heads with no exchange."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from block_sparse_attention_nsa_gb300.shard import kv_head_range, sequence_groups, slice_heads


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, result_path):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from workloads import WorkloadConfig, make_inputs
    cfg = WorkloadConfig("shard", (120, 77), 4, 2, 16, 16, 4, "bf16", "uniform", 1.0, 3,
                         with_dout=True)
    inp = make_inputs(cfg)
    lo, hi = kv_head_range(cfg.h_k, world, rank)
    f64 = {k: inp[k].double().numpy() for k in ("q", "k", "v", "dout")}
    f64["sel_idx"] = inp["sel_idx"]
    part = slice_heads(f64, cfg.h_k, cfg.g, lo, hi)
    out, lse = oracle.fwd(inp["cu_seqlens"], cfg.block, part["sel_idx"], part["q"], part["k"],
                          part["v"], cfg.scale)
    dq, dk, dv = oracle.bwd(inp["cu_seqlens"], cfg.block, part["sel_idx"], part["q"], part["k"],
                            part["v"], part["dout"], cfg.scale)
    pieces = {"out": out, "lse": lse, "dq": dq, "dk": dk, "dv": dv}
    gathered = {}
    for name, arr in pieces.items():
        t = torch.from_numpy(np.ascontiguousarray(arr))
        bucket = [None] * world
        dist.all_gather_object(bucket, t)
        gathered[name] = bucket
    # max over ranks, as bench.py reports its step time
    tm = torch.tensor([float(rank + 1)])
    dist.all_reduce(tm, op=dist.ReduceOp.MAX)
    if rank == 0:
        full_out, full_lse = oracle.fwd(inp["cu_seqlens"], cfg.block, inp["sel_idx"], f64["q"],
                                        f64["k"], f64["v"], cfg.scale)
        fq, fk, fv = oracle.bwd(inp["cu_seqlens"], cfg.block, inp["sel_idx"], f64["q"], f64["k"],
                                f64["v"], f64["dout"], cfg.scale)
        ok = (np.array_equal(torch.cat(gathered["out"], 1).numpy(), full_out)
              and np.array_equal(torch.cat(gathered["lse"], 0).numpy(), full_lse)
              and np.array_equal(torch.cat(gathered["dq"], 1).numpy(), fq)
              and np.array_equal(torch.cat(gathered["dk"], 1).numpy(), fk)
              and np.array_equal(torch.cat(gathered["dv"], 1).numpy(), fv)
              and float(tm.item()) == float(world))
        with open(result_path, "w") as f:
            f.write("ok" if ok else "mismatch")
    dist.barrier()
    dist.destroy_process_group()


def test_kv_head_sharding_two_gloo_ranks(tmp_path):
    path = str(tmp_path / "result.txt")
    mp.start_processes(_worker, args=(2, _free_port(), path), nprocs=2, start_method="spawn")
    assert open(path).read() == "ok"


def test_partition_helpers():
    assert [kv_head_range(4, 2, r) for r in range(2)] == [(0, 2), (2, 4)]
    assert [kv_head_range(5, 3, r) for r in range(3)] == [(0, 2), (2, 4), (4, 5)]
    assert kv_head_range(2, 4, 3) == (2, 2)
    groups = sequence_groups([16384, 32768, 8192, 8192], 2)
    assert sorted(sum(groups, [])) == [0, 1, 2, 3]
    loads = [sum([16384, 32768, 8192, 8192][i] for i in gr) for gr in groups]
    assert max(loads) == 32768
    with pytest.raises(ValueError):
        kv_head_range(4, 0, 0)
