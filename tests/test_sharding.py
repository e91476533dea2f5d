"""Multi-process (gloo, world size 2, CPU) checks of the sequence-sharding
host logic: shards partition the batch, per-shard results keyed by the global
sequence index reassemble into the whole-batch result, and the benchmark's
max-over-ranks time reduction behaves."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from speculative_decoding_verification_online_gb300.sharding import shard_bounds, weak_scaling_offset


def test_shard_bounds_partition():
    for B in (0, 1, 5, 64, 1023):
        for ws in (1, 2, 3, 8):
            spans = [shard_bounds(B, ws, r) for r in range(ws)]
            assert spans[0][0] == 0 and spans[-1][1] == B
            for (a, b), (c, _) in zip(spans, spans[1:]):
                assert b == c and a <= b
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shard_bounds(4, 2, 2)
    assert weak_scaling_offset(64, 3) == 192


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, ws, port, result_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import workloads
    from oracle import oracle as O
    w = workloads.make("b16_v32000_bf16", seed=5, B=6, gate="half")
    lo, hi = shard_bounds(w.B, ws, rank)
    out = O.verify(workloads.to_numpy_logits(w.Lt[lo:hi]), workloads.to_numpy_logits(w.Ld[lo:hi]),
                   w.D[lo:hi].numpy(), w.T, w.gate[lo:hi].numpy(), w.tau[lo:hi].numpy(),
                   seed=w.philox_seed, seq_offset=lo)
    parts = [None] * ws
    dist.all_gather_object(parts, {k: v for k, v in out.items()})
    t = torch.tensor([1.0 + rank], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    if rank == 0:
        merged = {k: np.concatenate([p[k] for p in parts]) for k in parts[0]}
        full = O.verify(workloads.to_numpy_logits(w.Lt), workloads.to_numpy_logits(w.Ld),
                        w.D.numpy(), w.T, w.gate.numpy(), w.tau.numpy(), seed=w.philox_seed)
        ok = all(np.array_equal(merged[k], full[k]) for k in full)
        with open(os.path.join(result_dir, "ok"), "w") as f:
            f.write(f"{int(ok)} {t.item()}")
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_shards_reassemble_the_whole_batch(tmp_path, monkeypatch):
    ws = 2
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    monkeypatch.setenv("PYTHONPATH", root + os.pathsep + os.environ.get("PYTHONPATH", ""))
    mp.start_processes(_worker, args=(ws, _free_port(), str(tmp_path)), nprocs=ws, join=True,
                       start_method="spawn")
    ok, tmax = open(tmp_path / "ok").read().split()
    assert ok == "1"
    assert float(tmax) == 2.0
