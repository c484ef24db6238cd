"""Multi-rank path on CPU: two gloo ranks shard a batch by request; each
verifies its share with its global request indices (the oracle stands in for
the GPU kernels, which take the same offset as request_offset), and the
gathered outputs equal the unsharded result.  Also the max-over-ranks timing
reduction the benchmark uses."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, result_path):
    import sys
    sys.path.insert(0, ROOT)
    import oracle
    from speculative_decoding_verification_51_gb300 import sharding
    from speculative_decoding_verification_51_gb300 import workloads as W
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        w = W.make_workload(2)                      # same seeded batch on every rank
        lo, hi = sharding.shard(w.B, rank, world)
        part = W.to_numpy(w.subset(list(range(lo, hi))))
        r = oracle.spec_verify(**part, req_index=np.arange(lo, hi))
        ids = sharding.gather_rows(torch.from_numpy(r["out_ids"]))
        nacc = sharding.gather_rows(torch.from_numpy(r["out_num_accepted"]))
        slowest = sharding.max_over_ranks(1.0 + rank)
        total = sharding.sum_over_ranks(float(hi - lo))
        if rank == 0:
            full = oracle.spec_verify(**W.to_numpy(w))
            ok = (np.array_equal(ids.numpy(), full["out_ids"]) and
                  np.array_equal(nacc.numpy(), full["out_num_accepted"]) and
                  slowest == float(world) and total == float(w.B))
            with open(result_path, "w") as f:
                f.write("ok" if ok else "mismatch")
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_sharded_oracle_equals_unsharded(world, tmp_path):
    out = tmp_path / "result.txt"
    mp.spawn(_worker, args=(world, _free_port(), str(out)), nprocs=world, join=True)
    assert out.read_text() == "ok"


def test_shard_bounds():
    from speculative_decoding_verification_51_gb300 import sharding
    for B in (0, 1, 7, 256):
        for world in (1, 2, 3, 8):
            spans = [sharding.shard(B, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == B
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
    assert sharding.weak_offset(3, 256) == 768
    assert sharding.max_over_ranks(2.5) == 2.5  # no process group: identity
