"""The pages' multi-rank ring protocol, emulated with CPU ranks over gloo.

Each rank i holds the query chunk Q_i and starts with its own K_i, V_i
("Training Long-Context Models Without OOM: Ring Attention", "Ring Attention
Demystified", steps 1-2).  Before computing on the chunk it holds, it posts
a non-blocking send of that chunk to rank (i + 1) % N and a receive from
rank (i - 1) % N (step 3), computes the partial while the transfer is in
flight (step 4) and merges it into its running (O, LSE); after N - 1 hops it
has seen every chunk (step 5; "Context Parallelism" guide, section 2).  The
per-step partial and the merge are the fp64 oracle's.

These tests cover the host-side exchange logic with world sizes 2 and 4: the
visit order against the schedule, coverage, exactness against unchunked
attention, and injected protocol faults (wrong direction, a dropped partial)
that the checks must catch.  No GPU is involved.
"""
import math
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q, k, v, causal, scale, fault, out_dir):
    os.environ["OMP_NUM_THREADS"] = "1"
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}",
                            rank=rank, world_size=world)
    B, H, S, d = q.shape
    C = S // world
    rows = slice(rank * C, (rank + 1) * C)
    q_i = q[:, :, rows]
    # the chunk in hand travels with its chunk id
    held = torch.cat([k[:, :, rows], v[:, :, rows]], dim=2).contiguous()
    held_j = torch.tensor([rank], dtype=torch.int64)
    o_run = np.zeros((B, H, C, d))
    lse_run = np.full((B, H, C), -np.inf)
    log = []
    if fault == "reverse":
        dst, src = (rank - 1) % world, (rank + 1) % world
    else:
        dst, src = (rank + 1) % world, (rank - 1) % world
    for t in range(world):
        j = int(held_j.item())
        reqs = []
        if t < world - 1:
            nxt = torch.empty_like(held)
            nxt_j = torch.empty_like(held_j)
            reqs = [dist.isend(held, dst), dist.isend(held_j, dst),
                    dist.irecv(nxt, src), dist.irecv(nxt_j, src)]
        skipped = causal and j > rank
        log.append((t, j, oracle.KIND_LOCAL if j == rank else
                    (oracle.KIND_SKIP if skipped else oracle.KIND_FULL)))
        drop = fault == "drop" and rank == world - 1 and t == 1
        if not skipped and not drop:
            kj = held[:, :, :C].numpy()
            vj = held[:, :, C:].numpy()
            for b in range(B):
                for h in range(H):
                    o_p, l_p = oracle.partial(q_i[b, h].numpy(), rank * C, kj[b, h], vj[b, h],
                                              j * C, causal, scale)
                    o_m, l_m = oracle.merge(o_run[b, h], lse_run[b, h], o_p, l_p)
                    o_run[b, h], lse_run[b, h] = o_m, l_m
        for r in reqs:
            r.wait()
        if reqs:
            held, held_j = nxt, nxt_j
    np.savez(os.path.join(out_dir, f"rank{rank}.npz"), o=o_run, lse=lse_run, log=np.array(log))
    dist.barrier()
    dist.destroy_process_group()


def _run(world, causal, fault, tmp_path, S=48, d=5):
    g = torch.Generator().manual_seed(7 + world)
    q = torch.randn(1, 2, S, d, generator=g, dtype=torch.float64)
    k = torch.randn(1, 2, S, d, generator=g, dtype=torch.float64)
    v = torch.randn(1, 2, S, d, generator=g, dtype=torch.float64)
    scale = 1.0 / math.sqrt(d)
    mp.start_processes(_rank_main, args=(world, _free_port(), q, k, v, causal, scale, fault,
                                         str(tmp_path)),
                       nprocs=world, join=True, start_method="spawn")
    outs = [np.load(os.path.join(tmp_path, f"rank{r}.npz")) for r in range(world)]
    o = np.concatenate([x["o"] for x in outs], axis=2)
    lse = np.concatenate([x["lse"] for x in outs], axis=2)
    logs = [[tuple(e) for e in x["log"].tolist()] for x in outs]
    o_ref, lse_ref = oracle.naive_fwd(q.numpy(), k.numpy(), v.numpy(), causal, scale)
    return o, lse, logs, o_ref, lse_ref


def _protocol_ok(world, causal, logs):
    """Visit order equals the schedule and coverage is complete."""
    for i in range(world):
        if logs[i] != oracle.ring_visits(world, causal, i):
            return False
    pairs = {(i, j) for i in range(world) for _, j, kind in logs[i] if kind != oracle.KIND_SKIP}
    want = world * (world + 1) // 2 if causal else world * world
    return len(pairs) == want


@pytest.mark.parametrize("world", [2, 4])
@pytest.mark.parametrize("causal", [False, True])
def test_ring_ranks_exact(world, causal, tmp_path):
    o, lse, logs, o_ref, lse_ref = _run(world, causal, None, tmp_path)
    assert _protocol_ok(world, causal, logs)
    np.testing.assert_allclose(o, o_ref, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, atol=1e-12)


def test_ring_ranks_wrong_direction_is_caught(tmp_path):
    # Sending left instead of right visits j = i, i+1, ...: the order check
    # fails even where the merged values still agree (non-causal).
    o, lse, logs, o_ref, _ = _run(4, False, "reverse", tmp_path)
    assert not _protocol_ok(4, False, logs)


def test_ring_ranks_dropped_partial_is_caught(tmp_path):
    o, lse, logs, o_ref, lse_ref = _run(2, False, "drop", tmp_path)
    assert np.abs(lse - lse_ref).max() > 1e-3
