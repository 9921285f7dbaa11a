"""The multi-GPU mode on CPU, as world-size-2 gloo process groups.

The decode path shards by sequence (each sequence's cache lives with it), so N GPUs run N
replicas with no exchange on the data path. Two things are checked: (1) the benchmark's replica
bookkeeping -- barriers, the maximum of each measured time over the ranks, the whole-job rate;
(2) that sharding is exact: every rank runs the oracle's decode step of both flows on its own
shard of the batch, and the shards' logits and appended cache entries equal the whole batch's,
bit for bit (the oracle stands in for the GPU step, which is tested against it elsewhere)."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

WORLD = 2


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, port):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(WORLD),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    return dist


def _timing_worker(rank, port, q):
    dist = _init(rank, port)
    try:
        import bench
        r, w, lr = bench.Replicas.from_env()
        reps = bench.Replicas(r, w, "cpu")
        reps.barrier()
        got = reps.max(1.0 + rank, 5.0 - 3.0 * rank, 2.5)
        reps.barrier()
        q.put((rank, (r, w, lr), got, reps.rate(32, 0.004)))
    finally:
        dist.destroy_process_group()


def _shard_worker(rank, port, q):
    dist = _init(rank, port)
    try:
        from tests.test_replicas_gloo import _oracle_step
        shard = list(range(rank, 4, WORLD))
        q.put((rank, shard, _oracle_step(shard)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _run(target):
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=target, args=(r, port, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    out = [q.get(timeout=240) for _ in range(WORLD)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(out, key=lambda x: x[0])


def _workload():
    from dfsynth import workloads as W
    return W.TINY_F32.replace(batch=4, ctx_len=0, ctx_lo=3, ctx_hi=40, n_kv_heads=2)


def _oracle_step(rows):
    """The oracle's decode step of both flows for the sequences `rows` of the batch."""
    import oracle as O
    from tests import gpu_harness as H
    w = _workload()
    caches = []
    for l in range(w.n_layers):
        K = H.host_f64(w, f"L{l}.K").reshape(w.cache_shape())[rows].copy()
        V = H.host_f64(w, f"L{l}.V").reshape(w.cache_shape())[rows].copy()
        caches.append(O.DenseCache(K=K, V=V))
    glob = {"E1": H.LazyRows(w, "E1"), "E2": H.LazyRows(w, "E2"), "W_lm": H.host_f64(w, "W_lm"),
            "g_final": H.host_f64(w, "g_final")}
    r = O.decode_step(H.hparams(w), glob, H.LazyLayers(w), caches, w.tokens()[rows], w.seq_lens()[rows],
                      aux_on=True, mirror=True)
    return {"logits": r["logits"], "k_new": r["k_new"], "v_new": r["v_new"]}


def test_replica_timing_bookkeeping_gloo():
    out = _run(_timing_worker)
    for rank, env, got, rate in out:
        assert env == (rank, WORLD, rank)
        assert got == [2.0, 5.0, 2.5]  # each value's maximum over both ranks, on every rank
        assert rate == pytest.approx(WORLD * 32 / 0.004)


def test_sequence_shards_equal_the_whole_batch_gloo():
    out = _run(_shard_worker)
    whole = _oracle_step(list(range(4)))
    covered = []
    for rank, shard, r in out:
        covered += shard
        assert np.array_equal(r["logits"], whole["logits"][:, shard])
        assert np.array_equal(r["k_new"], whole["k_new"][:, shard])
        assert np.array_equal(r["v_new"], whole["v_new"][:, shard])
    assert sorted(covered) == [0, 1, 2, 3]
