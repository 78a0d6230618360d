"""The column-parallel candidate read-out as real ranks on CPU (gloo): each
rank holds a vocabulary shard of the LM head (contiguous rows), runs the
package's readout_column_parallel with the oracle as its per-rank steps,
and must end with the one-device read-out's logits and probabilities bit
for bit (post "把决策模型推理从 vLLM 换到 Prism", sections 方案 and 实现要点: the
softmax over the candidates needs only the candidates' logits, so the ranks
exchange T floats).  Two and three ranks, even and uneven shards, an invalid
position included."""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(seed=41, P=9, K=256, V=300):
    sys.path.insert(0, ROOT)
    import workloads as wl
    rng = np.random.default_rng(seed)
    h = wl.bf16_bits(rng.standard_normal((P, K), dtype=np.float32))
    W = rng.integers(-127, 128, size=(V, K), dtype=np.int8)
    sc = rng.uniform(0.001, 0.02, V).astype(np.float32)
    counts = rng.integers(2, 11, size=P)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    ids = np.concatenate([rng.choice(V, size=c, replace=False) for c in counts]).astype(np.int32)
    ids[off[4] + 1] = ids[off[4]]           # position 4: a duplicate id (invalid)
    return h, W, sc, off, ids


class OracleReadoutOps:
    """The per-rank steps on the CPU oracle, on torch CPU tensors."""

    @staticmethod
    def candidate_logits(hidden, inv_s, lm_shard, lm_scale_shard, v0, V, off, ids, err):
        import oracle
        import torch
        _, lg = oracle.candidate_logits_shard(hidden.numpy().view(np.uint16), None if inv_s is None else inv_s.numpy(),
                                              lm_shard.numpy(), lm_scale_shard.numpy(), v0, V, off.numpy(),
                                              ids.numpy())
        return torch.from_numpy(lg)

    @staticmethod
    def candidate_softmax(logits, off, err):
        import oracle
        import torch
        _, pr = oracle.candidate_softmax(logits.numpy(), off.numpy())
        return torch.from_numpy(pr)


def _rank(rank, world, port, bounds, q):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import deterministic_w8a8_int8_gb300 as prism
        h, W, sc, off, ids = _inputs()
        v0, v1 = bounds[rank], bounds[rank + 1]
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
        lg, pr = prism.readout_column_parallel(t(h.view(np.int16)), None, t(W[v0:v1]), t(sc[v0:v1]), v0, W.shape[0],
                                               t(off), t(ids), ops=OracleReadoutOps)
        q.put((rank, lg.numpy().copy(), pr.numpy().copy()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("bounds", [[0, 150, 300], [0, 17, 300], [0, 100, 101, 300]])
def test_ranks_reproduce_one_device_readout(bounds):
    sys.path.insert(0, ROOT)
    import oracle
    world = len(bounds) - 1
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, bounds, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    h, W, sc, off, ids = _inputs()
    rc, lg_ref, pr_ref = oracle.candidate_readout(h, None, W, sc, off, ids)
    assert rc == -4                          # the planted duplicate
    b4, e4 = off[4], off[5]
    assert np.isnan(pr_ref[b4:e4]).all()
    for rank, lg, pr in got:
        assert np.array_equal(lg.view(np.uint32), lg_ref.view(np.uint32)), rank
        assert np.array_equal(pr.view(np.uint32), pr_ref.view(np.uint32)), rank
