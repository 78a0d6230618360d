"""The tensor-parallel integer combine as real ranks on CPU (gloo): each
rank holds a K-shard of the activations and of the weight, runs the
package's tp_row_parallel_linear with the oracle as its per-rank steps, and
must end with the one-device layer's output bit for bit (StartLux-Prism,
"Bitwise consistency is not lossless quantization": int32 partial sums are
combined before scaling).  Two and three ranks, even and uneven shards."""
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


def _inputs(seed=31, M=20, K=384, N=96):
    sys.path.insert(0, ROOT)
    import workloads as wl
    rng = np.random.default_rng(seed)
    x = wl.bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    x[:, 200] = wl.bf16_bits(rng.standard_normal(M, dtype=np.float32) * 50)   # outlier in one shard
    inv_s = rng.uniform(0.5, 2.0, K).astype(np.float32)
    w = wl.draw_weights(rng, (N, K), "normal")
    ws = rng.uniform(0.001, 0.02, N).astype(np.float32)
    res = wl.bf16_bits(rng.standard_normal((M, N), dtype=np.float32))
    return x, inv_s, w, ws, res


class OracleOps:
    """The per-rank steps on the CPU oracle, on torch CPU tensors."""

    @staticmethod
    def act_amax(x, inv_s):
        import oracle
        import torch
        return torch.from_numpy(oracle.act_amax(x.numpy().view(np.uint16), inv_s.numpy()))

    @staticmethod
    def quant_act_amax(x, inv_s, amax):
        import oracle
        import torch
        q, a = oracle.quant_act_amax(x.numpy().view(np.uint16), inv_s.numpy(), amax.numpy())
        return torch.from_numpy(q), torch.from_numpy(a)

    @staticmethod
    def gemm_s32(q, w):
        import oracle
        import torch
        return torch.from_numpy(oracle.gemm_s32(q.numpy(), w.numpy()))

    @staticmethod
    def epilogue(acc, a_scale, w_scale, residual):
        import oracle
        import torch
        r = None if residual is None else residual.numpy().view(np.uint16)
        return torch.from_numpy(oracle.epilogue(acc.numpy(), a_scale.numpy(), w_scale.numpy(), r).view(np.int16))


def _rank(rank, world, port, bounds, q):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import deterministic_w8a8_int8_gb300 as prism
        x, inv_s, w, ws, res = _inputs()
        b0, b1 = bounds[rank], bounds[rank + 1]
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
        out = prism.tp_row_parallel_linear(t(x[:, b0:b1].view(np.int16)), t(inv_s[b0:b1]), t(w[:, b0:b1]), t(ws),
                                           t(res.view(np.int16)), ops=OracleOps)
        # this rank's partial alone, scaled: what skipping the combine would give
        amax = OracleOps.act_amax(t(x[:, b0:b1].view(np.int16)), t(inv_s[b0:b1]))
        qq, aa = OracleOps.quant_act_amax(t(x[:, b0:b1].view(np.int16)), t(inv_s[b0:b1]), amax)
        alone = OracleOps.epilogue(OracleOps.gemm_s32(qq, t(w[:, b0:b1])), aa, t(ws), t(res.view(np.int16)))
        q.put((rank, out.numpy().view(np.uint16).copy(), alone.numpy().view(np.uint16).copy()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("bounds", [[0, 192, 384], [0, 48, 384], [0, 128, 208, 384]])
def test_ranks_reproduce_one_device_output(bounds):
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
    x, inv_s, w, ws, res = _inputs()
    qf, af = oracle.quant_act(x, inv_s)
    ref, _ = oracle.w8a8_linear(qf, af, w, ws, res)
    for rank, out, alone in got:
        assert np.array_equal(out, ref), rank
        assert not np.array_equal(alone, ref), rank     # the combine is what makes it exact
