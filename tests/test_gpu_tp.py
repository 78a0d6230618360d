"""The tensor-parallel building blocks on the GPU (StartLux-Prism, "Bitwise
consistency is not lossless quantization": with tensor parallelism the
int32 partial sums are combined before scaling).  One GPU plays every rank
in turn -- shard maxima, codes with the shared maximum, exact int32
partials -- and the test stands in for the two all-reduces (an elementwise
max and an integer sum); the epilogue kernel then must give the one-device
layer's output bit for bit, and every piece matches the oracle.

Covers the tcgen05 kernel's accumulator-only mode in both orientations with
the balanced schedule and explicit split-K, the few-row dp4a kernel, the
mma.sync kernel, uneven shards, and the epilogue kernel's vector and element
paths (odd strides, in-place residual)."""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_util import dev, dev_bf16, host, host_bits, padded

import deterministic_w8a8_int8_gb300 as prism

pytestmark = pytest.mark.gpu


def _inputs(M, K, N, seed):
    rng = np.random.default_rng(seed)
    x = wl.bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    x[:, rng.choice(K, size=max(1, K // 100), replace=False)] = wl.bf16_bits(
        rng.standard_normal((M, max(1, K // 100)), dtype=np.float32) * 30)
    inv_s = rng.uniform(0.5, 2.0, K).astype(np.float32)
    w = wl.draw_weights(rng, (N, K), "normal")
    ws = rng.uniform(0.001, 0.02, N).astype(np.float32)
    res = wl.bf16_bits(rng.standard_normal((M, N), dtype=np.float32))
    return x, inv_s, w, ws, res


def _with_path(path, fn):
    old = os.environ.get("PRISM_LINEAR_PATH")
    if path in ("mma", "tc", "gemv", "stream"):
        os.environ["PRISM_LINEAR_PATH"] = path
    else:
        os.environ.pop("PRISM_LINEAR_PATH", None)
    try:
        return fn()
    finally:
        if old is None:
            os.environ.pop("PRISM_LINEAR_PATH", None)
        else:
            os.environ["PRISM_LINEAR_PATH"] = old


@pytest.mark.parametrize("M,K,N,bounds,split,path", [
    (304, 5120, 15360, [0, 2560, 5120], 0, "auto"),   # forest QKV over two ranks (balanced schedule)
    (600, 2048, 1536, [0, 512, 2048], 0, "auto"),     # tokens on the 128-row side, uneven shards
    (304, 2048, 1536, [0, 1024, 2048], 4, "auto"),    # explicit split-K
    (1, 17408, 5120, [0, 4352, 8704, 13056, 17408], 0, "auto"),   # a decode row over four ranks: dp4a kernel
    (8, 5120, 640, [0, 2048, 5120], 0, "auto"),      # mma.sync weight stream, accumulator-only mode
    (8, 5120, 640, [0, 2048, 5120], 0, "gemv"),      # the dp4a kernel's accumulator-only mode
    (40, 5120, 1536, [0, 2048, 5120], 0, "auto"),     # tcgen05 accumulator-only mode on 128-K stages
    (8, 2048, 640, [0, 1024, 2048], 3, "tc"),         # the same, explicit split-K
    (300, 1024, 640, [0, 512, 1024], 0, "mma"),
])
def test_ranks_reproduce_one_device_layer(cuda_device, M, K, N, bounds, split, path):
    x, inv_s, w, ws, res = _inputs(M, K, N, M + K + N)
    X, I, W, S, R = dev_bf16(x), dev(inv_s), dev(w), dev(ws), dev_bf16(res)

    def run():
        shards = list(zip(bounds[:-1], bounds[1:]))
        amax = torch.stack([prism.prism_act_amax(X[:, b0:b1].contiguous(), I[b0:b1].contiguous())
                            for b0, b1 in shards]).amax(dim=0)               # the MAX all-reduce
        parts, qs = [], []
        for b0, b1 in shards:
            q, a = prism.prism_quant_act_amax(X[:, b0:b1].contiguous(), I[b0:b1].contiguous(), amax)
            qs.append(q)
            parts.append(prism.prism_w8a8_gemm_s32(q, W[:, b0:b1].contiguous(), split_k=split))
        acc = torch.stack(parts).sum(dim=0, dtype=torch.int32)                 # the SUM all-reduce
        out = prism.prism_w8a8_epilogue(acc, a, S, residual=R)
        qf, af = prism.prism_quant_act(X, I)
        full = prism.prism_w8a8_linear(qf, af, W, S, residual=R)
        torch.cuda.synchronize()
        return amax, qs, parts, acc, out, full, qf

    amax, qs, parts, acc, out, full, qf = _with_path(path, run)
    assert torch.equal(out.view(torch.int16), full.view(torch.int16))
    # every rank's codes are the full row's codes for its columns
    assert torch.equal(torch.cat(qs, dim=1), qf)
    # against the oracle: shard maxima, partials, combined output
    out_o, acc_o, parts_o = oracle.tp_row_parallel_linear(x, inv_s, w, ws, res, bounds)
    assert np.array_equal(host(acc), acc_o)
    for p, po in zip(parts, parts_o):
        assert np.array_equal(host(p), po)
    assert np.array_equal(host_bits(out), out_o)
    assert np.array_equal(host(amax).view(np.uint32), oracle.act_amax(x, inv_s).view(np.uint32))


@pytest.mark.parametrize("M,N,ldc_pad,ldo_pad", [(304, 5120, 0, 0), (37, 1001, 3, 5), (5, 16, 0, 1)])
@pytest.mark.parametrize("residual", [None, "separate", "in_place"])
def test_epilogue_kernel_matches_oracle(cuda_device, M, N, ldc_pad, ldo_pad, residual):
    rng = np.random.default_rng(M + N + ldc_pad)
    acc = rng.integers(-(2**31) + 1, 2**31 - 1, size=(M, N), dtype=np.int64).astype(np.int32)
    acc[:, :4] = [0, 1, -(2**24) - 1, 2**31 - 1]
    a = rng.uniform(1e-4, 1e-2, M).astype(np.float32)
    s = rng.uniform(1e-3, 2e-2, N).astype(np.float32)
    r = wl.bf16_bits(rng.standard_normal((M, N), dtype=np.float32))
    A = padded(M, N, N + ldc_pad, torch.int32)
    A.copy_(dev(acc))
    O = padded(M, N, N + ldo_pad, torch.bfloat16)
    R = None
    if residual == "separate":
        R = dev_bf16(r)
    elif residual == "in_place":
        O.copy_(dev_bf16(r))
        R = O
    prism.prism_w8a8_epilogue(A, dev(a), dev(s), residual=R, out=O)
    torch.cuda.synchronize()
    ref = oracle.epilogue(acc, a, s, None if residual is None else r)
    assert np.array_equal(host_bits(O), ref)
