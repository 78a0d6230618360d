"""W4A8 on packed 4-bit weights on the GPU, bit for bit against the oracle
and against the W8A8 linear on the unpacked codes (StartLux-Prism, "Compute
shared evidence once": Q4_K_M files and a W4A8 run; the contraction stays
exact int32 and the epilogue fixed).

Covers the few-row path (the dp4a kernel unpacking nibbles in registers) for
every row-count instance, the unpack + tcgen05 path for more rows (balanced
schedule and explicit split-K, and the mma.sync kernel), codes -8 and 7 at
the largest K, every byte pattern through the unpack kernel, strided packed
rows, workspace rules."""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_util import dev, dev_bf16, host, host_bits, padded

import deterministic_w8a8_int8_gb300 as prism

pytestmark = pytest.mark.gpu


def _problem(M, N, K, seed):
    rng = np.random.default_rng(seed)
    x = wl.bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    codes = wl.draw_w4_codes(rng, (N, K))
    ws = rng.uniform(0.005, 0.05, N).astype(np.float32)
    r = wl.bf16_bits(rng.standard_normal((M, N), dtype=np.float32))
    return x, codes, wl.pack_w4(codes), ws, r


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


def test_unpack_kernel_every_byte_pattern(cuda_device):
    b = np.tile(np.arange(256, dtype=np.uint8), (3, 4))          # [3, 1024] -> K = 2048
    w = prism.prism_unpack_w4(dev(b), 2048)
    torch.cuda.synchronize()
    assert np.array_equal(host(w), oracle.unpack_w4(b, 2048))


@pytest.mark.parametrize("M", [1, 2, 3, 4, 6, 8])
@pytest.mark.parametrize("N,K", [(1027, 5120), (64, 17408), (6, 32)])
def test_w4a8_few_rows_match_oracle(cuda_device, M, N, K):
    x, codes, w4, ws, r = _problem(M, N, K, 10 * M + N)
    q, a = prism.prism_quant_act(dev_bf16(x))
    assert prism.prism_w4a8_workspace_bytes(M, N, K, 0) == 0
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    out = prism.prism_w4a8_linear(q, a, dev(w4), dev(ws), residual=dev_bf16(r), acc_out=acc)
    torch.cuda.synchronize()
    out_o, acc_o = oracle.w4a8_linear(host(q), host(a), w4, ws, r)
    assert np.array_equal(host(acc), acc_o)
    assert np.array_equal(host_bits(out), out_o)


@pytest.mark.parametrize("M,N,K,split,path", [
    (304, 5120, 5120, 0, "auto"),       # tcgen05, balanced schedule
    (37, 384, 256, 0, "auto"),
    (600, 1024, 2048, 4, "auto"),       # explicit split-K
    (8, 1536, 5120, 0, "tc"),           # few rows forced onto unpack + tcgen05
    (5, 1536, 5120, 0, "stream"),       # few rows forced onto unpack + the mma.sync weight stream
    (300, 640, 1024, 0, "mma"),
])
def test_w4a8_more_rows_match_w8a8_and_oracle(cuda_device, M, N, K, split, path):
    x, codes, w4, ws, r = _problem(M, N, K, M + N + K)
    q, a = prism.prism_quant_act(dev_bf16(x))
    W4, S, R = dev(w4), dev(ws), dev_bf16(r)

    def run():
        need = prism.prism_w4a8_workspace_bytes(M, N, K, split)
        assert need >= N * K
        out = prism.prism_w4a8_linear(q, a, W4, S, residual=R, split_k=split)
        ref = prism.prism_w8a8_linear(q, a, dev(codes), S, residual=R, split_k=split)
        torch.cuda.synchronize()
        return out, ref

    out, ref = _with_path(path, run)
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    out_o, _ = oracle.w4a8_linear(host(q), host(a), w4, ws, r)
    assert np.array_equal(host_bits(out), out_o)


@pytest.mark.parametrize("M", [2, 40])
def test_w4a8_extremes_at_max_k(cuda_device, M):
    K, N = 133120, 8
    q = torch.full((M, K), 127, dtype=torch.int8, device="cuda")
    q[1::2] = -127
    w4 = torch.full((N, K // 2), 0x88, dtype=torch.uint8, device="cuda")   # every code -8
    w4[1::2] = 0x77                                                         # every code 7
    a = torch.ones(M, dtype=torch.float32, device="cuda")
    s = torch.ones(N, dtype=torch.float32, device="cuda")
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    prism.prism_w4a8_linear(q, a, w4, s, acc_out=acc)
    torch.cuda.synchronize()
    t8, t7 = K * 127 * 8, K * 127 * 7
    row = np.array([-t8, t7] * 4, np.int64)
    expect = np.stack([row if m % 2 == 0 else -row for m in range(M)])
    assert np.array_equal(host(acc).astype(np.int64), expect)


def test_w4a8_strided_packed_rows_and_workspace_rules(cuda_device):
    M, N, K = 5, 200, 1024
    x, codes, w4, ws, r = _problem(M, N, K, 3)
    q, a = prism.prism_quant_act(dev_bf16(x))
    W4 = padded(N, K // 2, K // 2 + 48, torch.uint8, fill=0x77)
    W4.copy_(dev(w4))
    out = prism.prism_w4a8_linear(q, a, W4, dev(ws), residual=dev_bf16(r))
    torch.cuda.synchronize()
    out_o, _ = oracle.w4a8_linear(host(q), host(a), w4, ws, r)
    assert np.array_equal(host_bits(out), out_o)
    # more rows without enough workspace are refused before any launch
    M2 = 64
    q2 = torch.zeros((M2, K), dtype=torch.int8, device="cuda")
    a2 = torch.ones(M2, dtype=torch.float32, device="cuda")
    small = torch.zeros(N * K // 2, dtype=torch.uint8, device="cuda")
    with pytest.raises(prism.PrismError) as e:
        prism.prism_w4a8_linear(q2, a2, W4, dev(ws), workspace=small)
    assert e.value.status == prism.PRISM_ERR_WORKSPACE
