"""The weight-streaming dp4a kernel that runs W8A8 linear calls of at most 2
token rows by default and of up to 8 under PRISM_LINEAR_PATH=gemv (decode
steps, answer rows of a restricted last layer): bit for bit against the
oracle and against the tcgen05 and mma.sync kernels
(StartLux-Prism, "Bitwise consistency is not lossless quantization": exact
int32 accumulation, fixed epilogue -- so every kernel gives the same bits).

Covers every row-count instance (1, 2, 4 and 8 rows, and the counts in
between), ragged channel counts (not a multiple of the 4 channels a warp
owns) and K tails (not a multiple of the 512 bytes a warp reads per step),
strided operands, in-place residual, the int32 extremes at the largest K,
and the decode shape at full size."""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_util import dev, dev_bf16, host, host_bits, padded

import deterministic_w8a8_int8_gb300 as prism

pytestmark = pytest.mark.gpu


def _problem(M, N, K, seed, residual=True):
    rng = np.random.default_rng(seed)
    x = wl.bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    w = wl.draw_weights(rng, (N, K), "uniform")
    ws = rng.uniform(0.001, 0.02, N).astype(np.float32)
    r = wl.bf16_bits(rng.standard_normal((M, N), dtype=np.float32)) if residual else None
    return x, w, ws, r


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


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 7, 8])
@pytest.mark.parametrize("N,K", [(1027, 5120), (6, 16), (130, 528), (64, 17408)])
def test_gemv_matches_oracle(cuda_device, monkeypatch, M, N, K):
    monkeypatch.setenv("PRISM_LINEAR_PATH", "gemv")   # the library's own choice is dp4a up to 2 rows
    x, w, ws, r = _problem(M, N, K, 100 * M + N)
    q, a = prism.prism_quant_act(dev_bf16(x))
    assert prism.prism_w8a8_kernel_kind(M, N, K) == 4
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    out = prism.prism_w8a8_linear(q, a, dev(w), dev(ws), residual=dev_bf16(r), acc_out=acc)
    torch.cuda.synchronize()
    out_o, acc_o = oracle.w8a8_linear(host(q), host(a), w, ws, r)
    assert np.array_equal(host(acc), acc_o)
    assert np.array_equal(host_bits(out), out_o)


@pytest.mark.parametrize("M,N,K", [(8, 1536, 5120), (3, 520, 2064), (1, 5120, 17408)])
def test_three_kernels_agree_on_few_rows(cuda_device, M, N, K):
    x, w, ws, r = _problem(M, N, K, 7 + M)
    q, a = prism.prism_quant_act(dev_bf16(x))
    W, S, R = dev(w), dev(ws), dev_bf16(r)
    kinds = {p: _with_path(p, lambda: prism.prism_w8a8_kernel_kind(M, N, K)) for p in ("gemv", "tc", "mma")}
    assert kinds == {"gemv": 4, "tc": 3, "mma": 1}
    outs = {p: _with_path(p, lambda: prism.prism_w8a8_linear(q, a, W, S, residual=R)) for p in kinds}
    torch.cuda.synchronize()
    assert torch.equal(outs["gemv"].view(torch.int16), outs["tc"].view(torch.int16))
    assert torch.equal(outs["gemv"].view(torch.int16), outs["mma"].view(torch.int16))


def test_gemv_strided_and_in_place(cuda_device, monkeypatch):
    monkeypatch.setenv("PRISM_LINEAR_PATH", "gemv")
    M, N, K = 5, 300, 1040
    x, w, ws, r = _problem(M, N, K, 9)
    q0, a = prism.prism_quant_act(dev_bf16(x))
    Q = padded(M, K, K + 32, torch.int8)
    Q.copy_(q0)
    W = padded(N, K, K + 16, torch.int8)
    W.copy_(dev(w))
    O = padded(M, N, N + 3, torch.bfloat16)            # odd output stride
    O.copy_(dev_bf16(r))
    prism.prism_w8a8_linear(Q, a, W, dev(ws), residual=O, out=O)   # residual added in place
    torch.cuda.synchronize()
    out_o, _ = oracle.w8a8_linear(host(q0), host(a), w, ws, r)
    assert np.array_equal(host_bits(O), out_o)


def test_gemv_int32_extremes_at_max_k(cuda_device, monkeypatch):
    monkeypatch.setenv("PRISM_LINEAR_PATH", "gemv")
    M, N, K = 2, 8, 133136
    q = torch.full((M, K), 127, dtype=torch.int8, device="cuda")
    q[1] = -127
    w = torch.full((N, K), 127, dtype=torch.int8, device="cuda")
    w[1::2] = -127
    a = torch.full((M,), 1.0, dtype=torch.float32, device="cuda")
    s = torch.full((N,), 1.0, dtype=torch.float32, device="cuda")
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    prism.prism_w8a8_linear(q, a, w, s, acc_out=acc)
    torch.cuda.synchronize()
    top = K * 127 * 127
    assert top <= 2**31 - 1
    expect = np.array([[top, -top] * 4, [-top, top] * 4], np.int64)
    assert np.array_equal(host(acc).astype(np.int64), expect)


def test_decode_full_size_all_rows(cuda_device):
    """The decode shape (K = 17408, N = 5120) for 1 and 8 rows: every output
    against the oracle, and row m the same whatever the other rows are."""
    c = wl.make_linear("decode_m64_k17408_n5120")
    W, S = dev(c.w), dev(c.w_scale)
    outs = {}
    for M in (1, 8):
        q, a = prism.prism_quant_act(dev_bf16(c.x_bits[:M]), dev(c.inv_s))
        R = dev_bf16(c.residual_bits[:M])
        outs[M] = prism.prism_w8a8_linear(q, a, W, S, residual=R)
        torch.cuda.synchronize()
        q_o, a_o = oracle.quant_act(c.x_bits[:M], c.inv_s)
        out_o, _ = oracle.w8a8_linear(q_o, a_o, c.w, c.w_scale, c.residual_bits[:M])
        assert np.array_equal(host_bits(outs[M]), out_o)
    assert torch.equal(outs[8][:1].view(torch.int16), outs[1].view(torch.int16))
