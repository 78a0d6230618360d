"""The mma.sync weight-streaming kernel that runs W8A8 linear calls of 9 to
16 token rows by default and of 1 to 16 under PRISM_LINEAR_PATH=stream
(decode steps, answer rows of a restricted last layer): bit for bit
against the oracle, across split-K factors and against the other kernels
(StartLux-Prism, "Bitwise consistency is not lossless quantization": int8
products accumulate exactly in int32 and split-K partial sums stay integers,
so every kernel and every split gives the same bits).

Covers both token-tile instances (1 and 2 tiles of 8 rows, and the counts
in between), ragged channel counts (not a multiple of a CTA's 16) and K tails
(not a multiple of the 128-K step or of the warps' quarters),
fp32 chunks at the 2^24 boundary, the int32 extremes at the largest K,
explicit splits with empty pieces, the automatic split of narrow weights
(workspace left zero), strided operands and in-place residual, the
restricted last layer's residual rows, the accumulator-only mode of the
tensor-parallel combine, and the decode shape at full size for every row
count and split."""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_util import dev, dev_bf16, host, host_bits, padded

import deterministic_w8a8_int8_gb300 as prism

pytestmark = pytest.mark.gpu


@pytest.fixture
def stream_path(monkeypatch):
    monkeypatch.setenv("PRISM_LINEAR_PATH", "stream")


def _problem(M, N, K, seed, residual=True, dist="normal"):
    rng = np.random.default_rng(seed)
    x = wl.bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    w = wl.draw_weights(rng, (N, K), dist)
    ws = rng.uniform(0.001, 0.02, N).astype(np.float32)
    r = wl.bf16_bits(rng.standard_normal((M, N), dtype=np.float32)) if residual else None
    return x, w, ws, r


def _run(q, a, W, S, R=None, split=0, acc=True, out=None, ws=None):
    M, N = q.shape[0], W.shape[0]
    acc_t = torch.full((M, N), -7, dtype=torch.int32, device="cuda") if acc else None
    o = prism.prism_w8a8_linear(q, a, W, S, residual=R, out=out, acc_out=acc_t, split_k=split, workspace=ws)
    torch.cuda.synchronize()
    return o, acc_t


@pytest.mark.parametrize("M", [1, 2, 7, 8, 9, 15, 16])
@pytest.mark.parametrize("N,K", [(130, 528), (257, 2064), (1, 16), (1040, 1088)])
@pytest.mark.parametrize("residual", [True, False])
def test_stream_matches_oracle(cuda_device, stream_path, M, N, K, residual):
    x, w, ws, r = _problem(M, N, K, 1000 * M + N + K, residual)
    q, a = prism.prism_quant_act(dev_bf16(x))
    assert prism.prism_w8a8_kernel_kind(M, N, K) == 5
    out, acc = _run(q, a, dev(w), dev(ws), None if r is None else dev_bf16(r))
    out_o, acc_o = oracle.w8a8_linear(host(q), host(a), w, ws, r)
    assert np.array_equal(host(acc), acc_o)
    assert np.array_equal(host_bits(out), out_o)


@pytest.mark.parametrize("M", [3, 16])
@pytest.mark.parametrize("split", [0, 1, 2, 3, 7, 16, 33, 64])
def test_stream_split_k_bit_identical(cuda_device, stream_path, M, split):
    """K = 2064 has 17 steps of 128 K: splits 7, 16, 33 and 64 leave pieces
    of uneven length and empty ones (which must still arrive on the
    counter)."""
    N, K = 390, 2064
    x, w, ws, r = _problem(M, N, K, 31 + M)
    q, a = prism.prism_quant_act(dev_bf16(x))
    wsp = prism.new_workspace(M, N, K, split, "cuda")
    for _ in range(2):     # the workspace must come back zero for the second call
        out, acc = _run(q, a, dev(w), dev(ws), dev_bf16(r), split=split, ws=wsp)
        out_o, acc_o = oracle.w8a8_linear(host(q), host(a), w, ws, r)
        assert np.array_equal(host(acc), acc_o)
        assert np.array_equal(host_bits(out), out_o)
        if wsp is not None:
            assert int(wsp.count_nonzero()) == 0


@pytest.mark.parametrize("M", [2, 16])
def test_stream_automatic_split_of_a_narrow_weight(cuda_device, stream_path, M):
    """390 channels are 25 tiles of 16, too few for the SMs: the automatic
    choice splits K = 17408 in pieces (workspace needed and left zero)."""
    N, K = 390, 17408
    assert prism.prism_w8a8_workspace_bytes(M, N, K, 0) > 0
    x, w, ws, r = _problem(M, N, K, 77 + M)
    q, a = prism.prism_quant_act(dev_bf16(x))
    wsp = prism.new_workspace(M, N, K, 0, "cuda")
    out_o, acc_o = oracle.w8a8_linear(host(q), host(a), w, ws, r)
    for _ in range(2):
        out, acc = _run(q, a, dev(w), dev(ws), dev_bf16(r), ws=wsp)
        assert np.array_equal(host(acc), acc_o)
        assert np.array_equal(host_bits(out), out_o)
        assert int(wsp.count_nonzero()) == 0


@pytest.mark.parametrize("M", [5, 16])
def test_stream_chunks_exact_at_2_pow_24(cuda_device, stream_path, M):
    """All +-127 operands give chunk partial sums up to 1024 * 16129 =
    16,516,096 (near 2^24); single +-1 terms beside them must stay exact."""
    K = 4096 + 1024 + 64
    rng = np.random.default_rng(M)
    N = 200
    q = np.where(rng.random((M, K)) < 0.5, 127, -127).astype(np.int8)
    w = np.full((N, K), 127, np.int8)
    w[1::3] = -127
    w[2::3] = np.where(rng.random((N // 3 + 1, K))[: w[2::3].shape[0]] < 0.5, 127, -127)
    q[:, 1000] = 1
    w[:, 1000] = 1
    a = rng.uniform(0.001, 0.01, M).astype(np.float32)
    s = rng.uniform(0.001, 0.02, N).astype(np.float32)
    out_o, acc_o = oracle.w8a8_linear(q, a, w, s, None)
    for split in (0, 1, 5):
        out, acc = _run(dev(q), dev(a), dev(w), dev(s), split=split)
        assert np.array_equal(host(acc), acc_o)
        assert np.array_equal(host_bits(out), out_o)


def test_stream_int32_extremes_at_max_k(cuda_device, stream_path):
    M, N, K = 12, 24, 133136
    q = torch.full((M, K), 127, dtype=torch.int8, device="cuda")
    q[1::2] = -127
    w = torch.full((N, K), 127, dtype=torch.int8, device="cuda")
    w[1::2] = -127
    a = torch.full((M,), 1.0, dtype=torch.float32, device="cuda")
    s = torch.full((N,), 1.0, dtype=torch.float32, device="cuda")
    top = K * 127 * 127
    assert top <= 2**31 - 1
    sign = np.where(np.arange(M)[:, None] % 2 == np.arange(N)[None, :] % 2, 1, -1)
    for split in (0, 1, 16):
        _, acc = _run(q, a, w, s, split=split)
        assert np.array_equal(host(acc).astype(np.int64), sign * top)


def test_stream_strided_and_in_place(cuda_device, stream_path):
    M, N, K = 20, 300, 1040
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


@pytest.mark.parametrize("M,N,K", [(16, 1536, 5120), (11, 520, 2064), (9, 384, 17408)])
def test_stream_agrees_with_other_kernels(cuda_device, monkeypatch, M, N, K):
    x, w, ws, r = _problem(M, N, K, 7 + M)
    q, a = prism.prism_quant_act(dev_bf16(x))
    W, S, R = dev(w), dev(ws), dev_bf16(r)
    outs = {}
    for path, kind in (("stream", 5), ("tc", 3), ("mma", 1)):
        monkeypatch.setenv("PRISM_LINEAR_PATH", path)
        assert prism.prism_w8a8_kernel_kind(M, N, K) == kind
        outs[path], _ = _run(q, a, W, S, R, acc=False)
    assert torch.equal(outs["stream"].view(torch.int16), outs["tc"].view(torch.int16))
    assert torch.equal(outs["stream"].view(torch.int16), outs["mma"].view(torch.int16))


@pytest.mark.parametrize("n", [3, 13])
def test_stream_restricted_rows(cuda_device, stream_path, n):
    """The last layer on answer rows: residual rows of the full hidden state
    through an index list, against the oracle."""
    M_x, K, N = 300, 2048, 640
    rng = np.random.default_rng(n)
    x = wl.bf16_bits(rng.standard_normal((M_x, K), dtype=np.float32))
    w = wl.draw_weights(rng, (N, K), "normal")
    ws = rng.uniform(0.001, 0.02, N).astype(np.float32)
    res = wl.bf16_bits(rng.standard_normal((M_x, N), dtype=np.float32))
    rows = rng.choice(M_x, size=n, replace=False).astype(np.int32)
    q, a = prism.prism_quant_act_rows(dev_bf16(x), dev(rows))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = prism.prism_w8a8_linear_rows(q, a, dev(w), dev(ws), dev_bf16(res), dev(rows), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    q_o, a_o, _ = oracle.quant_act_rows(x, rows, None)
    out_o, _, e_o = oracle.w8a8_linear_rows(q_o, a_o, w, ws, res, rows)
    assert e_o == 0
    assert np.array_equal(host_bits(out), out_o)


@pytest.mark.parametrize("M", [4, 12])
def test_stream_accumulator_only(cuda_device, stream_path, M):
    """prism_w8a8_gemm_s32 (a tensor-parallel rank's exact partial sums)."""
    N, K = 700, 3072
    x, w, _, _ = _problem(M, N, K, M, residual=False)
    q, a = prism.prism_quant_act(dev_bf16(x))
    acc = prism.prism_w8a8_gemm_s32(q, dev(w))
    torch.cuda.synchronize()
    _, acc_o = oracle.w8a8_linear(host(q), host(a), w, np.ones(N, np.float32), None)
    assert np.array_equal(host(acc), acc_o)


def test_stream_decode_full_size_every_m_and_split(cuda_device, monkeypatch):
    """The decode shape (K = 17408, N = 5120) in the library's own choice of
    kernel for 1..64 rows (dp4a, weight stream, tcgen05): every output of the
    64-row call against the oracle, and every row identical across M in
    {1, 8, 16, 64} and split-K in {0, 1, 4, 8, 16}."""
    monkeypatch.delenv("PRISM_LINEAR_PATH", raising=False)
    c = wl.make_linear("decode_m64_k17408_n5120")
    W, S = dev(c.w), dev(c.w_scale)
    q_o, a_o = oracle.quant_act(c.x_bits, c.inv_s)
    out_o, _ = oracle.w8a8_linear(q_o, a_o, c.w, c.w_scale, c.residual_bits)
    for M in wl.DECODE_M:
        q, a = prism.prism_quant_act(dev_bf16(c.x_bits[:M]), dev(c.inv_s))
        R = dev_bf16(c.residual_bits[:M])
        for split in (0,) + tuple(wl.DECODE_SPLITS):
            out = prism.prism_w8a8_linear(q, a, W, S, residual=R, split_k=split)
            torch.cuda.synchronize()
            assert np.array_equal(host_bits(out), out_o[:M]), (M, split)
