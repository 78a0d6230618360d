"""The last layer restricted to the positions needed for answers, on the GPU
(StartLux-Prism, "Compute shared evidence once").  The quantiser gathers the
answer rows of the full activation matrix; the linear adds the residual rows
of the full hidden state that an index list names.  Every output is compared
bit for bit with the oracle, and the restricted layer with the full layer's
rows at the answer positions (the restriction must not change an answer).

Shapes cover both orientations of the tensor-core kernel (few rows: weights
on the MMA's M side; many rows: tokens on it), explicit split-K, the
mma.sync kernel, the dp4a weight-streaming kernel that few-row calls take by
default, every quantiser team size, repeated and unordered indices,
out-of-range indices (error bit, NaN rows, the rest untouched) and the
overlap refusal."""
import ctypes
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_util import dev, dev_bf16, host, host_bits

import deterministic_w8a8_int8_gb300 as prism

pytestmark = pytest.mark.gpu


def _inputs(M_x, K, N, seed):
    rng = np.random.default_rng(seed)
    x = wl.bf16_bits(rng.standard_normal((M_x, K), dtype=np.float32))
    x[:, rng.choice(K, size=max(1, K // 100), replace=False)] = wl.bf16_bits(
        rng.standard_normal((M_x, max(1, K // 100)), dtype=np.float32) * 30)
    inv_s = rng.uniform(0.5, 2.0, K).astype(np.float32)
    w = wl.draw_weights(rng, (N, K), "normal")
    ws = rng.uniform(0.001, 0.02, N).astype(np.float32)
    res = wl.bf16_bits(rng.standard_normal((M_x, N), dtype=np.float32))
    return rng, x, inv_s, w, ws, res


def _with_path(path, fn):
    old = os.environ.get("PRISM_LINEAR_PATH")
    if path in ("mma", "tc", "gemv", "stream"):
        os.environ["PRISM_LINEAR_PATH"] = path
    else:                      # the library's own choice
        os.environ.pop("PRISM_LINEAR_PATH", None)
    try:
        return fn()
    finally:
        if old is None:
            os.environ.pop("PRISM_LINEAR_PATH", None)
        else:
            os.environ["PRISM_LINEAR_PATH"] = old


@pytest.mark.parametrize("M_x,K,n", [
    (37, 256, 5),          # 32-thread teams
    (304, 2048, 3),        # 64-thread teams: one request's three answer positions
    (300, 4096, 40),       # 128-thread teams
    (2048, 5120, 192),     # 256-thread teams: 64 clients x 3 answers
    (64, 17408, 17),       # five vectors per thread
    (2048, 5120, 2000),    # many gathered rows per CTA (the prefetching row loop)
])
def test_quant_rows_match_oracle(cuda_device, M_x, K, n):
    rng, x, inv_s, *_ = _inputs(M_x, K, 8, M_x + K)
    rows = rng.integers(0, M_x, size=n).astype(np.int32)
    rows[0], rows[-1] = M_x - 1, 0
    if n > 3:
        rows[1] = rows[2]                      # a repeat
    q_o, a_o, e_o = oracle.quant_act_rows(x, rows, inv_s)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q, a = prism.prism_quant_act_rows(dev_bf16(x), dev(rows), dev(inv_s), err=err)
    torch.cuda.synchronize()
    assert e_o == 0 and int(err.item()) == 0
    assert np.array_equal(host(q), q_o)
    assert np.array_equal(host(a).view(np.uint32), a_o.view(np.uint32))


@pytest.mark.parametrize("M_x,K,N,n,split,path", [
    (304, 5120, 5120, 3, 0, "tc"),        # forest request: o_proj on its 3 answer rows
    (2048, 5120, 5120, 192, 0, "tc"),     # 64 clients x 3 answers
    (600, 1024, 640, 300, 0, "tc"),       # enough rows for the token-side orientation
    (304, 2048, 1536, 3, 4, "tc"),        # explicit split-K
    (300, 1024, 640, 40, 0, "mma"),       # the mma.sync kernel
    (304, 5120, 5120, 3, 0, "auto"),      # the library's choice for 3 rows: the mma.sync weight stream
    (304, 5120, 5120, 3, 0, "gemv"),      # the dp4a weight stream
    (2048, 17408, 5120, 8, 0, "gemv"),
    (2048, 17408, 5120, 8, 0, "stream"),
    (2048, 5120, 5120, 2, 0, "auto"),     # the library's choice for 2 rows: the dp4a weight stream
])
def test_restricted_layer_matches_oracle_and_full_rows(cuda_device, M_x, K, N, n, split, path):
    rng, x, inv_s, w, ws, res = _inputs(M_x, K, N, 3 * M_x + N)
    rows = np.sort(rng.choice(M_x, size=n, replace=False)).astype(np.int32)[::-1].copy()
    X, I, W, S, R = dev_bf16(x), dev(inv_s), dev(w), dev(ws), dev_bf16(res)
    rows_d = dev(rows)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def run():
        q, a = prism.prism_quant_act_rows(X, rows_d, I, err=err)
        out = prism.prism_w8a8_linear_rows(q, a, W, S, R, rows_d, split_k=split, err=err)
        qf, af = prism.prism_quant_act(X, I)
        full = prism.prism_w8a8_linear(qf, af, W, S, residual=R, split_k=split)
        torch.cuda.synchronize()
        return out, full

    out, full = _with_path(path, run)
    assert int(err.item()) == 0
    # the restriction changes no answer: the full layer's rows, bit for bit
    assert np.array_equal(host_bits(out), host_bits(full)[rows])
    q_o, a_o, _ = oracle.quant_act_rows(x, rows, inv_s)
    out_o, _, e_o = oracle.w8a8_linear_rows(q_o, a_o, w, ws, res, rows)
    assert e_o == 0
    assert np.array_equal(host_bits(out), out_o)


@pytest.mark.parametrize("n", [3, 300])
def test_out_of_range_rows_flag_and_poison_only_their_rows(cuda_device, n):
    M_x, K, N = 304, 1024, 640
    rng, x, inv_s, w, ws, res = _inputs(M_x, K, N, 77 + n)
    rows = rng.integers(0, M_x, size=n).astype(np.int32)
    bad = [1] if n == 3 else [1, 100, 299]
    rows[bad] = [-1, M_x, 1 << 30][:len(bad)] if n > 3 else [-1]
    X, I, W, S, R = dev_bf16(x), dev(inv_s), dev(w), dev(ws), dev_bf16(res)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q, a = prism.prism_quant_act_rows(X, dev(rows), I, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == prism.PRISM_DEV_ERR_ROW_RANGE
    q_o, a_o, e_o = oracle.quant_act_rows(x, rows, inv_s)
    assert e_o == oracle.ERR_ROW_RANGE
    assert np.array_equal(host(q), q_o)
    assert np.array_equal(host(a).view(np.uint32), a_o.view(np.uint32))   # NaN rows included

    # the linear on valid inputs with invalid residual indices
    good = rows.copy()
    good[bad] = 0
    q, a = prism.prism_quant_act_rows(X, dev(good), I)
    err.zero_()
    out = prism.prism_w8a8_linear_rows(q, a, W, S, R, dev(rows), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == prism.PRISM_DEV_ERR_ROW_RANGE
    q_o, a_o, _ = oracle.quant_act_rows(x, good, inv_s)
    out_o, _, e_o = oracle.w8a8_linear_rows(q_o, a_o, w, ws, res, rows)
    assert e_o == oracle.ERR_ROW_RANGE
    assert np.array_equal(host_bits(out), out_o)
    assert (host_bits(out)[bad] == 0x7FC0).all()


def test_rows_argument_checks(cuda_device):
    M_x, K, N = 64, 256, 128
    rng, x, inv_s, w, ws, res = _inputs(M_x, K, N, 5)
    X, W, S, R = dev_bf16(x), dev(w), dev(ws), dev_bf16(res)
    rows = dev(np.arange(4, dtype=np.int32))
    q, a = prism.prism_quant_act_rows(X, rows)
    lib = prism.lib()
    P = ctypes.c_void_p
    stream = P(torch.cuda.current_stream().cuda_stream)
    # the output overlapping the residual is refused
    st = lib.prism_w8a8_linear_rows(P(q.data_ptr()), K, P(a.data_ptr()), P(W.data_ptr()), K, P(S.data_ptr()),
                                    P(R.data_ptr()), N, M_x, P(rows.data_ptr()), P(R.data_ptr()), N, None,
                                    4, N, K, 0, None, 0, None, stream)
    assert st == prism.PRISM_ERR_INVALID_ARG
    # the residual and its indices are required
    st = lib.prism_w8a8_linear_rows(P(q.data_ptr()), K, P(a.data_ptr()), P(W.data_ptr()), K, P(S.data_ptr()),
                                    None, N, M_x, P(rows.data_ptr()), P(R.data_ptr()), N, None,
                                    4, N, K, 0, None, 0, None, stream)
    assert st == prism.PRISM_ERR_INVALID_ARG
    # an empty selection enqueues nothing
    assert lib.prism_quant_act_rows(P(X.data_ptr()), K, M_x, P(rows.data_ptr()), 0, None, K,
                                    P(q.data_ptr()), K, P(a.data_ptr()), None, stream) == prism.PRISM_OK
    torch.cuda.synchronize()
