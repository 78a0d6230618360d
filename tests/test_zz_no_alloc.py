"""prism_w8a8_linear_noalloc, the allocation-free variant of the W8A8 linear.

Some callers cannot give the library device scratch memory (a plugin host
that passes only its own buffers, a loop that must not call cudaMalloc, a
fixed memory budget).  For them the library keeps a fixed scratch array of
its own.  These tests call that entry point through the C ABI and check that
its outputs equal prism_w8a8_linear's bit for bit -- the tolerance every
linear test here uses -- on two calls in a row (the second call reuses the
shared array the first one left behind), that on a shape with shared tiles
they also equal the CPU oracle's on their own, and that shapes whose scratch
would not fit are refused.  This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

import deterministic_w8a8_int8_gb300 as prism

pytestmark = pytest.mark.gpu


def _vp(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _problem(M, N, K, seed):
    rng = np.random.default_rng(seed)
    x = wl.bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    x = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    q, a = prism.prism_quant_act(x)
    w = torch.from_numpy(wl.draw_weights(rng, (N, K), "normal")).cuda()
    ws = torch.from_numpy(rng.uniform(0.001, 0.02, N).astype(np.float32)).cuda()
    r = wl.bf16_bits(rng.standard_normal((M, N), dtype=np.float32))
    r = torch.from_numpy(r.view(np.int16)).view(torch.bfloat16).cuda()
    return q, a, w, ws, r


def _noalloc(q, a, w, ws, r, out, acc, split):
    M, K = q.shape
    N = w.shape[0]
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return prism.lib().prism_w8a8_linear_noalloc(
        _vp(q), K, _vp(a), _vp(w), K, _vp(ws), _vp(r), N, _vp(out), N, _vp(acc), M, N, K, split, st)


@pytest.mark.parametrize("M,N,K,split", [(64, 5120, 17408, 8), (304, 5120, 5120, 3), (37, 384, 256, 1),
                                         (70, 520, 2064, 0)])
def test_noalloc_matches_workspace_entry_point(cuda_device, M, N, K, split):
    q, a, w, ws, r = _problem(M, N, K, M + N + K)
    ref_acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    ref = prism.prism_w8a8_linear(q, a, w, ws, residual=r, acc_out=ref_acc, split_k=split)
    torch.cuda.synchronize()
    for _ in range(2):   # two calls in a row share the library's scratch array
        out = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
        acc = torch.zeros((M, N), dtype=torch.int32, device="cuda")
        assert _noalloc(q, a, w, ws, r, out, acc, split) == prism.PRISM_OK
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
        assert torch.equal(acc, ref_acc)


def test_noalloc_matches_oracle(cuda_device):
    """A shape whose automatic schedule shares tiles between CTAs (so the
    scratch array is used), checked against the oracle directly, twice."""
    M, N, K = 70, 520, 2064
    assert prism.prism_w8a8_workspace_bytes(M, N, K, 0) > 0
    rng = np.random.default_rng(5)
    xb = wl.bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    w = wl.draw_weights(rng, (N, K), "normal")
    ws = rng.uniform(0.001, 0.02, N).astype(np.float32)
    rb = wl.bf16_bits(rng.standard_normal((M, N), dtype=np.float32))
    qo, ao = oracle.quant_act(xb, None)
    outo, acco = oracle.w8a8_linear(qo, ao, w, ws, rb)
    q = torch.from_numpy(qo).cuda()
    a = torch.from_numpy(ao).cuda()
    W, S = torch.from_numpy(w).cuda(), torch.from_numpy(ws).cuda()
    R = torch.from_numpy(rb.view(np.int16)).view(torch.bfloat16).cuda()
    for _ in range(2):
        out = torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda")
        acc = torch.full((M, N), -1, dtype=torch.int32, device="cuda")
        assert _noalloc(q, a, W, S, R, out, acc, 0) == prism.PRISM_OK
        torch.cuda.synchronize()
        assert np.array_equal(acc.cpu().numpy(), acco)
        assert np.array_equal(out.cpu().view(torch.int16).numpy().view(np.uint16), outo)


def test_noalloc_refuses_scratch_beyond_its_array(cuda_device):
    M, N, K = 2048, 2048, 1024          # split 4 would need ~16 MiB of scratch
    assert prism.prism_w8a8_workspace_bytes(M, N, K, 4) > prism.PRISM_NOALLOC_SCRATCH_BYTES
    q, a, w, ws, r = _problem(M, N, K, 3)
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(q, a, w, ws, r, out, None, 4) == prism.PRISM_ERR_UNSUPPORTED
    # split 1 needs no scratch and is accepted for the same shape
    assert _noalloc(q, a, w, ws, r, out, None, 1) == prism.PRISM_OK
    torch.cuda.synchronize()
    ref = prism.prism_w8a8_linear(q, a, w, ws, residual=r, split_k=1)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
