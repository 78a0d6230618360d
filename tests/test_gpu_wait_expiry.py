"""Failure detection on the GPU without a fault: the tensor-core kernels'
bounded on-chip waits, made to expire on purpose.

prism_debug_wait_expiry arms a test mode in which every CTA withholds one
completion signal, so a wait for it cannot complete (a flag that nothing
sets) and expires after a short limit.  The kernel must then return -- no
hang, no fault, the context usable -- with PRISM_DEVSTATUS_WAIT_TIMEOUT
raised for the host; and after the mode is disarmed and the workspace zeroed
again, the next call must give the oracle's bits.  Both contraction kernels
(int8 operands; binary16 codes), each with shared tiles in both MMA
orientations, with one CTA per tile, and with whole tiles in rounds."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_util import dev, dev_bf16, host_bits

import deterministic_w8a8_int8_gb300 as prism

pytestmark = pytest.mark.gpu

LIMIT_NS = 20_000_000   # 20 ms


@pytest.mark.parametrize("kernel", ["int8", "f16"])
@pytest.mark.parametrize("M,N,K", [(600, 2560, 2048), (304, 1536, 5120), (37, 384, 256), (304, 15360, 1024)])
def test_expired_wait_returns_reports_and_recovers(cuda_device, monkeypatch, kernel, M, N, K):
    monkeypatch.delenv("PRISM_LINEAR_PATH", raising=False)
    rng = np.random.default_rng(M + N + K)
    xb = wl.bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    w = wl.draw_weights(rng, (N, K), "normal")
    ws_ = rng.uniform(0.001, 0.02, N).astype(np.float32)
    rb = wl.bf16_bits(rng.standard_normal((M, N), dtype=np.float32))
    qo, ao = oracle.quant_act(xb, None)
    outo, _ = oracle.w8a8_linear(qo, ao, w, ws_, rb)
    X, S, R = dev_bf16(xb), dev(ws_), dev_bf16(rb)
    if kernel == "int8":
        q, a = prism.prism_quant_act(X)
        W = dev(w)
        buf = prism.new_workspace(M, N, K, 0, "cuda")
        call = lambda: prism.prism_w8a8_linear(q, a, W, S, residual=R, workspace=buf)
    else:
        q, a = prism.prism_quant_act_f16(X)
        W = prism.prism_codes_to_f16(dev(w))
        buf = prism.new_workspace_f16(M, N, K, 0, "cuda")
        call = lambda: prism.prism_w8a8_linear_f16(q, a, W, S, residual=R, workspace=buf)
    torch.cuda.synchronize()
    assert prism.prism_device_status() == 0

    prism.prism_debug_wait_expiry(LIMIT_NS)
    try:
        call()
        torch.cuda.synchronize()       # returns: the kernel wound down instead of hanging
    finally:
        prism.prism_debug_wait_expiry(0)
    assert prism.prism_device_status() == prism.PRISM_DEVSTATUS_WAIT_TIMEOUT

    # the context is usable, and with the workspace zeroed again the next call is exact
    if buf is not None:
        buf.zero_()
    out = call()
    torch.cuda.synchronize()
    assert prism.prism_device_status() == 0
    assert np.array_equal(host_bits(out), outo)
