"""Repeated runs of the shared-tile read-back under the restricted last layer
(StartLux-Prism, "Compute shared evidence once": read-out work restricted to
the answer positions; "Bitwise consistency is not lossless quantization":
split-K partial sums stay integers, so every run gives the same bits).

The case is 64 clients x 3 answers: 192 gathered answer rows of a
2048 x 5120 hidden state through a 5120 x 5120 projection with the full
hidden state's residual rows.  192 rows put the tensor-core kernel in its
swapped orientation (output channels on the 128 MMA rows, the tokens as its
N side) and its automatic schedule shares every one of the 40 output tiles
between CTAs: each CTA adds its int32 partial sums into the tile's slot
with integer reductions and the last one to arrive reads the slot back,
re-zeroes it and applies the epilogue.  An ordering fault anywhere in that
protocol (or in the gathered quantiser before it) shows up as a wrong bit in
some run; every run is compared with the oracle, bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_util import dev, dev_bf16

import deterministic_w8a8_int8_gb300 as prism

pytestmark = pytest.mark.gpu

M_X, K, N, N_ROWS = 2048, 5120, 5120, 192


@pytest.fixture(scope="module")
def problem():
    rng = np.random.default_rng(2024)
    x = wl.bf16_bits(rng.standard_normal((M_X, K), dtype=np.float32))
    outl = rng.choice(K, size=K // 100, replace=False)
    x[:, outl] = wl.bf16_bits(rng.standard_normal((M_X, outl.size), dtype=np.float32) * 30)
    inv_s = rng.uniform(0.5, 2.0, K).astype(np.float32)
    w = wl.draw_weights(rng, (N, K), "normal")
    ws = rng.uniform(0.001, 0.02, N).astype(np.float32)
    res = wl.bf16_bits(rng.standard_normal((M_X, N), dtype=np.float32))
    rows = np.sort(rng.choice(M_X, size=N_ROWS, replace=False)).astype(np.int32)[::-1].copy()
    q_o, a_o, e_o = oracle.quant_act_rows(x, rows, inv_s)
    out_o, acc_o, e2 = oracle.w8a8_linear_rows(q_o, a_o, w, ws, res, rows)
    assert e_o == 0 and e2 == 0
    return dict(X=dev_bf16(x), I=dev(inv_s), W=dev(w), S=dev(ws), R=dev_bf16(res), rows=dev(rows),
                q_o=torch.from_numpy(q_o).cuda(), a_o=torch.from_numpy(a_o).cuda(),
                out_o=torch.from_numpy(out_o.view(np.int16)).cuda(), acc_o=torch.from_numpy(acc_o).cuda())


def _tc_path(monkeypatch):
    monkeypatch.setenv("PRISM_LINEAR_PATH", "tc")
    assert prism.prism_w8a8_kernel_kind(N_ROWS, N, K) == 3          # swapped orientation
    assert prism.prism_w8a8_auto_split(N_ROWS, N, K) == 0            # balanced schedule
    assert prism.prism_w8a8_workspace_bytes(N_ROWS, N, K, 0) > 0     # with shared tiles


def _run(p, ws_buf, stream, reps):
    """reps back-to-back quantise + restricted-linear pairs on one stream,
    each into its own outputs; the workspace is reused by every call."""
    outs = []
    with torch.cuda.stream(stream):
        for _ in range(reps):
            q, a = prism.prism_quant_act_rows(p["X"], p["rows"], p["I"])
            acc = torch.empty((N_ROWS, N), dtype=torch.int32, device="cuda")
            out = prism.prism_w8a8_linear_rows(q, a, p["W"], p["S"], p["R"], p["rows"], acc_out=acc,
                                               workspace=ws_buf)
            outs.append((q, a, acc, out))
    return outs


def _count_bad(p, outs):
    bad = 0
    for q, a, acc, out in outs:
        ok = (torch.equal(q, p["q_o"]) and torch.equal(a.view(torch.int32), p["a_o"].view(torch.int32))
              and torch.equal(acc, p["acc_o"]) and torch.equal(out.view(torch.int16), p["out_o"]))
        bad += 0 if ok else 1
    return bad


def test_restricted_shared_tiles_many_runs_one_stream(cuda_device, problem, monkeypatch):
    """200 back-to-back calls on one stream, one workspace: all bit-exact."""
    _tc_path(monkeypatch)
    p = problem
    ws_buf = prism.new_workspace(N_ROWS, N, K, 0, "cuda")
    stream = torch.cuda.current_stream()
    outs = _run(p, ws_buf, stream, 200)
    torch.cuda.synchronize()
    assert prism.prism_device_status() == 0
    assert _count_bad(p, outs) == 0
    assert int(ws_buf.count_nonzero()) == 0     # every call leaves the slots and counters zero


def test_restricted_shared_tiles_two_streams(cuda_device, problem, monkeypatch):
    """Two streams with a workspace each, 100 calls per stream, launched
    alternately so that calls of the two streams overlap on the GPU."""
    _tc_path(monkeypatch)
    p = problem
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    bufs = [prism.new_workspace(N_ROWS, N, K, 0, "cuda") for _ in streams]
    torch.cuda.synchronize()
    outs = [[], []]
    for _ in range(100):
        for i, s in enumerate(streams):
            outs[i] += _run(p, bufs[i], s, 1)
    torch.cuda.synchronize()
    assert prism.prism_device_status() == 0
    assert _count_bad(p, outs[0]) == 0 and _count_bad(p, outs[1]) == 0
    assert all(int(b.count_nonzero()) == 0 for b in bufs)


def test_full_layer_rows_equal_restricted_rows_repeatedly(cuda_device, problem, monkeypatch):
    """The full 2048-row layer (tokens on the MMA rows, shared tiles read back
    in that orientation) run 20 times: its answer rows equal the oracle's
    restricted rows every time."""
    _tc_path(monkeypatch)
    p = problem
    assert prism.prism_w8a8_kernel_kind(M_X, N, K) == 2
    qf, af = prism.prism_quant_act(p["X"], p["I"])
    ws_buf = prism.new_workspace(M_X, N, K, 0, "cuda")
    outs = [prism.prism_w8a8_linear(qf, af, p["W"], p["S"], residual=p["R"], workspace=ws_buf)
            for _ in range(20)]
    torch.cuda.synchronize()
    assert prism.prism_device_status() == 0
    idx = p["rows"].long()
    bad = sum(0 if torch.equal(o.view(torch.int16)[idx], p["out_o"]) else 1 for o in outs)
    assert bad == 0
    assert int(ws_buf.count_nonzero()) == 0


def test_full_size_gateup_repeated_calls_identical(cuda_device, monkeypatch):
    """60 full-size gate/up calls (2048 x 34816 x 5120, int8 operands: 2176
    tiles of 80 widened stages a call) give identical accumulators, and the
    first one is the oracle's on one row of every 128-row block.  With an odd
    number of operand slots, shared by the two widening groups, about one
    call in 15 to 40 had a wrong tile; this repeats enough calls to see it."""
    monkeypatch.delenv("PRISM_LINEAR_PATH", raising=False)
    c = wl.make_linear("load_gateup_m2048_k5120_n34816")
    q, a = prism.prism_quant_act(dev_bf16(c.x_bits), dev(c.inv_s))
    W, S = dev(c.w), dev(c.w_scale)
    ws_buf = prism.new_workspace(c.M, c.N, c.K, 0, "cuda")
    ref = torch.empty((c.M, c.N), dtype=torch.int32, device="cuda")
    prism.prism_w8a8_linear(q, a, W, S, acc_out=ref, workspace=ws_buf)
    torch.cuda.synchronize()
    rows = np.unique(np.array([0, c.M - 1] + [b * 128 + 37 for b in range(c.M // 128)]))
    qo, ao = oracle.quant_act(c.x_bits[rows], c.inv_s)
    _, acco = oracle.w8a8_linear(qo, ao, c.w, c.w_scale, None)
    assert np.array_equal(ref.cpu().numpy()[rows], acco)
    acc = torch.empty_like(ref)
    bad = 0
    for _ in range(60):
        prism.prism_w8a8_linear(q, a, W, S, acc_out=acc, workspace=ws_buf)
        torch.cuda.synchronize()
        bad += 0 if torch.equal(acc, ref) else 1
    assert prism.prism_device_status() == 0
    assert bad == 0


def test_full_size_gateup_f16_repeated_calls_identical(cuda_device):
    """The same for the binary16-code kernel (whole tiles in rounds): 40
    calls, identical accumulators, the first one the oracle's."""
    c = wl.make_linear("load_gateup_m2048_k5120_n34816")
    qh, a = prism.prism_quant_act_f16(dev_bf16(c.x_bits), dev(c.inv_s))
    W = prism.prism_codes_to_f16(dev(c.w))
    S = dev(c.w_scale)
    ws_buf = prism.new_workspace_f16(c.M, c.N, c.K, 0, "cuda")
    ref = torch.empty((c.M, c.N), dtype=torch.int32, device="cuda")
    prism.prism_w8a8_linear_f16(qh, a, W, S, acc_out=ref, workspace=ws_buf)
    torch.cuda.synchronize()
    rows = np.unique(np.array([0, c.M - 1] + [b * 128 + 91 for b in range(c.M // 128)]))
    qo, ao = oracle.quant_act(c.x_bits[rows], c.inv_s)
    _, acco = oracle.w8a8_linear(qo, ao, c.w, c.w_scale, None)
    assert np.array_equal(ref.cpu().numpy()[rows], acco)
    acc = torch.empty_like(ref)
    bad = 0
    for _ in range(40):
        prism.prism_w8a8_linear_f16(qh, a, W, S, acc_out=acc, workspace=ws_buf)
        torch.cuda.synchronize()
        bad += 0 if torch.equal(acc, ref) else 1
    assert prism.prism_device_status() == 0
    assert bad == 0
