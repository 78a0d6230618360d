"""Load-time SmoothQuant requantisation of Q8_0 weights on the GPU, bit for bit
against the oracle (StartLux-Prism, "Compute shared evidence once": the
stored 8-bit weights are requantised with the smoothing factors folded in).

Shapes cover every register-cache width of the cached kernel (1, 2 and 3
vectors of 16 per thread, teams of 32 to 512 threads), more rows than one
resident grid (the prefetching row loop), the uncached kernel for long rows
up to the largest K, the three projections of the 27B model at full size,
special rows (zero, below 2^-120, subnormal and negative block scales), in
place and strided operation, argument errors, and the requantised weight fed
through the W8A8 linear."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_util import dev, host, padded

import deterministic_w8a8_int8_gb300 as prism

pytestmark = pytest.mark.gpu


def dev_f16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).cuda()


def check(case: wl.Q8Case, use_s: bool = True):
    s = case.s if use_s else None
    w_o, ws_o = oracle.smooth_requant(case.q, case.d, s)
    w, ws = prism.prism_smooth_requant(dev(case.q), dev_f16(case.d), None if s is None else dev(s))
    torch.cuda.synchronize()
    assert np.array_equal(host(w), w_o)
    assert np.array_equal(host(ws).view(np.uint32), ws_o.view(np.uint32))


@pytest.mark.parametrize("N,K,use_s", [
    (37, 32, True),        # one block per row, a single warp
    (5, 256, False),       # no smoothing vector
    (300, 5120, True),     # 320-thread teams, 1 vector each
    (3000, 5120, True),    # more rows than resident CTAs: prefetching row loop
    (50, 8192, True),      # 512 threads x 1 vector
    (50, 8224, True),      # just past it: 288 threads x 2 vectors
    (64, 16384, True),     # 512 threads x 2 vectors
    (40, 16416, True),     # just past it: 352 threads x 3 vectors
    (600, 17408, True),    # the down projection's K, several rows per CTA
    (12, 24576, True),     # the largest cached row: 512 threads x 3 vectors
    (6, 24608, True),      # uncached kernel
    (3, 133120, False),    # uncached, the largest K that is a multiple of 32
    # without smoothing, v * RN(127/amax) lands on exact ties x.5 hundreds of
    # times per million elements: each width must round them to even
    (600, 5120, False),
    (300, 16384, False),
    (200, 16416, False),
    (20, 24608, False),
])
def test_requant_matches_oracle(cuda_device, N, K, use_s):
    check(wl.q8_0_case("t", N, K, seed=N * 7 + K), use_s)


@pytest.mark.parametrize("name", sorted(wl.REQUANT_CONFIGS))
def test_requant_full_size(cuda_device, name):
    check(wl.make_q8_0(name))


def test_requant_special_rows(cuda_device):
    K = 64
    case = wl.q8_0_case("special", 8, K, seed=5)
    q, d, s = case.q.copy(), case.d.copy(), case.s.copy()
    q[0] = 0                                   # all-zero row -> zeros, scale 0
    d[1] = 0x0001                              # smallest subnormal scale, 2^-24 ...
    s[:] = np.float32(2.0 ** -100)             # ... times s = 2^-100: below 2^-120
    q[1] = 127
    d[2] = 0x0001                              # subnormal scale, s normal in row 3 below
    d[3] = 0x83FF                              # largest negative subnormal scale
    d[4] = 0xBC00                              # -1.0
    d[5, 0] = 0x0000                           # a zero block next to a normal one
    q[6] = 0
    q[6, 17] = -3                              # a single nonzero value -> -127 there
    d[7, 1] = 0x7BFF                           # largest finite binary16 scale in one block
    s2 = np.ones(K, np.float32)
    for sv in (s, s2):
        w_o, ws_o = oracle.smooth_requant(q, d, sv)
        w, ws = prism.prism_smooth_requant(dev(q), dev_f16(d), dev(sv))
        torch.cuda.synchronize()
        assert np.array_equal(host(w), w_o)
        assert np.array_equal(host(ws).view(np.uint32), ws_o.view(np.uint32))
    # the rows the construction pins down, stated from the definition
    w_o, ws_o = oracle.smooth_requant(q, d, s2)
    assert not w_o[0].any() and ws_o[0] == 0
    assert w_o[6, 17] == -127 and np.count_nonzero(w_o[6]) == 1


@pytest.mark.parametrize("N,K", [(300, 5120), (40, 16416), (4, 32800)])
def test_requant_in_place(cuda_device, N, K):
    case = wl.q8_0_case("inplace", N, K, seed=K)
    w_o, ws_o = oracle.smooth_requant(case.q, case.d, case.s)
    Q = dev(case.q)
    w, ws = prism.prism_smooth_requant(Q, dev_f16(case.d), dev(case.s), w=Q)
    torch.cuda.synchronize()
    assert w.data_ptr() == Q.data_ptr()
    assert np.array_equal(host(Q), w_o)
    assert np.array_equal(host(ws).view(np.uint32), ws_o.view(np.uint32))


@pytest.mark.parametrize("N,K", [(70, 5120), (9, 32800)])
def test_requant_strided(cuda_device, N, K):
    case = wl.q8_0_case("strided", N, K, seed=3 * K)
    w_o, ws_o = oracle.smooth_requant(case.q, case.d, case.s)
    Q = padded(N, K, K + 48, torch.int8, fill=5)
    Q.copy_(dev(case.q))
    D = padded(N, K // 32, K // 32 + 3, torch.int16, fill=0x7C00)   # +inf padding never read
    D.copy_(dev_f16(case.d))
    W = padded(N, K, K + 16, torch.int8, fill=-9)
    w, ws = prism.prism_smooth_requant(Q, D, dev(case.s), w=W)
    torch.cuda.synchronize()
    buf = host(W.as_strided((N, K + 16), (K + 16, 1)))
    assert np.array_equal(buf[:, :K], w_o)
    assert (buf[:, K:] == -9).all()           # row padding untouched
    assert np.array_equal(host(ws).view(np.uint32), ws_o.view(np.uint32))


def test_requant_rejects_bad_arguments(cuda_device):
    K, N = 64, 4
    q = torch.zeros((N, K), dtype=torch.int8, device="cuda")
    d = torch.zeros((N, K // 32), dtype=torch.int16, device="cuda")
    s_buf = torch.ones(K + 4, dtype=torch.float32, device="cuda")
    with pytest.raises(prism.PrismError) as e:                    # K not a multiple of 32
        prism.prism_smooth_requant(q[:, :48], d, None)
    assert e.value.status == prism.PRISM_ERR_ALIGNMENT
    with pytest.raises(prism.PrismError) as e:                    # smooth 4- but not 16-byte aligned
        prism.prism_smooth_requant(q, d, s_buf[1:K + 1])
    assert e.value.status == prism.PRISM_ERR_ALIGNMENT
    lib = prism.lib()
    w = torch.empty((N, 2 * K), dtype=torch.int8, device="cuda")
    ws = torch.empty((N,), dtype=torch.float32, device="cuda")
    P = ctypes.c_void_p
    stream = P(torch.cuda.current_stream().cuda_stream)
    # in place with two different strides
    assert lib.prism_smooth_requant(P(w.data_ptr()), 2 * K, P(d.data_ptr()), K // 32, None, N, K,
                                    P(w.data_ptr()), K, P(ws.data_ptr()), stream) == prism.PRISM_ERR_INVALID_ARG
    # block-scale stride shorter than K/32
    assert lib.prism_smooth_requant(P(q.data_ptr()), K, P(d.data_ptr()), 1, None, N, K,
                                    P(w.data_ptr()), 2 * K, P(ws.data_ptr()), stream) == prism.PRISM_ERR_INVALID_ARG
    # K beyond the limit
    assert lib.prism_smooth_requant(P(q.data_ptr()), 133184, P(d.data_ptr()), 4162, None, 1, 133184,
                                    P(w.data_ptr()), 133184, P(ws.data_ptr()), stream) == prism.PRISM_ERR_UNSUPPORTED
    # N == 0 enqueues nothing and succeeds
    assert lib.prism_smooth_requant(P(q.data_ptr()), K, P(d.data_ptr()), K // 32, None, 0, K,
                                    P(w.data_ptr()), 2 * K, P(ws.data_ptr()), stream) == prism.PRISM_OK
    torch.cuda.synchronize()


def test_requantised_weight_feeds_the_linear(cuda_device):
    """Load-time requantisation, then the serving layer on that weight: the
    whole chain matches the oracle's chain bit for bit."""
    N, K, M = 1536, 5120, 304
    case = wl.q8_0_case("chain", N, K, seed=21)
    rng = np.random.default_rng(22)
    x = wl.bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    inv_s = (np.float32(1.0) / case.s).astype(np.float32)
    w_o, ws_o = oracle.smooth_requant(case.q, case.d, case.s)
    qa_o, a_o = oracle.quant_act(x, inv_s)
    y_o, _ = oracle.w8a8_linear(qa_o, a_o, w_o, ws_o, None)

    W, WS = prism.prism_smooth_requant(dev(case.q), dev_f16(case.d), dev(case.s))
    X = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    qa, a = prism.prism_quant_act(X, dev(inv_s))
    y = prism.prism_w8a8_linear(qa, a, W, WS, workspace=prism.new_workspace(M, N, K, 0, X.device))
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().view(torch.int16).numpy().view(np.uint16), y_o)
