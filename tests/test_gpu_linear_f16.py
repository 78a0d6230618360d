"""GPU parity of the W8A8 linear on binary16 codes (prism_quant_act_f16,
prism_codes_to_f16, prism_w8a8_linear_f16) against the CPU oracle.

The codes are the int8 codes of the W8A8 linear stored as binary16 values,
so every result must equal the oracle's W8A8 linear on the int8 codes, bit
for bit (StartLux-Prism, "Bitwise consistency is not lossless quantization":
exact int32 accumulation, split-K partial sums kept as integers, a fixed
epilogue).  Covered: codes of the quantiser (both kernels: rows held in
registers and longer rows) and of the weight conversion (every byte value);
ragged shapes in both MMA orientations, strided and in-place outputs;
every explicit split-K factor and every branch of the balanced schedule;
fp32 chunks at the 2^24 boundary; int32 extremes at the largest K; agreement
with the int8-operand kernel; every 128-row block and every channel tile of
the full-size workloads."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_util import dev, dev_bf16, host, host_bits, padded
from tests.sched_util import balanced, f16_plan, f16_workspace

import deterministic_w8a8_int8_gb300 as prism

pytestmark = pytest.mark.gpu


def f16_codes(q: np.ndarray) -> np.ndarray:
    return q.astype(np.float16)


def run_f16(q, a, w, ws, res=None, split=0, acc=True, out=None):
    """The binary16-code linear on numpy int8 codes (converted on the GPU)."""
    M, N = q.shape[0], w.shape[0]
    Q = q if isinstance(q, torch.Tensor) else torch.from_numpy(f16_codes(q)).cuda()
    if isinstance(w, torch.Tensor) and w.dtype == torch.float16:
        W = w
    else:
        W = prism.prism_codes_to_f16(w if isinstance(w, torch.Tensor) else dev(w))
    acc_t = torch.empty((M, N), dtype=torch.int32, device="cuda") if acc else None
    A = a if isinstance(a, torch.Tensor) else dev(a)
    S = ws if isinstance(ws, torch.Tensor) else dev(ws)
    out = prism.prism_w8a8_linear_f16(Q, A, W, S, residual=res, out=out, acc_out=acc_t, split_k=split)
    torch.cuda.synchronize()
    return out, acc_t


def problem(M, N, K, seed, residual=True):
    rng = np.random.default_rng(seed)
    xb = wl.bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    w = wl.draw_weights(rng, (N, K), "normal")
    w_scale = rng.uniform(0.001, 0.02, N).astype(np.float32)
    rb = wl.bf16_bits(rng.standard_normal((M, N), dtype=np.float32)) if residual else None
    return xb, w, w_scale, rb


@pytest.mark.parametrize("M,K", [(37, 256), (304, 5120), (5, 17408), (64, 24576), (3, 32768), (2, 133136)])
def test_quant_codes_match_oracle(cuda_device, M, K):
    """The quantiser's binary16 codes are the oracle's int8 codes, exactly;
    the scales are the oracle's bits (persistent kernel up to K = 24576, the
    team kernel beyond)."""
    rng = np.random.default_rng(M + K)
    xb = wl.bf16_bits(rng.standard_normal((M, K), dtype=np.float32) * 3)
    inv_s = rng.uniform(0.5, 2.0, K).astype(np.float32)
    qo, ao = oracle.quant_act(xb, inv_s)
    qh, a = prism.prism_quant_act_f16(dev_bf16(xb), dev(inv_s))
    torch.cuda.synchronize()
    assert np.array_equal(host(qh).view(np.uint16), f16_codes(qo).view(np.uint16))
    assert np.array_equal(host(a).view(np.uint32), ao.view(np.uint32))


def test_quant_codes_zero_and_tie_rows(cuda_device):
    """A zero row gives +0 codes and scale 0; the hand-worked tie row rounds
    63.5 to 64 as in the int8 quantiser."""
    K = 16
    x = np.zeros((2, K), np.float32)
    x[1, :4] = [1.0, -0.5, 0.25, 2.0]
    xb = wl.bf16_bits(x)
    qh, a = prism.prism_quant_act_f16(dev_bf16(xb))
    torch.cuda.synchronize()
    got = host(qh)
    assert np.array_equal(got[0].view(np.uint16), np.zeros(K, np.uint16))
    assert list(got[1, :4]) == [64, -32, 16, 127]
    assert host(a)[0] == 0.0


def test_codes_to_f16_every_byte(cuda_device):
    w = np.arange(-128, 128, dtype=np.int16).astype(np.int8).reshape(16, 16)
    w = np.concatenate([w, w[::-1]], axis=1)        # K = 32
    wh = prism.prism_codes_to_f16(dev(w))
    torch.cuda.synchronize()
    assert np.array_equal(host(wh).view(np.uint16), w.astype(np.float16).view(np.uint16))


@pytest.mark.parametrize("M,N,K", [(1, 8, 16), (3, 130, 48), (129, 384, 256), (37, 131, 64),
                                   (130, 257, 528), (255, 136, 1040), (600, 520, 2064), (1000, 300, 1024),
                                   (513, 272, 1088)])
@pytest.mark.parametrize("residual", [True, False])
@pytest.mark.parametrize("orient", ["auto", "rows", "cols"])
def test_ragged_shapes(cuda_device, monkeypatch, M, N, K, residual, orient):
    """Both MMA orientations on every shape (PRISM_F16_ORIENT: tokens on the
    128 MMA rows, or on the N side in pieces), and the library's choice."""
    if orient != "auto":
        monkeypatch.setenv("PRISM_F16_ORIENT", orient)
    xb, w, w_scale, rb = problem(M, N, K, M * 131 + N * 7 + K, residual)
    qo, ao = oracle.quant_act(xb, None)
    outo, acco = oracle.w8a8_linear(qo, ao, w, w_scale, rb)
    qh, a = prism.prism_quant_act_f16(dev_bf16(xb))
    R = None if rb is None else dev_bf16(rb)
    out, acc = run_f16(qh, a, w, w_scale, R)
    assert np.array_equal(host(acc), acco)
    assert np.array_equal(host_bits(out), outo)


@pytest.mark.parametrize("M,N,K", [(70, 264, 1040), (700, 264, 1040)])
def test_strided_and_in_place_outputs(cuda_device, M, N, K):
    xb, w, w_scale, rb = problem(M, N, K, 11 * M + K)
    qo, ao = oracle.quant_act(xb, None)
    outo, _ = oracle.w8a8_linear(qo, ao, w, w_scale, rb)
    qh, a = prism.prism_quant_act_f16(dev_bf16(xb))
    for ld in (N + 1, N + 8):
        r = padded(M, N, ld, torch.bfloat16)
        r.copy_(dev_bf16(rb))
        out = padded(M, N, ld, torch.bfloat16)
        out, _ = run_f16(qh, a, w, w_scale, r, out=out)
        assert np.array_equal(host_bits(out), outo), ld
    buf = dev_bf16(rb)
    run_f16(qh, a, w, w_scale, buf, out=buf, acc=False)
    assert np.array_equal(host_bits(buf), outo)


@pytest.mark.parametrize("M", [70, 600])
def test_split_k_bit_identical(cuda_device, M):
    N, K = 520, 2064
    xb, w, w_scale, rb = problem(M, N, K, 17 + M)
    qo, ao = oracle.quant_act(xb, None)
    outo, acco = oracle.w8a8_linear(qo, ao, w, w_scale, rb)
    qh, a = prism.prism_quant_act_f16(dev_bf16(xb))
    R = dev_bf16(rb)
    for split in (0, 1, 2, 3, 4, 7, 8, 16, 33, 64):
        out, acc = run_f16(qh, a, w, w_scale, R, split=split)
        assert np.array_equal(host(acc), acco), split
        assert np.array_equal(host_bits(out), outo), split


@pytest.mark.parametrize("M,N,K", [
    (1024, 4864, 512),    # 152 tiles: one round of whole tiles
    (304, 1536, 5120),    # 24 tiles, each cut into 5 K pieces (lockstep)
    (600, 2560, 2048),    # 50 tiles, 2 pieces each
    (304, 15360, 1024),   # whole tiles in two rounds (the last 88 of 152)
    (37, 384, 256),       # one CTA per tile
    (640, 25600, 256),    # whole tiles in four rounds
    (96, 640, 17408),     # 5 tiles of 272 K stages, 17 pieces each
    (2048, 5120, 5120),   # two rounds, then 16 tiles in 5 pieces
    (1024, 5120, 1024),   # 160 tiles of 16 stages: the balanced schedule shares them all
])
def test_balanced_schedule_matches_single_piece(cuda_device, M, N, K):
    """Every branch of the balanced schedule gives the bits of one K piece
    per tile; a reused workspace stays zero."""
    rng = np.random.default_rng(M * 7 + N + K)
    q = rng.integers(-127, 128, (M, K), dtype=np.int8)
    w = rng.integers(-127, 128, (N, K), dtype=np.int8)
    a = (rng.random(M, dtype=np.float32) * 1e-3 + 1e-4).astype(np.float32)
    s = (rng.random(N, dtype=np.float32) * 1e-2 + 1e-3).astype(np.float32)
    rb = wl.bf16_bits(rng.normal(size=(M, N)).astype(np.float32))
    Q = torch.from_numpy(f16_codes(q)).cuda()
    W = prism.prism_codes_to_f16(dev(w))
    A, S, R = dev(a), dev(s), dev_bf16(rb)
    ref, ref_acc = run_f16(Q, A, W, S, R, split=1)
    ws_buf = prism.new_workspace_f16(M, N, K, 0, "cuda")
    counter_bytes, total = f16_workspace(M, N, K)
    assert (0 if ws_buf is None else ws_buf.numel()) == total
    for i in range(3):
        acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
        got = prism.prism_w8a8_linear_f16(Q, A, W, S, residual=R, split_k=0, workspace=ws_buf, acc_out=acc)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
        assert torch.equal(acc, ref_acc)
        if ws_buf is not None:
            # calls leave the arrival counters zero; the piece slots are
            # scratch whose stale contents never reach a result
            assert int(ws_buf[:counter_bytes].count_nonzero()) == 0
            ws_buf[counter_bytes:].fill_(0x5A + i)
    # and the single-piece result is the oracle's (sampled rows)
    rows = np.unique(np.linspace(0, M - 1, 9).astype(int))
    outo, acco = oracle.w8a8_linear(q[rows], a[rows], w, s, rb[rows])
    assert np.array_equal(host(ref_acc)[rows], acco)
    assert np.array_equal(host_bits(ref)[rows], outo)


@pytest.mark.parametrize("sched", ["whole", "balanced", "lock"])
@pytest.mark.parametrize("M,N,K", [(304, 1536, 5120), (2048, 5120, 2048), (300, 2600, 1040)])
def test_every_schedule_matches_oracle(cuda_device, monkeypatch, sched, M, N, K):
    """Each automatic schedule forced on the same shapes (PRISM_F16_SCHED):
    whole tiles in rounds, the balanced schedule's shared K ranges, and the
    rounds with the remainder tiles split in lockstep -- every one bit-exact
    against the oracle, with the workspace sized for it."""
    monkeypatch.setenv("PRISM_F16_SCHED", sched)
    xb, w, w_scale, rb = problem(M, N, K, 3 * M + N)
    rows = np.unique(np.linspace(0, M - 1, 11).astype(int))
    qo, ao = oracle.quant_act(xb[rows], None)
    outo, acco = oracle.w8a8_linear(qo, ao, w, w_scale, rb[rows])
    qh, a = prism.prism_quant_act_f16(dev_bf16(xb))
    W = prism.prism_codes_to_f16(dev(w))
    ws_buf = prism.new_workspace_f16(M, N, K, 0, "cuda")
    for i in range(2):
        acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
        out = prism.prism_w8a8_linear_f16(qh, a, W, dev(w_scale), residual=dev_bf16(rb), acc_out=acc,
                                          workspace=ws_buf)
        torch.cuda.synchronize()
        assert np.array_equal(host(acc)[rows], acco), i
        assert np.array_equal(host_bits(out)[rows], outo), i
        if ws_buf is not None:
            # slots are scratch; the counters (one per shared tile, first) stay zero
            T = f16_plan(M, N)[1]
            R = T % 152 if sched == "lock" else balanced(T, (K + 63) // 64, 16)[2]
            cb = (R * 4 + 255) & ~255
            assert int(ws_buf[:cb].count_nonzero()) == 0
            ws_buf[cb:].fill_(0x3C + i)


@pytest.mark.parametrize("M", [5, 40, 130, 600])
def test_chunks_exact_at_2_pow_24(cuda_device, M):
    """All +-127 operands (chunk partials up to 1024 * 16129) and single
    unit terms beside near-2^24 partials come out exact."""
    K = 4096 + 1024 + 64
    rng = np.random.default_rng(M)
    q = np.full((M, K), 127, np.int8)
    q[1::3] = -127
    q[2::3, 1023::1024] = 1
    N = 264
    w = np.where(rng.random((N, K)) < 0.5, 127, -127).astype(np.int8)
    w[0] = 127
    w[1] = -127
    w[2, 1023::1024] = -1
    w[3, ::2] = 1
    a = np.ones(M, np.float32)
    ws = np.ones(N, np.float32)
    outo, acco = oracle.w8a8_linear(q, a, w, ws, None)
    for split in (0, 1, 3):
        out, acc = run_f16(q, a, w, ws, None, split=split)
        assert np.array_equal(host(acc), acco), split
        assert np.array_equal(host_bits(out), outo), split


def test_int32_extremes_at_max_k(cuda_device):
    K = 133136
    q = np.full((3, K), 127, np.int8)
    q[1] = -127
    q[2, ::2] = -127
    w = np.full((16, K), 127, np.int8)
    w[1::2] = -127
    a = np.ones(3, np.float32)
    ws = np.ones(16, np.float32)
    outo, acco = oracle.w8a8_linear(q, a, w, ws, None)
    assert int(np.abs(acco).max()) == 127 * 127 * K
    for split in (0, 1, 5):
        out, acc = run_f16(q, a, w, ws, None, split=split)
        assert np.array_equal(host(acc), acco), split
        assert np.array_equal(host_bits(out), outo), split


@pytest.mark.parametrize("M,N,K", [(37, 384, 256), (304, 512, 5120), (600, 520, 2064), (2048, 1024, 1024)])
def test_agrees_with_int8_operand_kernel(cuda_device, M, N, K):
    """The binary16-code kernel and the int8-operand kernel give the same
    bits on the same codes."""
    xb, w, w_scale, rb = problem(M, N, K, 41 + M)
    q, a = prism.prism_quant_act(dev_bf16(xb))
    qh, ah = prism.prism_quant_act_f16(dev_bf16(xb))
    assert torch.equal(a, ah) and torch.equal(qh, q.to(torch.float16))
    W, S, R = dev(w), dev(w_scale), dev_bf16(rb)
    acc8 = torch.empty((M, N), dtype=torch.int32, device="cuda")
    out8 = prism.prism_w8a8_linear(q, a, W, S, residual=R, acc_out=acc8)
    out16, acc16 = run_f16(qh, ah, W, S, R)
    assert torch.equal(acc8, acc16)
    assert torch.equal(out8.view(torch.int16), out16.view(torch.int16))


@pytest.mark.parametrize("name", ["forest_qkv_m304_k5120_n15360", "forest_oproj_m304_k5120_n5120",
                                  "load_gateup_m2048_k5120_n34816", "load_down_m2048_k17408_n5120",
                                  "long_m8192_k5120_n5120"])
def test_full_size_every_tile(cuda_device, name):
    """Full-size call in the benchmark's launch configuration (balanced
    schedule): one row of every 128-row block (plus the first and last rows)
    checked against the oracle across ALL output channels, so every output
    tile of both orientations is covered; and the accumulators of those rows
    as well."""
    c = wl.make_linear(name)
    qh, a = prism.prism_quant_act_f16(dev_bf16(c.x_bits), dev(c.inv_s))
    W = prism.prism_codes_to_f16(dev(c.w))
    R = None if c.residual_bits is None else dev_bf16(c.residual_bits)
    acc = torch.empty((c.M, c.N), dtype=torch.int32, device="cuda")
    out = prism.prism_w8a8_linear_f16(qh, a, W, dev(c.w_scale), residual=R, acc_out=acc)
    torch.cuda.synchronize()
    rng = np.random.default_rng(11)
    rows = [0, c.M - 1] + [b * 128 + int(rng.integers(0, min(128, c.M - b * 128))) for b in range((c.M + 127) // 128)]
    rows = np.unique(np.array(rows))
    qo, ao = oracle.quant_act(c.x_bits[rows], c.inv_s)
    assert np.array_equal(host(qh)[rows].view(np.uint16), f16_codes(qo).view(np.uint16))
    assert np.array_equal(host(a)[rows], ao)
    rr = None if c.residual_bits is None else c.residual_bits[rows]
    outo, acco = oracle.w8a8_linear(qo, ao, c.w, c.w_scale, rr)
    assert np.array_equal(host(acc)[rows], acco)
    assert np.array_equal(host_bits(out)[rows], outo)


def test_argument_checks(cuda_device):
    L = prism.lib()
    import ctypes
    P = ctypes.c_void_p
    z = torch.zeros(64 * 64, dtype=torch.float16, device="cuda")
    s = torch.ones(64, device="cuda")
    o = torch.zeros(64 * 64, dtype=torch.bfloat16, device="cuda")
    st = P(torch.cuda.current_stream().cuda_stream)

    def call(M=64, N=64, K=64, ldq=64, ldw=64, q=z, split=0, ws=None, wsb=0):
        return L.prism_w8a8_linear_f16(P(q.data_ptr()), ldq, P(s.data_ptr()), P(z.data_ptr()), ldw, P(s.data_ptr()),
                                       None, 0, P(o.data_ptr()), 64, None, M, N, K, split,
                                       None if ws is None else P(ws), wsb, st)

    assert call(K=72, ldq=72, ldw=72) == prism.PRISM_ERR_ALIGNMENT
    assert call(ldq=60) == prism.PRISM_ERR_INVALID_ARG
    assert call(ldq=68) == prism.PRISM_ERR_ALIGNMENT
    assert call(split=65) == prism.PRISM_ERR_UNSUPPORTED
    assert call(K=133152, ldq=133152, ldw=133152) == prism.PRISM_ERR_UNSUPPORTED
    assert call(M=0) == prism.PRISM_OK
    M, N, K = 304, 1536, 5120
    assert prism.prism_w8a8_f16_workspace_bytes(M, N, K, 0) > 0
    assert L.prism_w8a8_linear_f16(P(z.data_ptr()), K, P(s.data_ptr()), P(z.data_ptr()), K, P(s.data_ptr()), None, 0,
                                   P(o.data_ptr()), N, None, M, N, K, 0, None, 0, st) == prism.PRISM_ERR_WORKSPACE
