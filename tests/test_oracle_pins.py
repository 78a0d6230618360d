"""Pins of the CPU oracle against things other than itself.

Each oracle function is checked here against what the pages and mathematics
fix: hand-worked examples, closed forms, brute force on tiny inputs, library
routines (numpy integer matmul, numpy binary32 arithmetic, torch's bf16
rounding), invariants, error bounds, and the pages' candidate-softmax identity
("把决策模型推理从 vLLM 换到 Prism", sections 方案 and 实现要点).  No GPU.
"""
import json
import math
import os
from fractions import Fraction as Fr

import numpy as np
import pytest

import oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers --
def rn32(v) -> float:
    """Round an exact rational to binary32, nearest-even (normal range and
    zero only; independent of any float unit)."""
    v = Fr(v)
    if v == 0:
        return 0.0
    s = -1 if v < 0 else 1
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fr(2) ** e > a:
        e -= 1
    while Fr(2) ** (e + 1) <= a:
        e += 1
    assert e >= -126, "helper covers normal numbers only"
    ulp = Fr(2) ** (e - 23)
    m = a / ulp
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > Fr(1, 2) or (rem == Fr(1, 2) and fl % 2 == 1):
        fl += 1
    return s * float(fl * ulp)


def rnbf16_bits(v) -> int:
    """Round an exact rational to bf16 (8 significant bits), nearest-even."""
    v = Fr(v)
    if v == 0:
        return 0
    s = 0x8000 if v < 0 else 0
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fr(2) ** e > a:
        e -= 1
    while Fr(2) ** (e + 1) <= a:
        e += 1
    ulp = Fr(2) ** (e - 7)
    m = a / ulp
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > Fr(1, 2) or (rem == Fr(1, 2) and fl % 2 == 1):
        fl += 1
    val = float(fl * ulp)
    return s | int(np.float32(val).view(np.uint32) >> 16)


def f32_bits(x) -> int:
    return int(np.float32(x).view(np.uint32))


def bits(x_f32: np.ndarray) -> np.ndarray:
    return wl.bf16_bits(np.asarray(x_f32, np.float32))


# ------------------------------------------- SmoothQuant requantisation ----
# StartLux-Prism, "Compute shared evidence once": Q8_0 weights (blocks of 32
# int8 with one binary16 scale) requantised with SmoothQuant at startup.
F16_ONE = 0x3C00


def _f16_bits(x) -> np.ndarray:
    return np.asarray(x, np.float16).view(np.uint16)


def test_f16_decoder_matches_library_on_every_pattern():
    h = np.arange(65536, dtype=np.uint16)
    got = oracle.f16_to_float(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_requant_unit_blocks_reduce_to_activation_quantiser():
    # with every block scale 1, requantising q * s is the activation
    # quantiser applied to x = q (integers <= 127 are exact in bf16) with
    # inv_s = s -- a special case of an independently pinned function
    rng = np.random.default_rng(31)
    for N, K in [(7, 64), (33, 256), (3, 1024)]:
        q = rng.integers(-127, 128, (N, K), dtype=np.int8)
        s = rng.uniform(0.25, 4.0, K).astype(np.float32)
        d = np.full((N, K // 32), F16_ONE, np.uint16)
        for sv in (s, None):
            w, ws = oracle.smooth_requant(q, d, sv)
            qa, aa = oracle.quant_act(wl.bf16_bits(q.astype(np.float32)), sv)
            assert np.array_equal(w, qa)
            assert np.array_equal(ws.view(np.uint32), aa.view(np.uint32))


def test_requant_block_scales_index_by_k_over_32():
    # a power-of-two block scale d moves into the smoothing factor exactly:
    # (d * q) * s == q * (d * s), one rounding either way; so each row must
    # equal the activation quantiser with inv_s_k = d[k // 32] * s_k
    rng = np.random.default_rng(32)
    N, K = 9, 256
    q = rng.integers(-127, 128, (N, K), dtype=np.int8)
    e = rng.integers(-6, 7, (N, K // 32))
    d = _f16_bits(np.exp2(e.astype(np.float64)))
    s = rng.uniform(0.5, 2.0, K).astype(np.float32)
    w, ws = oracle.smooth_requant(q, d, s)
    for n in range(N):
        fold = (np.exp2(e[n]).repeat(32) * s.astype(np.float64)).astype(np.float32)
        assert np.array_equal(fold.astype(np.float64), np.exp2(e[n]).repeat(32) * s.astype(np.float64))
        qa, aa = oracle.quant_act(wl.bf16_bits(q[n:n + 1].astype(np.float32)), fold)
        assert np.array_equal(w[n], qa[0]), n
        assert ws[n] == aa[0], n


def test_requant_closed_form_exact_rationals():
    # v = RN(d * q * s) (d * q exact), w_scale = RN(amax / 127),
    # w = clamp(rint(RN(v * RN(127 / amax)))), on exact rationals
    rng = np.random.default_rng(33)
    N, K = 6, 96
    q = rng.integers(-127, 128, (N, K), dtype=np.int8)
    d = _f16_bits(rng.uniform(1e-3, 3.0, (N, K // 32)))
    s = (rng.uniform(0.2, 5.0, K)).astype(np.float32)
    w, ws = oracle.smooth_requant(q, d, s)
    df = d.view(np.float16).astype(np.float64)
    for n in range(N):
        v = [rn32(Fr(float(df[n, k // 32])) * int(q[n, k]) * Fr(float(s[k]))) for k in range(K)]
        amax = max(abs(x) for x in v)
        assert ws[n] == np.float32(rn32(Fr(amax) / 127))
        inv = rn32(Fr(127) / Fr(amax))
        for k in range(K):
            t = rn32(Fr(v[k]) * Fr(inv))
            assert w[n, k] == max(-127, min(127, round(t)))


def test_requant_matches_library_binary32_arithmetic():
    # the same steps in numpy binary32 (each op one RN), on enough rows that
    # multiplying by RN(127/amax) and dividing by RN(amax/127) give different
    # codes somewhere: the test is sensitive to that reading
    rng = np.random.default_rng(36)
    N, K = 600, 256
    q = rng.integers(-127, 128, (N, K), dtype=np.int8)
    d = _f16_bits(rng.uniform(1e-3, 2.0, (N, K // 32)))
    s = rng.uniform(0.3, 3.0, K).astype(np.float32)
    w, ws = oracle.smooth_requant(q, d, s)
    df = d.view(np.float16).astype(np.float32).repeat(32, axis=1)
    v = (df * q.astype(np.float32)) * s[None, :]          # d*q exact, then one RN
    amax = np.abs(v).max(axis=1).astype(np.float32)
    inv = np.float32(127.0) / amax
    codes = np.clip(np.rint(v * inv[:, None]), -127, 127).astype(np.int8)
    assert np.array_equal(w, codes)
    assert np.array_equal(ws, amax / np.float32(127.0))
    # a row built so that the reading matters: amax = a (from q = 127 with
    # s_0 = RN(a / 127), RN(127 * s_0) == a) and one value v (q = 1, s_1 = v)
    # where rint(RN(v * RN(127 / a))) = 16 but rint(RN(v / RN(a / 127))) = 15
    a, vv = np.float32(3.7288472652435303), np.float32(0.455095499753952)
    s0 = a / np.float32(127.0)
    assert np.float32(127.0) * s0 == a
    K1 = 32
    q1 = np.zeros((1, K1), np.int8)
    q1[0, 0], q1[0, 1] = 127, 1
    s1 = np.zeros(K1, np.float32)
    s1[0], s1[1] = s0, vv
    w1, ws1 = oracle.smooth_requant(q1, np.full((1, 1), F16_ONE, np.uint16), s1)
    inv_r = rn32(Fr(127) / Fr(float(a)))
    mul = round(rn32(Fr(float(vv)) * Fr(inv_r)))
    div = round(rn32(Fr(float(vv)) / Fr(rn32(Fr(float(a)) / 127))))
    assert (mul, div) == (16, 15)
    assert w1[0, 0] == 127 and w1[0, 1] == mul


def test_requant_identity_equivariance_and_tiny_rows():
    rng = np.random.default_rng(34)
    N, K = 5, 128
    q = rng.integers(-127, 128, (N, K), dtype=np.int8)
    q[:, 0] = 127                                      # every row reaches 127
    one = np.full((N, K // 32), F16_ONE, np.uint16)
    w, ws = oracle.smooth_requant(q, one, None)
    assert np.array_equal(w, q) and np.all(ws == np.float32(1.0))
    # scaling every block scale by 2^e leaves the codes and scales w_scale by 2^e
    for e in (-8, 5):
        d2 = _f16_bits(np.full((N, K // 32), 2.0 ** e))
        w2, ws2 = oracle.smooth_requant(q, d2, None)
        assert np.array_equal(w2, q) and np.all(ws2 == np.float32(2.0 ** e))
    # all-zero rows and rows below 2^-120 give zero codes and scale 0
    qz = q.copy()
    qz[1] = 0
    tiny = one.copy()
    tiny[2] = 0x0001                                   # f16 2^-24: |v| <= 127 * 2^-134 < 2^-120
    s = np.full(K, 2.0 ** -110, np.float32)
    wz, wsz = oracle.smooth_requant(qz, tiny, s)
    assert not wz[1].any() and wsz[1] == 0.0
    assert not wz[2].any() and wsz[2] == 0.0
    assert wsz[0] > 0.0


def test_requant_error_bound():
    rng = np.random.default_rng(35)
    N, K = 16, 512
    q = rng.integers(-127, 128, (N, K), dtype=np.int8)
    d = _f16_bits(rng.uniform(1e-3, 0.1, (N, K // 32)))
    s = rng.uniform(0.5, 8.0, K).astype(np.float32)
    w, ws = oracle.smooth_requant(q, d, s)
    v = d.view(np.float16).astype(np.float64).repeat(32, axis=1) * q * s.astype(np.float64)
    err = np.abs(w.astype(np.float64) * ws[:, None].astype(np.float64) - v)
    # half a code step, plus the binary32 roundings of v, the scale and the reciprocal
    assert np.all(err <= ws[:, None] * (0.5 + 2.0 ** -20) + np.abs(v) * 2.0 ** -21)
    assert np.all(np.abs(w).max(axis=1) == 127)


# ------------------------------------------------------------ quantiser ----
def test_quant_hand_worked_examples():
    cases = json.load(open(os.path.join(GOLDEN, "quant_examples.json")))["cases"]
    for c in cases:
        x = np.array([c["x"]], np.float32)
        assert np.array_equal(wl.bits_to_f32(bits(x)), x), "example must be bf16-exact"
        inv_s = None if c["inv_s"] is None else np.array(c["inv_s"], np.float32)
        q, a = oracle.quant_act(bits(x), inv_s)
        assert q[0].tolist() == c["q"], c["name"]
        assert f32_bits(a[0]) == int(c["a_scale_bits"], 16), c["name"]


def test_quant_scale_closed_form():
    # a_scale = RN(amax / 127) on exact rationals, for a spread of amax values
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((64, 96)).astype(np.float32)
         * np.exp2(rng.integers(-20, 20, size=(64, 1))).astype(np.float32))
    xb = bits(x)
    q, a = oracle.quant_act(xb, None)
    xf = wl.bits_to_f32(xb)
    for m in range(64):
        amax = float(np.abs(xf[m]).max())
        assert a[m] == np.float32(rn32(Fr(amax) / 127))
        inv_a = rn32(Fr(127) / Fr(amax))
        # every code by exact rationals: rint(RN(xs * inv_a)), ties to even
        for k in range(0, 96, 7):
            t = rn32(Fr(float(xf[m, k])) * Fr(inv_a))
            assert q[m, k] == max(-127, min(127, round(t)))  # Python round: ties to even


def test_quant_invariants_and_error_bound():
    case = wl.make_linear("tiny_m37_k256_n384")
    q, a = oracle.quant_act(case.x_bits, case.inv_s)
    xs = wl.bits_to_f32(case.x_bits).astype(np.float64) * case.inv_s.astype(np.float64)
    assert np.abs(q.astype(np.int32)).max() <= 127
    for m in range(case.M):
        amax = np.abs(xs[m]).max()
        j = int(np.argmax(np.abs(xs[m])))
        assert abs(int(q[m, j])) == 127
        assert np.all(np.sign(q[m]) * np.sign(xs[m]) >= 0)
        # dequantisation error: at most half a step, plus the fp32 roundings
        step = amax / 127.0
        err = np.abs(q[m].astype(np.float64) * step - xs[m])
        assert err.max() <= 0.5 * step * (1 + 1e-5) + 1e-6 * amax


def test_quant_power_of_two_equivariance_and_unit_smoothing():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((9, 128)).astype(np.float32)
    q0, a0 = oracle.quant_act(bits(x), None)
    q1, a1 = oracle.quant_act(bits(x * np.float32(2.0 ** 9)), None)
    assert np.array_equal(q0, q1)
    assert np.array_equal(a1, a0 * np.float32(2.0 ** 9))
    q2, a2 = oracle.quant_act(bits(x), np.ones(128, np.float32))
    assert np.array_equal(q0, q2) and np.array_equal(a0, a2)
    # smoothing by 2^-k on input scaled by 2^k is the identity
    s = np.exp2(rng.integers(-6, 7, size=128)).astype(np.float32)
    q3, a3 = oracle.quant_act(bits(x * s), (1.0 / s).astype(np.float32))
    assert np.array_equal(q0, q3) and np.array_equal(a0, a3)


def test_quant_tiny_rows_are_zero():
    x = np.zeros((2, 32), np.float32)
    x[1, 5] = np.float32(2.0 ** -125)    # amax below 2^-120: treated as zero
    q, a = oracle.quant_act(bits(x), None)
    assert not q.any() and not a.any()


def test_quant_matches_library_binary32_arithmetic():
    # numpy's float32 ufuncs are single IEEE RN operations; np.rint ties to even
    case = wl.make_linear("tiny_m37_k256_n384")
    xf = wl.bits_to_f32(case.x_bits)
    xs = xf * case.inv_s
    amax = np.abs(xs).max(axis=1)
    inv_a = np.float32(127.0) / amax
    qn = np.clip(np.rint(xs * inv_a[:, None]), -127, 127).astype(np.int8)
    q, a = oracle.quant_act(case.x_bits, case.inv_s)
    assert np.array_equal(q, qn)
    assert np.array_equal(a, amax / np.float32(127.0))


# ------------------------------------------------------- contraction -------
def test_gemm_brute_force_tiny():
    rng = np.random.default_rng(5)
    for M, N, K in [(1, 1, 1), (2, 3, 16), (5, 4, 64), (3, 5, 33)]:
        q = rng.integers(-127, 128, size=(M, K), dtype=np.int8)
        w = rng.integers(-127, 128, size=(N, K), dtype=np.int8)
        acc = oracle.gemm_s32(q, w)
        for m in range(M):
            for n in range(N):
                assert acc[m, n] == sum(int(q[m, k]) * int(w[n, k]) for k in range(K))


def test_gemm_sign_patterns_and_extremes():
    # every sign pattern of 4 extreme terms, plus mixed magnitudes
    K = 4
    pats = np.array([[127 if (p >> i) & 1 else -127 for i in range(K)] for p in range(16)], np.int8)
    acc = oracle.gemm_s32(pats, pats)
    for i in range(16):
        for j in range(16):
            assert acc[i, j] == sum(int(pats[i, k]) * int(pats[j, k]) for k in range(K))


def test_gemm_matches_numpy_int64():
    case = wl.make_linear("tiny_m37_k256_n384")
    q, _ = oracle.quant_act(case.x_bits, case.inv_s)
    ref = q.astype(np.int64) @ case.w.astype(np.int64).T
    assert np.array_equal(oracle.gemm_s32(q, case.w), ref)
    rng = np.random.default_rng(1)
    w = wl.draw_weights(rng, (96, 5120), "normal")
    q2 = rng.integers(-127, 128, size=(12, 5120), dtype=np.int8)
    assert np.array_equal(oracle.gemm_s32(q2, w), q2.astype(np.int64) @ w.astype(np.int64).T)


@pytest.mark.parametrize("S", [1, 2, 3, 4, 7, 16, 64])
def test_gemm_split_k_invariant(S):
    rng = np.random.default_rng(S)
    q = rng.integers(-127, 128, size=(7, 1040), dtype=np.int8)
    w = rng.integers(-127, 128, size=(9, 1040), dtype=np.int8)
    assert np.array_equal(oracle.gemm_s32_splitk(q, w, S), oracle.gemm_s32(q, w))


def test_gemm_int32_range_closed_form():
    K = 133136   # largest multiple of 16 with K * 127^2 < 2^31
    assert K <= oracle.max_k() == 133144
    q = np.full((2, K), 127, np.int8)
    q[1] = -127
    w = np.full((1, K), 127, np.int8)
    acc = oracle.gemm_s32(q, w)
    assert acc[0, 0] == K * 16129 and acc[1, 0] == -K * 16129
    with pytest.raises(OverflowError):
        oracle.gemm_s32(np.full((1, 133145), 127, np.int8), np.full((1, 133145), 127, np.int8))


# ------------------------------------------------------------- epilogue ----
def _ep(acc, a, w, r=None):
    acc = np.array([[acc]], np.int32)
    rb = None if r is None else np.array([[r]], np.uint16)
    return int(oracle.epilogue(acc, np.array([a], np.float32), np.array([w], np.float32), rb)[0, 0])


def test_epilogue_small_integers_exact():
    accs = np.arange(-256, 257, dtype=np.int32).reshape(1, -1)
    out = oracle.epilogue(accs, np.ones(1, np.float32), np.ones(513, np.float32), None)
    assert np.array_equal(wl.bits_to_f32(out), accs.astype(np.float32))


def test_epilogue_zero_acc_returns_residual():
    rng = np.random.default_rng(2)
    r = bits(rng.standard_normal((3, 50)).astype(np.float32))
    out = oracle.epilogue(np.zeros((3, 50), np.int32), np.full(3, 0.01, np.float32),
                          np.full(50, 0.003, np.float32), r)
    assert np.array_equal(out, r)


def test_epilogue_int_to_float_and_bf16_ties():
    # int32 -> binary32 is round-to-nearest-even
    assert _ep(16777217, 1.0, 1.0) == rnbf16_bits(16777216)
    assert _ep(16777219, 1.0, 1.0) == rnbf16_bits(16777220)
    # bf16 ties to even: 257/256 lies halfway between 1 and 1 + 2^-7
    assert _ep(257, 2.0 ** -8, 1.0) == 0x3F80
    assert _ep(259, 2.0 ** -8, 1.0) == 0x3F82
    assert _ep(-259, 2.0 ** -8, 1.0) == 0xBF82


def test_epilogue_power_of_two_scales_closed_form():
    rng = np.random.default_rng(9)
    for acc in rng.integers(-2 ** 28, 2 ** 28, size=200):
        got = _ep(int(acc), 2.0 ** -7, 2.0 ** -11)
        assert got == rnbf16_bits(Fr(rn32(int(acc))) / 2 ** 18)


def test_epilogue_rounding_order_reading():
    # Reading: ((acc * a_scale) * w_scale) + residual, each step one binary32
    # RN operation, no FMA.  The final bf16 rounding hides most binary32
    # differences, so search (vectorised, numpy binary32) for inputs where the
    # other orders land on other bf16 values, then check the oracle against
    # exact-rational evaluation of the stated order on those inputs.
    rng = np.random.default_rng(4)
    n = 2_000_000
    acc = rng.integers(-2 ** 24, 2 ** 24, size=n).astype(np.int32)
    a = rng.uniform(1e-4, 1e-1, n).astype(np.float32)
    w = rng.uniform(1e-3, 2e-2, n).astype(np.float32)
    rb = bits((rng.standard_normal(n) * 64).astype(np.float32))
    r = wl.bits_to_f32(rb)
    t1 = acc.astype(np.float32) * a
    want = wl.bf16_bits((t1 * w) + r)
    alt = wl.bf16_bits((acc.astype(np.float32) * (a * w)) + r)
    fma = wl.bf16_bits(((t1.astype(np.float64) * w.astype(np.float64)) + r.astype(np.float64)).astype(np.float32))
    idx_order = np.nonzero(alt != want)[0][:20]
    idx_fma = np.nonzero(fma != want)[0][:20]
    assert idx_order.size > 0 and idx_fma.size > 0
    for i in np.concatenate([idx_order, idx_fma]):
        A, S, W, R = int(acc[i]), float(a[i]), float(w[i]), float(r[i])
        e1 = rn32(Fr(rn32(A)) * Fr(S))
        e2 = rn32(Fr(e1) * Fr(W))
        expect = rnbf16_bits(Fr(rn32(Fr(e2) + Fr(R))))
        other_order = rnbf16_bits(Fr(rn32(Fr(rn32(Fr(rn32(A)) * Fr(rn32(Fr(S) * Fr(W))))) + Fr(R))))
        fused = rnbf16_bits(Fr(rn32(Fr(e1) * Fr(W) + Fr(R))))
        assert expect != other_order or expect != fused
        assert _ep(A, S, W, int(rb[i])) == expect


def test_epilogue_matches_library_ops():
    import torch
    rng = np.random.default_rng(6)
    acc = rng.integers(-2 ** 27, 2 ** 27, size=(17, 40)).astype(np.int32)
    a = rng.uniform(1e-3, 1e-1, 17).astype(np.float32)
    w = rng.uniform(1e-3, 2e-2, 40).astype(np.float32)
    r = bits(rng.standard_normal((17, 40)).astype(np.float32))
    t = ((acc.astype(np.float32) * a[:, None]) * w[None, :]) + wl.bits_to_f32(r)
    ref = torch.from_numpy(t).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.epilogue(acc, a, w, r), ref)
    t0 = (acc.astype(np.float32) * a[:, None]) * w[None, :]
    ref0 = torch.from_numpy(t0).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.epilogue(acc, a, w, None), ref0)


def test_linear_batch_invariance():
    case = wl.make_linear("tiny_m37_k256_n384")
    q, a = oracle.quant_act(case.x_bits, case.inv_s)
    out, acc = oracle.w8a8_linear(q, a, case.w, case.w_scale, case.residual_bits)
    perm = np.random.default_rng(0).permutation(case.M)
    qp, ap = oracle.quant_act(case.x_bits[perm], case.inv_s)
    outp, _ = oracle.w8a8_linear(qp, ap, case.w, case.w_scale, case.residual_bits[perm])
    assert np.array_equal(outp, out[perm])
    for m in (0, 17, 36):
        q1, a1 = oracle.quant_act(case.x_bits[m:m + 1], case.inv_s)
        o1, _ = oracle.w8a8_linear(q1, a1, case.w, case.w_scale, case.residual_bits[m:m + 1])
        assert np.array_equal(o1[0], out[m])


# ------------------------------------------------------------------ exp ----
def test_exp_exact_points_and_underflow():
    assert oracle.exp(np.array([0.0], np.float32))[0] == np.float32(1.0)
    y = oracle.exp(np.array([-88.0, -100.0, -1e30], np.float32))
    assert np.all(y == 0.0)


def test_exp_error_bound_two_ulp():
    xs = np.concatenate([np.linspace(-87.0, 0.0, 400_001, dtype=np.float32),
                         -np.abs(np.random.default_rng(0).standard_normal(100_000).astype(np.float32)) * 10,
                         np.float32(-np.logspace(-30, 0, 2000))])
    y = oracle.exp(xs).astype(np.float64)
    ref = np.exp(xs.astype(np.float64))
    ulp = np.spacing(ref.astype(np.float32)).astype(np.float64)
    err = np.abs(y - ref) / ulp
    assert err.max() <= 2.0, float(err.max())


# ------------------------------------------------------------- read-out ----
def _full_logits(h_bits, inv_s, W, lm_scale):
    q, a = oracle.quant_act(h_bits, inv_s)
    acc = oracle.gemm_s32(q, W)
    return (acc.astype(np.float32) * a[:, None]) * lm_scale[None, :]


def test_readout_identity_on_subvocabulary():
    # The pages' identity: softmax over the candidate logits equals the
    # full-vocabulary softmax gathered on the candidates and renormalised.
    case = wl.make_readout("identity_p16_v32000", P=6)
    W = case.lm_head_full()
    rc, logits, probs = oracle.candidate_readout(case.h_bits, None, W, case.lm_scale,
                                                 case.cand_offsets, case.cand_ids)
    assert rc == 0
    full = _full_logits(case.h_bits, None, W, case.lm_scale).astype(np.float64)
    for p in range(case.P):
        b, e = case.cand_offsets[p], case.cand_offsets[p + 1]
        ids = case.cand_ids[b:e]
        z = full[p] - full[p].max()
        sm = np.exp(z) / np.exp(z).sum()
        ren = sm[ids] / sm[ids].sum()
        assert np.array_equal(logits[b:e], full[p, ids].astype(np.float32))
        d = np.abs(probs[b:e] - ren)
        # 1e-6 relative to the position's probability vector (its largest entry)
        assert d.max() <= 1e-6 * ren.max(), (p, probs[b:e], ren)
        # per element: binary32 error of (logit - max) grows with its magnitude
        x = (logits[b:e].astype(np.float64) - logits[b:e].max())
        bound = (np.abs(x) + (e - b) + 4) * 2.0 ** -23 * ren
        assert np.all(d <= bound + 1e-38), (p, d, bound)


def test_readout_single_candidate_and_ties():
    rng = np.random.default_rng(12)
    K = 256
    W = rng.integers(-127, 128, size=(20, K), dtype=np.int8)
    W[5] = W[3]
    W[9] = W[3]
    W[11] = W[3]
    sc = np.full(20, 0.01, np.float32)
    h = bits(rng.standard_normal((2, K)).astype(np.float32))
    off = np.array([0, 1, 5], np.int32)
    ids = np.array([7, 3, 5, 9, 11], np.int32)
    rc, logits, probs = oracle.candidate_readout(h, None, W, sc, off, ids)
    assert rc == 0
    assert probs[0] == np.float32(1.0)
    assert np.all(logits[1:] == logits[1]) and np.all(probs[1:] == np.float32(0.25))


def test_readout_rejects_bad_candidates():
    rng = np.random.default_rng(13)
    K, V = 64, 30
    W = rng.integers(-127, 128, size=(V, K), dtype=np.int8)
    sc = np.full(V, 0.01, np.float32)
    h = bits(rng.standard_normal((4, K)).astype(np.float32))
    off = np.array([0, 2, 4, 6, 8], np.int32)
    ids = np.array([1, 2, 3, 3, 4, 30, 5, 6], np.int32)   # dup in p1, out-of-range in p2
    rc, logits, probs = oracle.candidate_readout(h, None, W, sc, off, ids)
    assert rc < 0
    assert np.isnan(probs[2:6]).all() and np.isfinite(probs[[0, 1, 6, 7]]).all()
    off2 = np.array([0, 0, 2], np.int32)                  # an empty position
    rc, _, probs = oracle.candidate_readout(h[:2], None, W, sc, off2, ids[:2])
    assert rc == -2 and np.isfinite(probs).all()
    off3 = np.array([0, 65], np.int32)                    # over the cap
    ids3 = np.arange(65, dtype=np.int32) % V
    rc, _, _ = oracle.candidate_readout(h[:1], None, np.concatenate([W, W, W]),
                                        np.concatenate([sc, sc, sc]), off3, np.arange(65, dtype=np.int32))
    assert rc == -2


def test_readout_probs_sum_and_logit_consistency():
    case = wl.make_readout("readout_p192_v248000", P=24)
    uniq = np.unique(case.cand_ids)
    rows = case.lm_rows(uniq)
    remap = np.searchsorted(uniq, case.cand_ids).astype(np.int32)
    rc, logits, probs = oracle.candidate_readout(case.h_bits, None, rows, case.lm_scale[uniq],
                                                 case.cand_offsets, remap)
    assert rc == 0
    for p in range(case.P):
        b, e = case.cand_offsets[p], case.cand_offsets[p + 1]
        assert abs(float(probs[b:e].astype(np.float64).sum()) - 1.0) <= (e - b + 1) * 2 ** -23
        full = _full_logits(case.h_bits[p:p + 1], None, rows[remap[b:e]], case.lm_scale[case.cand_ids[b:e]])
        assert np.array_equal(full[0], logits[b:e])


def test_readout_softmax_arithmetic_exact_rationals():
    # Given the (pinned) logits and exp, the read-out's last steps are
    # binary32 RN: x = logit - max, s = e_1 + e_2 + ... in candidate order,
    # prob = e_i / s.  Check every bit against exact rationals.
    case = wl.make_readout("readout_p192_v248000", P=12)
    uniq = np.unique(case.cand_ids)
    rows = case.lm_rows(uniq)
    remap = np.searchsorted(uniq, case.cand_ids).astype(np.int32)
    rc, logits, probs = oracle.candidate_readout(case.h_bits, None, rows, case.lm_scale[uniq],
                                                 case.cand_offsets, remap)
    assert rc == 0
    for p in range(case.P):
        b, e = case.cand_offsets[p], case.cand_offsets[p + 1]
        lg = [float(v) for v in logits[b:e]]
        mx = max(lg)
        xs = [rn32(Fr(v) - Fr(mx)) for v in lg]
        ev = [float(v) for v in oracle.exp(np.array(xs, np.float32))]
        s = Fr(0)
        for v in ev:
            s = Fr(rn32(s + Fr(v))) if v or s else s
        for i, v in enumerate(ev):
            want = rn32(Fr(v) / s) if v else 0.0
            assert probs[b + i] == np.float32(want), (p, i)


# ---------------------------------------------- restriction to answer rows ---
# StartLux-Prism, "Compute shared evidence once": the last layer computes only
# the positions needed for answers.  Every step is per token, so the
# restricted layer must reproduce the full layer's rows at those positions:
# the pins compare the row-indexed oracle functions with the full ones.

def _layer_inputs(seed, M_x=40, K=256, N=96):
    rng = np.random.default_rng(seed)
    x = wl.bf16_bits(rng.standard_normal((M_x, K), dtype=np.float32) * 3)
    inv_s = rng.uniform(0.5, 2.0, K).astype(np.float32)
    w = wl.draw_weights(rng, (N, K), "normal")
    ws = rng.uniform(0.001, 0.02, N).astype(np.float32)
    res = wl.bf16_bits(rng.standard_normal((M_x, N), dtype=np.float32))
    return x, inv_s, w, ws, res


def test_rows_quantiser_is_the_full_quantiser_on_those_rows():
    x, inv_s, *_ = _layer_inputs(1)
    rows = np.array([7, 0, 39, 7, 13], np.int32)           # any order, repeats allowed
    q_full, a_full = oracle.quant_act(x, inv_s)
    q, a, err = oracle.quant_act_rows(x, rows, inv_s)
    assert err == 0
    assert np.array_equal(q, q_full[rows])
    assert np.array_equal(a.view(np.uint32), a_full[rows].view(np.uint32))


def test_restricted_layer_equals_full_layer_rows():
    x, inv_s, w, ws, res = _layer_inputs(2)
    rows = np.array([39, 2, 20], np.int32)
    q_full, a_full = oracle.quant_act(x, inv_s)
    out_full, acc_full = oracle.w8a8_linear(q_full, a_full, w, ws, res)
    q, a, err = oracle.quant_act_rows(x, rows, inv_s)
    out, acc, err2 = oracle.w8a8_linear_rows(q, a, w, ws, res, rows)
    assert err == 0 and err2 == 0
    assert np.array_equal(acc, acc_full[rows])
    assert np.array_equal(out, out_full[rows])
    # the residual row is the one the index names, not the output row's own
    out_wrong, _, _ = oracle.w8a8_linear_rows(q, a, w, ws, res, np.arange(3, dtype=np.int32))
    assert not np.array_equal(out_wrong, out)


def test_rows_out_of_range_flag_and_poison_only_their_row():
    x, inv_s, w, ws, res = _layer_inputs(3)
    q, a, err = oracle.quant_act_rows(x, np.array([5, -1, 40], np.int32), inv_s)
    assert err == oracle.ERR_ROW_RANGE
    assert np.isnan(a[1]) and np.isnan(a[2]) and not np.isnan(a[0])
    assert not q[1:].any()
    q_ok, a_ok, _ = oracle.quant_act_rows(x, np.array([5, 6, 7], np.int32), inv_s)
    out, _, err = oracle.w8a8_linear_rows(q_ok, a_ok, w, ws, res, np.array([5, 40, 7], np.int32))
    assert err == oracle.ERR_ROW_RANGE
    assert (out[1] == 0x7FC0).all()
    good, _, _ = oracle.w8a8_linear_rows(q_ok, a_ok, w, ws, res, np.array([5, 6, 7], np.int32))
    assert np.array_equal(out[[0, 2]], good[[0, 2]])


def test_rows_empty_selection():
    x, inv_s, *_ = _layer_inputs(4)
    q, a, err = oracle.quant_act_rows(x, np.zeros(0, np.int32), inv_s)
    assert q.shape == (0, x.shape[1]) and a.shape == (0,) and err == 0


# ------------------------------------------ tensor-parallel integer combine ---
# StartLux-Prism, "Bitwise consistency is not lossless quantization": with
# tensor parallelism the int32 partial sums are combined before any scaling,
# so the layer gives the same bits on any number of GPUs.  A row-parallel
# rank holds a K-shard of every token row: the ranks agree on the row's
# scale through a MAX all-reduce of their shard maxima, then SUM their exact
# partials.

def _tp_inputs(seed, M=24, K=320, N=72):
    rng = np.random.default_rng(seed)
    x = wl.bf16_bits(rng.standard_normal((M, K), dtype=np.float32) * 2)
    x[:, 7] = wl.bf16_bits(rng.standard_normal(M, dtype=np.float32) * 40)   # an outlier channel
    inv_s = rng.uniform(0.5, 2.0, K).astype(np.float32)
    w = wl.draw_weights(rng, (N, K), "uniform")
    ws = rng.uniform(0.001, 0.02, N).astype(np.float32)
    res = wl.bf16_bits(rng.standard_normal((M, N), dtype=np.float32))
    return x, inv_s, w, ws, res


def test_act_amax_restated_in_numpy():
    x, inv_s, *_ = _tp_inputs(11)
    xs = wl.bits_to_f32(x) * inv_s                      # binary32 products, RN
    assert np.array_equal(oracle.act_amax(x, inv_s).view(np.uint32),
                          np.abs(xs).max(axis=1).astype(np.float32).view(np.uint32))


def test_quant_with_a_larger_shared_amax_restated_in_numpy():
    """A rank quantises its shard with the whole row's (larger) maximum:
    q = clip(rint(xs * RN(127 / amax))), scale RN(amax / 127)."""
    x, inv_s, *_ = _tp_inputs(12)
    amax = oracle.act_amax(x, inv_s) * np.float32(3.0)
    q, a = oracle.quant_act_amax(x[:, :100], inv_s[:100], amax)
    xs = wl.bits_to_f32(x[:, :100]) * inv_s[:100]
    inv = (np.float32(127.0) / amax).astype(np.float32)
    ref = np.clip(np.rint((xs * inv[:, None]).astype(np.float32)), -127, 127).astype(np.int8)
    assert np.array_equal(q, ref)
    assert np.array_equal(a.view(np.uint32), (amax / np.float32(127.0)).astype(np.float32).view(np.uint32))
    assert np.abs(q).max() < 127                        # this shard does not hold the row maximum


@pytest.mark.parametrize("bounds", [[0, 160, 320], [0, 16, 48, 320], [0, 304, 320], [0, 64, 128, 192, 256, 320]])
def test_tp_row_parallel_equals_one_device(bounds):
    x, inv_s, w, ws, res = _tp_inputs(13)
    q, a = oracle.quant_act(x, inv_s)
    out1, acc1 = oracle.w8a8_linear(q, a, w, ws, res)
    out, acc, parts = oracle.tp_row_parallel_linear(x, inv_s, w, ws, res, bounds)
    assert np.array_equal(acc, acc1)
    assert np.array_equal(out, out1)
    # each rank's partial is its shard's own contraction with the shared scale
    assert len(parts) == len(bounds) - 1 and not np.array_equal(parts[0], acc1)


# ------------------------------------------------------------------- W4A8 ---
# StartLux-Prism, "Compute shared evidence once" (Q4_K_M files, a W4A8 run):
# 4-bit codes packed two per byte, then the W8A8 definition on the codes.

def test_unpack_w4_every_byte_restated_with_shifts():
    b = np.arange(256, dtype=np.uint8)[None, :]
    got = oracle.unpack_w4(b, 512)
    lo = (b.astype(np.int8) << 4).astype(np.int8) >> 4        # arithmetic shifts on int8
    hi = b.astype(np.int8) >> 4
    want = np.empty((1, 512), np.int8)
    want[:, 0::2], want[:, 1::2] = lo, hi
    assert np.array_equal(got, want)
    assert got.min() == -8 and got.max() == 7


def test_pack_then_unpack_is_identity():
    rng = np.random.default_rng(5)
    codes = rng.integers(-8, 8, size=(7, 96)).astype(np.int8)
    assert np.array_equal(oracle.unpack_w4(wl.pack_w4(codes), 96), codes)


def test_w4a8_brute_force_from_nibbles():
    rng = np.random.default_rng(6)
    M, K, N = 3, 32, 5
    q = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    w4 = rng.integers(0, 256, size=(N, K // 2)).astype(np.uint8)
    a = rng.uniform(1e-3, 1e-2, M).astype(np.float32)
    s = rng.uniform(1e-3, 1e-2, N).astype(np.float32)
    res = wl.bf16_bits(rng.standard_normal((M, N), dtype=np.float32))

    def nib(byte, high):
        v = (int(byte) >> 4) if high else (int(byte) & 15)
        return v - 16 if v >= 8 else v
    acc = np.array([[sum(int(q[m, k]) * nib(w4[n, k // 2], k % 2) for k in range(K)) for n in range(N)]
                    for m in range(M)], np.int64)
    out, acc_o = oracle.w4a8_linear(q, a, w4, s, res)
    assert np.array_equal(acc_o, acc)
    assert np.array_equal(out, oracle.epilogue(acc.astype(np.int32), a, s, res))


def test_w4a8_extremes_at_max_k():
    K = 133136
    q = np.full((2, K), 127, np.int8)
    q[1] = -127
    w4 = np.full((2, K // 2), 0x88, np.uint8)                 # every code -8
    w4[1] = 0x77                                              # every code 7
    _, acc = oracle.w4a8_linear(q, np.ones(2, np.float32), w4, np.ones(2, np.float32))
    assert acc.tolist() == [[-K * 127 * 8, K * 127 * 7], [K * 127 * 8, -K * 127 * 7]]


# ------------------------------------------- column-parallel read-out ----
def _shard_bounds(V, n, rng):
    cuts = np.sort(rng.choice(np.arange(1, V), size=n - 1, replace=False))
    return [0] + [int(c) for c in cuts] + [V]


def test_shard_logits_whole_head_is_the_readout():
    """The shard function over the whole head gives the (pinned) read-out's
    logits bit for bit, invalid positions included."""
    rng = np.random.default_rng(21)
    K, V = 128, 40
    W = rng.integers(-127, 128, size=(V, K), dtype=np.int8)
    sc = rng.uniform(0.001, 0.02, V).astype(np.float32)
    h = bits(rng.standard_normal((5, K)).astype(np.float32))
    off = np.array([0, 3, 5, 8, 10, 12], np.int32)
    ids = np.array([4, 9, 31, 2, 2, 7, 40, 1, 39, 0, 17, 23], np.int32)   # dup in p1, range in p2
    rc0, lg0, _ = oracle.candidate_readout(h, None, W, sc, off, ids)
    rc1, lg1 = oracle.candidate_logits_shard(h, None, W, sc, 0, V, off, ids)
    assert rc0 == rc1 < 0
    assert np.array_equal(lg0.view(np.uint32), lg1.view(np.uint32))


@pytest.mark.parametrize("n", [2, 3, 5])
def test_shard_logits_sum_to_the_readout(n):
    """Every candidate belongs to exactly one shard and the others write
    -0.0, so adding the shards' outputs in any order reproduces the one-head
    logits bit for bit (signs of zero included); the softmax of the sum is
    the read-out's probabilities bit for bit."""
    rng = np.random.default_rng(30 + n)
    case = wl.make_readout("readout_p192_v248000", P=12)
    uniq = np.unique(case.cand_ids)
    rows = case.lm_rows(uniq)
    ids = np.searchsorted(uniq, case.cand_ids).astype(np.int32)
    V = rows.shape[0]
    sc = case.lm_scale[uniq]
    rc, lg, pr = oracle.candidate_readout(case.h_bits, None, rows, sc, case.cand_offsets, ids)
    assert rc == 0
    bounds = _shard_bounds(V, n, rng)
    parts = []
    for r in range(n):
        v0, v1 = bounds[r], bounds[r + 1]
        rc_r, lg_r = oracle.candidate_logits_shard(case.h_bits, None, rows[v0:v1], sc[v0:v1], v0, V,
                                                   case.cand_offsets, ids)
        assert rc_r == 0
        owned = (ids >= v0) & (ids < v1)
        assert np.array_equal(lg_r[owned].view(np.uint32), lg[owned].view(np.uint32))
        assert np.all(lg_r[~owned].view(np.uint32) == np.float32(-0.0).view(np.uint32))
        parts.append(lg_r)
    for order in (range(n), reversed(range(n))):
        tot = np.full_like(lg, -0.0)
        for r in order:
            tot = (tot + parts[r]).astype(np.float32)
        assert np.array_equal(tot.view(np.uint32), lg.view(np.uint32))
    rc_s, pr_s = oracle.candidate_softmax(lg, case.cand_offsets)
    assert rc_s == 0 and np.array_equal(pr_s.view(np.uint32), pr.view(np.uint32))


def test_candidate_softmax_invalid_positions():
    lg = np.array([0.5, np.nan, 1.0, 2.0, 3.0], np.float32)
    rc, pr = oracle.candidate_softmax(lg, np.array([0, 2, 5], np.int32))
    assert rc == 0 and np.isnan(pr[:2]).all() and np.isfinite(pr[2:]).all()
    rc, pr = oracle.candidate_softmax(lg[2:], np.array([0, 0, 3], np.int32))
    assert rc == -2 and np.isfinite(pr).all()
