"""Host checks of the exactness argument behind the requantisation kernel's
arithmetic (StartLux-Prism, "Compute shared evidence once": Q8_0 weights
requantised with the smoothing factors folded in).

The kernel forms c * d for an int8 code c and a binary16 block scale d with
one fused multiply-add on the 2^23 binade,
    F * (d / 256) - (2^15 + 2^7) * d,   F = 2^23 + 256 * (c + 128),
and rounds t = RN(v * RN(127 / amax)) to an integer as the low byte of
RN(t + 1.5 * 2^23).  Both are exact only under conditions on the operands;
these tests check those conditions for every finite binary16 scale, every
code and every value t can take, in float64 (which holds every product here
exactly), independently of the GPU."""
import numpy as np


def finite_f16():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = h.view(np.float16)
    return f[np.isfinite(f)].astype(np.float64)


def representable_f32(x: np.ndarray) -> np.ndarray:
    return x.astype(np.float32).astype(np.float64) == x


def test_decode_constants_are_exact_binary32():
    d = finite_f16()
    assert representable_f32(d / 256).all()                 # d / 256: a power-of-two scaling
    assert representable_f32(d * 32896.0).all()            # (2^15 + 2^7) d: <= 20 significant bits


def test_fused_decode_equals_code_times_scale_exactly():
    d = finite_f16()
    c = np.arange(-127, 128, dtype=np.float64)
    F = 2.0 ** 23 + 256.0 * (c + 128.0)
    assert representable_f32(F).all()
    # exact value of the fused operation: F * (d/256) - 32896 d, all in float64
    exact = F[None, :] * (d[:, None] / 256.0) - 32896.0 * d[:, None]
    assert np.array_equal(exact, c[None, :] * d[:, None])
    # and that value needs no rounding in binary32, so the single rounding of
    # the fused operation returns it unchanged
    assert representable_f32(c[None, :] * d[:, None]).all()


def test_rounding_by_the_binade_ulp_is_round_half_even():
    # every binary32 t with |t| <= 127.00002 on a fine grid plus every tie
    ties = np.arange(-127, 127, dtype=np.float32) + np.float32(0.5)
    t = np.concatenate([
        np.linspace(-127.00002, 127.00002, 2_000_001, dtype=np.float32),
        ties, np.nextafter(ties, np.float32(0)), np.nextafter(ties, np.float32(200)),
        np.nextafter(ties, np.float32(-200)),
    ])
    t = t[np.abs(t) <= np.float32(127.00002)]
    s = (t + np.float32(12582912.0)).astype(np.float32)     # binary32 RN addition
    low = (s.view(np.uint32) & 0xFF).astype(np.uint8).view(np.int8)
    assert np.array_equal(low.astype(np.int64), np.rint(t.astype(np.float64)).astype(np.int64))
    assert np.abs(np.rint(t.astype(np.float64))).max() <= 127
