"""Seeded synthetic inputs for the W8A8 linear layer and the candidate read-out.

This module only draws inputs.  It holds none of the layer's arithmetic (no
quantiser, contraction, epilogue or softmax); both the CUDA path's tests and
benchmark and the CPU oracle take their inputs from here.

Workloads follow the shapes of the StartLux-Prism pages: a 27B decision model
with hidden size 5120 and FFN width 17408, a ~248,000-token vocabulary, short
requests of 256 evidence tokens plus three 16-token questions, 64 clients x 32
tokens under load, decode-like single rows, and 2-10 answer candidates per
answer position.  No dataset is used; every array is drawn from numpy's PCG64
generator with a fixed seed.

Draw recipe (per linear case, in this order): outlier channel indices,
activations X ~ N(0,1) (float32 draws) with the outlier columns multiplied by
the outlier factor, rounded to bf16 (round to nearest even); weights; weight
scales ~ U(0.001, 0.02); residual ~ N(0,1) in bf16.  Weights are either
``uniform`` integers in [-127, 127] or ``normal``: clip(rint(40 * N(0,1)),
-127, 127).

The SmoothQuant smoothing vector is a model parameter, not part of the hot
path's arithmetic: the path receives inv_s = 1/s and multiplies.  It is
synthesised here in float64 with the standard SmoothQuant migration
s_k = max|X[:,k]|^alpha / max|W_deq[:,k]|^(1-alpha) (alpha = 0.5, W_deq =
w * w_scale; s_k = 1 where either maximum is 0) and rounded once to float32.
"""
from __future__ import annotations

import dataclasses

import numpy as np

HIDDEN = 5120
FFN = 17408
VOCAB = 248_000


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 array -> bf16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bits_to_f32(h: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 (exact)."""
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def draw_weights(rng: np.random.Generator, shape, dist: str) -> np.ndarray:
    if dist == "uniform":
        return rng.integers(-127, 128, size=shape, dtype=np.int8)
    if dist == "normal":
        g = rng.standard_normal(shape, dtype=np.float32)
        g *= np.float32(40.0)
        np.rint(g, out=g)
        np.clip(g, -127, 127, out=g)
        return g.astype(np.int8)
    raise ValueError(dist)


def smoothing_inv_s(x_bits: np.ndarray, w: np.ndarray, w_scale: np.ndarray,
                    alpha: float = 0.5) -> np.ndarray:
    """SmoothQuant migration factors as float32 1/s (see module docstring)."""
    xmax = np.abs(bits_to_f32(x_bits).astype(np.float64)).max(axis=0)
    wdeq_max = np.zeros(w.shape[1], np.float64)
    # per-input-channel max of |w[n,k]| * w_scale[n], in chunks to bound memory
    for n0 in range(0, w.shape[0], 4096):
        blk = np.abs(w[n0:n0 + 4096].astype(np.float64)) * w_scale[n0:n0 + 4096, None].astype(np.float64)
        np.maximum(wdeq_max, blk.max(axis=0), out=wdeq_max)
    s = np.ones_like(xmax)
    ok = (xmax > 0) & (wdeq_max > 0)
    s[ok] = xmax[ok] ** alpha / wdeq_max[ok] ** (1.0 - alpha)
    return (1.0 / s).astype(np.float32)


@dataclasses.dataclass
class LinearCase:
    name: str
    M: int
    K: int
    N: int
    x_bits: np.ndarray          # uint16 [M, K]  bf16 activations
    inv_s: np.ndarray | None    # float32 [K]
    w: np.ndarray               # int8 [N, K]
    w_scale: np.ndarray         # float32 [N]
    residual_bits: np.ndarray | None  # uint16 [M, N]


def linear_case(name: str, M: int, K: int, N: int, seed: int, *, residual: bool,
                n_outliers: int, outlier_mult: float, w_dist: str,
                smooth: bool = True, alpha: float = 0.5) -> LinearCase:
    rng = np.random.default_rng(seed)
    out_idx = rng.choice(K, size=n_outliers, replace=False) if n_outliers else np.zeros(0, np.int64)
    x = rng.standard_normal((M, K), dtype=np.float32)
    if n_outliers:
        x[:, out_idx] *= np.float32(outlier_mult)
    x_bits = bf16_bits(x)
    del x
    w = draw_weights(rng, (N, K), w_dist)
    w_scale = rng.uniform(0.001, 0.02, size=N).astype(np.float32)
    res = bf16_bits(rng.standard_normal((M, N), dtype=np.float32)) if residual else None
    inv_s = smoothing_inv_s(x_bits, w, w_scale, alpha) if smooth else None
    return LinearCase(name, M, K, N, x_bits, inv_s, w, w_scale, res)


# ----------------------------------------------------------------- configs --
# name -> (M, K, N, seed, residual, n_outliers, outlier_mult, w_dist)
LINEAR_CONFIGS = {
    # tiny: 37 rows, 4 outlier channels x20, uniform weights
    "tiny_m37_k256_n384": (37, 256, 384, 0, True, 4, 20.0, "uniform"),
    # short-request forest bucket: 256 evidence + 3 x 16 question tokens
    "forest_qkv_m304_k5120_n15360": (304, HIDDEN, 15360, 1, False, HIDDEN // 100, 30.0, "normal"),
    "forest_oproj_m304_k5120_n5120": (304, HIDDEN, HIDDEN, 2, True, HIDDEN // 100, 30.0, "normal"),
    # 64 clients x 32 tokens, FFN
    "load_gateup_m2048_k5120_n34816": (2048, HIDDEN, 2 * FFN, 3, False, HIDDEN // 100, 30.0, "normal"),
    "load_down_m2048_k17408_n5120": (2048, FFN, HIDDEN, 4, True, FFN // 100, 30.0, "normal"),
    # decode-like weight streaming (M in {1, 8, 16, 64} are row slices of M=64)
    "decode_m64_k17408_n5120": (64, FFN, HIDDEN, 5, True, FFN // 100, 30.0, "normal"),
    # long evidence
    "long_m8192_k5120_n5120": (8192, HIDDEN, HIDDEN, 6, True, HIDDEN // 100, 30.0, "normal"),
}
DECODE_M = (1, 8, 16, 64)
DECODE_SPLITS = (1, 4, 8, 16)


def make_linear(name: str, **overrides) -> LinearCase:
    M, K, N, seed, residual, n_out, mult, dist = LINEAR_CONFIGS[name]
    kw = dict(M=M, K=K, N=N, seed=seed, residual=residual, n_outliers=n_out,
              outlier_mult=mult, w_dist=dist)
    kw.update(overrides)
    return linear_case(name, kw.pop("M"), kw.pop("K"), kw.pop("N"), kw.pop("seed"),
                       residual=kw["residual"], n_outliers=kw["n_outliers"],
                       outlier_mult=kw["outlier_mult"], w_dist=kw["w_dist"],
                       **{k: v for k, v in kw.items() if k in ("smooth", "alpha")})


# ------------------------------------------------------------ read-out ------
@dataclasses.dataclass
class ReadoutCase:
    name: str
    P: int
    K: int
    V: int
    seed: int
    h_bits: np.ndarray          # uint16 [P, K]  bf16 hidden states
    cand_offsets: np.ndarray    # int32 [P+1]   CSR
    cand_ids: np.ndarray        # int32 [T]
    lm_scale: np.ndarray        # float32 [V]

    def lm_rows(self, ids) -> np.ndarray:
        """LM-head rows for the given ids: int8 [len(ids), K].  Row c is drawn
        from its own generator seeded (seed, 1, c), so any subset of rows can be
        produced without drawing the whole 248,000 x 5120 head."""
        ids = np.asarray(ids)
        out = np.empty((ids.size, self.K), np.int8)
        for i, c in enumerate(ids.tolist()):
            out[i] = draw_weights(np.random.default_rng([self.seed, 1, int(c)]), (self.K,), "normal")
        return out

    def lm_head_full(self) -> np.ndarray:
        return self.lm_rows(np.arange(self.V))


def readout_case(name: str, P: int, K: int, V: int, seed: int,
                 cmin: int = 2, cmax: int = 10) -> ReadoutCase:
    rng = np.random.default_rng([seed, 0])
    h = bf16_bits(rng.standard_normal((P, K), dtype=np.float32))
    counts = rng.integers(cmin, cmax + 1, size=P)
    ids = [rng.choice(V, size=int(c), replace=False) for c in counts]
    off = np.zeros(P + 1, np.int32)
    off[1:] = np.cumsum(counts)
    cand = np.concatenate(ids).astype(np.int32) if P else np.zeros(0, np.int32)
    lm_scale = rng.uniform(0.001, 0.02, size=V).astype(np.float32)
    return ReadoutCase(name, P, K, V, seed, h, off, cand, lm_scale)


READOUT_CONFIGS = {
    "readout_p192_v248000": (192, HIDDEN, VOCAB, 7),
    "identity_p16_v32000": (16, HIDDEN, 32_000, 8),
}


def make_readout(name: str, **overrides) -> ReadoutCase:
    P, K, V, seed = READOUT_CONFIGS[name]
    kw = dict(P=P, K=K, V=V, seed=seed)
    kw.update(overrides)
    return readout_case(name, kw["P"], kw["K"], kw["V"], kw["seed"],
                        kw.get("cmin", 2), kw.get("cmax", 10))


# ------------------------------------------------- Q8_0 weights as stored ---
# Load-time requantisation inputs: the stored 8-bit codes of a weight [N, K]
# in 32-wide blocks, one binary16 scale per block, and the smoothing vector s
# [K] that the requantisation folds in.  Recipe, in draw order: codes
# clip(rint(40 N(0,1))); block scales U(2e-4, 2e-3) rounded to binary16;
# s = exp(N(0, 0.5)) in float32 with 1% of channels (at least one) multiplied
# by 30, the outlier channels that SmoothQuant moves into the weights.
REQUANT_CONFIGS = {
    # name: (N, K, seed) -- the projections of the 27B model as loaded
    "qkv_n15360_k5120": (15360, HIDDEN, 11),
    "gateup_n34816_k5120": (2 * FFN, HIDDEN, 12),
    "down_n5120_k17408": (HIDDEN, FFN, 13),
}


@dataclasses.dataclass
class Q8Case:
    name: str
    q: np.ndarray        # int8 [N, K]
    d: np.ndarray        # uint16 binary16 bits [N, K/32]
    s: np.ndarray        # float32 [K]


def q8_0_case(name: str, N: int, K: int, seed: int) -> Q8Case:
    rng = np.random.default_rng(seed)
    q = draw_weights(rng, (N, K), "normal")
    d = rng.uniform(2e-4, 2e-3, size=(N, K // 32)).astype(np.float16).view(np.uint16)
    s = np.exp(rng.standard_normal(K) * 0.5).astype(np.float32)
    out = rng.choice(K, size=max(1, K // 100), replace=False)
    s[out] *= np.float32(30.0)
    return Q8Case(name, q, d, s)


def make_q8_0(name: str) -> Q8Case:
    N, K, seed = REQUANT_CONFIGS[name]
    return q8_0_case(name, N, K, seed)


# ------------------------------------------------------------ W4 weights ---
# 4-bit weights for W4A8: codes clip(rint(2.5 N(0,1)), -7, 7) (symmetric per
# output channel, the form a load-time requantisation leaves), packed two
# per byte, code 2j in the low nibble of byte j, code 2j+1 in the high one.
def draw_w4_codes(rng: np.random.Generator, shape) -> np.ndarray:
    g = rng.standard_normal(shape, dtype=np.float32) * np.float32(2.5)
    return np.clip(np.rint(g), -7, 7).astype(np.int8)


def pack_w4(codes: np.ndarray) -> np.ndarray:
    """int8 codes in [-8, 7], [N, K] with K even -> uint8 [N, K/2]."""
    c = codes.astype(np.int16) & 0xF
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
