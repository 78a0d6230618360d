"""CPU oracle for the batch-invariant W8A8 linear layer and candidate read-out.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the benchmark's CPU-baseline leg may import this package.  The product path
(the CUDA library and its Python binding) never imports, links or runs it.

The arithmetic lives in ``prism_oracle.c`` (plain C99, built with
``-ffp-contract=off`` and no fast-math, so each float operation is a single
binary32 round-to-nearest-even step in program order).  This module only
compiles it and marshals numpy arrays through ctypes.  See the C file's
header for the sources each function follows.

Parity status: every exported function is pinned by tests in
``tests/test_oracle_pins.py`` (brute force, closed forms, library routines,
invariants and the pages' candidate-softmax identity); none is unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "prism_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_BASE_FLAGS = ["-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-Wall"]


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (gcc, OpenMP if
    available).  Returns the library path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", *_BASE_FLAGS, "-fopenmp", _SRC, "-o", tmp, "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:  # no OpenMP runtime: build single-threaded
        cmd = ["gcc", *_BASE_FLAGS, _SRC, "-o", tmp, "-lm"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("oracle build failed:\n" + r.stderr)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P, I64, I32, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
        sig = {
            "oracle_quant_act": (None, [P, I64, P, I64, I64, P, I64, P]),
            "oracle_act_amax": (None, [P, I64, P, I64, I64, P]),
            "oracle_quant_act_amax": (None, [P, I64, P, P, I64, I64, P, I64, P]),
            "oracle_gemm_s32": (I32, [P, I64, P, I64, I64, I64, I64, P, I64]),
            "oracle_gemm_s32_splitk": (I32, [P, I64, P, I64, I64, I64, I64, I32, P, I64]),
            "oracle_epilogue": (None, [P, I64, P, P, P, I64, I64, I64, P, I64]),
            "oracle_w8a8_linear": (I32, [P, I64, P, P, I64, P, P, I64, I64, I64, I64, P, I64, P]),
            "oracle_quant_act_rows": (ctypes.c_uint32, [P, I64, I64, P, I64, P, I64, P, I64, P]),
            "oracle_w8a8_linear_rows": (I32, [P, I64, P, P, I64, P, P, I64, I64, P, I64, I64, I64, P, I64,
                                              P, P]),
            "oracle_unpack_w4": (None, [P, I64, I64, I64, P, I64]),
            "oracle_w4a8_linear": (I32, [P, I64, P, P, I64, P, P, I64, I64, I64, I64, P, I64, P, P]),
            "oracle_exp": (F, [F]),
            "oracle_exp_batch": (None, [P, I64, P]),
            "oracle_candidate_readout": (I32, [P, I64, P, P, I64, P, I64, I64, P, P, I64, I64, P, P]),
            "oracle_candidate_logits_shard": (I32, [P, I64, P, P, I64, P, I64, I64, I64, I64, P, P, I64, I64, P]),
            "oracle_candidate_softmax": (I32, [P, P, I64, I64, P]),
            "oracle_bf16_to_float": (None, [P, I64, P]),
            "oracle_f16_to_float": (None, [P, I64, P]),
            "oracle_smooth_requant": (None, [P, I64, P, I64, P, I64, I64, P, I64, P]),
            "oracle_float_to_bf16": (None, [P, I64, P]),
            "oracle_set_threads": (None, [I32]),
            "oracle_get_threads": (I32, []),
            "oracle_max_k": (I32, []),
            "oracle_max_candidates": (I32, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    """Contiguous array of exactly ``dtype`` (no value conversion allowed)."""
    a = np.ascontiguousarray(a)
    if a.dtype != np.dtype(dtype):
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return a


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def get_threads() -> int:
    return int(_load().oracle_get_threads())


def max_k() -> int:
    return int(_load().oracle_max_k())


def max_candidates() -> int:
    return int(_load().oracle_max_candidates())


def quant_act(x_bf16_bits: np.ndarray, inv_s: np.ndarray | None):
    """Per-token smoothed quantisation.  ``x_bf16_bits``: uint16 [M, K] (bf16
    bit patterns).  Returns (q int8 [M, K], a_scale float32 [M])."""
    x = _c(x_bf16_bits, np.uint16)
    M, K = x.shape
    s = None if inv_s is None else _c(inv_s, np.float32)
    q = np.empty((M, K), np.int8)
    a = np.empty((M,), np.float32)
    _load().oracle_quant_act(_p(x), K, _p(s), M, K, _p(q), K, _p(a))
    return q, a


def act_amax(x_bf16_bits: np.ndarray, inv_s: np.ndarray | None) -> np.ndarray:
    """Per-row max |x * inv_s| (the quantiser's first half), float32 [M]."""
    x = _c(x_bf16_bits, np.uint16)
    M, K = x.shape
    s = None if inv_s is None else _c(inv_s, np.float32)
    amax = np.empty((M,), np.float32)
    _load().oracle_act_amax(_p(x), K, _p(s), M, K, _p(amax))
    return amax


def quant_act_amax(x_bf16_bits: np.ndarray, inv_s: np.ndarray | None, amax: np.ndarray):
    """The quantiser's second half with given row maxima.  Returns (q, a_scale)."""
    x = _c(x_bf16_bits, np.uint16)
    M, K = x.shape
    s = None if inv_s is None else _c(inv_s, np.float32)
    am = _c(amax, np.float32)
    q = np.empty((M, K), np.int8)
    a = np.empty((M,), np.float32)
    _load().oracle_quant_act_amax(_p(x), K, _p(s), _p(am), M, K, _p(q), K, _p(a))
    return q, a


def tp_row_parallel_linear(x_bf16_bits, inv_s, w, w_scale, residual_bits, bounds):
    """A row-parallel tensor-parallel linear over the K shards [bounds[r],
    bounds[r+1]): each rank's shard row maxima, their maximum (the MAX
    all-reduce), each rank's codes with that maximum, its exact int32 partial
    contraction, the partials' sum (the SUM all-reduce), then the epilogue.
    Returns (out bf16 bits, acc int32, per-rank partials)."""
    amax = np.max(np.stack([act_amax(x_bf16_bits[:, b0:b1], None if inv_s is None else inv_s[b0:b1])
                            for b0, b1 in zip(bounds[:-1], bounds[1:])]), axis=0)
    parts, a_scale = [], None
    for b0, b1 in zip(bounds[:-1], bounds[1:]):
        q, a_scale = quant_act_amax(x_bf16_bits[:, b0:b1], None if inv_s is None else inv_s[b0:b1], amax)
        parts.append(gemm_s32(q, w[:, b0:b1]))
    total = np.sum(np.stack(parts).astype(np.int64), axis=0)
    assert np.abs(total).max(initial=0) <= 2**31 - 1
    acc = total.astype(np.int32)
    return epilogue(acc, a_scale, w_scale, residual_bits), acc, parts


def smooth_requant(q: np.ndarray, d_f16_bits: np.ndarray, s: np.ndarray | None):
    """SmoothQuant startup requantisation of Q8_0 weights.  ``q`` int8 [N, K]
    (K a multiple of 32), ``d_f16_bits`` uint16 [N, K/32] (binary16 block
    scales), ``s`` float32 [K] or None.  Returns (w int8 [N, K], w_scale
    float32 [N])."""
    q = _c(q, np.int8)
    N, K = q.shape
    assert K % 32 == 0
    d = _c(d_f16_bits, np.uint16)
    assert d.shape == (N, K // 32)
    sv = None if s is None else _c(s, np.float32)
    w = np.empty((N, K), np.int8)
    ws = np.empty((N,), np.float32)
    _load().oracle_smooth_requant(_p(q), K, _p(d), K // 32, _p(sv), N, K, _p(w), K, _p(ws))
    return w, ws


def f16_to_float(h) -> np.ndarray:
    h = _c(h, np.uint16)
    f = np.empty(h.shape, np.float32)
    _load().oracle_f16_to_float(_p(h), h.size, _p(f))
    return f


def gemm_s32(q: np.ndarray, w: np.ndarray) -> np.ndarray:
    """Exact int32 contraction acc[m, n] = sum_k q[m, k] * w[n, k]."""
    q = _c(q, np.int8)
    w = _c(w, np.int8)
    M, K = q.shape
    N = w.shape[0]
    assert w.shape[1] == K
    acc = np.empty((M, N), np.int32)
    rc = _load().oracle_gemm_s32(_p(q), K, _p(w), K, M, N, K, _p(acc), N)
    if rc:
        raise OverflowError("int32 accumulator overflow")
    return acc


def gemm_s32_splitk(q: np.ndarray, w: np.ndarray, S: int) -> np.ndarray:
    """The same contraction as S contiguous K pieces added as int32."""
    q = _c(q, np.int8)
    w = _c(w, np.int8)
    M, K = q.shape
    N = w.shape[0]
    acc = np.empty((M, N), np.int32)
    rc = _load().oracle_gemm_s32_splitk(_p(q), K, _p(w), K, M, N, K, int(S), _p(acc), N)
    if rc:
        raise OverflowError("int32 accumulator overflow or bad S")
    return acc


def epilogue(acc: np.ndarray, a_scale: np.ndarray, w_scale: np.ndarray,
             residual_bits: np.ndarray | None) -> np.ndarray:
    """Fixed-order dequantise / scale / residual-add, rounded to bf16 bits."""
    acc = _c(acc, np.int32)
    M, N = acc.shape
    a = _c(a_scale, np.float32)
    ws = _c(w_scale, np.float32)
    r = None if residual_bits is None else _c(residual_bits, np.uint16)
    out = np.empty((M, N), np.uint16)
    _load().oracle_epilogue(_p(acc), N, _p(a), _p(ws), _p(r), N, M, N, _p(out), N)
    return out


def w8a8_linear(q, a_scale, w, w_scale, residual_bits=None):
    """Whole linear call.  Returns (out bf16 bits uint16 [M, N], acc int32)."""
    q = _c(q, np.int8)
    w = _c(w, np.int8)
    M, K = q.shape
    N = w.shape[0]
    a = _c(a_scale, np.float32)
    ws = _c(w_scale, np.float32)
    r = None if residual_bits is None else _c(residual_bits, np.uint16)
    out = np.empty((M, N), np.uint16)
    acc = np.empty((M, N), np.int32)
    rc = _load().oracle_w8a8_linear(_p(q), K, _p(a), _p(w), K, _p(ws), _p(r), N,
                                    M, N, K, _p(out), N, _p(acc))
    if rc:
        raise OverflowError("int32 accumulator overflow")
    return out, acc


def unpack_w4(w4: np.ndarray, K: int) -> np.ndarray:
    """Packed 4-bit codes uint8 [N, K/2] (low nibble = even k) -> int8 [N, K]."""
    w4 = _c(w4, np.uint8)
    N = w4.shape[0]
    assert K % 2 == 0 and w4.shape[1] == K // 2
    w = np.empty((N, K), np.int8)
    _load().oracle_unpack_w4(_p(w4), K // 2, N, K, _p(w), K)
    return w


def w4a8_linear(q, a_scale, w4, w_scale, residual_bits=None):
    """The W8A8 linear on packed 4-bit weights.  Returns (out bf16 bits, acc)."""
    q = _c(q, np.int8)
    w4 = _c(w4, np.uint8)
    M, K = q.shape
    N = w4.shape[0]
    assert w4.shape[1] == K // 2
    a = _c(a_scale, np.float32)
    ws = _c(w_scale, np.float32)
    r = None if residual_bits is None else _c(residual_bits, np.uint16)
    out = np.empty((M, N), np.uint16)
    acc = np.empty((M, N), np.int32)
    scratch = np.empty((N, K), np.int8)
    rc = _load().oracle_w4a8_linear(_p(q), K, _p(a), _p(w4), K // 2, _p(ws), _p(r), N, M, N, K,
                                    _p(out), N, _p(acc), _p(scratch))
    if rc:
        raise OverflowError("int32 accumulator overflow")
    return out, acc


ERR_ROW_RANGE = 16   # a row index outside the indexed matrix


def quant_act_rows(x_bf16_bits: np.ndarray, rows, inv_s: np.ndarray | None):
    """Quantisation of the rows ``rows`` of ``x_bf16_bits`` [M_x, K] (the last
    layer restricted to answer positions).  Returns (q int8 [n, K], a_scale
    float32 [n], error bits)."""
    x = _c(x_bf16_bits, np.uint16)
    M_x, K = x.shape
    r = _c(np.asarray(rows, dtype=np.int32), np.int32)
    n = r.size
    s = None if inv_s is None else _c(inv_s, np.float32)
    q = np.empty((n, K), np.int8)
    a = np.empty((n,), np.float32)
    err = _load().oracle_quant_act_rows(_p(x), K, M_x, _p(r), n, _p(s), K, _p(q), K, _p(a))
    return q, a, int(err)


def w8a8_linear_rows(q, a_scale, w, w_scale, residual_bits, res_rows):
    """The linear whose residual row m is ``residual_bits[res_rows[m]]``.
    Returns (out bf16 bits uint16 [M, N], acc int32, error bits)."""
    q = _c(q, np.int8)
    w = _c(w, np.int8)
    M, K = q.shape
    N = w.shape[0]
    a = _c(a_scale, np.float32)
    ws = _c(w_scale, np.float32)
    r = _c(residual_bits, np.uint16)
    M_res = r.shape[0]
    rr = _c(np.asarray(res_rows, dtype=np.int32), np.int32)
    assert rr.size == M
    out = np.empty((M, N), np.uint16)
    acc = np.empty((M, N), np.int32)
    err = ctypes.c_uint32(0)
    rc = _load().oracle_w8a8_linear_rows(_p(q), K, _p(a), _p(w), K, _p(ws), _p(r), N, M_res, _p(rr),
                                         M, N, K, _p(out), N, _p(acc), ctypes.byref(err))
    if rc:
        raise OverflowError("int32 accumulator overflow")
    return out, acc, int(err.value)


def exp(x) -> np.ndarray:
    """The read-out's exponential, elementwise on float32 (domain x <= 0)."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    y = np.empty_like(x)
    _load().oracle_exp_batch(_p(x), x.size, _p(y))
    return y


def candidate_readout(h_bits, inv_s, lm_head, lm_scale, cand_offsets, cand_ids):
    """Candidate-restricted read-out.  ``h_bits`` uint16 [P, K]; ``lm_head``
    int8 [V, K]; ``lm_scale`` float32 [V]; CSR int32 offsets [P+1], ids [T].
    Returns (status, logits float32 [T], probs float32 [T])."""
    h = _c(h_bits, np.uint16)
    P, K = h.shape
    W = _c(lm_head, np.int8)
    V = W.shape[0]
    assert W.shape[1] == K
    s = None if inv_s is None else _c(inv_s, np.float32)
    ls = _c(lm_scale, np.float32)
    off = _c(cand_offsets, np.int32)
    ids = _c(cand_ids, np.int32)
    T = ids.size
    assert off.size == P + 1
    logits = np.empty((T,), np.float32)
    probs = np.empty((T,), np.float32)
    rc = _load().oracle_candidate_readout(_p(h), K, _p(s), _p(W), K, _p(ls), V, K,
                                          _p(off), _p(ids), P, T, _p(logits), _p(probs))
    return int(rc), logits, probs


def candidate_logits_shard(h_bits, inv_s, lm_shard, lm_scale_shard, v0, V, cand_offsets, cand_ids):
    """Logits of the candidates held by rows v0 .. v0 + V_shard - 1 of a
    V-row head (``lm_shard`` int8 [V_shard, K]); -0.0 for the others.
    Returns (status, logits float32 [T])."""
    h = _c(h_bits, np.uint16)
    P, K = h.shape
    W = _c(lm_shard, np.int8).reshape(-1, K)
    Vs = W.shape[0]
    s = None if inv_s is None else _c(inv_s, np.float32)
    ls = _c(lm_scale_shard, np.float32)
    off = _c(cand_offsets, np.int32)
    ids = _c(cand_ids, np.int32)
    T = ids.size
    logits = np.empty((T,), np.float32)
    rc = _load().oracle_candidate_logits_shard(_p(h), K, _p(s), _p(W), K, _p(ls), int(v0), Vs, int(V), K,
                                               _p(off), _p(ids), P, T, _p(logits))
    return int(rc), logits


def candidate_softmax(logits, cand_offsets):
    """The read-out's candidate softmax on given logits.  Returns (status,
    probs float32 [T])."""
    lg = _c(logits, np.float32)
    off = _c(cand_offsets, np.int32)
    P, T = off.size - 1, lg.size
    probs = np.empty((T,), np.float32)
    rc = _load().oracle_candidate_softmax(_p(lg), _p(off), P, T, _p(probs))
    return int(rc), probs


def bf16_bits_to_float(h) -> np.ndarray:
    h = _c(h, np.uint16)
    f = np.empty(h.shape, np.float32)
    _load().oracle_bf16_to_float(_p(h), h.size, _p(f))
    return f


def float_to_bf16_bits(f) -> np.ndarray:
    f = _c(f, np.float32)
    h = np.empty(f.shape, np.uint16)
    _load().oracle_float_to_bf16(_p(f), f.size, _p(h))
    return h
