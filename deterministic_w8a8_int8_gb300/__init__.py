"""Batch-invariant W8A8 int8 linear layer and candidate read-out for GB300.

Thin Python binding over the C ABI of ``libprism.so`` (see ``include/prism.h``):
argument marshalling only.  Every step of the computation runs in the
library's CUDA kernels; there is no CPU or PyTorch fallback, and the import
of any compute entry point fails loudly when the library has not been built
(``deterministic_w8a8_int8_gb300.build.build()``).

PyTorch is used for device memory and the current CUDA stream only.

Entry points (same names as the C ABI):
  prism_quant_act(x, inv_s)                      -> (q, a_scale)
  prism_w8a8_linear(q, a_scale, w, w_scale, ...) -> out
  prism_smooth_requant(q, d, smooth)             -> (w, w_scale)
  prism_quant_act_rows(x, rows, inv_s)           -> (q, a_scale)   answer rows only
  prism_w8a8_linear_rows(q, a_scale, w, w_scale, residual, residual_rows) -> out
  prism_act_amax, prism_quant_act_amax, prism_w8a8_gemm_s32, prism_w8a8_epilogue
                                                 the tensor-parallel building blocks
  tp_row_parallel_linear(x_shard, ...)           those blocks around torch.distributed
  prism_w4a8_linear(q, a_scale, w4, w_scale, ...) -> out   packed 4-bit weights
  prism_unpack_w4(w4, K)                         -> int8 codes
  prism_candidate_readout(hidden, ...)           -> (logits, probs)
  prism_candidate_logits(hidden, ..., shard)     -> logits of one vocabulary shard
  prism_candidate_softmax(logits, cand_offsets)  -> probs
  readout_column_parallel(hidden, ..., shard)    those two around torch.distributed
  prism_quant_act_f16(x, inv_s)                  -> (codes as float16, a_scale)
  prism_codes_to_f16(w)                          -> int8 codes as float16 (load time)
  prism_w8a8_linear_f16(qh, a_scale, wh, w_scale, ...) -> out   codes given as float16
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "libprism.so")

PRISM_OK = 0
PRISM_ERR_INVALID_ARG = -1
PRISM_ERR_ALIGNMENT = -2
PRISM_ERR_UNSUPPORTED = -3
PRISM_ERR_WORKSPACE = -4
PRISM_ERR_CUDA = -5
PRISM_MAX_K = 133144
PRISM_MAX_SPLIT_K = 64
PRISM_MAX_CANDIDATES = 64
PRISM_MAX_READOUT_K = 65536
PRISM_NOALLOC_SCRATCH_BYTES = 8388608
PRISM_DEV_ERR_OFFSETS = 1
PRISM_DEV_ERR_COUNT = 2
PRISM_DEV_ERR_ID_RANGE = 4
PRISM_DEV_ERR_DUPLICATE = 8
PRISM_DEV_ERR_ROW_RANGE = 16
PRISM_DEVSTATUS_WAIT_TIMEOUT = 1

# (restype, argtypes) of every symbol the header declares
_P, _I64, _I32, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
SIGNATURES = {
    "prism_quant_act": (_I32, [_P, _I64, _P, _I64, _I64, _P, _I64, _P, _P]),
    "prism_w8a8_workspace_bytes": (_SZ, [_I64, _I64, _I64, _I32]),
    "prism_w8a8_linear": (_I32, [_P, _I64, _P, _P, _I64, _P, _P, _I64, _P, _I64, _P,
                                 _I64, _I64, _I64, _I32, _P, _SZ, _P]),
    "prism_w8a8_linear_noalloc": (_I32, [_P, _I64, _P, _P, _I64, _P, _P, _I64, _P, _I64, _P,
                                         _I64, _I64, _I64, _I32, _P]),
    "prism_candidate_readout": (_I32, [_P, _I64, _P, _P, _I64, _P, _I64, _I64, _P, _P,
                                       _I64, _I64, _P, _P, _P, _P, _SZ, _P]),
    "prism_readout_workspace_bytes": (_SZ, [_I64, _I64, _I64]),
    "prism_candidate_logits": (_I32, [_P, _I64, _P, _P, _I64, _P, _I64, _I64, _I64, _I64, _P, _P,
                                      _I64, _I64, _P, _P, _P]),
    "prism_candidate_softmax": (_I32, [_P, _P, _I64, _I64, _P, _P, _P]),
    "prism_quant_act_f16": (_I32, [_P, _I64, _P, _I64, _I64, _P, _I64, _P, _P]),
    "prism_codes_to_f16": (_I32, [_P, _I64, _I64, _I64, _P, _I64, _P]),
    "prism_w8a8_f16_workspace_bytes": (_SZ, [_I64, _I64, _I64, _I32]),
    "prism_w8a8_linear_f16": (_I32, [_P, _I64, _P, _P, _I64, _P, _P, _I64, _P, _I64, _P,
                                     _I64, _I64, _I64, _I32, _P, _SZ, _P]),
    "prism_debug_wait_expiry": (_I32, [ctypes.c_uint64]),
    "prism_smooth_requant": (_I32, [_P, _I64, _P, _I64, _P, _I64, _I64, _P, _I64, _P, _P]),
    "prism_quant_act_rows": (_I32, [_P, _I64, _I64, _P, _I64, _P, _I64, _P, _I64, _P, _P, _P]),
    "prism_w8a8_linear_rows": (_I32, [_P, _I64, _P, _P, _I64, _P, _P, _I64, _I64, _P, _P, _I64, _P,
                                      _I64, _I64, _I64, _I32, _P, _SZ, _P, _P]),
    "prism_act_amax": (_I32, [_P, _I64, _P, _I64, _I64, _P, _P]),
    "prism_quant_act_amax": (_I32, [_P, _I64, _P, _P, _I64, _I64, _P, _I64, _P, _P]),
    "prism_w8a8_gemm_s32": (_I32, [_P, _I64, _P, _I64, _P, _I64, _I64, _I64, _I32, _P, _SZ, _P]),
    "prism_w8a8_epilogue": (_I32, [_P, _I64, _P, _P, _P, _I64, _P, _I64, _I64, _I64, _P]),
    "prism_w4a8_workspace_bytes": (_SZ, [_I64, _I64, _I64, _I32]),
    "prism_w4a8_linear": (_I32, [_P, _I64, _P, _P, _I64, _P, _P, _I64, _P, _I64, _P, _I64, _I64, _I64, _I32,
                                 _P, _SZ, _P]),
    "prism_unpack_w4": (_I32, [_P, _I64, _I64, _I64, _P, _I64, _P]),
    "prism_status_string": (ctypes.c_char_p, [_I32]),
    "prism_version": (_I32, []),
    "prism_w8a8_kernel_kind": (_I32, [_I64, _I64, _I64]),
    "prism_w8a8_auto_split": (_I32, [_I64, _I64, _I64]),
    "prism_device_status": (_I32, [_P]),
    "prism_last_cuda_error": (_I32, [ctypes.c_char_p, _SZ]),
}

_lock = threading.Lock()
_lib = None


class PrismError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        detail = ""
        if status == PRISM_ERR_CUDA:
            buf = ctypes.create_string_buffer(256)
            code = lib().prism_last_cuda_error(buf, 256)
            detail = f"; CUDA error {code}: {buf.value.decode(errors='replace')}"
        super().__init__(f"{fn} failed: {status} ({status_string(status)}{detail})")


def lib() -> ctypes.CDLL:
    """The loaded libprism.so.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(
                    f"libprism.so is not built at {LIB_PATH}; run "
                    "deterministic_w8a8_int8_gb300.build.build() (needs nvcc)")
            handle = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
        return _lib


def status_string(status: int) -> str:
    return lib().prism_status_string(int(status)).decode()


def _check(fn: str, status: int) -> None:
    if status != PRISM_OK:
        raise PrismError(fn, status)


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _require(t, dtype, name, ndim, on_device=True):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if on_device and not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims")
    if ndim == 2 and t.stride(1) != 1:
        raise ValueError(f"{name} rows must be contiguous")
    if ndim == 1 and t.numel() > 1 and t.stride(0) != 1:
        raise ValueError(f"{name} must be contiguous")


def _linear_operands(q, a_scale, w, w_scale, residual, out, acc_out, on_device=True):
    """Checks the tensors of a linear call before anything is launched: dtypes,
    contiguous rows, and every shape against [M, K] x [N, K] (residual, out
    and acc_out [M, N]; acc_out dense).  Returns (M, N, K)."""
    import torch
    _require(q, torch.int8, "q", 2, on_device)
    _require(w, torch.int8, "w", 2, on_device)
    _require(a_scale, torch.float32, "a_scale", 1, on_device)
    _require(w_scale, torch.float32, "w_scale", 1, on_device)
    M, K = q.shape
    N = w.shape[0]
    if w.shape[1] != K or a_scale.numel() != M or w_scale.numel() != N:
        raise ValueError("shape mismatch")
    if residual is not None:
        _require(residual, torch.bfloat16, "residual", 2, on_device)
        if tuple(residual.shape) != (M, N):
            raise ValueError("residual must be [M, N]")
    if out is not None:
        _require(out, torch.bfloat16, "out", 2, on_device)
        if tuple(out.shape) != (M, N):
            raise ValueError("out must be [M, N]")
    if acc_out is not None:
        _require(acc_out, torch.int32, "acc_out", 2, on_device)
        if not acc_out.is_contiguous() or tuple(acc_out.shape) != (M, N):
            raise ValueError("acc_out must be a contiguous [M, N] int32 tensor")
    return M, N, K


def prism_w8a8_workspace_bytes(M: int, N: int, K: int, split_k: int = 0) -> int:
    return int(lib().prism_w8a8_workspace_bytes(M, N, K, split_k))


def prism_w8a8_kernel_kind(M: int, N: int, K: int) -> int:
    return int(lib().prism_w8a8_kernel_kind(M, N, K))


def prism_w8a8_auto_split(M: int, N: int, K: int) -> int:
    return int(lib().prism_w8a8_auto_split(M, N, K))


def prism_device_status() -> int:
    """Device error bits raised since the last query (0 = none); synchronous."""
    v = ctypes.c_uint32(0)
    _check("prism_device_status", lib().prism_device_status(ctypes.byref(v)))
    return int(v.value)


def prism_version() -> int:
    return int(lib().prism_version())


def prism_quant_act(x, inv_s=None, q=None, a_scale=None, stream=None):
    """Per-token quantisation of bf16 ``x`` [M, K] -> (int8 q [M, K], float32 a_scale [M])."""
    import torch
    _require(x, torch.bfloat16, "x", 2)
    M, K = x.shape
    if inv_s is not None:
        _require(inv_s, torch.float32, "inv_s", 1)
    if q is None:
        q = torch.empty((M, K), dtype=torch.int8, device=x.device)
    if a_scale is None:
        a_scale = torch.empty((M,), dtype=torch.float32, device=x.device)
    _require(q, torch.int8, "q", 2)
    _require(a_scale, torch.float32, "a_scale", 1)
    st = lib().prism_quant_act(_ptr(x), x.stride(0), _ptr(inv_s), M, K, _ptr(q), q.stride(0),
                               _ptr(a_scale), _stream(stream))
    _check("prism_quant_act", st)
    return q, a_scale


def prism_smooth_requant(q, d, smooth=None, w=None, w_scale=None, stream=None):
    """Requantise Q8_0 weights with SmoothQuant factors folded in.

    ``q`` int8 [N, K] codes, ``d`` [N, K/32] block scales (float16, or int16
    holding binary16 bits), ``smooth`` float32 [K] or None.  Returns
    (int8 w [N, K], float32 w_scale [N]); ``w`` may be ``q`` (in place)."""
    import torch
    _require(q, torch.int8, "q", 2)
    N, K = q.shape
    if d.dtype not in (torch.float16, torch.int16):
        raise TypeError(f"d must be float16 or int16 (binary16 bits), got {d.dtype}")
    if not d.is_cuda or d.dim() != 2 or (d.shape[1] > 1 and d.stride(1) != 1):
        raise ValueError("d must be a 2-D CUDA tensor with contiguous rows")
    if smooth is not None:
        _require(smooth, torch.float32, "smooth", 1)
    if w is None:
        w = torch.empty((N, K), dtype=torch.int8, device=q.device)
    if w_scale is None:
        w_scale = torch.empty((N,), dtype=torch.float32, device=q.device)
    _require(w, torch.int8, "w", 2)
    _require(w_scale, torch.float32, "w_scale", 1)
    st = lib().prism_smooth_requant(_ptr(q), q.stride(0), _ptr(d), d.stride(0), _ptr(smooth), N, K,
                                    _ptr(w), w.stride(0), _ptr(w_scale), _stream(stream))
    _check("prism_smooth_requant", st)
    return w, w_scale


def new_workspace(M: int, N: int, K: int, split_k: int = 0, device=None):
    """A zeroed workspace for prism_w8a8_linear (None when none is needed)."""
    import torch
    n = prism_w8a8_workspace_bytes(M, N, K, split_k)
    if n == 0:
        return None
    return torch.zeros((n,), dtype=torch.uint8, device=device)


def prism_w8a8_linear(q, a_scale, w, w_scale, residual=None, out=None, acc_out=None,
                      split_k: int = 0, workspace=None, stream=None):
    """out[M, N] (bf16) = epilogue(q @ w^T) with exact int32 accumulation.

    ``residual`` may be ``out`` itself (in-place residual add).  ``workspace``
    must be a zeroed uint8 tensor of at least prism_w8a8_workspace_bytes bytes
    when the schedule needs one (split-K > 1, or an automatic call that shares
    tiles between CTAs); one is allocated (and zeroed) per call when None."""
    import torch
    M, N, K = _linear_operands(q, a_scale, w, w_scale, residual, out, acc_out)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=q.device)
    if workspace is None:
        workspace = new_workspace(M, N, K, split_k, q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().prism_w8a8_linear(
        _ptr(q), q.stride(0), _ptr(a_scale), _ptr(w), w.stride(0), _ptr(w_scale),
        _ptr(residual), 0 if residual is None else residual.stride(0), _ptr(out), out.stride(0),
        _ptr(acc_out), M, N, K, int(split_k), _ptr(workspace), ws_bytes, _stream(stream))
    _check("prism_w8a8_linear", st)
    return out


def prism_quant_act_rows(x, rows, inv_s=None, q=None, a_scale=None, err=None, stream=None):
    """Quantisation of the rows ``rows`` (int32 [n]) of bf16 ``x`` [M_x, K]
    -> (int8 q [n, K], float32 a_scale [n]).  ``err``: optional int32 [1]
    device word that collects PRISM_DEV_ERR_ROW_RANGE."""
    import torch
    _require(x, torch.bfloat16, "x", 2)
    _require(rows, torch.int32, "rows", 1)
    M_x, K = x.shape
    n = rows.numel()
    if inv_s is not None:
        _require(inv_s, torch.float32, "inv_s", 1)
    if q is None:
        q = torch.empty((n, K), dtype=torch.int8, device=x.device)
    if a_scale is None:
        a_scale = torch.empty((n,), dtype=torch.float32, device=x.device)
    _require(q, torch.int8, "q", 2)
    _require(a_scale, torch.float32, "a_scale", 1)
    if err is not None:
        _require(err, torch.int32, "err", 1)
    st = lib().prism_quant_act_rows(_ptr(x), x.stride(0), M_x, _ptr(rows), n, _ptr(inv_s), K, _ptr(q),
                                    q.stride(0), _ptr(a_scale), _ptr(err), _stream(stream))
    _check("prism_quant_act_rows", st)
    return q, a_scale


def prism_w8a8_linear_rows(q, a_scale, w, w_scale, residual, residual_rows, out=None, acc_out=None,
                           split_k: int = 0, workspace=None, err=None, stream=None):
    """prism_w8a8_linear whose residual row for output row m is
    ``residual[residual_rows[m]]`` (``residual`` [M_res, N] bf16, the full
    hidden state; ``residual_rows`` int32 [M]).  ``out`` must not overlap
    ``residual``.  ``err``: optional int32 [1] device error word."""
    import torch
    _require(q, torch.int8, "q", 2)
    _require(w, torch.int8, "w", 2)
    _require(a_scale, torch.float32, "a_scale", 1)
    _require(w_scale, torch.float32, "w_scale", 1)
    _require(residual, torch.bfloat16, "residual", 2)
    _require(residual_rows, torch.int32, "residual_rows", 1)
    M, K = q.shape
    N = w.shape[0]
    if w.shape[1] != K or a_scale.numel() != M or w_scale.numel() != N or residual_rows.numel() != M:
        raise ValueError("shape mismatch")
    if residual.shape[1] != N:
        raise ValueError("residual shape")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=q.device)
    _require(out, torch.bfloat16, "out", 2)
    if acc_out is not None:
        _require(acc_out, torch.int32, "acc_out", 2)
        if not acc_out.is_contiguous() or tuple(acc_out.shape) != (M, N):
            raise ValueError("acc_out must be a contiguous [M, N] int32 tensor")
    if err is not None:
        _require(err, torch.int32, "err", 1)
    if workspace is None:
        workspace = new_workspace(M, N, K, split_k, q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().prism_w8a8_linear_rows(
        _ptr(q), q.stride(0), _ptr(a_scale), _ptr(w), w.stride(0), _ptr(w_scale),
        _ptr(residual), residual.stride(0), residual.shape[0], _ptr(residual_rows), _ptr(out), out.stride(0),
        _ptr(acc_out), M, N, K, int(split_k), _ptr(workspace), ws_bytes, _ptr(err), _stream(stream))
    _check("prism_w8a8_linear_rows", st)
    return out


def prism_w4a8_workspace_bytes(M: int, N: int, K: int, split_k: int = 0) -> int:
    return int(lib().prism_w4a8_workspace_bytes(M, N, K, split_k))


def prism_w4a8_linear(q, a_scale, w4, w_scale, residual=None, out=None, acc_out=None, split_k: int = 0,
                      workspace=None, stream=None):
    """The W8A8 linear on packed 4-bit weights ``w4`` uint8 [N, K/2] (code
    2j in the low nibble of byte j).  ``workspace``: a zeroed uint8 tensor of
    prism_w4a8_workspace_bytes bytes (allocated and zeroed when None)."""
    import torch
    _require(q, torch.int8, "q", 2)
    _require(w4, torch.uint8, "w4", 2)
    _require(a_scale, torch.float32, "a_scale", 1)
    _require(w_scale, torch.float32, "w_scale", 1)
    M, K = q.shape
    N = w4.shape[0]
    if 2 * w4.shape[1] != K or a_scale.numel() != M or w_scale.numel() != N:
        raise ValueError("shape mismatch")
    if residual is not None:
        _require(residual, torch.bfloat16, "residual", 2)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=q.device)
    _require(out, torch.bfloat16, "out", 2)
    if acc_out is not None and (acc_out.dtype != torch.int32 or not acc_out.is_contiguous()
                                or tuple(acc_out.shape) != (M, N)):
        raise ValueError("acc_out must be a contiguous [M, N] int32 tensor")
    if workspace is None:
        need = prism_w4a8_workspace_bytes(M, N, K, split_k)
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device) if need else None
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("prism_w4a8_linear", lib().prism_w4a8_linear(
        _ptr(q), q.stride(0), _ptr(a_scale), _ptr(w4), w4.stride(0), _ptr(w_scale), _ptr(residual),
        0 if residual is None else residual.stride(0), _ptr(out), out.stride(0), _ptr(acc_out), M, N, K,
        int(split_k), _ptr(workspace), ws_bytes, _stream(stream)))
    return out


def prism_unpack_w4(w4, K: int, w=None, stream=None):
    """Packed 4-bit codes uint8 [N, K/2] -> int8 [N, K]."""
    import torch
    _require(w4, torch.uint8, "w4", 2)
    N = w4.shape[0]
    if w is None:
        w = torch.empty((N, K), dtype=torch.int8, device=w4.device)
    _require(w, torch.int8, "w", 2)
    _check("prism_unpack_w4", lib().prism_unpack_w4(_ptr(w4), w4.stride(0), N, K, _ptr(w), w.stride(0),
                                                    _stream(stream)))
    return w


def prism_act_amax(x, inv_s=None, amax=None, stream=None):
    """Row maxima max_k |x * inv_s| of bf16 ``x`` [M, K] -> float32 [M]."""
    import torch
    _require(x, torch.bfloat16, "x", 2)
    M, K = x.shape
    if inv_s is not None:
        _require(inv_s, torch.float32, "inv_s", 1)
    if amax is None:
        amax = torch.empty((M,), dtype=torch.float32, device=x.device)
    _require(amax, torch.float32, "amax", 1)
    _check("prism_act_amax", lib().prism_act_amax(_ptr(x), x.stride(0), _ptr(inv_s), M, K, _ptr(amax),
                                                  _stream(stream)))
    return amax


def prism_quant_act_amax(x, inv_s, amax, q=None, a_scale=None, stream=None):
    """prism_quant_act with given row maxima ``amax`` [M] -> (q, a_scale)."""
    import torch
    _require(x, torch.bfloat16, "x", 2)
    _require(amax, torch.float32, "amax", 1)
    M, K = x.shape
    if inv_s is not None:
        _require(inv_s, torch.float32, "inv_s", 1)
    if q is None:
        q = torch.empty((M, K), dtype=torch.int8, device=x.device)
    if a_scale is None:
        a_scale = torch.empty((M,), dtype=torch.float32, device=x.device)
    _require(q, torch.int8, "q", 2)
    _require(a_scale, torch.float32, "a_scale", 1)
    _check("prism_quant_act_amax", lib().prism_quant_act_amax(
        _ptr(x), x.stride(0), _ptr(inv_s), _ptr(amax), M, K, _ptr(q), q.stride(0), _ptr(a_scale), _stream(stream)))
    return q, a_scale


def prism_w8a8_gemm_s32(q, w, acc=None, split_k: int = 0, workspace=None, stream=None):
    """Exact int32 ``q @ w^T`` -> dense int32 [M, N] (no scaling)."""
    import torch
    _require(q, torch.int8, "q", 2)
    _require(w, torch.int8, "w", 2)
    M, K = q.shape
    N = w.shape[0]
    if w.shape[1] != K:
        raise ValueError("shape mismatch")
    if acc is None:
        acc = torch.empty((M, N), dtype=torch.int32, device=q.device)
    if acc.dtype != torch.int32 or not acc.is_contiguous() or tuple(acc.shape) != (M, N):
        raise ValueError("acc must be a contiguous [M, N] int32 tensor")
    if workspace is None:
        workspace = new_workspace(M, N, K, split_k, q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("prism_w8a8_gemm_s32", lib().prism_w8a8_gemm_s32(
        _ptr(q), q.stride(0), _ptr(w), w.stride(0), _ptr(acc), M, N, K, int(split_k), _ptr(workspace), ws_bytes,
        _stream(stream)))
    return acc


def prism_w8a8_epilogue(acc, a_scale, w_scale, residual=None, out=None, stream=None):
    """bf16 out[M, N] from int32 ``acc`` [M, N] with the linear's epilogue."""
    import torch
    _require(acc, torch.int32, "acc", 2)
    _require(a_scale, torch.float32, "a_scale", 1)
    _require(w_scale, torch.float32, "w_scale", 1)
    M, N = acc.shape
    if a_scale.numel() != M or w_scale.numel() != N:
        raise ValueError("shape mismatch")
    if residual is not None:
        _require(residual, torch.bfloat16, "residual", 2)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=acc.device)
    _require(out, torch.bfloat16, "out", 2)
    _check("prism_w8a8_epilogue", lib().prism_w8a8_epilogue(
        _ptr(acc), acc.stride(0), _ptr(a_scale), _ptr(w_scale), _ptr(residual),
        0 if residual is None else residual.stride(0), _ptr(out), out.stride(0), M, N, _stream(stream)))
    return out


class KernelOps:
    """The per-rank steps of tp_row_parallel_linear on this library's kernels."""
    act_amax = staticmethod(lambda x, inv_s: prism_act_amax(x, inv_s))
    quant_act_amax = staticmethod(lambda x, inv_s, amax: prism_quant_act_amax(x, inv_s, amax))
    gemm_s32 = staticmethod(lambda q, w: prism_w8a8_gemm_s32(q, w))
    epilogue = staticmethod(lambda acc, a_scale, w_scale, residual: prism_w8a8_epilogue(acc, a_scale, w_scale,
                                                                                       residual))


def tp_row_parallel_linear(x, inv_s, w, w_scale, residual=None, group=None, ops=KernelOps):
    """One rank of a row-parallel tensor-parallel W8A8 linear.

    ``x`` [M, K_r] bf16 and ``inv_s`` [K_r] are this rank's columns of the
    activations, ``w`` [N, K_r] int8 its columns of the weight; ``w_scale``
    [N] and ``residual`` [M, N] are replicated.  The ranks agree on each
    token's scale (MAX all-reduce of the shard maxima), contract their shards
    exactly in int32, add the partial sums (SUM all-reduce) and scale once, so
    every rank returns the one-device output bit for bit.  ``group`` is a
    torch.distributed process group (None: the default group); ``ops`` holds
    the per-rank steps (act_amax, quant_act_amax, gemm_s32, epilogue)."""
    import torch.distributed as dist
    amax = ops.act_amax(x, inv_s)
    dist.all_reduce(amax, op=dist.ReduceOp.MAX, group=group)
    q, a_scale = ops.quant_act_amax(x, inv_s, amax)
    acc = ops.gemm_s32(q, w)
    dist.all_reduce(acc, op=dist.ReduceOp.SUM, group=group)
    return ops.epilogue(acc, a_scale, w_scale, residual)


def prism_w8a8_linear_noalloc(q, a_scale, w, w_scale, residual=None, out=None, acc_out=None,
                              split_k: int = 0, stream=None):
    """prism_w8a8_linear for callers that cannot supply scratch memory: split-K
    scratch comes from a fixed array inside the library (see include/prism.h
    for its size limit and the rule that overlapping calls must not share it)."""
    import torch
    M, N, K = _linear_operands(q, a_scale, w, w_scale, residual, out, acc_out)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=q.device)
    st = lib().prism_w8a8_linear_noalloc(
        _ptr(q), q.stride(0), _ptr(a_scale), _ptr(w), w.stride(0), _ptr(w_scale),
        _ptr(residual), 0 if residual is None else residual.stride(0), _ptr(out), out.stride(0),
        _ptr(acc_out), M, N, K, int(split_k), _stream(stream))
    _check("prism_w8a8_linear_noalloc", st)
    return out


def prism_readout_workspace_bytes(P: int, T: int, K: int) -> int:
    return int(lib().prism_readout_workspace_bytes(P, T, K))


def prism_candidate_readout(hidden, inv_s, lm_head, lm_scale, cand_offsets, cand_ids,
                            logits=None, probs=None, err=None, workspace=None, stream=None):
    """Candidate-restricted read-out -> (logits float32 [T], probs float32 [T]).
    ``err``: optional int32 [1] device error word; ``workspace``: optional
    uint8 device tensor of prism_readout_workspace_bytes bytes (allocated
    when None and that size is nonzero)."""
    import torch
    _require(hidden, torch.bfloat16, "hidden", 2)
    _require(lm_head, torch.int8, "lm_head", 2)
    _require(lm_scale, torch.float32, "lm_scale", 1)
    _require(cand_offsets, torch.int32, "cand_offsets", 1)
    _require(cand_ids, torch.int32, "cand_ids", 1)
    if inv_s is not None:
        _require(inv_s, torch.float32, "inv_s", 1)
    P, K = hidden.shape
    V = lm_head.shape[0]
    T = cand_ids.numel()
    if lm_head.shape[1] != K or cand_offsets.numel() != P + 1:
        raise ValueError("shape mismatch")
    if logits is None:
        logits = torch.empty((T,), dtype=torch.float32, device=hidden.device)
    if probs is None:
        probs = torch.empty((T,), dtype=torch.float32, device=hidden.device)
    _require(logits, torch.float32, "logits", 1)
    _require(probs, torch.float32, "probs", 1)
    if logits.numel() != T or probs.numel() != T:
        raise ValueError("logits and probs must hold T values")
    if err is not None:
        _require(err, torch.int32, "err", 1)
    if workspace is None:
        need = prism_readout_workspace_bytes(P, T, K)
        workspace = torch.zeros(need, dtype=torch.uint8, device=hidden.device) if need else None
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().prism_candidate_readout(
        _ptr(hidden), hidden.stride(0), _ptr(inv_s), _ptr(lm_head), lm_head.stride(0),
        _ptr(lm_scale), V, K, _ptr(cand_offsets), _ptr(cand_ids), P, T, _ptr(logits),
        _ptr(probs), _ptr(err), _ptr(workspace), ws_bytes, _stream(stream))
    _check("prism_candidate_readout", st)
    return logits, probs


def prism_candidate_logits(hidden, inv_s, lm_shard, lm_scale_shard, v0: int, V: int, cand_offsets, cand_ids,
                           logits=None, err=None, stream=None):
    """Logits float32 [T] of the candidates held by one vocabulary shard
    (``lm_shard`` [V_shard, K] int8 = rows v0 .. v0 + V_shard - 1 of a V-row
    head, ``lm_scale_shard`` [V_shard]); -0.0 for the other candidates, so
    that the SUM over the shards is the one-device read-out's logits."""
    import torch
    _require(hidden, torch.bfloat16, "hidden", 2)
    _require(lm_shard, torch.int8, "lm_shard", 2)
    _require(lm_scale_shard, torch.float32, "lm_scale_shard", 1)
    _require(cand_offsets, torch.int32, "cand_offsets", 1)
    _require(cand_ids, torch.int32, "cand_ids", 1)
    if inv_s is not None:
        _require(inv_s, torch.float32, "inv_s", 1)
    P, K = hidden.shape
    Vs = lm_shard.shape[0]
    T = cand_ids.numel()
    if lm_shard.shape[1] != K or lm_scale_shard.numel() != Vs or cand_offsets.numel() != P + 1:
        raise ValueError("shape mismatch")
    if logits is None:
        logits = torch.empty((T,), dtype=torch.float32, device=hidden.device)
    _require(logits, torch.float32, "logits", 1)
    if logits.numel() != T:
        raise ValueError("logits must hold T values")
    if err is not None:
        _require(err, torch.int32, "err", 1)
    st = lib().prism_candidate_logits(
        _ptr(hidden), hidden.stride(0), _ptr(inv_s), _ptr(lm_shard), lm_shard.stride(0), _ptr(lm_scale_shard),
        int(v0), Vs, int(V), K, _ptr(cand_offsets), _ptr(cand_ids), P, T, _ptr(logits), _ptr(err),
        _stream(stream))
    _check("prism_candidate_logits", st)
    return logits


def prism_candidate_softmax(logits, cand_offsets, probs=None, err=None, stream=None):
    """The read-out's candidate softmax on given logits -> probs float32 [T]."""
    import torch
    _require(logits, torch.float32, "logits", 1)
    _require(cand_offsets, torch.int32, "cand_offsets", 1)
    P, T = cand_offsets.numel() - 1, logits.numel()
    if probs is None:
        probs = torch.empty((T,), dtype=torch.float32, device=logits.device)
    _require(probs, torch.float32, "probs", 1)
    if probs.numel() != T:
        raise ValueError("probs must hold T values")
    if err is not None:
        _require(err, torch.int32, "err", 1)
    st = lib().prism_candidate_softmax(_ptr(logits), _ptr(cand_offsets), P, T, _ptr(probs), _ptr(err),
                                       _stream(stream))
    _check("prism_candidate_softmax", st)
    return probs


class ReadoutKernelOps:
    """The per-rank steps of readout_column_parallel on this library's kernels."""
    candidate_logits = staticmethod(lambda hidden, inv_s, lm_shard, lm_scale_shard, v0, V, off, ids, err:
                                    prism_candidate_logits(hidden, inv_s, lm_shard, lm_scale_shard, v0, V, off,
                                                           ids, err=err))
    candidate_softmax = staticmethod(lambda logits, off, err: prism_candidate_softmax(logits, off, err=err))


def readout_column_parallel(hidden, inv_s, lm_shard, lm_scale_shard, v0: int, V: int, cand_offsets, cand_ids,
                            err=None, group=None, ops=ReadoutKernelOps):
    """One rank of the column-parallel candidate read-out: this rank holds
    rows v0 .. v0 + V_shard - 1 of the V-row LM head; ``hidden`` and the
    candidate lists are replicated.  Each rank forms its candidates' logits
    (-0.0 for the others), the ranks add them (SUM all-reduce: one rank owns
    each candidate and x + -0.0 == x, so the sum is exact in any order), and
    every rank applies the candidate softmax -- returning the one-device
    read-out's (logits, probs) bit for bit.  ``ops`` holds the per-rank
    steps (candidate_logits, candidate_softmax)."""
    import torch.distributed as dist
    logits = ops.candidate_logits(hidden, inv_s, lm_shard, lm_scale_shard, v0, V, cand_offsets, cand_ids, err)
    dist.all_reduce(logits, op=dist.ReduceOp.SUM, group=group)
    return logits, ops.candidate_softmax(logits, cand_offsets, err)


def prism_debug_wait_expiry(limit_ns: int) -> None:
    """Arm (limit_ns > 0) or disarm (0) the test mode of the tensor-core
    kernels' bounded waits: each CTA withholds one completion signal and the
    wait for it expires after limit_ns (see include/prism.h)."""
    _check("prism_debug_wait_expiry", lib().prism_debug_wait_expiry(int(limit_ns)))


def prism_quant_act_f16(x, inv_s=None, qh=None, a_scale=None, stream=None):
    """prism_quant_act with the codes stored as float16 values (exact integers
    in [-127, 127]): bf16 ``x`` [M, K] -> (float16 qh [M, K], float32 a_scale [M])."""
    import torch
    _require(x, torch.bfloat16, "x", 2)
    M, K = x.shape
    if inv_s is not None:
        _require(inv_s, torch.float32, "inv_s", 1)
    if qh is None:
        qh = torch.empty((M, K), dtype=torch.float16, device=x.device)
    if a_scale is None:
        a_scale = torch.empty((M,), dtype=torch.float32, device=x.device)
    _require(qh, torch.float16, "qh", 2)
    _require(a_scale, torch.float32, "a_scale", 1)
    if tuple(qh.shape) != (M, K) or a_scale.numel() != M:
        raise ValueError("qh must be [M, K] and a_scale [M]")
    st = lib().prism_quant_act_f16(_ptr(x), x.stride(0), _ptr(inv_s), M, K, _ptr(qh), qh.stride(0),
                                   _ptr(a_scale), _stream(stream))
    _check("prism_quant_act_f16", st)
    return qh, a_scale


def prism_codes_to_f16(w, wh=None, stream=None):
    """int8 codes [N, K] -> the same codes as float16 [N, K] (exact; the weight
    operand of prism_w8a8_linear_f16, made once at load time)."""
    import torch
    _require(w, torch.int8, "w", 2)
    N, K = w.shape
    if wh is None:
        wh = torch.empty((N, K), dtype=torch.float16, device=w.device)
    _require(wh, torch.float16, "wh", 2)
    if tuple(wh.shape) != (N, K):
        raise ValueError("wh must be [N, K]")
    _check("prism_codes_to_f16", lib().prism_codes_to_f16(_ptr(w), w.stride(0), N, K, _ptr(wh), wh.stride(0),
                                                          _stream(stream)))
    return wh


def prism_w8a8_f16_workspace_bytes(M: int, N: int, K: int, split_k: int = 0) -> int:
    return int(lib().prism_w8a8_f16_workspace_bytes(M, N, K, split_k))


def new_workspace_f16(M: int, N: int, K: int, split_k: int = 0, device=None):
    """A zeroed workspace for prism_w8a8_linear_f16 (None when none is needed)."""
    import torch
    n = prism_w8a8_f16_workspace_bytes(M, N, K, split_k)
    if n == 0:
        return None
    return torch.zeros((n,), dtype=torch.uint8, device=device)


def prism_w8a8_linear_f16(qh, a_scale, wh, w_scale, residual=None, out=None, acc_out=None,
                          split_k: int = 0, workspace=None, stream=None):
    """prism_w8a8_linear with the codes given as float16 values: ``qh`` [M, K]
    (prism_quant_act_f16) and ``wh`` [N, K] (prism_codes_to_f16).  Same
    result, bit for bit; ``workspace`` as prism_w8a8_linear's, sized by
    prism_w8a8_f16_workspace_bytes."""
    import torch
    _require(qh, torch.float16, "qh", 2)
    _require(wh, torch.float16, "wh", 2)
    _require(a_scale, torch.float32, "a_scale", 1)
    _require(w_scale, torch.float32, "w_scale", 1)
    M, K = qh.shape
    N = wh.shape[0]
    if wh.shape[1] != K or a_scale.numel() != M or w_scale.numel() != N:
        raise ValueError("shape mismatch")
    if residual is not None:
        _require(residual, torch.bfloat16, "residual", 2)
        if tuple(residual.shape) != (M, N):
            raise ValueError("residual must be [M, N]")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=qh.device)
    _require(out, torch.bfloat16, "out", 2)
    if tuple(out.shape) != (M, N):
        raise ValueError("out must be [M, N]")
    if acc_out is not None:
        _require(acc_out, torch.int32, "acc_out", 2)
        if not acc_out.is_contiguous() or tuple(acc_out.shape) != (M, N):
            raise ValueError("acc_out must be a contiguous [M, N] int32 tensor")
    if workspace is None:
        workspace = new_workspace_f16(M, N, K, split_k, qh.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().prism_w8a8_linear_f16(
        _ptr(qh), qh.stride(0), _ptr(a_scale), _ptr(wh), wh.stride(0), _ptr(w_scale),
        _ptr(residual), 0 if residual is None else residual.stride(0), _ptr(out), out.stride(0),
        _ptr(acc_out), M, N, K, int(split_k), _ptr(workspace), ws_bytes, _stream(stream))
    _check("prism_w8a8_linear_f16", st)
    return out
