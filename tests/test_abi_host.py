"""Host-side tests of the C ABI: the library builds and loads, exports every
function include/prism.h declares, and rejects bad arguments with the right
status before anything is enqueued.  No GPU: every call below fails argument
validation by construction (the pointers are never dereferenced)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from deterministic_w8a8_int8_gb300 import build
    build.build()
    import deterministic_w8a8_int8_gb300 as p
    return p.lib()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(prism_\w+)\s*\(", src))
    return sorted(names)


def test_every_declared_symbol_is_exported(L):
    import deterministic_w8a8_int8_gb300 as p
    names = declared_functions()
    assert {"prism_quant_act", "prism_w8a8_linear", "prism_candidate_readout"} <= set(names)
    for n in names:
        assert hasattr(L, n), n
        assert n in p.SIGNATURES, f"binding lacks {n}"


def test_header_constants_match_binding():
    import deterministic_w8a8_int8_gb300 as p
    src = open(os.path.join(ROOT, "include", "prism.h")).read()
    for name in ("PRISM_MAX_K", "PRISM_MAX_SPLIT_K", "PRISM_MAX_CANDIDATES", "PRISM_MAX_READOUT_K"):
        v = int(re.search(rf"#define {name} (\d+)", src).group(1))
        assert getattr(p, name) == v
    for name, v in re.findall(r"(PRISM_ERR_\w+) = (-?\d+)", src):
        assert getattr(p, name) == int(v)
    for name, v in re.findall(r"#define (PRISM_DEV_ERR_\w+)\s+(\d+)u", src):
        assert getattr(p, name) == int(v)


def test_status_strings(L):
    for s in range(-5, 1):
        assert L.prism_status_string(s)
    assert L.prism_version() >= 100


A = 0x10000  # a 256-byte-aligned fake address; never dereferenced below


def quant(L, x=A, ldx=64, s=None, M=4, K=64, q=A, ldq=64, a=A):
    return L.prism_quant_act(x, ldx, s, M, K, q, ldq, a, None)


def test_quant_act_validation(L):
    assert quant(L, M=0) == 0                       # empty: nothing to do
    assert quant(L, M=-1) == -1
    assert quant(L, K=0) == -1
    assert quant(L, x=None) == -1
    assert quant(L, q=None) == -1
    assert quant(L, a=None) == -1
    assert quant(L, ldx=32) == -1                   # ldx < K
    assert quant(L, K=72, ldx=80, ldq=80) == -2     # K % 16
    assert quant(L, ldx=68, ldq=64) == -2           # ldx % 8
    assert quant(L, ldq=72) == -2                   # ldq % 16
    assert quant(L, x=A + 8) == -2
    assert quant(L, q=A + 4) == -2
    assert quant(L, a=A + 2) == -2
    assert quant(L, s=A + 4) == -2
    K = 133152                                      # multiple of 16 above the int32 bound
    assert quant(L, K=K, ldx=K, ldq=K) == -3


def lin(L, M=64, N=64, K=64, split=1, ws=None, wsb=0, q=A, w=A, out=A, res=None, ldr=0,
        ldq=None, ldw=None, ldo=None, a=A, ws_=A, acc=None):
    ldq = K if ldq is None else ldq
    ldw = K if ldw is None else ldw
    ldo = N if ldo is None else ldo
    return L.prism_w8a8_linear(q, ldq, a, w, ldw, ws_, res, ldr, out, ldo, acc, M, N, K, split,
                               ws, wsb, None)


def test_linear_validation(L):
    assert lin(L, M=0) == 0 and lin(L, N=0) == 0
    assert lin(L, M=-1) == -1 and lin(L, K=0) == -1
    assert lin(L, split=-1) == -1
    assert lin(L, split=65) == -3
    assert lin(L, q=None) == -1 and lin(L, w=None) == -1 and lin(L, out=None) == -1
    assert lin(L, a=None) == -1 and lin(L, ws_=None) == -1
    assert lin(L, ldq=32) == -1 and lin(L, ldo=32) == -1
    assert lin(L, res=A, ldr=32) == -1
    assert lin(L, K=72, ldq=80, ldw=80) == -2
    assert lin(L, ldq=72) == -2 and lin(L, ldw=72) == -2
    assert lin(L, q=A + 8) == -2 and lin(L, w=A + 8) == -2 and lin(L, out=A + 1) == -2
    assert lin(L, res=A + 1, ldr=64) == -2 and lin(L, a=A + 2) == -2
    assert lin(L, acc=A + 2) == -2
    K = 133152
    assert lin(L, K=K) == -3
    # split-K needs a workspace of the advertised size, 256-byte aligned
    need = L.prism_w8a8_workspace_bytes(64, 64, 4096, 4)
    assert need >= 64 * 64 * 4
    assert lin(L, K=4096, split=4) == -4
    assert lin(L, K=4096, split=4, ws=A, wsb=need - 1) == -4
    assert lin(L, K=4096, split=4, ws=A + 16, wsb=need) == -2


def test_workspace_and_dispatch_queries(L):
    assert L.prism_w8a8_workspace_bytes(64, 64, 64, 1) == 0
    assert L.prism_w8a8_workspace_bytes(0, 64, 64, 4) == 0
    assert L.prism_w8a8_workspace_bytes(64, 64, 64, 65) == 0
    for M, N, K in [(1, 5120, 17408), (304, 5120, 5120), (2048, 34816, 5120), (37, 384, 256)]:
        s = L.prism_w8a8_auto_split(M, N, K)
        assert 0 <= s <= 64   # 0: the balanced schedule of the tensor-core kernel
        if s > 0:
            assert L.prism_w8a8_workspace_bytes(M, N, K, 0) == L.prism_w8a8_workspace_bytes(M, N, K, s)
        assert L.prism_w8a8_kernel_kind(M, N, K) in (1, 2, 3, 4, 5)
    # calls of at most 2 token rows stream the weights through dp4a (kind 4),
    # with no workspace
    for M in (1, 2):
        assert L.prism_w8a8_kernel_kind(M, 5120, 17408) == 4
        assert L.prism_w8a8_workspace_bytes(M, 5120, 17408, 0) == 0
        assert L.prism_w8a8_workspace_bytes(M, 5120, 17408, 16) == 0
    # 3 to 16 rows: the mma.sync weight stream (kind 5), whole K per CTA on
    # a wide weight; more rows: tcgen05
    for M in (3, 8, 9, 16):
        assert L.prism_w8a8_kernel_kind(M, 5120, 17408) == 5
        assert L.prism_w8a8_workspace_bytes(M, 5120, 17408, 0) == 0
    assert L.prism_w8a8_workspace_bytes(16, 5120, 17408, 4) == ((16 * 5120 * 4 + 255) & ~255) + 1280
    assert L.prism_w8a8_kernel_kind(17, 5120, 17408) in (2, 3)
    # the balanced schedule keeps partial tiles only when it shares tiles
    assert L.prism_w8a8_workspace_bytes(37, 384, 256, 0) == 0
    assert L.prism_w8a8_workspace_bytes(304, 15360, 5120, 0) > 0
    assert L.prism_w8a8_kernel_kind(0, 5, 16) == 0


def _cdiv(x, y):
    return (x + y - 1) // y


def _balanced_workspace_bytes(M, N, K):
    """The automatic schedule restated: calls of 3 to 16 rows on the
    weight-streaming kernel (whole K per 16-channel CTA, unless the weight has
    too few tiles to fill the SMs: then [M, N] int32 partial sums and one
    counter per tile); more rows on the tensor-core kernel: orientation and
    token-piece width, 64- or 128-K stages, W rounds of whole tiles on the
    152 SMs and R tiles whose K stages are shared (shares of at least one
    1024-K chunk), then the bytes of R arrival counters and R int32 tiles."""
    if M <= 2:                                  # the dp4a weight stream
        return 0
    if M <= 16:                                 # the mma.sync weight stream
        tiles = _cdiv(N, 16)
        if 2 * tiles >= 2 * 152:                 # the tiles fill the SMs twice: whole K per CTA
            return 0
        pieces = min(_cdiv(2 * 152, tiles), max(1, _cdiv(K, 128) // 64))
        if pieces <= 1:
            return 0
        return ((M * N * 4 + 255) & ~255) + ((tiles * 4 + 255) & ~255)
    if M < 512:                                 # tokens on the MMA's N side
        bpiece = _cdiv(_cdiv(M, _cdiv(M, 256)), 32) * 32
        T = _cdiv(N, 128) * _cdiv(M, bpiece)
    else:
        bpiece = 256
        T = _cdiv(M, 128) * _cdiv(N, 256)
    sub = 2 if bpiece <= 96 and K >= 128 else 1
    S, min_units, sms = _cdiv(K, 64 * sub), 16 // sub, 152
    if T % sms == 0:
        return 0
    W, R = T // sms, T % sms
    if R * S < min_units * sms and W >= 1:
        W, R = W - 1, R + sms
    if R * S >= min_units * sms:
        G = sms
    elif W == 0:
        G = max(R, min(sms, R * S // min_units))
    else:
        return 0
    if R == 0 or G == R:
        return 0
    return ((R * 4 + 255) & ~255) + R * 128 * bpiece * 4


def test_balanced_schedule_workspace_matches_its_statement(L, monkeypatch):
    monkeypatch.delenv("PRISM_LINEAR_PATH", raising=False)
    for M in (1, 8, 9, 37, 64, 96, 97, 128, 160, 192, 304, 511, 512, 600, 2048, 8192):
        for N in (384, 640, 5120, 15360, 34816):
            for K in (64, 128, 2064, 5120, 17408):
                assert L.prism_w8a8_workspace_bytes(M, N, K, 0) == _balanced_workspace_bytes(M, N, K), (M, N, K)


def test_f16_workspace_matches_its_statement(L):
    """The binary16-code kernel's workspace: counters, then one slot per
    (shared tile, CTA) piece (tests/sched_util.py restates the schedule)."""
    from tests.sched_util import f16_workspace
    for M in (1, 8, 37, 64, 128, 160, 192, 304, 511, 512, 600, 2048, 8192):
        for N in (384, 640, 5120, 15360, 34816):
            for K in (64, 128, 2064, 5120, 17408):
                assert L.prism_w8a8_f16_workspace_bytes(M, N, K, 0) == f16_workspace(M, N, K)[1], (M, N, K)


def ro(L, P=4, T=8, V=100, K=64, h=A, ldh=64, s=None, W=A, ldw=64, sc=A, off=A, ids=A,
       lg=A, pr=A, err=None):
    return L.prism_candidate_readout(h, ldh, s, W, ldw, sc, V, K, off, ids, P, T, lg, pr, err, None, 0, None)


def test_readout_validation(L):
    assert ro(L, P=0, T=0) == 0
    assert ro(L, P=0, T=3) == -1
    assert ro(L, P=-1) == -1 and ro(L, V=0) == -1 and ro(L, K=0) == -1
    assert ro(L, h=None) == -1 and ro(L, W=None) == -1 and ro(L, sc=None) == -1
    assert ro(L, off=None) == -1 and ro(L, ids=None) == -1
    assert ro(L, lg=None) == -1 and ro(L, pr=None) == -1
    assert ro(L, ldh=32) == -1 and ro(L, ldw=32) == -1
    assert ro(L, K=72, ldh=80, ldw=80) == -2
    assert ro(L, T=4 * 64 + 1) == -3                # beyond the per-position cap
    assert ro(L, K=65536 + 16, ldh=65552, ldw=65552) == -3
    assert ro(L, ldh=68) == -2 and ro(L, ldw=72) == -2
    assert ro(L, h=A + 8) == -2 and ro(L, W=A + 8) == -2 and ro(L, off=A + 2) == -2
    assert ro(L, s=A + 4) == -2 and ro(L, err=A + 2) == -2
    # the read-out needs no scratch for any shape
    assert L.prism_readout_workspace_bytes(192, 1152, 5120) == 0 and L.prism_readout_workspace_bytes(0, 0, 16) == 0


def lo(L, P=4, T=8, V=100, K=64, h=A, ldh=64, s=None, W=A, ldw=64, sc=A, v0=0, Vs=50, off=A, ids=A, lg=A,
       err=None):
    return L.prism_candidate_logits(h, ldh, s, W, ldw, sc, v0, Vs, V, K, off, ids, P, T, lg, err, None)


def test_shard_logits_validation(L):
    """prism_candidate_logits: the shard must lie inside the head; an empty
    shard needs no rows; the read-out's own limits and alignments apply."""
    assert lo(L, P=0, T=0) == 0 and lo(L, P=0, T=3) == -1
    assert lo(L, P=-1) == -1 and lo(L, T=-1) == -1 and lo(L, V=0) == -1 and lo(L, K=0) == -1
    assert lo(L, v0=-1) == -1 and lo(L, Vs=-1) == -1
    assert lo(L, v0=60, Vs=50) == -1                     # past the head's last row
    # a shard ending at the head's last row, and an empty shard without rows,
    # pass the range checks (K = 72 then stops them before any launch)
    assert lo(L, v0=50, Vs=50, K=72, ldh=80, ldw=80) == -2
    assert lo(L, v0=100, Vs=0, W=None, sc=None, K=72, ldh=80, ldw=80) == -2
    assert lo(L, W=None) == -1 and lo(L, sc=None) == -1
    assert lo(L, h=None) == -1 and lo(L, off=None) == -1 and lo(L, lg=None) == -1 and lo(L, ids=None) == -1
    assert lo(L, ldh=32) == -1 and lo(L, ldw=32) == -1
    assert lo(L, K=72, ldh=80, ldw=80) == -2
    assert lo(L, T=4 * 64 + 1) == -3
    assert lo(L, P=1 << 62, T=1) == -3                   # refused before P * cap is formed
    assert lo(L, K=65536 + 16, ldh=65552, ldw=65552) == -3
    assert lo(L, ldh=68) == -2 and lo(L, ldw=72) == -2
    assert lo(L, h=A + 8) == -2 and lo(L, W=A + 8) == -2 and lo(L, off=A + 2) == -2 and lo(L, lg=A + 2) == -2
    assert lo(L, s=A + 4) == -2 and lo(L, err=A + 2) == -2


def test_candidate_softmax_validation(L):
    def sm(P=4, T=8, lg=A, off=A, pr=A, err=None):
        return L.prism_candidate_softmax(lg, off, P, T, pr, err, None)
    assert sm(P=0, T=0) == 0 and sm(P=0, T=2) == -1
    assert sm(P=-1) == -1 and sm(T=-1) == -1
    assert sm(off=None) == -1 and sm(pr=None) == -1 and sm(lg=None) == -1
    assert sm(T=4 * 64 + 1) == -3 and sm(P=1 << 62, T=1) == -3 and sm(P=1 << 31, T=1) == -3
    assert sm(lg=A + 2) == -2 and sm(off=A + 1) == -2 and sm(pr=A + 2) == -2 and sm(err=A + 2) == -2
    assert ro(L, P=1 << 62, T=1) == -3


def test_linear_operand_checks_before_any_launch():
    """The binding refuses mis-shaped or mis-typed outputs and residuals of a
    linear call (the W8A8 linear and its no-workspace variant share these
    checks) before the library is called: a short, strided or int64
    acc_out, or a residual / out with the wrong row count, would otherwise
    become out-of-bounds device accesses."""
    import torch
    import deterministic_w8a8_int8_gb300 as prism
    M, N, K = 4, 8, 32
    q = torch.zeros((M, K), dtype=torch.int8)
    w = torch.zeros((N, K), dtype=torch.int8)
    a, s = torch.ones(M), torch.ones(N)

    def chk(residual=None, out=None, acc_out=None):
        return prism._linear_operands(q, a, w, s, residual, out, acc_out, on_device=False)

    assert chk() == (M, N, K)
    assert chk(residual=torch.zeros((M, N), dtype=torch.bfloat16), out=torch.zeros((M, N), dtype=torch.bfloat16),
               acc_out=torch.zeros((M, N), dtype=torch.int32)) == (M, N, K)
    with pytest.raises(TypeError):
        chk(acc_out=torch.zeros((M, N), dtype=torch.int64))
    with pytest.raises(ValueError):
        chk(acc_out=torch.zeros((M, 2 * N), dtype=torch.int32)[:, :N])      # strided rows
    with pytest.raises(ValueError):
        chk(acc_out=torch.zeros((M - 1, N), dtype=torch.int32))
    with pytest.raises(ValueError):
        chk(residual=torch.zeros((M - 1, N), dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        chk(out=torch.zeros((M + 1, N), dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        prism.prism_w8a8_linear_noalloc(q, a, w, s, acc_out=torch.zeros((M, N), dtype=torch.int32))   # host tensors
