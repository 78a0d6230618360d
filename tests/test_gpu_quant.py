"""GPU parity of prism_quant_act against the CPU oracle: int8 codes and
per-token scales bit-exact, including ragged, strided, extreme and degenerate
rows, for every register-cache width of the persistent kernel, the long-row
kernel beyond it, and many rows per CTA."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_util import dev, dev_bf16, host, padded

import deterministic_w8a8_int8_gb300 as prism

pytestmark = pytest.mark.gpu


def run(x_bits, inv_s, ldx=None, ldq=None):
    M, K = x_bits.shape
    if ldx is None:
        x = dev_bf16(x_bits)
    else:
        x = padded(M, K, ldx, torch.bfloat16)
        x.copy_(dev_bf16(x_bits))
    q = None if ldq is None else padded(M, K, ldq, torch.int8, fill=99)
    s = None if inv_s is None else dev(inv_s)
    q, a = prism.prism_quant_act(x, s, q=q)
    torch.cuda.synchronize()
    return host(q), host(a)


def check(x_bits, inv_s, **kw):
    qg, ag = run(x_bits, inv_s, **kw)
    qo, ao = oracle.quant_act(x_bits, inv_s)
    assert np.array_equal(qg, qo)
    assert np.array_equal(ag.view(np.uint32), ao.view(np.uint32))


# The persistent kernel takes rows up to 24576 with C = 1..6 vectors of 8 per
# thread in teams of up to 512; every width appears, with the 24576 boundary
# and the long-row kernel past it, and shapes with many rows per CTA (the
# prefetching row loop: 3000 x 5120, 2048 x 17408).
@pytest.mark.parametrize("M,K", [(1, 16), (5, 48), (37, 256), (3, 272), (7, 1040), (9, 2064),
                                 (4, 4112), (3, 8192), (40, 12288), (40, 12304), (20, 16384),
                                 (2, 18432), (2, 20016), (64, 17408), (20, 24576), (8, 24592),
                                 (304, 5120), (3000, 5120), (2048, 17408)])
@pytest.mark.parametrize("smooth", [True, False])
def test_quant_parity_shapes(cuda_device, M, K, smooth):
    rng = np.random.default_rng(M * 7919 + K)
    x = rng.standard_normal((M, K), dtype=np.float32)
    x[:, rng.choice(K, size=max(1, K // 100), replace=False)] *= 30
    xb = wl.bf16_bits(x)
    inv_s = rng.uniform(0.05, 3.0, K).astype(np.float32) if smooth else None
    check(xb, inv_s)


def test_quant_tiny_config(cuda_device):
    case = wl.make_linear("tiny_m37_k256_n384")
    check(case.x_bits, case.inv_s)


def test_quant_strided(cuda_device):
    rng = np.random.default_rng(2)
    xb = wl.bf16_bits(rng.standard_normal((33, 528), dtype=np.float32))
    check(xb, None, ldx=552, ldq=560)


def test_quant_degenerate_rows(cuda_device):
    K = 512
    x = np.zeros((8, K), np.float32)
    x[1, 3] = 2.0 ** -125                         # below 2^-120: zero row
    x[2, :] = 3.0e38                               # near bf16 max
    x[2, 1::2] = -3.0e38
    x[3, :] = 1e-30                                # tiny but above 2^-120
    x[4, 0] = 127.0
    x[4, 1:9] = [0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 3.5, 126.5]   # exact ties
    x[5, :] = np.linspace(-1, 1, K)
    x[6, 7] = -4.0                                 # single negative spike
    x[7, :] = 1.0
    check(wl.bf16_bits(x), None)
    check(wl.bf16_bits(x), np.full(K, 0.5, np.float32))


def test_quant_max_k(cuda_device):
    K = 133136
    rng = np.random.default_rng(4)
    xb = wl.bf16_bits(rng.standard_normal((2, K), dtype=np.float32))
    check(xb, rng.uniform(0.5, 2.0, K).astype(np.float32))


def test_quant_empty_is_noop(cuda_device):
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    q, a = prism.prism_quant_act(x)
    assert q.shape == (0, 64) and a.shape == (0,)
