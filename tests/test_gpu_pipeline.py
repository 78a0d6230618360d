"""The whole hot path as one stream of dependent launches, with no host
synchronisation between them: quantise -> linear -> quantise -> linear with
an in-place residual -> candidate read-out of rows of the last output.  Every
library kernel may start while its predecessor finishes and waits for it
before reading data; a missing wait would let a kernel read a buffer its
predecessor is still writing.  Each round feeds new inputs through the same
device buffers, and every output is compared bit for bit with the oracle's
chain (StartLux-Prism, "Bitwise consistency is not lossless quantization";
"把决策模型推理从 vLLM 换到 Prism", sections 方案 and 实现要点)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_util import dev, host, host_bits

import deterministic_w8a8_int8_gb300 as prism

pytestmark = pytest.mark.gpu


def oracle_chain(x1, inv1, w1, s1, x2, inv2, w2, s2, res, rows, lm, lm_scale, off, ids):
    q1, a1 = oracle.quant_act(x1, inv1)
    y, _ = oracle.w8a8_linear(q1, a1, w1, s1, None)
    q2, a2 = oracle.quant_act(x2, inv2)
    h, _ = oracle.w8a8_linear(q2, a2, w2, s2, res)
    rc, logits, probs = oracle.candidate_readout(h[rows], None, lm, lm_scale, off, ids)
    assert rc == 0
    return y, h, logits, probs


@pytest.mark.parametrize("M,K,N1,N2", [(304, 512, 1536, 512), (96, 1024, 640, 1024)])
def test_dependent_launch_chain_matches_oracle(cuda_device, M, K, N1, N2):
    rng = np.random.default_rng(M + K)
    V = 4096
    w1 = wl.draw_weights(rng, (N1, K), "normal")
    w2 = wl.draw_weights(rng, (N2, K), "normal")
    s1 = rng.uniform(0.001, 0.02, N1).astype(np.float32)
    s2 = rng.uniform(0.001, 0.02, N2).astype(np.float32)
    lm = wl.draw_weights(rng, (V, N2), "normal")
    lm_scale = rng.uniform(0.001, 0.02, V).astype(np.float32)
    inv1 = rng.uniform(0.5, 2.0, K).astype(np.float32)
    inv2 = rng.uniform(0.5, 2.0, K).astype(np.float32)
    d = M // 4
    rows = np.array([d, 2 * d, 3 * d])   # equally spaced: a strided view, no gather kernel
    counts = np.array([3, 7, 2])
    off = np.zeros(4, np.int32)
    off[1:] = np.cumsum(counts)
    ids = np.concatenate([rng.choice(V, size=c, replace=False) for c in counts]).astype(np.int32)

    dv = torch.device("cuda", 0)
    W1, W2, S1, S2, LM, LS = dev(w1), dev(w2), dev(s1), dev(s2), dev(lm), dev(lm_scale)
    I1, I2, OFF, IDS = dev(inv1), dev(inv2), dev(off), dev(ids)
    X1 = torch.empty((M, K), dtype=torch.bfloat16, device=dv)
    X2 = torch.empty_like(X1)
    HR = torch.empty((M, N2), dtype=torch.bfloat16, device=dv)   # residual in, output out (in place)
    Y = torch.empty((M, N1), dtype=torch.bfloat16, device=dv)
    q1 = torch.empty((M, K), dtype=torch.int8, device=dv)
    q2 = torch.empty_like(q1)
    a1 = torch.empty((M,), dtype=torch.float32, device=dv)
    a2 = torch.empty_like(a1)
    ws1 = prism.new_workspace(M, N1, K, 0, dv)
    ws2 = prism.new_workspace(M, N2, K, 0, dv)
    T = int(off[-1])
    logits = torch.empty((T,), dtype=torch.float32, device=dv)
    probs = torch.empty((T,), dtype=torch.float32, device=dv)

    for rnd in range(3):
        x1 = wl.bf16_bits(rng.standard_normal((M, K), dtype=np.float32) * (rnd + 1))
        x2 = wl.bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
        res = wl.bf16_bits(rng.standard_normal((M, N2), dtype=np.float32))
        # inputs land by ordinary stream-ordered copies; the five launches
        # then follow one another with no synchronisation
        X1.copy_(torch.from_numpy(x1.view(np.int16)).view(torch.bfloat16))
        X2.copy_(torch.from_numpy(x2.view(np.int16)).view(torch.bfloat16))
        HR.copy_(torch.from_numpy(res.view(np.int16)).view(torch.bfloat16))
        prism.prism_quant_act(X1, I1, q=q1, a_scale=a1)
        prism.prism_w8a8_linear(q1, a1, W1, S1, out=Y, workspace=ws1)
        prism.prism_quant_act(X2, I2, q=q2, a_scale=a2)
        prism.prism_w8a8_linear(q2, a2, W2, S2, residual=HR, out=HR, workspace=ws2)
        prism.prism_candidate_readout(HR[d::d][:3], None, LM, LS, OFF, IDS, logits=logits, probs=probs)
        torch.cuda.synchronize()
        y_o, h_o, lg_o, pr_o = oracle_chain(x1, inv1, w1, s1, x2, inv2, w2, s2, res, rows, lm, lm_scale,
                                            off, ids)
        assert np.array_equal(host_bits(Y), y_o), rnd
        assert np.array_equal(host_bits(HR), h_o), rnd
        assert np.array_equal(host(logits).view(np.uint32), lg_o.view(np.uint32)), rnd
        assert np.array_equal(host(probs).view(np.uint32), pr_o.view(np.uint32)), rnd
