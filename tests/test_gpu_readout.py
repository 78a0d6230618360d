"""GPU parity of prism_candidate_readout against the CPU oracle: candidate
logits and probabilities bit-exact, on the full 248,000 x 5120 LM head and on
the 32,000-row identity instance; invalid candidate lists raise device error
bits and NaN outputs without trapping ("把决策模型推理从 vLLM 换到 Prism",
sections 方案, 实现要点 and 复盘)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_util import dev, dev_bf16, host

import deterministic_w8a8_int8_gb300 as prism

pytestmark = pytest.mark.gpu


def lm_head_on_device(case: wl.ReadoutCase, seed: int = 0):
    """Full [V, K] head: random filler drawn on the device, with the candidate
    rows (the only rows the outputs depend on) drawn by the seeded generator."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    W = torch.randint(-127, 128, (case.V, case.K), dtype=torch.int8, device="cuda", generator=g)
    uniq = np.unique(case.cand_ids)
    rows = case.lm_rows(uniq)
    W[torch.from_numpy(uniq.astype(np.int64)).cuda()] = dev(rows)
    return W, uniq, rows


def run(case, W, err=None, inv_s=None):
    logits, probs = prism.prism_candidate_readout(
        dev_bf16(case.h_bits), None if inv_s is None else dev(inv_s), W, dev(case.lm_scale),
        dev(case.cand_offsets), dev(case.cand_ids), err=err)
    torch.cuda.synchronize()
    return host(logits), host(probs)


def test_full_vocabulary_readout_parity(cuda_device):
    case = wl.make_readout("readout_p192_v248000")
    W, uniq, rows = lm_head_on_device(case)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lg, pr = run(case, W, err=err)
    assert int(err.item()) == 0
    remap = np.searchsorted(uniq, case.cand_ids).astype(np.int32)
    rc, lo, po = oracle.candidate_readout(case.h_bits, None, rows, case.lm_scale[uniq],
                                          case.cand_offsets, remap)
    assert rc == 0
    assert np.array_equal(lg.view(np.uint32), lo.view(np.uint32))
    assert np.array_equal(pr.view(np.uint32), po.view(np.uint32))


def test_identity_instance_parity_and_smoothing(cuda_device):
    case = wl.make_readout("identity_p16_v32000")
    Wn = case.lm_head_full()
    W = dev(Wn)
    for inv_s in (None, np.random.default_rng(3).uniform(0.5, 2.0, case.K).astype(np.float32)):
        lg, pr = run(case, W, inv_s=inv_s)
        rc, lo, po = oracle.candidate_readout(case.h_bits, inv_s, Wn, case.lm_scale,
                                              case.cand_offsets, case.cand_ids)
        assert rc == 0
        assert np.array_equal(lg.view(np.uint32), lo.view(np.uint32))
        assert np.array_equal(pr.view(np.uint32), po.view(np.uint32))


@pytest.mark.parametrize("cmin,cmax", [(1, 1), (2, 10), (60, 64)])
def test_candidate_count_range(cuda_device, cmin, cmax):
    case = wl.make_readout("identity_p16_v32000", P=40, K=1040, V=4000, cmin=cmin, cmax=cmax)
    Wn = case.lm_head_full()
    lg, pr = run(case, dev(Wn))
    rc, lo, po = oracle.candidate_readout(case.h_bits, None, Wn, case.lm_scale,
                                          case.cand_offsets, case.cand_ids)
    assert rc == 0
    assert np.array_equal(lg.view(np.uint32), lo.view(np.uint32))
    assert np.array_equal(pr.view(np.uint32), po.view(np.uint32))
    if cmax == 1:
        assert np.all(pr == 1.0)


def test_invalid_candidates_flag_and_nan(cuda_device):
    rng = np.random.default_rng(13)
    K, V = 256, 50
    Wn = rng.integers(-127, 128, size=(V, K), dtype=np.int8)
    sc = rng.uniform(0.001, 0.02, V).astype(np.float32)
    h = wl.bf16_bits(rng.standard_normal((5, K), dtype=np.float32))
    off = np.array([0, 2, 4, 6, 6, 8], np.int32)
    ids = np.array([1, 2, 3, 3, 4, 50, 7, 8], np.int32)   # dup, out of range, empty
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lg, pr = prism.prism_candidate_readout(dev_bf16(h), None, dev(Wn), dev(sc), dev(off), dev(ids), err=err)
    torch.cuda.synchronize()
    e = int(err.item())
    assert e == (prism.PRISM_DEV_ERR_DUPLICATE | prism.PRISM_DEV_ERR_ID_RANGE | prism.PRISM_DEV_ERR_COUNT)
    pr = host(pr)
    assert np.isnan(pr[2:6]).all()
    rc, lo, po = oracle.candidate_readout(h[[0, 4]], None, Wn, sc, np.array([0, 2, 4], np.int32),
                                          ids[[0, 1, 6, 7]])
    assert rc == 0
    assert np.array_equal(pr[[0, 1, 6, 7]].view(np.uint32), po.view(np.uint32))
    # offsets outside [0, T]: flagged, nothing written
    err.zero_()
    bad_off = np.array([0, 2, 9], np.int32)
    prism.prism_candidate_readout(dev_bf16(h[:2]), None, dev(Wn), dev(sc), dev(bad_off),
                                  dev(ids[:4]), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & prism.PRISM_DEV_ERR_OFFSETS


def test_empty_readout_is_noop(cuda_device):
    z = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((4, 64), dtype=torch.int8, device="cuda")
    lg, pr = prism.prism_candidate_readout(z, None, W, torch.ones(4, device="cuda"),
                                           torch.zeros(1, dtype=torch.int32, device="cuda"),
                                           torch.zeros(0, dtype=torch.int32, device="cuda"))
    assert lg.numel() == 0 and pr.numel() == 0
