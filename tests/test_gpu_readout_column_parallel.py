"""GPU parity of the column-parallel read-out building blocks
(prism_candidate_logits on vocabulary shards of the LM head, then
prism_candidate_softmax on the shards' summed logits) against the oracle and
the fused read-out: one GPU plays the ranks in turn, the test adding their
logits in place of the SUM all-reduce ("把决策模型推理从 vLLM 换到 Prism",
sections 方案 and 实现要点: the candidate softmax needs the candidates'
logits only).  Shard boundaries anywhere in the vocabulary, the full
248,000-row head, counts 1..64, smoothing, invalid lists."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_util import dev, dev_bf16, host

import deterministic_w8a8_int8_gb300 as prism

pytestmark = pytest.mark.gpu


def _sharded(h, inv_s, W, sc, off, ids, bounds, err=None, order=None):
    """Each shard's logits, summed on the device in the given order, then the
    candidate softmax."""
    V = W.shape[0]
    parts = [prism.prism_candidate_logits(h, inv_s, W[v0:v1], sc[v0:v1], v0, V, off, ids, err=err)
             for v0, v1 in zip(bounds[:-1], bounds[1:])]
    tot = torch.full_like(parts[0], -0.0)
    for r in (order if order is not None else range(len(parts))):
        tot = tot + parts[r]
    probs = prism.prism_candidate_softmax(tot, off, err=err)
    torch.cuda.synchronize()
    return host(tot), host(probs), [host(x) for x in parts]


@pytest.mark.parametrize("bounds", [[0, 32000], [0, 16000, 32000], [0, 1, 31999, 32000], [0, 5000, 11111, 20000, 32000]])
def test_shards_equal_fused_readout_and_oracle(cuda_device, bounds):
    case = wl.make_readout("identity_p16_v32000")
    Wn = case.lm_head_full()
    W, sc = dev(Wn), dev(case.lm_scale)
    h, off, ids = dev_bf16(case.h_bits), dev(case.cand_offsets), dev(case.cand_ids)
    inv_s = np.random.default_rng(5).uniform(0.5, 2.0, case.K).astype(np.float32)
    for s in (None, inv_s):
        S = None if s is None else dev(s)
        lg_f, pr_f = prism.prism_candidate_readout(h, S, W, sc, off, ids)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        lg, pr, parts = _sharded(h, S, W, sc, off, ids, bounds, err=err, order=reversed(range(len(bounds) - 1)))
        assert int(err.item()) == 0
        rc, lo, po = oracle.candidate_readout(case.h_bits, s, Wn, case.lm_scale, case.cand_offsets, case.cand_ids)
        assert rc == 0
        assert np.array_equal(lg.view(np.uint32), lo.view(np.uint32))
        assert np.array_equal(pr.view(np.uint32), po.view(np.uint32))
        assert np.array_equal(lg.view(np.uint32), host(lg_f).view(np.uint32))
        assert np.array_equal(pr.view(np.uint32), host(pr_f).view(np.uint32))
        for (v0, v1), part in zip(zip(bounds[:-1], bounds[1:]), parts):
            _, lo_r = oracle.candidate_logits_shard(case.h_bits, s, Wn[v0:v1], case.lm_scale[v0:v1], v0, Wn.shape[0],
                                                    case.cand_offsets, case.cand_ids)
            assert np.array_equal(part.view(np.uint32), lo_r.view(np.uint32))


def test_shards_of_the_full_vocabulary(cuda_device):
    """The 248,000-row head cut into four shards at arbitrary rows."""
    case = wl.make_readout("readout_p192_v248000", P=48)
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    W = torch.randint(-127, 128, (case.V, case.K), dtype=torch.int8, device="cuda", generator=g)
    uniq = np.unique(case.cand_ids)
    rows = case.lm_rows(uniq)
    W[torch.from_numpy(uniq.astype(np.int64)).cuda()] = dev(rows)
    sc = dev(case.lm_scale)
    h, off, ids = dev_bf16(case.h_bits), dev(case.cand_offsets), dev(case.cand_ids)
    lg, pr, _ = _sharded(h, None, W, sc, off, ids, [0, 61234, 123457, 200001, case.V])
    remap = np.searchsorted(uniq, case.cand_ids).astype(np.int32)
    rc, lo, po = oracle.candidate_readout(case.h_bits, None, rows, case.lm_scale[uniq], case.cand_offsets, remap)
    assert rc == 0
    assert np.array_equal(lg.view(np.uint32), lo.view(np.uint32))
    assert np.array_equal(pr.view(np.uint32), po.view(np.uint32))


@pytest.mark.parametrize("cmin,cmax", [(1, 1), (60, 64)])
def test_shards_candidate_count_range(cuda_device, cmin, cmax):
    case = wl.make_readout("identity_p16_v32000", P=40, K=1040, V=4000, cmin=cmin, cmax=cmax)
    Wn = case.lm_head_full()
    lg, pr, _ = _sharded(dev_bf16(case.h_bits), None, dev(Wn), dev(case.lm_scale), dev(case.cand_offsets),
                         dev(case.cand_ids), [0, 1333, 2500, 4000])
    rc, lo, po = oracle.candidate_readout(case.h_bits, None, Wn, case.lm_scale, case.cand_offsets, case.cand_ids)
    assert rc == 0
    assert np.array_equal(lg.view(np.uint32), lo.view(np.uint32))
    assert np.array_equal(pr.view(np.uint32), po.view(np.uint32))


def test_shards_invalid_lists(cuda_device):
    """A duplicate id and an id outside the whole head: every shard reports
    the bits and writes NaN logits for those positions, the softmax gives
    them NaN probabilities, the other positions are exact."""
    rng = np.random.default_rng(9)
    K, V, P = 128, 300, 6
    W = rng.integers(-127, 128, size=(V, K), dtype=np.int8)
    sc = rng.uniform(0.001, 0.02, V).astype(np.float32)
    h = wl.bf16_bits(rng.standard_normal((P, K), dtype=np.float32))
    off = np.array([0, 3, 6, 9, 12, 15, 18], np.int32)
    ids = rng.choice(V, size=18, replace=False).astype(np.int32)
    ids[4] = ids[3]          # position 1: duplicate
    ids[7] = V + 5           # position 2: outside the head
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lg, pr, _ = _sharded(dev_bf16(h), None, dev(W), dev(sc), dev(off), dev(ids), [0, 120, V], err=err)
    rc, lo, po = oracle.candidate_readout(h, None, W, sc, off, ids)
    e = int(err.item())
    assert e & prism.PRISM_DEV_ERR_DUPLICATE and e & prism.PRISM_DEV_ERR_ID_RANGE
    assert np.isnan(lg[3:9]).all() and np.isnan(pr[3:9]).all()
    good = np.r_[0:3, 9:18]
    assert np.array_equal(lg[good].view(np.uint32), lo[good].view(np.uint32))
    assert np.array_equal(pr[good].view(np.uint32), po[good].view(np.uint32))


def test_shard_argument_checks(cuda_device):
    L = prism.lib()
    import ctypes
    P_ = ctypes.c_void_p
    h = torch.zeros((2, 64), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((10, 64), dtype=torch.int8, device="cuda")
    sc = torch.ones(10, device="cuda")
    off = torch.tensor([0, 1, 2], dtype=torch.int32, device="cuda")
    ids = torch.tensor([1, 2], dtype=torch.int32, device="cuda")
    lg = torch.zeros(2, device="cuda")
    st = P_(torch.cuda.current_stream().cuda_stream)

    def call(v0=0, Vs=10, V=10):
        return L.prism_candidate_logits(P_(h.data_ptr()), 64, None, P_(W.data_ptr()), 64, P_(sc.data_ptr()), v0, Vs,
                                        V, 64, P_(off.data_ptr()), P_(ids.data_ptr()), 2, 2, P_(lg.data_ptr()), None,
                                        st)

    assert call(v0=5, Vs=10, V=10) == prism.PRISM_ERR_INVALID_ARG
    assert call(v0=-1) == prism.PRISM_ERR_INVALID_ARG
    assert call(V=0) == prism.PRISM_ERR_INVALID_ARG
    assert call() == prism.PRISM_OK
    torch.cuda.synchronize()
    assert L.prism_candidate_softmax(P_(lg.data_ptr()), P_(off.data_ptr()), 2, 129, P_(lg.data_ptr()), None, st) \
        == prism.PRISM_ERR_UNSUPPORTED
