"""GPU parity of prism_w8a8_linear against the CPU oracle, and the layer's
invariances: int32 accumulators and bf16 outputs bit-exact; identical bits
for every split-K factor, batch size, batch composition and row order
(StartLux-Prism, "Bitwise consistency is not lossless quantization")."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_util import dev, dev_bf16, host, host_bits, padded

import deterministic_w8a8_int8_gb300 as prism

pytestmark = pytest.mark.gpu


def gpu_linear(q, a, w, ws, res=None, split=0, acc=True, out=None):
    M, N = q.shape[0], w.shape[0]
    acc_t = torch.empty((M, N), dtype=torch.int32, device="cuda") if acc else None
    out = prism.prism_w8a8_linear(q, a, w, ws, residual=res, out=out, acc_out=acc_t, split_k=split)
    torch.cuda.synchronize()
    return out, acc_t


def random_problem(M, N, K, seed, residual=True):
    rng = np.random.default_rng(seed)
    xb = wl.bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    w = wl.draw_weights(rng, (N, K), "normal")
    w_scale = rng.uniform(0.001, 0.02, N).astype(np.float32)
    rb = wl.bf16_bits(rng.standard_normal((M, N), dtype=np.float32)) if residual else None
    return xb, w, w_scale, rb


def oracle_full(xb, inv_s, w, w_scale, rb):
    q, a = oracle.quant_act(xb, inv_s)
    out, acc = oracle.w8a8_linear(q, a, w, w_scale, rb)
    return q, a, out, acc


def test_tiny_config_end_to_end(cuda_device):
    c = wl.make_linear("tiny_m37_k256_n384")
    qo, ao, outo, acco = oracle_full(c.x_bits, c.inv_s, c.w, c.w_scale, c.residual_bits)
    q, a = prism.prism_quant_act(dev_bf16(c.x_bits), dev(c.inv_s))
    assert np.array_equal(host(q), qo) and np.array_equal(host(a), ao)
    w, ws, r = dev(c.w), dev(c.w_scale), dev_bf16(c.residual_bits)
    out, acc = gpu_linear(q, a, w, ws, r)
    assert np.array_equal(host(acc), acco)
    assert np.array_equal(host_bits(out), outo)
    # the same rows run one at a time give the same bits
    for m in range(c.M):
        q1, a1 = prism.prism_quant_act(dev_bf16(c.x_bits[m:m + 1]), dev(c.inv_s))
        o1, _ = gpu_linear(q1, a1, w, ws, r[m:m + 1], acc=False)
        assert np.array_equal(host_bits(o1)[0], outo[m]), m


@pytest.mark.parametrize("M,N,K", [(1, 8, 16), (3, 130, 48), (129, 384, 256), (37, 131, 64),
                                   (130, 257, 528), (255, 136, 1040), (1, 1, 16)])
@pytest.mark.parametrize("residual", [True, False])
@pytest.mark.parametrize("ld_pad", [8, 1])
def test_ragged_shapes(cuda_device, M, N, K, residual, ld_pad):
    xb, w, w_scale, rb = random_problem(M, N, K, M * 131 + N * 7 + K, residual)
    _, _, outo, acco = oracle_full(xb, None, w, w_scale, rb)
    q, a = prism.prism_quant_act(dev_bf16(xb))
    ld = (N + 7) // 8 * 8 + 8 if ld_pad == 8 else N + 1
    r = None
    if residual:
        r = padded(M, N, ld, torch.bfloat16)
        r.copy_(dev_bf16(rb))
    out = padded(M, N, ld, torch.bfloat16)
    out, acc = gpu_linear(q, a, dev(w), dev(w_scale), r, out=out)
    assert np.array_equal(host(acc), acco)
    assert np.array_equal(host_bits(out), outo)


@pytest.mark.parametrize("split", [1, 2, 3, 4, 7, 8, 16, 33, 64])
def test_split_k_bit_identical(cuda_device, split):
    M, N, K = 70, 520, 2064
    xb, w, w_scale, rb = random_problem(M, N, K, 17)
    _, _, outo, acco = oracle_full(xb, None, w, w_scale, rb)
    q, a = prism.prism_quant_act(dev_bf16(xb))
    out, acc = gpu_linear(q, a, dev(w), dev(w_scale), dev_bf16(rb), split=split)
    assert np.array_equal(host(acc), acco)
    assert np.array_equal(host_bits(out), outo)


def test_split_k_workspace_reuse_stays_zero(cuda_device):
    M, N, K = 40, 300, 4096
    xb, w, w_scale, rb = random_problem(M, N, K, 23)
    _, _, outo, _ = oracle_full(xb, None, w, w_scale, rb)
    q, a = prism.prism_quant_act(dev_bf16(xb))
    ws_buf = prism.new_workspace(M, N, K, 8, "cuda")
    W, S, R = dev(w), dev(w_scale), dev_bf16(rb)
    for _ in range(3):
        out = prism.prism_w8a8_linear(q, a, W, S, residual=R, split_k=8, workspace=ws_buf)
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(out), outo)
        assert int(ws_buf.count_nonzero()) == 0


def test_in_place_residual(cuda_device):
    M, N, K = 50, 264, 512
    xb, w, w_scale, rb = random_problem(M, N, K, 5)
    _, _, outo, _ = oracle_full(xb, None, w, w_scale, rb)
    q, a = prism.prism_quant_act(dev_bf16(xb))
    for split in (1, 4):
        buf = dev_bf16(rb)
        prism.prism_w8a8_linear(q, a, dev(w), dev(w_scale), residual=buf, out=buf, split_k=split)
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(buf), outo)


def test_int32_extremes_at_max_k(cuda_device):
    K = 133136
    q = np.full((3, K), 127, np.int8)
    q[1] = -127
    q[2, ::2] = -127
    w = np.full((16, K), 127, np.int8)
    w[1::2] = -127
    a = np.ones(3, np.float32)
    ws = np.full(16, 1.0, np.float32)
    outo, acco = oracle.w8a8_linear(q, a, w, ws, None)
    assert acco[0, 0] == K * 16129
    for split in (1, 5, 16):
        out, acc = gpu_linear(dev(q), dev(a), dev(w), dev(ws), None, split=split)
        assert np.array_equal(host(acc), acco)
        assert np.array_equal(host_bits(out), outo)


def test_batch_composition_and_row_order(cuda_device):
    M, N, K = 96, 640, 1024
    xb, w, w_scale, rb = random_problem(M, N, K, 31)
    W, S = dev(w), dev(w_scale)
    q, a = prism.prism_quant_act(dev_bf16(xb))
    base, _ = gpu_linear(q, a, W, S, dev_bf16(rb), acc=False)
    base = host_bits(base)
    perm = np.random.default_rng(0).permutation(M)
    qp, ap = prism.prism_quant_act(dev_bf16(xb[perm]))
    o, _ = gpu_linear(qp, ap, W, S, dev_bf16(rb[perm]), acc=False)
    assert np.array_equal(host_bits(o), base[perm])
    # unrelated extra rows added to the batch change nothing
    xe, _, _, re_ = random_problem(300, N, K, 99)
    xa = np.concatenate([xe[:150], xb, xe[150:]])
    ra = np.concatenate([re_[:150], rb, re_[150:]])
    qa, aa = prism.prism_quant_act(dev_bf16(xa))
    o, _ = gpu_linear(qa, aa, W, S, dev_bf16(ra), acc=False)
    assert np.array_equal(host_bits(o)[150:150 + M], base)


def test_decode_rows_invariant_across_m_and_split(cuda_device):
    c = wl.make_linear("decode_m64_k17408_n5120")
    W, S = dev(c.w), dev(c.w_scale)
    inv = dev(c.inv_s)
    ref = None
    for M in wl.DECODE_M:
        q, a = prism.prism_quant_act(dev_bf16(c.x_bits[:M]), inv)
        R = dev_bf16(c.residual_bits[:M])
        for split in wl.DECODE_SPLITS:
            o, _ = gpu_linear(q, a, W, S, R, split=split, acc=False)
            o = host_bits(o)
            if ref is None:
                ref = {}
            for m in range(M):
                if m in ref:
                    assert np.array_equal(o[m], ref[m]), (M, split, m)
                else:
                    ref[m] = o[m]
    # and the rows match the oracle on sampled output channels
    cols = np.random.default_rng(1).choice(c.N, 384, replace=False)
    qo, ao = oracle.quant_act(c.x_bits, c.inv_s)
    outo, _ = oracle.w8a8_linear(qo, ao, c.w[cols], c.w_scale[cols], c.residual_bits[:, cols])
    got = np.stack([ref[m] for m in range(64)])
    assert np.array_equal(got[:, cols], outo)


@pytest.mark.parametrize("name", ["forest_qkv_m304_k5120_n15360", "forest_oproj_m304_k5120_n5120",
                                  "load_gateup_m2048_k5120_n34816", "load_down_m2048_k17408_n5120",
                                  "long_m8192_k5120_n5120"])
def test_full_size_every_tile(cuda_device, name):
    """Full-size call in the benchmark's launch configuration (automatic
    schedule, so shared tiles and their read-back are included): one row of
    every 128-row block (plus the first and last rows) checked against the
    oracle across ALL output channels, accumulators and outputs -- every
    output tile of either orientation holds some of the checked elements."""
    c = wl.make_linear(name)
    q, a = prism.prism_quant_act(dev_bf16(c.x_bits), dev(c.inv_s))
    R = None if c.residual_bits is None else dev_bf16(c.residual_bits)
    out, acc = gpu_linear(q, a, dev(c.w), dev(c.w_scale), R, acc=True)
    rng = np.random.default_rng(7)
    rows = [0, c.M - 1] + [b * 128 + int(rng.integers(0, min(128, c.M - b * 128))) for b in range((c.M + 127) // 128)]
    rows = np.unique(np.array(rows))
    qo, ao = oracle.quant_act(c.x_bits[rows], c.inv_s)
    assert np.array_equal(host(q)[rows], qo) and np.array_equal(host(a)[rows], ao)
    rr = None if c.residual_bits is None else c.residual_bits[rows]
    outo, acco = oracle.w8a8_linear(qo, ao, c.w, c.w_scale, rr)
    assert np.array_equal(host(acc)[rows], acco)
    assert np.array_equal(host_bits(out)[rows], outo)


def _with_path(path, fn):
    import os
    old = os.environ.get("PRISM_LINEAR_PATH")
    if path in ("mma", "tc", "gemv", "stream"):
        os.environ["PRISM_LINEAR_PATH"] = path
    else:                      # the library's own choice
        os.environ.pop("PRISM_LINEAR_PATH", None)
    try:
        return fn()
    finally:
        if old is None:
            os.environ.pop("PRISM_LINEAR_PATH", None)
        else:
            os.environ["PRISM_LINEAR_PATH"] = old


@pytest.mark.parametrize("M", [5, 40, 130, 600])
def test_tensor_core_chunks_exact_at_2_pow_24(cuda_device, M):
    """Every fp32 chunk of <= 1024 products stays an exact integer: all
    +-127 operands (chunk partials up to 1024 * 16129 = 16,516,096) and single
    +-1 terms next to near-2^24 partials must come out exact."""
    K = 4096 + 1024 + 64
    rng = np.random.default_rng(M)
    q = np.full((M, K), 127, np.int8)
    q[1::3] = -127
    q[2::3, 1023::1024] = 1          # a unit term at the end of every chunk
    N = 264
    w = np.where(rng.random((N, K)) < 0.5, 127, -127).astype(np.int8)
    w[0] = 127
    w[1] = -127
    w[2, 1023::1024] = -1
    w[3, ::2] = 1
    a = np.ones(M, np.float32)
    ws = np.ones(N, np.float32)
    outo, acco = oracle.w8a8_linear(q, a, w, ws, None)
    assert abs(int(acco[0, 0])) == 127 * 127 * K
    for split in (1, 3):
        out, acc = gpu_linear(dev(q), dev(a), dev(w), dev(ws), None, split=split)
        assert np.array_equal(host(acc), acco)
        assert np.array_equal(host_bits(out), outo)
    assert prism.prism_device_status() == 0


@pytest.mark.parametrize("M", [9, 96, 97, 128])
@pytest.mark.parametrize("K", [64, 128, 192, 2064])
def test_stage_width_boundaries(cuda_device, M, K):
    """Tensor-core tiles up to 96 wide stream stages of 128 K (two 64-K f16
    slots per stage, 128-byte TMA rows), wider tiles stages of 64 K: both
    sides of that width boundary, one whole stage, a half-filled last stage
    and K below one stage give the oracle's bits, under the automatic
    schedule and explicit split-K alike."""
    N = 264
    xb, w, w_scale, rb = random_problem(M, N, K, 7 * M + K)
    _, _, outo, acco = oracle_full(xb, None, w, w_scale, rb)
    q, a = prism.prism_quant_act(dev_bf16(xb))
    W, S, R = dev(w), dev(w_scale), dev_bf16(rb)
    for split in (0, 3):
        out, acc = _with_path("tc", lambda: gpu_linear(q, a, W, S, R, split=split))
        assert np.array_equal(host(acc), acco), split
        assert np.array_equal(host_bits(out), outo), split
    assert prism.prism_device_status() == 0


@pytest.mark.parametrize("M,N,K", [(37, 384, 256), (304, 512, 5120), (600, 520, 2064), (64, 1024, 17408)])
def test_contraction_kernels_agree(cuda_device, M, N, K):
    """The tcgen05 kernel and the mma.sync s8 kernel give identical bits."""
    xb, w, w_scale, rb = random_problem(M, N, K, 41 + M)
    q, a = prism.prism_quant_act(dev_bf16(xb))
    W, S, R = dev(w), dev(w_scale), dev_bf16(rb)
    kinds = {p: _with_path(p, lambda: prism.prism_w8a8_kernel_kind(M, N, K)) for p in ("tc", "mma")}
    assert kinds["mma"] == 1 and kinds["tc"] in (2, 3)
    outs = {p: _with_path(p, lambda: gpu_linear(q, a, W, S, R)) for p in ("tc", "mma")}
    assert torch.equal(outs["tc"][1], outs["mma"][1])
    assert torch.equal(outs["tc"][0].view(torch.int16), outs["mma"][0].view(torch.int16))
    _, _, outo, _ = oracle_full(xb, None, w, w_scale, rb)
    assert np.array_equal(host_bits(outs["tc"][0]), outo)
    assert prism.prism_device_status() == 0


@pytest.mark.parametrize("M,N,K", [(600, 512, 4096), (64, 512, 3072), (304, 520, 5120), (1000, 300, 2048)])
def test_repeated_runs_bit_identical(cuda_device, M, N, K):
    """Twenty back-to-back calls (different pipeline timings each time) must
    all give the oracle's bits: a race between the staging, widening and MMA
    stages would show up as an intermittent mismatch."""
    rng = np.random.default_rng(M + N + K)
    q = rng.integers(-127, 128, (M, K), dtype=np.int8)
    w = rng.integers(-127, 128, (N, K), dtype=np.int8)
    acco = oracle.gemm_s32(q, w)
    Q, W = dev(q), dev(w)
    a = torch.ones(M, device="cuda")
    s = torch.ones(N, device="cuda")
    accs = [torch.empty((M, N), dtype=torch.int32, device="cuda") for _ in range(20)]
    for acc in accs:
        prism.prism_w8a8_linear(Q, a, W, s, acc_out=acc, split_k=1)
    torch.cuda.synchronize()
    for acc in accs:
        assert np.array_equal(host(acc), acco)
    assert prism.prism_device_status() == 0


@pytest.mark.gpu
@pytest.mark.parametrize("M,N,K", [
    (1024, 4864, 512),    # 152 tiles: whole tiles only, one round
    (304, 1536, 5120),    # 24 tiles shared out over 120 CTAs (5 K ranges each)
    (600, 2560, 2048),    # 50 tiles, K units shared over 152 CTAs
    (304, 15360, 1024),   # 240 tiles: one round of whole tiles, the rest shared
    (37, 384, 256),       # 3 tiles of 4 K stages: one CTA per tile
    (640, 25600, 256),    # 500 tiles of 4 K stages: whole tiles in rounds
    (96, 640, 17408),     # 5 tiles of 272 K stages over 152 CTAs
])
def test_balanced_schedule_matches_single_piece(cuda_device, M, N, K):
    """The automatic (balanced) schedule -- whole tiles, then K ranges of the
    remaining tiles shared between CTAs and summed from partial-tile slots --
    gives the same bits as one K piece per tile, for shapes that reach each
    branch of the schedule choice; the slots and counters are reused by a
    second call."""
    rng = np.random.default_rng(M * 7 + N + K)
    q = dev(rng.integers(-127, 128, (M, K), dtype=np.int8))
    w = dev(rng.integers(-127, 128, (N, K), dtype=np.int8))
    a = dev((rng.random(M, dtype=np.float32) * 1e-3 + 1e-4).astype(np.float32))
    s = dev((rng.random(N, dtype=np.float32) * 1e-2 + 1e-3).astype(np.float32))
    rb = wl.bf16_bits(rng.normal(size=(M, N)).astype(np.float32))
    ref, ref_acc = gpu_linear(q, a, w, s, dev_bf16(rb), split=1)
    ref_bits, ref_acc = ref.view(torch.int16).cpu().numpy(), ref_acc.cpu().numpy()
    ws_buf = prism.new_workspace(M, N, K, 0, torch.device("cuda", 0))
    for _ in range(2):
        acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
        got = prism.prism_w8a8_linear(q, a, w, s, residual=dev_bf16(rb), split_k=0, workspace=ws_buf, acc_out=acc)
        torch.cuda.synchronize()
        assert np.array_equal(got.view(torch.int16).cpu().numpy(), ref_bits)
        assert np.array_equal(acc.cpu().numpy(), ref_acc)


@pytest.mark.gpu
def test_balanced_schedule_without_room_uses_whole_tiles(cuda_device):
    """Given less workspace than the balanced schedule's partial tiles need,
    an automatic call is refused; the no-workspace entry point runs the same
    shape with whole tiles and gives the same bits."""
    M, N, K = 304, 15360, 1024
    rng = np.random.default_rng(5)
    q = dev(rng.integers(-127, 128, (M, K), dtype=np.int8))
    w = dev(rng.integers(-127, 128, (N, K), dtype=np.int8))
    a = dev(np.full(M, 1e-3, np.float32))
    s = dev(np.full(N, 1e-2, np.float32))
    ref, _ = gpu_linear(q, a, w, s, None, split=1)
    ref = ref.view(torch.int16).cpu().numpy()
    need = prism.prism_w8a8_workspace_bytes(M, N, K, 0)
    assert need > prism.PRISM_NOALLOC_SCRATCH_BYTES
    with pytest.raises(prism.PrismError):
        prism.prism_w8a8_linear(q, a, w, s, split_k=0,
                                workspace=torch.zeros(need // 2, dtype=torch.uint8, device="cuda"))
    out = prism.prism_w8a8_linear_noalloc(q, a, w, s, split_k=0)
    assert np.array_equal(out.view(torch.int16).cpu().numpy(), ref)
