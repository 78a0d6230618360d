// readout.cu -- candidate-restricted LM-head read-out with a softmax over the
// candidates only ("把决策模型推理从 vLLM 换到 Prism", sections 方案 and
// 实现要点; StartLux-Prism, "Compute shared evidence once": the last layer's
// read-out work is restricted to the positions needed for answers).
//
// One CTA per answer position p:
//   1. validate the position's CSR slice (count in [1, 64], ids in [0, V),
//      ids distinct); an invalid position ORs PRISM_DEV_ERR_* bits into the
//      caller's error word, writes NaN outputs and returns -- no trap;
//   2. quantise h_p exactly like prism_quant_act, into shared memory;
//   3. each warp takes candidates round-robin and streams the candidate's
//      LM-head row with 16-byte non-allocating loads, dp4a into exact int32,
//      warp-reduces, and forms logit = (float(acc) * a_scale) * lm_scale[c];
//   4. warp 0 forms the softmax: max over the logits, e_c = exp(logit_c -
//      max) and prob_c = e_c / s one candidate per lane, s = e_1 + ... + e_n
//      added in list order; every step binary32 RN.
// A vocabulary shard (the column-parallel read-out): the same kernel with
// the LM head's rows [v0, v0 + Vs) only computes the logits of the
// candidates it holds and writes -0.0 for the others (x + -0.0 == x for every
// x, so a SUM over the shards' outputs gives each logit bit for bit), and a
// separate kernel applies the softmax of step 4 to the combined logits with
// the same arithmetic (candidate_softmax below).
// Bytes: 2K (hidden row) + count * (K + 4) (candidate rows and scales) per
// position, plus 12 bytes per candidate (id, logit, prob) -- HBM- and
// latency-bound (a chain of dependent reads: offsets, ids, rows); nothing is
// written to global memory but the outputs.  The hidden row's loads and the
// candidate rows' copies into shared memory go out as early as their
// addresses are known, so the chain is three memory round trips long.
#include "common.cuh"

namespace prism {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// exp(x) for x <= 0: Cody-Waite reduction x = n ln2 + r (ln2 = 355/512 +
// RN(ln2 - 355/512)), e^r by its Taylor polynomial of degree 7 in Horner form
// with RN(1/k!) coefficients, scaled by 2^n through the exponent field;
// n < -126 gives 0.  Every step is one binary32 RN operation.
__device__ __forceinline__ float cw_exp(float x) {
  const float kLog2e = 0x1.715476p+0f;
  const float kLn2Hi = 0x1.63p-1f;
  const float kLn2Lo = -0x1.bd0106p-13f;
  const float kC2 = 0x1p-1f;
  const float kC3 = 0x1.555556p-3f;
  const float kC4 = 0x1.555556p-5f;
  const float kC5 = 0x1.111112p-7f;
  const float kC6 = 0x1.6c16c2p-10f;
  const float kC7 = 0x1.a01a02p-13f;
  if (x != x) return x;
  if (x > 0.0f) x = 0.0f;
  const float n = rintf(__fmul_rn(x, kLog2e));
  if (n < -126.0f) return 0.0f;
  float r = __fsub_rn(x, __fmul_rn(n, kLn2Hi));
  r = __fsub_rn(r, __fmul_rn(n, kLn2Lo));
  float p = kC7;
  p = __fadd_rn(__fmul_rn(p, r), kC6);
  p = __fadd_rn(__fmul_rn(p, r), kC5);
  p = __fadd_rn(__fmul_rn(p, r), kC4);
  p = __fadd_rn(__fmul_rn(p, r), kC3);
  p = __fadd_rn(__fmul_rn(p, r), kC2);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);
  const float two_n = __uint_as_float(static_cast<uint32_t>(static_cast<int>(n) + 127) << 23);
  return __fmul_rn(p, two_n);
}

__device__ __forceinline__ int dot16(const uint4 a, const uint4 b, int acc) {
  acc = __dp4a(static_cast<int>(a.x), static_cast<int>(b.x), acc);
  acc = __dp4a(static_cast<int>(a.y), static_cast<int>(b.y), acc);
  acc = __dp4a(static_cast<int>(a.z), static_cast<int>(b.z), acc);
  acc = __dp4a(static_cast<int>(a.w), static_cast<int>(b.w), acc);
  return acc;
}

__device__ __forceinline__ float smooth(float v, const float* inv_s, int64_t k) {
  return inv_s != nullptr ? __fmul_rn(v, __ldg(inv_s + k)) : v;
}

// Step 4 in one warp: lane i holds candidates i and 32 + i (l0, l1; lanes
// past the count hold -inf).  The maximum (exact, any order), e_c =
// exp(logit_c - max) and prob_c = e_c / s per lane, s = e_1 + ... + e_n added
// in list order (every lane forms the same sum from shuffled values); every
// step binary32 RN.
__device__ __forceinline__ void candidate_softmax(float l0, float l1, int64_t cnt, int lane, float& p0, float& p1) {
  float mx = fmaxf(l0, l1);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  const float e0 = lane < cnt ? cw_exp(__fsub_rn(l0, mx)) : 0.0f;
  const float e1 = lane + 32 < cnt ? cw_exp(__fsub_rn(l1, mx)) : 0.0f;
  float s = 0.0f;
  const int n0 = static_cast<int>(cnt < 32 ? cnt : 32);
  for (int i = 0; i < n0; ++i) s = __fadd_rn(s, __shfl_sync(0xffffffffu, e0, i));
  for (int i = 32; i < cnt; ++i) s = __fadd_rn(s, __shfl_sync(0xffffffffu, e1, i - 32));
  p0 = __fdiv_rn(e0, s);
  p1 = __fdiv_rn(e1, s);
}

// Hidden rows of up to kRegK elements are read once into registers, with
// loads issued before anything else (they depend on p alone).  The first
// pre_rows candidates of a position (pre_rows set by the launcher from the
// shared memory that two CTAs per SM leave: 16 rows of a 5120-wide head)
// are copied into shared memory with cp.async as soon as each id has passed
// its range check, together with their lm_scale values, so that all of the
// position's gathers are in flight while the list is validated and the
// hidden row quantised; candidates beyond pre_rows are streamed when the dot
// product reaches them.  Two CTAs fit on an SM (at most 128 registers), so
// 192 answer positions run in one wave on 152 SMs.
constexpr int kRegK = 8192;
constexpr int kHidVec = kRegK / 8 / kThreads;   // uint4 (8 bf16) per thread: 4
constexpr int kPreMax = 16;                     // staged candidate rows at most
constexpr int kPrePerWarp = kPreMax / kWarps;   // 2
constexpr int kSmemBudget = 110 * 1024;         // dynamic shared memory per CTA (two per SM)

// kLogits: logits only (a vocabulary shard, probs unused); W and lm_scale
// hold the rows [v0, v0 + Vs) of the V-row head (the whole head: v0 = 0,
// Vs = V).
template <bool kReg, bool kLogits>
__global__ void __launch_bounds__(kThreads, 2)
    readout_kernel(const uint16_t* __restrict__ h, int64_t ldh, const float* __restrict__ inv_s,
                   const int8_t* __restrict__ W, int64_t ldw, const float* __restrict__ lm_scale,
                   int64_t V, int64_t v0, int64_t Vs, int64_t K, const int32_t* __restrict__ off,
                   const int32_t* __restrict__ ids, int64_t T, float* __restrict__ logits,
                   float* __restrict__ probs, uint32_t* __restrict__ err, int pre_rows) {
  extern __shared__ __align__(16) int8_t smem[];
  int8_t* sq = smem;          // [K] the quantised hidden row
  int8_t* srow = smem + K;    // [pre_rows][K] staged candidate rows
  pdl_trigger();
  pdl_wait();
  __shared__ float s_logit[PRISM_MAX_CANDIDATES];
  __shared__ float s_red[kWarps];
  __shared__ unsigned s_bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t p = blockIdx.x;
  const int64_t nchunk = K >> 4;   // 16-byte chunks of a row

  // the hidden row depends on nothing but p: its loads go out first
  const uint16_t* hr = h + p * ldh;
  uint4 hv[kReg ? kHidVec : 1];
  if (kReg) {
#pragma unroll
    for (int i = 0; i < kHidVec; ++i) {
      const int64_t k = (static_cast<int64_t>(tid) + static_cast<int64_t>(i) * kThreads) * 8;
      hv[i] = k < K ? __ldg(reinterpret_cast<const uint4*>(hr + k)) : make_uint4(0u, 0u, 0u, 0u);
    }
  }

  // ---- 1. stage the first candidate rows, validate the candidate list
  const int64_t b = off[p], e = off[p + 1];
  const bool off_ok = b >= 0 && e <= T && b <= e;
  const int64_t cnt = off_ok ? e - b : 0;
  const bool cnt_ok = off_ok && cnt >= 1 && cnt <= PRISM_MAX_CANDIDATES;
  // the position's ids, held by every warp: candidate c is lane c % 32 of
  // id_l (c < 32) or id_h (two coalesced loads; L1 serves the other warps)
  int32_t id_l = -1, id_h = -1;
  if (cnt_ok) {
    if (lane < cnt) id_l = ids[b + lane];
    if (lane + 32 < cnt) id_h = ids[b + lane + 32];
  }
  auto id_of = [&](int64_t c) {   // c is the same in every lane
    return __shfl_sync(0xffffffffu, c < 32 ? id_l : id_h, static_cast<int>(c & 31));
  };
  const int nstage = cnt_ok ? static_cast<int>(cnt < pre_rows ? cnt : pre_rows) : 0;
  int32_t pre_id[kPrePerWarp];
  float pre_ls[kPrePerWarp];
#pragma unroll
  for (int j = 0; j < kPrePerWarp; ++j) {
    const int c = warp + j * kWarps;
    pre_id[j] = -1;
    pre_ls[j] = 0.0f;
    if (c < nstage) {
      const int32_t id = id_of(c);
      // out-of-range ids are never dereferenced, nor ids of another shard
      if (id >= 0 && id < V && id >= v0 && id - v0 < Vs) {
        pre_id[j] = id;
        pre_ls[j] = __ldg(lm_scale + (id - v0));
        const int8_t* wr = W + static_cast<int64_t>(id - v0) * ldw;
        const uint32_t dst = smem_u32(srow + static_cast<int64_t>(c) * K);
        for (int64_t ch = lane; ch < nchunk; ch += 32) cp_async_16(dst + static_cast<uint32_t>(ch * 16), wr + ch * 16, 16);
      }
    }
  }
  cp_async_commit();
  // warp 0 validates: offsets, count, every id in range, no id twice
  if (warp == 0) {
    unsigned bad = 0u;
    if (!off_ok) {
      bad = PRISM_DEV_ERR_OFFSETS;
    } else if (!cnt_ok) {
      bad = PRISM_DEV_ERR_COUNT;
    } else {
      const bool has_l = lane < cnt, has_h = lane + 32 < cnt;
      if ((has_l && (id_l < 0 || id_l >= V)) || (has_h && (id_h < 0 || id_h >= V))) bad |= PRISM_DEV_ERR_ID_RANGE;
      for (int64_t i = 0; i < cnt; ++i) {
        const int32_t o = id_of(i);
        if ((has_l && i < lane && o == id_l) || (has_h && i < lane + 32 && o == id_h)) bad |= PRISM_DEV_ERR_DUPLICATE;
      }
    }
    bad = __reduce_or_sync(0xffffffffu, bad);
    if (lane == 0) s_bad = bad;
  }
  __syncthreads();
  if (s_bad) {
    cp_async_wait<0>();   // no copy may land in shared memory after the CTA is gone
    if (tid == 0 && err != nullptr) atomicOr(err, s_bad);
    if (off_ok) {
      const float nan = __uint_as_float(0x7fc00000u);
      for (int64_t i = b + tid; i < e; i += kThreads) {
        logits[i] = nan;
        if (!kLogits) probs[i] = nan;
      }
    }
    return;
  }

  // ---- 2. quantise the hidden row into shared memory
  float amax = 0.0f;
  if (kReg) {
#pragma unroll
    for (int i = 0; i < kHidVec; ++i) {
      const int64_t k = (static_cast<int64_t>(tid) + static_cast<int64_t>(i) * kThreads) * 8;
      if (k < K) {
        const uint32_t w4[4] = {hv[i].x, hv[i].y, hv[i].z, hv[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          amax = fmaxf(amax, fabsf(smooth(bf16_lo(w4[j]), inv_s, k + 2 * j)));
          amax = fmaxf(amax, fabsf(smooth(bf16_hi(w4[j]), inv_s, k + 2 * j + 1)));
        }
      }
    }
  } else {
    for (int64_t k = static_cast<int64_t>(tid) * 8; k < K; k += kThreads * 8) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(hr + k));
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        amax = fmaxf(amax, fabsf(smooth(bf16_lo(w4[i]), inv_s, k + 2 * i)));
        amax = fmaxf(amax, fabsf(smooth(bf16_hi(w4[i]), inv_s, k + 2 * i + 1)));
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) s_red[warp] = amax;
  __syncthreads();
  amax = s_red[0];
#pragma unroll
  for (int i = 1; i < kWarps; ++i) amax = fmaxf(amax, s_red[i]);
  const bool zero_row = !(amax >= 0x1p-120f);
  const float inv_a = zero_row ? 0.0f : __fdiv_rn(127.0f, amax);
  const float a_scale = zero_row ? 0.0f : __fdiv_rn(amax, 127.0f);
  auto quant8 = [&](const uint4 v, int64_t k) {
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
    uint32_t packed[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int q0 = max(-127, min(127, __float2int_rn(__fmul_rn(smooth(bf16_lo(w4[i]), inv_s, k + 2 * i), inv_a))));
      const int q1 = max(-127, min(127, __float2int_rn(__fmul_rn(smooth(bf16_hi(w4[i]), inv_s, k + 2 * i + 1), inv_a))));
      const uint32_t two = (static_cast<uint32_t>(q0) & 0xffu) | ((static_cast<uint32_t>(q1) & 0xffu) << 8);
      packed[i >> 1] |= two << (16 * (i & 1));
    }
    *reinterpret_cast<uint2*>(sq + k) = make_uint2(packed[0], packed[1]);
  };
  if (kReg) {
#pragma unroll
    for (int i = 0; i < kHidVec; ++i) {
      const int64_t k = (static_cast<int64_t>(tid) + static_cast<int64_t>(i) * kThreads) * 8;
      if (k < K) quant8(hv[i], k);
    }
  } else {
    for (int64_t k = static_cast<int64_t>(tid) * 8; k < K; k += kThreads * 8)
      quant8(__ldg(reinterpret_cast<const uint4*>(hr + k)), k);
  }
  cp_async_wait<0>();
  __syncthreads();   // the quantised row and every staged candidate row are visible

  // ---- 3. one warp per candidate: exact int32 dot against the gathered row
  for (int64_t i = warp; i < cnt; i += kWarps) {
    int acc = 0;
    int32_t id;
    float ls;
    if (kLogits) {
      const int32_t ic = id_of(i);
      if (ic < v0 || ic - v0 >= Vs) {   // another shard's candidate
        if (lane == 0) s_logit[i] = -0.0f;
        continue;
      }
    }
    if (i < nstage) {
      const int j = static_cast<int>(i) / kWarps;
      id = pre_id[0];
#pragma unroll
      for (int jj = 1; jj < kPrePerWarp; ++jj)
        if (j == jj) id = pre_id[jj];
      ls = pre_ls[0];
#pragma unroll
      for (int jj = 1; jj < kPrePerWarp; ++jj)
        if (j == jj) ls = pre_ls[jj];
      const int8_t* rs = srow + i * K;
      for (int64_t c = lane; c < nchunk; c += 32)
        acc = dot16(*reinterpret_cast<const uint4*>(rs + c * 16), *reinterpret_cast<const uint4*>(sq + c * 16), acc);
    } else {
      id = id_of(i);
      ls = __ldg(lm_scale + (id - v0));
      const int8_t* wr = W + static_cast<int64_t>(id - v0) * ldw;
      int64_t c = lane;
      for (; c + 32 * 3 < nchunk; c += 32 * 4) {
        const uint4 w0 = ld_stream_16(wr + (c)*16);
        const uint4 w1 = ld_stream_16(wr + (c + 32) * 16);
        const uint4 w2 = ld_stream_16(wr + (c + 64) * 16);
        const uint4 w3 = ld_stream_16(wr + (c + 96) * 16);
        acc = dot16(w0, *reinterpret_cast<const uint4*>(sq + c * 16), acc);
        acc = dot16(w1, *reinterpret_cast<const uint4*>(sq + (c + 32) * 16), acc);
        acc = dot16(w2, *reinterpret_cast<const uint4*>(sq + (c + 64) * 16), acc);
        acc = dot16(w3, *reinterpret_cast<const uint4*>(sq + (c + 96) * 16), acc);
      }
      for (; c < nchunk; c += 32)
        acc = dot16(ld_stream_16(wr + c * 16), *reinterpret_cast<const uint4*>(sq + c * 16), acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) {
      float t = __int2float_rn(acc);
      t = __fmul_rn(t, a_scale);
      t = __fmul_rn(t, ls);
      s_logit[i] = t;
    }
  }
  __syncthreads();

  // ---- 4. softmax over the candidates in warp 0 (candidate_softmax), or
  // for a shard its logits only
  if (warp == 0) {
    const float l0 = lane < cnt ? s_logit[lane] : -INFINITY;
    const float l1 = lane + 32 < cnt ? s_logit[lane + 32] : -INFINITY;
    if (lane < cnt) logits[b + lane] = l0;
    if (lane + 32 < cnt) logits[b + lane + 32] = l1;
    if (!kLogits) {
      float p0, p1;
      candidate_softmax(l0, l1, cnt, lane, p0, p1);
      if (lane < cnt) probs[b + lane] = p0;
      if (lane + 32 < cnt) probs[b + lane + 32] = p1;
    }
  }
}

// The softmax of step 4 on logits combined from the vocabulary shards: one
// warp per position checks the CSR slice like the read-out (bad offsets or
// count: the error bit, NaN probabilities) and treats a position with a NaN
// logit (a shard found its list invalid and said so in the error word) as
// invalid too; the others get candidate_softmax, bit for bit the fused
// read-out's probabilities.
__global__ void __launch_bounds__(128)
    softmax_kernel(const float* __restrict__ logits, const int32_t* __restrict__ off, int64_t P, int64_t T,
                   float* __restrict__ probs, uint32_t* __restrict__ err) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t p = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  if (p >= P) return;
  const int64_t b = off[p], e = off[p + 1];
  const bool off_ok = b >= 0 && e <= T && b <= e;
  const int64_t cnt = off_ok ? e - b : 0;
  const bool cnt_ok = off_ok && cnt >= 1 && cnt <= PRISM_MAX_CANDIDATES;
  const float l0 = cnt_ok && lane < cnt ? logits[b + lane] : -INFINITY;
  const float l1 = cnt_ok && lane + 32 < cnt ? logits[b + lane + 32] : -INFINITY;
  const bool has_nan = __any_sync(0xffffffffu, l0 != l0 || l1 != l1);
  if (!cnt_ok || has_nan) {
    if (lane == 0 && err != nullptr && !cnt_ok) atomicOr(err, off_ok ? PRISM_DEV_ERR_COUNT : PRISM_DEV_ERR_OFFSETS);
    if (off_ok) {
      const float nan = __uint_as_float(0x7fc00000u);
      for (int64_t i = b + lane; i < e; i += 32) probs[i] = nan;
    }
    return;
  }
  float p0, p1;
  candidate_softmax(l0, l1, cnt, lane, p0, p1);
  if (lane < cnt) probs[b + lane] = p0;
  if (lane + 32 < cnt) probs[b + lane + 32] = p1;
}

}  // namespace

namespace {
template <bool kLogits>
cudaError_t launch_readout_impl(const void* h, int64_t ldh, const float* inv_s, const int8_t* W, int64_t ldw,
                                const float* lm_scale, int64_t V, int64_t v0, int64_t Vs, int64_t K,
                                const int32_t* off, const int32_t* ids, int64_t P, int64_t T, float* logits,
                                float* probs, uint32_t* err, cudaStream_t stream) {
  // staged rows: as many as fit beside the quantised row in kSmemBudget, at most kPreMax
  const int64_t fit = K < kSmemBudget ? (kSmemBudget - K) / K : 0;
  const int pre = static_cast<int>(std::min<int64_t>(kPreMax, fit));
  const size_t smem = static_cast<size_t>(K) * static_cast<size_t>(1 + pre);
  if (K <= kRegK) {
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(readout_kernel<true, kLogits>), kSmemBudget);
    if (e != cudaSuccess) return e;
    return launch_kernel(readout_kernel<true, kLogits>, dim3(static_cast<unsigned>(P)), dim3(kThreads), smem,
                         stream, true, static_cast<const uint16_t*>(h), ldh, inv_s, W, ldw, lm_scale, V, v0, Vs, K,
                         off, ids, T, logits, probs, err, pre);
  }
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(readout_kernel<false, kLogits>),
                                   std::max<int>(kSmemBudget, PRISM_MAX_READOUT_K));
  if (e != cudaSuccess) return e;
  return launch_kernel(readout_kernel<false, kLogits>, dim3(static_cast<unsigned>(P)), dim3(kThreads), smem, stream,
                       true, static_cast<const uint16_t*>(h), ldh, inv_s, W, ldw, lm_scale, V, v0, Vs, K, off, ids,
                       T, logits, probs, err, pre);
}
}  // namespace

cudaError_t launch_readout(const void* h, int64_t ldh, const float* inv_s, const int8_t* W,
                           int64_t ldw, const float* lm_scale, int64_t V, int64_t K,
                           const int32_t* off, const int32_t* ids, int64_t P, int64_t T,
                           float* logits, float* probs, uint32_t* err, cudaStream_t stream) {
  return launch_readout_impl<false>(h, ldh, inv_s, W, ldw, lm_scale, V, 0, V, K, off, ids, P, T, logits, probs, err,
                                    stream);
}

cudaError_t launch_readout_logits(const void* h, int64_t ldh, const float* inv_s, const int8_t* W_shard,
                                  int64_t ldw, const float* lm_scale_shard, int64_t v0, int64_t Vs, int64_t V,
                                  int64_t K, const int32_t* off, const int32_t* ids, int64_t P, int64_t T,
                                  float* logits, uint32_t* err, cudaStream_t stream) {
  return launch_readout_impl<true>(h, ldh, inv_s, W_shard, ldw, lm_scale_shard, V, v0, Vs, K, off, ids, P, T, logits,
                                   nullptr, err, stream);
}

cudaError_t launch_candidate_softmax(const float* logits, const int32_t* off, int64_t P, int64_t T, float* probs,
                                     uint32_t* err, cudaStream_t stream) {
  return launch_kernel(softmax_kernel, dim3(static_cast<unsigned>((P + 3) / 4)), dim3(128), 0, stream, true, logits,
                       off, P, T, probs, err);
}

}  // namespace prism
