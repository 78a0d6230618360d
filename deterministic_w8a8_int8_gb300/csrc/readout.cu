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
//   4. one thread forms the softmax in list order: e_c = exp(logit_c - max),
//      s = e_1 + ... + e_n, prob_c = e_c / s, every step binary32 RN.
// Bytes: 2K (hidden row) + count * (K + 4) (candidate rows and scales) per
// position, plus 12 bytes per candidate (id, logit, prob) -- HBM- and
// latency-bound; nothing is written to global memory but the outputs.  For K
// up to 8192 each warp starts streaming its first candidate row right after
// the offsets are checked (the id is range-checked first), and the hidden
// row is read once into registers.
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

// Hidden rows of up to kRegK elements are read once into registers; the
// first 5 KB of each warp's first candidate row (all of a 5120-wide row) are
// fetched into registers as soon as its id is known to be in range, so that
// their memory latency overlaps the quantisation of the hidden row (any rest
// of a longer row is read when the dot product reaches it).  Two CTAs fit on an SM (at most 128
// registers), so 192 answer positions run in one wave on 152 SMs.
constexpr int kRegK = 8192;
constexpr int kHidVec = kRegK / 8 / kThreads;   // uint4 (8 bf16) per thread: 4
constexpr int kRowVec = 10;                     // uint4 (16 int8) per lane: 5 KB of the row per warp

template <bool kReg>
__global__ void __launch_bounds__(kThreads, 2)
    readout_kernel(const uint16_t* __restrict__ h, int64_t ldh, const float* __restrict__ inv_s,
                   const int8_t* __restrict__ W, int64_t ldw, const float* __restrict__ lm_scale,
                   int64_t V, int64_t K, const int32_t* __restrict__ off,
                   const int32_t* __restrict__ ids, int64_t T, float* __restrict__ logits,
                   float* __restrict__ probs, uint32_t* __restrict__ err) {
  extern __shared__ __align__(16) int8_t sq[];
  pdl_trigger();
  pdl_wait();
  __shared__ float s_logit[PRISM_MAX_CANDIDATES];
  __shared__ float s_prob[PRISM_MAX_CANDIDATES];
  __shared__ float s_red[kWarps];
  __shared__ unsigned s_bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t p = blockIdx.x;
  const int64_t nchunk = K >> 4;   // 16-byte chunks of a row

  // ---- 1. validate this position's candidate list
  if (tid == 0) s_bad = 0u;
  __syncthreads();
  const int64_t b = off[p], e = off[p + 1];
  const bool off_ok = b >= 0 && e <= T && b <= e;
  const int64_t cnt = off_ok ? e - b : 0;
  const bool cnt_ok = off_ok && cnt >= 1 && cnt <= PRISM_MAX_CANDIDATES;
  // this warp's first candidate row, fetched early when its id is in range
  uint4 row[kReg ? kRowVec : 1];
  int32_t id0 = -1;
  if (kReg && cnt_ok && warp < cnt) {
    const int32_t id = ids[b + warp];
    if (id >= 0 && id < V) {
      id0 = id;
      const int8_t* wr = W + static_cast<int64_t>(id) * ldw;
#pragma unroll
      for (int i = 0; i < kRowVec; ++i) {
        const int64_t c = lane + 32 * i;
        row[i] = c < nchunk ? ld_stream_16(wr + c * 16) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }
  unsigned bad = 0u;
  if (!off_ok) {
    bad = PRISM_DEV_ERR_OFFSETS;
  } else if (!cnt_ok) {
    bad = PRISM_DEV_ERR_COUNT;
  } else if (tid < cnt) {
    const int32_t id = ids[b + tid];
    if (id < 0 || id >= V) bad |= PRISM_DEV_ERR_ID_RANGE;
    for (int j = 0; j < tid; ++j)
      if (ids[b + j] == id) bad |= PRISM_DEV_ERR_DUPLICATE;
  }
  if (bad) atomicOr(&s_bad, bad);
  __syncthreads();
  if (s_bad) {
    if (tid == 0 && err != nullptr) atomicOr(err, s_bad);
    if (off_ok) {
      const float nan = __uint_as_float(0x7fc00000u);
      for (int64_t i = b + tid; i < e; i += kThreads) {
        logits[i] = nan;
        probs[i] = nan;
      }
    }
    return;
  }

  // ---- 2. quantise the hidden row into shared memory
  const uint16_t* hr = h + p * ldh;
  uint4 hv[kReg ? kHidVec : 1];
  float amax = 0.0f;
  if (kReg) {
#pragma unroll
    for (int i = 0; i < kHidVec; ++i) {
      const int64_t k = (static_cast<int64_t>(tid) + static_cast<int64_t>(i) * kThreads) * 8;
      hv[i] = k < K ? __ldg(reinterpret_cast<const uint4*>(hr + k)) : make_uint4(0u, 0u, 0u, 0u);
    }
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
  __syncthreads();

  // ---- 3. one warp per candidate: exact int32 dot against the gathered row
  for (int64_t i = warp; i < cnt; i += kWarps) {
    const int32_t id = ids[b + i];
    const int8_t* wr = W + static_cast<int64_t>(id) * ldw;
    int acc = 0;
    if (kReg && i == warp && id == id0) {
#pragma unroll
      for (int j = 0; j < kRowVec; ++j) {
        const int64_t c = lane + 32 * j;
        if (c < nchunk) acc = dot16(row[j], *reinterpret_cast<const uint4*>(sq + c * 16), acc);
      }
      for (int64_t c = lane + 32 * kRowVec; c < nchunk; c += 32)
        acc = dot16(ld_stream_16(wr + c * 16), *reinterpret_cast<const uint4*>(sq + c * 16), acc);
    } else {
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
      t = __fmul_rn(t, __ldg(lm_scale + id));
      s_logit[i] = t;
    }
  }
  __syncthreads();

  // ---- 4. softmax over the candidates, fixed order
  if (tid == 0) {
    float mx = s_logit[0];
    for (int i = 1; i < cnt; ++i) mx = fmaxf(mx, s_logit[i]);
    float s = 0.0f;
    for (int i = 0; i < cnt; ++i) {
      const float ev = cw_exp(__fsub_rn(s_logit[i], mx));
      s_prob[i] = ev;
      s = __fadd_rn(s, ev);
    }
    for (int i = 0; i < cnt; ++i) s_prob[i] = __fdiv_rn(s_prob[i], s);
  }
  __syncthreads();
  if (tid < cnt) {
    logits[b + tid] = s_logit[tid];
    probs[b + tid] = s_prob[tid];
  }
}

}  // namespace

cudaError_t launch_readout(const void* h, int64_t ldh, const float* inv_s, const int8_t* W,
                           int64_t ldw, const float* lm_scale, int64_t V, int64_t K,
                           const int32_t* off, const int32_t* ids, int64_t P, int64_t T,
                           float* logits, float* probs, uint32_t* err, cudaStream_t stream) {
  const int smem = static_cast<int>((K + 15) & ~static_cast<int64_t>(15));
  if (K <= kRegK) {
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(readout_kernel<true>), kRegK);
    if (e != cudaSuccess) return e;
    return launch_kernel(readout_kernel<true>, dim3(static_cast<unsigned>(P)), dim3(kThreads),
                         static_cast<size_t>(smem), stream, true, static_cast<const uint16_t*>(h), ldh, inv_s, W, ldw,
                         lm_scale, V, K, off, ids, T, logits, probs, err);
  }
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(readout_kernel<false>), PRISM_MAX_READOUT_K);
  if (e != cudaSuccess) return e;
  return launch_kernel(readout_kernel<false>, dim3(static_cast<unsigned>(P)), dim3(kThreads),
                       static_cast<size_t>(smem), stream, true, static_cast<const uint16_t*>(h), ldh, inv_s, W, ldw,
                       lm_scale, V, K, off, ids, T, logits, probs, err);
}

}  // namespace prism
