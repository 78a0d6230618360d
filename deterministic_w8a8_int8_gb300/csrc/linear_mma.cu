// linear_mma.cu -- W8A8 linear on the warp-level int8 tensor-core path.
//
// acc[m,n] = sum_k q[m,k] * w[n,k] in exact int32 (mma.sync m16n8k32 s8*s8->s32),
// then y = bf16_rne(((float(acc) * a_scale[m]) * w_scale[n]) + residual[m,n])
// (StartLux-Prism, "Bitwise consistency is not lossless quantization").
//
// Tiling: a CTA computes a 128x128 output tile with 8 warps (2 x 4, 64x32
// each) over K-tiles of 64 bytes, staged through a 4-deep cp.async ring in
// shared memory (16-byte chunks XOR-swizzled by row pair so every ldmatrix
// phase touches 32 distinct banks).  Rows beyond M or N and chunks beyond K
// are zero-filled by the copy itself, so ragged edges need no extra branches
// in the main loop.
//
// Split-K (grid.z > 1): each CTA owns a contiguous range of K-tiles, adds its
// int32 partial tile into a workspace accumulator with integer atomics (exact
// and order-free), then bumps the tile's arrival counter.  The CTA that
// arrives last reads the complete integer sum, applies the epilogue, and
// returns the workspace tile and counter to zero for the next call.  No CTA
// ever waits for another, so there is no spin and no possible deadlock.
#include <algorithm>

#include "common.cuh"

namespace prism {
namespace {

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kBK = 64;  // bytes of K per stage
constexpr int kStages = 4;
constexpr int kThreads = 256;
constexpr int kStageA = kBM * kBK;
constexpr int kStageB = kBN * kBK;
constexpr int kSmemBytes = kStages * (kStageA + kStageB);

// byte offset of 16-byte chunk c (0..3) of row r inside a [rows][64 B] tile
__device__ __forceinline__ int swz(int r, int c) { return r * kBK + ((c ^ ((r >> 1) & 3)) << 4); }

__device__ __forceinline__ void store_pair(const LinearArgs& a, int64_t row, int64_t col, int32_t v0,
                                           int32_t v1) {
  const bool two = col + 1 < a.N;
  if (a.acc_only) {   // a tensor-parallel partial: the exact accumulators only
    int32_t* cp = a.acc_out + row * a.N + col;
    cp[0] = v0;
    if (two) cp[1] = v1;
    return;
  }
  const float as = __ldg(a.a_scale + row);
  if (!a.pair_io) {  // odd row strides or 2-byte-aligned bases: element stores
    const float as1 = __ldg(a.a_scale + row);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      if (e == 1 && !two) break;
      const int32_t v = e ? v1 : v0;
      const float ws1 = __ldg(a.w_scale + col + e);
      uint32_t o;
      if (a.residual != nullptr) {
        const uint16_t* rp = residual_row(a, row);
        o = epilogue_bf16_res(v, as1, ws1, bf16_bits_to_float(rp != nullptr ? rp[col + e] : kBf16NaN));
      } else {
        o = epilogue_bf16(v, as1, ws1);
      }
      a.out[row * a.ldo + col + e] = static_cast<uint16_t>(o);
      if (a.acc_out != nullptr) a.acc_out[row * a.N + col + e] = v;
    }
    return;
  }
  const float w0 = __ldg(a.w_scale + col);
  const float w1 = two ? __ldg(a.w_scale + col + 1) : 0.0f;
  uint32_t o0, o1 = 0;
  const uint16_t* rrow = a.residual != nullptr ? residual_row(a, row) : nullptr;
  if (a.residual != nullptr && rrow == nullptr) {
    o0 = epilogue_bf16_res(v0, as, w0, bf16_bits_to_float(kBf16NaN));
    if (two) o1 = epilogue_bf16_res(v1, as, w1, bf16_bits_to_float(kBf16NaN));
  } else if (a.residual != nullptr) {
    const uint16_t* rp = rrow + col;
    if (two) {
      const uint32_t rr = *reinterpret_cast<const uint32_t*>(rp);
      o0 = epilogue_bf16_res(v0, as, w0, bf16_lo(rr));
      o1 = epilogue_bf16_res(v1, as, w1, bf16_hi(rr));
    } else {
      o0 = epilogue_bf16_res(v0, as, w0, bf16_bits_to_float(*rp));
    }
  } else {
    o0 = epilogue_bf16(v0, as, w0);
    if (two) o1 = epilogue_bf16(v1, as, w1);
  }
  uint16_t* op = a.out + row * a.ldo + col;
  if (two) {
    *reinterpret_cast<uint32_t*>(op) = o0 | (o1 << 16);
  } else {
    *op = static_cast<uint16_t>(o0);
  }
  if (a.acc_out != nullptr) {
    int32_t* cp = a.acc_out + row * a.N + col;
    cp[0] = v0;
    if (two) cp[1] = v1;
  }
}

__global__ void __launch_bounds__(kThreads, 2) linear_mma_kernel(const LinearArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kStageA;
  __shared__ int s_last;
  pdl_trigger();
  pdl_wait();

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int wm = warp >> 2;  // 0..1
  const int wn = warp & 3;   // 0..3
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * kBM;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kBN;
  const int64_t ktiles = (a.K + kBK - 1) / kBK;
  const int64_t per = (ktiles + a.split - 1) / a.split;
  const int64_t kt0 = static_cast<int64_t>(blockIdx.z) * per;
  const int64_t kt1 = min(ktiles, kt0 + per);
  const int nk = kt1 > kt0 ? static_cast<int>(kt1 - kt0) : 0;

  auto load_stage = [&](int stage, int64_t kt) {
    const int64_t kb = kt * kBK;
#pragma unroll
    for (int i = 0; i < (kBM * kBK / 16) / kThreads; ++i) {
      const int id = tid + i * kThreads;
      const int r = id >> 2, c = id & 3;
      const int64_t gm = m0 + r, gk = kb + c * 16;
      const bool ok = gm < a.M && gk < a.K;
      cp_async_16(smem_u32(sA + stage * kStageA + swz(r, c)), ok ? a.q + gm * a.ldq + gk : a.q,
                  ok ? 16 : 0);
    }
#pragma unroll
    for (int i = 0; i < (kBN * kBK / 16) / kThreads; ++i) {
      const int id = tid + i * kThreads;
      const int r = id >> 2, c = id & 3;
      const int64_t gn = n0 + r, gk = kb + c * 16;
      const bool ok = gn < a.N && gk < a.K;
      cp_async_16(smem_u32(sB + stage * kStageB + swz(r, c)), ok ? a.w + gn * a.ldw + gk : a.w,
                  ok ? 16 : 0);
    }
  };

  int32_t acc[4][4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][j][e] = 0;

#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < nk) load_stage(s, kt0 + s);
    cp_async_commit();
  }

  for (int it = 0; it < nk; ++it) {
    cp_async_wait<kStages - 2>();
    __syncthreads();
    const int nxt = it + kStages - 1;
    if (nxt < nk) load_stage(nxt % kStages, kt0 + nxt);
    cp_async_commit();

    const uint8_t* tA = sA + (it % kStages) * kStageA;
    const uint8_t* tB = sB + (it % kStages) * kStageB;
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      uint32_t af[4][4];
      uint32_t bfr[4][2];
#pragma unroll
      for (int mi = 0; mi < 4; ++mi) {
        const int row = wm * 64 + mi * 16 + (lane & 15);
        const int ch = ks * 2 + (lane >> 4);
        ldmatrix_x4(smem_u32(tA + swz(row, ch)), af[mi][0], af[mi][1], af[mi][2], af[mi][3]);
      }
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        const int row = wn * 32 + p * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int ch = ks * 2 + ((lane >> 3) & 1);
        ldmatrix_x4(smem_u32(tB + swz(row, ch)), bfr[2 * p][0], bfr[2 * p][1], bfr[2 * p + 1][0],
                    bfr[2 * p + 1][1]);
      }
#pragma unroll
      for (int mi = 0; mi < 4; ++mi)
#pragma unroll
        for (int nj = 0; nj < 4; ++nj) mma_s8_16832(acc[mi][nj], af[mi], bfr[nj][0], bfr[nj][1]);
    }
  }
  cp_async_wait<0>();

  const int gid = lane >> 2, tig = lane & 3;
  if (a.split == 1) {
#pragma unroll
    for (int mi = 0; mi < 4; ++mi)
#pragma unroll
      for (int nj = 0; nj < 4; ++nj)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int64_t row = m0 + wm * 64 + mi * 16 + gid + h * 8;
          const int64_t col = n0 + wn * 32 + nj * 8 + tig * 2;
          if (row < a.M && col < a.N) store_pair(a, row, col, acc[mi][nj][2 * h], acc[mi][nj][2 * h + 1]);
        }
    return;
  }

  // ---- split-K: integer partials into the workspace, last arriver finishes
#pragma unroll
  for (int mi = 0; mi < 4; ++mi)
#pragma unroll
    for (int nj = 0; nj < 4; ++nj)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t row = m0 + wm * 64 + mi * 16 + gid + h * 8;
        const int64_t col = n0 + wn * 32 + nj * 8 + tig * 2;
        if (row < a.M && col < a.N) {
          int32_t* p = a.ws_acc + row * a.N + col;
          atomicAdd(p, acc[mi][nj][2 * h]);
          if (col + 1 < a.N) atomicAdd(p + 1, acc[mi][nj][2 * h + 1]);
        }
      }
  __threadfence();
  __syncthreads();
  const unsigned tile = blockIdx.y * gridDim.x + blockIdx.x;
  if (tid == 0) s_last = (atomicAdd(a.ws_count + tile, 1u) == static_cast<unsigned>(a.split - 1));
  __syncthreads();
  if (!s_last) return;
  __threadfence();
#pragma unroll
  for (int mi = 0; mi < 4; ++mi)
#pragma unroll
    for (int nj = 0; nj < 4; ++nj)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t row = m0 + wm * 64 + mi * 16 + gid + h * 8;
        const int64_t col = n0 + wn * 32 + nj * 8 + tig * 2;
        if (row < a.M && col < a.N) {
          int32_t* p = a.ws_acc + row * a.N + col;
          const bool two = col + 1 < a.N;
          const int32_t v0 = __ldcg(p);
          const int32_t v1 = two ? __ldcg(p + 1) : 0;
          __stcg(p, 0);
          if (two) __stcg(p + 1, 0);
          store_pair(a, row, col, v0, v1);
        }
      }
  if (tid == 0) a.ws_count[tile] = 0u;
}

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

int mma_auto_split(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0) return 1;
  const int64_t tiles = cdiv(M, kBM) * cdiv(N, kBN);
  const int64_t ktiles = cdiv(K, kBK);
  const int64_t want = 2 * 152;  // two resident CTAs on each of the 152 SMs
  int64_t s = cdiv(want, tiles);
  s = std::min<int64_t>(s, std::max<int64_t>(1, ktiles / 4));
  s = std::min<int64_t>(s, 16);
  return static_cast<int>(std::max<int64_t>(1, s));
}

cudaError_t launch_linear_mma(const LinearArgs& a, cudaStream_t stream) {
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(linear_mma_kernel), kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>(cdiv(a.N, kBN)), static_cast<unsigned>(cdiv(a.M, kBM)),
            static_cast<unsigned>(a.split));
  return launch_kernel(linear_mma_kernel, grid, dim3(kThreads), kSmemBytes, stream, a.no_pdl == 0, a);
}

}  // namespace prism
