// linear_gemv.cu -- the W8A8 linear for a few token rows (M <= 8): decode
// steps and the last layer restricted to answer positions (StartLux-Prism,
// "Bitwise consistency is not lossless quantization": int8 products
// accumulate exactly in int32, then a fixed fp32 epilogue).
//
// With so few rows the layer is a weight stream: every weight byte is used M
// times, far below the tensor cores' break-even, and the tcgen05 kernel's
// per-stage widening of 128 weight rows to f16 would set its speed.  Here S
// warps of a CTA own a group of R output channels, each warp a contiguous
// 1/S of K: each lane streams 16-byte chunks of the R weight rows (U chunks
// per row in flight, non-allocating loads), reads the matching 16 bytes of
// each token row through L1 (all warps share them), and accumulates with
// dp4a -- exact int32, so the sum does not depend on how K is split.  Warp
// reductions (redux.sync) and a shared-memory sum over the S warps give each
// channel's exact accumulator; lane m * R + r of the first warp applies the
// epilogue of token m, channel r.  Bit-identical to the other contraction
// kernels.
#include "common.cuh"

namespace prism {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

__device__ __forceinline__ int dp4a_16(const uint4& a, const uint4& b, int c) {
  c = __dp4a(static_cast<int>(a.x), static_cast<int>(b.x), c);
  c = __dp4a(static_cast<int>(a.y), static_cast<int>(b.y), c);
  c = __dp4a(static_cast<int>(a.z), static_cast<int>(b.z), c);
  return __dp4a(static_cast<int>(a.w), static_cast<int>(b.w), c);
}

// 4-bit weights (W4A8): 16 packed bytes hold codes 0..31 of a K-range, code
// 2j in the low nibble of byte j.  Unpacked in registers as 16 * code, an
// exact int8 byte (16 * [-8, 7] = [-128, 112]), in k order: for each word,
// lo = (w << 4) & 0xF0F0F0F0 holds the even codes, hi = w & 0xF0F0F0F0 the
// odd ones, and two byte permutes interleave them.  The dp4a sums are then
// 16 times the true ones; each lane shifts its partial right by 4 (exact: a
// multiple of 16) before the warp reduction, so the total stays within int32.
__device__ __forceinline__ void unpack_w4x16(const uint4& p, uint4& a, uint4& b) {
  auto two = [](uint32_t w, uint32_t& o0, uint32_t& o1) {
    const uint32_t lo = (w << 4) & 0xF0F0F0F0u, hi = w & 0xF0F0F0F0u;
    o0 = __byte_perm(lo, hi, 0x5140u);
    o1 = __byte_perm(lo, hi, 0x7362u);
  };
  two(p.x, a.x, a.y);
  two(p.y, a.z, a.w);
  two(p.z, b.x, b.y);
  two(p.w, b.z, b.w);
}

// MB: token rows rounded up (rows m >= M stay zero and are not written).
// kMode: 0 plain; 1 residual rows through a.res_rows (see residual_row); 2
// only the exact int32 accumulators, into acc_out.
// R: output channels per group; U: 16-byte chunks per channel in flight per
// lane; S: warps sharing one group, each over a contiguous 1/S of K (their
// exact partial sums are added through shared memory).
template <int MB, int kMode, int R, int U, int S, bool kW4 = false>
__global__ void __launch_bounds__(kThreads)
    linear_gemv_kernel(const __grid_constant__ LinearArgs a) {
  static_assert(MB * R <= 32 && kWarps % S == 0, "shape");
  __shared__ int part[kWarps][32];
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int slice = warp % S;
  const int64_t n0 = (static_cast<int64_t>(blockIdx.x) * (kWarps / S) + warp / S) * R;
  const bool live = n0 < a.N;
  const int M = static_cast<int>(a.M);
  const int nch = static_cast<int>(kW4 ? a.K >> 5 : a.K >> 4);   // 16-byte weight chunks per row
  const int c_begin = static_cast<int>(static_cast<int64_t>(nch) * slice / S);
  const int c_end = static_cast<int>(static_cast<int64_t>(nch) * (slice + 1) / S);
  const int8_t* wrow[R];
#pragma unroll
  for (int r = 0; r < R; ++r) wrow[r] = a.w + (live && n0 + r < a.N ? n0 + r : 0) * a.ldw;

  int acc[MB][R];
#pragma unroll
  for (int m = 0; m < MB; ++m)
#pragma unroll
    for (int r = 0; r < R; ++r) acc[m][r] = 0;

  if (live) {
    for (int c0 = c_begin; c0 < c_end; c0 += 32 * U) {
      uint4 wv[U][R];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + u * 32 + lane;
#pragma unroll
        for (int r = 0; r < R; ++r)
          wv[u][r] = c < c_end && n0 + r < a.N ? ld_stream_16(wrow[r] + 16 * static_cast<int64_t>(c))
                                               : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c >= c_end) break;
        if constexpr (kW4) {
          uint4 wa[R], wb[R];
#pragma unroll
          for (int r = 0; r < R; ++r) unpack_w4x16(wv[u][r], wa[r], wb[r]);
#pragma unroll
          for (int m = 0; m < MB; ++m) {
            if (m < M) {
              const uint4* qp = reinterpret_cast<const uint4*>(a.q + m * a.ldq) + 2 * static_cast<int64_t>(c);
              const uint4 qa = __ldg(qp), qb = __ldg(qp + 1);
#pragma unroll
              for (int r = 0; r < R; ++r) acc[m][r] = dp4a_16(qb, wb[r], dp4a_16(qa, wa[r], acc[m][r]));
            }
          }
        } else {
#pragma unroll
          for (int m = 0; m < MB; ++m) {
            if (m < M) {
              const uint4 qv = __ldg(reinterpret_cast<const uint4*>(a.q + m * a.ldq) + c);
#pragma unroll
              for (int r = 0; r < R; ++r) acc[m][r] = dp4a_16(qv, wv[u][r], acc[m][r]);
            }
          }
        }
      }
    }
  }
  if constexpr (kW4) {
#pragma unroll
    for (int m = 0; m < MB; ++m)
#pragma unroll
      for (int r = 0; r < R; ++r) acc[m][r] >>= 4;   // exact: every product was 16 times the true one
  }

  // exact int32 sums over the warp; lane m * R + r keeps (token m, channel r)
  int mine = 0;
#pragma unroll
  for (int m = 0; m < MB; ++m)
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int s = __reduce_add_sync(0xffffffffu, acc[m][r]);
      if (lane == m * R + r) mine = s;
    }
  if constexpr (S > 1) {
    part[warp][lane] = mine;
    __syncthreads();
    if (slice != 0) return;
#pragma unroll
    for (int j = 1; j < S; ++j) mine += part[warp + j][lane];
  }
  const int m = lane / R, r = lane % R;
  const int64_t n = n0 + r;
  if (!live || m >= MB || m >= M || n >= a.N) return;
  if constexpr (kMode == 2) {
    a.acc_out[m * a.N + n] = mine;
    return;
  }
  const float as = __ldg(a.a_scale + m), ws = __ldg(a.w_scale + n);
  uint32_t o;
  if (a.residual != nullptr) {
    uint16_t rv;
    if constexpr (kMode == 1) {
      const uint16_t* rp = residual_row(a, m);
      rv = rp != nullptr ? rp[n] : static_cast<uint16_t>(kBf16NaN);
    } else {
      rv = a.residual[m * a.ldr + n];
    }
    o = epilogue_bf16_res(mine, as, ws, bf16_bits_to_float(rv));
  } else {
    o = epilogue_bf16(mine, as, ws);
  }
  a.out[m * a.ldo + n] = static_cast<uint16_t>(o);
  if (a.acc_out != nullptr) a.acc_out[m * a.N + n] = mine;
}

template <int MB, int R, int U, int S>
cudaError_t launch_mb_w4(const LinearArgs& a, cudaStream_t stream) {
  const int64_t groups = (a.N + R - 1) / R;
  constexpr int kGroupsPerCta = kWarps / S;
  const dim3 grid(static_cast<unsigned>((groups + kGroupsPerCta - 1) / kGroupsPerCta));
  return launch_kernel(linear_gemv_kernel<MB, 0, R, U, S, true>, grid, dim3(kThreads), 0, stream, a.no_pdl == 0, a);
}

template <int MB, int R, int U, int S>
cudaError_t launch_mb(const LinearArgs& a, cudaStream_t stream) {
  const int64_t groups = (a.N + R - 1) / R;
  constexpr int kGroupsPerCta = kWarps / S;
  const dim3 grid(static_cast<unsigned>((groups + kGroupsPerCta - 1) / kGroupsPerCta));
  auto kernel = a.acc_only ? linear_gemv_kernel<MB, 2, R, U, S>
                : a.res_rows != nullptr ? linear_gemv_kernel<MB, 1, R, U, S> : linear_gemv_kernel<MB, 0, R, U, S>;
  return launch_kernel(kernel, grid, dim3(kThreads), 0, stream, a.no_pdl == 0, a);
}

}  // namespace

// Shapes (R, U, S) per row count, measured on the 5120 x 17408 decode
// weight (us for 1 / 3 / 8 rows): (4,4,1) 23.2 / 37.3 / 68.8; (4,2,2) 20.1 /
// 25.1 / 58.4; (2,2,4) 21.0 / 24.4 / 41.6; (4,1,8) 21.0 / 26.2 / 35.1.  More
// rows make each weight chunk cost more dp4a and token-row loads, so they
// want more warps per channel group and fewer chunks in flight per lane.
// 4-bit weights stream half the bytes per code and unpack in registers;
// shapes as for 8-bit weights.
cudaError_t launch_linear_gemv_w4(const LinearArgs& a, cudaStream_t stream) {
  if (a.M <= 1) return launch_mb_w4<1, 4, 2, 2>(a, stream);
  if (a.M <= 2) return launch_mb_w4<2, 4, 2, 2>(a, stream);
  if (a.M <= 4) return launch_mb_w4<4, 2, 2, 4>(a, stream);
  return launch_mb_w4<8, 4, 1, 8>(a, stream);
}

// Unpack 4-bit codes to int8: each thread turns 16 packed bytes (32 codes)
// into 32 bytes.  From the 16 * code bytes of unpack_w4x16, a logical shift
// of the word by 4 leaves each code's low nibble in its byte (the next
// byte's low nibble is zero), and the sign is spread over the high nibble
// with (u & 0x08) * 0x1E = 0xF0 per negative byte.
__global__ void __launch_bounds__(256)
    unpack_w4_kernel(const uint8_t* __restrict__ w4, int64_t ldw4, int64_t N, int64_t K, int8_t* __restrict__ w8,
                     int64_t ldw8) {
  pdl_trigger();
  pdl_wait();
  const int64_t chunks = K >> 5;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x; i < N * chunks;
       i += static_cast<int64_t>(gridDim.x) * 256) {
    const int64_t n = i / chunks, c = i - n * chunks;
    const uint4 p = __ldg(reinterpret_cast<const uint4*>(w4 + n * ldw4) + c);
    uint4 x[2];
    unpack_w4x16(p, x[0], x[1]);
    uint32_t* v = reinterpret_cast<uint32_t*>(x);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t u = v[j] >> 4;
      v[j] = u | ((u & 0x08080808u) * 0x1Eu);
    }
    uint4* dst = reinterpret_cast<uint4*>(w8 + n * ldw8) + 2 * c;
    dst[0] = x[0];
    dst[1] = x[1];
  }
}

cudaError_t launch_unpack_w4(const uint8_t* w4, int64_t ldw4, int64_t N, int64_t K, int8_t* w8, int64_t ldw8,
                             cudaStream_t stream) {
  const int64_t items = N * (K >> 5);
  const int64_t ctas = std::min<int64_t>((items + 255) / 256, 152 * 16);
  return launch_kernel(unpack_w4_kernel, dim3(static_cast<unsigned>(ctas)), dim3(256), 0, stream, true, w4, ldw4, N,
                       K, w8, ldw8);
}

cudaError_t launch_linear_gemv(const LinearArgs& a, cudaStream_t stream) {
  if (a.M <= 1) return launch_mb<1, 4, 2, 2>(a, stream);
  if (a.M <= 2) return launch_mb<2, 4, 2, 2>(a, stream);
  if (a.M <= 4) return launch_mb<4, 2, 2, 4>(a, stream);
  return launch_mb<8, 4, 1, 8>(a, stream);
}

}  // namespace prism
