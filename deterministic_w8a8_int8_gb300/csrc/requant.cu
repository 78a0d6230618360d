// requant.cu -- SmoothQuant requantisation of Q8_0 weights at load time
// (StartLux-Prism, "Compute shared evidence once": the stored 8-bit weights
// are requantised with the smoothing factors folded in before serving).
//
//   v_nk      = RN(RN(d_n,k/32 * q_nk) * s_k)      d * q is exact in binary32
//   amax_n    = max_k |v_nk|
//   w_nk      = rint_even(RN(v_nk * RN(127 / amax_n)))
//   w_scale_n = RN(amax_n / 127);   amax_n < 2^-120  =>  w_n = 0, w_scale_n = 0
//
// No clamp is needed: |v| <= amax, so |v * RN(127/amax)| <= 127 (1 + 2^-24)
// before rounding, which rounds to at most the next binary32 above 127 and
// then to the integer 127.
//
// HBM-bound, run once per weight: per element 1 byte of codes in, 1/16 byte
// of block scales in, 1 byte out.  One CTA is one team that owns a row at a
// time (persistent over rows).  Each thread holds C 16-element vectors of the
// row: it issues the loads of the next row's codes first, then smooths the
// current row into registers (pass 1, with the max), and quantises from those
// registers (pass 2), so that each element is decoded and smoothed once and
// the DRAM latency of row r+1 hides behind the arithmetic of row r.  s is
// staged once per CTA in shared memory, laid out [4][K/16] float4 so that
// consecutive threads read consecutive 16-byte words.  The arithmetic runs on
// packed pairs (Blackwell's f32x2 operations), which round each component
// like the scalar operation; the codes are decoded and multiplied by their
// block scale in one exact fused operation on the 2^23 binade, and rounded
// to integers with the same binade's unit in the last place.
#include <cuda_fp16.h>

#include "common.cuh"

namespace prism {
namespace {

constexpr int kMaxTeam = 512;
constexpr int kCachedMaxK = 24576;   // 512 threads x 3 vectors of 16; s in 96 KB of shared memory
constexpr float kTiny = 0x1p-120f;

// Exact c * d for codes i and i+1 of a word in one packed fused multiply-add.
// xw is the code word with every byte's top bit flipped (u = c + 128); the
// byte goes to bits 8..15 of 2^23, F = 2^23 + 256 u, and
//     F * (d / 256) - (2^15 + 2^7) d = (u - 128) d = c d.
// d / 256 is exact (d is a binary16 value, at least 2^-24 when nonzero),
// (2^15 + 2^7) d has at most 20 significant bits so it is exact too, and the
// fused operation rounds the exact result c d, which has at most 19
// significant bits, only once: it comes out exact.
__device__ __forceinline__ float2 code_pair_times_d(uint32_t xw, int i, float2 d_256, float2 neg_bias) {
  const uint32_t sel = 0x7504u | (static_cast<uint32_t>(i) << 4);
  const float lo = __uint_as_float(__byte_perm(xw, 0x4B000000u, sel));
  const float hi = __uint_as_float(__byte_perm(xw, 0x4B000000u, sel + 0x10u));
  return __ffma2_rn(make_float2(lo, hi), d_256, neg_bias);
}

// w = rint_even(RN(v * inv)) for two values, as the low 16 bits.  t =
// RN(v * inv) is one packed multiply; rint_even(t) for |t| < 2^22 is then the
// low byte of RN(t + 1.5 * 2^23): that sum lies in [2^23, 2^24), where the
// unit in the last place is 1, so the addition's single rounding rounds t to
// an integer, ties to even (1.5 * 2^23 is even), and the integer lands in the
// low mantissa bits.  t must be rounded on its own first -- a fused
// multiply-add would send the products that RN rounds up onto a tie x.5 to
// the odd neighbour -- so the additions are scalar __fadd_rn, which is never
// merged into a multiply-add.  (The packed add is: the assembler fuses a
// packed multiply and a packed add, even written as PTX with explicit .rn.)
__device__ __forceinline__ uint32_t round_pair_lo16(float2 v, float2 inv2) {
  const float2 t = __fmul2_rn(v, inv2);
  return __byte_perm(__float_as_uint(__fadd_rn(t.x, 12582912.0f)), __float_as_uint(__fadd_rn(t.y, 12582912.0f)),
                     0x0040u);
}

__device__ __forceinline__ float f16_bits_to_float(uint32_t h) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
}

// 16 smoothed values of one vector: codes (4 words), block scale df, s from
// shared memory (sv[j] holds s_k for k = 4j .. 4j+3 of the vector):
// v = RN(c * d * s), c * d exact.
struct Vec16 {
  float2 v[8];
};
__device__ __forceinline__ Vec16 smooth16(uint4 codes, float df, const float4 (&sv)[4]) {
  Vec16 r;
  const uint32_t w[4] = {codes.x ^ 0x80808080u, codes.y ^ 0x80808080u, codes.z ^ 0x80808080u,
                         codes.w ^ 0x80808080u};
  const float d256 = __fmul_rn(df, 0x1p-8f);
  const float nb = __fmul_rn(df, -32896.0f);
  const float2 d2 = make_float2(d256, d256), b2 = make_float2(nb, nb);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    r.v[2 * j] = __fmul2_rn(code_pair_times_d(w[j], 0, d2, b2), make_float2(sv[j].x, sv[j].y));
    r.v[2 * j + 1] = __fmul2_rn(code_pair_times_d(w[j], 2, d2, b2), make_float2(sv[j].z, sv[j].w));
  }
  return r;
}
__device__ __forceinline__ float absmax16(const Vec16& r, float m) {
#pragma unroll
  for (int e = 0; e < 8; ++e) m = fmaxf(fmaxf(m, fabsf(r.v[e].x)), fabsf(r.v[e].y));
  return m;
}
// |RN(v * inv)| <= 127.00001 (see the top of the file): every integer is
// within +-127.
__device__ __forceinline__ uint4 requant16(const Vec16& r, float inv) {
  const float2 inv2 = make_float2(inv, inv);
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    o[j] = __byte_perm(round_pair_lo16(r.v[2 * j], inv2), round_pair_lo16(r.v[2 * j + 1], inv2), 0x5410u);
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Coherent 16-byte load that does not allocate in L1 (w may be q: a row is
// read completely before it is written, by the same CTA).
__device__ __forceinline__ uint4 ld_codes(const int8_t* p) {
  uint4 v;
  asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// The max of m (>= 0) over the CTA, on its bit pattern (ordered like the
// value for non-negative floats) with warp reductions.  red is a [2][warps]
// double buffer indexed by row parity, so that one barrier per row suffices:
// a warp writes slot par of row r + 2 only after every thread has passed row
// r + 1's barrier, which is after every read of row r's slots.
__device__ __forceinline__ float team_max(float m, uint32_t (*red)[kMaxTeam / 32], int par) {
  const uint32_t wm = __reduce_max_sync(0xffffffffu, __float_as_uint(m));
  const int lane = threadIdx.x & 31;
  if (lane == 0) red[par][threadIdx.x >> 5] = wm;
  __syncthreads();
  const uint32_t x = lane < static_cast<int>(blockDim.x >> 5) ? red[par][lane] : 0u;
  return __uint_as_float(__reduce_max_sync(0xffffffffu, x));
}

// C: 16-element vectors per thread; P: rows whose codes are in registers at
// once (the current one and P - 1 prefetched); T: the largest CTA size.
template <int C, int P, int T>
__global__ void __launch_bounds__(T)
    smooth_requant_kernel(const int8_t* q, int64_t ldq, const uint16_t* __restrict__ d, int64_t ldd,
                          const float* __restrict__ s, int64_t N, int K, int8_t* w, int64_t ldw,
                          float* __restrict__ w_scale) {
  extern __shared__ float4 s_sm[];   // [4][nvec]
  __shared__ uint32_t red[2][kMaxTeam / 32];
  pdl_trigger();
  pdl_wait();
  const int team = blockDim.x;
  const int lt = threadIdx.x;
  const int nvec = K >> 4;
  for (int f = lt; f < (K >> 2); f += team) {
    const float4 sv = s != nullptr ? __ldg(reinterpret_cast<const float4*>(s) + f) : make_float4(1.f, 1.f, 1.f, 1.f);
    s_sm[(f & 3) * nvec + (f >> 2)] = sv;
  }
  __syncthreads();

  uint4 cur[P][C];      // cur[0]: this row; cur[j]: the row j steps ahead
  uint32_t dcur[P][C];
  int64_t r = blockIdx.x;
  auto load_row = [&](int64_t row, uint4(&c)[C], uint32_t(&dd)[C]) {
    const int8_t* qr = q + row * ldq;
    const uint16_t* dr = d + row * ldd;
#pragma unroll
    for (int i = 0; i < C; ++i) {
      const int v = lt + i * team;
      if (v < nvec) {
        c[i] = ld_codes(qr + 16 * static_cast<int64_t>(v));
        dd[i] = __ldg(dr + (v >> 1));
      }
    }
  };
#pragma unroll
  for (int j = 0; j < P; ++j)
    if (r + j * static_cast<int64_t>(gridDim.x) < N) load_row(r + j * static_cast<int64_t>(gridDim.x), cur[j], dcur[j]);
  int par = 0;
  for (; r < N; r += gridDim.x) {
    uint4 nxt[C];
    uint32_t dnxt[C];
    const int64_t rn = r + P * static_cast<int64_t>(gridDim.x);
    if (rn < N) load_row(rn, nxt, dnxt);

    // pass 1: the smoothed row, kept in registers for pass 2
    Vec16 x[C];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < C; ++i) {
      const int v = lt + i * team;
      if (v < nvec) {
        const float4 sv[4] = {s_sm[v], s_sm[nvec + v], s_sm[2 * nvec + v], s_sm[3 * nvec + v]};
        x[i] = smooth16(cur[0][i], f16_bits_to_float(dcur[0][i]), sv);
        amax = absmax16(x[i], amax);
      }
    }
    amax = team_max(amax, red, par);
    par ^= 1;
    const bool zero_row = !(amax >= kTiny);
    const float inv = zero_row ? 0.0f : __fdiv_rn(127.0f, amax);
    if (lt == 0) w_scale[r] = zero_row ? 0.0f : __fdiv_rn(amax, 127.0f);

    // pass 2
    int8_t* wr = w + r * ldw;
#pragma unroll
    for (int i = 0; i < C; ++i) {
      const int v = lt + i * team;
      if (v < nvec) *reinterpret_cast<uint4*>(wr + 16 * static_cast<int64_t>(v)) = requant16(x[i], inv);
    }
#pragma unroll
    for (int i = 0; i < C; ++i) {
#pragma unroll
      for (int j = 0; j + 1 < P; ++j) {
        cur[j][i] = cur[j + 1][i];
        dcur[j][i] = dcur[j + 1][i];
      }
      cur[P - 1][i] = nxt[i];
      dcur[P - 1][i] = dnxt[i];
    }
  }
}

// Rows longer than the register cache: the same arithmetic with every vector
// read from global memory in both passes (the second read hits L2).  One
// thread reads and later writes only its own vectors, so w may be q.
__global__ void __launch_bounds__(kMaxTeam)
    smooth_requant_long_kernel(const int8_t* q, int64_t ldq, const uint16_t* __restrict__ d, int64_t ldd,
                               const float* __restrict__ s, int64_t N, int K, int8_t* w, int64_t ldw,
                               float* __restrict__ w_scale) {
  __shared__ uint32_t red[2][kMaxTeam / 32];
  pdl_trigger();
  pdl_wait();
  const int nvec = K >> 4;
  const float4 one4 = make_float4(1.f, 1.f, 1.f, 1.f);
  const float4* s4g = reinterpret_cast<const float4*>(s);
  int par = 0;
  for (int64_t r = blockIdx.x; r < N; r += gridDim.x) {
    const int8_t* qr = q + r * ldq;
    const uint16_t* dr = d + r * ldd;
    float amax = 0.0f;
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
      const float4 sv[4] = {s4g ? __ldg(s4g + 4 * v) : one4, s4g ? __ldg(s4g + 4 * v + 1) : one4,
                            s4g ? __ldg(s4g + 4 * v + 2) : one4, s4g ? __ldg(s4g + 4 * v + 3) : one4};
      const Vec16 x = smooth16(ld_codes(qr + 16 * static_cast<int64_t>(v)), f16_bits_to_float(__ldg(dr + (v >> 1))), sv);
      amax = absmax16(x, amax);
    }
    amax = team_max(amax, red, par);
    par ^= 1;
    const bool zero_row = !(amax >= kTiny);
    const float inv = zero_row ? 0.0f : __fdiv_rn(127.0f, amax);
    if (threadIdx.x == 0) w_scale[r] = zero_row ? 0.0f : __fdiv_rn(amax, 127.0f);
    int8_t* wr = w + r * ldw;
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
      const float4 sv[4] = {s4g ? __ldg(s4g + 4 * v) : one4, s4g ? __ldg(s4g + 4 * v + 1) : one4,
                            s4g ? __ldg(s4g + 4 * v + 2) : one4, s4g ? __ldg(s4g + 4 * v + 3) : one4};
      const Vec16 x = smooth16(ld_codes(qr + 16 * static_cast<int64_t>(v)), f16_bits_to_float(__ldg(dr + (v >> 1))), sv);
      *reinterpret_cast<uint4*>(wr + 16 * static_cast<int64_t>(v)) = requant16(x, inv);
    }
  }
}

int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Persistent grid: as many CTAs as fit at once, then trimmed to
// ceil(N / rows_each) CTAs, rows_each = ceil(N / that), so that every CTA
// takes rows_each or rows_each - 1 rows and no partial last wave is left.
template <typename Kernel>
cudaError_t persistent_grid(Kernel kernel, int team, size_t smem, int64_t N, int* grid) {
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, team, smem);
  if (e != cudaSuccess) return e;
  const int64_t gmax = static_cast<int64_t>(sms) * (per_sm > 0 ? per_sm : 1);
  const int64_t rows_each = cdiv64(N, gmax);
  *grid = static_cast<int>(cdiv64(N, rows_each));
  return cudaSuccess;
}

template <int C, int P, int T>
cudaError_t launch_cached(int team, const int8_t* q, int64_t ldq, const uint16_t* d, int64_t ldd, const float* s,
                          int64_t N, int K, int8_t* w, int64_t ldw, float* w_scale, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(K) * sizeof(float);
  auto kernel = smooth_requant_kernel<C, P, T>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kernel), static_cast<int>(smem));
  int grid = 0;
  if (e == cudaSuccess) e = persistent_grid(kernel, team, smem, N, &grid);
  if (e != cudaSuccess) return e;
  return launch_kernel(kernel, dim3(grid), dim3(team), smem, stream, true, q, ldq, d, ldd, s, N, K, w, ldw,
                       w_scale);
}

}  // namespace

// Team shape for a row of K: the fewest 16-element vectors per thread (C of
// 1 to 3) that keep the team within kMaxTeam threads; returns C, or 0 for
// rows that take the uncached kernel.  *team gets the CTA size.
int requant_shape(int K, int* team) {
  const int nvec = K / 16;
  if (K <= kCachedMaxK) {
    for (int c = 1; c <= 3; ++c) {
      const int warps = (nvec + 32 * c - 1) / (32 * c);
      if (warps * 32 <= kMaxTeam) {
        *team = warps * 32;
        return c;
      }
    }
  }
  *team = kMaxTeam;
  return 0;
}

cudaError_t launch_smooth_requant(const int8_t* q, int64_t ldq, const uint16_t* d, int64_t ldd, const float* s,
                                  int64_t N, int64_t K, int8_t* w, int64_t ldw, float* w_scale,
                                  cudaStream_t stream) {
  int team = 0;
  const int k = static_cast<int>(K);
  switch (requant_shape(k, &team)) {
    case 1: return launch_cached<1, 1, kMaxTeam>(team, q, ldq, d, ldd, s, N, k, w, ldw, w_scale, stream);
    case 2: return launch_cached<2, 1, kMaxTeam>(team, q, ldq, d, ldd, s, N, k, w, ldw, w_scale, stream);
    case 3:
      // One such CTA fills an SM's registers, so its row loop alone must
      // keep the bytes in flight: rows up to 384 threads wide prefetch two
      // rows ahead (measured on the 5120 x 17408 down projection: 61 us with
      // none, 43.5 with one, 41.5 with two).
      if (team <= 384) return launch_cached<3, 3, 384>(team, q, ldq, d, ldd, s, N, k, w, ldw, w_scale, stream);
      return launch_cached<3, 1, kMaxTeam>(team, q, ldq, d, ldd, s, N, k, w, ldw, w_scale, stream);
    default: break;
  }
  int grid = 0;
  cudaError_t e = persistent_grid(smooth_requant_long_kernel, team, 0, N, &grid);
  if (e != cudaSuccess) return e;
  return launch_kernel(smooth_requant_long_kernel, dim3(grid), dim3(team), 0, stream, true, q, ldq, d, ldd, s, N, k,
                       w, ldw, w_scale);
}

}  // namespace prism
