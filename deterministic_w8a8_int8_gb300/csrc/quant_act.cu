// quant_act.cu -- per-token activation quantisation with the SmoothQuant
// divisor folded in (StartLux-Prism, "Compute shared evidence once").
//
//   xs_k    = x_k * inv_s_k                      binary32 RN
//   amax    = max_k |xs_k|                       exact (order free)
//   q_k     = clamp(rint_even(xs_k * RN(127/amax)), -127, 127)
//   a_scale = RN(amax / 127);  amax < 2^-120  =>  q = 0, a_scale = 0
//
// HBM-bound: each row is read once from DRAM (3 bytes per element in and
// out, plus 4 bytes of scale per row).  A team of TEAM threads owns one row:
// pass 1 streams the row with 16-byte loads and keeps the smoothed values in
// registers while they fit (CACHE vectors of 8 per thread), reduces amax with
// warp shuffles, pass 2 quantises from registers (or re-reads the row from L2
// when it is longer than the cache) and stores 8-byte int8 vectors.
#include <cuda_fp16.h>

#include "common.cuh"

namespace prism {
namespace {

constexpr int kBlock = 256;

struct Vec8 {
  float v[8];
};

__device__ __forceinline__ Vec8 load_smoothed(const uint16_t* __restrict__ xr,
                                              const float* __restrict__ inv_s, int64_t k0) {
  const uint4 xv = __ldg(reinterpret_cast<const uint4*>(xr + k0));
  Vec8 r;
  r.v[0] = bf16_lo(xv.x);
  r.v[1] = bf16_hi(xv.x);
  r.v[2] = bf16_lo(xv.y);
  r.v[3] = bf16_hi(xv.y);
  r.v[4] = bf16_lo(xv.z);
  r.v[5] = bf16_hi(xv.z);
  r.v[6] = bf16_lo(xv.w);
  r.v[7] = bf16_hi(xv.w);
  if (inv_s != nullptr) {
    const float4 s0 = __ldg(reinterpret_cast<const float4*>(inv_s + k0));
    const float4 s1 = __ldg(reinterpret_cast<const float4*>(inv_s + k0 + 4));
    r.v[0] = __fmul_rn(r.v[0], s0.x);
    r.v[1] = __fmul_rn(r.v[1], s0.y);
    r.v[2] = __fmul_rn(r.v[2], s0.z);
    r.v[3] = __fmul_rn(r.v[3], s0.w);
    r.v[4] = __fmul_rn(r.v[4], s1.x);
    r.v[5] = __fmul_rn(r.v[5], s1.y);
    r.v[6] = __fmul_rn(r.v[6], s1.z);
    r.v[7] = __fmul_rn(r.v[7], s1.w);
  }
  return r;
}

__device__ __forceinline__ uint32_t quant4(float a, float b, float c, float d, float inv_a) {
  int qa = max(-127, min(127, __float2int_rn(__fmul_rn(a, inv_a))));
  int qb = max(-127, min(127, __float2int_rn(__fmul_rn(b, inv_a))));
  int qc = max(-127, min(127, __float2int_rn(__fmul_rn(c, inv_a))));
  int qd = max(-127, min(127, __float2int_rn(__fmul_rn(d, inv_a))));
  return (static_cast<uint32_t>(qa) & 0xffu) | ((static_cast<uint32_t>(qb) & 0xffu) << 8) |
         ((static_cast<uint32_t>(qc) & 0xffu) << 16) | ((static_cast<uint32_t>(qd) & 0xffu) << 24);
}

__device__ __forceinline__ float vmaxabs(const Vec8& r, float m) {
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(r.v[i]));
  return m;
}

// Modes.  kPlain: the quantiser.  kRows: output row m quantises x row
// rows[m] of the M_x rows of x (the last layer restricted to answer
// positions); an index outside [0, M_x) gives a zero q row, a NaN scale and
// PRISM_DEV_ERR_ROW_RANGE in *err.  kAmaxOut: only the row maxima, into
// amax_io (a tensor-parallel rank's shard maxima).  kAmaxIn: the codes and
// scale from the given maxima amax_io (the maximum over the ranks).
enum QuantMode { kPlain = 0, kRows = 1, kAmaxOut = 2, kAmaxIn = 3 };

// The codes of 4 values (see quant4) as two packed binary16 pairs: integers
// of at most 127 in magnitude, so the conversions are exact.
__device__ __forceinline__ uint2 quant4_f16(float a, float b, float c, float d, float inv_a) {
  const int qa = max(-127, min(127, __float2int_rn(__fmul_rn(a, inv_a))));
  const int qb = max(-127, min(127, __float2int_rn(__fmul_rn(b, inv_a))));
  const int qc = max(-127, min(127, __float2int_rn(__fmul_rn(c, inv_a))));
  const int qd = max(-127, min(127, __float2int_rn(__fmul_rn(d, inv_a))));
  const __half2 lo = __halves2half2(__int2half_rn(qa), __int2half_rn(qb));
  const __half2 hi = __halves2half2(__int2half_rn(qc), __int2half_rn(qd));
  return make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
}

// kHalf: the codes are stored as binary16 values (qh, row stride ldqh
// elements) instead of int8 -- the operand form of the tensor-core kernel
// that reads f16 codes (linear_f16.cu).  Only with kPlain.
template <int TEAM, int CACHE, int kMode, bool kHalf>
__global__ void __launch_bounds__(kBlock)
    quant_act_kernel(const uint16_t* __restrict__ x, int64_t ldx, const float* __restrict__ inv_s,
                     int64_t M, int64_t K, int8_t* __restrict__ q, int64_t ldq,
                     float* __restrict__ a_scale, const int32_t* __restrict__ rows, int64_t M_x,
                     uint32_t* err, float* __restrict__ amax_io, uint16_t* __restrict__ qh, int64_t ldqh) {
  static_assert(!kHalf || kMode == kPlain, "binary16 codes only for the plain quantiser");
  constexpr int kTeams = kBlock / TEAM;
  constexpr int kWarpsPerTeam = TEAM / 32;
  __shared__ float red[kBlock / 32];
  pdl_trigger();
  pdl_wait();
  const int team = threadIdx.x / TEAM;
  const int lt = threadIdx.x % TEAM;
  const int64_t m = static_cast<int64_t>(blockIdx.x) * kTeams + team;
  const bool in_grid = m < M;
  int64_t src = m;
  if constexpr (kMode == kRows) src = in_grid ? __ldg(rows + m) : -1;
  const bool row_ok = kMode == kRows ? (src >= 0 && src < M_x) : in_grid;
  const bool active = in_grid && row_ok;
  const uint16_t* xr = x + (active ? src : 0) * ldx;
  const int64_t nvec = K >> 3;

  Vec8 cache[CACHE];
  float amax = 0.0f;
  if (active) {
#pragma unroll
    for (int c = 0; c < CACHE; ++c) {
      const int64_t v = lt + static_cast<int64_t>(c) * TEAM;
      if (v < nvec) {
        cache[c] = load_smoothed(xr, inv_s, v * 8);
        amax = vmaxabs(cache[c], amax);
      }
    }
    if constexpr (kMode != kAmaxIn)
      for (int64_t v = lt + static_cast<int64_t>(CACHE) * TEAM; v < nvec; v += TEAM)
        amax = vmaxabs(load_smoothed(xr, inv_s, v * 8), amax);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (kWarpsPerTeam > 1) {
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    const int w0 = team * kWarpsPerTeam;
#pragma unroll
    for (int i = 0; i < kWarpsPerTeam; ++i) amax = fmaxf(amax, red[w0 + i]);
  }
  if (!in_grid) return;
  if constexpr (kMode == kAmaxOut) {
    if (lt == 0) amax_io[m] = amax;
    return;
  }
  if constexpr (kMode == kAmaxIn) amax = __ldg(amax_io + m);
  if (kMode == kRows && !row_ok) {
    int8_t* qr = q + m * ldq;
    for (int64_t v = lt; v < (K >> 3); v += TEAM) *reinterpret_cast<uint2*>(qr + v * 8) = make_uint2(0u, 0u);
    if (lt == 0) {
      a_scale[m] = __uint_as_float(0x7fc00000u);
      if (err != nullptr) atomicOr(err, PRISM_DEV_ERR_ROW_RANGE);
    }
    return;
  }

  int8_t* qr = q + m * ldq;
  const bool zero_row = !(amax >= 0x1p-120f);
  const float inv_a = zero_row ? 0.0f : __fdiv_rn(127.0f, amax);
  if (lt == 0) a_scale[m] = zero_row ? 0.0f : __fdiv_rn(amax, 127.0f);
  auto store8 = [&](const Vec8& r, int64_t v) {
    if constexpr (kHalf) {
      const uint2 lo = quant4_f16(r.v[0], r.v[1], r.v[2], r.v[3], inv_a);
      const uint2 hi = quant4_f16(r.v[4], r.v[5], r.v[6], r.v[7], inv_a);
      *reinterpret_cast<uint4*>(qh + m * ldqh + v * 8) = make_uint4(lo.x, lo.y, hi.x, hi.y);
    } else {
      uint2 o;
      o.x = quant4(r.v[0], r.v[1], r.v[2], r.v[3], inv_a);
      o.y = quant4(r.v[4], r.v[5], r.v[6], r.v[7], inv_a);
      *reinterpret_cast<uint2*>(qr + v * 8) = o;
    }
  };

#pragma unroll
  for (int c = 0; c < CACHE; ++c) {
    const int64_t v = lt + static_cast<int64_t>(c) * TEAM;
    if (v < nvec) store8(cache[c], v);
  }
  for (int64_t v = lt + static_cast<int64_t>(CACHE) * TEAM; v < nvec; v += TEAM)
    store8(load_smoothed(xr, inv_s, v * 8), v);
}

// ----------------------------------------------------------------------
// Persistent form for rows of up to 512 threads x 6 vectors of 8 (K <=
// 24576): one CTA is one team that owns a row at a time.  Each thread keeps
// C raw 16-byte vectors of the row (8 bf16) and the same vectors of the next
// P - 1 rows, whose loads it issues before it works on the current row, so
// the DRAM latency of the next rows hides behind this one.  inv_s is staged
// once per CTA in shared memory as [2][K/8] float4 (consecutive threads read
// consecutive 16-byte words).  Pass 1 smooths the row and takes its max;
// pass 2 smooths it again from the raw registers (two operations per element,
// cheaper than holding floats) and quantises.  Smoothing and the 127/amax
// product run as packed f32x2 multiplies (each component rounded like the
// scalar operation); the rounding to an integer is RN(t + 1.5 * 2^23) with
// the scalar __fadd_rn, which is never merged into a multiply-add: on [2^23,
// 2^24) the unit in the last place is 1, so that single rounding is
// round-half-even of t and the integer sits in the low mantissa bits.
constexpr int kPMaxTeam = 512;
constexpr int kPCachedMaxK = kPMaxTeam * 6 * 8;

struct PArgs {
  const uint16_t* x;
  int64_t ldx;
  const float* inv_s;
  int64_t M, K;
  int8_t* q;
  int64_t ldq;
  float* a_scale;
  const int32_t* rows;
  int64_t M_x;
  uint32_t* err;
  float* amax_io;
  uint16_t* qh;      // binary16 codes out (kHalf), row stride ldqh elements
  int64_t ldqh;
};

__device__ __forceinline__ float2 smooth2(uint32_t pair, float4 s, int half) {
  const float2 v = make_float2(bf16_lo(pair), bf16_hi(pair));
  return __fmul2_rn(v, half ? make_float2(s.z, s.w) : make_float2(s.x, s.y));
}

template <int C, int P, int kMode, bool kHalf>
__global__ void __launch_bounds__(kPMaxTeam)
    quant_persist_kernel(const __grid_constant__ PArgs a) {
  static_assert(!kHalf || kMode == kPlain, "binary16 codes only for the plain quantiser");
  extern __shared__ float4 s_sm[];   // [2][K/8]
  __shared__ uint32_t red[2][kPMaxTeam / 32];
  pdl_trigger();
  pdl_wait();
  const int team = blockDim.x, lt = threadIdx.x, lane = lt & 31;
  const int nvec = static_cast<int>(a.K >> 3);
  for (int f = lt; f < (nvec << 1); f += team) {
    const float4 sv = a.inv_s != nullptr ? __ldg(reinterpret_cast<const float4*>(a.inv_s) + f)
                                         : make_float4(1.f, 1.f, 1.f, 1.f);
    s_sm[(f & 1) * nvec + (f >> 1)] = sv;
  }
  __syncthreads();

  // source row of output row r (kRows: the index list, -1 when out of range)
  auto source = [&](int64_t r) -> int64_t {
    if constexpr (kMode == kRows) {
      const int64_t s = __ldg(a.rows + r);
      return s >= 0 && s < a.M_x ? s : -1;
    }
    return r;
  };
  auto load_row = [&](int64_t r, uint4(&v)[C]) {
    const int64_t src = source(r);
    const uint16_t* xr = a.x + (src >= 0 ? src : 0) * a.ldx;
#pragma unroll
    for (int i = 0; i < C; ++i) {
      const int j = lt + i * team;
      v[i] = src >= 0 && j < nvec ? __ldg(reinterpret_cast<const uint4*>(xr) + j) : make_uint4(0u, 0u, 0u, 0u);
    }
  };

  uint4 cur[P][C];
  int64_t r = blockIdx.x;
#pragma unroll
  for (int j = 0; j < P; ++j)
    if (r + j * static_cast<int64_t>(gridDim.x) < a.M) load_row(r + j * static_cast<int64_t>(gridDim.x), cur[j]);
  int par = 0;
  for (; r < a.M; r += gridDim.x) {
    uint4 nxt[C];
    const int64_t rn = r + P * static_cast<int64_t>(gridDim.x);
    if (rn < a.M) load_row(rn, nxt);

    // pass 1: smoothed values, row max
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < C; ++i) {
      const int j = lt + i * team;
      if (j < nvec) {
        const float4 s0 = s_sm[j], s1 = s_sm[nvec + j];
        const float2 v0 = smooth2(cur[0][i].x, s0, 0), v1 = smooth2(cur[0][i].y, s0, 1);
        const float2 v2 = smooth2(cur[0][i].z, s1, 0), v3 = smooth2(cur[0][i].w, s1, 1);
        amax = fmaxf(fmaxf(fmaxf(amax, fabsf(v0.x)), fabsf(v0.y)), fmaxf(fabsf(v1.x), fabsf(v1.y)));
        amax = fmaxf(fmaxf(fmaxf(amax, fabsf(v2.x)), fabsf(v2.y)), fmaxf(fabsf(v3.x), fabsf(v3.y)));
      }
    }
    // the team's max on the bit patterns (ordered like the values for x >= 0)
    const uint32_t wm = __reduce_max_sync(0xffffffffu, __float_as_uint(amax));
    if (lane == 0) red[par][lt >> 5] = wm;
    __syncthreads();
    amax = __uint_as_float(__reduce_max_sync(0xffffffffu, lane < (team >> 5) ? red[par][lane] : 0u));
    par ^= 1;

    bool done = false;
    if constexpr (kMode == kAmaxOut) {
      if (lt == 0) a.amax_io[r] = amax;
      done = true;
    }
    if constexpr (kMode == kAmaxIn) amax = __ldg(a.amax_io + r);
    int8_t* qr = a.q + r * a.ldq;
    if constexpr (kMode == kRows) {
      if (source(r) < 0) {   // out-of-range index: zero codes, NaN scale, error bit
#pragma unroll
        for (int i = 0; i < C; ++i) {
          const int j = lt + i * team;
          if (j < nvec) *reinterpret_cast<uint2*>(qr + 8 * static_cast<int64_t>(j)) = make_uint2(0u, 0u);
        }
        if (lt == 0) {
          a.a_scale[r] = __uint_as_float(0x7fc00000u);
          if (a.err != nullptr) atomicOr(a.err, PRISM_DEV_ERR_ROW_RANGE);
        }
        done = true;
      }
    }
    if (!done) {
      const bool zero_row = !(amax >= 0x1p-120f);
      const float inv_a = zero_row ? 0.0f : __fdiv_rn(127.0f, amax);
      if (lt == 0) a.a_scale[r] = zero_row ? 0.0f : __fdiv_rn(amax, 127.0f);
      const float2 inv2 = make_float2(inv_a, inv_a);
      // pass 2: smooth again, scale, round, pack
#pragma unroll
      for (int i = 0; i < C; ++i) {
        const int j = lt + i * team;
        if (j < nvec) {
          const float4 s0 = s_sm[j], s1 = s_sm[nvec + j];
          const float2 t[4] = {__fmul2_rn(smooth2(cur[0][i].x, s0, 0), inv2),
                               __fmul2_rn(smooth2(cur[0][i].y, s0, 1), inv2),
                               __fmul2_rn(smooth2(cur[0][i].z, s1, 0), inv2),
                               __fmul2_rn(smooth2(cur[0][i].w, s1, 1), inv2)};
          uint32_t b[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float lo = t[e].x, hi = t[e].y;
            if constexpr (kMode == kAmaxIn) {   // a given maximum may be below this row's own
              lo = fminf(fmaxf(lo, -127.0f), 127.0f);
              hi = fminf(fmaxf(hi, -127.0f), 127.0f);
            }
            b[2 * e] = __float_as_uint(__fadd_rn(lo, 12582912.0f));
            b[2 * e + 1] = __float_as_uint(__fadd_rn(hi, 12582912.0f));
          }
          if constexpr (kHalf) {
            // the integer r = rint_even(t) back as a float (the subtraction of
            // 1.5 * 2^23 is exact), then exactly to binary16
            uint32_t h[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float lo = __fsub_rn(__uint_as_float(b[2 * e]), 12582912.0f);
              const float hi = __fsub_rn(__uint_as_float(b[2 * e + 1]), 12582912.0f);
              const __half2 hv = __floats2half2_rn(lo, hi);
              h[e] = *reinterpret_cast<const uint32_t*>(&hv);
            }
            *reinterpret_cast<uint4*>(a.qh + r * a.ldqh + 8 * static_cast<int64_t>(j)) =
                make_uint4(h[0], h[1], h[2], h[3]);
          } else {
            const uint32_t w0 =
                __byte_perm(__byte_perm(b[0], b[1], 0x0040u), __byte_perm(b[2], b[3], 0x0040u), 0x5410u);
            const uint32_t w1 =
                __byte_perm(__byte_perm(b[4], b[5], 0x0040u), __byte_perm(b[6], b[7], 0x0040u), 0x5410u);
            *reinterpret_cast<uint2*>(qr + 8 * static_cast<int64_t>(j)) = make_uint2(w0, w1);
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < C; ++i) {
#pragma unroll
      for (int j = 0; j + 1 < P; ++j) cur[j][i] = cur[j + 1][i];
      cur[P - 1][i] = nxt[i];
    }
  }
}

template <int C, int P>
cudaError_t launch_persist(const QuantCall& c, int team, cudaStream_t stream) {
  PArgs p{};
  p.x = static_cast<const uint16_t*>(c.x);
  p.ldx = c.ldx;
  p.inv_s = c.inv_s;
  p.M = c.M;
  p.K = c.K;
  p.q = c.q;
  p.ldq = c.ldq;
  p.a_scale = c.a_scale;
  p.rows = c.rows;
  p.M_x = c.rows != nullptr ? c.M_x : c.M;
  p.err = c.err;
  p.amax_io = c.amax_out != nullptr ? c.amax_out : const_cast<float*>(c.amax_in);
  p.qh = c.qh;
  p.ldqh = c.ldqh;
  auto kernel = c.qh != nullptr         ? quant_persist_kernel<C, P, kPlain, true>
                : c.rows != nullptr     ? quant_persist_kernel<C, P, kRows, false>
                : c.amax_out != nullptr ? quant_persist_kernel<C, P, kAmaxOut, false>
                : c.amax_in != nullptr  ? quant_persist_kernel<C, P, kAmaxIn, false>
                                        : quant_persist_kernel<C, P, kPlain, false>;
  const size_t smem = static_cast<size_t>(c.K) * sizeof(float);
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kernel), static_cast<int>(smem));
  int dev = 0, sms = 0, per_sm = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, team, smem);
  if (e != cudaSuccess) return e;
  const int64_t gmax = static_cast<int64_t>(sms) * std::max(per_sm, 1);
  const int64_t rows_each = (c.M + gmax - 1) / gmax;
  const int64_t grid = (c.M + rows_each - 1) / rows_each;
  return launch_kernel(kernel, dim3(static_cast<unsigned>(grid)), dim3(team), smem, stream, true, p);
}

template <int TEAM, int CACHE>
cudaError_t launch_team(const QuantCall& c, cudaStream_t stream) {
  constexpr int kTeams = kBlock / TEAM;
  const int64_t blocks = (c.M + kTeams - 1) / kTeams;
  auto kernel = c.qh != nullptr         ? quant_act_kernel<TEAM, CACHE, kPlain, true>
                : c.rows != nullptr     ? quant_act_kernel<TEAM, CACHE, kRows, false>
                : c.amax_out != nullptr ? quant_act_kernel<TEAM, CACHE, kAmaxOut, false>
                : c.amax_in != nullptr  ? quant_act_kernel<TEAM, CACHE, kAmaxIn, false>
                                        : quant_act_kernel<TEAM, CACHE, kPlain, false>;
  float* amax_io = c.amax_out != nullptr ? c.amax_out : const_cast<float*>(c.amax_in);
  return launch_kernel(kernel, dim3(static_cast<unsigned>(blocks)), dim3(kBlock), 0, stream, true,
                       static_cast<const uint16_t*>(c.x), c.ldx, c.inv_s, c.M, c.K, c.q, c.ldq, c.a_scale, c.rows,
                       c.rows != nullptr ? c.M_x : c.M, c.err, amax_io, c.qh, c.ldqh);
}

}  // namespace

cudaError_t launch_quant(const QuantCall& c, cudaStream_t stream) {
  if (c.K <= kPCachedMaxK) {
    // the fewest vectors per thread that keep the team within 512 threads
    const int64_t nvec = c.K / 8;
    for (int cv = 1; cv <= 6; ++cv) {
      const int64_t team = 32 * ((nvec + 32 * cv - 1) / (32 * cv));
      if (team > kPMaxTeam) continue;
      const int t = static_cast<int>(team);
      switch (cv) {
        case 1: return launch_persist<1, 2>(c, t, stream);
        case 2: return launch_persist<2, 2>(c, t, stream);
        case 3: return launch_persist<3, 2>(c, t, stream);
        case 4: return launch_persist<4, 2>(c, t, stream);
        case 5: return launch_persist<5, 2>(c, t, stream);
        default: return launch_persist<6, 2>(c, t, stream);
      }
    }
  }
  // Longer rows: a team of TEAM threads per row keeps CACHE vectors of
  // smoothed values per thread in registers and re-reads the rest from L2.
  if (c.K <= 32 * 8 * 4) return launch_team<32, 4>(c, stream);
  if (c.K <= 64 * 8 * 4) return launch_team<64, 4>(c, stream);
  if (c.K <= 128 * 8 * 4) return launch_team<128, 4>(c, stream);
  return launch_team<256, 9>(c, stream);
}

cudaError_t launch_quant_act(const void* x, int64_t ldx, const float* inv_s, int64_t M, int64_t K, int8_t* q,
                             int64_t ldq, float* a_scale, const int32_t* rows, int64_t M_x, uint32_t* err,
                             cudaStream_t stream) {
  QuantCall c{};
  c.x = x;
  c.ldx = ldx;
  c.inv_s = inv_s;
  c.M = M;
  c.K = K;
  c.q = q;
  c.ldq = ldq;
  c.a_scale = a_scale;
  c.rows = rows;
  c.M_x = M_x;
  c.err = err;
  return launch_quant(c, stream);
}

}  // namespace prism
