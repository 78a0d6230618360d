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

template <int TEAM, int CACHE, int kMode>
__global__ void __launch_bounds__(kBlock)
    quant_act_kernel(const uint16_t* __restrict__ x, int64_t ldx, const float* __restrict__ inv_s,
                     int64_t M, int64_t K, int8_t* __restrict__ q, int64_t ldq,
                     float* __restrict__ a_scale, const int32_t* __restrict__ rows, int64_t M_x,
                     uint32_t* err, float* __restrict__ amax_io) {
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

#pragma unroll
  for (int c = 0; c < CACHE; ++c) {
    const int64_t v = lt + static_cast<int64_t>(c) * TEAM;
    if (v < nvec) {
      const Vec8& r = cache[c];
      uint2 o;
      o.x = quant4(r.v[0], r.v[1], r.v[2], r.v[3], inv_a);
      o.y = quant4(r.v[4], r.v[5], r.v[6], r.v[7], inv_a);
      *reinterpret_cast<uint2*>(qr + v * 8) = o;
    }
  }
  for (int64_t v = lt + static_cast<int64_t>(CACHE) * TEAM; v < nvec; v += TEAM) {
    const Vec8 r = load_smoothed(xr, inv_s, v * 8);
    uint2 o;
    o.x = quant4(r.v[0], r.v[1], r.v[2], r.v[3], inv_a);
    o.y = quant4(r.v[4], r.v[5], r.v[6], r.v[7], inv_a);
    *reinterpret_cast<uint2*>(qr + v * 8) = o;
  }
}

template <int TEAM, int CACHE>
cudaError_t launch_team(const QuantCall& c, cudaStream_t stream) {
  constexpr int kTeams = kBlock / TEAM;
  const int64_t blocks = (c.M + kTeams - 1) / kTeams;
  auto kernel = c.rows != nullptr      ? quant_act_kernel<TEAM, CACHE, kRows>
                : c.amax_out != nullptr ? quant_act_kernel<TEAM, CACHE, kAmaxOut>
                : c.amax_in != nullptr  ? quant_act_kernel<TEAM, CACHE, kAmaxIn>
                                        : quant_act_kernel<TEAM, CACHE, kPlain>;
  float* amax_io = c.amax_out != nullptr ? c.amax_out : const_cast<float*>(c.amax_in);
  return launch_kernel(kernel, dim3(static_cast<unsigned>(blocks)), dim3(kBlock), 0, stream, true,
                       static_cast<const uint16_t*>(c.x), c.ldx, c.inv_s, c.M, c.K, c.q, c.ldq, c.a_scale, c.rows,
                       c.rows != nullptr ? c.M_x : c.M, c.err, amax_io);
}

}  // namespace

cudaError_t launch_quant(const QuantCall& c, cudaStream_t stream) {
  // Team size grows with K so that a row fits the team's register cache
  // (TEAM * CACHE * 8 elements); longer rows re-read their tail from L2.
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
