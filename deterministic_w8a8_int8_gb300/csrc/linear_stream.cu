// linear_stream.cu -- the W8A8 linear for a few token rows (up to 16): a
// weight stream through shared memory into the warp-level integer MMA
// (StartLux-Prism, "Bitwise consistency is not lossless quantization": int8
// products accumulate exactly in int32, split-K partial sums stay integers,
// then a fixed fp32 epilogue).
//
// With M <= 16 every weight byte is used at most 16 times: the call is a
// stream of N * K weight bytes with at most 32 operations per byte.  The
// legacy int8 MMA (mma.sync m16n8k32 s8 -> s32, about 155 TOP/s on this
// part, a thirteenth of the tcgen05 f16 rate) covers that for 8 token rows at
// the HBM rate, and it takes the int8 codes as they are: no widening, exact
// int32 sums in any order.  For 9 to 16 rows its rate falls short, and the
// f16 MMA (607 TFLOP/s measured) takes over on exactly widened codes, with
// fp32 sums drained into int32 every 1024 K (below 2^24, so exact).  What sets the speed is keeping enough weight
// bytes in flight, so each warp streams its own steps (no barrier between
// warps) and each CTA owns whole rows: no partial sums cross CTAs unless the
// weight is too narrow to fill the GPU or the caller asks for split-K.
//
// The sum over K may run in any order, so each lane takes its fragment
// elements in memory order: in a 128-K step, lane (g, t) = (lane / 4, lane %
// 4) reads the 16-byte pieces k0 + 16t and k0 + 64 + 16t of weight rows g and
// g + 8 and of token row g (the four lanes of a row read 64 contiguous bytes
// per load); those 32 bytes are 8 words, and MMA j (j = 0..3) takes words 2j
// and 2j + 1 of each as the fragment's K groups 4t .. 4t + 3 and
// 16 + 4t .. 16 + 4t + 3, in both operands alike.
//
// CTA: 16 output channels against all token rows (NT tiles of 8); its warps
// take the CTA's 128-K steps in turn, each copying its next steps into its
// own cp.async ring in shared memory -- eight warps with two-step rings for
// one token tile, four warps with four-step rings for two (48 or 64 KB per
// CTA, so that every CTA of a 5120-channel weight is resident at once) --
// and add their int32 sums through shared memory at the end.  The grid is one CTA per 16 channels (and per K piece when split).  A
// split K range has each piece add its int32 partial sums into the workspace
// accumulator with integer reductions; the last piece to arrive (an integer
// counter per channel tile) reads the sums back, zeroes them and applies the
// epilogue.  Integer addition is order-free: no split changes a bit.  The
// kernel waits on nothing but its own CTA barrier.
#include <algorithm>
#include <cstdint>

#include "common.cuh"

namespace prism {

int sm_count();

namespace {

constexpr int kWarps = 8;               // warps per CTA
constexpr int kRing = 2;                // steps in flight per warp (its shared-memory ring)
constexpr int kTileN = 16;              // output channels per CTA (one m16 tile)
constexpr int kStepK = 128;             // K per step: 32 bytes per lane, 4 int8 MMAs of K = 32
constexpr int kChunkSteps = 8;          // f16 MMA: steps per exact fp32 chunk (1024 K)
constexpr int kMinStepsPerWarp = 8;     // automatic split: at least 1024 K per warp

__host__ __device__ constexpr int64_t cdiv(int64_t x, int64_t y) { return (x + y - 1) / y; }

__device__ __forceinline__ uint32_t widen_lo(uint32_t u) {   // bytes 0, 1 of u (biased) -> f16x2
  uint32_t r;
  const uint32_t v = __byte_perm(u, 0x64646464u, 0x4140);
  asm("sub.f16x2 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(0x64806480u));
  return r;
}
__device__ __forceinline__ uint32_t widen_hi(uint32_t u) {   // bytes 2, 3 of u (biased) -> f16x2
  uint32_t r;
  const uint32_t v = __byte_perm(u, 0x64646464u, 0x4342);
  asm("sub.f16x2 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(0x64806480u));
  return r;
}
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t word(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

struct StreamParams {
  LinearArgs a;
  int pieces;        // K pieces (CTAs along K) per channel tile
  int steps;         // 128-K steps of the whole K
  int32_t* acc;      // pieces > 1: [M, N] int32 partial sums, zero between calls
  uint32_t* cnt;     // pieces > 1: one arrival counter per channel tile, zero between calls
};

// One 128-K step's operands of one lane: the 16-byte pieces 16t and 64 + 16t
// of weight rows g and g + 8 and of token rows 8 nt + g.
template <int NT>
struct StepRegs {
  uint4 w[2][2];    // [row g / g + 8][first / second 16 bytes]
  uint4 q[NT][2];
};

// The step's four m16n8k32 MMAs: MMA j takes words 2j and 2j + 1 of the
// lane's 32 bytes of each row (its a0 / a2 from row g, a1 / a3 from row
// g + 8) and of its token row (b0 / b1), exact int32 accumulation.
template <int NT>
__device__ __forceinline__ void mma_step(const StepRegs<NT>& r, int32_t (&acc)[NT][4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int h = j >> 1, w0 = 2 * (j & 1);
    const uint32_t a[4] = {word(r.w[0][h], w0), word(r.w[1][h], w0), word(r.w[0][h], w0 + 1),
                           word(r.w[1][h], w0 + 1)};
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      mma_s8_16832(acc[nt], a, word(r.q[nt][h], w0), word(r.q[nt][h], w0 + 1));
  }
}

// The same step on the f16 MMA (two token tiles: the int8 MMA's rate would
// fall short): MMA j (j = 0..7) takes word j of each row's and token row's 32
// bytes, bytes 0, 1 as the fragment's columns 2t, 2t + 1 and bytes 2, 3 as
// columns 2t + 8, 2t + 9; each byte is widened exactly to f16 (bias to
// u = b + 128, place u under the f16 pattern of 1024, subtract 1152) and the
// fp32 sums stay exact integers while a chunk holds at most 1024 K.
template <int NT>
__device__ __forceinline__ void mma_step_f16(const StepRegs<NT>& r, float (&facc)[NT][4]) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t u0 = word(r.w[0][j >> 2], j & 3) ^ 0x80808080u;
    const uint32_t u1 = word(r.w[1][j >> 2], j & 3) ^ 0x80808080u;
    const uint32_t a0 = widen_lo(u0), a1 = widen_lo(u1), a2 = widen_hi(u0), a3 = widen_hi(u1);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const uint32_t v = word(r.q[nt][j >> 2], j & 3) ^ 0x80808080u;
      mma_f16_16816(facc[nt], a0, a1, a2, a3, widen_lo(v), widen_hi(v));
    }
  }
}

// kMode: 0 plain; 1 residual rows through a.res_rows; 2 only the exact int32
// accumulators, into acc_out.  NT: token tiles of 8 rows (M <= 8 NT).  U:
// steps of loads in flight per warp.
template <int NT, int kMode, int U, int kW>
__global__ void __launch_bounds__(kW * 32, 3)
    linear_stream_kernel(const __grid_constant__ StreamParams p) {
  constexpr int kWarps = kW;
  constexpr int kThreads = kWarps * 32;
  extern __shared__ __align__(128) uint8_t ring[];   // per warp, U steps of (16 weight rows | token rows)
  constexpr int kElems = 4 * NT;                            // accumulator elements per lane
  constexpr int kOut = 32 * kElems;                         // accumulator elements of the CTA
  constexpr int kPer = static_cast<int>(cdiv(kOut, kThreads));   // of them per thread at the end
  __shared__ int32_t s_part[kWarps][32][kElems];
  __shared__ int s_last;
  pdl_trigger();
  pdl_wait();
  const LinearArgs& a = p.a;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kTileN;

  // this CTA's K piece (in steps)
  const int per_piece = static_cast<int>(cdiv(p.steps, p.pieces));
  const int pb = min(p.steps, static_cast<int>(blockIdx.y) * per_piece);
  const int pe = min(p.steps, pb + per_piece);
  // the warps take the piece's steps in turn (step pb + warp + i * kWarps is
  // this warp's i-th), so that at any time the CTA's warps read neighbouring
  // 128-byte pieces of the same 16 rows
  const int cnt = pe - pb > warp ? (pe - pb - warp + kWarps - 1) / kWarps : 0;
  auto step_of = [&](int i) { return pb + warp + i * kWarps; };

  int32_t iacc[NT][4];
  float facc[NT][4];   // the f16 MMA's fp32 chunk sums (NT > 1)
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      iacc[nt][i] = 0;
      facc[nt][i] = 0.0f;
    }

  {
    // U steps in flight through this warp's own cp.async ring in shared
    // memory (no registers held by loads in flight, no CTA barrier; every
    // copy has landed before the warp leaves the loop)
    constexpr int kStageBytes = (kTileN + 8 * NT) * kStepK;
    const uint32_t base = smem_u32(ring) + static_cast<uint32_t>(warp * U * kStageBytes);
    // 16-byte chunk c of row r (weights rows 0..15, then token rows) sits at
    // chunk c ^ 4 (r & 1) of the row: the lanes of a quarter-warp, reading
    // chunks t (or 4 + t) of rows g and g + 1, hit all 32 banks once
    auto issue = [&](int step, int slot) {
      const uint32_t sb = base + static_cast<uint32_t>(slot * kStageBytes);
#pragma unroll
      for (int i = 0; i < (kTileN + 8 * NT) * 8 / 32; ++i) {
        const int ci = lane + 32 * i;
        const int r = ci >> 3, c = ci & 7;
        const int64_t k = static_cast<int64_t>(step) * kStepK + 16 * c;
        const uint32_t dst = sb + static_cast<uint32_t>(r * kStepK + ((c ^ (4 * (r & 1))) * 16));
        if (r < kTileN) {
          const int64_t n = c0 + r;
          const bool in = n < a.N && k < a.K;
          cp_async_16(dst, in ? a.w + n * a.ldw + k : a.w, in ? 16 : 0);
        } else {
          const int64_t m = r - kTileN;
          const bool in = m < a.M && k < a.K;
          cp_async_16(dst, in ? a.q + m * a.ldq + k : a.q, in ? 16 : 0);
        }
      }
    };
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (u < cnt) issue(step_of(u), u);
      cp_async_commit();
    }
    const int sw = 4 * (g & 1);   // the swizzle of rows g, g + 8 and 8 nt + g
#pragma unroll 1
    for (int i = 0, slot = 0; i < cnt; ++i, slot = slot + 1 == U ? 0 : slot + 1) {
      cp_async_wait<U - 1>();
      __syncwarp();
      const uint8_t* sb = ring + (warp * U + slot) * kStageBytes;
      StepRegs<NT> r;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int pc = ((4 * h + t) ^ sw) * 16;
        r.w[0][h] = *reinterpret_cast<const uint4*>(sb + g * kStepK + pc);
        r.w[1][h] = *reinterpret_cast<const uint4*>(sb + (g + 8) * kStepK + pc);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          r.q[nt][h] = *reinterpret_cast<const uint4*>(sb + (kTileN + 8 * nt + g) * kStepK + pc);
      }
      __syncwarp();   // every lane has read the slot before it is refilled
      if (i + U < cnt) issue(step_of(i + U), slot);
      cp_async_commit();
      if constexpr (NT == 1) {
        mma_step<NT>(r, iacc);
      } else {
        mma_step_f16<NT>(r, facc);
        if ((i + 1) % kChunkSteps == 0 || i + 1 == cnt) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              iacc[nt][j] += __float2int_rn(facc[nt][j]);   // an exact integer below 2^24
              facc[nt][j] = 0.0f;
            }
        }
      }
    }
    cp_async_wait<0>();
  }

  // the four warps' sums through shared memory: element e = L * kElems + q
  // (lane L = 4g + t, fragment element q = 4 nt + i) is token
  // m = 8 nt + 2t + (i & 1) and channel n = c0 + g + 8 (i >> 1)
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) s_part[warp][lane][4 * nt + i] = iacc[nt][i];
  __syncthreads();
  int32_t sum[kPer];
#pragma unroll
  for (int r = 0; r < kPer; ++r) {
    const int e = tid + r * kThreads;
    sum[r] = 0;
    if (e < kOut) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) sum[r] += s_part[w][e / kElems][e % kElems];
    }
  }
  auto coords = [&](int e, int64_t& m, int64_t& n) {
    const int L = e / kElems, q = e % kElems;
    m = (q >> 2) * 8 + 2 * (L & 3) + (q & 1);
    n = c0 + (L >> 2) + 8 * ((q & 3) >> 1);
  };
  auto finish = [&](int e, int32_t v) {
    int64_t m, n;
    coords(e, m, n);
    if (m >= a.M || n >= a.N) return;
    if (a.acc_out != nullptr) a.acc_out[m * a.N + n] = v;
    if constexpr (kMode == 2) return;
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
      o = epilogue_bf16_res(v, as, ws, bf16_bits_to_float(rv));
    } else {
      o = epilogue_bf16(v, as, ws);
    }
    a.out[m * a.ldo + n] = static_cast<uint16_t>(o);
  };
  if (p.pieces == 1) {
#pragma unroll
    for (int r = 0; r < kPer; ++r)
      if (tid + r * kThreads < kOut) finish(tid + r * kThreads, sum[r]);
    return;
  }
  // a K piece: add the partial sums into the tile's accumulator; the last
  // piece to arrive reads the totals back, zeroes them and finishes the tile
#pragma unroll
  for (int r = 0; r < kPer; ++r) {
    const int e = tid + r * kThreads;
    int64_t m, n;
    coords(e, m, n);
    if (e < kOut && m < a.M && n < a.N) atomicAdd(p.acc + m * a.N + n, sum[r]);
  }
  __threadfence();
  __syncthreads();
  uint32_t* counter = p.cnt + blockIdx.x;
  if (tid == 0) {
    __threadfence();
    s_last = atomicAdd(counter, 1u) == static_cast<unsigned>(p.pieces - 1);
    __threadfence();
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
#pragma unroll
  for (int r = 0; r < kPer; ++r) {
    const int e = tid + r * kThreads;
    int64_t m, n;
    coords(e, m, n);
    if (e < kOut && m < a.M && n < a.N) {
      int32_t* src = p.acc + m * a.N + n;
      const int32_t v = __ldcg(src);
      __stcg(src, 0);
      finish(e, v);
    }
  }
  if (tid == 0) *counter = 0u;
}

// K pieces per channel tile: the caller's split, or for split 0 enough
// pieces that the tiles fill the GPU's SMs twice over (when there are too
// few tiles for that), each warp still getting at least one exact chunk.
int pieces_of(int64_t N, int64_t K, int split) {
  if (split >= 1) return split;
  const int64_t tiles = cdiv(N, kTileN);
  const int64_t target = 2 * static_cast<int64_t>(sm_count());
  if (2 * tiles >= target) return 1;
  const int64_t by_k = std::max<int64_t>(1, cdiv(K, kStepK) / (kWarps * kMinStepsPerWarp));
  return static_cast<int>(std::min<int64_t>(cdiv(target, tiles), by_k));
}

template <int NT, int kMode, int U, int kWarps>
cudaError_t launch_nt(const LinearArgs& a, cudaStream_t stream) {
  auto kernel = linear_stream_kernel<NT, kMode, U, kWarps>;
  const int smem = kWarps * U * (kTileN + 8 * NT) * kStepK;
  const cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kernel), smem);
  if (e != cudaSuccess) return e;
  StreamParams p{};
  p.a = a;
  p.steps = static_cast<int>(cdiv(a.K, kStepK));
  p.pieces = pieces_of(a.N, a.K, a.split);
  if (a.split == 0 && p.pieces > 1 && stream_workspace_bytes(a.M, a.N, a.K, 0) > a.ws_bytes)
    p.pieces = 1;   // the caller's scratch cannot hold the partial sums: whole K per CTA (same bits)
  if (p.pieces > 1) {
    const size_t acc_bytes =
        (static_cast<size_t>(a.M) * static_cast<size_t>(a.N) * 4 + 255) & ~static_cast<size_t>(255);
    p.acc = static_cast<int32_t*>(a.ws);
    p.cnt = reinterpret_cast<uint32_t*>(static_cast<char*>(a.ws) + acc_bytes);
  }
  const dim3 grid(static_cast<unsigned>(cdiv(a.N, kTileN)), static_cast<unsigned>(p.pieces));
  return launch_kernel(kernel, grid, dim3(kWarps * 32), static_cast<size_t>(smem), stream, a.no_pdl == 0, p);
}

template <int NT, int U, int W>
cudaError_t launch_modes(const LinearArgs& a, cudaStream_t stream) {
  if (a.acc_only) return launch_nt<NT, 2, U, W>(a, stream);
  if (a.res_rows != nullptr) return launch_nt<NT, 1, U, W>(a, stream);
  return launch_nt<NT, 0, U, W>(a, stream);
}

}  // namespace

// Workspace bytes of the weight-streaming kernel: the [M, N] int32
// accumulator and one arrival counter per 16-channel tile, when K is split
// between CTAs (an explicit split_k > 1, or the automatic choice for narrow
// weights).
size_t stream_workspace_bytes(int64_t M, int64_t N, int64_t K, int split) {
  if (pieces_of(N, K, split) <= 1) return 0;
  const size_t acc_bytes = (static_cast<size_t>(M) * static_cast<size_t>(N) * 4 + 255) & ~static_cast<size_t>(255);
  return acc_bytes + ((static_cast<size_t>(cdiv(N, kTileN)) * 4 + 255) & ~static_cast<size_t>(255));
}

cudaError_t launch_linear_stream(const LinearArgs& a, cudaStream_t stream) {
  // up to 8 rows: eight warps with two-step rings; 9-16 rows (the f16 MMA,
  // more registers per step): four warps with four-step rings
  return a.M <= 8 ? launch_modes<1, kRing, kWarps>(a, stream) : launch_modes<2, 4, 4>(a, stream);
}

}  // namespace prism
