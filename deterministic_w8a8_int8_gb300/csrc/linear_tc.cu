// linear_tc.cu -- W8A8 linear on the 5th-generation tensor cores (tcgen05).
//
// acc[m,n] = sum_k q[m,k] * w[n,k], exact int32, then the fixed-order
// epilogue y = bf16_rne(((float(acc) * a_scale[m]) * w_scale[n]) + r[m,n])
// (StartLux-Prism, "Bitwise consistency is not lossless quantization").
//
// sm_103a has no integer tcgen05 MMA, and its legacy int8 mma.sync pipe is
// slow, so the contraction runs on the f16 tensor pipe with exact arithmetic:
//   * every int8 value is exactly representable in f16 (11-bit significand);
//   * every product |q*w| <= 127*127 = 16129 is exact in the fp32 accumulator;
//   * a chunk of at most 1024 K-elements keeps every partial sum of products
//     below 1024 * 16129 < 2^24, so each fp32 partial is an exact integer no
//     matter in which order the tensor core adds the terms.
// The fp32 accumulator D lives in tensor memory (TMEM).  After each chunk the
// drain warps read D, convert it to int32 (exact) and add it into a second
// TMEM region I holding the int32 running sum; integer addition makes the
// result independent of chunking, tiling and split-K.  Where three tile widths
// fit the 512 TMEM columns (tiles of at most 160 B rows), D is double-buffered:
// chunk c accumulates in D[c % 2] while the workers drain D[(c - 1) % 2], so
// the tensor pipe does not wait for the drain.
//
// CTA roles (576 threads = 18 warps, one CTA per SM):
//   warp 17       lane 0 streams the raw int8 A and B tiles into a
//                 shared-memory staging ring (5 stages at width 256, up to 8
//                 for narrow tiles) with 2-D TMA loads;
//   warp 4        TMEM allocator; lane 0 issues every tcgen05.mma;
//   16 workers    (the other warps, four per TMEM lane quadrant) do all the
//                 rest: exact int8->f16 widening from the staging ring into
//                 128-byte-swizzled K-major f16 tiles (2 stages: one per
//                 group), in two groups of 8 warps that take alternate
//                 stages, so that one group's widening overlaps the other's
//                 wait for its data;
//                 at each 1024-K chunk boundary each warp drains its quarter
//                 of its quadrant's accumulator columns; at the end all 512
//                 threads write the tile out.
// mbarriers: s8_full (TMA transaction count), s8_empty and full (one arrival
// per warp of the stage's group), acc_empty (one per worker warp), empty and
// acc_full (tcgen05.commit).  Worker
// warps wait with all 32 lanes polling and agreeing on the outcome, so a warp
// never splits around a single polling lane.  Every
// wait is bounded by a 2-second global-timer limit; on expiry the CTA records
// kDevErrTimeout in the library's device error word and winds down.
//
// Two orientations:
//   normal (many rows)  A = q rows (tokens, 128 per tile), B = w rows
//                       (256 output channels per tile);
//   swapped (few rows)  A = w rows (128 channels), B = q rows (the tokens, one
//                       piece of up to 256), so small batches still fill the
//                       128-row MMA.
// Split-K reuses the integer-atomic / last-arriver protocol of the workspace.
#include <algorithm>
#include <atomic>
#include <climits>
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "tc_common.cuh"
#include "tc_sched.cuh"

namespace prism {

__device__ uint32_t g_kernel_error = 0;
// Limit of the pipeline waits (tests shorten it to drive the expiry path);
// the teardown waits always use kWaitLimitNs.
__device__ unsigned long long g_tc_wait_limit_ns = 2000000000ull;
// Test mode of the expiry path (prism_debug_wait_expiry): each CTA's MMA
// issuer withholds its first chunk-complete signal.
__device__ int g_tc_withhold = 0;

namespace {

constexpr int kMaxStages = 8;            // f16 operand / int8 staging stages (runtime count)
constexpr int kBM = 128;                  // A rows per tile = TMEM lanes
constexpr int kBNMax = 256;               // max B rows per tile = MMA N
constexpr int kBK = 64;                   // K elements per f16 operand slot (128 B of f16 per row)
constexpr int kChunkStages = 16;          // 16 * 64 = 1024 K per exact fp32 chunk
constexpr int kWorkerWarps = 16;          // convert, drain and write out; 4 per TMEM lane quadrant
constexpr int kWorkers = kWorkerWarps * 32;
constexpr int kMmaWarp = 4;               // TMEM allocator + MMA issuer
constexpr int kTmaWarp = 17;              // lane 0 issues the TMA loads
constexpr int kThreads = kWorkers + 64;   // 576: 18 warps, at most 96 registers each
constexpr int kStageA = kBM * 128;        // bytes of one f16 A stage
// One 216 KB region holds both rings: f16 operand stages first, then int8
// staging stages (the int8 ring gets whatever the f16 ring leaves, so that
// enough TMA loads are in flight to cover their latency).
constexpr int kRingRegion = 216 * 1024;
constexpr int kBarBytes = 512;
constexpr int kScaleBytes = 2 * 2 * kBNMax * 4;   // two items' a_scale and w_scale values
constexpr int kSmemBytes = 1024 + kRingRegion + kBarBytes + kScaleBytes;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColD = 0;             // fp32 chunk accumulator (single-buffered layout)
constexpr uint32_t kColI = 256;           // int32 running sum (single-buffered layout)
// The worker warps form two groups of 8 (two warps per TMEM lane quadrant)
// that widen alternate stages; a group thread converts 2 passes x 3
// segments of 16 int8 bytes per stage it owns.
constexpr int kGroupWarps = kWorkerWarps / 2;
constexpr int kSegPerThread = 3;
static_assert(2 * kSegPerThread * kGroupWarps * 32 == (kBM + kBNMax) * 4, "segment layout");
static_assert((kChunkStages & (kChunkStages - 1)) == 0, "chunk stages must be a power of two");
constexpr uint32_t kDevErrTimeout = 1u;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

struct TcParams {
  LinearArgs a;
  int swap;      // 0 normal, 1 swapped
  int bpiece;    // B rows per tile (multiple of 32, <= 256)
  int vec_io;    // vector epilogue loads/stores allowed (16-byte aligned out/residual, ldo/ldr % 8 == 0)
  int nst;       // f16 operand stages, each kSub slots of (128 + bpiece) x 128 bytes
  int nst8;      // int8 staging stages, each (128 + bpiece) x 64 kSub bytes
  SchedParams sp;  // work schedule (tc_sched.cuh); S counts stages of 64 kSub
  uint32_t* cnt;   // balanced schedule: arrival counters of the shared tiles (zero between calls)
  int32_t* acc;    // balanced schedule: one int32 accumulator per shared tile (zero between calls)
  int slot_elems;  // int32 elements of one accumulator (128 * bpiece)
};

// ------------------------------------------------------------ PTX helpers --
using tc::fence_proxy_async;
using tc::idesc_f16_f32;
using tc::mbar_arrive;
using tc::mbar_expect_tx;
using tc::mbar_init;
using tc::mbar_try_wait;
using tc::smem_desc_sw128;
using tc::tc_commit;
using tc::tc_fence_after;
using tc::tc_fence_before;
using tc::tc_mma;
using tc::tma_load_2d;
using tc::tmem_ld16;
using tc::tmem_st16;
using tc::tmem_wait_ld;
using tc::tmem_wait_st;

// Bounded wait (g_tc_wait_limit_ns, 2 s unless a test shortened it); an
// expiry raises kDevErrTimeout in g_kernel_error.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  return tc::mbar_wait_bounded(bar, parity, abort_flag, *reinterpret_cast<volatile unsigned long long*>(&g_tc_wait_limit_ns),
                               &g_kernel_error, kDevErrTimeout);
}
// Teardown wait: bounded by kWaitLimitNs, blind to the abort flag.
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity) {
  tc::mbar_wait_drain_bounded(bar, parity, kWaitLimitNs, &g_kernel_error, kDevErrTimeout);
}
// The same wait made by every lane of a warp: all lanes poll (one broadcast
// shared-memory read per poll) and the warp agrees on the outcome, so the warp
// never splits around a single polling lane.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
}

// Exact int8 -> f16 widening of 4 packed bytes: bias to u = b + 128 in
// [1, 255], place each byte under the f16 pattern of 1024 (0x6400 | u is the
// f16 of 1024 + u), subtract 1152 (0x6480) exactly.
__device__ __forceinline__ void widen4(uint32_t x, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = x ^ 0x80808080u;
  uint32_t p0, p1;
  asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(p0) : "r"(u), "r"(0x64646464u));
  asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(p1) : "r"(u), "r"(0x64646464u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(p0), "r"(0x64806480u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(p1), "r"(0x64806480u));
}

// 16-byte shared-memory load when pred holds, else zeros (predicated, no branch).
__device__ __forceinline__ uint4 ld_shared_v4_if(uint32_t addr, bool pred) {
  uint4 v;
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %5, 0;\n mov.u32 %0, 0;\n mov.u32 %1, 0;\n mov.u32 %2, 0;\n mov.u32 %3, 0;\n"
      " @p ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n}\n"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "r"(addr), "r"(static_cast<uint32_t>(pred)));
  return v;
}
// 16-byte shared-memory store when pred holds (predicated, no branch).
__device__ __forceinline__ void st_shared_v4_if(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                                bool pred) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %5, 0;\n @p st.shared.v4.u32 [%0], {%1,%2,%3,%4};\n}\n" ::"r"(addr),
      "r"(a), "r"(b), "r"(c), "r"(d), "r"(static_cast<uint32_t>(pred))
      : "memory");
}

// --------------------------------------------------------------- epilogue --

// Output of one accumulator round.  Lane trow of a TMEM quadrant holds the
// int32 results of A row a0 + trow for the 16 B rows b0 + 16 cb + j; in the
// swapped orientation A rows are output channels and B rows tokens, else the
// reverse.  s_as / s_ws hold the tile's a_scale (by token) and w_scale (by
// channel).  The residual values of the round are all loaded before any
// output is stored, so an in-place residual (residual == out) is safe.
// Kernel modes, each compiled into its own instance so that the ordinary
// path keeps its code: kTcPlain; kTcRows, the residual row of output row m
// is a.res_rows[m]; kTcAccOnly, only the exact int32 accumulators are
// written (a tensor-parallel rank's partial sums, scaled after their sum).
enum TcMode { kTcPlain = 0, kTcRows = 1, kTcAccOnly = 2 };

template <int kMode>
__device__ __forceinline__ void round_out(const TcParams& p, const float* s_as, const float* s_ws, int64_t a0,
                                          int64_t b0, int trow, int cb, const int32_t (&v)[16]) {
  const LinearArgs& a = p.a;
  if constexpr (kMode == kTcAccOnly) {
    if (p.swap) {
      const int64_t n = a0 + trow, mb = b0 + cb * 16;
      if (n >= a.N) return;
      const int jn = a.M - mb < 16 ? static_cast<int>(a.M - mb) : 16;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (j < jn) a.acc_out[(mb + j) * a.N + n] = v[j];
      return;
    }
    const int64_t m = a0 + trow, nb = b0 + cb * 16;
    if (m >= a.M) return;
    int32_t* dst = a.acc_out + m * a.N + nb;
    if (nb + 16 <= a.N && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        reinterpret_cast<int4*>(dst)[i] = make_int4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (nb + j < a.N) dst[j] = v[j];
    }
    return;
  }
  const bool res = a.residual != nullptr;
  if (p.swap) {
    const int64_t n = a0 + trow, mb = b0 + cb * 16;
    if (n >= a.N) return;
    const int jn = a.M - mb < 16 ? static_cast<int>(a.M - mb) : 16;
    const float ws = s_ws[trow];
    float r[16];
    if constexpr (kMode == kTcRows) {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        r[j] = 0.f;
        if (res && j < jn) {
          const uint16_t* rp = residual_row(a, mb + j);
          r[j] = bf16_bits_to_float(rp != nullptr ? rp[n] : kBf16NaN);
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j)
        r[j] = res && j < jn ? bf16_bits_to_float(a.residual[(mb + j) * a.ldr + n]) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (j < jn) {
        const float as = s_as[cb * 16 + j];
        const uint32_t o = res ? epilogue_bf16_res(v[j], as, ws, r[j]) : epilogue_bf16(v[j], as, ws);
        a.out[(mb + j) * a.ldo + n] = static_cast<uint16_t>(o);
        if (a.acc_out != nullptr) a.acc_out[(mb + j) * a.N + n] = v[j];
      }
    }
    return;
  }
  const int64_t m = a0 + trow, nb = b0 + cb * 16;
  if (m >= a.M) return;
  const float as = s_as[trow];
  const float* w = s_ws + cb * 16;
  if (p.vec_io && nb + 16 <= a.N) {
    uint4 r0 = make_uint4(0u, 0u, 0u, 0u), r1 = r0;
    if (res) {
      if constexpr (kMode == kTcRows) {
        const uint16_t* rp = residual_row(a, m);
        if (rp != nullptr) {
          r0 = *reinterpret_cast<const uint4*>(rp + nb);
          r1 = *reinterpret_cast<const uint4*>(rp + nb + 8);
        } else {
          r0 = r1 = make_uint4(kBf16NaN * 0x10001u, kBf16NaN * 0x10001u, kBf16NaN * 0x10001u, kBf16NaN * 0x10001u);
        }
      } else {
        r0 = *reinterpret_cast<const uint4*>(a.residual + m * a.ldr + nb);
        r1 = *reinterpret_cast<const uint4*>(a.residual + m * a.ldr + nb + 8);
      }
    }
    const uint32_t rw[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int j = 2 * i;
      o[i] = res ? (epilogue_bf16_res(v[j], as, w[j], bf16_lo(rw[i])) |
                    (epilogue_bf16_res(v[j + 1], as, w[j + 1], bf16_hi(rw[i])) << 16))
                 : (epilogue_bf16(v[j], as, w[j]) | (epilogue_bf16(v[j + 1], as, w[j + 1]) << 16));
    }
    *reinterpret_cast<uint4*>(a.out + m * a.ldo + nb) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4*>(a.out + m * a.ldo + nb + 8) = make_uint4(o[4], o[5], o[6], o[7]);
    if (a.acc_out != nullptr) {
#pragma unroll
      for (int j = 0; j < 16; ++j) a.acc_out[m * a.N + nb + j] = v[j];
    }
    return;
  }
  float r[16];
  if constexpr (kMode == kTcRows) {
    const uint16_t* rp = res ? residual_row(a, m) : nullptr;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      r[j] = res && nb + j < a.N ? bf16_bits_to_float(rp != nullptr ? rp[nb + j] : kBf16NaN) : 0.f;
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j) r[j] = res && nb + j < a.N ? bf16_bits_to_float(a.residual[m * a.ldr + nb + j]) : 0.f;
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if (nb + j < a.N) {
      const uint32_t o = res ? epilogue_bf16_res(v[j], as, w[j], r[j]) : epilogue_bf16(v[j], as, w[j]);
      a.out[m * a.ldo + nb + j] = static_cast<uint16_t>(o);
      if (a.acc_out != nullptr) a.acc_out[m * a.N + nb + j] = v[j];
    }
  }
}

// (m, n) of element j of a round, and whether it lies inside the matrix.
__device__ __forceinline__ bool round_elem(const TcParams& p, int64_t a0, int64_t b0, int trow, int cb, int j,
                                           int64_t& m, int64_t& n) {
  const int64_t ar = a0 + trow, br = b0 + cb * 16 + j;
  m = p.swap ? br : ar;
  n = p.swap ? ar : br;
  return m < p.a.M && n < p.a.N;
}

// Explicit split-K: add a round into the [M, N] int32 workspace.
__device__ __forceinline__ void round_atomic(const TcParams& p, int64_t a0, int64_t b0, int trow, int cb,
                                             const int32_t (&v)[16]) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    int64_t m, n;
    if (round_elem(p, a0, b0, trow, cb, j, m, n)) atomicAdd(p.a.ws_acc + m * p.a.N + n, v[j]);
  }
}

// A shared tile's accumulator is kept in TMEM order: element (trow, 16 cb +
// j) at word (16 cb + j) * 128 + trow, so that a warp's 32 lanes touch 128
// contiguous bytes.
__device__ __forceinline__ int slot_index(int trow, int cb, int j) { return (cb * 16 + j) * kBM + trow; }

// The last arriver's read-back of a shared tile in the swapped orientation
// (output channels on the TMEM lanes, tokens on the columns): unit u is
// column c = u / 32 and lanes 4 (u % 32) .. + 3 of the accumulator slot, one
// 16-byte load; its outputs are 4 consecutive channels n0 .. n0 + 3 of token
// row m = b0 + c.  A thread loads a batch of units (slots, then residuals)
// before it writes any, so their L2 round trips overlap; each output element
// is the same fixed-order epilogue as round_out, and an element's residual
// is read before its output is written (in-place residual).
template <int kMode>
__device__ __forceinline__ void readback_swap(const TcParams& p, const float* s_as, const float* s_ws, int64_t a0,
                                           int64_t b0, int bn, int32_t* tacc, int wt) {
  const LinearArgs& a = p.a;
  const bool res = kMode != kTcAccOnly && a.residual != nullptr;
  const int units = bn * (kBM / 4);
  constexpr int kB = 4;
  for (int u0 = wt; u0 < units; u0 += kB * kWorkers) {
    int4 v[kB];
    uint32_t r[kB][2];
#pragma unroll
    for (int b = 0; b < kB; ++b) {
      const int u = u0 + b * kWorkers;
      v[b] = make_int4(0, 0, 0, 0);
      r[b][0] = r[b][1] = 0u;
      if (u >= units) continue;
      const int c = u / (kBM / 4), r4 = (u % (kBM / 4)) * 4;
      v[b] = __ldcg(reinterpret_cast<const int4*>(tacc + c * kBM + r4));
      const int64_t m = b0 + c, n0 = a0 + r4;
      if (!res || m >= a.M) continue;
      const uint16_t* rp;
      if constexpr (kMode == kTcRows) {
        rp = residual_row(a, m);
      } else {
        rp = a.residual + m * a.ldr;
      }
      if (rp == nullptr) {
        r[b][0] = r[b][1] = kBf16NaN * 0x10001u;
      } else if (p.vec_io && n0 + 4 <= a.N) {
        const uint2 q = *reinterpret_cast<const uint2*>(rp + n0);
        r[b][0] = q.x;
        r[b][1] = q.y;
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (n0 + i < a.N) r[b][i >> 1] |= static_cast<uint32_t>(rp[n0 + i]) << (16 * (i & 1));
      }
    }
#pragma unroll
    for (int b = 0; b < kB; ++b) {
      const int u = u0 + b * kWorkers;
      if (u >= units) continue;
      const int c = u / (kBM / 4), r4 = (u % (kBM / 4)) * 4;
      __stcg(reinterpret_cast<int4*>(tacc + c * kBM + r4), make_int4(0, 0, 0, 0));
      const int64_t m = b0 + c, n0 = a0 + r4;
      if (m >= a.M || n0 >= a.N) continue;
      const int32_t vv[4] = {v[b].x, v[b].y, v[b].z, v[b].w};
      const bool quad = n0 + 4 <= a.N;
      if (a.acc_out != nullptr) {
        int32_t* dst = a.acc_out + m * a.N + n0;
        if (quad && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
          *reinterpret_cast<int4*>(dst) = v[b];
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (n0 + i < a.N) dst[i] = vv[i];
        }
      }
      if constexpr (kMode == kTcAccOnly) continue;
      const float as = s_as[c];
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float ws = s_ws[r4 + i];
        const uint16_t rb = static_cast<uint16_t>(r[b][i >> 1] >> (16 * (i & 1)));
        o[i] = res ? epilogue_bf16_res(vv[i], as, ws, bf16_bits_to_float(rb)) : epilogue_bf16(vv[i], as, ws);
      }
      uint16_t* op = a.out + m * a.ldo + n0;
      if (p.vec_io && quad) {
        *reinterpret_cast<uint2*>(op) = make_uint2(o[0] | (o[1] << 16), o[2] | (o[3] << 16));
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (n0 + i < a.N) op[i] = static_cast<uint16_t>(o[i]);
      }
    }
  }
}

// ------------------------------------------------------------------ kernel --

// Worker wt's share of an item's epilogue scales: a_scale of token wt of the
// tile (wt < 256) or w_scale of channel wt - 256 (0 beyond the tile or matrix).
__device__ __forceinline__ float item_scale(const TcParams& p, const Item& itm, int bn, int wt) {
  if (p.a.a_scale == nullptr) return 0.f;   // accumulators only: no scales
  const LinearArgs& a = p.a;
  const int64_t a0 = static_cast<int64_t>(itm.tx) * kBM, b0 = static_cast<int64_t>(itm.ty) * p.bpiece;
  if (wt < kBNMax) {
    const int64_t m = (p.swap ? b0 : a0) + wt;
    return wt < (p.swap ? bn : kBM) && m < a.M ? __ldg(a.a_scale + m) : 0.f;
  }
  const int i = wt - kBNMax;
  const int64_t n = (p.swap ? a0 : b0) + i;
  return i < (p.swap ? kBM : bn) && n < a.N ? __ldg(a.w_scale + n) : 0.f;
}

// kSub: f16 operand slots (64 K each) per stage.  Stages of 128 K (kSub = 2,
// narrow tiles) halve the barrier round trips, MMA-issue loop turns and TMA
// boxes per K (the boxes then carry 128-byte rows).
// kTA (swapped orientation, 128-K stages, narrow token tiles): the widened
// weight rows go to tensor memory instead of shared memory and the MMA reads
// its A operand from there.  Each worker thread then widens its own TMEM
// lane's row (the int8 A box arrives 128-byte swizzled, so a warp's 32 rows
// are read without bank conflicts) and only the token rows take the
// shared-memory round trip; per 128-K stage that removes 64 of the ~144 KB
// of shared-memory traffic of a 64-token tile.
template <int kMode, int kSub, bool kTA>
__global__ void __launch_bounds__(kThreads, 1)
    linear_tc_kernel(const __grid_constant__ TcParams p, const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB) {
  constexpr int kBK8 = kBK * kSub;               // K bytes per staging row
  constexpr int kS8A = kBM * kBK8;               // bytes of one int8 A box
  constexpr int kChunkL = kChunkStages / kSub;   // stages per 1024-K chunk
  extern __shared__ uint8_t smem_raw[];
  const LinearArgs& a = p.a;
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);
  const int nst = p.nst, nst8 = p.nst8;
  // f16 operand slot: A tile then B tile (kTA: the B tile alone)
  constexpr uint32_t kSlotB = kTA ? 0u : static_cast<uint32_t>(kStageA);
  const uint32_t kStageBytes = static_cast<uint32_t>(((kTA ? 0 : kBM) + p.bpiece) * 128);
  const uint32_t kS8Bytes = static_cast<uint32_t>((kBM + p.bpiece) * kBK8);
  const uint32_t sStage = base;                               // nst x kSub x (A tile | B tile), f16
  const uint32_t sS8 = sStage + nst * kSub * kStageBytes;     // nst8 x (A box | B box), int8
  const uint32_t bars = base + kRingRegion;
  uint8_t* bar_ptr = smem + (bars - base);
  const uint32_t bar_full = bars;                             // kMaxStages x 8 B each
  const uint32_t bar_empty = bars + 8 * kMaxStages;
  const uint32_t bar_s8_full = bars + 16 * kMaxStages;
  const uint32_t bar_s8_empty = bars + 24 * kMaxStages;
  const uint32_t bar_acc_full = bars + 32 * kMaxStages;      // 2 x 8 B: one per D buffer
  const uint32_t bar_acc_empty = bar_acc_full + 16;           // 2 x 8 B
  const uint32_t bar_done = bar_acc_full + 32;
  uint8_t* scalars = bar_ptr + (bar_done + 8 - bars);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(scalars);
  volatile int* s_abort = reinterpret_cast<volatile int*>(scalars + 4);
  int* s_last = reinterpret_cast<int*>(scalars + 8);
  float* s_as = reinterpret_cast<float*>(bar_ptr + kBarBytes);   // 2 x (kBNMax token + kBNMax channel scales)

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  // TMEM layout: double-buffered D[0] | D[1] | I when three widths fit, else D | I
  const bool dbuf = 3 * p.bpiece <= static_cast<int>(kTmemCols);
  const uint32_t col_i = dbuf ? 2u * static_cast<uint32_t>(p.bpiece) : kColI;
  // kTA: the widened A slots, 32 columns (64 f16 of K) per 64-K slot, after I
  const uint32_t col_a = col_i + static_cast<uint32_t>(p.bpiece);
  // B rows of piece ty that exist, rounded up to 32 (the MMA's N)
  auto tile_width = [&](int ty) -> int {
    const int64_t left = (p.swap ? a.M : a.N) - static_cast<int64_t>(ty) * p.bpiece;
    const int64_t rnd = (left + 31) & ~static_cast<int64_t>(31);
    return static_cast<int>(rnd < p.bpiece ? rnd : p.bpiece);
  };

  if (tid == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(bar_full + 8 * s, kGroupWarps);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int j = 0; j < nst8; ++j) {
      mbar_init(bar_s8_full + 8 * j, 1);
      mbar_init(bar_s8_empty + 8 * j, kGroupWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_acc_full + 8 * b, 1);
      mbar_init(bar_acc_empty + 8 * b, kWorkerWarps);
    }
    mbar_init(bar_done, 1);
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(s_tmem)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  // the prologue above touches no global data; inputs and workspace only now
  pdl_trigger();
  pdl_wait();

  if (warp == kMmaWarp) {
    // ======================= MMA issuer (one thread) =========================
    if (lane == 0) {
      const bool withhold = *reinterpret_cast<volatile int*>(&g_tc_withhold) != 0;
      int s = 0;
      uint32_t ph = 0;  // stage slot and its phase parity, advanced incrementally
      int c = -1;       // chunk counter over all items
      uint32_t dcol = kColD, dbar = 0;
      bool ok = true, issued = false;
      Item itm;
      for (int n = 0; ok && get_item(p.sp, n, itm); ++n) {
        const int nk = itm.k1 - itm.k0;
        const uint32_t idesc = idesc_f16_f32(tile_width(itm.ty));
        for (int it = 0; it < nk; ++it) {
          const int cpos = it & (kChunkL - 1);
          if (cpos == 0) {
            // chunk c reuses the D buffer of chunk c - 2 (double-buffered) or
            // c - 1: wait until the workers have drained it
            ++c;
            const int prev = c - (dbuf ? 2 : 1);
            dbar = dbuf ? static_cast<uint32_t>(c & 1) : 0u;
            dcol = dbuf && (c & 1) ? static_cast<uint32_t>(p.bpiece) : kColD;
            if (prev >= 0) {
              const uint32_t use = static_cast<uint32_t>(dbuf ? prev >> 1 : prev);
              if (!mbar_wait(bar_acc_empty + 8 * dbar, use & 1u, s_abort)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
          }
          if (!mbar_wait(bar_full + 8 * s, ph, s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int h = 0; h < kSub; ++h) {
            const uint64_t bd = smem_desc_sw128(sStage + (s * kSub + h) * kStageBytes + kSlotB);
            if constexpr (kTA) {
              // K = 16 is 8 columns of the slot's A rows in TMEM
              const uint32_t at = tmem + col_a + static_cast<uint32_t>(s * kSub + h) * 32u;
#pragma unroll
              for (int k = 0; k < kBK / 16; ++k)
                tc::tc_mma_ta(tmem + dcol, at + 8u * k, bd + 2 * k, idesc, (cpos | h | k) != 0 ? 1u : 0u);
            } else {
              const uint64_t ad = smem_desc_sw128(sStage + (s * kSub + h) * kStageBytes);
#pragma unroll
              for (int k = 0; k < kBK / 16; ++k)
                tc_mma(tmem + dcol, ad + 2 * k, bd + 2 * k, idesc, (cpos | h | k) != 0 ? 1u : 0u);
            }
          }
          issued = true;
          tc_commit(bar_empty + 8 * s);
          if ((cpos == kChunkL - 1 || it == nk - 1) && !(withhold && c == 0)) tc_commit(bar_acc_full + 8 * dbar);
          if (++s == nst) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (issued) {
        // every MMA issued above has completed before TMEM is released
        tc_commit(bar_done);
        mbar_wait_drain(bar_done, 0);
      }
    }
    __syncwarp();
  } else if (warp == kTmaWarp) {
    // ======================= TMA producer (one thread) ========================
    if (lane == 0) {
      const uint32_t tx = static_cast<uint32_t>(kS8A + kBK8 * p.bpiece);
      int j = 0;
      uint32_t ph = 0;
      int64_t issued = 0;
      bool ok = true;
      Item itm;
      for (int n = 0; ok && get_item(p.sp, n, itm); ++n) {
        const int32_t ya = itm.tx * kBM, yb = itm.ty * p.bpiece;
        for (int it = itm.k0; it < itm.k1; ++it) {
          if (!mbar_wait(bar_s8_empty + 8 * j, ph ^ 1u, s_abort)) {
            ok = false;
            break;
          }
          const uint32_t dst = sS8 + j * kS8Bytes;
          const int32_t x = it * kBK8;
          mbar_expect_tx(bar_s8_full + 8 * j, tx);
          tma_load_2d(dst, &tmA, x, ya, bar_s8_full + 8 * j);
          tma_load_2d(dst + kS8A, &tmB, x, yb, bar_s8_full + 8 * j);
          ++issued;
          if (++j == nst8) {
            j = 0;
            ph ^= 1u;
          }
        }
      }
      // Before the CTA may exit, every load issued must have landed: after an
      // expired wait the workers may stop consuming stages whose loads are
      // still in flight.  Stage x completes phase x / nst8 of slot x % nst8;
      // loads that were consumed pass at once.
      for (int64_t x = issued > nst8 ? issued - nst8 : 0; x < issued; ++x)
        mbar_wait_drain(bar_s8_full + 8 * static_cast<uint32_t>(x % nst8), static_cast<uint32_t>((x / nst8) & 1));
    }
    __syncwarp();
  } else {
    // ======================= workers (16 warps) ===============================
    // Conversion: worker thread wt owns 16-byte segment (wt % 4) of rows
    // wt / 4, wt / 4 + 128 and wt / 4 + 256 of the stacked [A | B] tile; the
    // shared-memory offsets are fixed, only K moves.
    // Drain: warp w reads TMEM lanes 32 (w % 4) .. +31; the four warps of a
    // quadrant take 16-column rounds j, j + 4, j + 8, ... of the accumulator,
    // and at an item's last chunk each thread writes out exactly the elements
    // it drained.
    // Every worker passes the same sequence of named barriers whatever
    // happens (a timed-out wait only skips work), so none can be left waiting.
    const int wi = warp < kMmaWarp ? warp : warp - 1;   // worker index 0..15
    const int wt = wi * 32 + lane;
    const int quad = warp & 3;
    const int slice = warp < kMmaWarp ? 0 : (warp - 1) / 4;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const int trow = quad * 32 + lane;                    // this thread's TMEM lane
    // widening: group grp (slices 0, 2 or 1, 3) owns the stages of its
    // parity in the CTA's stage sequence; group thread gt converts segment
    // gt % 4 of rows gt / 4 + 64 pass + 128 i of the stacked [A | B] tile
    const int grp = slice & 1;
    const int gt = (slice >> 1) * 128 + quad * 32 + lane;
    const int seg = gt & 3;
    // per segment of pass 0: offset of its 16 int8 bytes in a staging stage
    // (pass 1: + 64 rows), and per segment of both passes the offset of its
    // first 16-byte f16 chunk in an operand stage (the second is that ^ 16),
    // or ~0 when its B row lies beyond the current tile (set per item)
    uint32_t lo8[kSegPerThread], so[2 * kSegPerThread];
#pragma unroll
    for (int i = 0; i < kSegPerThread; ++i) {
      const int r = (gt >> 2) + i * kBM;
      const bool is_a = r < kBM;
      const int rr = is_a ? r : r - kBM;
      lo8[i] = (is_a ? 0u : static_cast<uint32_t>(kS8A)) + rr * kBK8 + seg * 16;
    }
    auto store_stage = [&](int s, int pass, const uint4 (&buf)[kSegPerThread]) {
      const uint32_t st_base = sStage + s * kStageBytes;
#pragma unroll
      for (int i = 0; i < kSegPerThread; ++i) {
        uint32_t w[8];
        widen4(buf[i].x, w[0], w[1]);
        widen4(buf[i].y, w[2], w[3]);
        widen4(buf[i].z, w[4], w[5]);
        widen4(buf[i].w, w[6], w[7]);
        const uint32_t o = so[pass * kSegPerThread + i];
        const bool valid = o != 0xFFFFFFFFu;   // rows beyond the tile lie outside the stage
        const uint32_t addr = st_base + (valid ? o : 0u);
        st_shared_v4_if(addr, w[0], w[1], w[2], w[3], valid);
        st_shared_v4_if(addr ^ 16u, w[4], w[5], w[6], w[7], valid);
      }
    };
    // kTA widening of the stage in staging slot j8 into operand slot s8op:
    // the group's two warps of a TMEM lane quadrant take the two 64-K halves
    // of their 32 weight rows (a thread its own lane's row: 64 bytes read
    // from the swizzled box, 32 columns stored); the group's 256 threads
    // share the token rows' 16-byte pieces (chunk u = row u / 8, K bytes
    // 16 (u % 8) ..), which go to the swizzled f16 B slot as before.
    auto widen_ta = [&](int j8, int s8op, uint32_t phase8, uint32_t phase, int bn) -> bool {
      constexpr int kTaB = 3;   // B pieces a thread: 96 rows x 8 pieces / 256 threads
      if (!mbar_wait_warp(bar_s8_full + 8 * j8, phase8, s_abort)) return false;
      const uint32_t s8 = sS8 + j8 * kS8Bytes;
      const int half = slice >> 1;
      uint4 av[4], bv[kTaB];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t c = static_cast<uint32_t>(4 * half + i);
        av[i] = ld_shared_v4_if(s8 + trow * 128u + ((c ^ static_cast<uint32_t>(trow & 7)) << 4), true);
      }
#pragma unroll
      for (int i = 0; i < kTaB; ++i) {
        const int u = gt + 256 * i;
        bv[i] = ld_shared_v4_if(s8 + kS8A + static_cast<uint32_t>(u) * 16u, (u >> 3) < bn);
      }
      // the operand slot's previous MMAs have completed
      if (!mbar_wait_warp(bar_empty + 8 * s8op, phase ^ 1u, s_abort)) return false;
      {
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          widen4(av[i].x, w[8 * i], w[8 * i + 1]);
          widen4(av[i].y, w[8 * i + 2], w[8 * i + 3]);
          widen4(av[i].z, w[8 * i + 4], w[8 * i + 5]);
          widen4(av[i].w, w[8 * i + 6], w[8 * i + 7]);
        }
        tc::tmem_st32(tmem + lane_base + col_a + static_cast<uint32_t>(s8op * kSub + half) * 32u, w);
      }
#pragma unroll
      for (int i = 0; i < kTaB; ++i) {
        const int u = gt + 256 * i;
        const int row = u >> 3, c = u & 7;
        uint32_t w[8];
        widen4(bv[i].x, w[0], w[1]);
        widen4(bv[i].y, w[2], w[3]);
        widen4(bv[i].z, w[4], w[5]);
        widen4(bv[i].w, w[6], w[7]);
        // 16 int8 K values of 64-K slot c / 4 become its f16 chunks 2 (c % 4)
        // and 2 (c % 4) + 1 of the row, 128-byte swizzled
        const uint32_t rb = sStage + static_cast<uint32_t>(s8op * kSub + (c >> 2)) * kStageBytes +
                            static_cast<uint32_t>(row) * 128u;
        const uint32_t f = static_cast<uint32_t>(2 * (c & 3)), sw = static_cast<uint32_t>(row & 7);
        st_shared_v4_if(rb + ((f ^ sw) << 4), w[0], w[1], w[2], w[3], row < bn);
        st_shared_v4_if(rb + (((f + 1u) ^ sw) << 4), w[4], w[5], w[6], w[7], row < bn);
      }
      tc::tmem_wait_st();
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_full + 8 * s8op);
      if (lane == 0) mbar_arrive(bar_s8_empty + 8 * j8);
      return true;
    };
    // Drain this warp's share of chunk gc (chunk lc of its item): I += int(D),
    // or, for the item's last chunk (out != nullptr), hand each round of final
    // int32 sums to out(cb, v).  Either way the D buffer is then handed back.
    auto drain = [&](int gc, int lc, int bn, auto&& out, bool last) -> bool {
      const uint32_t dbar = dbuf ? static_cast<uint32_t>(gc & 1) : 0u;
      const uint32_t use = static_cast<uint32_t>(dbuf ? gc >> 1 : gc);
      const uint32_t dcol = dbuf && (gc & 1) ? static_cast<uint32_t>(p.bpiece) : kColD;
      const bool got = mbar_wait_warp(bar_acc_full + 8 * dbar, use & 1u, s_abort);
      if (!got) return false;
      tc_fence_after();
      const int rounds = bn / 16;
      for (int cb = slice; cb < rounds; cb += 4) {
        uint32_t d[16], iv[16];
        tmem_ld16(tmem + lane_base + dcol + cb * 16, d);
        if (lc > 0) tmem_ld16(tmem + lane_base + col_i + cb * 16, iv);
        tmem_wait_ld();
        int32_t v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          v[j] = (lc > 0 ? static_cast<int32_t>(iv[j]) : 0) + __float2int_rn(__uint_as_float(d[j]));
        if (!last) {
          tmem_st16(tmem + lane_base + col_i + cb * 16, reinterpret_cast<const uint32_t(&)[16]>(v));
        } else {
          out(cb, v);
        }
      }
      if (!last) tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_acc_empty + 8 * dbar);
      return true;
    };
    auto no_out = [](int, const int32_t (&)[16]) {};

    bool ok = true;
    int gc = 0;                // chunk counter over all items
    int gst = 0;               // stage counter over all items
    int j = 0, s = 0;
    uint32_t ph8 = 0, ph = 0;  // staging / operand slots and phase parities
    // The epilogue scales of item n sit in buffer n % 2 of s_scale (token
    // scales then channel scales, 2 x kBNMax each); worker wt fills entry wt.
    // Item n + 1's are stored while item n finishes, and the next item-start
    // barrier orders them before any read.
    float* s_scale = s_as;
    {
      Item first;
      s_scale[wt] = get_item(p.sp, 0, first) ? item_scale(p, first, tile_width(first.ty), wt) : 0.f;
    }
    for (int n = 0;; ++n) {
      int bn, nk;
      {
        // (only n stays live through the stage loop; the item is looked up
        // again for its output)
        Item itm;
        if (!get_item(p.sp, n, itm)) break;
        // the previous item's output is finished and this item's scales are
        // in place
        asm volatile("bar.sync 1, %0;" ::"n"(kWorkers) : "memory");
        bn = tile_width(itm.ty);
        nk = itm.k1 > itm.k0 ? itm.k1 - itm.k0 : 0;
        if (a.residual != nullptr && itm.kind != 1) {
          // prefetch the item's residual tile into L2 for its epilogue
          const int64_t a0 = static_cast<int64_t>(itm.tx) * kBM, b0 = static_cast<int64_t>(itm.ty) * p.bpiece;
          const int64_t tok0 = p.swap ? b0 : a0, ch0 = p.swap ? a0 : b0;
          const int ntok = p.swap ? bn : kBM, nch = p.swap ? kBM : bn;
          const int lines = (nch * 2 + 127) / 128;  // 128-byte lines per token row
          for (int l = wt; l < ntok * lines; l += kWorkers) {
            const int r = l / lines;
            const int64_t m = tok0 + r, nn = ch0 + (l - r * lines) * 64;
            if constexpr (kMode == kTcRows) {
              const int64_t src = m < a.M ? __ldg(a.res_rows + m) : -1;
              if (nn < a.N && src >= 0 && src < a.M_res)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(a.residual + src * a.ldr + nn));
            } else if (m < a.M && nn < a.N) {
              asm volatile("prefetch.global.L2 [%0];" ::"l"(a.residual + m * a.ldr + nn));
            }
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 2 * kSegPerThread; ++i) {
        const int r = (gt >> 2) + (i % kSegPerThread) * kBM + (i / kSegPerThread) * 64;
        const bool is_a = r < kBM;
        const int rr = is_a ? r : r - kBM;
        so[i] = is_a || rr < bn ? (is_a ? 0u : static_cast<uint32_t>(kStageA)) + rr * 128 +
                                      static_cast<uint32_t>(((2 * seg) ^ (rr & 7)) * 16)
                                : 0xFFFFFFFFu;
      }
      const int nchunks = (nk + kChunkL - 1) / kChunkL;
      int next_drain = 0;  // next intermediate chunk to drain
      int next_trigger = kChunkL + nst - 1;
      for (int it = 0; it < nk && ok; ++it) {
        // chunk c's last MMA completes exactly when stage it - nst is
        // released, so drain it here, after the next chunk's first stages
        // have been prepared
        if (next_drain < nchunks - 1 && it == next_trigger) {
          ok = drain(gc + next_drain, next_drain, bn, no_out, false);
          ++next_drain;
          next_trigger += kChunkL;
          if (!ok) break;
        }
        if constexpr (kTA) {
          if (((gst + it) & 1) == grp) {
            ok = widen_ta(j, s, ph8, ph, bn);
            if (!ok) break;
          }
        } else if (((gst + it) & 1) == grp) {
          // this group's stage: widen it while the other group waits for
          // the next one
          ok = mbar_wait_warp(bar_s8_full + 8 * j, ph8, s_abort);
          if (!ok) break;
          uint4 buf[kSegPerThread];
          const uint32_t s8 = sS8 + j * kS8Bytes;
#pragma unroll
          for (int h = 0; h < kSub; ++h) {
#pragma unroll
            for (int pass = 0; pass < 2; ++pass) {
#pragma unroll
              for (int i = 0; i < kSegPerThread; ++i)  // rows beyond the tile lie outside the stage: skip
                buf[i] = ld_shared_v4_if(s8 + lo8[i] + pass * 64 * kBK8 + h * kBK,
                                         so[pass * kSegPerThread + i] != 0xFFFFFFFFu);
              if (h == 0 && pass == 0) {
                ok = mbar_wait_warp(bar_empty + 8 * s, ph ^ 1u, s_abort);
                if (!ok) break;
              }
              store_stage(s * kSub + h, pass, buf);
            }
            if (!ok) break;
          }
          if (!ok) break;
          fence_proxy_async();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_full + 8 * s);
          // released only now: every value read from the staging slot has
          // been consumed by the widening, so a TMA refill cannot overtake a
          // load
          if (lane == 0) mbar_arrive(bar_s8_empty + 8 * j);
        }
        if (++j == nst8) {
          j = 0;
          ph8 ^= 1u;
        }
        if (++s == nst) {
          s = 0;
          ph ^= 1u;
        }
      }
      while (ok && next_drain < nchunks - 1) {
        ok = drain(gc + next_drain, next_drain, bn, no_out, false);
        ++next_drain;
      }

      // ---- the item's last chunk: drain straight into its output
      Item itm;
      get_item(p.sp, n, itm);
      const int64_t a0 = static_cast<int64_t>(itm.tx) * kBM, b0 = static_cast<int64_t>(itm.ty) * p.bpiece;
      const float* sa = s_scale + (n & 1) * (2 * kBNMax);
      const float* sw = sa + kBNMax;
      float sc_next;  // loaded now, stored after the output (its latency overlaps)
      {
        Item nx;
        sc_next = get_item(p.sp, n + 1, nx) ? item_scale(p, nx, tile_width(nx.ty), wt) : 0.f;
      }
      const bool have = ok && nchunks > 0;
      const int glast = gc + nchunks - 1;
      if (itm.kind == 0) {
        if (have) {
          auto out = [&](int cb, const int32_t (&v)[16]) { round_out<kMode>(p, sa, sw, a0, b0, trow, cb, v); };
          ok = drain(glast, nchunks - 1, bn, out, true);
        }
      } else {
        // a K piece: this CTA's partial sums go to the workspace; the last CTA
        // to finish the tile sums all pieces and applies the epilogue
        int32_t* tacc = itm.kind == 2 ? p.acc + static_cast<int64_t>(itm.tile) * p.slot_elems : nullptr;
        if (have) {
          if (itm.kind == 1) {
            auto out = [&](int cb, const int32_t (&v)[16]) { round_atomic(p, a0, b0, trow, cb, v); };
            ok = drain(glast, nchunks - 1, bn, out, true);
          } else {
            auto out = [&](int cb, const int32_t (&v)[16]) {
#pragma unroll
              for (int jj = 0; jj < 16; ++jj) atomicAdd(tacc + slot_index(trow, cb, jj), v[jj]);
            };
            ok = drain(glast, nchunks - 1, bn, out, true);
          }
        }
        __threadfence();
        asm volatile("bar.sync 1, %0;" ::"n"(kWorkers) : "memory");
        int bf = 0, bl = 0;
        if (itm.kind == 2) shared_tile_ctas(p.sp, itm.tile, bf, bl);
        const unsigned target = itm.kind == 1 ? static_cast<unsigned>(a.split - 1) : static_cast<unsigned>(bl - bf);
        uint32_t* counter = itm.kind == 1 ? a.ws_count + itm.tile : p.cnt + itm.tile;
        // release: every worker's reductions reached thread 0 through the
        // barrier above; its fence makes them visible at GPU scope before its
        // arrival.  acquire: the last arriver's fence after the arrival
        // orders the read-back after every other CTA's reductions.
        if (wt == 0) {
          __threadfence();
          const bool last = atomicAdd(counter, 1u) == target;
          __threadfence();
          *s_last = last;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kWorkers) : "memory");
        if (*s_last && itm.kind == 2 && p.swap) {
          __threadfence();
          readback_swap<kMode>(p, sa, sw, a0, b0, bn, tacc, wt);
          if (wt == 0) *counter = 0u;
        } else if (*s_last) {
          __threadfence();
          for (int cb = slice; cb < bn / 16; cb += 4) {
            int32_t v[16];
            if (itm.kind == 1) {
#pragma unroll
              for (int jj = 0; jj < 16; ++jj) {
                int64_t m, nn;
                v[jj] = 0;
                if (round_elem(p, a0, b0, trow, cb, jj, m, nn)) {
                  int32_t* wp = a.ws_acc + m * a.N + nn;
                  v[jj] = __ldcg(wp);
                  __stcg(wp, 0);
                }
              }
            } else {
#pragma unroll
              for (int jj = 0; jj < 16; ++jj) v[jj] = __ldcg(tacc + slot_index(trow, cb, jj));
#pragma unroll
              for (int jj = 0; jj < 16; ++jj) __stcg(tacc + slot_index(trow, cb, jj), 0);
            }
            round_out<kMode>(p, sa, sw, a0, b0, trow, cb, v);
          }
          if (wt == 0) *counter = 0u;
        }
      }
      gc += nchunks;
      gst += nk;
      s_scale[((n + 1) & 1) * (2 * kBNMax) + wt] = sc_next;
    }
  }

  // ---- teardown: every role has finished its (bounded) work
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

inline int64_t cdiv(int64_t x, int64_t y) { return (x + y - 1) / y; }

}  // namespace

// Plan for the tensor-core path: orientation, B-piece width and the automatic
// split.  Few rows (M < 512) use the swapped orientation with the tokens as
// the MMA's N side (in equal pieces of at most 256); otherwise tokens fill the
// 128-row side.
struct TcPlan {
  int swap;
  int bpiece;
  int sub;       // f16 operand slots of 64 K per stage (see linear_tc_kernel)
  int64_t grid_x, grid_y;
};

static TcPlan tc_plan(int64_t M, int64_t N, int64_t K) {
  TcPlan pl{};
  pl.swap = M < 512 ? 1 : 0;
  if (pl.swap) {
    // tokens split into equal pieces (multiples of 32, at most 256) so that no
    // narrow leftover piece piles up on a few SMs
    const int64_t pieces = cdiv(M, kBNMax);
    pl.bpiece = static_cast<int>(cdiv(cdiv(M, pieces), 32) * 32);
    pl.grid_x = cdiv(N, kBM);
    pl.grid_y = cdiv(M, pl.bpiece);
  } else {
    pl.bpiece = 256;
    pl.grid_x = cdiv(M, kBM);
    pl.grid_y = cdiv(N, 256);
  }
  // two slots per stage for tiles up to 96 wide: 2 f16 stages and at least 3
  // int8 stages of 128 K fit the 216 KB ring (measured: 16-96 rows 7-13 %
  // faster; at 128 and 160 wide only 2 int8 stages fit, and the smaller
  // staging depth made them 7 % slower)
  pl.sub = pl.bpiece <= 96 && K >= 128 ? 2 : 1;
  return pl;
}

// Streaming multiprocessors of the current device (152 on a GB300), queried
// once per device; the balanced schedule runs one CTA per SM.  Without a
// usable device (a host that only sizes workspaces) the GB300's count is
// taken, so that sizes agree with the launches on that part.
int sm_count() {
  constexpr int kMaxDev = 64, kDefault = 152;
  static std::atomic<int> cache[kMaxDev];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
    cudaGetLastError();
    return kDefault;
  }
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      return kDefault;
    }
    n = std::min(n, 512);   // keeps the schedule's unit arithmetic within int32
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// The balanced schedule (tc_sched.cuh) over this device's SMs; a share of
// less than one 1024-K chunk per CTA is not worth its partial sums.
static TcSched tc_balanced(int64_t T, int64_t S, int sub) {
  return tc_balanced_sched(T, S, kChunkStages / sub, sm_count());
}

// Workspace of the balanced schedule: tile counters, then one int32
// accumulator per shared tile (all zero between calls); none when no tile is
// shared.
static size_t tc_balanced_bytes(int64_t M, int64_t N, int64_t K, size_t* counter_bytes) {
  const TcPlan pl = tc_plan(M, N, K);
  const TcSched sc = tc_balanced(pl.grid_x * pl.grid_y, cdiv(K, kBK * pl.sub), pl.sub);
  if (sc.R == 0 || sc.G == sc.R) {
    if (counter_bytes != nullptr) *counter_bytes = 0;
    return 0;
  }
  const size_t cb = (static_cast<size_t>(sc.R) * 4 + 255) & ~static_cast<size_t>(255);
  if (counter_bytes != nullptr) *counter_bytes = cb;
  return cb + static_cast<size_t>(sc.R) * kBM * pl.bpiece * 4;
}

// Workspace of explicit split-K (int32 atomics): the [M, N] accumulator, then
// one counter per tile (counted at 128 x 128, which covers both kernels' tiles).
static size_t atomic_bytes(int64_t M, int64_t N) {
  const size_t tiles = static_cast<size_t>(cdiv(M, 128) * cdiv(N, 128));
  return ((static_cast<size_t>(M) * static_cast<size_t>(N) * 4 + 255) & ~static_cast<size_t>(255)) +
         ((tiles * 4 + 255) & ~static_cast<size_t>(255));
}

using EncodeTiledFn = PFN_cuTensorMapEncodeTiled_v12000;

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
    tried = true;
  }
  return fn;
}

// Row-major int8 [rows, K] matrix with row stride ld bytes, read in boxes of
// box_k K-bytes x box_rows rows (128-byte swizzled when swz, which needs
// box_k = 128); out-of-range rows and K read as zero.
static cudaError_t make_map(CUtensorMap* m, const int8_t* ptr, int64_t rows, int64_t K, int64_t ld, int box_rows,
                            int box_k, bool swz = false) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_k), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swz ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Operand stages of the tensor-memory A variant: as many as the TMEM columns
// beside D[0] | D[1] | I hold (32 a 64-K slot), at most 4; 0 where the
// variant does not apply (the normal orientation, 64-K stages, tiles too
// wide for a double-buffered D).  PRISM_TC_A=smem keeps every call on the
// shared-memory A operand (a diagnostic: both give the same bits).
static int ta_stages(const TcPlan& pl) {
  if (!pl.swap || pl.sub != 2 || 3 * pl.bpiece > static_cast<int>(kTmemCols)) return 0;
  const char* e = std::getenv("PRISM_TC_A");
  if (e != nullptr && std::strcmp(e, "smem") == 0) return 0;
  const int cols = (static_cast<int>(kTmemCols) - 3 * pl.bpiece) / (32 * pl.sub);
  return cols >= 2 ? std::min(cols, 4) & ~1 : 0;   // an even number of slots (see launch_linear_tc)
}

static cudaError_t launch_linear_tc(const LinearArgs& a, cudaStream_t stream) {
  const TcPlan pl = tc_plan(a.M, a.N, a.K);
  const int ta = ta_stages(pl);
  auto kernel = ta > 0 ? (a.acc_only                ? linear_tc_kernel<kTcAccOnly, 2, true>
                          : a.res_rows != nullptr ? linear_tc_kernel<kTcRows, 2, true>
                                                  : linear_tc_kernel<kTcPlain, 2, true>)
                : pl.sub == 2 ? (a.acc_only                ? linear_tc_kernel<kTcAccOnly, 2, false>
                                 : a.res_rows != nullptr ? linear_tc_kernel<kTcRows, 2, false>
                                                         : linear_tc_kernel<kTcPlain, 2, false>)
                              : (a.acc_only                ? linear_tc_kernel<kTcAccOnly, 1, false>
                                 : a.res_rows != nullptr ? linear_tc_kernel<kTcRows, 1, false>
                                                         : linear_tc_kernel<kTcPlain, 1, false>);
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kernel), kSmemBytes);
  if (e != cudaSuccess) return e;
  TcParams p{};
  p.a = a;
  p.swap = pl.swap;
  p.bpiece = pl.bpiece;
  const uintptr_t ob = reinterpret_cast<uintptr_t>(a.out), rb = reinterpret_cast<uintptr_t>(a.residual);
  const uintptr_t wb = reinterpret_cast<uintptr_t>(a.w_scale);
  p.vec_io = (ob % 16 == 0) && (a.ldo % 8 == 0) && (wb % 16 == 0) &&
             (a.residual == nullptr || ((rb % 16 == 0) && (a.ldr % 8 == 0)));
  // f16 operand stages: an even number, so that every operand slot is only
  // ever written by one of the two worker groups (stage parity = slot
  // parity).  With three slots the groups took turns on each slot, and about
  // one full-size call in 15 to 40 had one tile whose products for one stage
  // used wrong values in the rows one group's warps write first (the first
  // pass); with an even count no call of 820 across five shapes did.
  // Four where four still leave three staging stages (tiles up to 160
  // wide), else two.
  const int f16_stage = pl.sub * ((ta > 0 ? 0 : kBM) + pl.bpiece) * 128, s8_stage = (kBM + pl.bpiece) * kBK * pl.sub;
  p.nst = ta > 0 ? ta : ((kRingRegion - 4 * f16_stage) / s8_stage >= 3 ? 4 : 2);
  p.nst8 = std::min(kMaxStages, (kRingRegion - p.nst * f16_stage) / s8_stage);
  p.sp.split = a.split;
  p.sp.gx = static_cast<int>(pl.grid_x);
  p.sp.gy = static_cast<int>(pl.grid_y);
  p.sp.a_w = pl.swap ? 1 : 0;
  p.sp.T = static_cast<int>(pl.grid_x * pl.grid_y);
  p.sp.S = static_cast<int>(cdiv(a.K, kBK * pl.sub));
  dim3 grid;
  if (a.split >= 1) {
    // explicit split-K: one CTA per tile and K piece; int32 atomics when split
    p.sp.sched = 0;
    if (a.split > 1) {
      p.a.ws_acc = static_cast<int32_t*>(a.ws);
      p.a.ws_count = reinterpret_cast<uint32_t*>(
          static_cast<char*>(a.ws) +
          ((static_cast<size_t>(a.M) * static_cast<size_t>(a.N) * 4 + 255) & ~static_cast<size_t>(255)));
    }
    grid = dim3(static_cast<unsigned>(pl.grid_x), static_cast<unsigned>(pl.grid_y), static_cast<unsigned>(a.split));
  } else {
    // automatic: the balanced schedule, falling back to whole tiles in rounds
    // when the caller's workspace cannot hold the shared tiles' partials
    p.sp.sched = 1;
    TcSched sc = tc_balanced(p.sp.T, p.sp.S, pl.sub);
    size_t cb = 0;
    const size_t need = tc_balanced_bytes(a.M, a.N, a.K, &cb);
    if (need > 0 && need > a.ws_bytes) {
      const int g = sm_count();
      sc = TcSched{g, static_cast<int>(cdiv(p.sp.T, g)), 0};
    }
    if (sc.R > 0 && need > 0) {
      p.cnt = static_cast<uint32_t*>(a.ws);
      p.acc = reinterpret_cast<int32_t*>(static_cast<char*>(a.ws) + cb);
    }
    p.sp.W = sc.W;
    p.sp.R = sc.R;
    p.slot_elems = kBM * pl.bpiece;
    const int64_t ctas = sc.R > 0 ? sc.G : std::min<int64_t>(sc.G, p.sp.T);
    grid = dim3(static_cast<unsigned>(ctas), 1, 1);
  }
  CUtensorMap tmA, tmB;
  const int8_t* Am = pl.swap ? a.w : a.q;
  const int8_t* Bm = pl.swap ? a.q : a.w;
  e = make_map(&tmA, Am, pl.swap ? a.N : a.M, a.K, pl.swap ? a.ldw : a.ldq, kBM, kBK * pl.sub, ta > 0);
  if (e != cudaSuccess) return e;
  e = make_map(&tmB, Bm, pl.swap ? a.M : a.N, a.K, pl.swap ? a.ldq : a.ldw, pl.bpiece, kBK * pl.sub);
  if (e != cudaSuccess) return e;
  return launch_kernel(kernel, grid, dim3(kThreads), kSmemBytes, stream, a.no_pdl == 0, p, tmA, tmB);
}

// PRISM_LINEAR_PATH=mma routes the linear to the mma.sync s8 kernel and
// PRISM_LINEAR_PATH=tc keeps calls of few rows on the tcgen05 kernel (both
// diagnostics for cross-checking the contraction kernels); read per call.
static bool path_is(const char* name) {
  const char* s = std::getenv("PRISM_LINEAR_PATH");
  return s != nullptr && std::strcmp(s, name) == 0;
}
static bool use_mma_path() { return path_is("mma"); }
// Calls of at most kGemvMaxM token rows stream the weights through the dp4a
// kernel (linear_gemv.cu), calls of up to kStreamMaxM rows through the
// mma.sync weight-streaming kernel (linear_stream.cu), more rows run on the
// tcgen05 kernel.  PRISM_LINEAR_PATH names a kernel instead (diagnostics;
// every kernel gives the same bits): "tc" or "mma" for every shape,
// "gemv" for calls of up to kGemvPathMaxM rows, "stream" for calls of up to
// kStreamMaxM rows.
constexpr int64_t kGemvMaxM = 2;
constexpr int64_t kGemvPathMaxM = 8;
constexpr int64_t kStreamMaxM = 16;
static bool use_gemv_path(int64_t M) {
  if (path_is("tc") || path_is("mma") || path_is("stream")) return false;
  return M <= (path_is("gemv") ? kGemvPathMaxM : kGemvMaxM);
}
static bool use_stream_path(int64_t M) {
  if (M > kStreamMaxM || path_is("tc") || path_is("mma") || use_gemv_path(M)) return false;
  return true;
}

int linear_kernel_kind(int64_t M, int64_t N, int64_t K) {
  (void)K;
  if (M <= 0 || N <= 0) return 0;
  if (use_mma_path()) return 1;
  if (use_gemv_path(M)) return 4;
  if (use_stream_path(M)) return 5;
  return tc_plan(M, N, K).swap ? 3 : 2;
}

// The packed 4-bit weights of W4A8 stream through the dp4a kernel for calls
// of up to kGemvPathMaxM rows unless another kernel is forced.
bool linear_w4_packed(int64_t M) {
  return M <= kGemvPathMaxM && !path_is("tc") && !path_is("mma") && !path_is("stream");
}

int linear_auto_split(int64_t M, int64_t N, int64_t K) {
  return use_mma_path() ? mma_auto_split(M, N, K) : 0;
}

size_t linear_workspace_bytes(int64_t M, int64_t N, int64_t K, int split) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  if (use_gemv_path(M)) return 0;
  if (use_stream_path(M)) return stream_workspace_bytes(M, N, K, split);
  if (use_mma_path() && split == 0) split = mma_auto_split(M, N, K);
  if (split == 0) return tc_balanced_bytes(M, N, K, nullptr);
  return split > 1 ? atomic_bytes(M, N) : 0;
}

size_t linear_workspace_zero_bytes(int64_t M, int64_t N, int64_t K, int split, size_t cap) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  if (use_gemv_path(M)) return 0;
  if (use_stream_path(M)) {
    const size_t need = stream_workspace_bytes(M, N, K, split);
    if (split == 0) return need <= cap ? need : 0;  // beyond cap: whole K per CTA
    return need <= cap ? need : SIZE_MAX;
  }
  if (use_mma_path() && split == 0) split = mma_auto_split(M, N, K);
  if (split == 0) {
    const size_t need = tc_balanced_bytes(M, N, K, nullptr);
    return need <= cap ? need : 0;  // beyond cap the call runs whole tiles only
  }
  const size_t need = split > 1 ? atomic_bytes(M, N) : 0;
  return need <= cap ? need : SIZE_MAX;
}

cudaError_t launch_linear(const LinearArgs& a, cudaStream_t stream) {
  if (use_gemv_path(a.M)) return launch_linear_gemv(a, stream);
  if (use_stream_path(a.M)) return launch_linear_stream(a, stream);
  if (!use_mma_path()) return launch_linear_tc(a, stream);
  LinearArgs b = a;
  if (b.split == 0) b.split = mma_auto_split(a.M, a.N, a.K);
  if (b.split > 1) {
    b.ws_acc = static_cast<int32_t*>(a.ws);
    b.ws_count = reinterpret_cast<uint32_t*>(
        static_cast<char*>(a.ws) +
        ((static_cast<size_t>(a.M) * static_cast<size_t>(a.N) * 4 + 255) & ~static_cast<size_t>(255)));
  }
  return launch_linear_mma(b, stream);
}

cudaError_t set_tc_wait_expiry(unsigned long long limit_ns, int withhold) {
  cudaError_t e = cudaMemcpyToSymbol(g_tc_wait_limit_ns, &limit_ns, sizeof limit_ns);
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_tc_withhold, &withhold, sizeof withhold);
  return e;
}

cudaError_t read_and_clear_kernel_error(uint32_t* out) {
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_kernel_error, sizeof v);
  if (e != cudaSuccess) return e;
  if (v != 0) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_kernel_error, &zero, sizeof zero);
  }
  *out = v;
  return e;
}

}  // namespace prism
