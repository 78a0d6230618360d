// linear_f16.cu -- the W8A8 linear on the tcgen05 tensor cores with the int8
// codes held as binary16 values ("f16 codes") in global memory.
//
// acc[m,n] = sum_k q[m,k] * w[n,k] exactly in int32, then the fixed-order
// epilogue y = bf16_rne(((float(acc) * a_scale[m]) * w_scale[n]) + r[m,n])
// (StartLux-Prism, "Bitwise consistency is not lossless quantization").
//
// sm_103a has no integer tcgen05 MMA; its f16 MMA is exact on these integers:
//   * a code in [-127, 127] is exact in binary16;
//   * a product |q w| <= 127 * 127 = 16129 is exact in the fp32 accumulator;
//   * a chunk of at most 1024 K-elements keeps every partial sum below
//     1024 * 16129 < 2^24, so the fp32 accumulator holds exact integers in any
//     summation order.
// The int8-operand kernel (linear_tc.cu) widens every stage from int8 to f16
// in shared memory, and that pass competes with the MMA for shared-memory
// bandwidth.  Here the codes are stored as binary16 (the weight once at load
// time by prism_codes_to_f16, the activations by the quantiser), so TMA drops
// each 64-K stage straight into the MMA's 128-byte-swizzled K-major operand
// layout and no thread touches the operands.  The price is twice the operand
// bytes, which compute-bound shapes (hundreds of token rows and more) afford.
//
// CTA (576 threads, one per SM, persistent over the work items of tc_sched.cuh):
//   warp 0       lane 0: TMA producer -- per 64-K stage, the A tile (128 rows
//                x 128 bytes) and the B tile (bpiece rows x 128 bytes) into a
//                4-8 stage ring (216 KB);
//   warp 1       TMEM allocator (512 columns: two fp32 accumulator buffers of
//                up to 256 columns) and, lane 0, the MMA issuer: 4 MMAs of
//                K = 16 per stage, a commit that frees the stage, and a
//                commit at each chunk's end;
//   warps 2-17   epilogue: warp w reads TMEM lane quadrant w % 4, and the four
//                warps of a quadrant split the tile's 16-column groups
//                (group cb belongs to slice cb % 4).  Each thread keeps the
//                int32 running sums of its elements (up to 4 groups of 16)
//                in registers, adds every drained chunk into them, and at the
//                item's end writes the output, or adds its partial sums into
//                the shared tile's slot (tc_sched.cuh).
// Chunk c accumulates into buffer c % 2 while the epilogue drains chunk c - 1,
// so the tensor pipe never waits for a drain.
//
// Orientation: many rows (M >= 512) put 128 tokens on the MMA's rows and 256
// output channels on its N side; fewer rows put 128 output channels on the
// rows and the tokens on N, in equal pieces of at most 256.
//
// Every mbarrier wait is bounded (2 s of global time; prism_debug_wait_expiry
// shortens it for tests and withholds one signal so that a wait expires).  On expiry the CTA raises
// PRISM_DEVSTATUS_WAIT_TIMEOUT and winds down: the producer stops issuing and
// then waits (bounded by 2 s, whatever the debug limit) until every TMA load
// it issued has landed, the MMA thread waits for its last commit before TMEM
// is released, and the epilogue warps take every named barrier together (the
// decision to skip a tile's output is a barrier reduction, so no warp is left
// waiting).  Outputs of such a call are invalid, and a workspace it used must
// be zeroed again before its next use.
#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "tc_common.cuh"
#include "tc_sched.cuh"

namespace prism {

__device__ uint32_t g_f16_status = 0;
__device__ unsigned long long g_f16_wait_limit_ns = 2000000000ull;
// Test mode of the expiry path (prism_debug_wait_expiry): each CTA's MMA
// issuer withholds its first chunk-complete signal, so the first drain wait
// cannot complete and expires after g_f16_wait_limit_ns.
__device__ int g_f16_withhold = 0;

namespace {

using tc::mbar_arrive;
using tc::mbar_init;
using tc::mbar_try_wait;
using tc::tc_fence_after;
using tc::tc_fence_before;

constexpr int kBM = 128;                 // A rows per tile = TMEM lanes
constexpr int kBNMax = 256;              // B rows per tile at most = MMA N
constexpr int kBK = 64;                  // K elements per stage: one 128-byte swizzled row of f16
constexpr int kChunk = 16;               // stages per exact fp32 chunk (1024 K)
constexpr int kEpiWarps = 16;
constexpr int kEpi = kEpiWarps * 32;     // 512 epilogue threads
constexpr int kThreads = kEpi + 64;      // 576
constexpr int kTmaWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kGroups = kBNMax / 16 / 4; // 16-column groups per epilogue thread: 4
constexpr int kRing = 216 * 1024;
constexpr int kMaxStages = 8;
constexpr int kBarBytes = 256;
// the epilogue scales of two items: per item kBNMax token scales (a_scale)
// and kBNMax channel scales (w_scale)
constexpr int kScaleBytes = 2 * 2 * kBNMax * 4;
constexpr int kSmemBytes = 1024 + kRing + kBarBytes + kScaleBytes;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kStatusTimeout = 1u;
constexpr unsigned long long kDrainLimitNs = 2000000000ull;
static_assert(kGroups * 4 * 16 == kBNMax, "column groups");

struct HParams {
  const float* a_scale;      // [M]
  const float* w_scale;      // [N]
  const uint16_t* residual;  // [M, N] bf16 or null
  int64_t ldr;
  uint16_t* out;             // [M, N] bf16
  int64_t ldo;
  int32_t* acc_out;          // [M, N] dense int32 or null
  int64_t M, N, K;
  int swap;                  // 0: tokens on the MMA rows; 1: channels on the MMA rows
  int bpiece;                // B rows per tile (multiple of 32, <= 256)
  int vec_io;                // out / residual rows and w_scale 16-byte aligned, ld % 8 == 0
  int nst;                   // ring stages
  SchedParams sp;
  uint32_t* cnt;             // automatic: arrival counters of the shared tiles
  int32_t* slots;            // automatic: piece slots of 128 x bpiece int32 (shared_tile_slots in
                             // tc_sched.cuh: balanced, one per (shared tile st, CTA b) pair at index st + b;
                             // lockstep rounds, P per remainder tile)
  int32_t* ws_acc;           // explicit split: [M, N] int32 accumulator
  uint32_t* ws_count;        // explicit split: per-tile arrival counters
};

// Wait made by one thread (TMA producer, MMA issuer); the limit is read only
// when the phase has not completed at the first look.
__device__ __forceinline__ bool wait1(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  return tc::mbar_wait_bounded(bar, parity, abort_flag,
                               *reinterpret_cast<volatile unsigned long long*>(&g_f16_wait_limit_ns),
                               &g_f16_status, kStatusTimeout);
}
// Wait made by all lanes of a warp, which agree on the outcome.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  return __all_sync(0xffffffffu, wait1(bar, parity, abort_flag));
}
// Teardown wait: bounded by kDrainLimitNs, blind to the abort flag.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity) {
  tc::mbar_wait_drain_bounded(bar, parity, kDrainLimitNs, &g_f16_status, kStatusTimeout);
}
// Named barrier 1 over the epilogue warps, returning whether any thread
// passed `pred` (the same answer in every thread).
__device__ __forceinline__ bool epi_barrier_any(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, %2, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "n"(kEpi)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void epi_barrier() { asm volatile("bar.sync 1, %0;" ::"n"(kEpi) : "memory"); }

// The output of one 16-column group: lane trow of a TMEM quadrant holds the
// int32 sums of A row a0 + trow with the 16 B rows b0 + 16 cb + j.  In the
// normal orientation A rows are tokens and B rows channels, in the swapped
// one the reverse.  Each element's residual is read before its output is
// written by the same thread, so residual == out is safe.
// s_tok / s_ch: the item's token scales (a_scale of token t0 + i at i) and
// channel scales (w_scale of channel c0 + i at i) in shared memory.
__device__ __forceinline__ void emit_group(const HParams& p, const float* s_tok, const float* s_ch, int64_t a0,
                                           int64_t b0, int trow, int cb, const int32_t (&v)[16]) {
  // The group goes out in two halves of 8 elements, and the residual values
  // of a half are loaded before its first output store: the stores may alias
  // the residual, so a load placed after one would wait for a memory round
  // trip of its own.  The scales come from shared memory.
  const bool res = p.residual != nullptr;
  if (p.swap) {
    const int64_t n = a0 + trow;
    if (n >= p.N) return;
    const float ws = s_ch[trow];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t mb = b0 + cb * 16 + 8 * h;
      uint32_t rb[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        rb[j] = res && mb + j < p.M ? static_cast<uint32_t>(p.residual[(mb + j) * p.ldr + n]) : 0u;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int64_t m = mb + j;
        if (m < p.M) {
          const int32_t x = v[8 * h + j];
          const float as = s_tok[cb * 16 + 8 * h + j];
          const uint32_t o = res ? epilogue_bf16_res(x, as, ws, bf16_bits_to_float(static_cast<uint16_t>(rb[j])))
                                 : epilogue_bf16(x, as, ws);
          p.out[m * p.ldo + n] = static_cast<uint16_t>(o);
          if (p.acc_out != nullptr) p.acc_out[m * p.N + n] = x;
        }
      }
    }
    return;
  }
  const int64_t m = a0 + trow, nb = b0 + cb * 16;
  if (m >= p.M) return;
  const float as = s_tok[trow];
  const float* w = s_ch + cb * 16;
  if (p.vec_io && nb + 16 <= p.N) {
    uint4 rv[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
    if (res) {
      rv[0] = *reinterpret_cast<const uint4*>(p.residual + m * p.ldr + nb);
      rv[1] = *reinterpret_cast<const uint4*>(p.residual + m * p.ldr + nb + 8);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t rw[4] = {rv[h].x, rv[h].y, rv[h].z, rv[h].w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int j = 8 * h + 2 * i;
        o[i] = res ? (epilogue_bf16_res(v[j], as, w[j], bf16_lo(rw[i])) |
                      (epilogue_bf16_res(v[j + 1], as, w[j + 1], bf16_hi(rw[i])) << 16))
                   : (epilogue_bf16(v[j], as, w[j]) | (epilogue_bf16(v[j + 1], as, w[j + 1]) << 16));
      }
      *reinterpret_cast<uint4*>(p.out + m * p.ldo + nb + 8 * h) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (p.acc_out != nullptr) {
#pragma unroll
      for (int j = 0; j < 16; ++j) p.acc_out[m * p.N + nb + j] = v[j];
    }
    return;
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t rb[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      rb[j] = res && nb + 8 * h + j < p.N ? static_cast<uint32_t>(p.residual[m * p.ldr + nb + 8 * h + j]) : 0u;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int64_t n = nb + 8 * h + j;
      if (n < p.N) {
        const int32_t x = v[8 * h + j];
        const uint32_t o = res ? epilogue_bf16_res(x, as, w[8 * h + j], bf16_bits_to_float(static_cast<uint16_t>(rb[j])))
                               : epilogue_bf16(x, as, w[8 * h + j]);
        p.out[m * p.ldo + n] = static_cast<uint16_t>(o);
        if (p.acc_out != nullptr) p.acc_out[m * p.N + n] = x;
      }
    }
  }
}

// Epilogue thread et's share of an item's scales: the a_scale of the tile's
// token et (et < kBNMax) or the w_scale of its channel et - kBNMax (0 past
// the tile or the matrix).
__device__ __forceinline__ float item_scale(const HParams& p, const Item& itm, int bn, int et) {
  const int64_t a0 = static_cast<int64_t>(itm.tx) * kBM, b0 = static_cast<int64_t>(itm.ty) * p.bpiece;
  if (et < kBNMax) {
    const int64_t m = (p.swap ? b0 : a0) + et;
    return et < (p.swap ? bn : kBM) && m < p.M ? __ldg(p.a_scale + m) : 0.f;
  }
  const int i = et - kBNMax;
  const int64_t n = (p.swap ? a0 : b0) + i;
  return i < (p.swap ? kBM : bn) && n < p.N ? __ldg(p.w_scale + n) : 0.f;
}

// (m, n) of element j of group cb, and whether it lies inside the matrix.
__device__ __forceinline__ bool group_elem(const HParams& p, int64_t a0, int64_t b0, int trow, int cb, int j,
                                           int64_t& m, int64_t& n) {
  const int64_t ar = a0 + trow, br = b0 + cb * 16 + j;
  m = p.swap ? br : ar;
  n = p.swap ? ar : br;
  return m < p.M && n < p.N;
}

// A piece slot holds a CTA's int32 partial sums of one shared tile: the 16
// values of group cb of TMEM lane trow at words ((cb * 128) + trow) * 16 ..
// + 15, so each thread moves its group as four 16-byte vectors and a warp's
// vectors cover 2 KB contiguously.
__device__ __forceinline__ int64_t piece_group(int trow, int cb) { return (static_cast<int64_t>(cb) * kBM + trow) * 16; }

// kExplicit: the explicit split-K instance (items of kind 0 and 1); the
// other instance runs the automatic schedules (kinds 0 and 2).  Each carries
// only its own protocol, which keeps the epilogue within its registers.
template <bool kExplicit>
__global__ void __launch_bounds__(kThreads, 1)
    linear_f16_kernel(const __grid_constant__ HParams p, const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);
  const int nst = p.nst;
  const uint32_t stage_bytes = static_cast<uint32_t>((kBM + p.bpiece) * 128);
  const uint32_t bars = base + kRing;
  const uint32_t bar_full = bars;                        // kMaxStages x 8 B: TMA bytes landed
  const uint32_t bar_empty = bars + 8 * kMaxStages;      // kMaxStages x 8 B: MMAs done with the stage
  const uint32_t bar_accf = bars + 16 * kMaxStages;      // 2 x 8 B: chunk in D[b] complete
  const uint32_t bar_acce = bar_accf + 16;               // 2 x 8 B: D[b] drained
  const uint32_t bar_done = bar_acce + 16;               // every MMA complete (teardown)
  uint8_t* scalars = smem + (bar_done + 8 - base);
  float* s_scale = reinterpret_cast<float*>(smem + kRing + kBarBytes);   // [2][2 * kBNMax]
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(scalars);
  volatile int* s_abort = reinterpret_cast<volatile int*>(scalars + 4);
  int* s_last = reinterpret_cast<int*>(scalars + 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // B rows of piece ty that exist, rounded up to 16 (the MMA's N granule)
  auto tile_width = [&](int ty) -> int {
    const int64_t left = (p.swap ? p.M : p.N) - static_cast<int64_t>(ty) * p.bpiece;
    const int64_t rnd = (left + 15) & ~static_cast<int64_t>(15);
    return static_cast<int>(rnd < p.bpiece ? rnd : p.bpiece);
  };

  if (tid == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_accf + 8 * b, 1);
      mbar_init(bar_acce + 8 * b, kEpiWarps);
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
  // nothing above touched global data; inputs and workspace only from here
  pdl_trigger();
  pdl_wait();

  if (warp == kTmaWarp) {
    // ============================ TMA producer ================================
    if (lane == 0) {
      int j = 0;
      uint32_t ph = 0;
      int64_t issued = 0;
      bool ok = true;
      Item itm;
      for (int n = 0; ok && get_item(p.sp, n, itm); ++n) {
        const int32_t ya = itm.tx * kBM, yb = itm.ty * p.bpiece;
        for (int it = itm.k0; it < itm.k1; ++it) {
          if (!wait1(bar_empty + 8 * j, ph ^ 1u, s_abort)) {
            ok = false;
            break;
          }
          const uint32_t dst = base + j * stage_bytes;
          tc::mbar_expect_tx(bar_full + 8 * j, stage_bytes);
          tc::tma_load_2d(dst, &tmA, it * kBK, ya, bar_full + 8 * j);
          tc::tma_load_2d(dst + kBM * 128, &tmB, it * kBK, yb, bar_full + 8 * j);
          ++issued;
          if (++j == nst) {
            j = 0;
            ph ^= 1u;
          }
        }
      }
      // Before the CTA may exit, every load issued must have landed: after an
      // expired wait anywhere in the CTA the MMA issuer may stop consuming
      // stages whose loads are still in flight.  Stage x completes phase
      // x / nst of slot x % nst; loads that were consumed pass at once.
      for (int64_t x = issued > nst ? issued - nst : 0; x < issued; ++x)
        wait_drain(bar_full + 8 * static_cast<uint32_t>(x % nst), static_cast<uint32_t>((x / nst) & 1));
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ============================ MMA issuer ==================================
    if (lane == 0) {
      const bool withhold = *reinterpret_cast<volatile int*>(&g_f16_withhold) != 0;
      int s = 0;
      uint32_t ph = 0;
      int c = -1;  // chunk counter over all items
      bool ok = true, issued = false;
      Item itm;
      for (int n = 0; ok && get_item(p.sp, n, itm); ++n) {
        const int nk = itm.k1 - itm.k0;
        const uint32_t idesc = tc::idesc_f16_f32(tile_width(itm.ty));
        uint32_t dcol = 0, buf = 0;
        for (int it = 0; it < nk; ++it) {
          const int cpos = it & (kChunk - 1);
          if (cpos == 0) {
            // chunk c reuses buffer c % 2: wait until chunk c - 2 was drained
            ++c;
            buf = static_cast<uint32_t>(c & 1);
            dcol = buf * kBNMax;
            if (c >= 2) {
              if (!wait1(bar_acce + 8 * buf, static_cast<uint32_t>(((c >> 1) - 1) & 1), s_abort)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
          }
          if (!wait1(bar_full + 8 * s, ph, s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st_addr = base + s * stage_bytes;
          const uint64_t ad = tc::smem_desc_sw128(st_addr);
          const uint64_t bd = tc::smem_desc_sw128(st_addr + kBM * 128);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            tc::tc_mma(tmem + dcol, ad + 2 * k, bd + 2 * k, idesc, (cpos | k) != 0 ? 1u : 0u);
          issued = true;
          tc::tc_commit(bar_empty + 8 * s);
          if ((cpos == kChunk - 1 || it == nk - 1) && !(withhold && c == 0)) tc::tc_commit(bar_accf + 8 * buf);
          if (++s == nst) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (issued) {
        // every MMA issued above has completed before TMEM is released
        tc::tc_commit(bar_done);
        wait_drain(bar_done, 0);
      }
    }
    __syncwarp();
  } else {
    // ============================ epilogue (16 warps) =========================
    const int ew = warp - 2;                       // 0..15
    const int quad = warp & 3;                     // TMEM lane quadrant this warp may access
    const int slice = ew >> 2;                     // column groups slice, slice + 4, ...
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const int trow = quad * 32 + lane;             // this thread's TMEM lane = A row of the tile
    const int et = ew * 32 + lane;
    bool ok = true;
    int gc = 0;                                    // chunk counter over all items
    {
      // item 0's scales; item n + 1's are stored while item n finishes, and
      // the barrier at item n + 1's output orders them before any read
      Item first;
      s_scale[et] = get_item(p.sp, 0, first) ? item_scale(p, first, tile_width(first.ty), et) : 0.f;
    }
    for (int n = 0;; ++n) {
      int groups, nchunks;
      {
        // only n stays live through the chunk loop; the item is looked up
        // again for its output
        Item itm;
        if (!get_item(p.sp, n, itm)) break;
        groups = tile_width(itm.ty) >> 4;
        nchunks = (itm.k1 - itm.k0 + kChunk - 1) / kChunk;
      }
      int32_t acc[kGroups][16];
#pragma unroll
      for (int r = 0; r < kGroups; ++r)
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[r][j] = 0;
      for (int lc = 0; lc < nchunks; ++lc, ++gc) {
        if (!ok) continue;
        const uint32_t buf = static_cast<uint32_t>(gc & 1);
        ok = wait_warp(bar_accf + 8 * buf, static_cast<uint32_t>((gc >> 1) & 1), s_abort);
        if (!ok) continue;
        tc_fence_after();
#pragma unroll
        for (int r = 0; r < kGroups; ++r) {
          const int cb = slice + 4 * r;
          if (cb < groups) {
            uint32_t d[16];
            tc::tmem_ld16(tmem + lane_base + buf * kBNMax + cb * 16, d);
            tc::tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[r][j] += __float2int_rn(__uint_as_float(d[j]));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_acce + 8 * buf);
      }

      Item itm;
      get_item(p.sp, n, itm);
      const int64_t a0 = static_cast<int64_t>(itm.tx) * kBM, b0 = static_cast<int64_t>(itm.ty) * p.bpiece;
      // this item's scales are in place (and every thread is done with the
      // previous item's, whose buffer takes item n + 1's below)
      epi_barrier();
      const float* s_tok = s_scale + (n & 1) * (2 * kBNMax);
      const float* s_ch = s_tok + kBNMax;
      {
        Item nx;
        const float sc = get_item(p.sp, n + 1, nx) ? item_scale(p, nx, tile_width(nx.ty), et) : 0.f;
        s_scale[((n + 1) & 1) * (2 * kBNMax) + et] = sc;
      }
      if (itm.kind == 0) {
        if (ok && nchunks > 0) {
#pragma unroll
          for (int r = 0; r < kGroups; ++r)
            if (slice + 4 * r < groups) emit_group(p, s_tok, s_ch, a0, b0, trow, slice + 4 * r, acc[r]);
        }
        continue;
      }
      // a K piece: the partial sums go to the workspace; the last CTA to finish
      // the tile adds the other pieces to its own and applies the epilogue.
      // Balanced schedule: every piece has a slot of its own, written with
      // plain 16-byte stores (no reductions, nothing to re-zero).  Explicit
      // split-K: integer atomics into the [M, N] accumulator.
      const int64_t slot_elems = static_cast<int64_t>(kBM) * p.bpiece;
      int sfirst = 0, sn = 0, smine = 0;
      if (!kExplicit) shared_tile_slots(p.sp, itm.tile, sfirst, sn, smine);
      if (ok) {
        if (!kExplicit) {
          int32_t* mine = p.slots + static_cast<int64_t>(smine) * slot_elems;
#pragma unroll
          for (int r = 0; r < kGroups; ++r) {
            const int cb = slice + 4 * r;
            if (cb >= groups) continue;
            int4* dst = reinterpret_cast<int4*>(mine + piece_group(trow, cb));
#pragma unroll
            for (int q = 0; q < 4; ++q)
              __stcg(dst + q, make_int4(acc[r][4 * q], acc[r][4 * q + 1], acc[r][4 * q + 2], acc[r][4 * q + 3]));
          }
        } else {
#pragma unroll
          for (int r = 0; r < kGroups; ++r) {
            const int cb = slice + 4 * r;
            if (cb >= groups) continue;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              int64_t m, nn;
              if (group_elem(p, a0, b0, trow, cb, j, m, nn)) atomicAdd(p.ws_acc + m * p.N + nn, acc[r][j]);
            }
          }
        }
      }
      __threadfence();
      // every epilogue thread takes both barriers; a tile that any thread
      // could not finish (an expired wait) is not counted and not written
      const bool bad = epi_barrier_any(!ok);
      uint32_t* counter = kExplicit ? p.ws_count + itm.tile : p.cnt + itm.tile;
      if (!bad && et == 0) {
        const unsigned target = kExplicit ? static_cast<unsigned>(p.sp.split - 1) : static_cast<unsigned>(sn - 1);
        // release: the stores of every epilogue thread reached thread 0
        // through the barrier; its fence orders them before the arrival.
        // acquire: the last arriver's fence orders the read-back after them.
        __threadfence();
        const bool last = atomicAdd(counter, 1u) == target;
        __threadfence();
        *s_last = last;
      }
      epi_barrier();
      if (bad || !*s_last) continue;
      __threadfence();
      if (!kExplicit) {
        // the other CTAs' pieces, added to this CTA's own sums in registers
        for (int so = sfirst; so < sfirst + sn; ++so) {
          if (so == smine) continue;
          const int32_t* other = p.slots + static_cast<int64_t>(so) * slot_elems;
#pragma unroll
          for (int r = 0; r < kGroups; ++r) {
            const int cb = slice + 4 * r;
            if (cb >= groups) continue;
            const int4* src = reinterpret_cast<const int4*>(other + piece_group(trow, cb));
            int4 in[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) in[q] = __ldcg(src + q);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              acc[r][4 * q] += in[q].x;
              acc[r][4 * q + 1] += in[q].y;
              acc[r][4 * q + 2] += in[q].z;
              acc[r][4 * q + 3] += in[q].w;
            }
          }
        }
      } else {
        // explicit split-K: the total from the accumulator, which is re-zeroed
#pragma unroll
        for (int r = 0; r < kGroups; ++r) {
          const int cb = slice + 4 * r;
          if (cb >= groups) continue;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            int64_t m, nn;
            acc[r][j] = group_elem(p, a0, b0, trow, cb, j, m, nn) ? __ldcg(p.ws_acc + m * p.N + nn) : 0;
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            int64_t m, nn;
            if (group_elem(p, a0, b0, trow, cb, j, m, nn)) __stcg(p.ws_acc + m * p.N + nn, 0);
          }
        }
      }
#pragma unroll
      for (int r = 0; r < kGroups; ++r)
        if (slice + 4 * r < groups) emit_group(p, s_tok, s_ch, a0, b0, trow, slice + 4 * r, acc[r]);
      if (et == 0) *counter = 0u;
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

// Orientation and B-piece width: few rows (M < 512) put the tokens on the
// MMA's N side in equal pieces (multiples of 32, at most 256); otherwise the
// tokens fill the 128 MMA rows and 256 output channels form N.
struct HPlan {
  int swap, bpiece;
  int64_t gx, gy;
};

// PRISM_F16_ORIENT=rows / =cols forces the tokens onto the MMA's rows / its
// N side whatever M (a diagnostic: both orientations give the same bits).
int orient_override() {
  const char* e = std::getenv("PRISM_F16_ORIENT");
  if (e == nullptr) return -1;
  if (std::strcmp(e, "rows") == 0) return 0;
  if (std::strcmp(e, "cols") == 0) return 1;
  return -1;
}

HPlan plan(int64_t M, int64_t N) {
  HPlan pl{};
  const int forced = orient_override();
  pl.swap = forced >= 0 ? forced : (M < 512 ? 1 : 0);
  if (pl.swap) {
    const int64_t pieces = cdiv(M, kBNMax);
    pl.bpiece = static_cast<int>(cdiv(cdiv(M, pieces), 32) * 32);
    pl.gx = cdiv(N, kBM);
    pl.gy = cdiv(M, pl.bpiece);
  } else {
    pl.bpiece = kBNMax;
    pl.gx = cdiv(M, kBM);
    pl.gy = cdiv(N, kBNMax);
  }
  return pl;
}

// The automatic schedule (tc_sched.cuh).  Whole tiles in rounds (tile b,
// b + G, ... on CTA b) unless the last round would leave most SMs idle:
// then the rounds with the last one split in lockstep (each remainder tile
// cut into P equal K pieces on P CTAs, the pieces of tiles that share a
// weight operand running side by side), or, where no such split fits, the
// balanced schedule.  The balanced schedule's arbitrary cuts cost this
// kernel more than they gain -- each shared piece's private slot (128 x
// width int32) written, counted and read back; keeping the pieces of a
// weight tile side by side did not recover it.  Measured per call (whole /
// balanced / lockstep, us): gate/up 458 / 481 / 463; 8192 rows 313 / 334 /
// 313; down (2 rounds and 16 tiles) 311 / 295 / 275; QKV 64.8 whole against
// 72 balanced; o_proj 40.5 against 50.  PRISM_F16_SCHED = whole, balanced or
// lock forces one (a diagnostic: every schedule gives the same bits).
struct F16Sched {
  int sched, G, W, R, P;
};

F16Sched schedule(const HPlan& pl, int64_t K) {
  const int64_t T = pl.gx * pl.gy, g = sm_count(), S = cdiv(K, kBK);
  auto whole = [&] { return F16Sched{1, static_cast<int>(g), static_cast<int>(cdiv(T, g)), 0, 1}; };
  auto bal = [&] {
    const TcSched sc = tc_balanced_sched(T, S, kChunk, g);
    return F16Sched{1, sc.G, sc.W, sc.R, 1};
  };
  auto lock = [&] {
    const int64_t W = T / g, R = T % g;
    const int64_t P = R == 0 ? 1 : std::min<int64_t>(g / R, S / kChunk);
    if (P <= 1) return whole();
    return F16Sched{2, static_cast<int>(W > 0 ? g : R * P), static_cast<int>(W), static_cast<int>(R),
                    static_cast<int>(P)};
  };
  if (const char* e = std::getenv("PRISM_F16_SCHED")) {
    if (std::strcmp(e, "whole") == 0) return whole();
    if (std::strcmp(e, "balanced") == 0) return bal();
    if (std::strcmp(e, "lock") == 0) return lock();
  }
  if (T >= g / 2 && T % g >= g / 5) return whole();
  const F16Sched l = lock();
  return l.sched == 2 ? l : bal();
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Automatic schedule's workspace: counters of the shared tiles, then the
// piece slots of 128 x bpiece int32 -- balanced: one per (shared tile st,
// CTA b) pair at index st + b, R + G - 1 slots; lockstep rounds: P per
// remainder tile.
size_t balanced_bytes(int64_t M, int64_t N, int64_t K, size_t* counter_bytes) {
  const HPlan pl = plan(M, N);
  const F16Sched sc = schedule(pl, K);
  const size_t slots = sc.sched == 2 ? static_cast<size_t>(sc.R) * sc.P
                                     : (sc.R == 0 || sc.G == sc.R ? 0 : static_cast<size_t>(sc.R + sc.G - 1));
  if (slots == 0) {   // no tile shared between CTAs
    if (counter_bytes != nullptr) *counter_bytes = 0;
    return 0;
  }
  const size_t cb = round256(static_cast<size_t>(sc.R) * 4);
  if (counter_bytes != nullptr) *counter_bytes = cb;
  return cb + slots * kBM * pl.bpiece * 4;
}

// Explicit split-K: the [M, N] int32 accumulator, then one counter per tile.
size_t split_bytes(int64_t M, int64_t N) {
  const HPlan pl = plan(M, N);
  return round256(static_cast<size_t>(M) * static_cast<size_t>(N) * 4) +
         round256(static_cast<size_t>(pl.gx * pl.gy) * 4);
}

using EncodeTiledFn = PFN_cuTensorMapEncodeTiled_v12000;

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(f);
    return static_cast<EncodeTiledFn>(nullptr);
  }();
  return fn;
}

// Row-major binary16 [rows, K] with row stride ld elements, read in boxes of
// 64 K-elements (128 bytes) x box_rows rows, 128-byte swizzled into shared
// memory (the MMA's K-major operand layout); out-of-range rows and K read 0.
cudaError_t make_map(CUtensorMap* m, const uint16_t* ptr, int64_t rows, int64_t K, int64_t ld, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

size_t linear_f16_workspace_bytes(int64_t M, int64_t N, int64_t K, int split) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  if (split == 0) return balanced_bytes(M, N, K, nullptr);
  return split > 1 ? split_bytes(M, N) : 0;
}

cudaError_t launch_linear_f16(const LinearF16Args& a, cudaStream_t stream) {
  const HPlan pl = plan(a.M, a.N);
  auto kernel = a.split >= 1 ? linear_f16_kernel<true> : linear_f16_kernel<false>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kernel), kSmemBytes);
  if (e != cudaSuccess) return e;
  HParams p{};
  p.a_scale = a.a_scale;
  p.w_scale = a.w_scale;
  p.residual = a.residual;
  p.ldr = a.ldr;
  p.out = a.out;
  p.ldo = a.ldo;
  p.acc_out = a.acc_out;
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.swap = pl.swap;
  p.bpiece = pl.bpiece;
  const uintptr_t ob = reinterpret_cast<uintptr_t>(a.out), rb = reinterpret_cast<uintptr_t>(a.residual);
  const uintptr_t wb = reinterpret_cast<uintptr_t>(a.w_scale);
  p.vec_io = (ob % 16 == 0) && (a.ldo % 8 == 0) && (wb % 16 == 0) &&
             (a.residual == nullptr || ((rb % 16 == 0) && (a.ldr % 8 == 0)));
  p.nst = std::min(kMaxStages, kRing / ((kBM + pl.bpiece) * 128));
  p.sp.split = a.split;
  p.sp.gx = static_cast<int>(pl.gx);
  p.sp.gy = static_cast<int>(pl.gy);
  p.sp.a_w = pl.swap ? 1 : 0;
  p.sp.T = static_cast<int>(pl.gx * pl.gy);
  p.sp.S = static_cast<int>(cdiv(a.K, kBK));
  dim3 grid;
  if (a.split >= 1) {
    p.sp.sched = 0;
    if (a.split > 1) {
      p.ws_acc = static_cast<int32_t*>(a.ws);
      p.ws_count = reinterpret_cast<uint32_t*>(static_cast<char*>(a.ws) +
                                               round256(static_cast<size_t>(a.M) * static_cast<size_t>(a.N) * 4));
    }
    grid = dim3(static_cast<unsigned>(pl.gx), static_cast<unsigned>(pl.gy), static_cast<unsigned>(a.split));
  } else {
    const F16Sched sc = schedule(pl, a.K);
    p.sp.sched = sc.sched;
    size_t cb = 0;
    const size_t need = balanced_bytes(a.M, a.N, a.K, &cb);
    if (need > 0) {
      p.cnt = static_cast<uint32_t*>(a.ws);
      p.slots = reinterpret_cast<int32_t*>(static_cast<char*>(a.ws) + cb);
    }
    p.sp.W = sc.W;
    p.sp.R = sc.R;
    p.sp.P = sc.P;
    const int64_t ctas = sc.sched == 2 || sc.R > 0 ? sc.G : std::min<int64_t>(sc.G, p.sp.T);
    grid = dim3(static_cast<unsigned>(ctas), 1, 1);
  }
  CUtensorMap tmA, tmB;
  const uint16_t* Am = pl.swap ? a.wh : a.qh;
  const uint16_t* Bm = pl.swap ? a.qh : a.wh;
  e = make_map(&tmA, Am, pl.swap ? a.N : a.M, a.K, pl.swap ? a.ldw : a.ldq, kBM);
  if (e != cudaSuccess) return e;
  e = make_map(&tmB, Bm, pl.swap ? a.M : a.N, a.K, pl.swap ? a.ldq : a.ldw, pl.bpiece);
  if (e != cudaSuccess) return e;
  return launch_kernel(kernel, grid, dim3(kThreads), kSmemBytes, stream, true, p, tmA, tmB);
}

cudaError_t read_and_clear_f16_status(uint32_t* out) {
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_f16_status, sizeof v);
  if (e != cudaSuccess) return e;
  if (v != 0) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_f16_status, &zero, sizeof zero);
  }
  *out = v;
  return e;
}

cudaError_t set_f16_wait_expiry(unsigned long long limit_ns, int withhold) {
  cudaError_t e = cudaMemcpyToSymbol(g_f16_wait_limit_ns, &limit_ns, sizeof limit_ns);
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_f16_withhold, &withhold, sizeof withhold);
  return e;
}

// ------------------------------------------------------- int8 -> binary16 --
namespace {

// Exact widening of int8 codes to binary16: each byte b becomes the f16 of
// 1024 + (b + 128) (pattern 0x6400 | (b ^ 0x80)), minus 1152, both exact.
__global__ void __launch_bounds__(256) codes_to_f16_kernel(const int8_t* __restrict__ w, int64_t ldw, int64_t rows,
                                                          int64_t K, uint16_t* __restrict__ wh, int64_t ldwh) {
  pdl_trigger();
  pdl_wait();
  const int64_t per_row = K >> 4;   // 16-byte chunks of a row
  const int64_t total = rows * per_row;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / per_row, c = i - r * per_row;
    const uint4 v = ld_stream_16(w + r * ldw + c * 16);
    const uint32_t x[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t u = x[k] ^ 0x80808080u;
      uint32_t p0, p1;
      asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(p0) : "r"(u), "r"(0x64646464u));
      asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(p1) : "r"(u), "r"(0x64646464u));
      asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(o[2 * k]) : "r"(p0), "r"(0x64806480u));
      asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(o[2 * k + 1]) : "r"(p1), "r"(0x64806480u));
    }
    uint4* dst = reinterpret_cast<uint4*>(wh + r * ldwh + c * 16);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

}  // namespace

cudaError_t launch_codes_to_f16(const int8_t* w, int64_t ldw, int64_t rows, int64_t K, uint16_t* wh, int64_t ldwh,
                                cudaStream_t stream) {
  const int64_t total = rows * (K >> 4);
  const int64_t ctas = std::max<int64_t>(1, std::min<int64_t>(cdiv(total, 256), static_cast<int64_t>(sm_count()) * 8));
  return launch_kernel(codes_to_f16_kernel, dim3(static_cast<unsigned>(ctas)), dim3(256), 0, stream, true, w, ldw,
                       rows, K, wh, ldwh);
}

}  // namespace prism
