// tc_sched.cuh -- the work schedule of the persistent tcgen05 contraction
// kernels: which output tile and which range of K stages each CTA computes.
//
// Output tile (tx, ty) is A block tx (128 rows) by B piece ty.  The balanced
// schedule numbers tiles so that consecutive indices share the weight
// operand: t = ty * gx + tx when the weights are B (tokens on the MMA rows),
// t = tx * gy + ty when they are A (output channels on the MMA rows), so the
// CTAs that run side by side read the same weight stages and all but the
// first of them find those stages in L2.  K is cut into S stages of 64
// elements.
//   sched 0: one item per CTA: tile (blockIdx.x, blockIdx.y), K piece
//            blockIdx.z of `split` equal pieces (explicit split-K; the
//            pieces' int32 partial sums are added with integer atomics).
//   sched 1: the balanced schedule over G = gridDim.x CTAs: CTA b first
//            takes whole tiles b, b + G, ... (W rounds, indices below T),
//            then the K stages [b U / G, (b + 1) U / G) of the last R tiles,
//            U = R * S, shared tile st covering stages [st S, (st + 1) S).
//            Every CTA gets the same number of stages; a tile shared by
//            several CTAs has their int32 partial sums added (integer
//            reductions) into its accumulator slot, and the last CTA to
//            finish the tile reads the slot back and applies the epilogue.
//   sched 2: rounds with the last one split in lockstep: CTA b takes whole
//            tiles b, b + G, ... (W rounds), then, when b < R * P, K piece
//            b / R of the P equal pieces of remainder tile b % R, so that the
//            pieces of tiles that share a weight operand run side by side
//            and start together; the last piece of a tile to finish adds
//            the others' partial sums.
// Integer addition is order-free, so no choice here changes a result bit.
#pragma once

#include <algorithm>
#include <cstdint>

namespace prism {

struct SchedParams {
  int sched;  // 0: one item per CTA (explicit split-K); 1: balanced
  int split;  // explicit split-K factor (sched 0)
  int gx;     // A blocks of 128 rows
  int gy;     // B pieces
  int a_w;    // 1: the weights are the A operand (tile index runs over B pieces fastest)
  int T;      // tiles
  int S;      // K stages of 64 elements
  int W;      // balanced: rounds of whole tiles per CTA
  int R;      // balanced: tiles whose K stages are shared out
  int P;      // sched 2: K pieces of each remainder tile
};

// One unit of work: tile (tx, ty) over K stages [k0, k1).
//   kind 0: the whole K range; the epilogue is applied directly.
//   kind 1: one of `split` equal K pieces (explicit split-K).
//   kind 2: a K range of a tile the balanced schedule shares between CTAs.
struct Item {
  int tx, ty, k0, k1, kind, tile;
};

// Tile index t of the balanced schedule -> (tx, ty).
__device__ __forceinline__ void tile_coords(const SchedParams& p, int t, Item& it) {
  if (p.a_w) {
    it.tx = t / p.gy;
    it.ty = t % p.gy;
  } else {
    it.tx = t % p.gx;
    it.ty = t / p.gx;
  }
}

// Work item n of this CTA; every role of the CTA walks the same list.
__device__ __forceinline__ bool get_item(const SchedParams& p, int n, Item& it) {
  if (p.sched == 0) {
    if (n > 0) return false;
    const int per = (p.S + p.split - 1) / p.split;
    it.tx = static_cast<int>(blockIdx.x);
    it.ty = static_cast<int>(blockIdx.y);
    const int k0 = static_cast<int>(blockIdx.z) * per;
    it.k0 = k0 < p.S ? k0 : p.S;
    it.k1 = it.k0 + per < p.S ? it.k0 + per : p.S;
    it.kind = p.split > 1 ? 1 : 0;
    it.tile = it.ty * p.gx + it.tx;
    return true;
  }
  const int G = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x);
  if (p.sched == 2) {
    if (n < p.W) {
      const int t = n * G + b;
      if (t >= p.T) return false;
      tile_coords(p, t, it);
      it.k0 = 0;
      it.k1 = p.S;
      it.kind = 0;
      it.tile = t;
      return true;
    }
    if (n > p.W || b >= p.R * p.P) return false;
    const int r = b % p.R, kp = b / p.R;
    tile_coords(p, p.W * G + r, it);
    it.k0 = kp * p.S / p.P;
    it.k1 = (kp + 1) * p.S / p.P;
    it.kind = p.P > 1 ? 2 : 0;
    it.tile = r;
    return true;
  }
  if (n < p.W) {
    const int t = n * G + b;
    if (t >= p.T) return false;
    tile_coords(p, t, it);
    it.k0 = 0;
    it.k1 = p.S;
    it.kind = 0;
    it.tile = t;
    return true;
  }
  if (p.R == 0) return false;
  // U * G < 2^31: R < 2 G, S <= 2081 (K <= 133144) and G <= 512 (sm_count's cap)
  const int j = n - p.W;
  const int U = p.R * p.S;
  const int u0 = b * U / G, u1 = (b + 1) * U / G;
  const int st = u0 / p.S + j;
  const int ts = st * p.S;
  if (u0 >= u1 || ts >= u1) return false;
  const int t = p.W * G + st;
  tile_coords(p, t, it);
  it.k0 = (u0 > ts ? u0 : ts) - ts;
  it.k1 = (u1 < ts + p.S ? u1 : ts + p.S) - ts;
  it.kind = (it.k0 == 0 && it.k1 == p.S) ? 0 : 2;
  it.tile = st;
  return true;
}

// CTAs bf..bl of the balanced schedule whose K ranges meet shared tile st
// (the CTA holding unit u is floor(((u + 1) G - 1) / U)).
__device__ __forceinline__ void shared_tile_ctas(const SchedParams& p, int st, int& bf, int& bl) {
  const int G = static_cast<int>(gridDim.x);
  const int U = p.R * p.S;
  bf = ((st * p.S + 1) * G - 1) / U;
  bl = ((st * p.S + p.S) * G - 1) / U;
}

// The partial-sum slots of shared tile st: this CTA's (mine) and the tile's
// ns slots first, first + 1, ... (one per CTA sharing the tile: the sched-1
// pair index st + b over the tile's CTAs bf..bl, or st * P + piece).
__device__ __forceinline__ void shared_tile_slots(const SchedParams& p, int st, int& first, int& ns, int& mine) {
  const int b = static_cast<int>(blockIdx.x);
  if (p.sched == 2) {
    first = st * p.P;
    ns = p.P;
    mine = first + b / p.R;
    return;
  }
  int bf, bl;
  shared_tile_ctas(p, st, bf, bl);
  first = st + bf;
  ns = bl - bf + 1;
  mine = st + b;
}

// The balanced schedule for T tiles of S K-stages on `sms` CTAs: whole tiles
// in W rounds, then the K stages of the last R tiles shared out evenly.
// Shares below min_units stages (one exact 1024-K chunk) per CTA are not
// worth their partial-sum traffic: then one round fewer of whole tiles is
// taken, or, with few tiles, fewer CTAs share them, or (little K) only whole
// tiles are used.
struct TcSched {
  int G, W, R;
};

inline TcSched tc_balanced_sched(int64_t T, int64_t S, int64_t min_units, int64_t sms) {
  TcSched sc{static_cast<int>(sms), 0, 0};
  if (T % sms == 0) {
    sc.W = static_cast<int>(T / sms);
    return sc;
  }
  int64_t W = T / sms, R = T - W * sms;
  if (R * S < min_units * sms && W >= 1) {
    W -= 1;
    R += sms;
  }
  if (R * S >= min_units * sms) {
    sc.W = static_cast<int>(W);
    sc.R = static_cast<int>(R);
  } else if (W == 0) {
    sc.G = static_cast<int>(std::max<int64_t>(R, std::min<int64_t>(sms, R * S / min_units)));
    sc.R = static_cast<int>(R);
  } else {
    sc.W = static_cast<int>((T + sms - 1) / sms);
  }
  return sc;
}

}  // namespace prism
