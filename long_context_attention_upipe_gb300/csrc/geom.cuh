// Row geometry of the attention kernels and the tile-skip table: which keys a query row sees.
//
// Plain launches: query and key row i share position i, and a query sees the keys of its segment
// up to itself (causal) or all of them, one interval [seg start, r or seg end] (MaxText article,
// Splash attention paragraph: packed sequences without padding).
//
// Zigzag ring steps (MaxText article, strategy table, row "P2P (Ring)", and the paragraph on
// causal load balancing): a plane holds one device's two chunks, the query rows of device r and
// the key rows of the visiting shard of device src = (r - step) mod P.  Positions increase with
// the local row in both, so the keys a query sees (an earlier-or-equal position, the same segment)
// again form one interval, and the queries that see a key form one interval too; both interval
// ends are non-decreasing in the row, which is what the table's tile ranges rely on.
#pragma once

#include "internal.h"

namespace upipe {

__host__ __device__ __forceinline__ int ring_mod(int x, int P) {
  x %= P;
  return x < 0 ? x + P : x;
}

// Row geometry of one (query device, key shard) pair of a launch.
struct Zig {
  const int32_t* seg;  // plain: [S] by row; ring: [2PC] by position; NULL: one segment
  int64_t S;           // rows per plane
  int causal;
  int P;               // 0: plain
  int64_t C;
  int r, src;          // ring devices of the query rows and of the key rows

  __device__ __forceinline__ int64_t pos(int dev, int64_t i) const {
    return i < C ? (int64_t)dev * C + i : (int64_t)(2 * P - 1 - dev) * C + (i - C);
  }
  // last local row j of device dev with pos(dev, j) <= p (-1: none)
  __device__ __forceinline__ int64_t last_le(int dev, int64_t p) const {
    const int64_t a0 = (int64_t)dev * C, b0 = (int64_t)(2 * P - 1 - dev) * C;
    if (p >= b0) return C + min(C - 1, p - b0);
    if (p >= a0) return min(C - 1, p - a0);
    return -1;
  }
  // first local row i of device dev with pos(dev, i) >= p (2C: none)
  __device__ __forceinline__ int64_t first_ge(int dev, int64_t p) const {
    const int64_t a0 = (int64_t)dev * C, b0 = (int64_t)(2 * P - 1 - dev) * C;
    if (p <= a0) return 0;
    if (p < a0 + C) return p - a0;
    if (p <= b0) return C;
    if (p < b0 + C) return C + (p - b0);
    return 2 * C;
  }
  // first local row of device dev whose segment id is >= v, and last whose id is <= v
  __device__ __forceinline__ int64_t seg_lo(int dev, int32_t v) const {
    int64_t lo = 0, hi = 2 * C;
    while (lo < hi) {
      const int64_t mid = (lo + hi) >> 1;
      if (seg[pos(dev, mid)] >= v) hi = mid; else lo = mid + 1;
    }
    return lo;
  }
  __device__ __forceinline__ int64_t seg_hi(int dev, int32_t v) const {
    int64_t lo = -1, hi = 2 * C - 1;
    while (lo < hi) {
      const int64_t mid = (lo + hi + 1) >> 1;
      if (seg[pos(dev, mid)] <= v) lo = mid; else hi = mid - 1;
    }
    return lo;
  }

  // The keys query row `row` (< S) sees: [lo, hi] (empty when lo > hi).
  __device__ __forceinline__ void q_interval(int64_t row, int64_t& lo, int64_t& hi) const {
    if (P == 0) {
      lo = seg_first(seg, row);
      hi = causal ? row : seg_last(seg, S, row);
      return;
    }
    const int64_t p = pos(r, row);
    lo = 0;
    hi = causal ? last_le(src, p) : 2 * C - 1;
    if (seg) {
      const int32_t v = seg[p];
      lo = seg_lo(src, v);
      hi = min(hi, seg_hi(src, v));
    }
  }
  // The queries that see key row `krow` (< S): [lo, hi].
  __device__ __forceinline__ void k_interval(int64_t krow, int64_t& lo, int64_t& hi) const {
    if (P == 0) {
      lo = causal ? krow : seg_first(seg, krow);
      hi = seg_last(seg, S, krow);
      return;
    }
    const int64_t p = pos(src, krow);
    lo = causal ? first_ge(r, p) : 0;
    hi = 2 * C - 1;
    if (seg) {
      const int32_t v = seg[p];
      lo = max(lo, seg_lo(r, v));
      hi = seg_hi(r, v);
    }
  }
};

// Geometry of batch device d (its query planes and the key shard it reads).
__device__ __forceinline__ Zig make_zig(const int32_t* seg, int64_t S, int causal, const RingGeom& g, int d) {
  Zig z{seg, S, causal, g.P, g.C, 0, 0};
  if (g.P) {
    z.r = ring_mod(g.r0 + d, g.P);
    z.src = ring_mod(z.r - g.step, g.P);
  }
  return z;
}

// Memory index of the key/value shard that batch device d reads, and the batch device that key
// shard m serves at this step (>= ndev: none of the launch).
__device__ __forceinline__ int kv_shard_of(const RingGeom& g, int d) {
  return g.P ? ring_mod(g.r0 + d - g.step - g.kv0, g.P) : 0;
}
__device__ __forceinline__ int dev_of_shard(const RingGeom& g, int m) {
  return g.P ? ring_mod(g.kv0 + m + g.step - g.r0, g.P) : 0;
}

// Does a later step of the ring touch query tile qt of batch device d (non-empty table row)?
__device__ __forceinline__ bool q_tile_touched_later(const AttnArgs& a, int d, int qt, int nt) {
  for (int s2 = a.ring.step + 1; s2 < a.ring.P; ++s2) {
    const int4 r = reinterpret_cast<const int4*>(a.ring_tables + s2 * a.ring_table_stride +
                                                 sizeof(TableHeader))[(int64_t)d * nt + qt];
    if (r.x < r.w) return true;
  }
  return false;
}
// ... key tile jt of key shard m (valid when the shards are the launch's own at every step)
__device__ __forceinline__ bool kv_tile_touched_later(const AttnArgs& a, int m, int jt, int nt) {
  for (int s2 = a.ring.step + 1; s2 < a.ring.P; ++s2) {
    const int4 r = reinterpret_cast<const int4*>(a.ring_tables + s2 * a.ring_table_stride + sizeof(TableHeader) +
                                                 (size_t)a.ndev * nt * sizeof(int4))[(int64_t)m * nt + jt];
    if (r.x < r.w) return true;
  }
  return false;
}

}  // namespace upipe
