// Tile-skip table for 128x128 tiles under the causal + same-segment mask.
//
// Splash attention skips blocks whose every (query, key) pair is masked and handles packed
// sequences without padding (MaxText long-context article, techmoon.xyz, paragraph on the
// shared attention kernel).  With non-decreasing segment ids, query row r sees exactly the
// keys [segstart(r), causal ? r : segend(r)]; both ends are non-decreasing in r, so for a
// query tile the non-empty key tiles form one range and the full ones a sub-range, and the
// same holds per key tile.  Each thread derives one row of the table from a few binary
// searches over the segment ids; nothing is materialised per element.
//
// A ring step's table (the zigzag geometry of geom.cuh) has one such set of rows per batched
// device and per key shard, and its dispatch orders rank the work of all of them together, so a
// single launch runs the whole step with the longest CTAs first.
#include "geom.cuh"

namespace upipe {

namespace {

// Raw range functions of query tile i (all non-decreasing in i for non-decreasing ids).
struct QTileRanges {
  int32_t b, e;    // non-empty key tiles [b, e)
  int32_t fb, fe;  // full key tiles [fb, fe), possibly empty (fb >= fe)
};

// From the intervals of the tile's first and last rows: with both interval ends non-decreasing in
// the row, every row's keys lie in [lo(first), hi(last)], and the keys in [lo(last), hi(first)]
// are seen by every row.
__device__ __forceinline__ QTileRanges q_tile_ranges(const Zig& z, int64_t i, int64_t nt) {
  const int64_t S = z.S;
  const int64_t r0 = i * kTile;
  const int64_t rl = min(S, r0 + kTile) - 1;
  int64_t lo0, hi0, lo1, hi1;
  z.q_interval(r0, lo0, hi0);
  z.q_interval(rl, lo1, hi1);
  QTileRanges q;
  q.b = (int32_t)(lo0 / kTile);
  q.e = hi1 < 0 ? 0 : (int32_t)(hi1 / kTile + 1);
  q.fb = (int32_t)ceil_div(lo1, kTile);
  const int64_t last = (hi0 >= S - 1) ? nt - 1 : (hi0 + 1) / kTile - 1;  // every key column <= hi0 is seen by all rows
  q.fe = (int32_t)(last + 1);
  return q;
}

__global__ void k_table_init(TableHeader* h, int n_tiles) {
  if (threadIdx.x == 0 && blockIdx.x == 0) {
    h->n_partial = 0;
    h->n_full = 0;
    h->error = 0;
    h->n_tiles = n_tiles;
    h->reserved = 0;
  }
}

__global__ void k_check_monotone(const int32_t* __restrict__ seg, int64_t S, TableHeader* h) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  bool bad = false;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i + 1 < S; i += stride)
    bad |= seg[i] > seg[i + 1];
  if (__syncthreads_or(bad) && threadIdx.x == 0) set_error(&h->error, UPIPE_ERR_SEGMENTS_NOT_CONTIGUOUS);
}

struct Geo {
  const int32_t* seg;
  int64_t S;
  int causal;
  RingGeom g;
  int ndev, kv_count;
};

// one thread per (device, query tile)
__global__ void k_q_rows(Geo geo, int64_t nt, int4* __restrict__ rows, TableHeader* h) {
  const int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  long long part = 0, full = 0;
  if (x < geo.ndev * nt) {
    const int d = (int)(x / nt);
    const int64_t i = x - d * nt;
    const Zig z = make_zig(geo.seg, geo.S, geo.causal, geo.g, d);
    QTileRanges q = q_tile_ranges(z, i, nt);
    int32_t fb = q.fb, fe = q.fe;
    if (fb >= fe) fb = fe = q.e;
    // clamp (only matters when the ids are not sorted; the error word is set then)
    int32_t b = max(0, min(q.b, (int32_t)nt)), e = max(b, min(q.e, (int32_t)nt));
    fb = max(b, min(fb, e));
    fe = max(fb, min(fe, e));
    rows[x] = b < e ? make_int4(b, fb, fe, e) : make_int4(0, 0, 0, 0);  // empty (ring steps only)
    full = fe - fb;
    part = (e - b) - full;
  }
  // block reduction of the per-tile counts
  __shared__ long long sp[32], sf[32];
  for (int o = 16; o > 0; o >>= 1) {
    part += __shfl_down_sync(0xffffffffu, part, o);
    full += __shfl_down_sync(0xffffffffu, full, o);
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) { sp[w] = part; sf[w] = full; }
  __syncthreads();
  if (w == 0) {
    const int nw = blockDim.x >> 5;
    part = l < nw ? sp[l] : 0;
    full = l < nw ? sf[l] : 0;
    for (int o = 16; o > 0; o >>= 1) {
      part += __shfl_down_sync(0xffffffffu, part, o);
      full += __shfl_down_sync(0xffffffffu, full, o);
    }
    if (l == 0) {
      atomicAdd(reinterpret_cast<unsigned long long*>(&h->n_partial), (unsigned long long)part);
      atomicAdd(reinterpret_cast<unsigned long long*>(&h->n_full), (unsigned long long)full);
    }
  }
}

// one thread per (key shard, key tile j): the query tiles of the device the shard serves whose
// ranges contain j, found by binary search over the tile index.
__global__ void k_kv_rows(Geo geo, int64_t nt, int4* __restrict__ rows) {
  const int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (x >= geo.kv_count * nt) return;
  const int m = (int)(x / nt);
  const int64_t j = x - m * nt;
  const int d = dev_of_shard(geo.g, m);
  if (d >= geo.ndev) {  // the shard serves no device of the launch at this step
    rows[x] = make_int4(0, 0, 0, 0);
    return;
  }
  const Zig z = make_zig(geo.seg, geo.S, geo.causal, geo.g, d);
  // min i with e(i) > j ; max i with b(i) <= j ; min i with fe(i) > j ; max i with fb(i) <= j
  int64_t lo, hi;
  lo = 0; hi = nt;
  while (lo < hi) { int64_t md = (lo + hi) >> 1; if (q_tile_ranges(z, md, nt).e > j) hi = md; else lo = md + 1; }
  const int64_t qb = lo;
  lo = -1; hi = nt - 1;
  while (lo < hi) { int64_t md = (lo + hi + 1) >> 1; if (q_tile_ranges(z, md, nt).b <= j) lo = md; else hi = md - 1; }
  const int64_t qe = lo + 1;
  lo = 0; hi = nt;
  while (lo < hi) { int64_t md = (lo + hi) >> 1; if (q_tile_ranges(z, md, nt).fe > j) hi = md; else lo = md + 1; }
  int64_t qfb = lo;
  lo = -1; hi = nt - 1;
  while (lo < hi) { int64_t md = (lo + hi + 1) >> 1; if (q_tile_ranges(z, md, nt).fb <= j) lo = md; else hi = md - 1; }
  int64_t qfe = lo + 1;
  int32_t b = (int32_t)max((int64_t)0, min(qb, nt)), e = (int32_t)max((int64_t)b, min(qe, nt));
  if (qfb >= qfe) qfb = qfe = e;
  int32_t fb = (int32_t)max((int64_t)b, min(qfb, (int64_t)e));
  int32_t fe = (int32_t)max((int64_t)fb, min(qfe, (int64_t)e));
  rows[x] = b < e ? make_int4(b, fb, fe, e) : make_int4(0, 0, 0, 0);  // empty (ring steps only)
}

// Ring steps: the first or last row of a tile may see no key of the visiting shard while others
// do (a packed segment that began before the shard's chunks, or a tile straddling the device's two
// chunks), so the tile's range is reduced over all of its rows instead of read off its end rows.
// The keys seen by the rows of one tile still form one interval (the geometry leaves no gap), so
// [min lo, max hi] over the rows that see any key is exact; the full tiles are those inside
// [max lo, min hi] when every row sees some key.  One 128-thread block per tile; side 0 reduces the
// query rows of (device, query tile) blocks, side 1 the key rows of (shard, key tile) blocks.
__device__ __forceinline__ int64_t block_min(int64_t v, int64_t* sh) {
  for (int o = 16; o > 0; o >>= 1) v = min(v, (int64_t)__shfl_down_sync(0xffffffffu, v, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = v;
  __syncthreads();
  return min(min(sh[0], sh[1]), min(sh[2], sh[3]));
}

__global__ void __launch_bounds__(kTile) k_ring_rows(Geo geo, int64_t nt, int side, int4* __restrict__ rows,
                                                     TableHeader* h) {
  __shared__ int64_t sh[4];
  const int64_t x = blockIdx.x;
  const int u = (int)(x / nt);  // device (side 0) or key shard (side 1)
  const int64_t t = x - u * nt;
  const int d = side ? dev_of_shard(geo.g, u) : u;
  if (d >= geo.ndev) {  // a shard that serves no device of the launch at this step
    if (threadIdx.x == 0) rows[x] = make_int4(0, 0, 0, 0);
    return;
  }
  const Zig z = make_zig(geo.seg, geo.S, geo.causal, geo.g, d);
  const int64_t row = t * kTile + threadIdx.x;
  const int64_t big = INT64_MAX / 2;
  int64_t lo = big, hi = -1, lo_all = -big, hi_all = big;  // lo_all / hi_all: for max lo, min hi
  int64_t empty = 0;
  if (row < geo.S) {
    int64_t l, r;
    if (side) z.k_interval(row, l, r); else z.q_interval(row, l, r);
    if (l <= r) {
      lo = l; hi = r; lo_all = l; hi_all = r;
    } else {
      empty = 1;
    }
  }
  const int64_t min_lo = block_min(lo, sh);
  const int64_t max_hi = -block_min(-hi, sh);
  const int64_t max_lo = -block_min(-lo_all, sh);
  const int64_t min_hi = block_min(hi_all, sh);
  const int64_t any_empty = -block_min(-empty, sh);
  if (threadIdx.x != 0) return;
  if (max_hi < 0) {
    rows[x] = make_int4(0, 0, 0, 0);
    return;
  }
  const int32_t b = (int32_t)(min_lo / kTile), e = (int32_t)(max_hi / kTile + 1);
  int32_t fb = e, fe = e;
  if (!any_empty) {
    const int64_t f0 = ceil_div(max_lo, kTile);
    const int64_t f1 = min_hi >= geo.S - 1 ? nt : (min_hi + 1) / kTile;
    if (f0 < f1) {
      fb = (int32_t)max((int64_t)b, f0);
      fe = (int32_t)min((int64_t)e, f1);
    }
  }
  rows[x] = make_int4(b, fb, fe, e);
  if (side == 0) {
    atomicAdd(reinterpret_cast<unsigned long long*>(&h->n_partial), (unsigned long long)((e - b) - (fe - fb)));
    atomicAdd(reinterpret_cast<unsigned long long*>(&h->n_full), (unsigned long long)(fe - fb));
  }
}

// Dispatch orders by rank: entry x goes to position #{y : work(y) > work(x)} + #{y : work(y) ==
// work(x), y before x in the tie order}, a permutation.  Blocks [0, nbq) rank the query-tile pairs
// of all devices (ties: later entry first), the rest the key tiles of all shards (ties: earlier
// entry first).  Each block stages the works 256 at a time in shared memory.
__global__ void k_orders(const int4* __restrict__ q_rows, const int4* __restrict__ kv_rows, int64_t nt, int ndev,
                         int kv_count, int nbq, int32_t* __restrict__ q_order, int32_t* __restrict__ kv_order) {
  const bool qside = (int)blockIdx.x < nbq;
  const int64_t npairs = (nt + 1) / 2;
  const int64_t n = qside ? ndev * npairs : kv_count * nt;
  const int64_t x = (int64_t)(qside ? blockIdx.x : blockIdx.x - nbq) * blockDim.x + threadIdx.x;
  auto work = [&](int64_t y) -> int32_t {
    if (qside) {
      const int64_t d = y / npairs, p = y - d * npairs;
      const int4 a = q_rows[d * nt + 2 * p];
      int32_t w = a.w - a.x;
      if (2 * p + 1 < nt) {
        const int4 b = q_rows[d * nt + 2 * p + 1];
        w += b.w - b.x;
      }
      return w;
    }
    const int4 a = kv_rows[y];
    return a.w - a.x;
  };
  const int32_t wx = x < n ? work(x) : 0;
  __shared__ int32_t ws[256];
  int64_t rank = 0;
  for (int64_t base = 0; base < n; base += 256) {
    __syncthreads();
    if (base + threadIdx.x < n) ws[threadIdx.x] = work(base + threadIdx.x);
    __syncthreads();
    const int cnt = (int)min((int64_t)256, n - base);
    for (int t = 0; t < cnt; ++t) {
      const int64_t y = base + t;
      const int32_t wy = ws[t];
      rank += (wy > wx) || (wy == wx && (qside ? y > x : y < x));
    }
  }
  if (x < n) (qside ? q_order : kv_order)[rank] = (int32_t)x;
}

cudaError_t build(const Geo& geo, int64_t seg_len, void* table, cudaStream_t st) {
  const int64_t S = geo.S;
  const int64_t nt = ceil_div(S, kTile);
  TableHeader* h = reinterpret_cast<TableHeader*>(table);
  int4* q_rows = const_cast<int4*>(table_q_rows(table));
  int4* kv_rows = const_cast<int4*>(table_kv_rows(table, S, geo.ndev));
  k_table_init<<<1, 32, 0, st>>>(h, (int)nt);
  note_launch();
  if (geo.seg && seg_len > 1) {
    int64_t blocks = std::min<int64_t>(ceil_div(seg_len, 256), 152 * 8);
    k_check_monotone<<<(unsigned)blocks, 256, 0, st>>>(geo.seg, seg_len, h);
    note_launch();
  }
  if (geo.g.P == 0) {
    k_q_rows<<<(unsigned)ceil_div(nt, 256), 256, 0, st>>>(geo, nt, q_rows, h);
    note_launch();
    k_kv_rows<<<(unsigned)ceil_div(nt, 256), 256, 0, st>>>(geo, nt, kv_rows);
    note_launch();
  } else {
    k_ring_rows<<<(unsigned)(geo.ndev * nt), kTile, 0, st>>>(geo, nt, 0, q_rows, h);
    note_launch();
    k_ring_rows<<<(unsigned)(geo.kv_count * nt), kTile, 0, st>>>(geo, nt, 1, kv_rows, h);
    note_launch();
  }
  const int nbq = (int)ceil_div(geo.ndev * ((nt + 1) / 2), 256), nbk = (int)ceil_div(geo.kv_count * nt, 256);
  k_orders<<<nbq + nbk, 256, 0, st>>>(q_rows, kv_rows, nt, geo.ndev, geo.kv_count, nbq,
                                      const_cast<int32_t*>(table_q_order(table, S, geo.ndev, geo.kv_count)),
                                      const_cast<int32_t*>(table_kv_order(table, S, geo.ndev, geo.kv_count)));
  note_launch();
  return cudaGetLastError();
}

}  // namespace

size_t tile_table_bytes(int64_t S, int ndev, int kv_count) {
  const size_t nt = (size_t)ceil_div(S, kTile);
  const size_t bytes = sizeof(TableHeader) + (size_t)(ndev + kv_count) * nt * 16 + 4 * (ndev * ((nt + 1) / 2) + kv_count * nt);
  return (bytes + 15) & ~(size_t)15;
}

cudaError_t launch_tile_table(int64_t S, int causal, const int32_t* seg, void* table, cudaStream_t st) {
  return build(Geo{seg, S, causal, RingGeom{}, 1, 1}, S, table, st);
}

cudaError_t launch_ring_table(int64_t S, int causal, const int32_t* seg, const RingGeom& g, int ndev, int kv_count,
                              void* table, cudaStream_t st) {
  return build(Geo{seg, S, causal, g, ndev, kv_count}, 2 * (int64_t)g.P * g.C, table, st);
}

}  // namespace upipe
