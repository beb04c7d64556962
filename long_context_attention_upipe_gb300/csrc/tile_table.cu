// Tile-skip table for 128x128 tiles under the causal + same-segment mask.
//
// Splash attention skips blocks whose every (query, key) pair is masked and handles packed
// sequences without padding (MaxText long-context article, techmoon.xyz, paragraph on the
// shared attention kernel).  With non-decreasing segment ids, query row r sees exactly the
// keys [segstart(r), causal ? r : segend(r)]; both ends are non-decreasing in r, so for a
// query tile the non-empty key tiles form one range and the full ones a sub-range, and the
// same holds per key tile.  Each thread derives one row of the table from four binary
// searches over the segment ids; nothing is materialised per element.
#include "common.cuh"
#include "internal.h"

namespace upipe {

namespace {

struct SegView {
  const int32_t* seg;  // NULL: one segment
  int64_t S;
  __device__ __forceinline__ int64_t start(int64_t r) const {  // first position of r's segment
    if (!seg) return 0;
    const int32_t v = seg[r];
    int64_t lo = 0, hi = r;  // first p in [0, r] with seg[p] >= v
    while (lo < hi) {
      int64_t mid = (lo + hi) >> 1;
      if (seg[mid] >= v) hi = mid; else lo = mid + 1;
    }
    return lo;
  }
  __device__ __forceinline__ int64_t end(int64_t r) const {  // last position of r's segment
    if (!seg) return S - 1;
    const int32_t v = seg[r];
    int64_t lo = r, hi = S - 1;  // last p in [r, S) with seg[p] <= v
    while (lo < hi) {
      int64_t mid = (lo + hi + 1) >> 1;
      if (seg[mid] <= v) lo = mid; else hi = mid - 1;
    }
    return lo;
  }
};

// Raw range functions of query tile i (all non-decreasing in i for non-decreasing ids).
struct QTileRanges {
  int32_t b, e;    // non-empty key tiles [b, e)
  int32_t fb, fe;  // full key tiles [fb, fe), possibly empty (fb >= fe)
};

__device__ __forceinline__ QTileRanges q_tile_ranges(const SegView& sv, int64_t i, int causal, int64_t nt) {
  const int64_t S = sv.S;
  const int64_t r0 = i * kTile;
  const int64_t rl = min(S, r0 + kTile) - 1;
  const int64_t lo = sv.start(r0);
  const int64_t hi = causal ? rl : sv.end(rl);
  QTileRanges q;
  q.b = (int32_t)(lo / kTile);
  q.e = (int32_t)(hi / kTile + 1);
  q.fb = (int32_t)ceil_div(sv.start(rl), kTile);
  const int64_t lim = causal ? r0 : sv.end(r0);  // every key column c <= lim is seen by all rows
  const int64_t last = (lim >= S - 1) ? nt - 1 : (lim + 1) / kTile - 1;
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

__global__ void k_q_rows(SegView sv, int causal, int64_t nt, int4* __restrict__ rows, TableHeader* h) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  long long part = 0, full = 0;
  if (i < nt) {
    QTileRanges q = q_tile_ranges(sv, i, causal, nt);
    int32_t fb = q.fb, fe = q.fe;
    if (fb >= fe) fb = fe = q.e;
    // clamp (only matters when the ids are not sorted; the error word is set then)
    int32_t b = max(0, min(q.b, (int32_t)nt)), e = max(b, min(q.e, (int32_t)nt));
    fb = max(b, min(fb, e));
    fe = max(fb, min(fe, e));
    rows[i] = make_int4(b, fb, fe, e);
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

// kv tile j: the query tiles whose ranges contain j, found by binary search over i.
__global__ void k_kv_rows(SegView sv, int causal, int64_t nt, int4* __restrict__ rows) {
  const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= nt) return;
  // min i with e(i) > j ; max i with b(i) <= j ; min i with fe(i) > j ; max i with fb(i) <= j
  int64_t lo, hi;
  lo = 0; hi = nt;
  while (lo < hi) { int64_t m = (lo + hi) >> 1; if (q_tile_ranges(sv, m, causal, nt).e > j) hi = m; else lo = m + 1; }
  const int64_t qb = lo;
  lo = -1; hi = nt - 1;
  while (lo < hi) { int64_t m = (lo + hi + 1) >> 1; if (q_tile_ranges(sv, m, causal, nt).b <= j) lo = m; else hi = m - 1; }
  const int64_t qe = lo + 1;
  lo = 0; hi = nt;
  while (lo < hi) { int64_t m = (lo + hi) >> 1; if (q_tile_ranges(sv, m, causal, nt).fe > j) hi = m; else lo = m + 1; }
  int64_t qfb = lo;
  lo = -1; hi = nt - 1;
  while (lo < hi) { int64_t m = (lo + hi + 1) >> 1; if (q_tile_ranges(sv, m, causal, nt).fb <= j) lo = m; else hi = m - 1; }
  int64_t qfe = lo + 1;
  int32_t b = (int32_t)max((int64_t)0, min(qb, nt)), e = (int32_t)max((int64_t)b, min(qe, nt));
  if (qfb >= qfe) qfb = qfe = e;
  int32_t fb = (int32_t)max((int64_t)b, min(qfb, (int64_t)e));
  int32_t fe = (int32_t)max((int64_t)fb, min(qfe, (int64_t)e));
  rows[j] = make_int4(b, fb, fe, e);
}

// Dispatch orders by rank: entry x goes to position #{y : work(y) > work(x)} + #{y : work(y) ==
// work(x), y before x in the tie order}, a permutation.  Blocks [0, nbq) rank the query-tile pairs
// (ties: later pair first), the rest the key tiles (ties: earlier tile first).  Each block stages
// the works 256 at a time in shared memory.
__global__ void k_orders(const int4* __restrict__ q_rows, const int4* __restrict__ kv_rows, int64_t nt, int nbq,
                         int32_t* __restrict__ q_order, int32_t* __restrict__ kv_order) {
  const bool qside = (int)blockIdx.x < nbq;
  const int64_t n = qside ? (nt + 1) / 2 : nt;
  const int64_t x = (int64_t)(qside ? blockIdx.x : blockIdx.x - nbq) * blockDim.x + threadIdx.x;
  auto work = [&](int64_t y) -> int32_t {
    if (qside) {
      const int4 a = q_rows[2 * y];
      int32_t w = a.w - a.x;
      if (2 * y + 1 < nt) {
        const int4 b = q_rows[2 * y + 1];
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

}  // namespace

size_t tile_table_bytes(int64_t S) {
  const size_t nt = (size_t)ceil_div(S, kTile);
  const size_t bytes = sizeof(TableHeader) + 2 * nt * 16 + 4 * ((nt + 1) / 2 + nt);
  return (bytes + 15) & ~(size_t)15;
}

cudaError_t launch_tile_table(int64_t S, int causal, const int32_t* seg, void* table, cudaStream_t st) {
  const int64_t nt = ceil_div(S, kTile);
  TableHeader* h = reinterpret_cast<TableHeader*>(table);
  int4* q_rows = reinterpret_cast<int4*>(reinterpret_cast<char*>(table) + sizeof(TableHeader));
  int4* kv_rows = q_rows + nt;
  k_table_init<<<1, 32, 0, st>>>(h, (int)nt);
  note_launch();
  if (seg && S > 1) {
    int64_t blocks = std::min<int64_t>(ceil_div(S, 256), 152 * 8);
    k_check_monotone<<<(unsigned)blocks, 256, 0, st>>>(seg, S, h);
    note_launch();
  }
  SegView sv{seg, S};
  const unsigned tb = (unsigned)ceil_div(nt, 256);
  k_q_rows<<<tb, 256, 0, st>>>(sv, causal, nt, q_rows, h);
  note_launch();
  k_kv_rows<<<tb, 256, 0, st>>>(sv, causal, nt, kv_rows);
  note_launch();
  const int nbq = (int)ceil_div((nt + 1) / 2, 256), nbk = (int)ceil_div(nt, 256);
  k_orders<<<nbq + nbk, 256, 0, st>>>(q_rows, kv_rows, nt, nbq, const_cast<int32_t*>(table_q_order(table, S)),
                                      const_cast<int32_t*>(table_kv_order(table, S)));
  note_launch();
  return cudaGetLastError();
}

}  // namespace upipe
