// Projection GEMMs of the layer on the 5th-generation tensor cores (tcgen05, TMEM, TMA).
//
// C[M, N] = A[M, K] * B[N, K]^T, bf16 operands, fp32 accumulation in TMEM, one of the epilogues
// of GemmEpilogue.  Every operand is read by TMA in 64 x 64 boxes (128-byte swizzle) from a 2-D
// or 3-D tensor map, K-major or MN-major, so each projection of the chunk loop reads its
// operands in place: head-major activations ([heads][S][Dh], a 3-D map whose third coordinate
// is the head), column slices of Wo (a 2-D map with the row stride of Wo) and the row blocks of
// Wqkv that belong to a chunk (a 2-D map plus the first row of each block).
//
// Persistent kernel, one CTA per SM, launched as CTA pairs (clusters of two) that compute one
// 256 x 256 output tile with the pair form of the tensor core (tcgen05 cta_group::2): each CTA
// holds its own 128 rows of A and one half (128 columns) of B, the even CTA issues M256 N256
// MMAs that read both CTAs' shared memory, and each CTA's TMEM receives its 128 rows of D.  A
// stage is 32 KB per CTA (half of a single-CTA 128 x 256 tile's 48 KB), so six stages fit and
// the tensor core reads half as many shared-memory bytes per FLOP.  6 warps per CTA:
//   warps 0, 6, 7, 8  TMA producers, one 64 x 64 box of a stage each (A rows 0-63, A rows 64-127,
//              B rows 0-63, B rows 64-127; one thread could not issue a stage's four loads within
//              its MMA time) over a 6-stage ring of (A 128x64, B half 128x64) tiles; both CTAs'
//              loads count on the even CTA's stage barrier; a stage is refilled once the MMAs
//              that read it have completed (a pair commit arrives in both CTAs)
//   warp 1     TMEM owner in both CTAs; in the even CTA the MMA issuer (one thread): 4 MMAs
//              (M256 N256 K16) per stage into one of two TMEM accumulators, so the epilogue of
//              a tile overlaps the next tile
//   warps 2-5  epilogue: one output row per thread (TMEM lane), 32 columns at a time; both CTAs'
//              epilogues release an accumulator on the even CTA's barrier
// Plain row-major fp32 outputs (and split-K partials) leave through shared memory: each epilogue
// warp stages a 32 x 32 fp32 box (128-byte swizzle, double-buffered) and one lane hands it to a
// TMA bulk store, or to a TMA bulk reduce-add for C += A B^T, so the read-modify-write of an
// accumulator runs in L2 without the SM waiting on its loads.  Other outputs are stored per
// thread.  Split-K (weight gradients, K = S) writes fp32 partials that k_split_reduce sums in order.
#include <cstring>

#include "internal.h"
#include "tc_common.cuh"

namespace upipe {

namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 6, THREADS = 288;  // BM: rows per CTA of the pair
constexpr uint32_t BOX = 64 * 64 * 2;          // one 64 x 64 bf16 box, 8 KB
constexpr uint32_t TILE_A = 2 * BOX;           // 128 x 64 A tile (this CTA's rows)
constexpr uint32_t TILE_B = 2 * BOX;           // 128 x 64: this CTA's half of the 256-wide B tile
constexpr uint32_t STAGE = TILE_A + TILE_B;
constexpr uint32_t STG_OFF = STAGES * STAGE;         // epilogue staging: 4 warps x 2 boxes of 32 x 32 fp32
constexpr uint32_t STG_BOX = 32 * 32 * 4;
constexpr uint32_t BAR_OFF = STG_OFF + 8 * STG_BOX;
constexpr uint32_t SMEM_BYTES = BAR_OFF + 256 + 1024;

struct TcOpDev {
  int k_major, rank, blk_shift, blk_dim;
  int32_t row_base[kMaxBlocks];
};

struct TcGemmParams {
  int64_t M, N, K;
  TcOpDev a, b;
  GemmOutput c;
  int epi;
  int split_k;
  int64_t k_per_split;  // multiple of BK
  int tiles_m, tiles_n;
  float* split_out;
  int tma_out;  // 0: per-thread stores; 1: TMA store (2-D map); 2: TMA reduce-add (2-D); 3: TMA store of split partials (3-D)
  uint64_t wait_ns;  // limit of each bounded wait
  int m_fast;   // unit order: M-tile pairs fastest (B, the larger operand, read once) or N tiles fastest
};

enum : int { TMA_OUT_NONE = 0, TMA_OUT_STORE = 1, TMA_OUT_ADD = 2, TMA_OUT_SPLIT = 3 };

// TMA coordinates of the 64 x 64 box that starts at logical (mn, k).
__device__ __forceinline__ void box_coords(const TcOpDev& o, int64_t mn, int64_t k, int& c0, int& c1, int& c2) {
  int b = 0;
  if (o.blk_shift >= 0) {
    const int64_t mask = (int64_t(1) << o.blk_shift) - 1;
    if (o.blk_dim == 0) { b = (int)(mn >> o.blk_shift); mn &= mask; }
    else { b = (int)(k >> o.blk_shift); k &= mask; }
  }
  const int64_t inner = o.k_major ? k : mn, outer = o.k_major ? mn : k;
  if (o.rank == 3) {
    c0 = (int)inner; c1 = (int)outer; c2 = b;
  } else {
    c0 = (int)inner; c1 = (int)(outer + (o.blk_shift >= 0 ? o.row_base[b] : 0)); c2 = 0;
  }
}

// A box into this CTA's shared memory, counted on the even CTA's barrier (shared::cluster address).
__device__ __forceinline__ void load_box_pair(uint8_t* dst, const CUtensorMap* map, const TcOpDev& o,
                                              uint32_t bar_cluster, int64_t mn, int64_t k) {
  int c0, c1, c2;
  box_coords(o, mn, k, c0, c1, c2);
  if (o.rank == 3) tc::tma_load_3d_pair(dst, map, bar_cluster, c0, c1, c2);
  else tc::tma_load_2d_pair(dst, map, bar_cluster, c0, c1);
}

// smem descriptor of one operand tile at MMA K-step k16 (16 elements)
__device__ __forceinline__ uint64_t tile_desc(uint32_t base, int k_major, int k16) {
  return k_major ? tc::sdesc_sw128(base + k16 * 32, 16, 1024)        // 128 rows x 128 B, 8-row groups
                 : tc::sdesc_sw128(base + k16 * 2048, BOX, 1024);    // two 64-wide MN atoms, BOX apart
}

template <typename T>
__device__ __forceinline__ T* out_ptr(const GemmOutput& o, int64_t m, int64_t n) {
  int b = 0;
  if (o.blk_shift >= 0) {
    const int64_t idx = o.blk_dim == 0 ? m : n;
    b = (int)(idx >> o.blk_shift);
    const int64_t local = idx & ((int64_t(1) << o.blk_shift) - 1);
    if (o.blk_dim == 0) m = local; else n = local;
  }
  return reinterpret_cast<T*>(o.blk[b]) + m * o.ld + n;
}

__global__ void __launch_bounds__(THREADS, 1) k_gemm_tc(const __grid_constant__ CUtensorMap ta,
                                                        const __grid_constant__ CUtensorMap tb,
                                                        const __grid_constant__ CUtensorMap tout, TcGemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BAR_OFF);
  uint64_t* full = bars;                // [STAGES]
  uint64_t* empty = bars + STAGES;      // [STAGES]
  uint64_t* acc_full = bars + 2 * STAGES;       // [2]
  uint64_t* acc_empty = bars + 2 * STAGES + 2;  // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * STAGES + 5);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // work unit = a pair of M tiles (2 pm, 2 pm + 1) of one N tile and K split; CTA `crank` of the
  // cluster takes M tile 2 pm + crank (a tile past M is computed on zero-filled rows and dropped)
  const int crank = (int)tc::cluster_ctarank();
  const int cid = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;
  const int tiles_mp = (p.tiles_m + 1) >> 1;
  const int64_t tiles_pn = (int64_t)tiles_mp * p.tiles_n;
  const int64_t n_tiles = tiles_pn * p.split_k;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      tc::mbar_init(&full[i], 1);   // even CTA: its producer's arrival + both CTAs' bytes
      tc::mbar_init(&empty[i], 1);  // the even CTA's MMA commit (a pair commit arrives in both)
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&acc_full[i], 1);
      tc::mbar_init(&acc_empty[i], 2 * 128);  // even CTA: both CTAs' epilogue threads
    }
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc_pair(tmem_slot, 2 * BN);
    tc::tmem_relinquish_pair();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::cluster_sync();  // the peer's barriers are initialised before any pair commit or load reaches them
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  // unit t -> (m tile, n tile, split).  The fast index sweeps its whole operand once for every
  // step of the slow index: with N fastest B is re-read for every pair of M tiles, with M fastest
  // A for every N tile.  The launcher sweeps the smaller operand (the one L2 can hold), so the
  // larger one is read from DRAM about once: an MLP's gate/up weights (28672 x 4096) do not fit in
  // L2 and are swept over its 8192-row tiles of X otherwise.
  auto decode = [&](int64_t t, int& tm, int& tn, int& ks) {
    ks = (int)(t / tiles_pn);
    const int64_t r = t % tiles_pn;
    if (p.m_fast) {
      tm = 2 * (int)(r % tiles_mp) + crank;
      tn = (int)(r / tiles_mp);
    } else {
      tm = 2 * (int)(r / p.tiles_n) + crank;
      tn = (int)(r % p.tiles_n);
    }
  };
  auto k_tiles = [&](int ks) {
    const int64_t kb = (int64_t)ks * p.k_per_split;
    const int64_t ke = min(p.K, kb + p.k_per_split);
    return ke > kb ? (int)ceil_div(ke - kb, BK) : 0;
  };

  if (warp == 0 || warp >= 6) {
    // one box per warp and stage: warps 0, 6 load A rows 0-63 / 64-127 (warp 0 also announces the
    // stage's bytes), warps 7, 8 load this CTA's half of B, rows 0-63 / 64-127
    const int q = warp == 0 ? 0 : warp - 5;  // 0..3
    const bool is_a = q < 2;
    if (lane == 0) {
      tc::prefetch_tmap(is_a ? &ta : &tb);
      const uint32_t full0 = tc::mapa_cluster(smem_u32(&full[0]), 0);  // the even CTA's stage barriers
      int it = 0;
      bool ok = true;
      for (int64_t t = cid; ok && t < n_tiles; t += n_clusters) {
        int tm, tn, ks;
        decode(t, tm, tn, ks);
        const int nk = k_tiles(ks);
        for (int kt = 0; kt < nk; ++kt, ++it) {
          const int s = it % STAGES;
          if (it >= STAGES && !(ok = tc::mbar_wait(&empty[s], ((it / STAGES) - 1) & 1, abort_flag, nullptr, p.wait_ns))) break;
          if (q == 0 && crank == 0) tc::mbar_arrive_expect_tx(&full[s], 2 * STAGE);  // both CTAs' A and B halves
          const uint32_t bar = full0 + s * 8;
          uint8_t* sa = smem + s * STAGE;
          const int64_t k = (int64_t)ks * p.k_per_split + (int64_t)kt * BK;
          const int i = q & 1;
          if (is_a) load_box_pair(sa + i * BOX, &ta, p.a, bar, (int64_t)tm * BM + 64 * i, k);
          else  // B columns [tn*BN + 128*crank, +128): this CTA's half
            load_box_pair(sa + TILE_A + i * BOX, &tb, p.b, bar, (int64_t)tn * BN + 128 * crank + 64 * i, k);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && crank == 0) {
      const uint32_t idesc = tc::idesc_bf16(2 * BM, BN, !p.a.k_major, !p.b.k_major);
      // descriptors of stage 0, stepped by constant offsets (stage, K step) in the loop
      const uint32_t s0 = smem_u32(smem);
      const uint64_t a0 = tile_desc(s0, p.a.k_major, 0), b0 = tile_desc(s0 + TILE_A, p.b.k_major, 0);
      const uint32_t a_step = p.a.k_major ? 32 : 2048, b_step = p.b.k_major ? 32 : 2048;  // bytes per K16 step
      int it = 0, tcount = 0;
      bool ok = true;
      for (int64_t t = cid; ok && t < n_tiles; t += n_clusters, ++tcount) {
        int tm, tn, ks;
        decode(t, tm, tn, ks);
        const int nk = k_tiles(ks);
        const int buf = tcount & 1;
        if (tcount >= 2 && !(ok = tc::mbar_wait(&acc_empty[buf], ((tcount >> 1) - 1) & 1, abort_flag, nullptr, p.wait_ns))) break;
        tc::fence_after_sync();
        const uint32_t d = tmem + buf * BN;
        for (int kt = 0; kt < nk; ++kt, ++it) {
          const int s = it % STAGES;
          if (!(ok = tc::mbar_wait(&full[s], (it / STAGES) & 1, abort_flag, nullptr, p.wait_ns))) break;
          tc::fence_after_sync();
          const uint64_t ad = tc::opaque(tc::sdesc_add(a0, s * STAGE)), bd = tc::opaque(tc::sdesc_add(b0, s * STAGE));
#pragma unroll
          for (int k16 = 0; k16 < BK / 16; ++k16)
            tc::mma_ss_pair(d, tc::sdesc_add(ad, k16 * a_step), tc::sdesc_add(bd, k16 * b_step), idesc, kt > 0 || k16 > 0);
          tc::mma_commit_pair(&empty[s]);  // release the stage in both CTAs
        }
        tc::mma_commit_pair(&acc_full[buf]);
      }
    }
    __syncwarp();
  } else {
    // epilogue warps 2..5: TMEM lanes 32 * (warp % 4) + lane
    const int row_in_tile = 32 * (warp & 3) + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    int tcount = 0, nstage = 0;
    bool ok = true;
    for (int64_t t = cid; t < n_tiles; t += n_clusters, ++tcount) {
      int tm, tn, ks;
      decode(t, tm, tn, ks);
      const int nk = k_tiles(ks);
      const int buf = tcount & 1;
      if (ok) ok = tc::mbar_wait(&acc_full[buf], (tcount >> 1) & 1, abort_flag, nullptr, p.wait_ns);
      tc::fence_after_sync();
      const int64_t m = (int64_t)tm * BM + row_in_tile;
      const bool m_ok = m < p.M;
#pragma unroll 1
      for (int ch = 0; ch < BN / 32; ++ch) {
        uint32_t v[32];
        tc::tmem_ld32(lane_addr + buf * BN + ch * 32, v);
        tc::tmem_ld_wait();
        if (nk == 0) {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;
        }
        const int64_t n0 = (int64_t)tn * BN + ch * 32;
        if (p.tma_out != TMA_OUT_NONE) {
          // stage this warp's 32 rows x 32 columns, row `lane` with 128-byte swizzle (16-byte
          // chunk j of row r at chunk j ^ (r % 8)), then one lane issues the bulk copy.  Only
          // boxes that are issued are staged, so the two buffers alternate with the committed
          // groups and "at most one group still reading" frees the buffer about to be written.
          const int64_t y = (int64_t)tm * BM + 32 * (warp & 3);
          if (!__all_sync(0xffffffffu, ok) || n0 >= p.N || y >= p.M) continue;
          uint8_t* box = smem + STG_OFF + ((warp & 3) * 2 + (nstage & 1)) * STG_BOX;
          ++nstage;
          if (lane == 0) tc::bulk_wait_read<1>();  // the copy that last read this buffer is done
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<float4*>(box + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]), __uint_as_float(v[4 * j + 2]),
                            __uint_as_float(v[4 * j + 3]));
          tc::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (p.tma_out == TMA_OUT_STORE) tc::tma_store_2d(&tout, box, (int)n0, (int)y);
            else if (p.tma_out == TMA_OUT_ADD) tc::tma_reduce_add_2d(&tout, box, (int)n0, (int)y);
            else tc::tma_store_3d(&tout, box, (int)n0, (int)y, ks);
            tc::bulk_commit();
          }
          continue;
        }
        if (!ok || !m_ok || n0 >= p.N) continue;
        const int ncols = (int)min((int64_t)32, p.N - n0);  // multiple of 8
        if (p.split_out) {
          float* dst = p.split_out + ((int64_t)ks * p.M + m) * p.N + n0;
          _Pragma("unroll") for (int i = 0; i < 32; i += 4) if (i < ncols)
            *reinterpret_cast<float4*>(dst + i) = make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                                                              __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
          continue;
        }
        switch (p.epi) {
          case EPI_STORE_BF16: {
            bf16* dst = out_ptr<bf16>(p.c, m, n0);
            _Pragma("unroll") for (int i = 0; i < 32; i += 8) if (i < ncols) {
              uint4 q;
              q.x = tc::pack_bf16x2(__uint_as_float(v[i]), __uint_as_float(v[i + 1]));
              q.y = tc::pack_bf16x2(__uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
              q.z = tc::pack_bf16x2(__uint_as_float(v[i + 4]), __uint_as_float(v[i + 5]));
              q.w = tc::pack_bf16x2(__uint_as_float(v[i + 6]), __uint_as_float(v[i + 7]));
              *reinterpret_cast<uint4*>(dst + i) = q;
            }
            break;
          }
          case EPI_STORE_F32: {
            float* dst = out_ptr<float>(p.c, m, n0);
            _Pragma("unroll") for (int i = 0; i < 32; i += 4) if (i < ncols)
              *reinterpret_cast<float4*>(dst + i) = make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                                                                __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
            break;
          }
          case EPI_ACC_F32: {
            float* dst = out_ptr<float>(p.c, m, n0);
            _Pragma("unroll") for (int i = 0; i < 32; i += 4) if (i < ncols) {
              float4 o = *reinterpret_cast<float4*>(dst + i);
              o.x += __uint_as_float(v[i]); o.y += __uint_as_float(v[i + 1]);
              o.z += __uint_as_float(v[i + 2]); o.w += __uint_as_float(v[i + 3]);
              *reinterpret_cast<float4*>(dst + i) = o;
            }
            break;
          }
          case EPI_ACC_BF16: {
            bf16* dst = out_ptr<bf16>(p.c, m, n0);
            _Pragma("unroll") for (int i = 0; i < 32; i += 8) if (i < ncols) {
              uint4 q = *reinterpret_cast<uint4*>(dst + i);
              __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&q);
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const float2 f = __bfloat1622float2(h2[u]);
                h2[u] = __floats2bfloat162_rn(f.x + __uint_as_float(v[i + 2 * u]), f.y + __uint_as_float(v[i + 2 * u + 1]));
              }
              *reinterpret_cast<uint4*>(dst + i) = q;
            }
            break;
          }
        }
      }
      tc::fence_before_sync();
      tc::mbar_arrive_cluster(tc::mapa_cluster(smem_u32(&acc_empty[buf]), 0));  // on the even CTA's barrier
    }
    if (lane == 0) tc::bulk_wait_all();  // bulk stores complete before the CTA exits
    __syncwarp();
  }
  tc::fence_before_sync();
  __syncthreads();
  // the peer may still load into this CTA's shared memory or arrive on its barriers until
  // its own last MMAs are done: leave together
  tc::cluster_sync();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc_pair(tmem, 2 * BN);
  }
}

// Fixed-order reduction of split-K partials into the (blocked) fp32 output (or onto it).
__global__ void k_split_reduce(const float* __restrict__ part, int splits, int64_t M, int64_t N, GemmOutput out,
                               int accumulate) {
  const int64_t total = M * N / 4;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int64_t e = i * 4;
    const int64_t m = e / N, n = e % N;
    float4 s = reinterpret_cast<const float4*>(part)[i];
    for (int z = 1; z < splits; ++z) {
      const float4 v = reinterpret_cast<const float4*>(part + (int64_t)z * M * N)[i];
      s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
    }
    float4* dst = reinterpret_cast<float4*>(out_ptr<float>(out, m, n));
    if (accumulate) {
      const float4 o = *dst;
      s.x += o.x; s.y += o.y; s.z += o.z; s.w += o.w;
    }
    *dst = s;
  }
}

bool make_map(CUtensorMap* map, const TcOperand& o) {
  if (o.rank == 3) return make_tmap_3d_bf16(map, o.base, o.inner, o.outer, o.planes, 64, 64, o.plane_stride);
  return make_tmap_2d_bf16(map, o.base, o.inner, o.outer, o.row_stride, 64, 64);
}

bool aligned16(const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; }

TcOpDev dev_op(const TcOperand& o) {
  TcOpDev d{};
  d.k_major = o.k_major;
  d.rank = o.rank;
  d.blk_shift = o.blk_shift;
  d.blk_dim = o.blk_dim;
  for (int i = 0; i < kMaxBlocks; ++i) d.row_base[i] = o.row_base[i];
  return d;
}

}  // namespace

size_t gemm_split_scratch_bytes(int64_t M, int64_t N, int split_k) {
  return split_k > 1 ? (size_t)split_k * M * N * sizeof(float) : 0;
}

// Split K until the tile count covers two waves of the SMs (each split keeps >= 2048 of K).
int gemm_pick_split(int64_t M, int64_t N, int64_t K, int num_sms) {
  const int64_t tiles = ceil_div(M, BM) * ceil_div(N, BN);
  int split = 1;
  while (tiles * split < 2 * num_sms && K / (split * 2) >= 2048 && split < 32) split *= 2;
  return split;
}

cudaError_t launch_split_reduce(const float* part, int splits, int64_t M, int64_t N, const GemmOutput& out,
                                int accumulate, cudaStream_t st) {
  const int64_t total4 = M * N / 4;
  const unsigned blocks = (unsigned)std::max<int64_t>(1, std::min<int64_t>(ceil_div(total4, 256), 152 * 8));
  k_split_reduce<<<blocks, 256, 0, st>>>(part, splits, M, N, out, accumulate);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_gemm_tc(const TcGemmArgs& g, int split_k, float* split_scratch, cudaStream_t st) {
  if (g.M <= 0 || g.N <= 0) return cudaSuccess;
  CUtensorMap ta, tb;
  if (!make_map(&ta, g.a) || !make_map(&tb, g.b)) return cudaErrorInvalidValue;
  TcGemmParams p{};
  p.M = g.M; p.N = g.N; p.K = g.K;
  p.a = dev_op(g.a);
  p.b = dev_op(g.b);
  p.c = g.c;
  p.epi = g.epi;
  const int64_t ktiles = ceil_div(g.K, BK);
  if (split_k < 1) split_k = 1;
  if (split_k > ktiles) split_k = (int)std::max<int64_t>(1, ktiles);
  p.split_k = split_k;
  p.k_per_split = ceil_div(ktiles, split_k) * BK;
  p.tiles_m = (int)ceil_div(g.M, BM);
  p.tiles_n = (int)ceil_div(g.N, BN);
  p.split_out = split_k > 1 ? split_scratch : nullptr;
  p.wait_ns = wait_limit_ns();
  p.m_fast = g.N > g.M;  // sweep the smaller operand A [M, K]
  // fp32 outputs through TMA where the layout allows it (16-byte aligned base and rows)
  CUtensorMap tout;
  std::memset(&tout, 0, sizeof(tout));
  p.tma_out = TMA_OUT_NONE;
  if (split_k > 1) {
    const uint64_t dims[3] = {(uint64_t)g.N, (uint64_t)g.M, (uint64_t)split_k};
    const uint64_t strides[2] = {(uint64_t)g.N * 4, (uint64_t)g.M * g.N * 4};
    if (g.N % 4 == 0 && aligned16(split_scratch) && make_tmap_f32_out(&tout, split_scratch, 3, dims, strides))
      p.tma_out = TMA_OUT_SPLIT;
  } else if ((g.epi == EPI_STORE_F32 || g.epi == EPI_ACC_F32) && g.c.blk_shift < 0) {
    const uint64_t dims[2] = {(uint64_t)g.N, (uint64_t)g.M};
    const uint64_t strides[1] = {(uint64_t)g.c.ld * 4};
    if (g.N % 4 == 0 && g.c.ld % 4 == 0 && aligned16(g.c.blk[0]) &&
        make_tmap_f32_out(&tout, g.c.blk[0], 2, dims, strides))
      p.tma_out = g.epi == EPI_ACC_F32 ? TMA_OUT_ADD : TMA_OUT_STORE;
  }
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      sms = 152;
  }
  const int64_t n_units = (int64_t)((p.tiles_m + 1) / 2) * p.tiles_n * split_k;  // M-tile pairs
  const int clusters = (int)std::max<int64_t>(1, std::min<int64_t>(n_units, sms / 2));
  cudaError_t e = cudaFuncSetAttribute(k_gemm_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(2 * clusters));
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k_gemm_tc, ta, tb, tout, p);
  note_launch();
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess || split_k <= 1) return e;
  return launch_split_reduce(split_scratch, split_k, g.M, g.N, g.c, g.split_accumulate, st);
}

}  // namespace upipe
