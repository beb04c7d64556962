// Projection GEMMs of the layer on the warp-level tensor core path (mma.sync m16n8k16).
//
// C[M, N] = A[M, K] * B[N, K]^T with bf16 operands and fp32 accumulation.  Operands and output
// are sets of row-major blocks (see GemmOperand), which covers every projection of the chunk
// loop without copies: the head-major Q/K/V/O/dO/dQ buffers, column slices of Wo and row
// slices of Wqkv.  CTA tile 128 x 128 x 32, 8 warps (2 x 4, warp tile 64 x 32), three-stage
// cp.async pipeline, padded shared-memory rows (conflict-free ldmatrix).
#include "common.cuh"
#include "internal.h"

namespace upipe {

namespace {

constexpr int BM = 128, BN = 128, BK = 32, STAGES = 3, THREADS = 256;
constexpr int KM_LD = BK + 8;    // k-major tile row: 40 elements (80 B)
constexpr int MN_LD = BM + 8;    // mn-major tile row: 136 elements (272 B)
constexpr int TILE_ELEMS = (BM * KM_LD > BK * MN_LD) ? BM * KM_LD : BK * MN_LD;

__device__ __forceinline__ const bf16* op_addr(const GemmOperand& op, int64_t mn, int64_t k) {
  int b = 0;
  if (op.blk_shift >= 0) {
    const int64_t idx = op.blk_dim == 0 ? mn : k;
    b = (int)(idx >> op.blk_shift);
    const int64_t local = idx & ((int64_t(1) << op.blk_shift) - 1);
    if (op.blk_dim == 0) mn = local; else k = local;
  }
  const bf16* base = reinterpret_cast<const bf16*>(op.blk[b]);
  return op.k_major ? base + mn * op.ld + k : base + k * op.ld + mn;
}

template <typename T>
__device__ __forceinline__ T* out_addr(const GemmOutput& o, int64_t m, int64_t n) {
  int b = 0;
  if (o.blk_shift >= 0) {
    const int64_t idx = o.blk_dim == 0 ? m : n;
    b = (int)(idx >> o.blk_shift);
    const int64_t local = idx & ((int64_t(1) << o.blk_shift) - 1);
    if (o.blk_dim == 0) m = local; else n = local;
  }
  return reinterpret_cast<T*>(o.blk[b]) + m * o.ld + n;
}

// Load one 128 x 32 operand tile (rows = M or N) into shared memory.
template <bool KM>
__device__ __forceinline__ void load_tile(bf16* s, const GemmOperand& op, int64_t mn0, int64_t mn_lim, int64_t k0,
                                          int64_t k_lim, int tid) {
#pragma unroll
  for (int it = 0; it < 2; ++it) {
    const int c = tid + it * THREADS;  // 512 chunks of 8 elements
    if (KM) {
      const int r = c >> 2, kc = (c & 3) * 8;
      const int64_t mn = mn0 + r, k = k0 + kc;
      const bool ok = mn < mn_lim && k < k_lim;
      const bf16* g = ok ? op_addr(op, mn, k) : reinterpret_cast<const bf16*>(op.blk[0]);
      cp_async16(s + r * KM_LD + kc, g, ok ? 16 : 0);
    } else {
      const int kr = c >> 4, mc = (c & 15) * 8;
      const int64_t mn = mn0 + mc, k = k0 + kr;
      const bool ok = mn < mn_lim && k < k_lim;
      const bf16* g = ok ? op_addr(op, mn, k) : reinterpret_cast<const bf16*>(op.blk[0]);
      cp_async16(s + kr * MN_LD + mc, g, ok ? 16 : 0);
    }
  }
}

template <bool AKM, bool BKM>
__global__ void __launch_bounds__(THREADS) k_gemm(GemmArgs args, int64_t k_per_split, float* split_out) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  bf16* sA = reinterpret_cast<bf16*>(smem_raw);
  bf16* sB = sA + STAGES * TILE_ELEMS;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wm = warp >> 2, wn = warp & 3;  // 2 x 4 warps
  const int64_t m0 = (int64_t)blockIdx.x * BM, n0 = (int64_t)blockIdx.y * BN;
  const int64_t kb = (int64_t)blockIdx.z * k_per_split;
  const int64_t ke = min(args.K, kb + k_per_split);
  const int nk = (int)ceil_div(max(ke - kb, (int64_t)0), BK);

  float acc[4][4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][j][e] = 0.f;

#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < nk) {
      load_tile<AKM>(sA + s * TILE_ELEMS, args.a, m0, args.M, kb + s * BK, ke, tid);
      load_tile<BKM>(sB + s * TILE_ELEMS, args.b, n0, args.N, kb + s * BK, ke, tid);
    }
    cp_async_commit();
  }

  for (int kt = 0; kt < nk; ++kt) {
    cp_async_wait<STAGES - 2>();
    __syncthreads();
    {  // prefetch tile kt + STAGES - 1
      const int nt = kt + STAGES - 1;
      if (nt < nk) {
        const int st = nt % STAGES;
        load_tile<AKM>(sA + st * TILE_ELEMS, args.a, m0, args.M, kb + (int64_t)nt * BK, ke, tid);
        load_tile<BKM>(sB + st * TILE_ELEMS, args.b, n0, args.N, kb + (int64_t)nt * BK, ke, tid);
      }
      cp_async_commit();
    }
    const bf16* a = sA + (kt % STAGES) * TILE_ELEMS;
    const bf16* b = sB + (kt % STAGES) * TILE_ELEMS;
#pragma unroll
    for (int kk = 0; kk < BK / 16; ++kk) {
      uint32_t af[4][4], bfr[2][4];
#pragma unroll
      for (int mi = 0; mi < 4; ++mi) {
        const int mrow = wm * 64 + mi * 16;
        if (AKM) {
          ldmatrix_x4(af[mi], a + (mrow + (lane & 15)) * KM_LD + kk * 16 + (lane >> 4) * 8);
        } else {
          const int q = lane >> 3, r = lane & 7;
          ldmatrix_x4_trans(af[mi], a + (kk * 16 + (q >> 1) * 8 + r) * MN_LD + mrow + (q & 1) * 8);
        }
      }
#pragma unroll
      for (int nj = 0; nj < 2; ++nj) {
        const int ncol = wn * 32 + nj * 16;
        const int q = lane >> 3, r = lane & 7;
        if (BKM) {
          ldmatrix_x4(bfr[nj], b + (ncol + (q >> 1) * 8 + r) * KM_LD + kk * 16 + (q & 1) * 8);
        } else {
          ldmatrix_x4_trans(bfr[nj], b + (kk * 16 + (q & 1) * 8 + r) * MN_LD + ncol + (q >> 1) * 8);
        }
      }
#pragma unroll
      for (int mi = 0; mi < 4; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) mma_bf16_16816(acc[mi][ni], af[mi], &bfr[ni >> 1][(ni & 1) * 2]);
    }
  }
  cp_async_wait<0>();

  // epilogue
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int mi = 0; mi < 4; ++mi)
#pragma unroll
    for (int ni = 0; ni < 4; ++ni)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int64_t m = m0 + wm * 64 + mi * 16 + g + hh * 8;
        const int64_t n = n0 + wn * 32 + ni * 8 + 2 * t;
        if (m >= args.M || n >= args.N) continue;
        const float v0 = acc[mi][ni][hh * 2], v1 = acc[mi][ni][hh * 2 + 1];
        if (split_out) {
          float2* p = reinterpret_cast<float2*>(split_out + ((int64_t)blockIdx.z * args.M + m) * args.N + n);
          *p = make_float2(v0, v1);
          continue;
        }
        switch (args.epi) {
          case EPI_STORE_BF16:
            *reinterpret_cast<uint32_t*>(out_addr<bf16>(args.c, m, n)) = pack_bf16(v0, v1);
            break;
          case EPI_STORE_F32:
            *reinterpret_cast<float2*>(out_addr<float>(args.c, m, n)) = make_float2(v0, v1);
            break;
          case EPI_ACC_F32: {
            float2* p = reinterpret_cast<float2*>(out_addr<float>(args.c, m, n));
            float2 o = *p;
            *p = make_float2(o.x + v0, o.y + v1);
            break;
          }
          case EPI_ACC_F32_TO_BF16: {
            const float2 o = *reinterpret_cast<const float2*>(args.c.aux + m * args.c.aux_ld + n);
            *reinterpret_cast<uint32_t*>(out_addr<bf16>(args.c, m, n)) = pack_bf16(o.x + v0, o.y + v1);
            break;
          }
          case EPI_ACC_BF16: {
            uint32_t* p = reinterpret_cast<uint32_t*>(out_addr<bf16>(args.c, m, n));
            __nv_bfloat162 o = *reinterpret_cast<__nv_bfloat162*>(p);
            *p = pack_bf16(__low2float(o) + v0, __high2float(o) + v1);
            break;
          }
        }
      }
}

// Fixed-order reduction of split-K partials into the (blocked) f32 output.
__global__ void k_split_reduce(const float* __restrict__ part, int splits, int64_t M, int64_t N, GemmOutput out) {
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
    *reinterpret_cast<float4*>(out_addr<float>(out, m, n)) = s;
  }
}

}  // namespace

size_t gemm_split_scratch_bytes(int64_t M, int64_t N, int split_k) {
  return split_k > 1 ? (size_t)split_k * M * N * sizeof(float) : 0;
}

int gemm_pick_split(int64_t M, int64_t N, int64_t K, int num_sms) {
  const int64_t tiles = ceil_div(M, BM) * ceil_div(N, BN);
  int split = 1;
  while (tiles * split < 2 * num_sms && K / (split * 2) >= 2048 && split < 32) split *= 2;
  return split;
}

cudaError_t launch_gemm(const GemmArgs& args, int split_k, float* split_scratch, cudaStream_t st) {
  if (args.M <= 0 || args.N <= 0) return cudaSuccess;
  const size_t smem = 2 * STAGES * TILE_ELEMS * sizeof(bf16);
  int64_t kps = args.K;
  if (split_k > 1) kps = ceil_div(ceil_div(args.K, split_k), BK) * BK;
  dim3 grid((unsigned)ceil_div(args.M, BM), (unsigned)ceil_div(args.N, BN), (unsigned)(split_k > 1 ? split_k : 1));
  float* so = split_k > 1 ? split_scratch : nullptr;
  const int key = (args.a.k_major ? 2 : 0) | (args.b.k_major ? 1 : 0);
  cudaError_t e = cudaSuccess;
#define UPIPE_GEMM_CASE(AK, BK_)                                                                \
  {                                                                                            \
    auto kfn = k_gemm<AK, BK_>;                                                                \
    e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);     \
    if (e != cudaSuccess) return e;                                                            \
    kfn<<<grid, THREADS, smem, st>>>(args, kps, so);                                           \
  }
  switch (key) {
    case 3: UPIPE_GEMM_CASE(true, true) break;
    case 2: UPIPE_GEMM_CASE(true, false) break;
    case 1: UPIPE_GEMM_CASE(false, true) break;
    default: UPIPE_GEMM_CASE(false, false) break;
  }
#undef UPIPE_GEMM_CASE
  e = cudaGetLastError();
  if (e != cudaSuccess || split_k <= 1) return e;
  const int64_t total4 = args.M * args.N / 4;
  const unsigned blocks = (unsigned)std::min<int64_t>(ceil_div(total4, 256), 152 * 8);
  k_split_reduce<<<blocks, 256, 0, st>>>(split_scratch, split_k, args.M, args.N, args.c);
  return cudaGetLastError();
}

}  // namespace upipe
