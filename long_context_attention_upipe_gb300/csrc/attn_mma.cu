// Flash-style attention core on the warp-level tensor core path (mma.sync m16n8k16).
//
// Each head is computed over the whole sequence with online softmax (podcast summary "Road to
// 5 Million Tokens", chapter on DeepSpeed Ulysses: each GPU computes its heads over the full
// sequence, so flash attention applies).  Tiles come from the skip table: key tiles outside a
// query tile's range are never touched, full tiles run without a mask, partial ones (and the
// ragged last tile) apply  seg[q] == seg[k] && (!causal || k <= q) && k < S  per element.
//
//   bwd dq     : dQ = scale * dS K, dS = P * (dP - D), dP = dO V^T       (grid: q tile x head)
//   bwd dkdv   : dV = sum_h P^T dO, dK = scale * sum_h dS^T Q  over the query heads of a
//                KV head (GQA reduction in registers)                    (grid: kv tile x kv head)
#include "common.cuh"
#include "internal.h"

namespace upipe {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kThreads = 256;  // 8 warps, 16 rows each
constexpr int kSub = 64;       // key rows per step in the query-major kernels
constexpr int kQSub = 32;      // query rows per step in the key-major kernel

template <int DH>
struct Smem {
  static constexpr int LD = DH + 8;  // padded row (conflict-free ldmatrix)
};

// Copy `rows` rows of a head-major [S, DH] matrix starting at row r0 into shared memory
// (rows >= S are zero-filled).
template <int DH>
__device__ __forceinline__ void load_rows(bf16* s, const bf16* g, int64_t r0, int rows, int64_t S, int tid) {
  constexpr int CPR = DH / 8;  // 16-byte chunks per row
  for (int c = tid; c < rows * CPR; c += kThreads) {
    const int r = c / CPR, cc = (c % CPR) * 8;
    const int64_t gr = r0 + r;
    const bool ok = gr < S;
    cp_async16(s + r * Smem<DH>::LD + cc, ok ? g + gr * DH + cc : g, ok ? 16 : 0);
  }
}

__device__ __forceinline__ bool visible(const int32_t* seg, int32_t sq, int32_t sk, int64_t q, int64_t k, int64_t S,
                                        int causal) {
  return k < S && q < S && (!seg || sq == sk) && (!causal || k <= q);
}

// S (16 x 64 per warp) = Q_w K_sub^T : A rows from sQ (warp rows), B rows from sK.
template <int DH>
__device__ __forceinline__ void qk_tile(float (&s)[8][4], const bf16* sQw, const bf16* sK, int lane) {
  constexpr int LD = Smem<DH>::LD;
#pragma unroll
  for (int nb = 0; nb < 8; ++nb)
#pragma unroll
    for (int e = 0; e < 4; ++e) s[nb][e] = 0.f;
#pragma unroll
  for (int kk = 0; kk < DH / 16; ++kk) {
    uint32_t a[4];
    ldmatrix_x4(a, sQw + (lane & 15) * LD + kk * 16 + (lane >> 4) * 8);
#pragma unroll
    for (int nj = 0; nj < 4; ++nj) {
      uint32_t b[4];
      const int q = lane >> 3, r = lane & 7;
      ldmatrix_x4(b, sK + (nj * 16 + (q >> 1) * 8 + r) * LD + kk * 16 + (q & 1) * 8);
      mma_bf16_16816(s[2 * nj], a, b);
      mma_bf16_16816(s[2 * nj + 1], a, b + 2);
    }
  }
}

// acc (16 x DH per warp) += P (16 x 64, registers) * V_sub (64 x DH, shared, row-major)
template <int DH>
__device__ __forceinline__ void pv_tile(float (&acc)[DH / 8][4], const float (&p)[8][4], const bf16* sV, int lane) {
  constexpr int LD = Smem<DH>::LD;
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    uint32_t a[4];
    a[0] = pack_bf16(p[2 * kk][0], p[2 * kk][1]);
    a[1] = pack_bf16(p[2 * kk][2], p[2 * kk][3]);
    a[2] = pack_bf16(p[2 * kk + 1][0], p[2 * kk + 1][1]);
    a[3] = pack_bf16(p[2 * kk + 1][2], p[2 * kk + 1][3]);
#pragma unroll
    for (int nj = 0; nj < DH / 16; ++nj) {
      uint32_t b[4];
      const int q = lane >> 3, r = lane & 7;
      ldmatrix_x4_trans(b, sV + (kk * 16 + (q & 1) * 8 + r) * LD + nj * 16 + (q >> 1) * 8);
      mma_bf16_16816(acc[2 * nj], a, b);
      mma_bf16_16816(acc[2 * nj + 1], a, b + 2);
    }
  }
}

// ---------------------------------------------------------------------------------------------
// backward, dQ (query-major)
// ---------------------------------------------------------------------------------------------
template <int DH>
__global__ void __launch_bounds__(kThreads, 1) k_attn_bwd_dq(AttnBwdArgs b) {
  constexpr int LD = Smem<DH>::LD;
  const AttnArgs& a = b.f;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  bf16* sQ = reinterpret_cast<bf16*>(smem_raw);
  bf16* sdO = sQ + kTile * LD;
  bf16* sK = sdO + kTile * LD;      // [2][kSub][LD]
  bf16* sV = sK + 2 * kSub * LD;    // [2][kSub][LD]
  int32_t* sSeg = reinterpret_cast<int32_t*>(sV + 2 * kSub * LD);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t S = a.S;
  const int64_t nt = ceil_div(S, kTile);
  const int64_t qt = nt - 1 - blockIdx.x;
  const int h = blockIdx.y;
  const int kvh = h / a.g;
  const bf16* Qh = a.q + (int64_t)h * S * DH;
  const bf16* dOh = a.dO + (int64_t)h * S * DH;
  const bf16* Kh = a.k + (int64_t)kvh * S * DH;
  const bf16* Vh = a.v + (int64_t)kvh * S * DH;
  const int64_t row0 = qt * kTile;
  const int4 tr = a.q_rows[qt];
  const bool ragged = (S % kTile) != 0;

  load_rows<DH>(sQ, Qh, row0, kTile, S, tid);
  load_rows<DH>(sdO, dOh, row0, kTile, S, tid);
  cp_async_commit();
  auto sub_row = [&](int s) { return (int64_t)tr.x * kTile + (int64_t)s * kSub; };
  int n_sub = 2 * (tr.w - tr.x);
  while (n_sub > 0 && sub_row(n_sub - 1) >= S) --n_sub;
  auto prefetch = [&](int s, int buf) {
    const int64_t kr0 = sub_row(s);
    load_rows<DH>(sK + buf * kSub * LD, Kh, kr0, kSub, S, tid);
    load_rows<DH>(sV + buf * kSub * LD, Vh, kr0, kSub, S, tid);
    if (a.seg && tid < kSub) sSeg[buf * kSub + tid] = (kr0 + tid < S) ? a.seg[kr0 + tid] : 0;
  };
  if (n_sub > 0) prefetch(0, 0);
  cp_async_commit();

  const int g = lane >> 2, t = lane & 3;
  const int64_t rA = row0 + warp * 16 + g, rB = rA + 8;
  const int32_t segA = (a.seg && rA < S) ? a.seg[rA] : 0;
  const int32_t segB = (a.seg && rB < S) ? a.seg[rB] : 0;
  const float c = a.scale * kLog2e;
  const float lse2[2] = {rA < S ? a.lse[(int64_t)h * S + rA] * kLog2e : 0.f,
                         rB < S ? a.lse[(int64_t)h * S + rB] * kLog2e : 0.f};
  const float Dr[2] = {rA < S ? a.D[(int64_t)h * S + rA] : 0.f, rB < S ? a.D[(int64_t)h * S + rB] : 0.f};

  float acc[DH / 8][4];
#pragma unroll
  for (int i = 0; i < DH / 8; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[i][e] = 0.f;

  for (int s = 0; s < n_sub; ++s) {
    const int buf = s & 1;
    if (s + 1 < n_sub) prefetch(s + 1, buf ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const bf16* k_s = sK + buf * kSub * LD;
    const bf16* v_s = sV + buf * kSub * LD;
    float p[8][4], dp[8][4];
    qk_tile<DH>(p, sQ + warp * 16 * LD, k_s, lane);
    qk_tile<DH>(dp, sdO + warp * 16 * LD, v_s, lane);
    const int64_t kr0 = sub_row(s);
    const int64_t jt = kr0 / kTile;
    const bool partial = jt < tr.y || jt >= tr.z || (ragged && jt == nt - 1);
#pragma unroll
    for (int nb = 0; nb < 8; ++nb)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = e >> 1;
        float pv = fast_exp2(p[nb][e] * c - lse2[r]);
        if (partial) {
          const int col = nb * 8 + 2 * t + (e & 1);
          const int32_t sk = a.seg ? sSeg[buf * kSub + col] : 0;
          if (!visible(a.seg, r ? segB : segA, sk, r ? rB : rA, kr0 + col, S, a.causal)) pv = 0.f;
        }
        p[nb][e] = pv * (dp[nb][e] - Dr[r]);  // dS
      }
    // dQ += dS K_sub  (K rows are the contraction index: same access as V in the forward)
    pv_tile<DH>(acc, p, k_s, lane);
    __syncthreads();
  }
  cp_async_wait<0>();
  bf16* dQh = b.dq + (int64_t)h * S * DH;
#pragma unroll
  for (int i = 0; i < DH / 8; ++i) {
    const int col = i * 8 + 2 * t;
    if (rA < S) *reinterpret_cast<uint32_t*>(dQh + rA * DH + col) = pack_bf16(acc[i][0] * a.scale, acc[i][1] * a.scale);
    if (rB < S) *reinterpret_cast<uint32_t*>(dQh + rB * DH + col) = pack_bf16(acc[i][2] * a.scale, acc[i][3] * a.scale);
  }
}

// ---------------------------------------------------------------------------------------------
// backward, dK and dV (key-major), GQA heads reduced in registers
// ---------------------------------------------------------------------------------------------
template <int DH>
__global__ void __launch_bounds__(kThreads, 1) k_attn_bwd_dkdv(AttnBwdArgs b) {
  constexpr int LD = Smem<DH>::LD;
  const AttnArgs& a = b.f;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  bf16* sK = reinterpret_cast<bf16*>(smem_raw);
  bf16* sV = sK + kTile * LD;
  bf16* sQ = sV + kTile * LD;        // [2][kQSub][LD]
  bf16* sdO = sQ + 2 * kQSub * LD;   // [2][kQSub][LD]
  float* sL = reinterpret_cast<float*>(sdO + 2 * kQSub * LD);  // [2][kQSub] lse * log2e
  float* sD = sL + 2 * kQSub;                                  // [2][kQSub]
  int32_t* sSeg = reinterpret_cast<int32_t*>(sD + 2 * kQSub);  // [2][kQSub]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t S = a.S;
  const int64_t nt = ceil_div(S, kTile);
  const int64_t jt = blockIdx.x;  // kv tile (small j has the most query tiles under causality)
  const int kvh = blockIdx.y;
  const int64_t kv0 = jt * kTile;
  const int4 tr = a.kv_rows[jt];  // {q_begin, q_full_begin, q_full_end, q_end}
  const bool ragged = (S % kTile) != 0;

  load_rows<DH>(sK, a.k + (int64_t)kvh * S * DH, kv0, kTile, S, tid);
  load_rows<DH>(sV, a.v + (int64_t)kvh * S * DH, kv0, kTile, S, tid);
  cp_async_commit();

  // work items: (query head of this KV head within the launch) x (query sub-tile of 32 rows)
  const int h_first = kvh * a.g;
  const int h_last = min(a.nh, h_first + a.g);  // exclusive
  const int n_heads = max(0, h_last - h_first);
  auto qsub_row = [&](int s) { return (int64_t)tr.x * kTile + (int64_t)s * kQSub; };
  int n_qs = (tr.w - tr.x) * (kTile / kQSub);
  while (n_qs > 0 && qsub_row(n_qs - 1) >= S) --n_qs;
  const int n_items = n_heads * n_qs;

  auto prefetch = [&](int it, int buf) {
    const int h = h_first + it / n_qs;
    const int64_t q0 = qsub_row(it % n_qs);
    load_rows<DH>(sQ + buf * kQSub * LD, a.q + (int64_t)h * S * DH, q0, kQSub, S, tid);
    load_rows<DH>(sdO + buf * kQSub * LD, a.dO + (int64_t)h * S * DH, q0, kQSub, S, tid);
    if (tid < kQSub) {
      const int64_t q = q0 + tid;
      const bool ok = q < S;
      sL[buf * kQSub + tid] = ok ? a.lse[(int64_t)h * S + q] * kLog2e : 0.f;
      sD[buf * kQSub + tid] = ok ? a.D[(int64_t)h * S + q] : 0.f;
      sSeg[buf * kQSub + tid] = (ok && a.seg) ? a.seg[q] : 0;
    }
  };
  if (n_items > 0) prefetch(0, 0);
  cp_async_commit();

  const int g = lane >> 2, t = lane & 3;
  const int64_t kA = kv0 + warp * 16 + g, kB = kA + 8;  // this thread's two key rows
  const int32_t segA = (a.seg && kA < S) ? a.seg[kA] : 0;
  const int32_t segB = (a.seg && kB < S) ? a.seg[kB] : 0;
  const float c = a.scale * kLog2e;

  float dk[DH / 8][4], dv[DH / 8][4];
#pragma unroll
  for (int i = 0; i < DH / 8; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) dk[i][e] = dv[i][e] = 0.f;

  for (int it = 0; it < n_items; ++it) {
    const int buf = it & 1;
    if (it + 1 < n_items) prefetch(it + 1, buf ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const bf16* q_s = sQ + buf * kQSub * LD;
    const bf16* do_s = sdO + buf * kQSub * LD;
    const int64_t q0 = qsub_row(it % n_qs);
    const int64_t qt = q0 / kTile;
    const bool partial = qt < tr.y || qt >= tr.z || (ragged && (qt == nt - 1 || jt == nt - 1));

    // S^T (16 keys x 32 queries) = K_w Q_sub^T ; dP^T = V_w dO_sub^T
    float st[4][4], dpt[4][4];
#pragma unroll
    for (int nb = 0; nb < 4; ++nb)
#pragma unroll
      for (int e = 0; e < 4; ++e) st[nb][e] = dpt[nb][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < DH / 16; ++kk) {
      uint32_t ak[4], av[4];
      ldmatrix_x4(ak, sK + (warp * 16 + (lane & 15)) * LD + kk * 16 + (lane >> 4) * 8);
      ldmatrix_x4(av, sV + (warp * 16 + (lane & 15)) * LD + kk * 16 + (lane >> 4) * 8);
#pragma unroll
      for (int nj = 0; nj < 2; ++nj) {
        uint32_t bq[4], bd[4];
        const int q = lane >> 3, r = lane & 7;
        ldmatrix_x4(bq, q_s + (nj * 16 + (q >> 1) * 8 + r) * LD + kk * 16 + (q & 1) * 8);
        ldmatrix_x4(bd, do_s + (nj * 16 + (q >> 1) * 8 + r) * LD + kk * 16 + (q & 1) * 8);
        mma_bf16_16816(st[2 * nj], ak, bq);
        mma_bf16_16816(st[2 * nj + 1], ak, bq + 2);
        mma_bf16_16816(dpt[2 * nj], av, bd);
        mma_bf16_16816(dpt[2 * nj + 1], av, bd + 2);
      }
    }
    // P^T and dS^T
#pragma unroll
    for (int nb = 0; nb < 4; ++nb)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int col = nb * 8 + 2 * t + (e & 1);  // query index within the sub-tile
        const int r = e >> 1;                      // key row A or B
        float pv = fast_exp2(st[nb][e] * c - sL[buf * kQSub + col]);
        if (partial) {
          const int32_t sq = a.seg ? sSeg[buf * kQSub + col] : 0;
          if (!visible(a.seg, sq, r ? segB : segA, q0 + col, r ? kB : kA, S, a.causal)) pv = 0.f;
        }
        st[nb][e] = pv;
        dpt[nb][e] = pv * (dpt[nb][e] - sD[buf * kQSub + col]);
      }
    // dV += P^T dO_sub ; dK += dS^T Q_sub  (contraction over the 32 queries)
#pragma unroll
    for (int kk = 0; kk < kQSub / 16; ++kk) {
      uint32_t ap[4], as[4];
      ap[0] = pack_bf16(st[2 * kk][0], st[2 * kk][1]);
      ap[1] = pack_bf16(st[2 * kk][2], st[2 * kk][3]);
      ap[2] = pack_bf16(st[2 * kk + 1][0], st[2 * kk + 1][1]);
      ap[3] = pack_bf16(st[2 * kk + 1][2], st[2 * kk + 1][3]);
      as[0] = pack_bf16(dpt[2 * kk][0], dpt[2 * kk][1]);
      as[1] = pack_bf16(dpt[2 * kk][2], dpt[2 * kk][3]);
      as[2] = pack_bf16(dpt[2 * kk + 1][0], dpt[2 * kk + 1][1]);
      as[3] = pack_bf16(dpt[2 * kk + 1][2], dpt[2 * kk + 1][3]);
#pragma unroll
      for (int nj = 0; nj < DH / 16; ++nj) {
        uint32_t bo[4], bq[4];
        const int q = lane >> 3, r = lane & 7;
        ldmatrix_x4_trans(bo, do_s + (kk * 16 + (q & 1) * 8 + r) * LD + nj * 16 + (q >> 1) * 8);
        ldmatrix_x4_trans(bq, q_s + (kk * 16 + (q & 1) * 8 + r) * LD + nj * 16 + (q >> 1) * 8);
        mma_bf16_16816(dv[2 * nj], ap, bo);
        mma_bf16_16816(dv[2 * nj + 1], ap, bo + 2);
        mma_bf16_16816(dk[2 * nj], as, bq);
        mma_bf16_16816(dk[2 * nj + 1], as, bq + 2);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

#pragma unroll
  for (int i = 0; i < DH / 8; ++i) {
    const int col = i * 8 + 2 * t;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int64_t row = r ? kB : kA;
      if (row >= S) continue;
      const float k0 = dk[i][2 * r] * a.scale, k1 = dk[i][2 * r + 1] * a.scale;
      const float v0 = dv[i][2 * r], v1 = dv[i][2 * r + 1];
      const int64_t off = ((int64_t)kvh * S + row) * DH + col;
      if (b.acc_kv) {
        float2* pk = reinterpret_cast<float2*>(b.dk_acc + off);
        float2* pv = reinterpret_cast<float2*>(b.dv_acc + off);
        float2 ok = *pk, ov = *pv;
        *pk = make_float2(ok.x + k0, ok.y + k1);
        *pv = make_float2(ov.x + v0, ov.y + v1);
      } else {
        *reinterpret_cast<uint32_t*>(b.dk + off) = pack_bf16(k0, k1);
        *reinterpret_cast<uint32_t*>(b.dv + off) = pack_bf16(v0, v1);
      }
    }
  }
}

template <int DH>
size_t dq_smem() {
  return (size_t)(2 * kTile + 4 * kSub) * Smem<DH>::LD * sizeof(bf16) + 2 * kSub * sizeof(int32_t);
}
template <int DH>
size_t dkdv_smem() {
  return (size_t)(2 * kTile + 4 * kQSub) * Smem<DH>::LD * sizeof(bf16) + 6 * kQSub * sizeof(float);
}

template <int DH>
cudaError_t run_bwd_dq(const AttnBwdArgs& b, cudaStream_t st) {
  const size_t smem = dq_smem<DH>();
  cudaError_t e = cudaFuncSetAttribute(k_attn_bwd_dq<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)ceil_div(b.f.S, kTile), (unsigned)b.f.nh);
  k_attn_bwd_dq<DH><<<grid, kThreads, smem, st>>>(b);
  return cudaGetLastError();
}

template <int DH>
cudaError_t run_bwd_dkdv(const AttnBwdArgs& b, cudaStream_t st) {
  const size_t smem = dkdv_smem<DH>();
  cudaError_t e = cudaFuncSetAttribute(k_attn_bwd_dkdv<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)ceil_div(b.f.S, kTile), (unsigned)b.nkv);
  k_attn_bwd_dkdv<DH><<<grid, kThreads, smem, st>>>(b);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_bwd_dq(const AttnBwdArgs& b, int head_dim, cudaStream_t st) {
  return head_dim == 64 ? run_bwd_dq<64>(b, st) : run_bwd_dq<128>(b, st);
}
cudaError_t launch_attn_bwd_dkdv(const AttnBwdArgs& b, int head_dim, cudaStream_t st) {
  return head_dim == 64 ? run_bwd_dkdv<64>(b, st) : run_bwd_dkdv<128>(b, st);
}

}  // namespace upipe
