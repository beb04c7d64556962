// Element-wise halves of the sequence-tiled SwiGLU feed-forward step (the MLP beside the
// attention layer, computed a tile of rows at a time so that no buffer spans the whole sequence:
// "Road to 5 Million Tokens" podcast summary, chapter on sequence tiling; neuro-slop.ru transcript,
// Полезные советы).  The projections run on the tensor-core GEMM; these kernels sit between them.
//
// H [rows][2F] bf16 holds the gate projection G in columns [0, F) and the up projection U in
// [F, 2F) (the row order of Wgu = [Wg; Wu]).
//   forward : A = silu(G) * U                                       (A bf16 [rows][F])
//   backward: A as above, dG = dA * U * silu'(G), dU = dA * silu(G)  (dH = [dG | dU] bf16)
// with silu(g) = g * s, s = 1 / (1 + e^-g), silu'(g) = s * (1 + g * (1 - s)); fp32 math on the
// bf16 inputs, one bf16 rounding per output.  Each thread takes 8 consecutive columns (16-byte
// loads and stores); grid-stride over rows x F/8, a few waves of the 152 SMs.  HBM-bound:
// 6 bytes per (row, f) forward, 12 backward.
#include "common.cuh"
#include "internal.h"

namespace upipe {

namespace {

struct F8 {
  float v[8];
};

__device__ __forceinline__ F8 load8(const bf16* p) {
  const uint4 q = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
  F8 f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(h[i]);
    f.v[2 * i] = t.x;
    f.v[2 * i + 1] = t.y;
  }
  return f;
}

__device__ __forceinline__ void store8(bf16* p, const F8& f) {
  uint4 q;
  q.x = pack_bf16(f.v[0], f.v[1]);
  q.y = pack_bf16(f.v[2], f.v[3]);
  q.z = pack_bf16(f.v[4], f.v[5]);
  q.w = pack_bf16(f.v[6], f.v[7]);
  *reinterpret_cast<uint4*>(p) = q;
}

__device__ __forceinline__ float sigmoid(float g) { return __fdividef(1.f, 1.f + __expf(-g)); }

__global__ void k_swiglu_fwd(const bf16* __restrict__ H, bf16* __restrict__ A, int64_t rows, int64_t F) {
  const int64_t per_row = F / 8;
  const int64_t n = rows * per_row;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const int64_t r = i / per_row, c = (i - r * per_row) * 8;
    const F8 g = load8(H + r * 2 * F + c), u = load8(H + r * 2 * F + F + c);
    F8 a;
#pragma unroll
    for (int k = 0; k < 8; ++k) a.v[k] = g.v[k] * sigmoid(g.v[k]) * u.v[k];
    store8(A + r * F + c, a);
  }
}

__global__ void k_swiglu_bwd(const bf16* __restrict__ H, const bf16* __restrict__ dA, bf16* __restrict__ A,
                             bf16* __restrict__ dH, int64_t rows, int64_t F) {
  const int64_t per_row = F / 8;
  const int64_t n = rows * per_row;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const int64_t r = i / per_row, c = (i - r * per_row) * 8;
    const F8 g = load8(H + r * 2 * F + c), u = load8(H + r * 2 * F + F + c), da = load8(dA + r * F + c);
    F8 a, dg, du;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float s = sigmoid(g.v[k]);
      const float sl = g.v[k] * s;
      a.v[k] = sl * u.v[k];
      du.v[k] = da.v[k] * sl;
      dg.v[k] = da.v[k] * u.v[k] * (s * (1.f + g.v[k] * (1.f - s)));
    }
    store8(A + r * F + c, a);
    store8(dH + r * 2 * F + c, dg);
    store8(dH + r * 2 * F + F + c, du);
  }
}

unsigned grid_for(int64_t work) { return (unsigned)std::max<int64_t>(1, std::min<int64_t>(ceil_div(work, 256), 152 * 8)); }

}  // namespace

cudaError_t launch_swiglu_fwd(const bf16* H, bf16* A, int64_t rows, int64_t F, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  k_swiglu_fwd<<<grid_for(rows * F / 8), 256, 0, st>>>(H, A, rows, F);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_swiglu_bwd(const bf16* H, const bf16* dA, bf16* A, bf16* dH, int64_t rows, int64_t F,
                              cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  k_swiglu_bwd<<<grid_for(rows * F / 8), 256, 0, st>>>(H, dA, A, dH, rows, F);
  note_launch();
  return cudaGetLastError();
}

}  // namespace upipe
