// Merge of block attention results: the single-GPU share of ring (P2P) context parallelism.
//
// In the ring strategy the key/value blocks travel from device to device and each device attends
// its query block to the block that is visiting (MaxText long-context article, techmoon.xyz,
// table of the four context-parallel strategies, row "P2P (Ring)").  Attention over a union of
// disjoint key sets follows from the per-set results: with L = log sum exp of the scores,
//   L = log(e^{L_a} + e^{L_b}),   O = (e^{L_a} O_a + e^{L_b} O_b) / e^{L},
// so each visiting block's (O_b, L_b), as upipe_attn_core_fwd writes them, is folded into an fp32
// accumulator.  One warp per (head, query row): lanes hold 4 (head_dim 128) or 2 (head_dim 64)
// consecutive elements, so every access is coalesced; the kernel is bound by HBM bandwidth
// (10 bytes per element, 12 with the bf16 output).
#include "common.cuh"
#include "internal.h"

namespace upipe {

namespace {

template <int DH>
__global__ void k_lse_merge(int64_t rows, const bf16* __restrict__ ob, const float* __restrict__ lb,
                            float* __restrict__ oacc, float* __restrict__ lacc, bf16* __restrict__ oout) {
  constexpr int E = DH / 32;  // elements per lane
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
    const float la = lacc[r], lbr = lb[r];
    const float m = fmaxf(la, lbr);
    float wa = 0.f, wb = 0.f, lnew = -INFINITY;
    if (m != -INFINITY) {
      wa = expf(la - m);   // 0 when la = -inf
      wb = expf(lbr - m);
      const float s = wa + wb;
      lnew = m + logf(s);
      wa /= s;
      wb /= s;
    }
    // a side with weight 0 contributes nothing, whatever its O holds (an accumulator that has
    // seen no key yet, or a block row that sees none)
    auto mix = [&](float x, float y) { return (wa != 0.f ? wa * x : 0.f) + (wb != 0.f ? wb * y : 0.f); };
    float* orow = oacc + r * DH + lane * E;
    const bf16* brow = ob + r * DH + lane * E;
    if constexpr (E == 4) {
      const float4 a = *reinterpret_cast<const float4*>(orow);
      const uint2 b2 = *reinterpret_cast<const uint2*>(brow);
      const float2 b01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&b2.x));
      const float2 b23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&b2.y));
      const float4 o = make_float4(mix(a.x, b01.x), mix(a.y, b01.y), mix(a.z, b23.x), mix(a.w, b23.y));
      *reinterpret_cast<float4*>(orow) = o;
      if (oout) *reinterpret_cast<uint2*>(oout + r * DH + lane * E) = make_uint2(pack_bf16(o.x, o.y), pack_bf16(o.z, o.w));
    } else {
      const float2 a = *reinterpret_cast<const float2*>(orow);
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(brow));
      const float2 o = make_float2(mix(a.x, b.x), mix(a.y, b.y));
      *reinterpret_cast<float2*>(orow) = o;
      if (oout) *reinterpret_cast<uint32_t*>(oout + r * DH + lane * E) = pack_bf16(o.x, o.y);
    }
    __syncwarp();  // every lane has read lacc[r]
    if (lane == 0) lacc[r] = lnew;
  }
}

// Backward of the ring: every block (query chunk, key chunk) runs the dQ and dK/dV kernels with the
// softmax of the whole key set, i.e. the query chunk's final log-sum-exp L and D = rowsum(dO * O)
// of its final output.  This fills the kernels' D buffer [2][heads][Sp] (D, then L * log2(e);
// zero rows past the chunk) from O, dO and L.  One warp per (head, row).
template <int DH>
__global__ void k_ring_bwd_prep(int nh, int64_t S, const bf16* __restrict__ o, const bf16* __restrict__ dout,
                                const float* __restrict__ lse, float* __restrict__ D) {
  constexpr int E = DH / 32;
  const int lane = threadIdx.x & 31;
  const int64_t sp = ceil_div(S, kTile) * kTile;
  const int64_t rows = (int64_t)nh * sp;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
    const int64_t h = r / sp, i = r % sp;
    float dsum = 0.f, l2 = 0.f;
    if (i < S) {
      const int64_t row = h * S + i;
      const bf16* orow = o + row * DH + lane * E;
      const bf16* grow = dout + row * DH + lane * E;
#pragma unroll
      for (int e = 0; e < E; e += 2) {
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(orow + e));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(grow + e));
        dsum += a.x * b.x + a.y * b.y;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, off);
      l2 = lse[row] * 1.4426950408889634f;
    }
    if (lane == 0) {
      D[h * sp + i] = dsum;
      D[((int64_t)nh + h) * sp + i] = l2;
    }
  }
}

// acc += src (bf16 -> fp32); out (optional) = bf16(acc).  Blocks' gradient contributions summed in
// fp32 and rounded once.
__global__ void k_accumulate(int64_t n, const bf16* __restrict__ src, float* __restrict__ acc, bf16* __restrict__ out) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n / 4; i += stride) {
    const uint2 s2 = reinterpret_cast<const uint2*>(src)[i];
    const float2 s01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&s2.x));
    const float2 s23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&s2.y));
    float4 a = reinterpret_cast<float4*>(acc)[i];
    a.x += s01.x; a.y += s01.y; a.z += s23.x; a.w += s23.y;
    reinterpret_cast<float4*>(acc)[i] = a;
    if (out) reinterpret_cast<uint2*>(out)[i] = make_uint2(pack_bf16(a.x, a.y), pack_bf16(a.z, a.w));
  }
  for (int64_t i = (n / 4) * 4 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    acc[i] += __bfloat162float(src[i]);
    if (out) out[i] = __float2bfloat16_rn(acc[i]);
  }
}

}  // namespace

cudaError_t launch_ring_bwd_prep(int nh, int64_t S, int head_dim, const bf16* o, const bf16* dout, const float* lse,
                                 float* D, cudaStream_t st) {
  const int64_t rows = (int64_t)nh * ceil_div(S, kTile) * kTile;
  if (rows <= 0) return cudaSuccess;
  const unsigned blocks = (unsigned)std::max<int64_t>(1, std::min<int64_t>(ceil_div(rows, 8), 152 * 16));
  if (head_dim == 128) k_ring_bwd_prep<128><<<blocks, 256, 0, st>>>(nh, S, o, dout, lse, D);
  else k_ring_bwd_prep<64><<<blocks, 256, 0, st>>>(nh, S, o, dout, lse, D);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_accumulate(int64_t n, const bf16* src, float* acc, bf16* out, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const unsigned blocks = (unsigned)std::max<int64_t>(1, std::min<int64_t>(ceil_div(n / 4 + 1, 256), 152 * 16));
  k_accumulate<<<blocks, 256, 0, st>>>(n, src, acc, out);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_lse_merge(int64_t rows, int head_dim, const bf16* ob, const float* lb, float* oacc, float* lacc,
                             bf16* oout, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const unsigned blocks = (unsigned)std::max<int64_t>(1, std::min<int64_t>(ceil_div(rows, 8), 152 * 16));
  if (head_dim == 128) k_lse_merge<128><<<blocks, 256, 0, st>>>(rows, ob, lb, oacc, lacc, oout);
  else k_lse_merge<64><<<blocks, 256, 0, st>>>(rows, ob, lb, oacc, lacc, oout);
  note_launch();
  return cudaGetLastError();
}

}  // namespace upipe
