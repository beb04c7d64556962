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

}  // namespace

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
