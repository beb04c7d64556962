// Bandwidth-bound helpers of the chunk loop: fp32 -> bf16 conversion with a scale, zeroing.
// Grid-stride loops over 16-byte vectors, grid sized to a few waves of the 152 SMs.
#include "common.cuh"
#include "internal.h"

namespace upipe {

namespace {

__global__ void k_f32_to_bf16(const float* __restrict__ in, bf16* __restrict__ out, int64_t n, float mul) {
  const int64_t n8 = n / 8;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride) {
    const float4 a = reinterpret_cast<const float4*>(in)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(in)[2 * i + 1];
    uint4 o;
    o.x = pack_bf16(a.x * mul, a.y * mul);
    o.y = pack_bf16(a.z * mul, a.w * mul);
    o.z = pack_bf16(b.x * mul, b.y * mul);
    o.w = pack_bf16(b.z * mul, b.w * mul);
    reinterpret_cast<uint4*>(out)[i] = o;
  }
  for (int64_t i = n8 * 8 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    out[i] = __float2bfloat16_rn(in[i] * mul);
}

__global__ void k_zero(uint4* __restrict__ p, int64_t n16) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride) p[i] = make_uint4(0, 0, 0, 0);
}

unsigned grid_for(int64_t work) { return (unsigned)std::max<int64_t>(1, std::min<int64_t>(ceil_div(work, 256), 152 * 16)); }

}  // namespace

cudaError_t launch_f32_to_bf16(const float* in, bf16* out, int64_t n, float mul, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  k_f32_to_bf16<<<grid_for(n / 8 + 1), 256, 0, st>>>(in, out, n, mul);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_zero(void* p, int64_t bytes, cudaStream_t st) {
  if (bytes <= 0) return cudaSuccess;
  k_zero<<<grid_for(bytes / 16), 256, 0, st>>>(reinterpret_cast<uint4*>(p), bytes / 16);
  note_launch();
  return cudaGetLastError();
}

}  // namespace upipe
