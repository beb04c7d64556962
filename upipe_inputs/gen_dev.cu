// Device fill of seeded bf16 tensors: same generator (gen.h) as the host fill, same bits.
#include <cuda_runtime.h>
#include <stdint.h>
#include "gen.h"

static __global__ void ug_fill_kernel(uint16_t* __restrict__ out, int64_t n, uint64_t key, int64_t first,
                                      double mean, double stddev) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    out[i] = ug_normal_bf16(key, (uint64_t)(first + i), mean, stddev);
}

extern "C" int ug_fill_normal_bf16_device(uint16_t* out, int64_t n, uint64_t seed, uint64_t tid, int64_t first,
                                          double mean, double stddev, void* stream) {
  if (n <= 0) return 0;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (n + 255) / 256;
  int64_t cap = (int64_t)sms * 16;
  if (blocks > cap) blocks = cap;
  ug_fill_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(out, n, ug_key(seed, tid), first, mean, stddev);
  return (int)cudaGetLastError();
}
