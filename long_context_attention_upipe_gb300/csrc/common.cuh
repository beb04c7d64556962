// Device helpers shared by the kernels of the head-chunked attention library (sm_103a).
#pragma once

#include <algorithm>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "upipe_attn.h"

namespace upipe {

typedef __nv_bfloat16 bf16;

constexpr int kTile = 128;  // tile edge of the skip table and of the attention kernels

// Workspace / table header: int64 n_partial, int64 n_full, int32 error, int32 n_tiles, int64 reserved
struct TableHeader {
  long long n_partial;
  long long n_full;
  int error;
  int n_tiles;
  long long reserved;
};
static_assert(sizeof(TableHeader) == 32, "table header is 32 bytes");

inline __host__ __device__ int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Segment bounds of position r for non-decreasing segment ids (NULL: one segment [0, S)).
// With contiguous segments, query r sees exactly the keys [seg_first(r), causal ? r : seg_last(r)].
__device__ __forceinline__ int64_t seg_first(const int32_t* seg, int64_t r) {
  if (!seg) return 0;
  const int32_t v = seg[r];
  int64_t lo = 0, hi = r;  // first p in [0, r] with seg[p] >= v
  while (lo < hi) {
    const int64_t mid = (lo + hi) >> 1;
    if (seg[mid] >= v) hi = mid; else lo = mid + 1;
  }
  return lo;
}
__device__ __forceinline__ int64_t seg_last(const int32_t* seg, int64_t S, int64_t r) {
  if (!seg) return S - 1;
  const int32_t v = seg[r];
  int64_t lo = r, hi = S - 1;  // last p in [r, S) with seg[p] <= v
  while (lo < hi) {
    const int64_t mid = (lo + hi + 1) >> 1;
    if (seg[mid] <= v) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Programmatic dependent launch between consecutive ring steps: a CTA lets the next step's grid
// start on the SMs this grid leaves free (trigger), and a step waits for the previous step to
// complete, with its writes visible, before it touches the accumulators they share (wait).  Both
// are no-ops for a grid launched without programmatic stream serialisation.
__device__ __forceinline__ void grid_dep_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// First error wins; the word lives in the table header.
__device__ __forceinline__ void set_error(int* word, int code) { atomicCAS(word, 0, code); }

// ------------------------------------------------------------------------------------------------
// bf16 packing
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// max(a, b, c) in one instruction (three-input max of sm_100-family GPUs)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace upipe
