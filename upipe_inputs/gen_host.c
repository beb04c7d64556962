/* Host fill of seeded bf16 tensors (OpenMP); the generator itself is in gen.h. */
#include <stdint.h>
#include "gen.h"

/* out[i] = normal_bf16(seed, tid, first + i) for i in [0, n) */
void ug_fill_normal_bf16_host(uint16_t* out, int64_t n, uint64_t seed, uint64_t tid, int64_t first,
                              double mean, double stddev) {
  const uint64_t key = ug_key(seed, tid);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = ug_normal_bf16(key, (uint64_t)(first + i), mean, stddev);
}

/* rows of a row-major [*, cols] tensor: out[r, :] = element (rows[r] * cols + c) */
void ug_fill_rows_normal_bf16_host(uint16_t* out, const int64_t* rows, int64_t n_rows, int64_t cols,
                                   uint64_t seed, uint64_t tid, double mean, double stddev) {
  const uint64_t key = ug_key(seed, tid);
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < n_rows; ++r)
    for (int64_t c = 0; c < cols; ++c)
      out[r * cols + c] = ug_normal_bf16(key, (uint64_t)(rows[r] * cols + c), mean, stddev);
}

/* uniform (0,1) draws, used for the segment-length recipe */
void ug_uniform_host(double* out, int64_t n, uint64_t seed, uint64_t tid) {
  const uint64_t key = ug_key(seed, tid);
  for (int64_t i = 0; i < n; ++i) out[i] = ug_uniform(ug_draw(key, (uint64_t)i));
}

/* exposed for the generator's own tests */
double ug_log_host(double x) { return ug_log(x); }
uint16_t ug_bf16_rne_host(double x) { return ug_bf16_rne(x); }
uint64_t ug_mix64_host(uint64_t z) { return ug_mix64(z); }
