// C-ABI entry points and the head-chunk scheduler.
//
// UPipe: the query heads one GPU owns are processed a chunk at a time; every chunk's Q/K/V
// projection, attention and output-projection accumulation run in one workspace that the next
// chunk reuses, and only the partial output sum is carried from chunk to chunk ("Road to 5
// Million Tokens" podcast summary, chapters "主要貢獻 UPipe" and "分批算 heads"; neuro-slop.ru
// transcript, insight 02).  The backward pass recomputes each chunk's activations from X and
// the saved log-sum-exp (activation checkpointing, same summary, chapter "Activation
// checkpointing"), so no per-head activation survives a chunk.
//
// Workspace carve-up (every region 256-byte aligned, offsets from the workspace base):
//   table   skip table (its header holds the device error word)              both passes
//   K, V    bf16 [kvc, S, Dh]: the KV heads of the current group, resident     both
//           while the chunks of that group run
//   Q, O    bf16 [hpc, S, Dh]                                                   both
//   Yacc    f32 [S, d] partial output projection (fwd, several chunks, accum_mode 0)
//   dO      bf16 [hpc, S, Dh]; D f32 [2][hpc][Sp] (D and lse*log2e, Sp = S rounded to 128)
//   dQKV    bf16 [hpc + 2 kvc, S, Dh]: dQ heads, then dK, dV heads (one tensor, so the dX and
//           dWqkv GEMMs read it through one 3-D tensor map)                     bwd
//   dKacc, dVacc f32 [S, Dh] when a chunk holds only part of a KV group (hpc < g)  bwd
//   dXacc   f32 [S, d] partial input gradient (several chunks, accum_mode 0)   bwd
//   split   f32 split-K partials of the weight-gradient GEMMs                  bwd
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace upipe {

// Default limit of a bounded device wait (4 s), and the largest a caller may set (60 s).
constexpr uint64_t tc_wait_default_ns = 4000000000ull;
constexpr uint64_t kMaxWaitLimitNs = 60000000000ull;

// Name of the CUDA error behind the last UPIPE_ERR_CUDA returned on this host thread.
thread_local const char* g_last_cuda_error = "cudaSuccess";

std::atomic<uint64_t> g_launch_count{0};
void note_launch() { g_launch_count.fetch_add(1, std::memory_order_relaxed); }

std::atomic<uint64_t> g_wait_limit_ns{tc_wait_default_ns};
uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

// Longest run of dK / dV accumulations into the same tensor-memory tile before the dK/dV kernel
// adds it into fp32 sums in global memory (upipe_attn_set_dkdv_window; even).
constexpr int kDkvWindowDefault = 4096;
std::atomic<int> g_dkdv_window{kDkvWindowDefault};
int dkdv_window() { return g_dkdv_window.load(std::memory_order_relaxed); }

upipe_status_t cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return UPIPE_OK;
  g_last_cuda_error = cudaGetErrorName(e);
  return UPIPE_ERR_CUDA;
}

// ------------------------------------------------------------------------ per-launch timing
// When enabled (upipe_attn_timing_enable), every kernel launch of the fwd/bwd schedule is
// bracketed by two CUDA events on its stream and logged with its kind and shape; the caller
// collects the durations after the work has run.  Off by default, and then free.
namespace {
struct TimingRec {
  int32_t kind, epi, split_k, chunk;
  int64_t m, n, k;
  cudaEvent_t e0, e1;
};
std::atomic<int> g_timing_on{0};
std::mutex g_timing_mutex;
std::vector<TimingRec> g_timing;

class Timed {
 public:
  Timed(int kind, int epi, int64_t m, int64_t n, int64_t k, int split_k, int chunk, cudaStream_t st) : st_(st) {
    if (!g_timing_on.load(std::memory_order_relaxed)) return;
    rec_ = TimingRec{kind, epi, split_k, chunk, m, n, k, nullptr, nullptr};
    if (cudaEventCreate(&rec_.e0) != cudaSuccess || cudaEventCreate(&rec_.e1) != cudaSuccess ||
        cudaEventRecord(rec_.e0, st_) != cudaSuccess)
      return;
    on_ = true;
  }
  ~Timed() {
    if (!on_) return;
    if (cudaEventRecord(rec_.e1, st_) != cudaSuccess) return;
    std::lock_guard<std::mutex> lock(g_timing_mutex);
    g_timing.push_back(rec_);
  }

 private:
  cudaStream_t st_;
  TimingRec rec_{};
  bool on_ = false;
};
}  // namespace

namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Plan {
  int64_t S;
  int d, Hq, Hkv, Dh, hpc, g, kvc, n_chunks, causal, accum;
  float scale;
  // workspace offsets
  size_t table, k, v, q, o, yacc, dO, D, dq, dk, dv, dkacc, dvacc, dxacc, split, total;
  int split_wo, split_wqkv_q, split_wqkv_full;
  // host-resident X / dY: rows per staged block, the two staging buffers of each, and the K
  // splits of the weight-gradient GEMMs over one block
  int64_t R;
  size_t xs[2], dys[2];
  int split_wo_blk, split_wqkv_q_blk, split_wqkv_full_blk;
  // dK / dV summed in fp32 workspace buffers (dkacc, dvacc: [kvc][S][Dh]) rather than written in
  // bf16 by the dK/dV kernel: always for a KV group split over chunks, and for whole groups once a
  // key tile's work items (the group's query heads x query tiles) exceed the accumulation window
  bool kv_sums;
  int window;
};

constexpr int64_t kDefaultStageRows = 65536;

int num_sms() {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      sms = 152;
  }
  return sms;
}

upipe_status_t check_desc(const upipe_attn_desc_t* d) {
  if (!d) return UPIPE_ERR_INVALID_ARG;
  if (d->seq_len < 1 || d->seq_len > INT32_MAX) return UPIPE_ERR_INVALID_ARG;
  if (d->hidden <= 0 || d->n_q_heads <= 0 || d->n_kv_heads <= 0 || d->heads_per_chunk <= 0) return UPIPE_ERR_INVALID_ARG;
  if (d->n_q_heads % d->n_kv_heads != 0 || d->n_q_heads % d->heads_per_chunk != 0) return UPIPE_ERR_INVALID_ARG;
  const int g = d->n_q_heads / d->n_kv_heads;
  if (d->heads_per_chunk % g != 0 && g % d->heads_per_chunk != 0) return UPIPE_ERR_INVALID_ARG;
  if (d->causal != 0 && d->causal != 1) return UPIPE_ERR_INVALID_ARG;
  if (d->accum_mode != 0 && d->accum_mode != 1) return UPIPE_ERR_INVALID_ARG;
  if (!(d->softmax_scale >= 0.f) || !std::isfinite(d->softmax_scale)) return UPIPE_ERR_INVALID_ARG;
  if (d->head_dim != 64 && d->head_dim != 128) return UPIPE_ERR_UNSUPPORTED;
  if (d->hidden % 64 != 0) return UPIPE_ERR_UNSUPPORTED;
  const int kvc = d->heads_per_chunk >= g ? d->heads_per_chunk / g : 1;
  if (d->heads_per_chunk + 2 * kvc > kMaxBlocks) return UPIPE_ERR_UNSUPPORTED;
  return UPIPE_OK;
}

// stage_rows > 0: X (and dY) stay in host memory and are staged in blocks of that many rows.
Plan make_plan(const upipe_attn_desc_t* desc, int pass, int64_t stage_rows = 0) {
  Plan p;
  p.S = desc->seq_len;
  p.d = desc->hidden;
  p.Hq = desc->n_q_heads;
  p.Hkv = desc->n_kv_heads;
  p.Dh = desc->head_dim;
  p.hpc = desc->heads_per_chunk;
  p.g = p.Hq / p.Hkv;
  p.kvc = p.hpc >= p.g ? p.hpc / p.g : 1;
  p.n_chunks = p.Hq / p.hpc;
  p.causal = desc->causal;
  p.accum = desc->accum_mode;
  p.scale = desc->softmax_scale > 0.f ? desc->softmax_scale : 1.0f / std::sqrt((float)p.Dh);
  const size_t head = (size_t)p.S * p.Dh * sizeof(bf16);
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes); return o; };
  p.table = take(tile_table_bytes(p.S));
  p.k = take(p.kvc * head);
  p.v = take(p.kvc * head);
  p.q = take(p.hpc * head);
  p.o = take(p.hpc * head);
  p.yacc = p.dO = p.D = p.dq = p.dk = p.dv = p.dkacc = p.dvacc = p.dxacc = p.split = 0;
  p.split_wo = p.split_wqkv_q = p.split_wqkv_full = 1;
  p.R = 0;
  p.xs[0] = p.xs[1] = p.dys[0] = p.dys[1] = 0;
  p.split_wo_blk = p.split_wqkv_q_blk = p.split_wqkv_full_blk = 1;
  if (stage_rows > 0) {
    p.R = std::min<int64_t>(stage_rows, p.S);
    const size_t blk = (size_t)p.R * p.d * sizeof(bf16);
    p.xs[0] = take(blk);
    p.xs[1] = take(blk);
    if (pass == 1) {
      p.dys[0] = take(blk);
      p.dys[1] = take(blk);
    }
  }
  const bool multi = p.n_chunks > 1;
  if (pass == 0) {
    if (multi && p.accum == 0) p.yacc = take((size_t)p.S * p.d * sizeof(float));
  } else {
    p.dO = take(p.hpc * head);
    p.D = take(2 * (size_t)p.hpc * ceil_div(p.S, kTile) * kTile * sizeof(float));
    p.dq = take((p.hpc + 2 * p.kvc) * head);  // [dQ heads | dK heads | dV heads], one 3-D tensor
    p.dk = p.dq + p.hpc * head;
    p.dv = p.dk + p.kvc * head;
    p.window = dkdv_window();
    p.kv_sums = p.hpc < p.g || (int64_t)p.g * ceil_div(p.S, kTile) > p.window;
    if (p.kv_sums) {
      p.dkacc = take((size_t)p.kvc * p.S * p.Dh * sizeof(float));
      p.dvacc = take((size_t)p.kvc * p.S * p.Dh * sizeof(float));
    }
    if (multi && p.accum == 0) p.dxacc = take((size_t)p.S * p.d * sizeof(float));
    const int sms = num_sms();
    p.split_wo = gemm_pick_split(p.d, (int64_t)p.hpc * p.Dh, p.S, sms);
    p.split_wqkv_q = gemm_pick_split((int64_t)p.hpc * p.Dh, p.d, p.S, sms);
    const int64_t full_rows = (int64_t)(p.hpc + 2 * p.kvc) * p.Dh;
    p.split_wqkv_full = gemm_pick_split(full_rows, p.d, p.S, sms);
    size_t sb = gemm_split_scratch_bytes(p.d, (int64_t)p.hpc * p.Dh, p.split_wo);
    sb = std::max(sb, gemm_split_scratch_bytes((int64_t)p.hpc * p.Dh, p.d, p.split_wqkv_q));
    sb = std::max(sb, gemm_split_scratch_bytes(full_rows, p.d, p.split_wqkv_full));
    if (p.R) {  // the weight gradients are summed block by block: K = one block's rows
      p.split_wo_blk = gemm_pick_split(p.d, (int64_t)p.hpc * p.Dh, p.R, sms);
      p.split_wqkv_q_blk = gemm_pick_split((int64_t)p.hpc * p.Dh, p.d, p.R, sms);
      p.split_wqkv_full_blk = gemm_pick_split(full_rows, p.d, p.R, sms);
      sb = std::max(sb, gemm_split_scratch_bytes(p.d, (int64_t)p.hpc * p.Dh, p.split_wo_blk));
      sb = std::max(sb, gemm_split_scratch_bytes((int64_t)p.hpc * p.Dh, p.d, p.split_wqkv_q_blk));
      sb = std::max(sb, gemm_split_scratch_bytes(full_rows, p.d, p.split_wqkv_full_blk));
    }
    if (sb) p.split = take(sb);
  }
  p.total = off;
  return p;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(reinterpret_cast<char*>(ws) + off);
}

#define UPIPE_CUDA(x)                                 \
  do {                                                \
    const cudaError_t e_ = (x);                       \
    if (e_ != cudaSuccess) return cuda_status(e_);    \
  } while (0)

// Wqkv row of the first weight row of a head: Q heads, then K heads, then V heads.
inline int64_t wrow_q(const Plan& p, int h) { return (int64_t)h * p.Dh; }
inline int64_t wrow_k(const Plan& p, int kv) { return (int64_t)(p.Hq + kv) * p.Dh; }
inline int64_t wrow_v(const Plan& p, int kv) { return (int64_t)(p.Hq + p.Hkv + kv) * p.Dh; }

int log2i(int x) {
  int s = 0;
  while ((1 << s) < x) ++s;
  return s;
}

TcOperand op2d(const void* base, uint64_t inner, uint64_t outer, uint64_t row_stride, int k_major) {
  TcOperand o{};
  o.base = base; o.rank = 2; o.inner = inner; o.outer = outer; o.planes = 1; o.row_stride = row_stride;
  o.k_major = k_major; o.blk_shift = -1; o.blk_dim = 0;
  return o;
}

TcOperand op3d(const void* base, uint64_t inner, uint64_t outer, uint64_t planes, int k_major, int blk_shift,
               int blk_dim) {
  TcOperand o{};
  o.base = base; o.rank = 3; o.inner = inner; o.outer = outer; o.planes = planes; o.row_stride = inner;
  o.k_major = k_major; o.blk_shift = blk_shift; o.blk_dim = blk_dim;
  return o;
}

// Rows [r0, r0 + rows) of a head-major [planes][S][Dh] workspace tensor as a 3-D operand.
TcOperand op3d_rows(const Plan& p, const bf16* base, uint64_t planes, int64_t r0, int64_t rows, int k_major,
                    int blk_shift, int blk_dim) {
  TcOperand o = op3d(base + r0 * p.Dh, p.Dh, (uint64_t)rows, planes, k_major, blk_shift, blk_dim);
  o.plane_stride = (uint64_t)p.S * p.Dh;
  return o;
}

// Q (and, at the start of a KV group, K and V) of chunk c:  [Q|K|V]_c = X * Wqkv_c^T for the
// sequence rows [r0, r0 + rows); Xr points at row r0's hidden state (rows of d elements).
// B = the chunk's rows of Wqkv (a 2-D map with one starting row per head), output head-major.
cudaError_t project_qkv(const Plan& p, int c, bool with_kv, const bf16* Xr, int64_t r0, int64_t rows,
                        const bf16* Wqkv, void* ws, cudaStream_t st) {
  TcGemmArgs g{};
  const int sh = log2i(p.Dh);
  const uint64_t wrows = (uint64_t)(p.Hq + 2 * p.Hkv) * p.Dh;
  g.a = op2d(Xr, p.d, (uint64_t)rows, p.d, 1);
  g.b = op2d(Wqkv, p.d, wrows, p.d, 1);
  g.b.blk_shift = sh; g.b.blk_dim = 0;
  g.c.ld = p.Dh; g.c.blk_shift = sh; g.c.blk_dim = 1;
  int nb = 0;
  for (int hl = 0; hl < p.hpc; ++hl, ++nb) {
    g.b.row_base[nb] = (int32_t)wrow_q(p, c * p.hpc + hl);
    g.c.blk[nb] = at<bf16>(ws, p.q) + (int64_t)hl * p.S * p.Dh + r0 * p.Dh;
  }
  if (with_kv) {
    const int kv0 = (c * p.hpc) / p.g;
    for (int j = 0; j < p.kvc; ++j, ++nb) {
      g.b.row_base[nb] = (int32_t)wrow_k(p, kv0 + j);
      g.c.blk[nb] = at<bf16>(ws, p.k) + (int64_t)j * p.S * p.Dh + r0 * p.Dh;
    }
    for (int j = 0; j < p.kvc; ++j, ++nb) {
      g.b.row_base[nb] = (int32_t)wrow_v(p, kv0 + j);
      g.c.blk[nb] = at<bf16>(ws, p.v) + (int64_t)j * p.S * p.Dh + r0 * p.Dh;
    }
  }
  g.M = rows; g.N = (int64_t)nb * p.Dh; g.K = p.d;
  g.epi = EPI_STORE_BF16;
  return launch_gemm_tc(g, 1, nullptr, st);
}

// dO_c rows [r0, r0 + rows) = dY rows * Wo_c   (Wo_c: columns of Wo, read as [K = d][N = hpc Dh])
cudaError_t project_do(const Plan& p, int c, const bf16* dYr, int64_t r0, int64_t rows, const bf16* Wo, void* ws,
                       cudaStream_t st) {
  TcGemmArgs g{};
  g.M = rows; g.N = (int64_t)p.hpc * p.Dh; g.K = p.d;
  g.a = op2d(dYr, p.d, (uint64_t)rows, p.d, 1);
  g.b = op2d(Wo + (int64_t)c * p.hpc * p.Dh, (uint64_t)p.hpc * p.Dh, p.d, (uint64_t)p.Hq * p.Dh, 0);
  for (int hl = 0; hl < p.hpc; ++hl) g.c.blk[hl] = at<bf16>(ws, p.dO) + (int64_t)hl * p.S * p.Dh + r0 * p.Dh;
  g.c.ld = p.Dh; g.c.blk_shift = log2i(p.Dh); g.c.blk_dim = 1;
  g.epi = EPI_STORE_BF16;
  return launch_gemm_tc(g, 1, nullptr, st);
}

// Epilogue schedule of a quantity accumulated over the n_chunks chunks (Y, dX): the first chunk
// stores, later chunks add (accum_mode 0: into the fp32 workspace sum, reduced in L2 by TMA;
// accum_mode 1: into the bf16 output in place).  With accum_mode 0 the fp32 sum is rounded to
// bf16 once, after the last chunk (accum_finish).
int accum_epi(const Plan& p, int c) {
  if (p.n_chunks == 1) return EPI_STORE_BF16;
  if (p.accum == 1) return c == 0 ? EPI_STORE_BF16 : EPI_ACC_BF16;
  return c == 0 ? EPI_STORE_F32 : EPI_ACC_F32;
}

bool finishes_accum(const Plan& p, int c) { return p.n_chunks > 1 && p.accum == 0 && c == p.n_chunks - 1; }

cudaError_t accum_finish(const Plan& p, int c, const float* acc, bf16* out, cudaStream_t st) {
  if (!finishes_accum(p, c)) return cudaSuccess;
  return launch_f32_to_bf16(acc, out, p.S * p.d, 1.f, st);
}

void set_accum_out(GemmOutput& o, const Plan& p, int epi, void* bf16_out, float* acc) {
  o.blk_shift = -1; o.blk_dim = 0; o.ld = p.d;
  if (epi == EPI_STORE_F32 || epi == EPI_ACC_F32) o.blk[0] = acc;
  else o.blk[0] = bf16_out;
}

AttnArgs attn_args(const Plan& p, int c, void* ws, const int32_t* seg, float* lse) {
  AttnArgs a{};
  a.q = at<bf16>(ws, p.q);
  a.k = at<bf16>(ws, p.k);
  a.v = at<bf16>(ws, p.v);
  a.o = at<bf16>(ws, p.o);
  a.lse = lse + (int64_t)c * p.hpc * p.S;
  a.seg = seg;
  a.q_rows = table_q_rows(at<char>(ws, p.table));
  a.kv_rows = table_kv_rows(at<char>(ws, p.table), p.S);
  a.q_order = table_q_order(at<char>(ws, p.table), p.S);
  a.kv_order = table_kv_order(at<char>(ws, p.table), p.S);
  a.S = p.S;
  a.nh = p.hpc;
  a.nkv = p.kvc;
  a.g = p.g;
  a.causal = p.causal;
  a.scale = p.scale;
  a.err = &at<TableHeader>(ws, p.table)->error;
  return a;
}

// width (columns) of the chunk's Q (and, at a group start, K and V) projection
int64_t qkv_width(const Plan& p, bool with_kv) { return (int64_t)(p.hpc + (with_kv ? 2 * p.kvc : 0)) * p.Dh; }

upipe_status_t run_fwd(const Plan& p, const bf16* X, const bf16* Wqkv, const bf16* Wo, const int32_t* seg, bf16* Y,
                       float* lse, void* ws, cudaStream_t st) {
  {
    Timed t(UPIPE_K_TILE_TABLE, 0, p.S, 0, 0, 1, -1, st);
    UPIPE_CUDA(launch_tile_table(p.S, p.causal, seg, at<char>(ws, p.table), st));
  }
  const int sh = log2i(p.Dh);
  for (int c = 0; c < p.n_chunks; ++c) {
    const bool new_group = p.hpc >= p.g || (c * p.hpc) % p.g == 0;
    {
      Timed t(UPIPE_K_QKV_PROJ, EPI_STORE_BF16, p.S, qkv_width(p, new_group), p.d, 1, c, st);
      UPIPE_CUDA(project_qkv(p, c, new_group, X, 0, p.S, Wqkv, ws, st));
    }
    AttnArgs a = attn_args(p, c, ws, seg, lse);
    {
      Timed t(UPIPE_K_ATTN_FWD, 0, p.S, p.hpc, p.Dh, 1, c, st);
      UPIPE_CUDA(launch_attn_fwd(a, p.Dh, st));
    }
    // Y (+)= O_c * Wo_c^T
    TcGemmArgs g{};
    g.M = p.S; g.N = p.d; g.K = (int64_t)p.hpc * p.Dh;
    g.a = op3d(at<bf16>(ws, p.o), p.Dh, p.S, p.hpc, 1, sh, 1);                        // O_c, K blocked by head
    g.b = op2d(Wo + (int64_t)c * p.hpc * p.Dh, (uint64_t)p.hpc * p.Dh, p.d, (uint64_t)p.Hq * p.Dh, 1);  // Wo_c
    g.epi = accum_epi(p, c);
    set_accum_out(g.c, p, g.epi, Y, p.yacc ? at<float>(ws, p.yacc) : nullptr);
    {
      Timed t(UPIPE_K_O_PROJ, g.epi, g.M, g.N, g.K, 1, c, st);
      UPIPE_CUDA(launch_gemm_tc(g, 1, nullptr, st));
    }
    if (finishes_accum(p, c)) {
      Timed t(UPIPE_K_CONVERT, 0, p.S * p.d, 1, 1, 1, c, st);
      UPIPE_CUDA(accum_finish(p, c, p.yacc ? at<float>(ws, p.yacc) : nullptr, Y, st));
    }
  }
  return UPIPE_OK;
}

upipe_status_t run_bwd(const Plan& p, const bf16* X, const bf16* Wqkv, const bf16* Wo, const int32_t* seg,
                       const bf16* dY, const float* lse, bf16* dX, float* dWqkv, float* dWo, void* ws, cudaStream_t st) {
  {
    Timed t(UPIPE_K_TILE_TABLE, 0, p.S, 0, 0, 1, -1, st);
    UPIPE_CUDA(launch_tile_table(p.S, p.causal, seg, at<char>(ws, p.table), st));
  }
  const int sh = log2i(p.Dh);
  const int64_t HD = (int64_t)p.Hq * p.Dh;
  float* split = p.split ? at<float>(ws, p.split) : nullptr;
  for (int c = 0; c < p.n_chunks; ++c) {
    const bool new_group = p.hpc >= p.g || (c * p.hpc) % p.g == 0;
    const bool end_group = p.hpc >= p.g || ((c + 1) * p.hpc) % p.g == 0;
    const int kv0 = (c * p.hpc) / p.g;
    {
      Timed t(UPIPE_K_QKV_PROJ, EPI_STORE_BF16, p.S, qkv_width(p, new_group), p.d, 1, c, st);
      UPIPE_CUDA(project_qkv(p, c, new_group, X, 0, p.S, Wqkv, ws, st));
    }
    if (new_group && p.kv_sums) {
      Timed t(UPIPE_K_ZERO, 0, 2 * p.kvc * p.S * p.Dh, 1, 1, 1, c, st);
      UPIPE_CUDA(launch_zero(at<char>(ws, p.dkacc), (int64_t)p.kvc * p.S * p.Dh * 4, st));
      UPIPE_CUDA(launch_zero(at<char>(ws, p.dvacc), (int64_t)p.kvc * p.S * p.Dh * 4, st));
    }
    {  // dO_c = dY * Wo_c
      Timed t(UPIPE_K_DO_PROJ, EPI_STORE_BF16, p.S, (int64_t)p.hpc * p.Dh, p.d, 1, c, st);
      UPIPE_CUDA(project_do(p, c, dY, 0, p.S, Wo, ws, st));
    }
    AttnArgs a = attn_args(p, c, ws, seg, const_cast<float*>(lse));
    a.dO = at<bf16>(ws, p.dO);
    a.D = at<float>(ws, p.D);
    {
      Timed t(UPIPE_K_RECOMPUTE, 0, p.S, p.hpc, p.Dh, 1, c, st);
      UPIPE_CUDA(launch_attn_recompute(a, p.Dh, st));
    }
    {  // dWo_c = dY^T * O_c   (split-K over S)
      TcGemmArgs g{};
      g.M = p.d; g.N = (int64_t)p.hpc * p.Dh; g.K = p.S;
      g.a = op2d(dY, p.d, p.S, p.d, 0);                              // dY^T: M runs along d
      g.b = op3d(at<bf16>(ws, p.o), p.Dh, p.S, p.hpc, 0, sh, 0);    // O_c: N blocked by head
      g.c.blk[0] = dWo + (int64_t)c * p.hpc * p.Dh; g.c.ld = HD; g.c.blk_shift = -1;
      g.epi = EPI_STORE_F32;
      Timed t(UPIPE_K_DWO, g.epi, g.M, g.N, g.K, p.split_wo, c, st);
      UPIPE_CUDA(launch_gemm_tc(g, p.split_wo, split, st));
    }
    AttnBwdArgs b{};
    b.f = a;
    b.dq = at<bf16>(ws, p.dq);
    b.dk = at<bf16>(ws, p.dk);
    b.dv = at<bf16>(ws, p.dv);
    b.acc_kv = p.kv_sums;
    b.flush_items = p.window;
    b.dk_acc = p.dkacc ? at<float>(ws, p.dkacc) : nullptr;
    b.dv_acc = p.dvacc ? at<float>(ws, p.dvacc) : nullptr;
    b.nkv = p.kvc;
    {
      Timed t(UPIPE_K_BWD_DQ, 0, p.S, p.hpc, p.Dh, 1, c, st);
      UPIPE_CUDA(launch_attn_bwd_dq(b, p.Dh, st));
    }
    {
      Timed t(UPIPE_K_BWD_DKDV, 0, p.S, p.hpc, p.Dh, 1, c, st);
      UPIPE_CUDA(launch_attn_bwd_dkdv(b, p.Dh, st));
    }
    if (end_group && p.kv_sums) {
      Timed t(UPIPE_K_CONVERT, 0, 2 * p.kvc * p.S * p.Dh, 1, 1, 1, c, st);
      UPIPE_CUDA(launch_f32_to_bf16(at<float>(ws, p.dkacc), at<bf16>(ws, p.dk), p.kvc * p.S * p.Dh, 1.f, st));
      UPIPE_CUDA(launch_f32_to_bf16(at<float>(ws, p.dvacc), at<bf16>(ws, p.dv), p.kvc * p.S * p.Dh, 1.f, st));
    }
    // blocks of dQKV_c that are final now: the chunk's dQ heads, plus dK/dV at a group end.
    // They are planes [0, nb) of the [dQ | dK | dV] tensor of the workspace.
    int32_t blk_row[kMaxBlocks];
    int nb = 0;
    for (int hl = 0; hl < p.hpc; ++hl, ++nb) blk_row[nb] = (int32_t)wrow_q(p, c * p.hpc + hl);
    if (end_group) {
      for (int j = 0; j < p.kvc; ++j, ++nb) blk_row[nb] = (int32_t)wrow_k(p, kv0 + j);
      for (int j = 0; j < p.kvc; ++j, ++nb) blk_row[nb] = (int32_t)wrow_v(p, kv0 + j);
    }
    const uint64_t planes = (uint64_t)(p.hpc + 2 * p.kvc);
    const uint64_t wrows = (uint64_t)(p.Hq + 2 * p.Hkv) * p.Dh;
    {  // dX (+)= dQKV_c * Wqkv_c
      TcGemmArgs g{};
      g.M = p.S; g.N = p.d; g.K = (int64_t)nb * p.Dh;
      g.a = op3d(at<bf16>(ws, p.dq), p.Dh, p.S, planes, 1, sh, 1);   // K blocked by head
      g.b = op2d(Wqkv, p.d, wrows, p.d, 0);                           // rows of the blocks, N along d
      g.b.blk_shift = sh; g.b.blk_dim = 1;
      for (int i = 0; i < nb; ++i) g.b.row_base[i] = blk_row[i];
      g.epi = accum_epi(p, c);
      set_accum_out(g.c, p, g.epi, dX, p.dxacc ? at<float>(ws, p.dxacc) : nullptr);
      {
        Timed t(UPIPE_K_DX_PROJ, g.epi, g.M, g.N, g.K, 1, c, st);
        UPIPE_CUDA(launch_gemm_tc(g, 1, nullptr, st));
      }
      if (finishes_accum(p, c)) {
        Timed t(UPIPE_K_CONVERT, 0, p.S * p.d, 1, 1, 1, c, st);
        UPIPE_CUDA(accum_finish(p, c, p.dxacc ? at<float>(ws, p.dxacc) : nullptr, dX, st));
      }
    }
    {  // dWqkv rows of these blocks = dQKV_block^T * X   (split-K over S)
      TcGemmArgs g{};
      g.M = (int64_t)nb * p.Dh; g.N = p.d; g.K = p.S;
      g.a = op3d(at<bf16>(ws, p.dq), p.Dh, p.S, planes, 0, sh, 0);   // M blocked by head
      g.b = op2d(X, p.d, p.S, p.d, 0);
      for (int i = 0; i < nb; ++i) g.c.blk[i] = dWqkv + (int64_t)blk_row[i] * p.d;
      g.c.ld = p.d; g.c.blk_shift = sh; g.c.blk_dim = 0;
      g.epi = EPI_STORE_F32;
      const int split_k = nb == p.hpc ? p.split_wqkv_q : p.split_wqkv_full;
      Timed t(UPIPE_K_DWQKV, g.epi, g.M, g.N, g.K, split_k, c, st);
      UPIPE_CUDA(launch_gemm_tc(g, split_k, split, st));
    }
  }
  return UPIPE_OK;
}

// ------------------------------------------------------------------------ host-resident X / dY
// CPU offload of the layer's inputs ("Road to 5 Million Tokens" podcast summary, chapter on
// offloading part of the inputs to the CPU; neuro-slop.ru transcript, implementation plan step
// 2): X and dY stay in pinned host memory and are brought in block by block, R rows at a time,
// into two device staging buffers each.  Every block is one cudaMemcpyAsync on the device's copy
// stream (created once and kept), issued one block ahead, so the copy of block b + 1 runs while the
// projections of block b do.
// Events order the reuse of a staging buffer after the kernels that read it.
// The staging copy stream of a device: created on first use and kept for the life of the process
// (one per device; calls that run concurrently share it, which only orders their copies).
cudaError_t copy_stream(cudaStream_t* out) {
  static std::mutex mu;
  static cudaStream_t streams[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!streams[dev]) {
    e = cudaStreamCreateWithFlags(&streams[dev], cudaStreamNonBlocking);
    if (e != cudaSuccess) return e;
  }
  *out = streams[dev];
  return cudaSuccess;
}

class Stager {
 public:
  // hx / hdy: the tensors; those with *_host set are staged, the others are device memory read in
  // place (a device-resident dY, for instance, as a training stack produces it in the backward)
  Stager(const Plan& p, void* ws, cudaStream_t st, const bf16* hx, bool x_host, const bf16* hdy, bool dy_host)
      : p_(p), ws_(ws), st_(st), hx_(hx), hdy_(hdy), x_host_(x_host), dy_host_(dy_host) {}
  ~Stager() {
    for (cudaEvent_t e : {entry_, ready_[0], ready_[1], free_[0], free_[1]})
      if (e) cudaEventDestroy(e);
  }
  cudaError_t begin() {
    cudaError_t e = copy_stream(&cs_);
    for (cudaEvent_t* ev : {&entry_, &ready_[0], &ready_[1], &free_[0], &free_[1]})
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    // the copies start after the work queued before this call (which may still read the buffers)
    if (e == cudaSuccess) e = cudaEventRecord(entry_, st_);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs_, entry_, 0);
    for (int k = 0; k < 2 && e == cudaSuccess; ++k) e = cudaEventRecord(free_[k], st_);
    return e;
  }
  int64_t blocks() const { return ceil_div(p_.S, p_.R); }
  int64_t row0(int64_t b) const { return b * p_.R; }
  int64_t rows(int64_t b) const { return std::min(p_.R, p_.S - b * p_.R); }
  const bf16* x(int64_t b) const { return x_host_ ? at<bf16>(ws_, p_.xs[b & 1]) : hx_ + row0(b) * p_.d; }
  const bf16* dy(int64_t b) const { return dy_host_ ? at<bf16>(ws_, p_.dys[b & 1]) : hdy_ + row0(b) * p_.d; }
  // copy block b of each host tensor into staging buffer b % 2 once its last readers are done
  cudaError_t prefetch(int64_t b) {
    const int k = (int)(b & 1);
    const size_t bytes = (size_t)rows(b) * p_.d * sizeof(bf16);
    const size_t off = (size_t)row0(b) * p_.d;
    cudaError_t e = cudaStreamWaitEvent(cs_, free_[k], 0);
    Timed t(UPIPE_K_H2D, 0, (int64_t)bytes * ((x_host_ ? 1 : 0) + (hdy_ && dy_host_ ? 1 : 0)), 1, 1, 1, (int)b, cs_);
    if (e == cudaSuccess && x_host_)
      e = cudaMemcpyAsync(at<bf16>(ws_, p_.xs[k]), hx_ + off, bytes, cudaMemcpyHostToDevice, cs_);
    if (e == cudaSuccess && hdy_ && dy_host_)
      e = cudaMemcpyAsync(at<bf16>(ws_, p_.dys[k]), hdy_ + off, bytes, cudaMemcpyHostToDevice, cs_);
    if (e == cudaSuccess) e = cudaEventRecord(ready_[k], cs_);
    return e;
  }
  cudaError_t acquire(int64_t b) { return cudaStreamWaitEvent(st_, ready_[b & 1], 0); }
  cudaError_t release(int64_t b) { return cudaEventRecord(free_[b & 1], st_); }

 private:
  const Plan& p_;
  void* ws_;
  cudaStream_t st_;
  const bf16* hx_;
  const bf16* hdy_;
  bool x_host_, dy_host_;
  cudaStream_t cs_ = nullptr;
  cudaEvent_t entry_ = nullptr, ready_[2] = {nullptr, nullptr}, free_[2] = {nullptr, nullptr};
};

// f(b, r0, rows) for every staged block, each with its block resident in the staging buffers.
template <typename F>
upipe_status_t over_blocks(Stager& sg, F&& f) {
  const int64_t nb = sg.blocks();
  UPIPE_CUDA(sg.prefetch(0));
  for (int64_t b = 0; b < nb; ++b) {
    if (b + 1 < nb) UPIPE_CUDA(sg.prefetch(b + 1));
    UPIPE_CUDA(sg.acquire(b));
    const upipe_status_t s = f(b, sg.row0(b), sg.rows(b));
    if (s != UPIPE_OK) return s;
    UPIPE_CUDA(sg.release(b));
  }
  return UPIPE_OK;
}

// A weight gradient summed over the staged blocks: block 0 stores, later blocks add (split-K
// partials of a block are reduced in a fixed order, onto the running sum).
cudaError_t block_weight_grad(TcGemmArgs g, int64_t b, int split, float* scratch, cudaStream_t st) {
  if (split > 1) {
    g.epi = EPI_STORE_F32;
    g.split_accumulate = b > 0;
  } else {
    g.epi = b > 0 ? EPI_ACC_F32 : EPI_STORE_F32;
  }
  return launch_gemm_tc(g, split, scratch, st);
}

upipe_status_t run_fwd_offload(const Plan& p, const bf16* hX, bool x_host, const bf16* Wqkv, const bf16* Wo,
                               const int32_t* seg, bf16* Y, float* lse, void* ws, cudaStream_t st) {
  Stager sg(p, ws, st, hX, x_host, nullptr, false);
  UPIPE_CUDA(sg.begin());
  {
    Timed t(UPIPE_K_TILE_TABLE, 0, p.S, 0, 0, 1, -1, st);
    UPIPE_CUDA(launch_tile_table(p.S, p.causal, seg, at<char>(ws, p.table), st));
  }
  const int sh = log2i(p.Dh);
  for (int c = 0; c < p.n_chunks; ++c) {
    const bool new_group = p.hpc >= p.g || (c * p.hpc) % p.g == 0;
    upipe_status_t s = over_blocks(sg, [&](int64_t b, int64_t r0, int64_t rows) -> upipe_status_t {
      Timed t(UPIPE_K_QKV_PROJ, EPI_STORE_BF16, rows, qkv_width(p, new_group), p.d, 1, c, st);
      UPIPE_CUDA(project_qkv(p, c, new_group, sg.x(b), r0, rows, Wqkv, ws, st));
      return UPIPE_OK;
    });
    if (s != UPIPE_OK) return s;
    AttnArgs a = attn_args(p, c, ws, seg, lse);
    {
      Timed t(UPIPE_K_ATTN_FWD, 0, p.S, p.hpc, p.Dh, 1, c, st);
      UPIPE_CUDA(launch_attn_fwd(a, p.Dh, st));
    }
    TcGemmArgs g{};
    g.M = p.S; g.N = p.d; g.K = (int64_t)p.hpc * p.Dh;
    g.a = op3d(at<bf16>(ws, p.o), p.Dh, p.S, p.hpc, 1, sh, 1);
    g.b = op2d(Wo + (int64_t)c * p.hpc * p.Dh, (uint64_t)p.hpc * p.Dh, p.d, (uint64_t)p.Hq * p.Dh, 1);
    g.epi = accum_epi(p, c);
    set_accum_out(g.c, p, g.epi, Y, p.yacc ? at<float>(ws, p.yacc) : nullptr);
    {
      Timed t(UPIPE_K_O_PROJ, g.epi, g.M, g.N, g.K, 1, c, st);
      UPIPE_CUDA(launch_gemm_tc(g, 1, nullptr, st));
    }
    if (finishes_accum(p, c)) {
      Timed t(UPIPE_K_CONVERT, 0, p.S * p.d, 1, 1, 1, c, st);
      UPIPE_CUDA(accum_finish(p, c, p.yacc ? at<float>(ws, p.yacc) : nullptr, Y, st));
    }
  }
  return UPIPE_OK;
}

// Backward with X and dY in host memory.  Per chunk, two passes over the staged blocks: before
// the attention kernels the chunk's Q (K, V) and dO projections; after them the weight
// gradients dWo_c = dY^T O_c and dWqkv_c = dQKV_c^T X, summed block by block.  dX needs neither
// X nor dY and runs over the whole sequence as in upipe_attn_bwd.
upipe_status_t run_bwd_offload(const Plan& p, const bf16* hX, bool x_host, const bf16* Wqkv, const bf16* Wo,
                               const int32_t* seg, const bf16* hdY, bool dy_host, const float* lse, bf16* dX,
                               float* dWqkv, float* dWo, void* ws, cudaStream_t st) {
  Stager sg(p, ws, st, hX, x_host, hdY, dy_host);
  UPIPE_CUDA(sg.begin());
  {
    Timed t(UPIPE_K_TILE_TABLE, 0, p.S, 0, 0, 1, -1, st);
    UPIPE_CUDA(launch_tile_table(p.S, p.causal, seg, at<char>(ws, p.table), st));
  }
  const int sh = log2i(p.Dh);
  const int64_t HD = (int64_t)p.Hq * p.Dh;
  float* split = p.split ? at<float>(ws, p.split) : nullptr;
  for (int c = 0; c < p.n_chunks; ++c) {
    const bool new_group = p.hpc >= p.g || (c * p.hpc) % p.g == 0;
    const bool end_group = p.hpc >= p.g || ((c + 1) * p.hpc) % p.g == 0;
    const int kv0 = (c * p.hpc) / p.g;
    if (new_group && p.kv_sums) {
      Timed t(UPIPE_K_ZERO, 0, 2 * p.kvc * p.S * p.Dh, 1, 1, 1, c, st);
      UPIPE_CUDA(launch_zero(at<char>(ws, p.dkacc), (int64_t)p.kvc * p.S * p.Dh * 4, st));
      UPIPE_CUDA(launch_zero(at<char>(ws, p.dvacc), (int64_t)p.kvc * p.S * p.Dh * 4, st));
    }
    upipe_status_t s = over_blocks(sg, [&](int64_t b, int64_t r0, int64_t rows) -> upipe_status_t {
      {
        Timed t(UPIPE_K_QKV_PROJ, EPI_STORE_BF16, rows, qkv_width(p, new_group), p.d, 1, c, st);
        UPIPE_CUDA(project_qkv(p, c, new_group, sg.x(b), r0, rows, Wqkv, ws, st));
      }
      Timed t(UPIPE_K_DO_PROJ, EPI_STORE_BF16, rows, (int64_t)p.hpc * p.Dh, p.d, 1, c, st);
      UPIPE_CUDA(project_do(p, c, sg.dy(b), r0, rows, Wo, ws, st));
      return UPIPE_OK;
    });
    if (s != UPIPE_OK) return s;
    AttnArgs a = attn_args(p, c, ws, seg, const_cast<float*>(lse));
    a.dO = at<bf16>(ws, p.dO);
    a.D = at<float>(ws, p.D);
    {
      Timed t(UPIPE_K_RECOMPUTE, 0, p.S, p.hpc, p.Dh, 1, c, st);
      UPIPE_CUDA(launch_attn_recompute(a, p.Dh, st));
    }
    AttnBwdArgs bw{};
    bw.f = a;
    bw.dq = at<bf16>(ws, p.dq);
    bw.dk = at<bf16>(ws, p.dk);
    bw.dv = at<bf16>(ws, p.dv);
    bw.acc_kv = p.kv_sums;
    bw.flush_items = p.window;
    bw.dk_acc = p.dkacc ? at<float>(ws, p.dkacc) : nullptr;
    bw.dv_acc = p.dvacc ? at<float>(ws, p.dvacc) : nullptr;
    bw.nkv = p.kvc;
    {
      Timed t(UPIPE_K_BWD_DQ, 0, p.S, p.hpc, p.Dh, 1, c, st);
      UPIPE_CUDA(launch_attn_bwd_dq(bw, p.Dh, st));
    }
    {
      Timed t(UPIPE_K_BWD_DKDV, 0, p.S, p.hpc, p.Dh, 1, c, st);
      UPIPE_CUDA(launch_attn_bwd_dkdv(bw, p.Dh, st));
    }
    if (end_group && p.kv_sums) {
      Timed t(UPIPE_K_CONVERT, 0, 2 * p.kvc * p.S * p.Dh, 1, 1, 1, c, st);
      UPIPE_CUDA(launch_f32_to_bf16(at<float>(ws, p.dkacc), at<bf16>(ws, p.dk), p.kvc * p.S * p.Dh, 1.f, st));
      UPIPE_CUDA(launch_f32_to_bf16(at<float>(ws, p.dvacc), at<bf16>(ws, p.dv), p.kvc * p.S * p.Dh, 1.f, st));
    }
    int32_t blk_row[kMaxBlocks];
    int nb = 0;
    for (int hl = 0; hl < p.hpc; ++hl, ++nb) blk_row[nb] = (int32_t)wrow_q(p, c * p.hpc + hl);
    if (end_group) {
      for (int j = 0; j < p.kvc; ++j, ++nb) blk_row[nb] = (int32_t)wrow_k(p, kv0 + j);
      for (int j = 0; j < p.kvc; ++j, ++nb) blk_row[nb] = (int32_t)wrow_v(p, kv0 + j);
    }
    const uint64_t planes = (uint64_t)(p.hpc + 2 * p.kvc);
    const uint64_t wrows = (uint64_t)(p.Hq + 2 * p.Hkv) * p.Dh;
    {  // dX (+)= dQKV_c * Wqkv_c over the whole sequence
      TcGemmArgs g{};
      g.M = p.S; g.N = p.d; g.K = (int64_t)nb * p.Dh;
      g.a = op3d(at<bf16>(ws, p.dq), p.Dh, p.S, planes, 1, sh, 1);
      g.b = op2d(Wqkv, p.d, wrows, p.d, 0);
      g.b.blk_shift = sh; g.b.blk_dim = 1;
      for (int i = 0; i < nb; ++i) g.b.row_base[i] = blk_row[i];
      g.epi = accum_epi(p, c);
      set_accum_out(g.c, p, g.epi, dX, p.dxacc ? at<float>(ws, p.dxacc) : nullptr);
      {
        Timed t(UPIPE_K_DX_PROJ, g.epi, g.M, g.N, g.K, 1, c, st);
        UPIPE_CUDA(launch_gemm_tc(g, 1, nullptr, st));
      }
      if (finishes_accum(p, c)) {
        Timed t(UPIPE_K_CONVERT, 0, p.S * p.d, 1, 1, 1, c, st);
        UPIPE_CUDA(accum_finish(p, c, p.dxacc ? at<float>(ws, p.dxacc) : nullptr, dX, st));
      }
    }
    const int split_qkv = nb == p.hpc ? p.split_wqkv_q_blk : p.split_wqkv_full_blk;
    s = over_blocks(sg, [&](int64_t b, int64_t r0, int64_t rows) -> upipe_status_t {
      {  // dWo_c (+)= dY_b^T * O_c rows of the block
        TcGemmArgs g{};
        g.M = p.d; g.N = (int64_t)p.hpc * p.Dh; g.K = rows;
        g.a = op2d(sg.dy(b), p.d, (uint64_t)rows, p.d, 0);
        g.b = op3d_rows(p, at<bf16>(ws, p.o), p.hpc, r0, rows, 0, sh, 0);
        g.c.blk[0] = dWo + (int64_t)c * p.hpc * p.Dh; g.c.ld = HD; g.c.blk_shift = -1;
        Timed t(UPIPE_K_DWO, b > 0 ? EPI_ACC_F32 : EPI_STORE_F32, g.M, g.N, g.K, p.split_wo_blk, c, st);
        UPIPE_CUDA(block_weight_grad(g, b, p.split_wo_blk, split, st));
      }
      // dWqkv rows of the final blocks (+)= dQKV_b^T * X_b
      TcGemmArgs g{};
      g.M = (int64_t)nb * p.Dh; g.N = p.d; g.K = rows;
      g.a = op3d_rows(p, at<bf16>(ws, p.dq), planes, r0, rows, 0, sh, 0);
      g.b = op2d(sg.x(b), p.d, (uint64_t)rows, p.d, 0);
      for (int i = 0; i < nb; ++i) g.c.blk[i] = dWqkv + (int64_t)blk_row[i] * p.d;
      g.c.ld = p.d; g.c.blk_shift = sh; g.c.blk_dim = 0;
      Timed t(UPIPE_K_DWQKV, b > 0 ? EPI_ACC_F32 : EPI_STORE_F32, g.M, g.N, g.K, split_qkv, c, st);
      UPIPE_CUDA(block_weight_grad(g, b, split_qkv, split, st));
      return UPIPE_OK;
    });
    if (s != UPIPE_OK) return s;
  }
  return UPIPE_OK;
}

// ------------------------------------------------------------------------ sequence-tiled MLP
// SwiGLU feed-forward computed a tile of rows at a time (the element-wise steps beside the layer,
// tiled along the sequence: podcast summary, chapter on sequence tiling).  Workspace: one tile's
// H = [G | U] bf16 [T][2F] and A bf16 [T][F] (forward), plus dA [T][F] and dH [T][2F] (backward)
// and the weight gradients' split-K partials.
struct MlpPlan {
  int64_t S, T;
  int d, F;
  size_t H, A, dA, dH, split, total;
  int split_dwd, split_dwgu;
};

upipe_status_t check_mlp(const upipe_mlp_desc_t* m) {
  if (!m || m->seq_len < 1 || m->seq_len > INT32_MAX || m->hidden <= 0 || m->ffn <= 0) return UPIPE_ERR_INVALID_ARG;
  if (m->tile_rows < 0 || m->tile_rows % kTile != 0) return UPIPE_ERR_INVALID_ARG;
  if (m->hidden % 64 != 0 || m->ffn % 64 != 0) return UPIPE_ERR_UNSUPPORTED;
  return UPIPE_OK;
}

MlpPlan make_mlp_plan(const upipe_mlp_desc_t* m, int pass) {
  MlpPlan p{};
  p.S = m->seq_len;
  p.d = m->hidden;
  p.F = m->ffn;
  p.T = m->tile_rows == 0 ? p.S : std::min<int64_t>(m->tile_rows, p.S);
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes); return o; };
  p.H = take((size_t)p.T * 2 * p.F * sizeof(bf16));
  p.A = take((size_t)p.T * p.F * sizeof(bf16));
  p.dA = p.dH = p.split = 0;
  p.split_dwd = p.split_dwgu = 1;
  if (pass == 1) {
    p.dA = take((size_t)p.T * p.F * sizeof(bf16));
    p.dH = take((size_t)p.T * 2 * p.F * sizeof(bf16));
    const int sms = num_sms();
    p.split_dwd = gemm_pick_split(p.d, p.F, p.T, sms);
    p.split_dwgu = gemm_pick_split(2 * (int64_t)p.F, p.d, p.T, sms);
    const size_t sb = std::max(gemm_split_scratch_bytes(p.d, p.F, p.split_dwd),
                               gemm_split_scratch_bytes(2 * (int64_t)p.F, p.d, p.split_dwgu));
    if (sb) p.split = take(sb);
  }
  p.total = off;
  return p;
}

// C[rows, N] (bf16, ld) = A[rows, K] B[N, K]^T with A, B plain row-major 2-D operands
TcGemmArgs gemm2d(int64_t M, int64_t N, int64_t K, TcOperand a, TcOperand b, void* out, int64_t ld, int epi) {
  TcGemmArgs g{};
  g.M = M; g.N = N; g.K = K;
  g.a = a; g.b = b;
  g.c.blk[0] = out; g.c.ld = ld; g.c.blk_shift = -1; g.c.blk_dim = 0;
  g.epi = epi;
  return g;
}

upipe_status_t run_mlp_fwd(const MlpPlan& p, const bf16* X, const bf16* Wgu, const bf16* Wd, bf16* Y, void* ws,
                           cudaStream_t st) {
  const int64_t F2 = 2 * (int64_t)p.F;
  bf16* H = at<bf16>(ws, p.H);
  bf16* A = at<bf16>(ws, p.A);
  for (int64_t r0 = 0, t = 0; r0 < p.S; r0 += p.T, ++t) {
    const int64_t rows = std::min(p.T, p.S - r0);
    {  // H = X_t [Wg; Wu]^T
      TcGemmArgs g = gemm2d(rows, F2, p.d, op2d(X + r0 * p.d, p.d, rows, p.d, 1), op2d(Wgu, p.d, F2, p.d, 1), H, F2,
                            EPI_STORE_BF16);
      Timed tm(UPIPE_K_MLP_GATE_UP, g.epi, g.M, g.N, g.K, 1, (int)t, st);
      UPIPE_CUDA(launch_gemm_tc(g, 1, nullptr, st));
    }
    {
      Timed tm(UPIPE_K_MLP_ACT, 0, rows * p.F, 1, 1, 1, (int)t, st);
      UPIPE_CUDA(launch_swiglu_fwd(H, A, rows, p.F, st));
    }
    {  // Y_t = A Wd^T
      TcGemmArgs g = gemm2d(rows, p.d, p.F, op2d(A, p.F, rows, p.F, 1), op2d(Wd, p.F, p.d, p.F, 1), Y + r0 * p.d, p.d,
                            EPI_STORE_BF16);
      Timed tm(UPIPE_K_MLP_DOWN, g.epi, g.M, g.N, g.K, 1, (int)t, st);
      UPIPE_CUDA(launch_gemm_tc(g, 1, nullptr, st));
    }
  }
  return UPIPE_OK;
}

upipe_status_t run_mlp_bwd(const MlpPlan& p, const bf16* X, const bf16* Wgu, const bf16* Wd, const bf16* dY, bf16* dX,
                           float* dWgu, float* dWd, void* ws, cudaStream_t st) {
  const int64_t F2 = 2 * (int64_t)p.F;
  bf16* H = at<bf16>(ws, p.H);
  bf16* A = at<bf16>(ws, p.A);
  bf16* dA = at<bf16>(ws, p.dA);
  bf16* dH = at<bf16>(ws, p.dH);
  float* split = p.split ? at<float>(ws, p.split) : nullptr;
  for (int64_t r0 = 0, t = 0; r0 < p.S; r0 += p.T, ++t) {
    const int64_t rows = std::min(p.T, p.S - r0);
    {  // recompute H = X_t [Wg; Wu]^T
      TcGemmArgs g = gemm2d(rows, F2, p.d, op2d(X + r0 * p.d, p.d, rows, p.d, 1), op2d(Wgu, p.d, F2, p.d, 1), H, F2,
                            EPI_STORE_BF16);
      Timed tm(UPIPE_K_MLP_GATE_UP, g.epi, g.M, g.N, g.K, 1, (int)t, st);
      UPIPE_CUDA(launch_gemm_tc(g, 1, nullptr, st));
    }
    {  // dA = dY_t Wd   (Wd read as [K = d][N = F])
      TcGemmArgs g = gemm2d(rows, p.F, p.d, op2d(dY + r0 * p.d, p.d, rows, p.d, 1), op2d(Wd, p.F, p.d, p.F, 0), dA,
                            p.F, EPI_STORE_BF16);
      Timed tm(UPIPE_K_MLP_DACT, g.epi, g.M, g.N, g.K, 1, (int)t, st);
      UPIPE_CUDA(launch_gemm_tc(g, 1, nullptr, st));
    }
    {
      Timed tm(UPIPE_K_MLP_ACT_BWD, 0, rows * p.F, 1, 1, 1, (int)t, st);
      UPIPE_CUDA(launch_swiglu_bwd(H, dA, A, dH, rows, p.F, st));
    }
    {  // dWd (+)= dY_t^T A
      TcGemmArgs g = gemm2d(p.d, p.F, rows, op2d(dY + r0 * p.d, p.d, rows, p.d, 0), op2d(A, p.F, rows, p.F, 0), dWd,
                            p.F, EPI_STORE_F32);
      Timed tm(UPIPE_K_MLP_DWD, t > 0 ? EPI_ACC_F32 : EPI_STORE_F32, g.M, g.N, g.K, p.split_dwd, (int)t, st);
      UPIPE_CUDA(block_weight_grad(g, t, p.split_dwd, split, st));
    }
    {  // dX_t = [dG | dU] [Wg; Wu]   (Wgu read as [K = 2F][N = d])
      TcGemmArgs g = gemm2d(rows, p.d, F2, op2d(dH, F2, rows, F2, 1), op2d(Wgu, p.d, F2, p.d, 0), dX + r0 * p.d, p.d,
                            EPI_STORE_BF16);
      Timed tm(UPIPE_K_MLP_DX, g.epi, g.M, g.N, g.K, 1, (int)t, st);
      UPIPE_CUDA(launch_gemm_tc(g, 1, nullptr, st));
    }
    {  // dWgu (+)= [dG | dU]^T X_t
      TcGemmArgs g = gemm2d(F2, p.d, rows, op2d(dH, F2, rows, F2, 0), op2d(X + r0 * p.d, p.d, rows, p.d, 0), dWgu,
                            p.d, EPI_STORE_F32);
      Timed tm(UPIPE_K_MLP_DWGU, t > 0 ? EPI_ACC_F32 : EPI_STORE_F32, g.M, g.N, g.K, p.split_dwgu, (int)t, st);
      UPIPE_CUDA(block_weight_grad(g, t, p.split_dwgu, split, st));
    }
  }
  return UPIPE_OK;
}

// Where a tensor of the offloaded entry points lives: page-locked host memory (staged), device
// memory (read in place), or neither (pageable host memory: rejected).
enum class Where { Host, Device, Invalid };
Where where_is(const void* ptr) {
  cudaPointerAttributes attr{};
  if (cudaPointerGetAttributes(&attr, ptr) != cudaSuccess) {
    cudaGetLastError();  // the failed query's error is not sticky: clear it
    return Where::Invalid;
  }
  if (attr.type == cudaMemoryTypeHost) return Where::Host;
  if (attr.type == cudaMemoryTypeDevice || attr.type == cudaMemoryTypeManaged) return Where::Device;
  return Where::Invalid;
}

upipe_status_t check_stage_rows(int64_t stage_rows) {
  if (stage_rows < 0 || (stage_rows > 0 && stage_rows % kTile != 0)) return UPIPE_ERR_INVALID_ARG;
  return UPIPE_OK;
}

}  // namespace
}  // namespace upipe

using namespace upipe;

extern "C" {

const char* upipe_attn_last_error_string(void) { return upipe::g_last_cuda_error; }

const char* upipe_attn_status_string(upipe_status_t s) {
  switch (s) {
    case UPIPE_OK: return "ok";
    case UPIPE_ERR_INVALID_ARG: return "invalid argument";
    case UPIPE_ERR_UNSUPPORTED: return "unsupported configuration";
    case UPIPE_ERR_ALIGNMENT: return "device pointer not 16-byte aligned";
    case UPIPE_ERR_WORKSPACE_TOO_SMALL: return "workspace or table buffer too small";
    case UPIPE_ERR_SEGMENTS_NOT_CONTIGUOUS: return "segment ids are not non-decreasing";
    case UPIPE_ERR_CUDA: return "CUDA runtime error";
    case UPIPE_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

upipe_status_t upipe_attn_workspace_size(const upipe_attn_desc_t* desc, int pass, size_t* bytes) {
  upipe_status_t s = check_desc(desc);
  if (s != UPIPE_OK) return s;
  if (!bytes || (pass != 0 && pass != 1)) return UPIPE_ERR_INVALID_ARG;
  *bytes = make_plan(desc, pass).total;
  return UPIPE_OK;
}

upipe_status_t upipe_attn_tile_table_size(const upipe_attn_desc_t* desc, size_t* bytes) {
  if (!desc || !bytes || desc->seq_len < 1 || desc->seq_len > INT32_MAX) return UPIPE_ERR_INVALID_ARG;
  *bytes = tile_table_bytes(desc->seq_len);
  return UPIPE_OK;
}

// Splash-style table of the tiles that are not fully masked (MaxText long-context article, Splash
// attention paragraph); optionally hands the visited-tile counts back to the host.
upipe_status_t upipe_attn_build_tile_table(const upipe_attn_desc_t* desc, const int32_t* seg, void* table,
                                           size_t table_bytes, int64_t* visited_counts_host, void* stream) {
  if (!desc || !table || desc->seq_len < 1 || desc->seq_len > INT32_MAX) return UPIPE_ERR_INVALID_ARG;
  if (desc->causal != 0 && desc->causal != 1) return UPIPE_ERR_INVALID_ARG;
  if (!aligned16(table) || (seg && !aligned16(seg))) return UPIPE_ERR_ALIGNMENT;
  if (table_bytes < tile_table_bytes(desc->seq_len)) return UPIPE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = (cudaStream_t)stream;
  UPIPE_CUDA(launch_tile_table(desc->seq_len, desc->causal, seg, table, st));
  if (visited_counts_host) {
    long long counts[2];
    UPIPE_CUDA(cudaMemcpyAsync(counts, table, sizeof(counts), cudaMemcpyDeviceToHost, st));
    UPIPE_CUDA(cudaStreamSynchronize(st));
    visited_counts_host[0] = counts[0];
    visited_counts_host[1] = counts[1];
  }
  return UPIPE_OK;
}

// The layer's forward, one chunk of query heads after another in one reused workspace ("Road to
// 5 Million Tokens" podcast summary, chapters "主要貢獻 UPipe" and "分批算 heads").
upipe_status_t upipe_attn_fwd(const upipe_attn_desc_t* desc, const uint16_t* X, const uint16_t* Wqkv, const uint16_t* Wo,
                              const int32_t* seg, uint16_t* Y, float* lse, void* ws, size_t ws_bytes, void* stream) {
  upipe_status_t s = check_desc(desc);
  if (s != UPIPE_OK) return s;
  if (!X || !Wqkv || !Wo || !Y || !lse || !ws) return UPIPE_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(Wqkv) || !aligned16(Wo) || !aligned16(Y) || !aligned16(lse) || !aligned16(ws) ||
      (seg && !aligned16(seg)))
    return UPIPE_ERR_ALIGNMENT;
  const Plan p = make_plan(desc, 0);
  if (ws_bytes < p.total) return UPIPE_ERR_WORKSPACE_TOO_SMALL;
  return run_fwd(p, reinterpret_cast<const bf16*>(X), reinterpret_cast<const bf16*>(Wqkv),
                 reinterpret_cast<const bf16*>(Wo), seg, reinterpret_cast<bf16*>(Y), lse, ws, (cudaStream_t)stream);
}

// The layer's backward, chunk by chunk, recomputing each chunk's activations from X and lse
// (same summary, chapter "Activation checkpointing").
upipe_status_t upipe_attn_bwd(const upipe_attn_desc_t* desc, const uint16_t* X, const uint16_t* Wqkv, const uint16_t* Wo,
                              const int32_t* seg, const uint16_t* dY, const float* lse, uint16_t* dX, float* dWqkv,
                              float* dWo, void* ws, size_t ws_bytes, void* stream) {
  upipe_status_t s = check_desc(desc);
  if (s != UPIPE_OK) return s;
  if (!X || !Wqkv || !Wo || !dY || !lse || !dX || !dWqkv || !dWo || !ws) return UPIPE_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(Wqkv) || !aligned16(Wo) || !aligned16(dY) || !aligned16(lse) || !aligned16(dX) ||
      !aligned16(dWqkv) || !aligned16(dWo) || !aligned16(ws) || (seg && !aligned16(seg)))
    return UPIPE_ERR_ALIGNMENT;
  const Plan p = make_plan(desc, 1);
  if (ws_bytes < p.total) return UPIPE_ERR_WORKSPACE_TOO_SMALL;
  return run_bwd(p, reinterpret_cast<const bf16*>(X), reinterpret_cast<const bf16*>(Wqkv),
                 reinterpret_cast<const bf16*>(Wo), seg, reinterpret_cast<const bf16*>(dY), lse,
                 reinterpret_cast<bf16*>(dX), dWqkv, dWo, ws, (cudaStream_t)stream);
}

static upipe_status_t check_core(const upipe_attn_desc_t* desc) {
  if (!desc || desc->seq_len < 1 || desc->seq_len > INT32_MAX || desc->n_q_heads <= 0 || desc->n_kv_heads <= 0 ||
      desc->n_q_heads % desc->n_kv_heads != 0 || (desc->causal != 0 && desc->causal != 1))
    return UPIPE_ERR_INVALID_ARG;
  if (desc->head_dim != 64 && desc->head_dim != 128) return UPIPE_ERR_UNSUPPORTED;
  return UPIPE_OK;
}

static AttnArgs core_args(const upipe_attn_desc_t* desc, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                          const int32_t* seg, void* table) {
  AttnArgs a{};
  a.q = reinterpret_cast<const bf16*>(q);
  a.k = reinterpret_cast<const bf16*>(k);
  a.v = reinterpret_cast<const bf16*>(v);
  a.seg = seg;
  a.q_rows = table_q_rows(table);
  a.kv_rows = table_kv_rows(table, desc->seq_len);
  a.q_order = table_q_order(table, desc->seq_len);
  a.kv_order = table_kv_order(table, desc->seq_len);
  a.S = desc->seq_len;
  a.nh = desc->n_q_heads;
  a.nkv = desc->n_kv_heads;
  a.g = desc->n_q_heads / desc->n_kv_heads;
  a.causal = desc->causal;
  a.scale = desc->softmax_scale > 0.f ? desc->softmax_scale : 1.0f / std::sqrt((float)desc->head_dim);
  a.err = &reinterpret_cast<TableHeader*>(table)->error;
  return a;
}

// Flash-style attention forward over whole heads (podcast summary, chapter "DeepSpeed Ulysses").
upipe_status_t upipe_attn_core_fwd(const upipe_attn_desc_t* desc, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                   const int32_t* seg, void* table, uint16_t* o, float* lse, void* stream) {
  upipe_status_t s = check_core(desc);
  if (s != UPIPE_OK) return s;
  if (!q || !k || !v || !table || !o || !lse) return UPIPE_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(table) || !aligned16(o) || !aligned16(lse))
    return UPIPE_ERR_ALIGNMENT;
  AttnArgs a = core_args(desc, q, k, v, seg, table);
  a.o = reinterpret_cast<bf16*>(o);
  a.lse = lse;
  return cuda_status(launch_attn_fwd(a, desc->head_dim, (cudaStream_t)stream));
}

// O and D recomputed from the saved lse (podcast summary, chapter "Activation checkpointing").
upipe_status_t upipe_attn_core_recompute(const upipe_attn_desc_t* desc, const uint16_t* q, const uint16_t* k,
                                         const uint16_t* v, const uint16_t* dO, const float* lse, const int32_t* seg,
                                         void* table, uint16_t* o, float* D, void* stream) {
  upipe_status_t s = check_core(desc);
  if (s != UPIPE_OK) return s;
  if (!q || !k || !v || !dO || !lse || !table || !o || !D) return UPIPE_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(lse) || !aligned16(table) ||
      !aligned16(o) || !aligned16(D))
    return UPIPE_ERR_ALIGNMENT;
  AttnArgs a = core_args(desc, q, k, v, seg, table);
  a.lse = const_cast<float*>(lse);
  a.dO = reinterpret_cast<const bf16*>(dO);
  a.D = D;
  a.o = reinterpret_cast<bf16*>(o);
  return cuda_status(launch_attn_recompute(a, desc->head_dim, (cudaStream_t)stream));
}

static upipe_status_t core_bwd_common(const upipe_attn_desc_t* desc, const uint16_t* q, const uint16_t* k,
                                      const uint16_t* v, const uint16_t* dO, const float* lse, const float* D,
                                      const int32_t* seg, void* table, AttnBwdArgs* b) {
  upipe_status_t s = check_core(desc);
  if (s != UPIPE_OK) return s;
  if (!q || !k || !v || !dO || !lse || !D || !table) return UPIPE_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(lse) || !aligned16(D) ||
      !aligned16(table))
    return UPIPE_ERR_ALIGNMENT;
  *b = AttnBwdArgs{};
  b->f = core_args(desc, q, k, v, seg, table);
  b->f.lse = const_cast<float*>(lse);
  b->f.dO = reinterpret_cast<const bf16*>(dO);
  b->f.D = const_cast<float*>(D);
  b->nkv = desc->n_kv_heads;
  return UPIPE_OK;
}

// dQ of the attention backward (chain rule of the same softmax; recompute as above).
upipe_status_t upipe_attn_core_bwd_dq(const upipe_attn_desc_t* desc, const uint16_t* q, const uint16_t* k,
                                      const uint16_t* v, const uint16_t* dO, const float* lse, const float* D,
                                      const int32_t* seg, void* table, uint16_t* dq, void* stream) {
  AttnBwdArgs b;
  upipe_status_t s = core_bwd_common(desc, q, k, v, dO, lse, D, seg, table, &b);
  if (s != UPIPE_OK) return s;
  if (!dq) return UPIPE_ERR_INVALID_ARG;
  if (!aligned16(dq)) return UPIPE_ERR_ALIGNMENT;
  b.dq = reinterpret_cast<bf16*>(dq);
  return cuda_status(launch_attn_bwd_dq(b, desc->head_dim, (cudaStream_t)stream));
}

// dK, dV with the GQA heads of each KV head summed (MaxText article, Splash paragraph: GQA).
upipe_status_t upipe_attn_core_bwd_dkdv(const upipe_attn_desc_t* desc, const uint16_t* q, const uint16_t* k,
                                        const uint16_t* v, const uint16_t* dO, const float* lse, const float* D,
                                        const int32_t* seg, void* table, uint16_t* dk, uint16_t* dv,
                                        void* stream) {
  AttnBwdArgs b;
  upipe_status_t s = core_bwd_common(desc, q, k, v, dO, lse, D, seg, table, &b);
  if (s != UPIPE_OK) return s;
  if (!dk || !dv) return UPIPE_ERR_INVALID_ARG;
  if (!aligned16(dk) || !aligned16(dv)) return UPIPE_ERR_ALIGNMENT;
  b.dk = reinterpret_cast<bf16*>(dk);
  b.dv = reinterpret_cast<bf16*>(dv);
  return cuda_status(launch_attn_bwd_dkdv(b, desc->head_dim, (cudaStream_t)stream));
}

// The same into fp32 sums, flushed in windows (the layer's launch for partial KV groups and long
// key tiles).
upipe_status_t upipe_attn_core_bwd_dkdv_acc(const upipe_attn_desc_t* desc, const uint16_t* q, const uint16_t* k,
                                            const uint16_t* v, const uint16_t* dO, const float* lse,
                                            const float* D, const int32_t* seg, void* table, float* dk_acc,
                                            float* dv_acc, uint16_t* dk, uint16_t* dv, void* stream) {
  AttnBwdArgs b;
  upipe_status_t s = core_bwd_common(desc, q, k, v, dO, lse, D, seg, table, &b);
  if (s != UPIPE_OK) return s;
  if (!dk_acc || !dv_acc || (!dk) != (!dv)) return UPIPE_ERR_INVALID_ARG;
  if (!aligned16(dk_acc) || !aligned16(dv_acc) || (dk && (!aligned16(dk) || !aligned16(dv))))
    return UPIPE_ERR_ALIGNMENT;
  b.acc_kv = 1;
  b.flush_items = dkdv_window();
  b.dk_acc = dk_acc;
  b.dv_acc = dv_acc;
  b.dk_out = reinterpret_cast<bf16*>(dk);
  b.dv_out = reinterpret_cast<bf16*>(dv);
  return cuda_status(launch_attn_bwd_dkdv(b, desc->head_dim, (cudaStream_t)stream));
}

upipe_status_t upipe_attn_gemm_nt(int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda, const uint16_t* B,
                                  int64_t ldb, float* C, int64_t ldc, void* stream) {
  if (M <= 0 || N <= 0 || K <= 0 || !A || !B || !C || lda < K || ldb < K || ldc < N) return UPIPE_ERR_INVALID_ARG;
  if (K % 8 || N % 8 || lda % 8 || ldb % 8 || ldc % 4) return UPIPE_ERR_UNSUPPORTED;
  if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return UPIPE_ERR_ALIGNMENT;
  TcGemmArgs g{};
  g.M = M; g.N = N; g.K = K;
  g.a = op2d(A, K, M, lda, 1);
  g.b = op2d(B, K, N, ldb, 1);
  g.c.blk[0] = C; g.c.ld = ldc; g.c.blk_shift = -1;
  g.epi = EPI_STORE_F32;
  return cuda_status(launch_gemm_tc(g, 1, nullptr, (cudaStream_t)stream));
}

upipe_status_t upipe_attn_lse_merge(int64_t rows, int32_t head_dim, const uint16_t* O_b, const float* lse_b,
                                    float* O_acc, float* lse_acc, uint16_t* O_out, void* stream) {
  if (rows < 0 || !O_b || !lse_b || !O_acc || !lse_acc) return UPIPE_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return UPIPE_ERR_UNSUPPORTED;
  if (!aligned16(O_b) || !aligned16(lse_b) || !aligned16(O_acc) || !aligned16(lse_acc) || (O_out && !aligned16(O_out)))
    return UPIPE_ERR_ALIGNMENT;
  return cuda_status(launch_lse_merge(rows, head_dim, reinterpret_cast<const bf16*>(O_b), lse_b, O_acc, lse_acc,
                                      reinterpret_cast<bf16*>(O_out), (cudaStream_t)stream));
}

upipe_status_t upipe_attn_ring_bwd_prep(int32_t n_heads, int64_t seq_len, int32_t head_dim, const uint16_t* O,
                                        const uint16_t* dO, const float* lse, float* D, void* stream) {
  if (n_heads <= 0 || seq_len < 1 || seq_len > INT32_MAX || !O || !dO || !lse || !D) return UPIPE_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return UPIPE_ERR_UNSUPPORTED;
  if (!aligned16(O) || !aligned16(dO) || !aligned16(lse) || !aligned16(D)) return UPIPE_ERR_ALIGNMENT;
  return cuda_status(launch_ring_bwd_prep(n_heads, seq_len, head_dim, reinterpret_cast<const bf16*>(O),
                                          reinterpret_cast<const bf16*>(dO), lse, D, (cudaStream_t)stream));
}

upipe_status_t upipe_attn_accumulate(int64_t n, const uint16_t* src, float* acc, uint16_t* out, void* stream) {
  if (n < 0 || !src || !acc) return UPIPE_ERR_INVALID_ARG;
  if (!aligned16(src) || !aligned16(acc) || (out && !aligned16(out))) return UPIPE_ERR_ALIGNMENT;
  return cuda_status(launch_accumulate(n, reinterpret_cast<const bf16*>(src), acc, reinterpret_cast<bf16*>(out),
                                       (cudaStream_t)stream));
}

// ------------------------------------------------------------------------------------------------
// Ring (P2P) steps (MaxText article, strategy table row "P2P (Ring)" and the paragraph on causal
// load balancing): the zigzag shards of dev_count devices against the visiting key/value shards,
// one launch per step and pass kernel, accumulating in fp32.
// ------------------------------------------------------------------------------------------------
static upipe_status_t check_ring(const upipe_ring_desc_t* d) {
  if (!d || d->ring_size < 1 || d->chunk_len < 1 || 2 * d->chunk_len > INT32_MAX || d->n_q_heads <= 0 ||
      d->n_kv_heads <= 0 || d->n_q_heads % d->n_kv_heads != 0 || (d->causal != 0 && d->causal != 1))
    return UPIPE_ERR_INVALID_ARG;
  if (d->dev_first < 0 || d->dev_count < 1 || d->dev_first + d->dev_count > d->ring_size) return UPIPE_ERR_INVALID_ARG;
  if (d->kv_count != d->ring_size && d->kv_count != d->dev_count) return UPIPE_ERR_INVALID_ARG;
  if (d->head_dim != 64 && d->head_dim != 128) return UPIPE_ERR_UNSUPPORTED;
  // the launches' second grid dimension runs over the query-tile pairs of all batched devices
  // (forward, dQ) and over the key tiles of all shards (dK/dV)
  const int64_t nt = ceil_div(2 * d->chunk_len, kTile);
  if ((int64_t)d->dev_count * ceil_div(nt, 2) > 65535 || (int64_t)d->kv_count * nt > 65535) return UPIPE_ERR_UNSUPPORTED;
  return UPIPE_OK;
}

// Geometry of step `step`: k/v hold every shard in device order (kv0 = 0) or the visiting ones in
// batch order (kv0 = the owner of the first batched device's visitor).
static RingGeom ring_geom(const upipe_ring_desc_t* d, int step) {
  RingGeom g{};
  g.P = d->ring_size;
  g.r0 = d->dev_first;
  g.step = step;
  g.kv0 = d->kv_count == d->ring_size ? 0 : ((d->dev_first - step) % d->ring_size + d->ring_size) % d->ring_size;
  g.C = d->chunk_len;
  return g;
}

static size_t ring_table_bytes(const upipe_ring_desc_t* d) {
  return tile_table_bytes(2 * d->chunk_len, d->dev_count, d->kv_count);
}

upipe_status_t upipe_attn_ring_tables_size(const upipe_ring_desc_t* desc, size_t* bytes) {
  upipe_status_t s = check_ring(desc);
  if (s != UPIPE_OK) return s;
  if (!bytes) return UPIPE_ERR_INVALID_ARG;
  *bytes = (size_t)desc->ring_size * ring_table_bytes(desc);
  return UPIPE_OK;
}

upipe_status_t upipe_attn_ring_build_tables(const upipe_ring_desc_t* desc, const int32_t* seg, void* tables,
                                            size_t bytes, void* stream) {
  upipe_status_t s = check_ring(desc);
  if (s != UPIPE_OK) return s;
  if (!tables) return UPIPE_ERR_INVALID_ARG;
  if (!aligned16(tables) || (seg && !aligned16(seg))) return UPIPE_ERR_ALIGNMENT;
  const size_t per = ring_table_bytes(desc);
  if (bytes < per * desc->ring_size) return UPIPE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = (cudaStream_t)stream;
  for (int step = 0; step < desc->ring_size; ++step) {
    Timed t(UPIPE_K_TILE_TABLE, 0, 2 * desc->chunk_len, 0, 0, 1, -1, st);
    UPIPE_CUDA(launch_ring_table(2 * desc->chunk_len, desc->causal, seg, ring_geom(desc, step), desc->dev_count,
                                 desc->kv_count, at<char>(tables, per * step), st));
  }
  return UPIPE_OK;
}

static AttnArgs ring_args(const upipe_ring_desc_t* d, int step, const uint16_t* q, const uint16_t* k,
                          const uint16_t* v, const int32_t* seg, void* tables) {
  const size_t per = ring_table_bytes(d);
  void* table = at<char>(tables, per * step);
  const int64_t S = 2 * d->chunk_len;
  AttnArgs a{};
  a.q = reinterpret_cast<const bf16*>(q);
  a.k = reinterpret_cast<const bf16*>(k);
  a.v = reinterpret_cast<const bf16*>(v);
  a.seg = seg;
  a.q_rows = table_q_rows(table);
  a.kv_rows = table_kv_rows(table, S, d->dev_count);
  a.q_order = table_q_order(table, S, d->dev_count, d->kv_count);
  a.kv_order = table_kv_order(table, S, d->dev_count, d->kv_count);
  a.S = S;
  a.nh = d->dev_count * d->n_q_heads;
  a.nkv = d->kv_count * d->n_kv_heads;
  a.g = d->n_q_heads / d->n_kv_heads;
  a.hq = d->n_q_heads;
  a.hkv = d->n_kv_heads;
  a.ndev = d->dev_count;
  a.kv_count = d->kv_count;
  a.causal = d->causal;
  a.scale = d->softmax_scale > 0.f ? d->softmax_scale : 1.0f / std::sqrt((float)d->head_dim);
  a.err = &reinterpret_cast<TableHeader*>(tables)->error;  // every step reports into the first table
  a.ring = ring_geom(d, step);
  a.acc_first = step == 0;
  a.acc_last = step == d->ring_size - 1;
  a.ring_tables = reinterpret_cast<const char*>(tables);
  a.ring_table_stride = per;
  a.kv_last_touch = d->dev_count == d->ring_size && d->kv_count == d->ring_size;
  return a;
}

static upipe_status_t ring_fwd_checks(const upipe_ring_desc_t* desc, const uint16_t* q, const uint16_t* k,
                                      const uint16_t* v, const int32_t* seg, void* tables, float* o_acc, float* lse,
                                      uint16_t* o) {
  upipe_status_t s = check_ring(desc);
  if (s != UPIPE_OK) return s;
  if (!q || !k || !v || !tables || !o_acc || !lse) return UPIPE_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(tables) || !aligned16(o_acc) || !aligned16(lse) ||
      (o && !aligned16(o)) || (seg && !aligned16(seg)))
    return UPIPE_ERR_ALIGNMENT;
  return UPIPE_OK;
}

static upipe_status_t ring_fwd_launch(const upipe_ring_desc_t* desc, int step, bool chained, const uint16_t* q,
                                      const uint16_t* k, const uint16_t* v, const int32_t* seg, void* tables,
                                      float* o_acc, float* lse, uint16_t* o, cudaStream_t st) {
  AttnArgs a = ring_args(desc, step, q, k, v, seg, tables);
  a.o_acc = o_acc;
  a.lse = lse;
  a.o = reinterpret_cast<bf16*>(o);
  a.pdl = chained;
  Timed t(UPIPE_K_RING_FWD, 0, a.S, a.nh, desc->head_dim, 1, step, st);
  return cuda_status(launch_attn_ring_fwd(a, desc->head_dim, st));
}

upipe_status_t upipe_attn_ring_fwd_step(const upipe_ring_desc_t* desc, int32_t step, const uint16_t* q,
                                        const uint16_t* k, const uint16_t* v, const int32_t* seg, void* tables,
                                        float* o_acc, float* lse, uint16_t* o, void* stream) {
  upipe_status_t s = ring_fwd_checks(desc, q, k, v, seg, tables, o_acc, lse, o);
  if (s != UPIPE_OK) return s;
  if (step < 0 || step >= desc->ring_size) return UPIPE_ERR_INVALID_ARG;
  return ring_fwd_launch(desc, step, false, q, k, v, seg, tables, o_acc, lse, o, (cudaStream_t)stream);
}

upipe_status_t upipe_attn_ring_fwd(const upipe_ring_desc_t* desc, const uint16_t* q, const uint16_t* k,
                                   const uint16_t* v, const int32_t* seg, void* tables, float* o_acc, float* lse,
                                   uint16_t* o, void* stream) {
  upipe_status_t s = ring_fwd_checks(desc, q, k, v, seg, tables, o_acc, lse, o);
  if (s != UPIPE_OK) return s;
  // timing events between the launches would break the chain: chain only while timing is off
  const bool chain = !g_timing_on.load(std::memory_order_relaxed);
  for (int step = 0; step < desc->ring_size; ++step) {
    s = ring_fwd_launch(desc, step, chain && step > 0, q, k, v, seg, tables, o_acc, lse, o, (cudaStream_t)stream);
    if (s != UPIPE_OK) return s;
  }
  return UPIPE_OK;
}

static upipe_status_t ring_bwd_checks(const upipe_ring_desc_t* desc, const uint16_t* q, const uint16_t* k,
                                      const uint16_t* v, const uint16_t* dO, const float* D, const int32_t* seg,
                                      void* tables, float* dq_acc, float* dk_acc, float* dv_acc, uint16_t* dq,
                                      uint16_t* dk, uint16_t* dv) {
  upipe_status_t s = check_ring(desc);
  if (s != UPIPE_OK) return s;
  if (!q || !k || !v || !dO || !D || !tables || !dq_acc || !dk_acc || !dv_acc) return UPIPE_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(D) || !aligned16(tables) ||
      !aligned16(dq_acc) || !aligned16(dk_acc) || !aligned16(dv_acc) || (dq && !aligned16(dq)) ||
      (dk && !aligned16(dk)) || (dv && !aligned16(dv)) || (seg && !aligned16(seg)))
    return UPIPE_ERR_ALIGNMENT;
  return UPIPE_OK;
}

// dQ then dK/dV of one step.  dq_chained: the previous kernel on the stream is the previous step's
// dK/dV launch; kv_chained: chain the dK/dV launch to this step's dQ launch, which it follows
// directly and whose output it does not read (it still waits for it before its epilogue, so it
// never completes first).
static upipe_status_t ring_bwd_launch(const upipe_ring_desc_t* desc, int step, bool dq_chained, bool kv_chained,
                                      const uint16_t* q,
                                      const uint16_t* k, const uint16_t* v, const uint16_t* dO, const float* D,
                                      const int32_t* seg, void* tables, float* dq_acc, float* dk_acc, float* dv_acc,
                                      uint16_t* dq, uint16_t* dk, uint16_t* dv, cudaStream_t st) {
  AttnBwdArgs b{};
  b.f = ring_args(desc, step, q, k, v, seg, tables);
  b.f.dO = reinterpret_cast<const bf16*>(dO);
  b.f.D = const_cast<float*>(D);
  b.nkv = b.f.nkv;
  b.dq_acc = dq_acc;
  b.dq = reinterpret_cast<bf16*>(dq);
  b.acc_kv = 1;
  b.flush_items = dkdv_window();
  b.dk_acc = dk_acc;
  b.dv_acc = dv_acc;
  b.dk_out = reinterpret_cast<bf16*>(dk);
  b.dv_out = reinterpret_cast<bf16*>(dv);
  {
    b.f.pdl = dq_chained;
    Timed t(UPIPE_K_RING_DQ, 0, b.f.S, b.f.nh, desc->head_dim, 1, step, st);
    UPIPE_CUDA(launch_attn_bwd_dq(b, desc->head_dim, st));
  }
  b.f.pdl = kv_chained;
  Timed t(UPIPE_K_RING_DKDV, 0, b.f.S, b.f.nh, desc->head_dim, 1, step, st);
  return cuda_status(launch_attn_bwd_dkdv(b, desc->head_dim, st));
}

upipe_status_t upipe_attn_ring_bwd_step(const upipe_ring_desc_t* desc, int32_t step, const uint16_t* q,
                                        const uint16_t* k, const uint16_t* v, const uint16_t* dO, const float* D,
                                        const int32_t* seg, void* tables, float* dq_acc, float* dk_acc,
                                        float* dv_acc, uint16_t* dq, uint16_t* dk, uint16_t* dv, void* stream) {
  upipe_status_t s = ring_bwd_checks(desc, q, k, v, dO, D, seg, tables, dq_acc, dk_acc, dv_acc, dq, dk, dv);
  if (s != UPIPE_OK) return s;
  if (step < 0 || step >= desc->ring_size) return UPIPE_ERR_INVALID_ARG;
  // timing events between the launches would break a chain: chain only while timing is off
  const bool chain = !g_timing_on.load(std::memory_order_relaxed);
  return ring_bwd_launch(desc, step, false, chain, q, k, v, dO, D, seg, tables, dq_acc, dk_acc, dv_acc, dq, dk, dv,
                         (cudaStream_t)stream);
}

upipe_status_t upipe_attn_ring_bwd(const upipe_ring_desc_t* desc, const uint16_t* q, const uint16_t* k,
                                   const uint16_t* v, const uint16_t* o, const uint16_t* dO, const float* lse,
                                   const int32_t* seg, void* tables, float* D, float* dq_acc, float* dk_acc,
                                   float* dv_acc, uint16_t* dq, uint16_t* dk, uint16_t* dv, void* stream) {
  upipe_status_t s = ring_bwd_checks(desc, q, k, v, dO, D, seg, tables, dq_acc, dk_acc, dv_acc, dq, dk, dv);
  if (s != UPIPE_OK) return s;
  if (!o || !lse) return UPIPE_ERR_INVALID_ARG;
  if (!aligned16(o) || !aligned16(lse)) return UPIPE_ERR_ALIGNMENT;
  cudaStream_t st = (cudaStream_t)stream;
  UPIPE_CUDA(launch_ring_bwd_prep(desc->dev_count * desc->n_q_heads, 2 * desc->chunk_len, desc->head_dim,
                                  reinterpret_cast<const bf16*>(o), reinterpret_cast<const bf16*>(dO), lse, D, st));
  const bool chain = !g_timing_on.load(std::memory_order_relaxed);
  for (int step = 0; step < desc->ring_size; ++step) {
    // the first dQ launch follows the prep kernel, whose D it reads: not chained
    s = ring_bwd_launch(desc, step, chain && step > 0, chain, q, k, v, dO, D, seg, tables, dq_acc, dk_acc, dv_acc,
                        dq, dk, dv, st);
    if (s != UPIPE_OK) return s;
  }
  return UPIPE_OK;
}

uint64_t upipe_attn_launch_count(void) { return upipe::g_launch_count.load(std::memory_order_relaxed); }

// Error word of a workspace or table header (bounded device waits, segment order check).
upipe_status_t upipe_attn_device_status(const void* buf, int32_t* code, void* stream) {
  if (!buf || !code) return UPIPE_ERR_INVALID_ARG;
  int32_t v = 0;
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(&v, reinterpret_cast<const char*>(buf) + offsetof(TableHeader, error), sizeof(v),
                                  cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_status(e);
  *code = v;
  return UPIPE_OK;
}

upipe_status_t upipe_attn_workspace_size_offload(const upipe_attn_desc_t* desc, int pass, int64_t stage_rows,
                                                 size_t* bytes) {
  upipe_status_t s = check_desc(desc);
  if (s != UPIPE_OK) return s;
  if (!bytes || (pass != 0 && pass != 1)) return UPIPE_ERR_INVALID_ARG;
  if ((s = check_stage_rows(stage_rows)) != UPIPE_OK) return s;
  *bytes = make_plan(desc, pass, stage_rows ? stage_rows : kDefaultStageRows).total;
  return UPIPE_OK;
}

// The layer's forward with X in host memory (CPU offload of the inputs: podcast summary, chapter
// on offloading inputs to the CPU; transcript, implementation plan step 2).
upipe_status_t upipe_attn_fwd_offload(const upipe_attn_desc_t* desc, const uint16_t* X_host, const uint16_t* Wqkv,
                                      const uint16_t* Wo, const int32_t* seg, uint16_t* Y, float* lse, void* ws,
                                      size_t ws_bytes, int64_t stage_rows, void* stream) {
  upipe_status_t s = check_desc(desc);
  if (s != UPIPE_OK) return s;
  if ((s = check_stage_rows(stage_rows)) != UPIPE_OK) return s;
  if (!X_host || !Wqkv || !Wo || !Y || !lse || !ws) return UPIPE_ERR_INVALID_ARG;
  if (!aligned16(X_host) || !aligned16(Wqkv) || !aligned16(Wo) || !aligned16(Y) || !aligned16(lse) || !aligned16(ws) ||
      (seg && !aligned16(seg)))
    return UPIPE_ERR_ALIGNMENT;
  const Plan p = make_plan(desc, 0, stage_rows ? stage_rows : kDefaultStageRows);
  if (ws_bytes < p.total) return UPIPE_ERR_WORKSPACE_TOO_SMALL;
  const Where wx = where_is(X_host);
  if (wx == Where::Invalid) return UPIPE_ERR_INVALID_ARG;
  return run_fwd_offload(p, reinterpret_cast<const bf16*>(X_host), wx == Where::Host, reinterpret_cast<const bf16*>(Wqkv),
                         reinterpret_cast<const bf16*>(Wo), seg, reinterpret_cast<bf16*>(Y), lse, ws,
                         (cudaStream_t)stream);
}

// The layer's backward with X and dY in host memory (same passages).
upipe_status_t upipe_attn_bwd_offload(const upipe_attn_desc_t* desc, const uint16_t* X_host, const uint16_t* Wqkv,
                                      const uint16_t* Wo, const int32_t* seg, const uint16_t* dY_host, const float* lse,
                                      uint16_t* dX, float* dWqkv, float* dWo, void* ws, size_t ws_bytes,
                                      int64_t stage_rows, void* stream) {
  upipe_status_t s = check_desc(desc);
  if (s != UPIPE_OK) return s;
  if ((s = check_stage_rows(stage_rows)) != UPIPE_OK) return s;
  if (!X_host || !Wqkv || !Wo || !dY_host || !lse || !dX || !dWqkv || !dWo || !ws) return UPIPE_ERR_INVALID_ARG;
  if (!aligned16(X_host) || !aligned16(Wqkv) || !aligned16(Wo) || !aligned16(dY_host) || !aligned16(lse) ||
      !aligned16(dX) || !aligned16(dWqkv) || !aligned16(dWo) || !aligned16(ws) || (seg && !aligned16(seg)))
    return UPIPE_ERR_ALIGNMENT;
  const Plan p = make_plan(desc, 1, stage_rows ? stage_rows : kDefaultStageRows);
  if (ws_bytes < p.total) return UPIPE_ERR_WORKSPACE_TOO_SMALL;
  const Where wx = where_is(X_host), wdy = where_is(dY_host);
  if (wx == Where::Invalid || wdy == Where::Invalid) return UPIPE_ERR_INVALID_ARG;
  return run_bwd_offload(p, reinterpret_cast<const bf16*>(X_host), wx == Where::Host, reinterpret_cast<const bf16*>(Wqkv),
                         reinterpret_cast<const bf16*>(Wo), seg, reinterpret_cast<const bf16*>(dY_host),
                         wdy == Where::Host, lse, reinterpret_cast<bf16*>(dX), dWqkv, dWo, ws, (cudaStream_t)stream);
}

upipe_status_t upipe_mlp_workspace_size(const upipe_mlp_desc_t* desc, int pass, size_t* bytes) {
  upipe_status_t s = check_mlp(desc);
  if (s != UPIPE_OK) return s;
  if (!bytes || (pass != 0 && pass != 1)) return UPIPE_ERR_INVALID_ARG;
  *bytes = make_mlp_plan(desc, pass).total;
  return UPIPE_OK;
}

// The feed-forward step in sequence tiles (podcast summary, chapter on sequence tiling; transcript,
// Полезные советы: the MLP computed in pieces).
upipe_status_t upipe_mlp_fwd(const upipe_mlp_desc_t* desc, const uint16_t* X, const uint16_t* Wgu, const uint16_t* Wd,
                             uint16_t* Y, void* ws, size_t ws_bytes, void* stream) {
  upipe_status_t s = check_mlp(desc);
  if (s != UPIPE_OK) return s;
  if (!X || !Wgu || !Wd || !Y || !ws) return UPIPE_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(Wgu) || !aligned16(Wd) || !aligned16(Y) || !aligned16(ws)) return UPIPE_ERR_ALIGNMENT;
  const MlpPlan p = make_mlp_plan(desc, 0);
  if (ws_bytes < p.total) return UPIPE_ERR_WORKSPACE_TOO_SMALL;
  return run_mlp_fwd(p, reinterpret_cast<const bf16*>(X), reinterpret_cast<const bf16*>(Wgu),
                     reinterpret_cast<const bf16*>(Wd), reinterpret_cast<bf16*>(Y), ws, (cudaStream_t)stream);
}

upipe_status_t upipe_mlp_bwd(const upipe_mlp_desc_t* desc, const uint16_t* X, const uint16_t* Wgu, const uint16_t* Wd,
                             const uint16_t* dY, uint16_t* dX, float* dWgu, float* dWd, void* ws, size_t ws_bytes,
                             void* stream) {
  upipe_status_t s = check_mlp(desc);
  if (s != UPIPE_OK) return s;
  if (!X || !Wgu || !Wd || !dY || !dX || !dWgu || !dWd || !ws) return UPIPE_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(Wgu) || !aligned16(Wd) || !aligned16(dY) || !aligned16(dX) || !aligned16(dWgu) ||
      !aligned16(dWd) || !aligned16(ws))
    return UPIPE_ERR_ALIGNMENT;
  const MlpPlan p = make_mlp_plan(desc, 1);
  if (ws_bytes < p.total) return UPIPE_ERR_WORKSPACE_TOO_SMALL;
  return run_mlp_bwd(p, reinterpret_cast<const bf16*>(X), reinterpret_cast<const bf16*>(Wgu),
                     reinterpret_cast<const bf16*>(Wd), reinterpret_cast<const bf16*>(dY), reinterpret_cast<bf16*>(dX),
                     dWgu, dWd, ws, (cudaStream_t)stream);
}

upipe_status_t upipe_attn_timing_enable(int32_t on) {
  if (on != 0 && on != 1) return UPIPE_ERR_INVALID_ARG;
  g_timing_on.store(on, std::memory_order_relaxed);
  return UPIPE_OK;
}

upipe_status_t upipe_attn_timing_collect(upipe_attn_timing_t* out, int32_t cap, int32_t* n) {
  if (!n || cap < 0 || (cap > 0 && !out)) return UPIPE_ERR_INVALID_ARG;
  std::vector<TimingRec> recs;
  {
    std::lock_guard<std::mutex> lock(g_timing_mutex);
    recs.swap(g_timing);
  }
  upipe_status_t status = UPIPE_OK;
  int32_t k = 0;
  for (const TimingRec& r : recs) {
    float ms = -1.f, start = -1.f;
    cudaError_t e = cudaEventSynchronize(r.e1);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.e0, r.e1);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&start, recs.front().e0, r.e0);
    if (e != cudaSuccess && status == UPIPE_OK) status = cuda_status(e);
    if (k < cap) {
      upipe_attn_timing_t& o = out[k];
      o.kind = r.kind; o.epilogue = r.epi; o.split_k = r.split_k; o.chunk = r.chunk;
      o.m = r.m; o.n = r.n; o.k = r.k; o.ms = ms; o.start_ms = start;
    }
    ++k;
  }
  for (const TimingRec& r : recs) {
    cudaEventDestroy(r.e0);
    cudaEventDestroy(r.e1);
  }
  *n = k;
  return status;
}

upipe_status_t upipe_attn_set_dkdv_window(int32_t items) {
  if (items < 0 || (items && (items < 2 || items % 2 || items > (1 << 24)))) return UPIPE_ERR_INVALID_ARG;
  g_dkdv_window.store(items ? items : kDkvWindowDefault, std::memory_order_relaxed);
  return UPIPE_OK;
}

upipe_status_t upipe_attn_set_wait_limit_ns(uint64_t ns) {
  if (ns > kMaxWaitLimitNs) return UPIPE_ERR_INVALID_ARG;
  g_wait_limit_ns.store(ns ? ns : tc_wait_default_ns, std::memory_order_relaxed);
  return UPIPE_OK;
}

upipe_status_t upipe_attn_wait_probe(void* buf, size_t bytes, int32_t arrive, void* stream) {
  if (!buf || bytes < sizeof(TableHeader) || (arrive != 0 && arrive != 1)) return UPIPE_ERR_INVALID_ARG;
  if (!aligned16(buf)) return UPIPE_ERR_ALIGNMENT;
  return cuda_status(launch_wait_probe(buf, arrive, (cudaStream_t)stream));
}

upipe_status_t upipe_attn_last_device_error(const void* ws, void* stream, int32_t* code) {
  return upipe_attn_device_status(ws, code, stream);
}

}  // extern "C"
