// Internal launch interfaces of the head-chunked attention library.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace upipe {

// Every kernel launch of the library calls this once (a process-wide counter, read through
// upipe_attn_launch_count).
void note_launch();

// Limit of every bounded device-side wait, in nanoseconds, passed to each kernel at launch
// (upipe_attn_set_wait_limit_ns; 4 s by default).
uint64_t wait_limit_ns();
// A kernel whose one bounded wait nothing satisfies (arrive = 0), or one that is satisfied at
// once (arrive = 1): the timeout path of the wait helper, reported in a table header's error word.
cudaError_t launch_wait_probe(void* header, int arrive, cudaStream_t st);

// ---------------------------------------------------------------- row geometry
// Zigzag ring (P2P context parallelism with causal load balancing: MaxText long-context article,
// strategy table and the paragraph after it).  The sequence is cut into 2P chunks of C rows; ring
// device r holds chunks r and 2P-1-r as one plane of 2C rows, so local row i sits at position
// i < C ? rC + i : (2P-1-r)C + i - C.  At ring step s device r attends to the key/value shard of
// device (r - s) mod P.  A launch may batch the query shards of `ndev` devices r0, r0+1, ... (as
// extra planes) against `kv_count` key/value shards; shard m in memory belongs to device
// (kv0 + m) mod P.  P == 0: plain geometry, query and key row i share position i.
struct RingGeom {
  int P;
  int r0, step, kv0;
  int64_t C;
};

// ---------------------------------------------------------------- tile-skip table
// Layout: header, q_rows [ndev][nt] int4, kv_rows [kv_count][nt] int4, q_order [ndev * npairs]
// int32 (entry = device * npairs + pair), kv_order [kv_count * nt] (entry = shard * nt + tile),
// with nt = ceil(S / 128) tiles per plane and npairs = ceil(nt / 2).
size_t tile_table_bytes(int64_t S, int ndev = 1, int kv_count = 1);
cudaError_t launch_tile_table(int64_t S, int causal, const int32_t* seg, void* table, cudaStream_t st);
// The table of one ring step: seg (NULL or [2PC]) is indexed by global position.
cudaError_t launch_ring_table(int64_t S, int causal, const int32_t* seg, const RingGeom& g, int ndev, int kv_count,
                              void* table, cudaStream_t st);

inline const int4* table_q_rows(const void* table) {
  return reinterpret_cast<const int4*>(reinterpret_cast<const char*>(table) + sizeof(TableHeader));
}
inline const int4* table_kv_rows(const void* table, int64_t S, int ndev = 1) {
  return table_q_rows(table) + ndev * ceil_div(S, kTile);
}
// Dispatch orders: query-tile pairs (2p, 2p + 1) and key tiles, each by non-increasing number of
// non-empty tiles (the work of the CTA that takes it), ties by the position the kernels used before
// (later pairs first, earlier key tiles first).
inline const int32_t* table_q_order(const void* table, int64_t S, int ndev = 1, int kv_count = 1) {
  return reinterpret_cast<const int32_t*>(table_kv_rows(table, S, ndev) + kv_count * ceil_div(S, kTile));
}
inline const int32_t* table_kv_order(const void* table, int64_t S, int ndev = 1, int kv_count = 1) {
  return table_q_order(table, S, ndev, kv_count) + ndev * ceil_div(ceil_div(S, kTile), 2);
}

// ---------------------------------------------------------------- projection GEMMs
// Logical operands: A is [M, K], B is [N, K]; C[M, N] = A * B^T.
constexpr int kMaxBlocks = 64;

enum GemmEpilogue : int {
  EPI_STORE_BF16 = 0,      // out(bf16) = acc
  EPI_STORE_F32 = 1,       // out(f32) = acc
  EPI_ACC_F32 = 2,         // out(f32) += acc
  EPI_ACC_BF16 = 3,        // out(bf16) = out(bf16) + acc (fp32 math)
};

struct GemmOutput {
  void* blk[kMaxBlocks];  // row-major [M][N] blocks; blocked along blk_dim (0: M, 1: N)
  int64_t ld;
  int blk_shift;          // -1: unblocked
  int blk_dim;
};

size_t gemm_split_scratch_bytes(int64_t M, int64_t N, int split_k);
int gemm_pick_split(int64_t M, int64_t N, int64_t K, int num_sms);

// Operand of the tensor-core GEMM as a TMA tensor map.  rank 2: rows of `row_stride` elements,
// [outer][inner]; rank 3: dense [planes][outer][inner].  k_major: the logical K index runs along
// `inner` (else the M/N index does).  With blk_shift >= 0 the logical index along blk_dim
// (0: M/N, 1: K) is split into blocks of 2^blk_shift (>= 64): rank 3 takes the block as the
// plane; rank 2 (blocked dimension outer only) starts block b at outer coordinate row_base[b].
struct TcOperand {
  const void* base;
  int rank;
  uint64_t inner, outer, planes, row_stride;
  uint64_t plane_stride;  // rank 3: elements between planes (0: dense, outer * inner)
  int k_major;
  int blk_shift;
  int blk_dim;
  int32_t row_base[kMaxBlocks];
};

struct TcGemmArgs {
  int64_t M, N, K;
  TcOperand a, b;
  GemmOutput c;
  int epi;
  int split_accumulate;  // split_k > 1: the reduction adds the splits' sum to the fp32 output
};

// C = A * B^T with the given epilogue on the tcgen05 path.  split_k > 1 requires
// epi == EPI_STORE_F32 and a scratch of split_k * M * N floats; the splits are reduced in a
// fixed order (deterministic), into C (or onto it with split_accumulate).
cudaError_t launch_gemm_tc(const TcGemmArgs& args, int split_k, float* split_scratch, cudaStream_t st);
cudaError_t launch_split_reduce(const float* part, int splits, int64_t M, int64_t N, const GemmOutput& out,
                                int accumulate, cudaStream_t st);

// ---------------------------------------------------------------- attention core
struct AttnArgs {
  const bf16* q;    // [nh, S, Dh]   query heads of this launch
  const bf16* k;    // [nkv, S, Dh]  KV heads; local query head h reads KV head h / g
  const bf16* v;
  bf16* o;          // [nh, S, Dh]
  float* lse;       // [nh] rows of stride S: natural-log normaliser (written in fwd, read in bwd)
  const bf16* dO;   // [nh, S, Dh]   (recompute mode and backward)
  float* D;         // [2][nh][ceil(S/128)*128]: rowsum(dO * O), then lse*log2e; zero past S
                    // (recompute mode writes, backward reads)
  const int32_t* seg;
  const int4* q_rows;   // q-major skip table
  const int4* kv_rows;  // kv-major skip table
  const int32_t* q_order;   // query-tile pairs, most work first
  const int32_t* kv_order;  // key tiles, most work first
  int64_t S;
  int nh;           // query heads of the launch
  int nkv;          // KV heads of the launch
  int g;            // query heads per KV head (local head h -> KV head h / g)
  int causal;
  float scale;      // softmax scale
  int* err;         // device error word (table header), set by bounded waits that time out
  uint64_t wait_ns; // limit of each bounded wait (set at launch)
  // Planes: the nh query planes are ndev devices x hq heads, the nkv KV planes kv_count shards x
  // hkv heads.  Zero (plain launches) means ndev = kv_count = 1, hq = nh, hkv = nkv.
  int hq, hkv, ndev, kv_count;
  RingGeom ring;    // ring.P == 0: plain geometry
  // Ring steps fold their result into fp32 accumulators: acc_first (step 0) writes them instead
  // of reading them; acc_last skips storing the fp32 state once only the bf16 result is needed.
  int acc_first, acc_last;
  float* o_acc;     // ring forward: [nh, S, Dh] fp32 running output (lse holds the running lse);
                    // o (if not NULL) receives the merged output rounded to bf16
  int pdl;          // launch with programmatic stream serialisation: the previous kernel on the
                    // stream is the previous ring step of the same call (see grid_dep_wait)
  // Ring steps: every step's table (step s at ring_tables + s * ring_table_stride), so that a tile
  // knows whether a later step touches it again; only the step that touches a row last writes its
  // bf16 result and that step skips the fp32 store.  kv_last_touch: the same holds for the key
  // shards' dK / dV sums (they are the launch's own shards at every step: all devices batched).
  const char* ring_tables;
  size_t ring_table_stride;
  int kv_last_touch;
};

// Launch with programmatic stream serialisation allowed (the grid may start while the previous
// kernel on the stream finishes; it synchronises with grid_dep_wait).
template <typename K, typename... Args>
cudaError_t launch_pdl(K kfn, dim3 grid, dim3 block, size_t smem, cudaStream_t st, const Args&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kfn, args...);
}

// Plain launches leave the plane fields zero: one device, one key shard, all heads of the launch.
inline void fill_planes(AttnArgs& a) {
  if (a.hq == 0) a.hq = a.nh;
  if (a.hkv == 0) a.hkv = a.nkv;
  if (a.ndev == 0) a.ndev = 1;
  if (a.kv_count == 0) a.kv_count = 1;
}

cudaError_t launch_attn_fwd(const AttnArgs& a, int head_dim, cudaStream_t st);
// One ring step of the forward: the block results are merged into o_acc / lse (see AttnArgs).
cudaError_t launch_attn_ring_fwd(const AttnArgs& a, int head_dim, cudaStream_t st);
// O and D from the saved lse (no online rescaling): activation recompute for the backward pass.
cudaError_t launch_attn_recompute(const AttnArgs& a, int head_dim, cudaStream_t st);

struct AttnBwdArgs {
  AttnArgs f;       // q, k, v, dO, lse, D, seg, tables
  bf16* dq;         // [nh, S, Dh]
  bf16* dk;         // [nkv, S, Dh]  written when acc_kv == 0
  bf16* dv;
  float* dk_acc;    // [nkv, S, Dh]  f32 accumulators when acc_kv == 1 (partial KV group, ring)
  float* dv_acc;
  int acc_kv;
  int nkv;
  int flush_items;  // > 0 (even; acc_kv launches): every flush_items work items the
                    // dK / dV tensor-memory accumulators are added into dk_acc / dv_acc and
                    // restarted, so no accumulation runs longer than that (see k_attn_bwd_dkdv_tc)
  float* dq_acc;    // ring: [nh, S, Dh] f32 accumulator of dQ (dq, if not NULL, gets it in bf16)
  bf16* dk_out;     // ring: the accumulated dK, dV rounded to bf16 (NULL: not written)
  bf16* dv_out;
};
cudaError_t launch_attn_bwd_dq(const AttnBwdArgs& a, int head_dim, cudaStream_t st);
cudaError_t launch_attn_bwd_dkdv(const AttnBwdArgs& a, int head_dim, cudaStream_t st);

// ---------------------------------------------------------------- small kernels
cudaError_t launch_f32_to_bf16(const float* in, bf16* out, int64_t n, float mul, cudaStream_t st);
cudaError_t launch_zero(void* p, int64_t bytes, cudaStream_t st);
cudaError_t launch_lse_merge(int64_t rows, int head_dim, const bf16* ob, const float* lb, float* oacc, float* lacc,
                             bf16* oout, cudaStream_t st);
cudaError_t launch_ring_bwd_prep(int nh, int64_t S, int head_dim, const bf16* o, const bf16* dout, const float* lse,
                                 float* D, cudaStream_t st);
cudaError_t launch_accumulate(int64_t n, const bf16* src, float* acc, bf16* out, cudaStream_t st);
// SwiGLU halves of the sequence-tiled MLP: H = [G | U] bf16 [rows][2F]
cudaError_t launch_swiglu_fwd(const bf16* H, bf16* A, int64_t rows, int64_t F, cudaStream_t st);
cudaError_t launch_swiglu_bwd(const bf16* H, const bf16* dA, bf16* A, bf16* dH, int64_t rows, int64_t F,
                              cudaStream_t st);

}  // namespace upipe
