/*
 * upipe_attn: head-chunked causal self-attention (forward and backward) on one GB300.
 *
 * The layer is  Y = concat_h softmax(Q_h K_{h/g}^T * scale + M) V_{h/g} * Wo^T  with
 * [Q | K | V] = X * Wqkv^T, for a sequence of S tokens of hidden size d.  Its query heads are
 * processed in chunks of `heads_per_chunk`, one chunk after another, and every chunk's Q/K/V
 * projection, attention and output-projection accumulation run inside one caller-provided
 * workspace that is reused from chunk to chunk, so activation memory grows with the chunk
 * size and not with the number of heads.
 *
 * Sources: "Road to 5 Million Tokens" (podcast summary, chapters "主要貢獻 UPipe" and
 * "分批算 heads": heads on one GPU run in groups, one group after another; partial results
 * are kept and the next group reuses the buffer the previous one allocated; Q&A chapter: it
 * concerns the layer's query, key and value matrices).  neuro-slop.ru transcript ("Как
 * уместить 5 млн токенов...", quiz answer on U-Pipe and insight 02: one set of heads already
 * saturates the GPU, so heads are chunked in time with one small reused buffer).  Packed
 * sequences and skipping of fully masked tiles: MaxText long-context article (techmoon.xyz),
 * paragraph on Splash attention.  GQA: same paragraph.
 *
 * Conventions for every entry point
 *  - All tensors are row-major.  bf16 tensors are passed as uint16_t bit patterns.
 *  - Weights follow the nn.Linear layout [out, in].  Wqkv rows are [Q heads | K heads | V heads],
 *    head_dim rows per head; query head h uses KV head h / (n_q_heads / n_kv_heads).
 *  - Pointers marked "device" are CUDA device addresses; every device pointer must be 16-byte
 *    aligned.  `stream` is a cudaStream_t (NULL = the legacy default stream).
 *  - The caller owns every buffer, including the workspace.  The library allocates no device
 *    memory and keeps no state between calls.  Calls are stream-ordered and asynchronous;
 *    two calls may run concurrently only with different workspaces.
 *  - Every check that depends only on the arguments is made on the host before any launch; a
 *    failing check returns a status and launches nothing.  Conditions only the device can see
 *    (segment ids that are not non-decreasing) set an error word in the workspace or table,
 *    read with upipe_attn_device_status().  No call aborts, traps or throws.
 */
#ifndef UPIPE_ATTN_H
#define UPIPE_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  UPIPE_OK = 0,
  UPIPE_ERR_INVALID_ARG = 1,             /* NULL pointer, bad size or shape                    */
  UPIPE_ERR_UNSUPPORTED = 2,             /* valid but not supported (e.g. head_dim 96)         */
  UPIPE_ERR_ALIGNMENT = 3,               /* a device pointer is not 16-byte aligned            */
  UPIPE_ERR_WORKSPACE_TOO_SMALL = 4,     /* ws_bytes / table_bytes below the required size     */
  UPIPE_ERR_SEGMENTS_NOT_CONTIGUOUS = 5, /* device-detected: segment ids decrease somewhere    */
  UPIPE_ERR_CUDA = 6,                    /* a CUDA runtime call failed (launch error)          */
  UPIPE_ERR_DEVICE_TIMEOUT = 7           /* a bounded device-side wait ran out                 */
} upipe_status_t;

typedef struct {
  int64_t seq_len;         /* S: 1 .. 2^31 - 1 tokens (TMA tile coordinates are signed 32-bit)  */
  int32_t hidden;          /* d: multiple of 64                                                */
  int32_t n_q_heads;       /* Hq                                                               */
  int32_t n_kv_heads;      /* Hkv; Hq % Hkv == 0 (g = Hq / Hkv query heads share a KV head)     */
  int32_t head_dim;        /* Dh: 64 or 128                                                    */
  int32_t heads_per_chunk; /* query heads per chunk; Hq % hpc == 0 and (hpc % g == 0 or
                              g % hpc == 0), so a chunk holds whole KV groups or part of one */
  int32_t causal;          /* 1: key j visible to query i only if j <= i                       */
  int32_t accum_mode;      /* 0: fp32 accumulators for Y / dX in the workspace (default);
                              1: accumulate in place in the bf16 output (fp32 math per chunk,
                              one bf16 rounding per chunk; smaller workspace)                  */
  float softmax_scale;     /* 0 selects 1/sqrt(head_dim)                                       */
} upipe_attn_desc_t;

/* Human-readable name of a status code (static string, never NULL).  No counterpart on the
 * pages (they print no interface); a convenience of this library. */
const char* upipe_attn_status_string(upipe_status_t status);

/* Name of the CUDA runtime error (e.g. "cudaErrorInvalidValue") behind the most recent
 * UPIPE_ERR_CUDA returned on the calling host thread; "cudaSuccess" if none.  Static string. */
const char* upipe_attn_last_error_string(void);

/* Workspace bytes needed by upipe_attn_fwd (pass = 0) or upipe_attn_bwd (pass = 1) for this
 * descriptor.  Host-only; writes *bytes.  The size grows with heads_per_chunk (per-chunk
 * Q/O/dO/dQ buffers and the resident K/V of one KV group), not with n_q_heads: the one reused
 * group-sized buffer of UPipe ("Road to 5 Million Tokens" podcast summary, chapter "主要貢獻
 * UPipe": the next group reuses the buffer the previous group allocated). */
upipe_status_t upipe_attn_workspace_size(const upipe_attn_desc_t* desc, int pass, size_t* bytes);

/* Bytes of the tile-skip table for seq_len S, with n = ceil(S/128):
 * 32-byte header + 2 * n * 16 + 4 * (ceil(n/2) + n), rounded up to a multiple of 16.
 * (MaxText long-context article, Splash attention paragraph: the table is what lets fully
 * masked blocks be skipped.) */
upipe_status_t upipe_attn_tile_table_size(const upipe_attn_desc_t* desc, size_t* bytes);

/* Tile-skip table (Splash-style skipping of fully masked blocks, MaxText article).
 * For 128x128 tiles (query tile i, key tile j) a tile is EMPTY when no (query, key) pair in it
 * is visible, FULL when every in-range pair is, PARTIAL otherwise; visible means
 * seg[q] == seg[k] and (not causal or k <= q).  With non-decreasing segment ids the non-empty
 * tiles of a row form one range with the full ones in the middle, so the table stores
 *   header  : int64 n_partial, int64 n_full (tile pairs per head), int32 error (0 or
 *             UPIPE_ERR_SEGMENTS_NOT_CONTIGUOUS), int32 n_tiles, int64 reserved
 *   q-major : int32[n_tiles][4] {kv_begin, kv_full_begin, kv_full_end, kv_end}
 *   kv-major: int32[n_tiles][4] {q_begin, q_full_begin, q_full_end, q_end}
 *   q-order : int32[ceil(n_tiles/2)] query-tile pairs p (tiles 2p, 2p + 1) by non-increasing
 *             number of non-empty tiles in their rows, ties later pair first
 *   kv-order: int32[n_tiles] key tiles by non-increasing number of non-empty tiles in their
 *             rows, ties earlier tile first
 * (half-open ranges of tile indices; a row with no full tile has full_begin = full_end = end).
 * The two orders are the attention kernels' dispatch orders (most work first); they do not change
 * any result.
 * seg: device int32[S] or NULL (one segment).  table: device, table_bytes from
 * upipe_attn_tile_table_size.  Only desc->seq_len and desc->causal are read.
 * visited_counts_host: NULL, or host int64[2] that receives {n_partial, n_full} (the visited
 *   tile pairs per head); then the call waits for the stream (a synchronous read of the header).
 *   With NULL the call is asynchronous and the counts stay readable in the header. */
upipe_status_t upipe_attn_build_tile_table(const upipe_attn_desc_t* desc, const int32_t* seg, void* table,
                                           size_t table_bytes, int64_t* visited_counts_host, void* stream);

/* Forward pass of the layer.
 *   X    device bf16 [S, d]                      hidden states
 *   Wqkv device bf16 [(Hq + 2 Hkv) * Dh, d]
 *   Wo   device bf16 [d, Hq * Dh]
 *   seg  device int32 [S] non-decreasing segment ids, or NULL (one segment)
 *   Y    device bf16 [S, d]                      output (written)
 *   lse  device fp32 [Hq, S]                     natural-log softmax normaliser per query row,
 *                                                the only state the backward pass needs
 *   ws   device workspace of ws_bytes >= upipe_attn_workspace_size(desc, 0)
 * Chunks run in ascending head order; the K/V of a KV group stay resident in the workspace
 * while the chunks of that group run. */
upipe_status_t upipe_attn_fwd(const upipe_attn_desc_t* desc, const uint16_t* X, const uint16_t* Wqkv,
                              const uint16_t* Wo, const int32_t* seg, uint16_t* Y, float* lse, void* ws,
                              size_t ws_bytes, void* stream);

/* Backward pass: gradients of sum(dY * Y).  Activations are recomputed chunk by chunk from X
 * and the saved lse (activation checkpointing inside the layer: podcast summary, chapter
 * "Activation checkpointing").
 *   dY    device bf16 [S, d]
 *   lse   device fp32 [Hq, S] as written by upipe_attn_fwd for the same inputs
 *   dX    device bf16 [S, d]                    (written)
 *   dWqkv device fp32 [(Hq + 2 Hkv) * Dh, d]     (written, not accumulated)
 *   dWo   device fp32 [d, Hq * Dh]               (written, not accumulated)
 *   ws    device workspace of ws_bytes >= upipe_attn_workspace_size(desc, 1) */
upipe_status_t upipe_attn_bwd(const upipe_attn_desc_t* desc, const uint16_t* X, const uint16_t* Wqkv,
                              const uint16_t* Wo, const int32_t* seg, const uint16_t* dY, const float* lse,
                              uint16_t* dX, float* dWqkv, float* dWo, void* ws, size_t ws_bytes,
                              void* stream);

/* CPU offload of the layer's inputs ("Road to 5 Million Tokens" podcast summary, chapter on moving
 * part of the inputs to the CPU; neuro-slop.ru transcript, implementation plan step 2: block
 * inputs offloaded to the CPU).  Same layer, same results as upipe_attn_fwd / upipe_attn_bwd, but
 * X (and, in the backward, dY) stay in page-locked host memory and never occupy device memory as a
 * whole: the library brings them in `stage_rows` rows at a time (0 selects 65536; otherwise a
 * multiple of 128) into two staging buffers per tensor inside the workspace, one
 * cudaMemcpyAsync per block on a copy stream the library keeps per device, issued one block ahead so that copies
 * overlap the projections.  Per chunk the forward streams X once (the Q/K/V projection); the
 * backward streams X and dY twice (the Q/K/V and dO projections before the attention kernels,
 * the weight gradients dWo and dWqkv after them, summed block by block in a fixed order).
 *   X_host, dY_host  bf16 [S, d], each either page-locked host memory (cudaHostAlloc or
 *                    cudaHostRegister), which is staged, or device memory, which is read in place
 *                    (a training stack offloads the block input X; its dY is produced on the device
 *                    during the backward); pageable host memory is rejected with
 *                    UPIPE_ERR_INVALID_ARG before any launch
 *   ws               device workspace of upipe_attn_workspace_size_offload(desc, pass, stage_rows)
 *                    bytes (the regular workspace plus 2 or 4 staging buffers of stage_rows x d)
 * Y, lse and dX are bit-identical to the regular calls'; dWqkv and dWo equal theirs to rounding
 * (their sums over S are split at other places).  The host buffers must not change until the
 * call's work on `stream` has completed. */
upipe_status_t upipe_attn_workspace_size_offload(const upipe_attn_desc_t* desc, int pass, int64_t stage_rows,
                                                 size_t* bytes);
upipe_status_t upipe_attn_fwd_offload(const upipe_attn_desc_t* desc, const uint16_t* X_host, const uint16_t* Wqkv,
                                      const uint16_t* Wo, const int32_t* seg, uint16_t* Y, float* lse, void* ws,
                                      size_t ws_bytes, int64_t stage_rows, void* stream);
upipe_status_t upipe_attn_bwd_offload(const upipe_attn_desc_t* desc, const uint16_t* X_host, const uint16_t* Wqkv,
                                      const uint16_t* Wo, const int32_t* seg, const uint16_t* dY_host, const float* lse,
                                      uint16_t* dX, float* dWqkv, float* dWo, void* ws, size_t ws_bytes,
                                      int64_t stage_rows, void* stream);

/* The feed-forward step beside the attention layer, computed in tiles of rows along the sequence
 * so that no intermediate spans the whole sequence (sequence tiling of the element-wise steps:
 * "Road to 5 Million Tokens" podcast summary, 概要 and the chapter on tiling; neuro-slop.ru
 * transcript, Полезные советы: the loss and the MLP can be computed in pieces).  The pages do not
 * write the MLP; for the Llama-3.1-shaped layers it is the Llama feed-forward block (SwiGLU):
 *   Y = (silu(X Wg^T) * (X Wu^T)) Wd^T,  silu(x) = x / (1 + e^-x).
 * Per tile of T rows: H = X_t [Wg; Wu]^T (tensor cores, bf16 [T][2F]), A = silu(G) * U (bf16
 * [T][F]), Y_t = A Wd^T.  The backward recomputes H per tile, then dA = dY_t Wd, [dG | dU] and A,
 * dX_t = [dG | dU] [Wg; Wu], and adds the tile's dWd = dY_t^T A and dWgu = [dG | dU]^T X_t to the
 * weight gradients (summed over tiles in a fixed order).  The workspace holds one tile's H, A,
 * dA and dH: 2T(2F + F) bytes forward, 2T(6F) backward (plus split-K partials), so memory
 * grows with tile_rows, not with S.
 *   seq_len    S (1 .. 2^31 - 1)
 *   hidden     d, multiple of 64;  ffn  F, multiple of 64
 *   tile_rows  rows per tile, a multiple of 128, or 0 for one tile of all S rows (untiled)
 *   X, Y, dY, dX  device bf16 [S, d];  Wgu device bf16 [2F, d] (gate rows, then up rows);
 *   Wd device bf16 [d, F];  dWgu, dWd device fp32, same shapes (written, not accumulated). */
typedef struct {
  int64_t seq_len;
  int32_t hidden;
  int32_t ffn;
  int64_t tile_rows;
} upipe_mlp_desc_t;
upipe_status_t upipe_mlp_workspace_size(const upipe_mlp_desc_t* desc, int pass, size_t* bytes);
upipe_status_t upipe_mlp_fwd(const upipe_mlp_desc_t* desc, const uint16_t* X, const uint16_t* Wgu, const uint16_t* Wd,
                             uint16_t* Y, void* ws, size_t ws_bytes, void* stream);
upipe_status_t upipe_mlp_bwd(const upipe_mlp_desc_t* desc, const uint16_t* X, const uint16_t* Wgu, const uint16_t* Wd,
                             const uint16_t* dY, uint16_t* dX, float* dWgu, float* dWd, void* ws, size_t ws_bytes,
                             void* stream);

/* Forward pass for callers that cannot allocate device memory (for example code recorded into
 * someone else's CUDA graph, or a plugin that only receives input and output pointers).  The
 * pages describe nothing like it; it is a convenience of this library.  Same arguments and
 * results as upipe_attn_fwd, without ws/ws_bytes: the workspace is a 32 MiB device array
 * inside the library, which every GPU that loads the library holds until the process exits.
 *  - Descriptors whose forward workspace (upipe_attn_workspace_size, pass 0) exceeds 32 MiB
 *    are rejected with UPIPE_ERR_WORKSPACE_TOO_SMALL before any launch.
 *  - No cudaMalloc, cudaFree or other allocating call is made.
 *  - The first call on a device looks up the array's device address on that (current)
 *    device; make that first call before any stream capture.  The address is kept for the
 *    life of the process: do not use this entry point across cudaDeviceReset.
 *  - Device-detected errors land in the array's own error word: read them with
 *    upipe_attn_no_alloc_device_status.
 *  - Every call uses the same array and leaves its contents behind; the forward pass
 *    initialises everything it reads.  Calls whose executions overlap on the GPU (different
 *    streams, or concurrent host threads) race on the array: serialise them. */
upipe_status_t upipe_attn_fwd_no_alloc(const upipe_attn_desc_t* desc, const uint16_t* X, const uint16_t* Wqkv,
                                       const uint16_t* Wo, const int32_t* seg, uint16_t* Y, float* lse,
                                       void* stream);

/* Attention core alone, Q/K/V given directly (head-major), for testing the kernels in isolation
 * (flash attention over whole heads: podcast summary, chapter "DeepSpeed Ulysses").
 *   q [Hq, S, Dh], k, v [Hkv, S, Dh] device bf16; table from upipe_attn_build_tile_table (its
 *   header's error word is set if a bounded device wait runs out, so it is not const);
 *   o [Hq, S, Dh] device bf16 (written); lse [Hq, S] device fp32 (written).
 * heads_per_chunk and hidden are ignored. */
upipe_status_t upipe_attn_core_fwd(const upipe_attn_desc_t* desc, const uint16_t* q, const uint16_t* k,
                                   const uint16_t* v, const int32_t* seg, void* table, uint16_t* o,
                                   float* lse, void* stream);

/* The three kernels of the attention backward, one launch each, in the order the layer runs
 * them (activation recompute: podcast summary, chapter "Activation checkpointing").  Arguments as in upipe_attn_core_fwd; dO [Hq, S, Dh] device bf16; lse [Hq, S] from the
 * forward pass.
 *   recompute: o [Hq, S, Dh] bf16 and D, device fp32 [2][Hq][Sp] with Sp = ceil(S/128)*128:
 *              D[0][h][i] = rowsum(dO * O) of query row i, D[1][h][i] = lse * log2(e), zeros
 *              for i >= S; from q, k, v and lse without online rescaling (activation
 *              recompute).  bwd_dq and bwd_dkdv read D in this layout.
 *   bwd_dq   : dq [Hq, S, Dh] bf16 = scale * sum_j P_ij (dP_ij - D_i) k_j,  dP = dO v^T.
 *   bwd_dkdv : dk, dv [Hkv, S, Dh] bf16, summed over the query heads of each KV head:
 *              dv_j = sum P_ij dO_i,  dk_j = scale * sum P_ij (dP_ij - D_i) q_i. */
upipe_status_t upipe_attn_core_recompute(const upipe_attn_desc_t* desc, const uint16_t* q, const uint16_t* k,
                                         const uint16_t* v, const uint16_t* dO, const float* lse, const int32_t* seg,
                                         void* table, uint16_t* o, float* D, void* stream);
upipe_status_t upipe_attn_core_bwd_dq(const upipe_attn_desc_t* desc, const uint16_t* q, const uint16_t* k,
                                      const uint16_t* v, const uint16_t* dO, const float* lse, const float* D,
                                      const int32_t* seg, void* table, uint16_t* dq, void* stream);
upipe_status_t upipe_attn_core_bwd_dkdv(const upipe_attn_desc_t* desc, const uint16_t* q, const uint16_t* k,
                                        const uint16_t* v, const uint16_t* dO, const float* lse, const float* D,
                                        const int32_t* seg, void* table, uint16_t* dk, uint16_t* dv,
                                        void* stream);
/* bwd_dkdv into fp32 sums, as the layer launches it for a KV group split over head chunks or for
 * key tiles of more work items than the window of upipe_attn_set_dkdv_window:
 *   dk_acc, dv_acc  device fp32 [Hkv, S, Dh]: this call's dK, dV are added to what they hold
 *                   (in windows of work items: see upipe_attn_set_dkdv_window)
 *   dk, dv          both NULL, or device bf16 [Hkv, S, Dh] that receive the sums rounded. */
upipe_status_t upipe_attn_core_bwd_dkdv_acc(const upipe_attn_desc_t* desc, const uint16_t* q, const uint16_t* k,
                                            const uint16_t* v, const uint16_t* dO, const float* lse,
                                            const float* D, const int32_t* seg, void* table, float* dk_acc,
                                            float* dv_acc, uint16_t* dk, uint16_t* dv, void* stream);

/* Projection GEMM alone, for testing: C[M, N] (fp32, row-major, ldc) = A[M, K] * B[N, K]^T with
 * A, B device bf16 row-major (lda, ldb in elements).  The per-chunk Q/K/V and O projections of
 * the layer run on this kernel (podcast summary, Q&A chapter: UPipe concerns the layer's Q/K/V). */
upipe_status_t upipe_attn_gemm_nt(int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda,
                                  const uint16_t* B, int64_t ldb, float* C, int64_t ldc, void* stream);

/* Merge of block attention results: the single-GPU share of ring (P2P) context parallelism, where
 * key/value blocks travel around a ring of devices and each device attends its query block to
 * the visiting block (MaxText long-context article, table of context-parallel strategies, row
 * "P2P (Ring)").  For `rows` query rows (e.g. n_heads * block length, head-major as
 * upipe_attn_core_fwd writes them), with L the natural-log log-sum-exp of a row's scores:
 *   L_acc <- log(e^{L_acc} + e^{L_b}),   O_acc <- (e^{L_acc,old} O_acc + e^{L_b} O_b) / e^{L_acc,new}
 * which is attention over the union of the key sets seen so far and the block's.
 *   O_b      device bf16 [rows][head_dim]: the block's output (upipe_attn_core_fwd `o`)
 *   lse_b    device fp32 [rows]: the block's log-sum-exp (upipe_attn_core_fwd `lse`)
 *   O_acc    device fp32 [rows][head_dim], updated in place; start from zeros
 *   lse_acc  device fp32 [rows], updated in place; start from -inf
 *   O_out    NULL, or device bf16 [rows][head_dim] that receives the merged O rounded to bf16
 * A side whose L is -inf contributes nothing; a row with both -inf stays O = 0, L = -inf.
 * head_dim 64 or 128; all pointers 16-byte aligned.  Stream-ordered, asynchronous. */
upipe_status_t upipe_attn_lse_merge(int64_t rows, int32_t head_dim, const uint16_t* O_b, const float* lse_b,
                                    float* O_acc, float* lse_acc, uint16_t* O_out, void* stream);

/* Backward of the ring share.  Every block (query chunk, key chunk) runs upipe_attn_core_bwd_dq
 * and upipe_attn_core_bwd_dkdv with the softmax over the whole key set: the query chunk's final
 * log-sum-exp and D = rowsum(dO * O) of its final (merged) output.  This fills their D buffer
 * from those: D device fp32 [2][n_heads][Sp], Sp = ceil(seq_len/128)*128, D[0][h][i] = sum over
 * the head dimension of dO * O, D[1][h][i] = lse * log2(e), zeros for i >= seq_len.
 *   O, dO  device bf16 [n_heads][seq_len][head_dim]: the chunk's final output and its gradient
 *   lse    device fp32 [n_heads][seq_len]: the chunk's final log-sum-exp (natural log)
 * head_dim 64 or 128; pointers 16-byte aligned. */
upipe_status_t upipe_attn_ring_bwd_prep(int32_t n_heads, int64_t seq_len, int32_t head_dim, const uint16_t* O,
                                        const uint16_t* dO, const float* lse, float* D, void* stream);

/* acc[i] += src[i] for n elements (src device bf16, acc device fp32, in place); out, if not NULL,
 * receives bf16(acc[i]) (round to nearest even).  The ring backward sums the blocks' dQ, dK and dV
 * contributions with it and rounds each gradient once.  Pointers 16-byte aligned. */
upipe_status_t upipe_attn_accumulate(int64_t n, const uint16_t* src, float* acc, uint16_t* out, void* stream);

/* ------------------------------------------------------------------------------------------
 * Ring (P2P) context parallelism, one call per ring step (MaxText long-context article: table of
 * the context-parallel strategies, row "P2P (Ring)", and the paragraph after it on the causal
 * load balancing the ring needs).  The sequence of 2PC rows is cut into 2P chunks of C rows;
 * ring device r holds chunks r and 2P-1-r as its shard, one plane of 2C rows per head (local
 * row i is at position i < C ? rC + i : (2P-1-r)C + i - C), so every device does the same work.
 * At step s device r attends its queries to the key/value shard of device (r - s) mod P: keys
 * at an earlier or equal position (causal) and of the same segment.  Every step is one launch
 * for all batched devices; its result is folded into fp32 accumulators (the log-sum-exp merge
 * L = log(e^L_acc + e^L_b), O = (e^L_acc O_acc + e^L_b O_b) / e^L), so after the last step they
 * hold attention over the whole sequence.  One GPU can run the shares of several devices
 * (dev_count > 1, their shards as consecutive planes); the exchange of the shards between
 * devices is not part of the library.
 *
 * Shapes (planes of 2C rows, row-major, head-major inside a device):
 *   q, o, dO        [dev_count][n_q_heads][2C][head_dim]   bf16
 *   k, v            [kv_count][n_kv_heads][2C][head_dim]   bf16
 *   lse             [dev_count][n_q_heads][2C]             fp32
 * kv_count == P: k and v hold every device's shard, in device order (shard m is device m's);
 * otherwise kv_count == dev_count and they hold, in batch order, the shards that visit the
 * batched devices at the step of the call (a device of a real ring passes its receive buffer).
 * seg: NULL (one sequence) or device int32 [2PC] segment ids in SEQUENCE order (non-decreasing;
 * packed sequences attend within their segment only). */
typedef struct {
  int32_t ring_size;    /* P >= 1 */
  int32_t n_q_heads, n_kv_heads, head_dim; /* head_dim 64 or 128; n_q_heads a multiple of n_kv_heads */
  int64_t chunk_len;    /* C >= 1, 2C <= 2^31 - 1 */
  int32_t causal;       /* 1: causal (the ring's use); 0: every key of the segment */
  float softmax_scale;  /* <= 0: 1/sqrt(head_dim) */
  int32_t dev_first, dev_count; /* the ring devices dev_first .. dev_first + dev_count - 1 (<= P) */
  int32_t kv_count;     /* P, or dev_count (see above) */
} upipe_ring_desc_t;
/* A descriptor whose launches would exceed the grid's second dimension (dev_count * ceil(2C/256)
 * query-tile pairs or kv_count * ceil(2C/128) key tiles above 65535) is UPIPE_ERR_UNSUPPORTED. */

/* Bytes of the P per-step tile tables of a ring (device memory the caller owns, 16-byte
 * aligned).  The tables depend on the descriptor and on seg only: build them once per segment
 * layout and reuse them for every layer and both passes. */
upipe_status_t upipe_attn_ring_tables_size(const upipe_ring_desc_t* desc, size_t* bytes);
/* Builds the tables of every step (stream-ordered).  Segment ids that are not non-decreasing set
 * UPIPE_ERR_SEGMENTS_NOT_CONTIGUOUS in the error word read by upipe_attn_device_status(tables);
 * so does a bounded device wait of any ring step that runs out. */
upipe_status_t upipe_attn_ring_build_tables(const upipe_ring_desc_t* desc, const int32_t* seg, void* tables,
                                            size_t bytes, void* stream);

/* Forward of ring step `step` (0 .. P-1, called in order on the same accumulators): one
 * attention launch over all batched devices.
 *   o_acc  device fp32 [dev_count][n_q_heads][2C][head_dim]: running output (step 0 writes it,
 *          later steps fold into it)
 *   lse    device fp32 [dev_count][n_q_heads][2C]: running log-sum-exp (natural log), final
 *          after the last step
 *   o      NULL, or device bf16 like q: the result.  A 128-row tile's rows are written by the
 *          last step that changes them (the steps' tables say which), and that step does not
 *          store them to o_acc; with o NULL, o_acc holds the result after the last step.
 * Query tiles that see no key of the visiting shard are not touched. */
upipe_status_t upipe_attn_ring_fwd_step(const upipe_ring_desc_t* desc, int32_t step, const uint16_t* q,
                                        const uint16_t* k, const uint16_t* v, const int32_t* seg, void* tables,
                                        float* o_acc, float* lse, uint16_t* o, void* stream);

/* Backward of ring step `step` (0 .. P-1, in order), two launches (dQ, then dK and dV).  Every
 * block uses the softmax over the whole key set: D from upipe_attn_ring_bwd_prep over the
 * final o, dO and lse (n_heads = dev_count * n_q_heads, seq_len = 2C).
 *   dq_acc          device fp32 like o_acc: dQ summed over the steps (step 0 writes it)
 *   dk_acc, dv_acc  device fp32 [kv_count][n_kv_heads][2C][head_dim]: dK, dV of the key shards,
 *                   indexed like k and v, summed over the steps and the query heads of each KV
 *                   head (on a real ring they travel with their shard)
 *   dq, dk, dv      NULL, or device bf16 like q / k / v: the sums rounded.  dq's rows are
 *                   written by the last step that changes their tile, which then does not store
 *                   dq_acc; likewise dk / dv when one call batches every device with every
 *                   shard (dev_count = kv_count = P), else every step writes the key tiles it
 *                   changes (so dk / dv travel with their shard like dk_acc / dv_acc) and the
 *                   ring's last step does not store dk_acc / dv_acc (for a key tile of more
 *                   work items than upipe_attn_set_dkdv_window's window they then hold partial
 *                   sums).  With a NULL bf16 output the fp32 sums hold the result after the
 *                   last step.
 * Tiles that no query of a step sees are not touched by that step. */
upipe_status_t upipe_attn_ring_bwd_step(const upipe_ring_desc_t* desc, int32_t step, const uint16_t* q,
                                        const uint16_t* k, const uint16_t* v, const uint16_t* dO, const float* D,
                                        const int32_t* seg, void* tables, float* dq_acc, float* dk_acc,
                                        float* dv_acc, uint16_t* dq, uint16_t* dk, uint16_t* dv, void* stream);

/* All P steps of the forward (steps 0 .. P-1 in order) in one call, with the arguments of
 * upipe_attn_ring_fwd_step.  Each step after the first may start on the SMs the previous step's
 * last CTAs leave idle: it computes its blocks and waits for the previous step to complete only
 * before it touches the accumulators (programmatic dependent launch).  For a GPU that holds
 * every shard (the batched single-GPU share); a device of a real ring calls the steps one by one
 * as its shards arrive. */
upipe_status_t upipe_attn_ring_fwd(const upipe_ring_desc_t* desc, const uint16_t* q, const uint16_t* k,
                                   const uint16_t* v, const int32_t* seg, void* tables, float* o_acc, float* lse,
                                   uint16_t* o, void* stream);

/* All P steps of the backward in one call: D (device fp32 [2][dev_count * n_q_heads][Sp], Sp =
 * ceil(2C/128)*128, written) from the final o, dO and lse as upipe_attn_ring_bwd_prep writes it,
 * then steps 0 .. P-1 chained as in upipe_attn_ring_fwd; other arguments as in
 * upipe_attn_ring_bwd_step. */
upipe_status_t upipe_attn_ring_bwd(const upipe_ring_desc_t* desc, const uint16_t* q, const uint16_t* k,
                                   const uint16_t* v, const uint16_t* o, const uint16_t* dO, const float* lse,
                                   const int32_t* seg, void* tables, float* D, float* dq_acc, float* dk_acc,
                                   float* dv_acc, uint16_t* dq, uint16_t* dk, uint16_t* dv, void* stream);

/* Reads the device error word of a workspace (after fwd/bwd) or of a table (after
 * build_tile_table) into *code (a upipe_status_t value; UPIPE_OK when none).  Synchronises
 * `stream`.  `buf` is the workspace or the table.  No counterpart on the pages. */
upipe_status_t upipe_attn_device_status(const void* buf, int32_t* code, void* stream);

/* The same read with the argument order of the library's original interface sketch: `ws` is a
 * workspace (or a table), *code receives its device error word after `stream` has drained. */
upipe_status_t upipe_attn_last_device_error(const void* ws, void* stream, int32_t* code);

/* Device error word of the array upipe_attn_fwd_no_alloc uses as its workspace, on the current
 * device, after `stream` has drained: segment ids that are not non-decreasing
 * (UPIPE_ERR_SEGMENTS_NOT_CONTIGUOUS) or a bounded device wait that ran out.  Allocates nothing.
 * The word describes the most recent upipe_attn_fwd_no_alloc call on this device (each call
 * clears it first).  Before the first such call on a device it reports UPIPE_OK. */
upipe_status_t upipe_attn_no_alloc_device_status(int32_t* code, void* stream);

/* Per-launch timing of the layer's kernels, a diagnostic with no counterpart on the pages (the
 * pages point to a profiler to find where memory and time go: podcast summary, chapter
 * "PyTorch profiler").  While enabled, every kernel launch of upipe_attn_fwd / upipe_attn_bwd
 * (and their offloaded forms), upipe_mlp_fwd / upipe_mlp_bwd and the ring steps is
 * bracketed by two CUDA events on the call's stream and logged with its kind and shape; do not
 * enable it while a stream is being captured into a CUDA graph.  Process-wide; off by default.
 *   kind      UPIPE_K_* below
 *   epilogue  GEMMs: 0 store bf16, 1 store fp32, 2 fp32 C += A B^T, 3 bf16 C += A B^T
 *   m, n, k   GEMMs: C[m, n] = A[m, k] B[n, k]^T; attention kernels: m = S, n = query heads,
 *             k = head_dim; conversions / zeroing: m = elements; tile table: m = S
 *   split_k   GEMM K splits (> 1: the record includes the split reduction)
 *   chunk     head chunk index (-1 for the tile table)
 *   ms        device time between the two events
 *   start_ms  when the first event fired, relative to the first record of the collect
 * upipe_attn_timing_collect waits for the logged launches, copies up to `cap` records (in
 * launch order) into `out`, writes the total count to *n and clears the log. */
enum {
  UPIPE_K_TILE_TABLE = 0, UPIPE_K_QKV_PROJ = 1, UPIPE_K_ATTN_FWD = 2, UPIPE_K_O_PROJ = 3, UPIPE_K_CONVERT = 4,
  UPIPE_K_DO_PROJ = 5, UPIPE_K_RECOMPUTE = 6, UPIPE_K_DWO = 7, UPIPE_K_BWD_DQ = 8, UPIPE_K_BWD_DKDV = 9,
  UPIPE_K_DX_PROJ = 10, UPIPE_K_DWQKV = 11, UPIPE_K_ZERO = 12,
  /* the sequence-tiled MLP (upipe_mlp_fwd / upipe_mlp_bwd) */
  UPIPE_K_MLP_GATE_UP = 13, UPIPE_K_MLP_ACT = 14, UPIPE_K_MLP_DOWN = 15, UPIPE_K_MLP_DACT = 16,
  UPIPE_K_MLP_ACT_BWD = 17, UPIPE_K_MLP_DWD = 18, UPIPE_K_MLP_DX = 19, UPIPE_K_MLP_DWGU = 20,
  /* a host-to-device staging copy of the offloaded calls (on their copy stream; m = bytes,
     chunk = row block) */
  UPIPE_K_H2D = 21,
  /* ring steps (m = 2C, n = dev_count * n_q_heads, k = head_dim, chunk = step) */
  UPIPE_K_RING_FWD = 22, UPIPE_K_RING_DQ = 23, UPIPE_K_RING_DKDV = 24
};
typedef struct {
  int32_t kind, epilogue, split_k, chunk;
  int64_t m, n, k;
  float ms;
  float start_ms; /* start relative to the first record of the same collect call */
} upipe_attn_timing_t;
upipe_status_t upipe_attn_timing_enable(int32_t on);
upipe_status_t upipe_attn_timing_collect(upipe_attn_timing_t* out, int32_t cap, int32_t* n);

/* Accumulation window of the layer backward's dK / dV kernel, in work items (query head x query
 * tile) per key tile; 0 restores the default of 4096, otherwise even, 2 .. 2^24, else
 * UPIPE_ERR_INVALID_ARG.  The kernel sums each key tile's dK and dV over all query heads of its KV
 * group and all query tiles that see it (MaxText article, Splash paragraph: GQA) in tensor-memory
 * fp32 accumulators; a very long accumulation into the same accumulator drifts low, so once a key
 * tile has more items than the window, the layer backward entry points (upipe_attn_bwd and its
 * offload variant) keep dK / dV as fp32 sums in their workspace and the kernel adds its
 * accumulators into them after every full window.  Takes effect for workspaces planned (and
 * sizes queried) after the call: a workspace must be sized under the same window it runs with.
 * Ring backward steps flush into their dk_acc / dv_acc the same way (a key tile of a step has
 * n_q_heads / n_kv_heads x ceil(2C/128) items at most), and so does
 * upipe_attn_core_bwd_dkdv_acc; upipe_attn_core_bwd_dkdv, which writes bf16 only, does not flush. */
upipe_status_t upipe_attn_set_dkdv_window(int32_t items);

/* Limit of every bounded device-side wait of the library's kernels, in nanoseconds (0 restores the
 * default of 4 s; at most 60 s).  Each kernel receives the value in effect when it is launched.
 * When a wait runs out, the kernel raises UPIPE_ERR_DEVICE_TIMEOUT in the error word of its
 * workspace or table and returns instead of hanging.  A diagnostic with no counterpart on the
 * pages: shorter limits are for testing the timeout path with upipe_attn_wait_probe. */
upipe_status_t upipe_attn_set_wait_limit_ns(uint64_t ns);

/* Runs the library's bounded wait on a barrier that nothing completes (arrive = 0) or on one it
 * completes itself first (arrive = 1), under the current wait limit.  `buf` is a device buffer
 * of at least 32 bytes laid out as a table header; its error word is cleared, then set to
 * UPIPE_ERR_DEVICE_TIMEOUT if the wait runs out (read it with upipe_attn_device_status). */
upipe_status_t upipe_attn_wait_probe(void* buf, size_t bytes, int32_t arrive, void* stream);

/* Number of GPU kernels this library has launched in the process so far (every entry point
 * counts its own launches; a diagnostic with no counterpart in the method).  The difference of
 * two reads brackets the launches of the calls between them on any thread. */
uint64_t upipe_attn_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* UPIPE_ATTN_H */
