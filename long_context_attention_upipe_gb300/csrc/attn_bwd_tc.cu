// Attention backward on the 5th-generation tensor cores (tcgen05, TMEM, TMA).
//
// Chain rule of softmax(Q K^T * scale + M) V per head, with P rebuilt from the saved
// log-sum-exp (activation recompute: podcast summary "Road to 5 Million Tokens", chapter
// "Activation checkpointing").  The recompute kernel leaves, per query row, D = rowsum(dO * O)
// and lse*log2e in a padded buffer Dbuf [2][nh][ceil(S/128)*128] (zeros past the end).
//   dP = dO V^T,  dS = P * (dP - D),  dQ = scale * dS K,  dK = scale * dS^T Q,  dV = P^T dO.
// Two kernels, both over the skip table's tiles:
//
// k_attn_bwd_dq_tc  (one head x two 128-row query tiles per CTA, 12 warps)
//   warp 0 TMA: Q_t, dO_t once, then K_j through a 2-slot ring and V_j through one slot (V_j is
//   only read by dP, so its slot is refilled early); warp 1 MMA + TMEM owner; warps 4-7 / 8-11
//   element-wise for tile a / b, one query row per thread (TMEM lane).
//   TMEM per tile: a 128-column region that holds S, then dP, then dS (bf16, columns 0-63),
//   and the dQ accumulator.  Per key tile:  S = Q K^T -> P = exp2(S c - lse2) kept in
//   registers in fp32 -> region free -> dP = dO V^T -> dS = P (dP - D) written to TMEM ->
//   dQ += dS K (A operand from TMEM, K in shared memory read MN-major).
//
// k_attn_bwd_dkdv_tc  (one KV head x one 128-row key tile per CTA, 12 warps)
//   warp 0 TMA: K_j, V_j once, then per work item (query head of the group x query tile) Q_i
//   into a 3-slot ring and dO_i into a 2-slot ring; warps 1 and 2 issue the MMAs of the even
//   and the odd items; warps 4-7 and 8-11 take the even and the odd items, one key row per
//   thread.  TMEM: dK and dV accumulators and two 128-column regions, one per element-wise
//   group.  Per item:  S^T = K Q^T -> P^T written to TMEM (kept in registers) -> dV += P^T dO
//   and dP^T = V dO^T into the same region -> dS^T = P^T (dP^T - D) written to TMEM ->
//   dK += dS^T Q.  Query heads sharing the KV head accumulate in TMEM (GQA reduction inside the
//   CTA).  The two issuers keep the shared dK / dV accumulations in item order through token
//   barriers; the two element-wise groups take turns phase by phase (named-barrier ping-pong).
//   A long accumulation into the same TMEM tile drifts low (against an fp64 sum of the same bf16
//   products: 0.6% after 32K work items, 4.8% after 312K), so launches that keep fp32 sums in
//   global memory (acc_kv) with flush_items > 0 add the accumulators into them and restart them
//   every flush_items items (a window): each element-wise group, after its last item of the
//   window, waits for the window's last MMAs (the Q-slot releases of its last two items), adds
//   its accumulator (group 0 dK, group 1 dV) to the global sum and arrives on win_empty; group 0
//   hands the next window's first P^T to the issuer (whose dV MMA restarts the accumulators) only
//   after win_empty completes.  The issuers only restart the accumulation at window starts.
// Every wait on an mbarrier is bounded (see tc::mbar_wait); registers are split per role with
// setmaxnreg (launch 168 x 384; control warpgroup 72, element-wise warpgroups 216).
#include "geom.cuh"
#include "tc_common.cuh"

namespace upipe {

namespace {

constexpr int kThreads = 384;
constexpr uint32_t kBoxBytes = 128 * 128;  // one TMA box: 128 rows x 64 bf16 (128 B, swizzled)

__device__ __forceinline__ bool in_range(const int4& r, int j) { return j >= r.x && j < r.w; }

// Start loading 64 fp32 columns of this thread's TMEM lane (complete after tmem_ld_wait_for).
__device__ __forceinline__ void tmem_ld64(uint32_t addr, uint32_t (&v)[64]) {
  tc::tmem_ld32(addr + 0, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
  tc::tmem_ld32(addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
}

// Wait for outstanding TMEM loads, then tie the registers of `v` to the wait so the compiler
// cannot move their uses above it (the load writes them asynchronously).
__device__ __forceinline__ void tmem_ld_wait_for(uint32_t (&v)[64]) {
  tc::tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 64; ++i) asm volatile("" : "+r"(v[i]));
}

// The MMA-issuing thread shares its SM sub-partition with two busy element-wise warps, so its
// issue path is kept short: operand descriptors are built once per buffer (kdesc / mndesc) and
// stepped by constant offsets (tc::sdesc_add).
__device__ __forceinline__ uint64_t kdesc(uint32_t saddr) { return tc::sdesc_sw128(saddr, 16, 1024); }          // K-major tile
__device__ __forceinline__ uint64_t mndesc(uint32_t saddr) { return tc::sdesc_sw128(saddr, kBoxBytes, 1024); }  // MN-major tile

template <int DH>
__device__ __forceinline__ void mma_nt(uint32_t d, uint64_t adesc, uint64_t bdesc) {  // D = A B^T, both K-major
  constexpr uint32_t kId = tc::idesc_bf16(128, 128, false, false);
  adesc = tc::opaque(adesc);
  bdesc = tc::opaque(bdesc);
#pragma unroll
  for (int k = 0; k < DH / 16; ++k) {
    const uint32_t off = (k >> 2) * kBoxBytes + (k & 3) * 32;
    tc::mma_ss(d, tc::sdesc_add(adesc, off), tc::sdesc_add(bdesc, off), kId, k > 0);
  }
}

template <int DH>
__device__ __forceinline__ void mma_acc(uint32_t d, uint32_t a_tmem, uint64_t bdesc, bool acc) {  // D (+)= A[tmem] B
  constexpr uint32_t kId = tc::idesc_bf16(128, DH, false, true);  // B [128 rows x Dh] read MN-major
  bdesc = tc::opaque(bdesc);
#pragma unroll
  for (int k = 0; k < 128 / 16; ++k) tc::mma_ts(d, a_tmem + k * 8, tc::sdesc_add(bdesc, k * 2048), kId, acc || k > 0);
}

// dS = P (dP - D) with P kept in fp32 registers (pa: columns 0-63, pb: 64-127); ndval(k)
// returns (-D[k], -D[k+1]).  dP is read 32 columns at a time and dS chunk c (bf16 pairs) written
// to columns [16c, 16c + 16), all of which earlier chunks have already read.
template <typename DFn>
__device__ __forceinline__ void ds_pass_f32(uint32_t r_addr, const uint32_t (&pa)[64], const uint32_t (&pb)[64],
                                            DFn ndval) {
  // chunk c + 1 loads while chunk c is computed and stored: its columns [32c + 32, 32c + 64) are
  // disjoint from the store's [16c, 16c + 16)
  uint32_t v[2][32];
  tc::tmem_ld32(r_addr, v[0]);
  tc::tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 32; ++i) asm volatile("" : "+r"(v[0][i]));
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t o[16];
    if (c + 1 < 4) tc::tmem_ld32(r_addr + 32 * (c + 1), v[(c + 1) & 1]);
    const uint32_t* pp = c < 2 ? &pa[32 * c] : &pb[32 * (c - 2)];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float2 d = __fadd2_rn(make_float2(__uint_as_float(v[c & 1][2 * i]), __uint_as_float(v[c & 1][2 * i + 1])),
                                  ndval(32 * c + 2 * i));
      const float2 r = __fmul2_rn(make_float2(__uint_as_float(pp[2 * i]), __uint_as_float(pp[2 * i + 1])), d);
      o[i] = tc::pack_bf16x2(r.x, r.y);
    }
    tc::tmem_st16(r_addr + 16 * c, o);
    if (c + 1 < 4) {
      tc::tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; ++i) asm volatile("" : "+r"(v[(c + 1) & 1][i]));
    }
  }
  tc::tmem_st_wait();
}

// ================================================================================================
// dQ
// ================================================================================================
template <int DH>
struct DqLayout {
  static constexpr uint32_t TB = 128 * DH * 2;
  static constexpr uint32_t Q = 0, DO = 2 * TB, KR = 4 * TB, VR = 6 * TB, BAR = 7 * TB;  // K ring 2, V 1
  static constexpr uint32_t BYTES = BAR + 256;
  static constexpr uint32_t TMEM_COLS = 512;
  __device__ static constexpr uint32_t r_col(int t) { return t * 128; }        // S / dP / dS
  __device__ static constexpr uint32_t q_col(int t) { return 256 + t * 128; }  // dQ accumulator
};

template <int DH>
__global__ void __launch_bounds__(kThreads, 1) k_attn_bwd_dq_tc(const __grid_constant__ CUtensorMap tq,
                                                                const __grid_constant__ CUtensorMap tdo,
                                                                const __grid_constant__ CUtensorMap tk,
                                                                const __grid_constant__ CUtensorMap tv,
                                                                AttnBwdArgs b) {
  using L = DqLayout<DH>;
  const AttnArgs& a = b.f;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* s_full = bars + 1;    // [2] S ready in the region
  uint64_t* s_free = bars + 3;    // [2] S consumed (P in registers)
  uint64_t* dp_full = bars + 5;   // [2]
  uint64_t* ds_full = bars + 7;   // [2]
  uint64_t* dq_full = bars + 9;   // [2]
  uint64_t* k_full = bars + 11;   // [2]
  uint64_t* k_empty = bars + 13;  // [2]
  uint64_t* v_full = bars + 15;
  uint64_t* v_empty = bars + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 17);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 18);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t S = a.S;
  const int nt = (int)ceil_div(S, kTile);
  const int64_t sp = (int64_t)nt * kTile;
  // most work first (table dispatch order), across all heads and batched devices
  const int npairs = (int)ceil_div(nt, 2);
  const int entry = a.q_order[blockIdx.y];
  const int dev = entry / npairs, pair = entry - dev * npairs;
  const int h = dev * a.hq + blockIdx.x;                                // query plane
  const int kvh = kv_shard_of(a.ring, dev) * a.hkv + blockIdx.x / a.g;  // KV plane
  const int qt0 = 2 * pair, qt1 = 2 * pair + 1;
  const bool valid1 = qt1 < nt;
  const int4 rng0 = a.q_rows[dev * nt + qt0];
  const int4 rng1 = valid1 ? a.q_rows[dev * nt + qt1] : make_int4(0, 0, 0, 0);
  // key tiles of the CTA: the union of its query tiles' ranges (a ring step's tile may have none)
  const bool has0 = rng0.x < rng0.w, has1 = valid1 && rng1.x < rng1.w;
  const int j0 = has0 && has1 ? min(rng0.x, rng1.x) : (has0 ? rng0.x : (has1 ? rng1.x : 0));
  const int j1 = has0 && has1 ? max(rng0.w, rng1.w) : (has0 ? rng0.w : (has1 ? rng1.w : 0));
  if (b.dq_acc) {
    grid_dep_trigger();
    // a ring step adds nothing to query tiles that see no key of the visiting shard (plain
    // launches always have keys: every row sees itself); the first CTA in dispatch order still
    // waits for the previous kernel of the chain, so that this grid never completes before it
    if (j0 >= j1) {
      if (blockIdx.x == 0 && blockIdx.y == 0) grid_dep_wait();
      return;
    }
  }

  if (threadIdx.x == 0) {
    tc::mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&s_full[i], 1);
      tc::mbar_init(&s_free[i], 128);
      tc::mbar_init(&dp_full[i], 1);
      tc::mbar_init(&ds_full[i], 128);
      tc::mbar_init(&dq_full[i], 1);
      tc::mbar_init(&k_full[i], 1);
      tc::mbar_init(&k_empty[i], 1);
    }
    tc::mbar_init(v_full, 1);
    tc::mbar_init(v_empty, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, L::TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 72;\n" ::: "memory");
    if (warp == 0) {
      if (lane == 0) {
        tc::prefetch_tmap(&tq);
        tc::prefetch_tmap(&tdo);
        tc::prefetch_tmap(&tk);
        tc::prefetch_tmap(&tv);
        tc::mbar_arrive_expect_tx(q_full, (valid1 ? 4 : 2) * L::TB);
        for (int at = 0; at < DH / 64; ++at) {
          tc::tma_load_3d(smem + L::Q + at * kBoxBytes, &tq, q_full, at * 64, qt0 * kTile, h);
          tc::tma_load_3d(smem + L::DO + at * kBoxBytes, &tdo, q_full, at * 64, qt0 * kTile, h);
          if (valid1) {
            tc::tma_load_3d(smem + L::Q + L::TB + at * kBoxBytes, &tq, q_full, at * 64, qt1 * kTile, h);
            tc::tma_load_3d(smem + L::DO + L::TB + at * kBoxBytes, &tdo, q_full, at * 64, qt1 * kTile, h);
          }
        }
        for (int j = j0, n = 0; j < j1; ++j, ++n) {
          // K_j into K slot n % 2 once K_{j-2} is released; V_j into the V slot once dP of V_{j-1} is done
          if (n >= 2 && !tc::mbar_wait(&k_empty[n & 1], ((n >> 1) - 1) & 1, abort_flag, a.err, a.wait_ns)) break;
          tc::mbar_arrive_expect_tx(&k_full[n & 1], L::TB);
          for (int at = 0; at < DH / 64; ++at)
            tc::tma_load_3d(smem + L::KR + (n & 1) * L::TB + at * kBoxBytes, &tk, &k_full[n & 1], at * 64, j * kTile, kvh);
          if (n >= 1 && !tc::mbar_wait(v_empty, (n - 1) & 1, abort_flag, a.err, a.wait_ns)) break;
          tc::mbar_arrive_expect_tx(v_full, L::TB);
          for (int at = 0; at < DH / 64; ++at)
            tc::tma_load_3d(smem + L::VR + at * kBoxBytes, &tv, v_full, at * 64, j * kTile, kvh);
        }
      }
      __syncwarp();
    } else if (warp == 1) {
      if (lane == 0) {
        const uint64_t dQ = kdesc(smem_u32(smem + L::Q)), dDO = kdesc(smem_u32(smem + L::DO));
        const uint64_t dK = kdesc(smem_u32(smem + L::KR)), dKmn = mndesc(smem_u32(smem + L::KR));
        const uint64_t dV = kdesc(smem_u32(smem + L::VR));
        bool ok = tc::mbar_wait(q_full, 0, abort_flag, a.err, a.wait_ns);
        const int4 rng[2] = {rng0, rng1};
        int cnt[2] = {0, 0};
        bool first[2] = {true, true};
        if (ok) {
          ok = tc::mbar_wait(&k_full[0], 0, abort_flag, a.err, a.wait_ns);
          tc::fence_after_sync();
          for (int t = 0; t < 2 && ok; ++t)
            if (in_range(rng[t], j0)) {
              mma_nt<DH>(tmem + L::r_col(t), tc::sdesc_add(dQ, t * L::TB), dK);
              tc::mma_commit(&s_full[t]);
            }
        }
        for (int j = j0, n = 0; ok && j < j1; ++j, ++n) {
          const uint64_t kb = tc::sdesc_add(dKmn, (n & 1) * L::TB);
          ok = tc::mbar_wait(v_full, n & 1, abort_flag, a.err, a.wait_ns);  // V_j
          if (!ok) break;
          tc::fence_after_sync();
          for (int t = 0; t < 2 && ok; ++t)
            if (in_range(rng[t], j)) {
              ok = tc::mbar_wait(&s_free[t], cnt[t] & 1, abort_flag, a.err, a.wait_ns);
              if (!ok) break;
              tc::fence_after_sync();
              mma_nt<DH>(tmem + L::r_col(t), tc::sdesc_add(dDO, t * L::TB), dV);  // dP = dO V^T
              tc::mma_commit(&dp_full[t]);
            }
          if (!ok) break;
          tc::mma_commit(v_empty);
          if (j + 1 < j1) {
            ok = tc::mbar_wait(&k_full[(n + 1) & 1], ((n + 1) >> 1) & 1, abort_flag, a.err, a.wait_ns);  // K_j+1
            tc::fence_after_sync();
          }
          for (int t = 0; t < 2 && ok; ++t) {
            if (in_range(rng[t], j)) {
              ok = tc::mbar_wait(&ds_full[t], cnt[t] & 1, abort_flag, a.err, a.wait_ns);
              if (!ok) break;
              ++cnt[t];
              tc::fence_after_sync();
              mma_acc<DH>(tmem + L::q_col(t), tmem + L::r_col(t), kb, !first[t]);  // dQ += dS K_j
              first[t] = false;
              if (j == rng[t].w - 1) tc::mma_commit(&dq_full[t]);
            }
            if (in_range(rng[t], j + 1)) {
              mma_nt<DH>(tmem + L::r_col(t), tc::sdesc_add(dQ, t * L::TB), tc::sdesc_add(dK, ((n + 1) & 1) * L::TB));
              tc::mma_commit(&s_full[t]);
            }
          }
          if (ok) tc::mma_commit(&k_empty[n & 1]);
        }
      }
      __syncwarp();
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 216;\n" ::: "memory");
    const int t = (warp - 4) >> 2;
    const int r = 32 * (warp & 3) + lane;
    const int4 rg = t ? rng1 : rng0;
    if (t == 0 || valid1) {
      const int64_t row = (int64_t)(t ? qt1 : qt0) * kTile + r;
      const bool row_ok = row < S;
      const bool has_keys = rg.x < rg.w;  // false only in a ring step
      int64_t vis_lo = 0, vis_hi = -1;
      if (row_ok) make_zig(a.seg, S, a.causal, a.ring, dev).q_interval(row, vis_lo, vis_hi);
      const float Dr = a.D[(int64_t)h * sp + row];
      const float lse2 = a.D[((int64_t)a.nh + h) * sp + row];
      const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
      const uint32_t r_addr = lane_addr + L::r_col(t), q_addr = lane_addr + L::q_col(t);
      const float c = a.scale * 1.4426950408889634f;
      const bool ragged = (S % kTile) != 0;
      bool ok = true;
      int cnt = 0;
      for (int j = rg.x; j < rg.w; ++j, ++cnt) {
        const bool partial = j < rg.y || j >= rg.z || (ragged && j == nt - 1);
        ok = tc::mbar_wait(&s_full[t], cnt & 1, abort_flag, a.err, a.wait_ns);
        if (!ok) break;
        tc::fence_after_sync();
        // P = exp2(s c - lse2) in fp32, in place of the scores (P only feeds dS here, so it is
        // never rounded to bf16); the second half's TMEM load overlaps the first half's math
        uint32_t sa[64], sb[64];
        {
          int lo = 0, hi = 127;
          if (partial) {
            const int64_t col0 = (int64_t)j * kTile;
            lo = (int)max((int64_t)-1, min(vis_lo - col0, (int64_t)128));
            hi = (int)max((int64_t)-1, min(vis_hi - col0, (int64_t)128));
          }
          const float2 cc = make_float2(c, c), nl = make_float2(-lse2, -lse2);
          // masked scores become -inf (exp2 -> 0) in a separate pass that only partial tiles run
          auto half = [&](uint32_t (&sv)[64], int hf) {
            if (partial) {
#pragma unroll
              for (int i = 0; i < 64; ++i)
                if (hf * 64 + i < lo || hf * 64 + i > hi) sv[i] = 0xff800000u;
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float2 arg = __ffma2_rn(make_float2(__uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1])), cc, nl);
              sv[2 * i] = __float_as_uint(fast_exp2(arg.x));
              sv[2 * i + 1] = __float_as_uint(fast_exp2(arg.y));
            }
          };
          tmem_ld64(r_addr, sa);
          tmem_ld_wait_for(sa);
          tmem_ld64(r_addr + 64, sb);
          half(sa, 0);
          tmem_ld_wait_for(sb);
          half(sb, 1);
        }
        tc::fence_before_sync();
        tc::mbar_arrive(&s_free[t]);
        ok = tc::mbar_wait(&dp_full[t], cnt & 1, abort_flag, a.err, a.wait_ns);
        if (!ok) break;
        tc::fence_after_sync();
        ds_pass_f32(r_addr, sa, sb, [&](int) { return make_float2(-Dr, -Dr); });
        tc::fence_before_sync();
        tc::mbar_arrive(&ds_full[t]);
      }
      float* accrow = b.dq_acc ? b.dq_acc + ((int64_t)h * S + (row_ok ? row : 0)) * DH : nullptr;
      // ring step: only the last step that touches this tile writes its bf16 result, and that
      // step skips the fp32 store
      const bool last = accrow && b.dq && !q_tile_touched_later(a, dev, t ? qt1 : qt0, nt);
      bf16* dqrow = (b.dq && (!accrow || last)) ? b.dq + ((int64_t)h * S + (row_ok ? row : 0)) * DH : nullptr;
      // ring step: this row's running sum, loaded while the last dS K completes (all loads in
      // flight at once)
      float4 pa[DH / 4];
      if (accrow) {
        grid_dep_wait();  // the previous ring step's sums are complete and visible
#pragma unroll
        for (int i = 0; i < DH / 4; ++i) pa[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (ok && row_ok && has_keys && !a.acc_first) {
#pragma unroll
          for (int i = 0; i < DH / 4; ++i) pa[i] = reinterpret_cast<const float4*>(accrow)[i];
        }
      }
      if (ok && has_keys) ok = tc::mbar_wait(&dq_full[t], 0, abort_flag, a.err, a.wait_ns);
      tc::fence_after_sync();
#pragma unroll
      for (int ch = 0; ch < DH / 32; ++ch) {
        uint32_t v[32];
        tc::tmem_ld32(q_addr + ch * 32, v);
        tc::tmem_ld_wait();
        if (!has_keys) {  // never in plain launches; dQ = 0 then
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;
        }
        if (accrow) {  // ring step: fold into the fp32 sum (empty tiles returned or add nothing)
          if (ok && row_ok && has_keys) {
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
              float4 o4 = pa[ch * 8 + q4];
              o4.x += __uint_as_float(v[q4 * 4 + 0]) * a.scale;
              o4.y += __uint_as_float(v[q4 * 4 + 1]) * a.scale;
              o4.z += __uint_as_float(v[q4 * 4 + 2]) * a.scale;
              o4.w += __uint_as_float(v[q4 * 4 + 3]) * a.scale;
              if (!last) *reinterpret_cast<float4*>(accrow + ch * 32 + q4 * 4) = o4;
              if (dqrow)
                *reinterpret_cast<uint2*>(dqrow + ch * 32 + q4 * 4) =
                    make_uint2(tc::pack_bf16x2(o4.x, o4.y), tc::pack_bf16x2(o4.z, o4.w));
            }
          }
        } else if (ok && row_ok) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 pkt;
            uint32_t* pw = reinterpret_cast<uint32_t*>(&pkt);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              pw[i] = tc::pack_bf16x2(__uint_as_float(v[q4 * 8 + 2 * i]) * a.scale,
                                      __uint_as_float(v[q4 * 8 + 2 * i + 1]) * a.scale);
            *reinterpret_cast<uint4*>(dqrow + ch * 32 + q4 * 8) = pkt;
          }
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

// ================================================================================================
// dK, dV
// ================================================================================================
// Adds one TMEM accumulator row (this thread's lane, DH fp32 columns, times mul) to its fp32 sum
// in global memory (or stores it there when !add), 32 columns at a time.
template <int DH>
__device__ __forceinline__ void flush_window(uint32_t acc_addr, float* row, float mul, bool store, bool add) {
#pragma unroll 1
  for (int ch = 0; ch < DH / 32; ++ch) {
    uint32_t v[32];
    tc::tmem_ld32(acc_addr + ch * 32, v);
    float4 w4[8];
#pragma unroll
    for (int q4 = 0; q4 < 8; ++q4) w4[q4] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (store && add) {
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4) w4[q4] = reinterpret_cast<const float4*>(row + ch * 32)[q4];
    }
    tc::tmem_ld_wait();
    if (store) {
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4) {
        float4 o4 = w4[q4];
        o4.x += __uint_as_float(v[q4 * 4 + 0]) * mul;
        o4.y += __uint_as_float(v[q4 * 4 + 1]) * mul;
        o4.z += __uint_as_float(v[q4 * 4 + 2]) * mul;
        o4.w += __uint_as_float(v[q4 * 4 + 3]) * mul;
        reinterpret_cast<float4*>(row + ch * 32)[q4] = o4;
      }
    }
  }
}

template <int DH>
struct DkvLayout {
  static constexpr uint32_t TB = 128 * DH * 2;
  static constexpr int NQ = 3, NO = 2;  // Q ring, dO ring
  static constexpr uint32_t K = 0, V = TB, QR = 2 * TB, OR = QR + NQ * TB, VEC = OR + NO * TB;
  static constexpr uint32_t BAR = VEC + 2 * 256 * 4;  // per element-wise group: -lse*log2e [128], -D [128]
  static constexpr uint32_t BYTES = BAR + 256;
  static constexpr uint32_t TMEM_COLS = 512;
  __device__ static constexpr uint32_t r_col(int t) { return t * 128; }  // S^T / P^T / dP^T / dS^T
  static constexpr uint32_t DK_COL = 256, DV_COL = 384;
};

template <int DH, bool FLUSH>
__global__ void __launch_bounds__(kThreads, 1) k_attn_bwd_dkdv_tc(const __grid_constant__ CUtensorMap tq,
                                                                  const __grid_constant__ CUtensorMap tdo,
                                                                  const __grid_constant__ CUtensorMap tk,
                                                                  const __grid_constant__ CUtensorMap tv,
                                                                  AttnBwdArgs b) {
  using L = DkvLayout<DH>;
  constexpr int NQ = L::NQ, NO = L::NO;
  const AttnArgs& a = b.f;
  extern __shared__ uint8_t smem_raw[];
  // this kernel uses all but ~0.7 KB of the 227 KB: no room to round the base up, so it relies on
  // the dynamic shared memory window starting 1024-byte aligned and reports otherwise
  uint8_t* smem = smem_raw;
  if (smem_u32(smem_raw) & 1023) {
    if (threadIdx.x == 0 && b.f.err) atomicCAS(b.f.err, 0, (int)UPIPE_ERR_UNSUPPORTED);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR);
  uint64_t* kv_full = bars + 0;
  uint64_t* s_full = bars + 1;    // [2] per region
  uint64_t* p_full = bars + 3;    // [2]
  uint64_t* dp_full = bars + 5;   // [2]
  uint64_t* ds_full = bars + 7;   // [2]
  uint64_t* acc_full = bars + 9;
  uint64_t* q_full = bars + 10;   // [NQ]
  uint64_t* q_empty = bars + 13;  // [NQ]
  uint64_t* o_full = bars + 16;   // [NO]
  uint64_t* o_empty = bars + 18;  // [NO]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 20);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 21);
  uint64_t* dv_tok = bars + 22;   // phase n completes once dV(n) is issued
  uint64_t* dk_tok = bars + 23;   // phase n completes once dK(n) is issued
  uint64_t* win_empty = bars + 24;  // both groups have added the window's sums to global memory

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t S = a.S;
  const int nt = (int)ceil_div(S, kTile);
  const int64_t sp = (int64_t)nt * kTile;
  // grid (KV heads, key tiles of all key shards) with the head fastest, the key tiles in the
  // table's dispatch order: the key tiles seen by the most query tiles (under causality the first
  // ones of each segment) of every head are dispatched first
  const int entry = a.kv_order[blockIdx.y];
  const int shard = entry / nt, jt = entry - shard * nt;
  const int kvh = shard * a.hkv + blockIdx.x;  // KV plane
  const int dev = dev_of_shard(a.ring, shard);  // the batched device whose queries see this shard
  const int4 tr = a.kv_rows[entry];             // query tiles {begin, full_begin, full_end, end}
  const int h_first = dev * a.hq + blockIdx.x * a.g;
  const int n_heads = dev < a.ndev ? max(0, min(a.hq, (int)blockIdx.x * a.g + a.g) - (int)blockIdx.x * a.g) : 0;
  const int nq = tr.w - tr.x;
  const int n_items = n_heads * nq;
  // windows flushed into the global fp32 sums: every full window followed by more items (FLUSH:
  // the launch has key tiles with more items than the window; the other instantiation carries
  // none of the flush's code)
  const int F = FLUSH ? b.flush_items : 0;
  const int n_win = (F > 0 && n_items > 0) ? (n_items - 1) / F : 0;
  if (a.ring.P) {
    grid_dep_trigger();
    // a ring step adds nothing to key tiles that no query of the step sees (plain launches write
    // zeros there; the first ring step has none); the first CTA in dispatch order still waits for
    // the previous kernel of the chain
    if (!a.acc_first && n_items == 0) {
      if (blockIdx.x == 0 && blockIdx.y == 0) grid_dep_wait();
      return;
    }
  }

  if (threadIdx.x == 0) {
    tc::mbar_init(kv_full, 1);
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&s_full[i], 1);
      tc::mbar_init(&p_full[i], 128);
      tc::mbar_init(&dp_full[i], 1);
      tc::mbar_init(&ds_full[i], 128);
    }
    tc::mbar_init(acc_full, n_items >= 2 ? 2 : 1);  // the last MMAs of each issuer
    tc::mbar_init(dv_tok, 1);
    tc::mbar_init(dk_tok, 1);
    tc::mbar_init(win_empty, 256);
    for (int i = 0; i < NQ; ++i) {
      tc::mbar_init(&q_full[i], 1);
      tc::mbar_init(&q_empty[i], 1);
    }
    for (int i = 0; i < NO; ++i) {
      tc::mbar_init(&o_full[i], 1);
      tc::mbar_init(&o_empty[i], 1);
    }
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, L::TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 72;\n" ::: "memory");
    if (warp == 0) {
      if (lane == 0) {
        tc::prefetch_tmap(&tq);
        tc::prefetch_tmap(&tdo);
        tc::mbar_arrive_expect_tx(kv_full, 2 * L::TB);
        for (int at = 0; at < DH / 64; ++at) {
          tc::tma_load_3d(smem + L::K + at * kBoxBytes, &tk, kv_full, at * 64, jt * kTile, kvh);
          tc::tma_load_3d(smem + L::V + at * kBoxBytes, &tv, kv_full, at * 64, jt * kTile, kvh);
        }
        for (int n = 0; n < n_items; ++n) {
          const int hh = h_first + n / nq;
          const int qi = tr.x + n % nq;
          const int sq = n % NQ, so = n % NO;
          if (n >= NQ && !tc::mbar_wait(&q_empty[sq], ((n / NQ) - 1) & 1, abort_flag, a.err, a.wait_ns)) break;
          tc::mbar_arrive_expect_tx(&q_full[sq], L::TB);
          for (int at = 0; at < DH / 64; ++at)
            tc::tma_load_3d(smem + L::QR + sq * L::TB + at * kBoxBytes, &tq, &q_full[sq], at * 64, qi * kTile, hh);
          if (n >= NO && !tc::mbar_wait(&o_empty[so], ((n / NO) - 1) & 1, abort_flag, a.err, a.wait_ns)) break;
          tc::mbar_arrive_expect_tx(&o_full[so], L::TB);
          for (int at = 0; at < DH / 64; ++at)
            tc::tma_load_3d(smem + L::OR + so * L::TB + at * kBoxBytes, &tdo, &o_full[so], at * 64, qi * kTile, hh);
        }
      }
      __syncwarp();
    } else if (warp == 1 || warp == 2) {
      // One MMA-issuing thread per element-wise group (warp 1: even items, warp 2: odd items),
      // so the two groups' waits and handshakes overlap.  The dK and dV accumulators are shared:
      // the accumulating MMA groups stay in item order across the two threads through token
      // barriers (tcgen05 fence before the arrival, fence after the wait), exactly as if one
      // thread had issued them.
      const int g = warp - 1;
      if (lane == 0 && g < n_items) {
        const uint64_t dK = kdesc(smem_u32(smem + L::K)), dV = kdesc(smem_u32(smem + L::V));
        const uint64_t dQ = kdesc(smem_u32(smem + L::QR)), dQmn = mndesc(smem_u32(smem + L::QR));
        const uint64_t dO = tc::sdesc_add(kdesc(smem_u32(smem + L::OR)), (g % NO) * L::TB);  // item n uses dO slot n % 2 == g
        const uint64_t dOmn = tc::sdesc_add(mndesc(smem_u32(smem + L::OR)), (g % NO) * L::TB);
        const uint32_t r_tm = tmem + L::r_col(g);
        bool ok = tc::mbar_wait(kv_full, 0, abort_flag, a.err, a.wait_ns);
        auto issue_st = [&](int n) {  // S^T of item n into this group's region
          if (ok) ok = tc::mbar_wait(&q_full[n % NQ], (n / NQ) & 1, abort_flag, a.err, a.wait_ns);
          if (!ok) return;
          tc::fence_after_sync();
          mma_nt<DH>(r_tm, dK, tc::sdesc_add(dQ, (n % NQ) * L::TB));
          tc::mma_commit(&s_full[g]);
        };
        issue_st(g);
        // windows of F items (FLUSH), each restarting the accumulators: the element-wise groups
        // hand the first P^T of a window over only once the previous window's sums are out
        for (int w0 = 0; ok && w0 < n_items; w0 += FLUSH ? F : n_items) {
          const int w1 = FLUSH ? min(n_items, w0 + F) : n_items;
          for (int n = w0 + g; ok && n < w1; n += 2) {
            const uint32_t ph = (n >> 1) & 1;
            // the waits that are normally already satisfied come first, so that the issue of dV
            // follows the element-wise group's P^T arrival as closely as possible
            ok = tc::mbar_wait(&o_full[g], (n / NO) & 1, abort_flag, a.err, a.wait_ns);
            if (ok && n > 0) ok = tc::mbar_wait(dv_tok, (n - 1) & 1, abort_flag, a.err, a.wait_ns);  // dV(n-1) issued
            const bool acc_in = n > w0;  // the window's first item restarts the accumulators
            if (ok) ok = tc::mbar_wait(&p_full[g], ph, abort_flag, a.err, a.wait_ns);
            if (!ok) break;
            tc::fence_after_sync();
            mma_acc<DH>(tmem + L::DV_COL, r_tm, dOmn, acc_in);  // dV += P^T dO
            tc::fence_before_sync();
            tc::mbar_arrive(dv_tok);
            mma_nt<DH>(r_tm, dV, dO);  // dP^T = V dO^T
            tc::mma_commit(&dp_full[g]);
            tc::mma_commit(&o_empty[g]);
            if (n > 0) ok = tc::mbar_wait(dk_tok, (n - 1) & 1, abort_flag, a.err, a.wait_ns);  // dK(n-1) issued
            if (ok) ok = tc::mbar_wait(&ds_full[g], ph, abort_flag, a.err, a.wait_ns);
            if (!ok) break;
            tc::fence_after_sync();
            mma_acc<DH>(tmem + L::DK_COL, r_tm, tc::sdesc_add(dQmn, (n % NQ) * L::TB), acc_in);  // dK += dS^T Q
            tc::fence_before_sync();
            tc::mbar_arrive(dk_tok);
            tc::mma_commit(&q_empty[n % NQ]);
            if (n + 2 >= n_items) tc::mma_commit(acc_full);  // this issuer's last item
            if (n + 2 < n_items) issue_st(n + 2);
          }
        }
      }
      __syncwarp();
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 216;\n" ::: "memory");
    const int grp = (warp - 4) >> 2;       // element-wise group: items n with n % 2 == grp
    const int r = 32 * (warp & 3) + lane;  // key row within the tile == TMEM lane
    const int64_t krow = (int64_t)jt * kTile + r;
    const bool k_ok = krow < S;
    // the queries that see this key: [vis_lo, vis_hi]
    int64_t vis_lo = 0, vis_hi = -1;
    if (k_ok) make_zig(a.seg, S, a.causal, a.ring, dev).k_interval(krow, vis_lo, vis_hi);
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const uint32_t r_addr = lane_addr + L::r_col(grp);
    float* nvec = reinterpret_cast<float*>(smem + L::VEC) + grp * 256;  // this group's -lse2 | -D
    const float c = a.scale * 1.4426950408889634f;
    const bool ragged = (S % kTile) != 0;
    bool ok = true;
    // -lse*log2e and -D of query r of item n (one value pair per thread), loaded one item ahead
    auto load_vec = [&](int n) {
      const int64_t qoff = (int64_t)(tr.x + n % nq) * kTile + r;
      const int hh = h_first + n / nq;
      return make_float2(-a.D[((int64_t)a.nh + hh) * sp + qoff], -a.D[(int64_t)hh * sp + qoff]);
    };
    float2 vec_next = grp < n_items ? load_vec(grp) : make_float2(0.f, 0.f);
    // Ping-pong: the groups take turns phase by phase (P of items n and n+1, then dS of both),
    // so one group's element-wise work overlaps the tensor core's work on the other's item.
    // Group grp waits for its turn at named barrier kPing + grp (ids 1 and 2 stage lse/D).
    constexpr int kPing = 3;
    const int n_pp = 2 * min((n_items + 1) / 2, n_items / 2);
    const int n_give = grp == 0 ? n_pp : n_pp - 1;
    if (grp == 1 && n_pp > 0) tc::named_bar_arrive(kPing + 0, 256);
    int turn = 0;
    auto take_turn = [&]() { if (turn < n_pp) tc::named_bar_sync(kPing + grp, 256); };
    auto give_turn = [&]() {
      if (turn < n_give) tc::named_bar_arrive(kPing + 1 - grp, 256);
      ++turn;
    };
    for (int n = grp; n < n_items;) {
      // this group's items up to the end of the current window (all of them when no flush
      // follows), so that the per-item loop carries none of the flush
      const int Fd = FLUSH ? F : 1;  // F as a divisor (the other instantiation never divides)
      const bool flush = F > 0 && n / Fd < n_win;
      const int w_end = flush ? (n / Fd + 1) * F : n_items;
      for (; n < w_end; n += 2) {
        const int qi = tr.x + n % nq;
        const bool partial = qi < tr.y || qi >= tr.z || (ragged && (qi == nt - 1 || jt == nt - 1));
        const int cyc = (n >> 1) & 1;
        int lo = 0, hi = 127;
        if (partial) {
          const int64_t col0 = (int64_t)qi * kTile;
          lo = (int)max((int64_t)-1, min(vis_lo - col0, (int64_t)128));
          hi = (int)max((int64_t)-1, min(vis_hi - col0, (int64_t)128));
        }
        // stage the item's 128 (-lse2, -D) pairs in shared memory, then start the next item's loads
        tc::named_bar_sync(1 + grp, 128);  // the previous item's readers are done
        nvec[r] = vec_next.x;
        nvec[128 + r] = vec_next.y;
        tc::named_bar_sync(1 + grp, 128);
        if (n + 2 < n_items) vec_next = load_vec(n + 2);
        take_turn();
        ok = tc::mbar_wait(&s_full[grp], cyc, abort_flag, a.err, a.wait_ns);
        if (!ok) break;
        tc::fence_after_sync();
        // P^T = exp2(s c - lse2) kept in fp32 in place of the scores (for dS^T); its bf16 copy goes
        // to TMEM as the A operand of dV += P^T dO
        uint32_t sa[64], sb[64];
        {
          const float2 cc = make_float2(c, c);
          // two halves of 64 columns, the second loading while the first is computed (as in dQ)
          auto half = [&](uint32_t (&sv)[64], int hf) {
            if (partial) {  // masked scores -> -inf (exp2 -> 0), only on partial tiles
#pragma unroll
              for (int i = 0; i < 64; ++i)
                if (hf * 64 + i < lo || hf * 64 + i > hi) sv[i] = 0xff800000u;
            }
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float4 l4 = *reinterpret_cast<const float4*>(nvec + hf * 64 + 2 * i);
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                const int kk = 2 * (i + u);
                const float2 arg = __ffma2_rn(make_float2(__uint_as_float(sv[kk]), __uint_as_float(sv[kk + 1])), cc,
                                              u ? make_float2(l4.z, l4.w) : make_float2(l4.x, l4.y));
                sv[kk] = __float_as_uint(fast_exp2(arg.x));
                sv[kk + 1] = __float_as_uint(fast_exp2(arg.y));
              }
            }
          };
          tmem_ld64(r_addr, sa);
          tmem_ld_wait_for(sa);
          tmem_ld64(r_addr + 64, sb);
          half(sa, 0);
          tmem_ld_wait_for(sb);
          half(sb, 1);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // bf16 pairs of columns [32q, 32q + 32) -> TMEM columns [16q, 16q + 16)
          const uint32_t* pp = q < 2 ? &sa[32 * q] : &sb[32 * (q - 2)];
          uint32_t o[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] = tc::pack_bf16x2(__uint_as_float(pp[2 * i]), __uint_as_float(pp[2 * i + 1]));
          tc::tmem_st16(r_addr + 16 * q, o);
        }
        tc::tmem_st_wait();
        tc::fence_before_sync();
        tc::mbar_arrive(&p_full[grp]);
        give_turn();
        take_turn();
        ok = tc::mbar_wait(&dp_full[grp], cyc, abort_flag, a.err, a.wait_ns);
        if (!ok) break;
        tc::fence_after_sync();
        ds_pass_f32(r_addr, sa, sb, [&](int k) { return *reinterpret_cast<const float2*>(nvec + 128 + k); });
        tc::fence_before_sync();
        tc::mbar_arrive(&ds_full[grp]);
        give_turn();
      }
      if (!ok) break;
      if (flush) {
        // the window's last items are done: add this group's accumulator (group 0 dK, group 1 dV)
        // to the global fp32 sum, 32 columns at a time
        const int w = w_end / Fd - 1;
        float* wrow = (grp == 0 ? b.dk_acc : b.dv_acc) + ((int64_t)kvh * S + (k_ok ? krow : 0)) * DH;
        if (a.ring.P) grid_dep_wait();  // the previous ring step's sums are complete and visible
        // the window's last two items (one per issuer) are complete once their dK MMAs have
        // released their Q slots (each issuer's commit covers its earlier MMAs; no later phase of
        // these barriers can complete before this group hands over its next item)
        const int m0 = w_end - 2, m1 = w_end - 1;
        ok = tc::mbar_wait(&q_empty[m0 % NQ], (m0 / NQ) & 1, abort_flag, a.err, a.wait_ns);
        if (ok) ok = tc::mbar_wait(&q_empty[m1 % NQ], (m1 / NQ) & 1, abort_flag, a.err, a.wait_ns);
        tc::fence_after_sync();
        // the first ring step starts the sums (nothing to add to), later flushes add to them
        flush_window<DH>(lane_addr + (grp == 0 ? L::DK_COL : L::DV_COL), wrow, grp == 0 ? a.scale : 1.f, ok && k_ok,
                         !(a.acc_first && w == 0));
        tc::fence_before_sync();
        tc::mbar_arrive(win_empty);
        // group 0 hands the next window's first P^T (whose dV MMA restarts the accumulators) over
        // only once both groups' sums are out
        if (grp == 0 && ok) ok = tc::mbar_wait(win_empty, w & 1, abort_flag, a.err, a.wait_ns);
        tc::fence_after_sync();
        if (!ok) break;
      }
    }
    // after an abort, hand over the turns still owed so the other group never blocks on them
    for (int k = turn; k < n_give; ++k) tc::named_bar_arrive(kPing + 1 - grp, 256);
    // epilogue: group 0 writes dK rows (scaled), group 1 writes dV rows.  Ring steps: the fp32 sum
    // is not stored by the last step that touches the key tile (with the shards the launch's own
    // at every step; otherwise by the ring's last step) and only that step writes the bf16 result.
    const bool last = a.ring.P && b.dk_out && b.dv_out &&
                      (a.kv_last_touch ? !kv_tile_touched_later(a, shard, jt, nt) : a.acc_last != 0);
    const uint32_t acc_addr = lane_addr + (grp == 0 ? L::DK_COL : L::DV_COL);
    const float mul = grp == 0 ? a.scale : 1.f;
    const int64_t off = ((int64_t)kvh * S + (k_ok ? krow : 0)) * DH;
    // fp32 sums: this row's running sum, loaded while the last MMAs complete (all loads in flight
    // at once)
    float4 pa[DH / 4];
    if (b.acc_kv) {
      if (a.ring.P) grid_dep_wait();  // the previous ring step's sums are complete and visible
#pragma unroll
      for (int i = 0; i < DH / 4; ++i) pa[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (ok && k_ok && (!a.acc_first || n_win > 0)) {
        const float4* src = reinterpret_cast<const float4*>((grp == 0 ? b.dk_acc : b.dv_acc) + off);
#pragma unroll
        for (int i = 0; i < DH / 4; ++i) pa[i] = src[i];
      }
    }
    if (ok && n_items > 0) ok = tc::mbar_wait(acc_full, 0, abort_flag, a.err, a.wait_ns);
    tc::fence_after_sync();
#pragma unroll
    for (int ch = 0; ch < DH / 32; ++ch) {
      uint32_t v[32];
      tc::tmem_ld32(acc_addr + ch * 32, v);
      tc::tmem_ld_wait();
      if (n_items == 0) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0u;
      }
      if (ok && k_ok) {
        if (b.acc_kv) {
          // fp32 sums over a partial KV group's chunks or over the ring's steps; a ring step also
          // leaves the running sum rounded to bf16 if asked
          float* dst = (grp == 0 ? b.dk_acc : b.dv_acc) + off + ch * 32;
          bf16* out = grp == 0 ? b.dk_out : b.dv_out;
          if (out && !(last || !a.kv_last_touch)) out = nullptr;  // written by a later step
          if (out) out += off + ch * 32;
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            float4 o4 = pa[ch * 8 + q4];
            o4.x += __uint_as_float(v[q4 * 4 + 0]) * mul;
            o4.y += __uint_as_float(v[q4 * 4 + 1]) * mul;
            o4.z += __uint_as_float(v[q4 * 4 + 2]) * mul;
            o4.w += __uint_as_float(v[q4 * 4 + 3]) * mul;
            if (!last) *reinterpret_cast<float4*>(dst + q4 * 4) = o4;
            if (out)
              *reinterpret_cast<uint2*>(out + q4 * 4) = make_uint2(tc::pack_bf16x2(o4.x, o4.y), tc::pack_bf16x2(o4.z, o4.w));
          }
        } else {
          bf16* dst = (grp == 0 ? b.dk : b.dv) + off + ch * 32;
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 pkt;
            uint32_t* pw = reinterpret_cast<uint32_t*>(&pkt);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              pw[i] = tc::pack_bf16x2(__uint_as_float(v[q4 * 8 + 2 * i]) * mul, __uint_as_float(v[q4 * 8 + 2 * i + 1]) * mul);
            *reinterpret_cast<uint4*>(dst + q4 * 8) = pkt;
          }
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

template <int DH>
bool make_maps(const AttnArgs& a, CUtensorMap* tq, CUtensorMap* tdo, CUtensorMap* tk, CUtensorMap* tv) {
  return make_tmap_3d_bf16(tq, a.q, DH, a.S, a.nh, 64, 128) && make_tmap_3d_bf16(tdo, a.dO, DH, a.S, a.nh, 64, 128) &&
         make_tmap_3d_bf16(tk, a.k, DH, a.S, a.nkv, 64, 128) && make_tmap_3d_bf16(tv, a.v, DH, a.S, a.nkv, 64, 128);
}

template <typename KFN>
cudaError_t launch(KFN kfn, size_t bytes, dim3 grid, const CUtensorMap& tq, const CUtensorMap& tdo,
                   const CUtensorMap& tk, const CUtensorMap& tv, const AttnBwdArgs& b, cudaStream_t st) {
  // at least 120 KB so that two CTAs never share an SM (each takes all 512 TMEM columns)
  const size_t smem = bytes > 120 * 1024 ? bytes : 120 * 1024;
  cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  AttnBwdArgs args = b;
  fill_planes(args.f);
  args.f.wait_ns = wait_limit_ns();
  if (args.f.pdl) {
    e = launch_pdl(kfn, grid, dim3(kThreads), smem, st, tq, tdo, tk, tv, args);
  } else {
    kfn<<<grid, kThreads, smem, st>>>(tq, tdo, tk, tv, args);
    e = cudaGetLastError();
  }
  note_launch();
  return e;
}

template <int DH>
cudaError_t run_dq(const AttnBwdArgs& b, cudaStream_t st) {
  CUtensorMap tq, tdo, tk, tv;
  if (!make_maps<DH>(b.f, &tq, &tdo, &tk, &tv)) return cudaErrorInvalidValue;
  const int nt = (int)ceil_div(b.f.S, kTile);
  AttnArgs f = b.f;
  fill_planes(f);
  return launch(k_attn_bwd_dq_tc<DH>, DqLayout<DH>::BYTES + 1024,
                dim3((unsigned)f.hq, (unsigned)(f.ndev * ceil_div(nt, 2))), tq, tdo, tk, tv, b, st);
}

template <int DH>
cudaError_t run_dkdv(const AttnBwdArgs& b, cudaStream_t st) {
  CUtensorMap tq, tdo, tk, tv;
  if (!make_maps<DH>(b.f, &tq, &tdo, &tk, &tv)) return cudaErrorInvalidValue;
  const int nt = (int)ceil_div(b.f.S, kTile);
  AttnArgs f = b.f;
  fill_planes(f);
  // a key tile has at most min(g, hq) x nt work items (the launch's query heads of its KV head x
  // the query tiles)
  const bool flush = b.acc_kv && b.flush_items > 0 && (int64_t)std::min(f.g, f.hq) * nt > b.flush_items;
  const dim3 grid((unsigned)f.hkv, (unsigned)(f.kv_count * nt));
  return flush ? launch(k_attn_bwd_dkdv_tc<DH, true>, DkvLayout<DH>::BYTES, grid, tq, tdo, tk, tv, b, st)
               : launch(k_attn_bwd_dkdv_tc<DH, false>, DkvLayout<DH>::BYTES, grid, tq, tdo, tk, tv, b, st);
}

}  // namespace

cudaError_t launch_attn_bwd_dq(const AttnBwdArgs& b, int head_dim, cudaStream_t st) {
  return head_dim == 64 ? run_dq<64>(b, st) : run_dq<128>(b, st);
}
cudaError_t launch_attn_bwd_dkdv(const AttnBwdArgs& b, int head_dim, cudaStream_t st) {
  return head_dim == 64 ? run_dkdv<64>(b, st) : run_dkdv<128>(b, st);
}

}  // namespace upipe
