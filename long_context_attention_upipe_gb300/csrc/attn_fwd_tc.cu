// Flash-style attention forward on the 5th-generation tensor cores (tcgen05, TMEM, TMA).
//
// Per head, softmax(Q K^T * scale + M) V over the whole sequence with online softmax (podcast
// summary "Road to 5 Million Tokens", chapter on DeepSpeed Ulysses: each GPU computes whole
// heads, so flash attention applies).  Key tiles come from the skip table (MaxText article,
// Splash attention paragraph): tiles outside a query tile's range are never loaded, full tiles
// run unmasked, partial tiles and the ragged last tile apply the causal / segment mask.  With
// contiguous segments a query row sees one interval of keys, so the mask of a partial tile is
// two integer compares per element.
//
// One CTA = one head x two 128-row query tiles (a, b), 12 warps (warp 3 idle):
//   warp 0     TMA producer: Q_a, Q_b once, then K_j, V_j, K_j+1, ... through a ring of
//              tile-sized slots; a slot is refilled once both MMA issuers have released it
//   warps 1, 2 MMA issuers (one thread each), one per query tile: S_t = Q_t K^T (both operands
//              in shared memory), O_t += P_t V (P_t read from TMEM, V from shared memory); two
//              independent streams keep the tensor pipe fed; warp 1 owns the TMEM allocation
//   warps 4-7  softmax of tile a, warps 8-11 softmax of tile b: each thread owns one query row
//              (TMEM lane 32 * (warp % 4) + lane): row max, exp2, row sum, P written back over
//              S as bf16, all from one TMEM read of the row.  On the key tiles both query tiles
//              see, the two groups take turns (named-barrier ping-pong), so one group's softmax
//              overlaps the tensor core's work on the other tile.
// TMEM columns: S/P_a [0,128) S/P_b [128,256) O_a [256,256+Dh) O_b [256+Dh, 256+2Dh).
// While one softmax group works, the tensor core runs the other tile's P V and next Q K^T.
// The softmax offset is optimistic: the first tile with a visible key sets it to that tile's row
// maximum and later tiles reuse it without computing their maximum; only when a tile's row sum of P
// exceeds 2^16 (a score outgrew the offset by 16 in exp2 units) is the offset moved to the true
// maximum, O and l rescaled and the tile's P redone.  Every P stays <= 2^16, so O and l stay far from
// fp32 overflow, and O / l does not depend on the offset.
//
// MODE 1 (activation recompute for the backward pass): P = exp2(S*scale*log2e - lse*log2e)
// from the saved log-sum-exp, no rescaling; the epilogue also writes D = rowsum(dO * O).
// MODE 2 (one step of the zigzag ring, all batched devices in one launch): MODE 0's softmax,
// with the epilogue folding the block's (O, lse) into the fp32 running output and lse
// (L = log(e^L_acc + e^L_b), O = (e^L_acc O_acc + e^L_b O_b) / e^L); query tiles that see no key
// of the visiting shard are left alone.
#include "geom.cuh"
#include "tc_common.cuh"

namespace upipe {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kFwdThreads = 384;
constexpr uint32_t kBoxBytes = 128 * 128;  // one TMA box: 128 rows x 64 bf16 (128 B, swizzled)

template <int DH>
struct FwdLayout {
  static constexpr uint32_t TB = 128 * DH * 2;     // one 128-row tile of Q, K or V
  static constexpr int NSLOT = DH == 128 ? 5 : 8;  // K/V ring slots
  static constexpr uint32_t Q = 0, RING = 2 * TB, BAR = RING + NSLOT * TB;
  static constexpr uint32_t BYTES = BAR + 512;     // + 1024 alignment slack at launch
  static constexpr uint32_t TMEM_COLS = 512;
  __device__ static constexpr uint32_t s_col(int t) { return t * 128; }
  __device__ static constexpr uint32_t o_col(int t) { return 256 + t * DH; }
};

__device__ __forceinline__ bool in_range(const int4& r, int j) { return j >= r.x && j < r.w; }

// Launched with 168 registers per thread (12 warps, 3 per SM sub-partition of 16K registers).
// The control warpgroup then drops to 72 and the two softmax warpgroups rise to 216: per
// sub-partition 72 + 216 + 216 = 504 <= 512 per lane, per CTA 64,512 = the launch's 384 x 168.
template <int DH, int MODE>
__global__ void __launch_bounds__(kFwdThreads, 1)
    k_attn_fwd_tc(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, AttnArgs a) {
  using L = FwdLayout<DH>;
  constexpr int NS = L::NSLOT;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* s_full = bars + 1;           // [2] per query tile
  uint64_t* p_full = bars + 3;           // [2]
  uint64_t* o_full = bars + 5;           // [2]
  uint64_t* slot_full = bars + 7;        // [NS]
  uint64_t* slot_empty = bars + 7 + NS;  // [NS]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 7 + 2 * NS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 8 + 2 * NS);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t S = a.S;
  const int nt = (int)ceil_div(S, kTile);
  // grid (heads, query-tile pairs of all batched devices) with the head fastest, the pairs in the
  // table's dispatch order, so the CTAs are dispatched most work first across all heads (a late
  // long CTA would leave the others idle at the end); with packed segments the work depends on
  // the position in the segment
  const int npairs = (int)ceil_div(nt, 2);
  const int entry = a.q_order[blockIdx.y];
  const int dev = entry / npairs, pair = entry - dev * npairs;
  const int h = dev * a.hq + blockIdx.x;                            // query plane
  const int kvh = kv_shard_of(a.ring, dev) * a.hkv + blockIdx.x / a.g;  // KV plane
  const int qt0 = 2 * pair, qt1 = 2 * pair + 1;
  const bool valid1 = qt1 < nt;
  const int4 rng0 = a.q_rows[dev * nt + qt0];
  const int4 rng1 = valid1 ? a.q_rows[dev * nt + qt1] : make_int4(0, 0, 0, 0);
  // key tiles of the CTA: the union of its query tiles' ranges (a ring step's tile may have none)
  const bool has0 = rng0.x < rng0.w, has1 = valid1 && rng1.x < rng1.w;
  const int j0 = has0 && has1 ? min(rng0.x, rng1.x) : (has0 ? rng0.x : (has1 ? rng1.x : 0));
  const int j1 = has0 && has1 ? max(rng0.w, rng1.w) : (has0 ? rng0.w : (has1 ? rng1.w : 0));
  if (MODE == 2) {
    grid_dep_trigger();
    // a ring step adds nothing to query tiles that see no key of the visiting shard (plain
    // launches always have keys: every row sees itself).  The first CTA in dispatch order waits
    // for the previous step even then, so that this grid never completes before it.
    if (j0 >= j1) {
      if (blockIdx.x == 0 && blockIdx.y == 0) grid_dep_wait();
      return;
    }
  }

  if (threadIdx.x == 0) {
    tc::mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&s_full[i], 1);
      tc::mbar_init(&p_full[i], 128);
      tc::mbar_init(&o_full[i], 1);
    }
    for (int i = 0; i < NS; ++i) {
      tc::mbar_init(&slot_full[i], 1);
      tc::mbar_init(&slot_empty[i], valid1 ? 2 : 1);  // released by each MMA issuer
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
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tc::prefetch_tmap(&tq);
      tc::prefetch_tmap(&tk);
      tc::prefetch_tmap(&tv);
      tc::mbar_arrive_expect_tx(q_full, (valid1 ? 2 : 1) * L::TB);
      for (int at = 0; at < DH / 64; ++at) {
        tc::tma_load_3d(smem + L::Q + at * kBoxBytes, &tq, q_full, at * 64, qt0 * kTile, h);
        if (valid1) tc::tma_load_3d(smem + L::Q + L::TB + at * kBoxBytes, &tq, q_full, at * 64, qt1 * kTile, h);
      }
      // item 2n = K of the n-th key tile, item 2n+1 = its V
      const int n_items = 2 * (j1 - j0);
      for (int it = 0; it < n_items; ++it) {
        const int sl = it % NS;
        if (it >= NS && !tc::mbar_wait(&slot_empty[sl], ((it / NS) - 1) & 1, abort_flag, a.err, a.wait_ns)) break;
        tc::mbar_arrive_expect_tx(&slot_full[sl], L::TB);
        const CUtensorMap* map = (it & 1) ? &tv : &tk;
        const int row = (j0 + (it >> 1)) * kTile;
        for (int at = 0; at < DH / 64; ++at)
          tc::tma_load_3d(smem + L::RING + sl * L::TB + at * kBoxBytes, map, &slot_full[sl], at * 64, row, kvh);
      }
    }
    __syncwarp();
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------------ MMA issuers
    // One issuing thread per query tile (warp 1: tile a, warp 2: tile b), so the two tiles' MMA
    // streams are independent and the tensor pipe takes whichever is ready.  Both walk all key
    // tiles of the CTA and release every K/V slot (the slot barriers count one arrival per
    // issuer).  The issue path is lean: descriptors are built once and stepped by constant
    // offsets, ring slots and phases are tracked incrementally.
    const int t = warp - 1;
    if (lane == 0 && (t == 0 || valid1)) {
      constexpr uint32_t kIdS = tc::idesc_bf16(128, 128, false, false);
      constexpr uint32_t kIdO = tc::idesc_bf16(128, DH, false, true);
      const uint32_t sQ = smem_u32(smem + L::Q), sR = smem_u32(smem + L::RING);
      const uint64_t dQt = tc::sdesc_add(tc::sdesc_sw128(sQ, 16, 1024), t * L::TB);  // Q_t, K-major
      const uint64_t dK = tc::sdesc_sw128(sR, 16, 1024);           // ring slot 0 read as K (K-major)
      const uint64_t dV = tc::sdesc_sw128(sR, kBoxBytes, 1024);    // ring slot 0 read as V (MN-major)
      const uint32_t s_tm = tmem + L::s_col(t), o_tm = tmem + L::o_col(t);
      const int4 rg = t ? rng1 : rng0;
      bool ok = tc::mbar_wait(q_full, 0, abort_flag, a.err, a.wait_ns);
      struct Pos { int slot; uint32_t phase; };
      auto next = [](Pos p) { return p.slot + 1 == NS ? Pos{0, p.phase ^ 1u} : Pos{p.slot + 1, p.phase}; };
      auto wait_item = [&](Pos p) {
        if (ok) ok = tc::mbar_wait(&slot_full[p.slot], p.phase, abort_flag, a.err, a.wait_ns);
        tc::fence_after_sync();
      };
      auto issue_s = [&](int slot) {
        const uint64_t kd = tc::opaque(tc::sdesc_add(dK, slot * L::TB));
#pragma unroll
        for (int k = 0; k < DH / 16; ++k) {
          const uint32_t off = (k >> 2) * kBoxBytes + (k & 3) * 32;
          tc::mma_ss(s_tm, tc::sdesc_add(dQt, off), tc::sdesc_add(kd, off), kIdS, k > 0);
        }
        tc::mma_commit(&s_full[t]);
      };
      auto issue_pv = [&](int slot, bool first) {
        const uint64_t vd = tc::opaque(tc::sdesc_add(dV, slot * L::TB));
#pragma unroll
        for (int k = 0; k < 128 / 16; ++k)
          tc::mma_ts(o_tm, s_tm + k * 8, tc::sdesc_add(vd, k * 2048), kIdO, (!first) || k > 0);
      };
      int cnt_p = 0;
      bool first_pv = true;
      Pos kpos{0, 0u};  // ring position of K_j (item 2n); V_j follows it, then K_j+1
      if (ok) {
        wait_item(kpos);
        if (ok && in_range(rg, j0)) issue_s(kpos.slot);
        if (ok) tc::mma_commit(&slot_empty[kpos.slot]);
      }
      for (int j = j0; ok && j < j1; ++j) {
        const Pos vpos = next(kpos), knext = next(vpos);
        wait_item(vpos);                       // V_j
        if (j + 1 < j1) wait_item(knext);      // K_j+1
        if (!ok) break;
        if (in_range(rg, j)) {
          ok = tc::mbar_wait(&p_full[t], cnt_p & 1, abort_flag, a.err, a.wait_ns);
          if (!ok) break;
          ++cnt_p;
          tc::fence_after_sync();
          issue_pv(vpos.slot, first_pv);
          first_pv = false;
          if (j == rg.w - 1) tc::mma_commit(&o_full[t]);
        }
        tc::mma_commit(&slot_empty[vpos.slot]);                   // V_j released by this issuer
        if (in_range(rg, j + 1)) issue_s(knext.slot);
        if (j + 1 < j1) tc::mma_commit(&slot_empty[knext.slot]);  // K_j+1 released by this issuer
        kpos = knext;
      }
    }
    __syncwarp();
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 216;\n" ::: "memory");
    // ------------------------------------------------------------------ softmax groups
    const int t = (warp - 4) >> 2;
    const int r = 32 * (warp & 3) + lane;  // row within the tile == TMEM lane this warp may access
    const int4 rg = t ? rng1 : rng0;
    if (t == 0 || valid1) {
      const int64_t row = (int64_t)(t ? qt1 : qt0) * kTile + r;
      const bool row_ok = row < S;
      const bool has_keys = rg.x < rg.w;  // false only in a ring step
      // the keys this row sees: [vis_lo, vis_hi] (empty for rows past the end)
      int64_t vis_lo = 0, vis_hi = -1;
      if (row_ok) make_zig(a.seg, S, a.causal, a.ring, dev).q_interval(row, vis_lo, vis_hi);
      const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
      const uint32_t s_addr = lane_addr + L::s_col(t), o_addr = lane_addr + L::o_col(t);
      const float c = a.scale * kLog2e;
      const bool ragged = (S % kTile) != 0;
      float m_used = -INFINITY, l = 0.f;
      if (MODE == 1) m_used = row_ok ? a.lse[(int64_t)h * S + row] * kLog2e : 0.f;
      // Ping-pong: on the key tiles that both query tiles see, the two softmax groups take turns
      // (a then b on each key tile), so one group's softmax overlaps the tensor core's work on
      // the other tile instead of both competing for the same issue slots.  Named barrier
      // kPing + t is where group t waits for its turn; the other group's arrival grants it.
      // Turns pair the same key tile in both groups, so the shared K/V ring never waits on a
      // group that is waiting for its turn (on other key tiles the groups run free).
      constexpr int kPing = 3;
      const int pp_lo = max(rng0.x, rng1.x), pp_hi = valid1 ? min(rng0.w, rng1.w) : pp_lo;
      const int n_pp = max(0, pp_hi - pp_lo);       // shared key tiles: one turn each per group
      const int n_give = t == 0 ? n_pp : n_pp - 1;  // turns this group hands over inside the loop
      if (t == 1 && n_pp > 0) tc::named_bar_arrive(kPing + 0, 256);
      int turn = 0;
      bool ok = true;
      int cnt = 0;
      for (int j = rg.x; j < rg.w; ++j, ++cnt) {
        const bool partial = j < rg.y || j >= rg.z || (ragged && j == nt - 1);
        const bool pp = j >= pp_lo && j < pp_hi;
        if (pp) tc::named_bar_sync(kPing + t, 256);
        ok = tc::mbar_wait(&s_full[t], cnt & 1, abort_flag, a.err, a.wait_ns);
        if (!ok) break;
        tc::fence_after_sync();
        uint32_t sv[128];
        tc::tmem_ld32(s_addr + 0, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
        tc::tmem_ld32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
        tc::tmem_ld32(s_addr + 64, *reinterpret_cast<uint32_t(*)[32]>(&sv[64]));
        tc::tmem_ld32(s_addr + 96, *reinterpret_cast<uint32_t(*)[32]>(&sv[96]));
        tc::tmem_ld_wait();
        if (partial) {
          const int64_t col0 = (int64_t)j * kTile;
          const int lo = (int)max((int64_t)-1, min(vis_lo - col0, (int64_t)128));
          const int hi = (int)max((int64_t)-1, min(vis_hi - col0, (int64_t)128));
#pragma unroll
          for (int k = 0; k < 128; ++k)
            if (k < lo || k > hi) sv[k] = 0xff800000u;  // -inf
        }
        float f = 1.f;
        bool rescale_o = false;
        // row maximum of the tile's (masked) scores, in exp2 units
        auto row_max = [&]() {
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int k = 0; k < 128; k += 2)
            m4[(k >> 1) & 3] = fmax3(m4[(k >> 1) & 3], __uint_as_float(sv[k]), __uint_as_float(sv[k + 1]));
          return fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * c;
        };
        // The offset only has to keep P in range: O / l is the same for any offset.  The first
        // tile with a visible key sets it to that tile's maximum; later tiles reuse it and their
        // P's row sum tells whether a score outgrew it (below).
        if (MODE != 1 && m_used == -INFINITY) m_used = row_max();  // stays -inf if all masked
        float mu = m_used == -INFINITY ? 0.f : m_used;
        // P = exp2(s * c - mu) as bf16 pairs into the first 64 columns of S (already read)
        float lt;
        auto exp_store = [&]() {
          float2 l2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
          const float2 cc = make_float2(c, c), nmu = make_float2(-mu, -mu);
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            uint32_t pk[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float2 arg = __ffma2_rn(
                  make_float2(__uint_as_float(sv[hf * 64 + 2 * i]), __uint_as_float(sv[hf * 64 + 2 * i + 1])), cc, nmu);
              const float2 p = make_float2(fast_exp2(arg.x), fast_exp2(arg.y));
              l2[i & 1] = __fadd2_rn(l2[i & 1], p);
              pk[i] = tc::pack_bf16x2(p.x, p.y);
            }
            tc::tmem_st32(s_addr + hf * 32, pk);
          }
          lt = (l2[0].x + l2[0].y) + (l2[1].x + l2[1].y);
        };
        exp_store();
        if (MODE != 1) {
          // A row sum above 2^16 (or inf) means some P exceeded 2^16: move the offset to the true
          // maximum, rescale the running O and l, and redo the tile's P (rare: the scores have to
          // outgrow the first visible tile's maximum by 16 in exp2 units).  P <= 2^16 keeps O and
          // l far from fp32 overflow, and bf16 P has the same relative precision at any size.
          const bool redo = !(lt <= 65536.f);
          if (__any_sync(0xffffffffu, redo)) {  // warp-uniform: the TMEM stores are collective
            if (redo) {
              const float mx = fmaxf(m_used, row_max());
              rescale_o = cnt > 0;
              f = fast_exp2(m_used - mx);
              m_used = mx;
              mu = mx;
            }
            tc::tmem_st_wait();
            exp_store();
          }
        }
        tc::tmem_st_wait();
        if (MODE != 1 && __any_sync(0xffffffffu, rescale_o)) {
          // O_t is idle here: P V of the previous tile completed before this S was ready, and
          // this tile's P V waits for the arrival below
#pragma unroll
          for (int ch = 0; ch < DH / 32; ++ch) {
            uint32_t v[32];
            tc::tmem_ld32(o_addr + ch * 32, v);
            tc::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * f);
            tc::tmem_st32(o_addr + ch * 32, v);
          }
          tc::tmem_st_wait();
        }
        l = l * f + lt;
        tc::fence_before_sync();
        tc::mbar_arrive(&p_full[t]);
        if (pp) {
          if (turn < n_give) tc::named_bar_arrive(kPing + 1 - t, 256);
          ++turn;
        }
      }
      // after an abort, hand over the turns still owed so the other group never blocks on them
      for (int k = turn; k < n_give; ++k) tc::named_bar_arrive(kPing + 1 - t, 256);
      // ring step: the running output of this row, loaded while the last P V completes (all
      // loads in flight at once: one memory latency, not one per vector)
      float4 pa[MODE == 2 ? DH / 4 : 1];
      float la2 = -INFINITY;
      if constexpr (MODE == 2) {
        grid_dep_wait();  // the previous step's accumulators are complete and visible
        if (ok && row_ok && has_keys && !a.acc_first) {
          const float4* src = reinterpret_cast<const float4*>(a.o_acc + ((int64_t)h * S + row) * DH);
          la2 = a.lse[(int64_t)h * S + row] * kLog2e;
#pragma unroll
          for (int i = 0; i < DH / 4; ++i) pa[i] = src[i];
        }
      }
      if (ok && has_keys) ok = tc::mbar_wait(&o_full[t], 0, abort_flag, a.err, a.wait_ns);
      tc::fence_after_sync();
      // epilogue: O / l -> bf16 row; lse or D
      const float inv = (MODE != 1) ? (l > 0.f ? 1.f / l : 0.f) : 1.f;
      if constexpr (MODE == 2) {
        // fold the block into the running (O_acc, lse): weights of the two sides in exp2 units
        const float lb2 = l > 0.f ? m_used + log2f(l) : -INFINITY;
        const float mx = fmaxf(la2, lb2);
        float wa = 0.f, wb = 0.f, lnew = -INFINITY;
        if (mx != -INFINITY) {
          wa = exp2f(la2 - mx);  // 0 when la2 = -inf (first step)
          wb = exp2f(lb2 - mx);
          const float sum = wa + wb;
          lnew = (mx + log2f(sum)) * kLn2;
          wa /= sum;
          wb = wb / sum * inv;
        }
        const bool act = ok && row_ok && has_keys;
        // the last step that touches this tile writes its bf16 result and no fp32 state (without a
        // bf16 output, the fp32 state is the result and always stored)
        const bool last = a.o && !q_tile_touched_later(a, dev, t ? qt1 : qt0, nt);
        float* arow = a.o_acc + ((int64_t)h * S + (row_ok ? row : 0)) * DH;
        bf16* orow = last ? a.o + ((int64_t)h * S + (row_ok ? row : 0)) * DH : nullptr;
#pragma unroll
        for (int ch = 0; ch < DH / 32; ++ch) {
          uint32_t v[32];
          tc::tmem_ld32(o_addr + ch * 32, v);
          tc::tmem_ld_wait();
          if (act) {
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
              float4 o4 = make_float4(0.f, 0.f, 0.f, 0.f);
              if (wa != 0.f) {  // a side with weight 0 contributes nothing, whatever it holds
                const float4 p4 = pa[ch * 8 + q4];
                o4 = make_float4(wa * p4.x, wa * p4.y, wa * p4.z, wa * p4.w);
              }
              if (wb != 0.f) {
                o4.x += wb * __uint_as_float(v[q4 * 4 + 0]);
                o4.y += wb * __uint_as_float(v[q4 * 4 + 1]);
                o4.z += wb * __uint_as_float(v[q4 * 4 + 2]);
                o4.w += wb * __uint_as_float(v[q4 * 4 + 3]);
              }
              if (!last) *reinterpret_cast<float4*>(arow + ch * 32 + q4 * 4) = o4;
              if (orow)
                *reinterpret_cast<uint2*>(orow + ch * 32 + q4 * 4) =
                    make_uint2(tc::pack_bf16x2(o4.x, o4.y), tc::pack_bf16x2(o4.z, o4.w));
            }
          }
        }
        if (act) a.lse[(int64_t)h * S + row] = lnew;
      } else {
      bf16* orow = a.o + ((int64_t)h * S + (row_ok ? row : 0)) * DH;
      const bf16* dorow = (MODE == 1) ? a.dO + ((int64_t)h * S + (row_ok ? row : 0)) * DH : nullptr;
      float dsum = 0.f;
#pragma unroll
      for (int ch = 0; ch < DH / 32; ++ch) {
        uint32_t v[32];
        tc::tmem_ld32(o_addr + ch * 32, v);
        tc::tmem_ld_wait();
        if (!has_keys) {  // never in plain launches (every row sees itself); O = 0 then
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;
        }
        if (ok && row_ok) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 pkt;
            uint32_t* pw = reinterpret_cast<uint32_t*>(&pkt);
            uint4 dv4;
            if (MODE == 1) dv4 = *reinterpret_cast<const uint4*>(dorow + ch * 32 + q4 * 8);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float o0 = __uint_as_float(v[q4 * 8 + 2 * i]) * inv;
              const float o1 = __uint_as_float(v[q4 * 8 + 2 * i + 1]) * inv;
              pw[i] = tc::pack_bf16x2(o0, o1);
              if (MODE == 1) {
                const __nv_bfloat162 d2 = reinterpret_cast<const __nv_bfloat162*>(&dv4)[i];
                dsum += o0 * __low2float(d2) + o1 * __high2float(d2);
              }
            }
            *reinterpret_cast<uint4*>(orow + ch * 32 + q4 * 8) = pkt;
          }
        }
      }
      if (MODE == 0) {
        if (ok && row_ok) a.lse[(int64_t)h * S + row] = l > 0.f ? (m_used + log2f(l)) * kLn2 : -INFINITY;
      } else if (ok) {
        // padded [2][nh][nt*128]: D, then lse*log2e; zeros past the end of the sequence
        const int64_t sp = (int64_t)nt * kTile;
        a.D[(int64_t)h * sp + row] = row_ok ? dsum : 0.f;
        a.D[((int64_t)a.nh + h) * sp + row] = row_ok ? m_used : 0.f;
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

template <int DH, int MODE>
cudaError_t run(const AttnArgs& a, cudaStream_t st) {
  using L = FwdLayout<DH>;
  CUtensorMap tq, tk, tv;
  if (!make_tmap_3d_bf16(&tq, a.q, DH, a.S, a.nh, 64, 128) || !make_tmap_3d_bf16(&tk, a.k, DH, a.S, a.nkv, 64, 128) ||
      !make_tmap_3d_bf16(&tv, a.v, DH, a.S, a.nkv, 64, 128))
    return cudaErrorInvalidValue;
  // at least 120 KB so that two CTAs never share an SM (each takes all 512 TMEM columns)
  const size_t smem = L::BYTES + 1024 > 120 * 1024 ? L::BYTES + 1024 : 120 * 1024;
  auto kfn = k_attn_fwd_tc<DH, MODE>;
  cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  AttnArgs args = a;
  fill_planes(args);
  const int nt = (int)ceil_div(a.S, kTile);
  dim3 grid((unsigned)args.hq, (unsigned)(args.ndev * ceil_div(nt, 2)));
  args.wait_ns = wait_limit_ns();
  if (args.pdl) {
    e = launch_pdl(kfn, grid, dim3(kFwdThreads), smem, st, tq, tk, tv, args);
  } else {
    kfn<<<grid, kFwdThreads, smem, st>>>(tq, tk, tv, args);
    e = cudaGetLastError();
  }
  note_launch();
  return e;
}

}  // namespace

cudaError_t launch_attn_fwd(const AttnArgs& a, int head_dim, cudaStream_t st) {
  return head_dim == 64 ? run<64, 0>(a, st) : run<128, 0>(a, st);
}
cudaError_t launch_attn_recompute(const AttnArgs& a, int head_dim, cudaStream_t st) {
  return head_dim == 64 ? run<64, 1>(a, st) : run<128, 1>(a, st);
}
cudaError_t launch_attn_ring_fwd(const AttnArgs& a, int head_dim, cudaStream_t st) {
  return head_dim == 64 ? run<64, 2>(a, st) : run<128, 2>(a, st);
}

}  // namespace upipe
