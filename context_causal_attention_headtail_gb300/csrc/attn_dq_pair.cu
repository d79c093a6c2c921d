// dQ of the ring-attention backward computed by CTA pairs with two-SM MMAs
// (d = 128, inputs already rotated or no RoPE). Same mathematics and ring
// order as the query-stationary kernel of attn_bwd2_tc.cu ("Claude Logs",
// 2026-03-24: P from the saved LSE, dS = P * (dP - D); dQ owned by one place,
// no atomics): per key tile, S = Q K^T, dP = dO V^T, dS, dQ += dS K.
//
// What changes is the layout. A cluster of two CTAs owns 256 consecutive
// query rows of one chunk (128 per CTA) and streams each key tile once for
// both: every product is one M = 256 MMA issued by the pair's leader, each CTA
// supplying half of the B operand, so each SM reads half of B from its shared
// memory. That leaves room to keep Q in shared memory (S is an SS product)
// and to give dS its own tensor-memory columns: dP(n+1) no longer waits for
// dQ(n) to consume dS(n), only for the softmax to have read dP(n), and
// S(n+1) only for the softmax to have read S(n).
//
// Per CTA, shared memory: Q (its 128 rows, K-major), NK stages of K holding
//   Kr: keys [64r, 64r+64) of the key tile, K-major  (B half of S = Q K^T)
//   Kc: all 128 keys, d columns [64r, 64r+64)          (B half of dQ += dS K)
// and NV stages of V holding
//   Vr: keys [64r, 64r+64), K-major                   (B half of dP = dO V^T)
// (r = the CTA's rank in the pair). K is in use from S(n) to dQ(n), the
// longest span, so its ring is the deeper one: a K stage is refilled while
// three other key tiles are in flight, which covers the L2 latency of the
// refill (a timeline of the pair showed the issuer waiting ~300-600 cycles
// per tile for K/V with three shared stages). Tensor memory: dO (bf16 A operand) 0..63,
// dS (bf16 A operand) 64..127, S 128..255, dP 256..383, dQ 384..511.
// Warps 0-7: softmax (warpgroup h owns key columns [64h, 64h+64)); warp 8:
// TMA producer and TMEM allocator; warp 9: MMA issuer (leader only).
// With the forward's O given, warpgroup 1 computes its rows'
// D = rowsum(dO * O) (the backward's preprocess, "Claude Logs", 2026-03-24)
// from the dO row it loads into TMEM anyway, after handing dO over, so the
// O loads overlap the first products; D goes to warpgroup 0 through shared
// memory (d_ready) and out to the dK/dV kernel, which then runs after this
// one: no separate D pass.
#include <math.h>

#include "attn_common.cuh"

namespace cpattn {
namespace {

constexpr float kLog2eP = 1.4426950408889634f;

struct DqPairParams {
  const __nv_bfloat16 *dO;   // sharded [BH, T, 128]
  const __nv_bfloat16 *o;    // the forward's O: D = rowsum(dO * O) is computed here and written to D; nullptr: read D
  const float *lse;          // [BH, T]
  float *D;                  // [BH, T]
  __nv_bfloat16 *dq;
  int *err;
  int BH, T, T_valid, c, cp, causal, tpc;
  int group;                 // query heads per K/V head
  const int *doc_lo, *doc_hi;
  float scale, scale_log2;
  RopeTheta theta;           // R^T of the epilogue (EPI)
};

struct DqPairCfg {
  static constexpr int D = 128;
  static constexpr int NK = 4, NV = 3;               // K and V stages
  static constexpr int QT = kTile * D * 2;           // Q tile, 32 KiB
  static constexpr int HT = 64 * D * 2;              // half tile, 16 KiB
  static constexpr int KSTAGE = 2 * HT;              // Kr, Kc
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = QT;
  static constexpr int OFF_V = OFF_K + NK * KSTAGE;
  static constexpr int OFF_BAR = OFF_V + NV * HT;
  // q_full, qdo_ready, s_full, s_free, dp_full, dp_free, ds_ready, dq_done, fin, d_ready,
  // k_full[NK], k_empty[NK], v_full[NV], v_empty[NV]
  static constexpr int NBAR = 10 + 2 * NK + 2 * NV;
  static constexpr int OFF_DROW = OFF_BAR + NBAR * 8;   // D of the tile's 128 rows (fp32)
  static constexpr int OFF_MISC = OFF_DROW + 512;
  static constexpr int SMEM = OFF_MISC + 16 + kMaxTiles * 8 + 1024;   // misc, tile table, alignment slack
  static_assert(SMEM <= 232448, "over the 227 KiB of shared memory a CTA may opt into");
  static constexpr uint32_t colDO = 0, colDS = 64, colS = 128, colDP = 256, colDQ = 384;
  // arrivals on the leader's softmax barriers: 8 warps in each CTA of the pair
  static constexpr uint32_t kWarpArrivals = 16;
};

// Heads per launch-order group of the paired dQ kernel.
constexpr int kDqHeadGroup = 1;

__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %clusterid.x;" : "=r"(r));
  return r;
}

// EPI: q and k arrive rotated (in-kernel RoPE done by the forward); dQ leaves
// through R^T at the query's position.
template <bool EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(320, 1)
    dq_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kc,
                   const __grid_constant__ CUtensorMap tm_kr, const __grid_constant__ CUtensorMap tm_vr,
                   const __grid_constant__ DqPairParams p) {
  using C = DqPairCfg;
  constexpr int NK = C::NK, NV = C::NV, D = C::D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = tc::smem_u32(smem);
  const uint32_t rank = tc::cluster_rank();
  const bool leader = rank == 0;
  const uint32_t sQ = sbase + C::OFF_Q;
  auto sKr = [&](int st) { return sbase + C::OFF_K + st * C::KSTAGE; };
  auto sKc = [&](int st) { return sbase + C::OFF_K + st * C::KSTAGE + C::HT; };
  auto sVr = [&](int st) { return sbase + C::OFF_V + st * C::HT; };
  const uint32_t bar0 = sbase + C::OFF_BAR;
  const uint32_t bar_q_full = bar0, bar_qdo = bar0 + 8, bar_s_full = bar0 + 16, bar_s_free = bar0 + 24,
                 bar_dp_full = bar0 + 32, bar_dp_free = bar0 + 40, bar_ds_ready = bar0 + 48,
                 bar_dq_done = bar0 + 56, bar_fin = bar0 + 64, bar_d_ready = bar0 + 72;
  float *s_drow = reinterpret_cast<float *>(smem + C::OFF_DROW);
  auto bar_k_full = [&](int st) { return bar0 + 80 + 8 * st; };
  auto bar_k_empty = [&](int st) { return bar0 + 80 + 8 * NK + 8 * st; };
  auto bar_v_full = [&](int st) { return bar0 + 80 + 16 * NK + 8 * st; };
  auto bar_v_empty = [&](int st) { return bar0 + 80 + 16 * NK + 8 * NV + 8 * st; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
  int *ntiles_slot = reinterpret_cast<int *>(smem + C::OFF_MISC + 12);
  TileEntry *tab = reinterpret_cast<TileEntry *>(smem + C::OFF_MISC + 16);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cp = p.cp, c = p.c, tpc = p.tpc;
  const int ppc = (tpc + 1) / 2;                  // tile pairs per chunk
  const int pair = (int)cluster_id_x();
  int bh, g;   // a few heads at a time (K/V tiles shared in L2), heaviest pairs first
  head_group_order<kDqHeadGroup>(pair, 2 * cp * ppc, p.BH, bh, g);
  const int bkv = bh / p.group;                   // K/V head of this query head
  const int kq = 2 * cp - 1 - g / ppc;            // latest chunks first: they carry the most work
  const int pq = ppc - 1 - g % ppc;
  int rq, hq;
  owner_of(kq, cp, rq, hq);
  const int y_pair = pq * 2 * kTile;              // first row of the pair inside the chunk
  const int y_own = y_pair + (int)rank * kTile;   // first row of this CTA's tile
  const int pair_rows = min(2 * kTile, c - y_pair);
  const int q_rows = min(kTile, c - y_own);       // <= 0 for the peer of a lone last tile
  const int q_pos_pair = kq * c + y_pair;
  const int q_pos0 = kq * c + y_own;
  const int q_z = bh * 2 * cp + 2 * rq + hq;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NBAR; ++i) {
      const uint32_t b = bar0 + 8 * i;
      const bool by_warps = b == bar_qdo || b == bar_s_free || b == bar_dp_free || b == bar_ds_ready;
      tc::mbar_init(b, by_warps ? C::kWarpArrivals : b == bar_d_ready ? 128 : 1);
    }
    abort_flag[0] = 0;
    abort_flag[1] = 0;
    tc::mbar_fence_init();
  }
  tc::cluster_sync_all();          // both CTAs' barriers exist before either touches the other's
  if (warp == 8) {
    if (lane == 0) {   // the stationary Q tiles load while the tile table is built
      if (leader) tc::mbar_arrive_expect_tx(bar_q_full, 2 * C::QT);
      const uint32_t lq = tc::mapa_shared(bar_q_full, 0);
      for (int blk = 0; blk < D / 64; ++blk)
        tc::tma_load_3d_pair(sQ + blk * kTile * 128, &tm_q, lq, blk * 64, y_own, q_z);
    }
    __syncwarp();
    tc::tmem_alloc_pair(tc::smem_u32(tmem_slot), 512);
    tc::tmem_relinquish_pair();
    const KvBounds kb = kv_bounds(p.doc_lo, p.doc_hi, p.T, p.T_valid, p.causal, q_pos_pair,
                                  q_pos_pair + pair_rows - 1);
    const int nt = build_kv_table(tab, cp, c, rq, p.causal, p.T_valid, kb, lane);
    if (lane == 0) *ntiles_slot = nt;
  }
  tc::tc_fence_before();
  tc::cluster_arrive();
  // Warpgroup 1 of the softmax warps: this thread's rows of dO (and of O, for
  // D) are loaded while the pair waits at the barrier (a release arrival
  // after the loads would wait for them).
  const long long grow = (long long)bh * p.T + (long long)(2 * c * rq + hq * c + y_own + (threadIdx.x & 127));
  const bool row_valid = (int)(threadIdx.x & 127) < q_rows;
  uint4 pre_do[D / 8], pre_o[D / 8];
  if (warp >= 4 && warp < 8) {
    const uint4 *src = reinterpret_cast<const uint4 *>(p.dO + grow * D);
#pragma unroll
    for (int v = 0; v < D / 8; ++v) pre_do[v] = row_valid ? src[v] : make_uint4(0u, 0u, 0u, 0u);
    if (p.o) {
      const uint4 *o_src = reinterpret_cast<const uint4 *>(p.o + grow * D);
#pragma unroll
      for (int v = 0; v < D / 8; ++v) pre_o[v] = row_valid ? o_src[v] : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  tc::cluster_wait();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int ntiles = *ntiles_slot;
  const tc::WaitCtx wc{abort_flag, p.err};
  const tc::WaitCtx drain{abort_flag + 1, p.err};

  TileInfo t;

  if (warp == 8) {
    // ---------------------------------------------------- TMA producer (both CTAs)
    if (lane == 0) {
      tc::tma_prefetch_desc(&tm_kr);
      tc::tma_prefetch_desc(&tm_kc);
      tc::tma_prefetch_desc(&tm_vr);
      int nk = 0, nv = 0;   // K / V tiles issued
      while (nk < ntiles && (decode_tile(tab[nk], t), true)) {
        const int z = bkv * 2 * cp + t.slot;
        const int yr = t.y0 + 64 * (int)rank;
        const int sk = nk % NK, sv = nk % NV;
        if (nk >= NK && !tc::mbar_wait(bar_k_empty(sk), ((nk / NK) - 1) & 1, wc)) break;
        const uint32_t lk = tc::mapa_shared(bar_k_full(sk), 0);
        if (leader) tc::mbar_arrive_expect_tx(bar_k_full(sk), 2 * C::KSTAGE);
        for (int blk = 0; blk < D / 64; ++blk)
          tc::tma_load_3d_pair(sKr(sk) + blk * 64 * 128, &tm_kr, lk, blk * 64, yr, z);
        tc::tma_load_3d_pair(sKc(sk), &tm_kc, lk, 64 * (int)rank, t.y0, z);
        ++nk;
        if (nv >= NV && !tc::mbar_wait(bar_v_empty(sv), ((nv / NV) - 1) & 1, wc)) break;
        const uint32_t lv = tc::mapa_shared(bar_v_full(sv), 0);
        if (leader) tc::mbar_arrive_expect_tx(bar_v_full(sv), 2 * C::HT);
        for (int blk = 0; blk < D / 64; ++blk)
          tc::tma_load_3d_pair(sVr(sv) + blk * 64 * 128, &tm_vr, lv, blk * 64, yr, z);
        ++nv;
      }
      // every issued stage is consumed by the pair's MMAs (multicast k_empty /
      // v_empty) before this CTA's shared memory goes away
      for (int m = (nk > NK ? nk - NK : 0); m < nk; ++m) tc::mbar_wait(bar_k_empty(m % NK), (m / NK) & 1, drain);
      for (int m = (nv > NV ? nv - NV : 0); m < nv; ++m) tc::mbar_wait(bar_v_empty(m % NV), (m / NV) & 1, drain);
    }
  } else if (warp == 9) {
    // ------------------------------------------------ MMA issuer (leader only)
    auto wait_all = [&](uint32_t bar, uint32_t par, const tc::WaitCtx &w) {
      return __all_sync(0xffffffffu, tc::mbar_wait(bar, par, w));
    };
    if (leader) {
      constexpr uint32_t idS = tc::idesc_bf16(256, 128, false, false);
      constexpr uint32_t idQ = tc::idesc_bf16(256, D, false, true);
      const uint64_t aq0 = tc::kdesc0(sQ);
      auto issue_s = [&](int n) {
        const uint64_t b0 = tc::kdesc0(sKr(n % NK));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc::mma2_ss_w(tmem + C::colS, aq0 + tc::koff(kTile, kk), b0 + tc::koff(64, kk), idS, kk > 0 ? 1u : 0u);
        tc::mma2_commit_both_w(bar_s_full);
      };
      auto issue_dp = [&](int n) {
        const uint64_t b0 = tc::kdesc0(sVr(n % NV));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc::mma2_ts_w(tmem + C::colDP, tmem + C::colDO + kk * 8, b0 + tc::koff(64, kk), idS, kk > 0 ? 1u : 0u);
        tc::mma2_commit_both_w(bar_dp_full);
        tc::mma2_commit_both_w(bar_v_empty(n % NV));   // dP(n) is the only reader of V(n)
      };
      bool ok = wait_all(bar_q_full, 0, wc) && wait_all(bar_qdo, 0, wc);
      if (ok && ntiles > 0) {
        ok = wait_all(bar_k_full(0), 0, wc) && wait_all(bar_v_full(0), 0, wc);
        if (ok) {
          tc::tc_fence_after();
          issue_s(0);
          issue_dp(0);
        }
        for (int n = 0; ok; ++n) {
          const bool more = n + 1 < ntiles;
          const int sk = n % NK;
          if (more) {   // S(n+1) once S(n) has been read, dP(n+1) once dP(n) has been read
            if (!(ok = wait_all(bar_k_full((n + 1) % NK), ((n + 1) / NK) & 1, wc))) break;
            if (!(ok = wait_all(bar_s_free, n & 1, wc))) break;
            tc::tc_fence_after();
            issue_s(n + 1);
            if (!(ok = wait_all(bar_v_full((n + 1) % NV), ((n + 1) / NV) & 1, wc))) break;
            if (!(ok = wait_all(bar_dp_free, n & 1, wc))) break;
            tc::tc_fence_after();
            issue_dp(n + 1);
          }
          if (!(ok = wait_all(bar_ds_ready, n & 1, wc))) break;
          tc::tc_fence_after();
          {   // dQ += dS(n) K(n): dS in its own columns, 128 keys = 64 packed columns
            const uint64_t b0 = tc::mndesc0(sKc(sk), kTile);
            const uint32_t acc0 = n > 0 ? 1u : 0u;
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              tc::mma2_ts_w(tmem + C::colDQ, tmem + C::colDS + kk * 8, b0 + tc::mnoff(kk), idQ, kk > 0 ? 1u : acc0);
            tc::mma2_commit_both_w(bar_dq_done);
            tc::mma2_commit_both_w(bar_k_empty(sk));   // dQ(n) is the last reader of K(n)
          }
          if (!more) break;
        }
      }
      tc::mma2_commit_both_w(bar_fin);
    }
    // both CTAs: every arrival of the pair's MMAs has landed before teardown
    wait_all(bar_fin, 0, drain);
  } else {
    // ------------------------------------ softmax warpgroups (both CTAs, key halves)
    const int h = warp >> 2;
    const int row = threadIdx.x & 127;
    const int q_pos = q_pos0 + row;
    const bool valid = row_valid;
    const uint32_t t_row = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const float lse2 = valid ? p.lse[grow] * kLog2eP : INFINITY;
    float Drow = (!p.o && valid) ? p.D[grow] : 0.f;   // with O given: computed below
    const uint32_t l_qdo = tc::mapa_shared(bar_qdo, 0), l_s_free = tc::mapa_shared(bar_s_free, 0),
                   l_dp_free = tc::mapa_shared(bar_dp_free, 0), l_ds_ready = tc::mapa_shared(bar_ds_ready, 0);
    auto warp_arrive = [&](uint32_t leader_bar) {   // after this warp's TMEM accesses are complete
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_cluster(leader_bar);
    };
    if (h == 1) {   // this thread's row of dO into TMEM (A operand of dP), then D
      uint32_t r[D / 64][32];
#pragma unroll
      for (int v = 0; v < D / 8; ++v) {
        const uint4 x = pre_do[v];
        uint32_t *rv = &r[v / 8][4 * (v % 8)];
        rv[0] = x.x; rv[1] = x.y; rv[2] = x.z; rv[3] = x.w;
      }
#pragma unroll
      for (int cb = 0; cb < D / 64; ++cb) tc::tmem_st32(t_row + C::colDO + cb * 32, r[cb]);
      tc::tmem_st_wait();
      tc::tc_fence_before();
      warp_arrive(l_qdo);
      if (p.o) {   // D = rowsum(dO * O), fixed summation order (bitwise reproducible)
        uint64_t acc[4] = {tc::f2(0.f, 0.f), tc::f2(0.f, 0.f), tc::f2(0.f, 0.f), tc::f2(0.f, 0.f)};
#pragma unroll
        for (int v = 0; v < D / 8; ++v) {
          const uint4 b = pre_o[v];
          const uint32_t *aw = &r[v / 8][4 * (v % 8)];
          const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
          for (int w = 0; w < 4; ++w)
            acc[w] = tc::ffma2(tc::f2(bf16lo_to_f32(aw[w]), bf16hi_to_f32(aw[w])),
                               tc::f2(bf16lo_to_f32(bw[w]), bf16hi_to_f32(bw[w])), acc[w]);
        }
        float a0, a1, a2, a3, a4, a5, a6, a7;
        tc::unf2(acc[0], a0, a1);
        tc::unf2(acc[1], a2, a3);
        tc::unf2(acc[2], a4, a5);
        tc::unf2(acc[3], a6, a7);
        Drow = ((a0 + a1) + (a2 + a3)) + ((a4 + a5) + (a6 + a7));
        s_drow[row] = Drow;
        if (valid) p.D[grow] = Drow;
        tc::mbar_arrive(bar_d_ready);
      }
    } else {
      tc::tc_fence_before();
      warp_arrive(l_qdo);
    }
    const float sl2 = p.scale_log2;
    int dlo, dhi;   // this row's document [dlo, dhi)
    doc_bounds_at(p.doc_lo, p.doc_hi, min(q_pos, p.T - 1), p.T, dlo, dhi);
    int n = 0;
    bool ok = true;
    while (n < ntiles && (decode_tile(tab[n], t), true)) {
      ok = __all_sync(0xffffffffu, tc::mbar_wait(bar_s_full, n & 1, wc));
      if (!ok) break;
      tc::tc_fence_after();
      float pr[64];
      {
        uint32_t r[2][32];
        tc::tmem_ld32(t_row + C::colS + 64 * h, r[0]);
        tc::tmem_ld32(t_row + C::colS + 64 * h + 32, r[1]);
        tc::tmem_ld_wait();
        tc::tc_fence_before();
        warp_arrive(l_s_free);                        // S may now be overwritten by S(n+1)
        // keep key columns lo <= j < lim (see the forward kernel)
        int lim = kTile, lo = 0;
        if (t.need_mask) {
          lim = min(min(t.nvalid, p.T_valid - t.pos0), dhi - t.pos0);
          if (p.causal) lim = min(lim, q_pos - t.pos0 + 1);
          lo = dlo - t.pos0;
        }
        lim -= 64 * h;
        lo -= 64 * h;
        const uint64_t sl2x2 = tc::f2(sl2, sl2), nl2 = tc::f2(-lse2, -lse2);
#pragma unroll
        for (int j = 0; j < 64; j += 2) {
          float x0, x1;
          tc::unf2(tc::ffma2(tc::f2(__uint_as_float(r[j >> 5][j & 31]), __uint_as_float(r[j >> 5][(j & 31) + 1])),
                             sl2x2, nl2), x0, x1);
          pr[j] = tc::ex2(x0);
          pr[j + 1] = tc::ex2(x1);
        }
        if (__any_sync(0xffffffffu, lim < 64 || lo > 0)) {
          const unsigned width = (unsigned)max(lim - lo, 0);
#pragma unroll
          for (int j = 0; j < 64; ++j)
            if ((unsigned)(j - lo) >= width) pr[j] = 0.f;
        }
      }
      ok = __all_sync(0xffffffffu, tc::mbar_wait(bar_dp_full, n & 1, wc));
      if (!ok) break;
      if (n == 0 && p.o && h == 0) {   // D of this row, from warpgroup 1
        ok = __all_sync(0xffffffffu, tc::mbar_wait(bar_d_ready, 0, wc));
        if (!ok) break;
        Drow = s_drow[row];
      }
      tc::tc_fence_after();
      uint32_t pk[2][16];
      {
        uint32_t rd[2][32];
        tc::tmem_ld32(t_row + C::colDP + 64 * h, rd[0]);
        tc::tmem_ld32(t_row + C::colDP + 64 * h + 32, rd[1]);
        tc::tmem_ld_wait();
        tc::tc_fence_before();
        warp_arrive(l_dp_free);                       // dP may now be overwritten by dP(n+1)
        const uint64_t nD2 = tc::f2(-Drow, -Drow);
#pragma unroll
        for (int cb = 0; cb < 2; ++cb)
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int j = cb * 32 + 2 * e;
            const uint64_t dp = tc::fadd2(tc::f2(__uint_as_float(rd[cb][2 * e]), __uint_as_float(rd[cb][2 * e + 1])), nD2);
            pk[cb][e] = tc::pack_bf16x2_2(tc::fmul2(tc::f2(pr[j], pr[j + 1]), dp));
          }
      }
      if (n > 0) {   // dS(n-1) consumed by dQ(n-1) before dS(n) overwrites it
        ok = __all_sync(0xffffffffu, tc::mbar_wait(bar_dq_done, (n - 1) & 1, wc));
        if (!ok) break;
        tc::tc_fence_after();
      }
      tc::tmem_st16(t_row + C::colDS + 32 * h, pk[0]);
      tc::tmem_st16(t_row + C::colDS + 32 * h + 16, pk[1]);
      tc::tmem_st_wait();
      tc::tc_fence_before();
      warp_arrive(l_ds_ready);
      ++n;
    }
    if (ok && n > 0) {
      ok = __all_sync(0xffffffffu, tc::mbar_wait(bar_dq_done, (n - 1) & 1, wc));
      if (ok && EPI) {   // frequencies 32h..32h+31 of dQ and their partners 64 columns on: R^T
        tc::tc_fence_after();
        store_tmem_pair_rope<D>(t_row + C::colDQ, h, p.scale, q_pos, p.theta, p.dq + grow * D, valid);
      } else if (ok) {
        tc::tc_fence_after();
#pragma unroll 1
        for (int cb = 0; cb < 2; ++cb) {   // this warpgroup's 64 columns of dQ, scaled, as bf16
          uint32_t r[32];
          tc::tmem_ld32(t_row + C::colDQ + h * 64 + cb * 32, r);
          tc::tmem_ld_wait();
          uint32_t o[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            o[e] = pack_bf16x2(__uint_as_float(r[2 * e]) * p.scale, __uint_as_float(r[2 * e + 1]) * p.scale);
          if (valid) {
            uint4 *d4 = reinterpret_cast<uint4 *>(p.dq + grow * D + h * 64 + cb * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v) d4[v] = make_uint4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
          }
        }
      }
    } else if (ok && valid) {   // no key tile at all (rows outside every document)
      uint4 *d4 = reinterpret_cast<uint4 *>(p.dq + grow * D + h * (D / 2));
#pragma unroll 1
      for (int v = 0; v < D / 16; ++v) d4[v] = make_uint4(0u, 0u, 0u, 0u);
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  tc::cluster_sync_all();          // both CTAs are done with the pair's tensor memory and barriers
  if (warp == 8) {
    tc::tc_fence_after();
    tc::tmem_dealloc_pair(tmem, 512);
  }
  tc::cluster_sync_all();
}

}  // namespace

cpattn_status launch_dq_pair_bf16(const void *q, const void *k, const void *v, const float *lse,
                                  const void *dO, void *dq, float *D, const Geometry &g,
                                  cudaStream_t s) {
  using C = DqPairCfg;
  if (g.d != C::D || g.rope) return fail(CPATTN_ERR_UNSUPPORTED, "paired dQ kernel: d = 128, q and k not rotated in-kernel");
  const long long BH = (long long)g.B * g.H;
  const long long n_slots = BH * 2 * g.cp;
  const long long n_kv_slots = (long long)g.B * g.Hkv * 2 * g.cp;
  CUtensorMap mq, mkc, mkr, mvr;
  if (!make_tile_map(&mq, q, g.d, g.c, n_slots) || !make_tile_map(&mkc, k, g.d, g.c, n_kv_slots) ||
      !make_tile_map(&mkr, k, g.d, g.c, n_kv_slots, 64) || !make_tile_map(&mvr, v, g.d, g.c, n_kv_slots, 64))
    return fail(CPATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed (is the driver too old?)");
  DqPairParams dp;
  dp.dO = static_cast<const __nv_bfloat16 *>(dO);
  dp.o = static_cast<const __nv_bfloat16 *>(g.o_for_D);
  dp.lse = lse;
  dp.D = D;
  dp.dq = static_cast<__nv_bfloat16 *>(dq);
  dp.err = device_err_flag();
  dp.BH = (int)BH;
  dp.group = g.H / g.Hkv;
  dp.doc_lo = g.doc_lo;
  dp.doc_hi = g.doc_hi;
  dp.T = g.T;
  dp.T_valid = g.T_valid;
  dp.c = g.c;
  dp.cp = g.cp;
  dp.causal = g.causal;
  dp.tpc = (g.c + kTile - 1) / kTile;
  dp.scale = (float)(1.0 / sqrt((double)g.d));
  dp.scale_log2 = (float)(1.4426950408889634 / sqrt((double)g.d));
  const long long pairs = BH * 2 * g.cp * ((dp.tpc + 1) / 2);
  if (2 * pairs > 0x7fffffffLL) return fail(CPATTN_ERR_SHAPE, "too many query tiles");
  make_rope_theta(g.d, &dp.theta, g.rope_cfg);
  auto kern = g.rope_epi ? dq_pair_kernel<true> : dq_pair_kernel<false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
    return fail(CPATTN_ERR_CUDA, "cannot set %d bytes of shared memory for the paired dQ kernel", C::SMEM);
  kern<<<(unsigned)(2 * pairs), 320, C::SMEM, s>>>(mq, mkc, mkr, mvr, dp);
  return check_launch("tensor-core dQ kernel (CTA pairs)");
}

}  // namespace cpattn
