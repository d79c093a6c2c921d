// Ring attention backward, pipelined form (inputs already rotated, or no
// RoPE). Same mathematics and ring order as the kernels in attn_bwd_tc.cu
// (P from the saved LSE, dS = P * (dP - D), dK/dV and dQ each owned by one
// CTA, no atomics); the difference is scheduling. Every tcgen05.mma is
// 128 x 128 (or 128 x D) so the tensor core runs at full rate, and the two
// softmax warpgroups split each tile's 128 columns. The work on a tile is cut
// into a P phase (exponentials) and a dS phase, and the MMA issuer starts the
// products that need only one of them as soon as it is ready, so softmax
// work overlaps the matrix products of the same and of the next tile.
//  * dq2_tc_kernel (query-stationary): Q and dO are the A operands of
//    S = Q K^T and dP = dO V^T straight from TMEM.
//  * dkdv2_tc_kernel (key-stationary): dK and dV stay in TMEM across every
//    ring step of every rank (the ring's travelling accumulator).
#include <math.h>

#include "attn_common.cuh"

namespace cpattn {
namespace {

constexpr float kLog2eB = 1.4426950408889634f;

struct Bwd2Params {
  const __nv_bfloat16 *q, *dO;  // sharded [BH, T, D] (dq kernel: TMEM operands)
  const float *lse, *D;         // [BH, T]
  __nv_bfloat16 *dq, *dk, *dv;
  int *err;
  int BH, T, T_valid, c, cp, causal, tpc;
  int group;   // query heads per K/V head
  const int *doc_lo, *doc_hi;   // packed documents: [T] bounds per natural position, or nullptr
  float scale, scale_log2;
  RopeTheta theta;   // in-kernel RoPE frequencies (ROPE kernels)
};

// Scales 32-column chunks [c0, c0 + n*32) of a TMEM row and stores them as
// bf16 at dst + c0 (every lane of the warp must call this).
__device__ __forceinline__ void store_tmem_cols(uint32_t t_row, int c0, int nchunks, float scale,
                                                __nv_bfloat16 *dst, bool valid) {
#pragma unroll 1
  for (int cb = 0; cb < nchunks; ++cb) {
    uint32_t r[32];
    tc::tmem_ld32(t_row + c0 + cb * 32, r);
    tc::tmem_ld_wait();
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 16; ++e)
      pk[e] = pack_bf16x2(__uint_as_float(r[2 * e]) * scale, __uint_as_float(r[2 * e + 1]) * scale);
    if (valid) {
      uint4 *d4 = reinterpret_cast<uint4 *>(dst + c0 + cb * 32);
#pragma unroll
      for (int v = 0; v < 4; ++v) d4[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
    }
  }
}

// Rotate-half RoPE of a bf16 row held as D/2 words in registers (word k holds
// columns 2k, 2k+1; word k < D/4 pairs with word k + D/4) at natural
// position pos: m R for FORWARD, its transpose otherwise (m the temperature
// of the RoPE configuration, 1 for the standard rotation).
template <int D, bool FORWARD>
__device__ __forceinline__ void rope_row_words(uint32_t *w, int pos, const RopeTheta &th) {
#pragma unroll
  for (int k = 0; k < D / 4; ++k) {
    float s0, c0, s1, c1;
    rope_sincos(pos, th.hi[2 * k], th.lo[2 * k], s0, c0);
    rope_sincos(pos, th.hi[2 * k + 1], th.lo[2 * k + 1], s1, c1);
    c0 *= th.mscale; s0 *= th.mscale; c1 *= th.mscale; s1 *= th.mscale;   // m R (YaRN temperature)
    if (!FORWARD) { s0 = -s0; s1 = -s1; }
    const float x0 = bf16lo_to_f32(w[k]), x1 = bf16hi_to_f32(w[k]);
    const float y0 = bf16lo_to_f32(w[k + D / 4]), y1 = bf16hi_to_f32(w[k + D / 4]);
    w[k] = pack_bf16x2(fmaf(x0, c0, -y0 * s0), fmaf(x1, c1, -y1 * s1));
    w[k + D / 4] = pack_bf16x2(fmaf(y0, c0, x0 * s0), fmaf(y1, c1, x1 * s1));
  }
}

// ================================================================== dQ
// Query-stationary. TMEM: Q (bf16 A operand) 0, dO 64, S 128, dP 256, dQ 384.
// Warpgroup h owns key columns [64h, 64h+64) of each tile and writes its
// half of dS (bf16 pairs, 32 columns) over the start of its own half of dP,
// at 256 + 64h, so neither warpgroup waits for the other; the dQ MMA reads
// its A operand from columns 256..287 then 320..351. Per key tile n the MMA
// issuer runs S(n+1) as soon as both softmax warpgroups have read S(n), then
// dQ(n) once dS(n) is in TMEM, then dP(n+1) once dQ(n) has consumed dS(n).
// With in-kernel RoPE (ROPE) warpgroup 0 rotates its Q row before it goes to
// TMEM, warps 10-11 rotate every K tile in shared memory (k_ready), and dQ
// leaves through R^T at the query's position.
template <int D>
struct Dq3Cfg {
  static constexpr int NS = (D == 128) ? 3 : 4;  // K/V stages
  static constexpr int TILE = kTile * D * 2;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = NS * TILE;
  static constexpr int OFF_BAR = 2 * NS * TILE;
  // qdo_ready, fin, s_full, dp_full, s_free, (spare), ds_ready, dq_done, kv_full[NS], kv_empty[NS],
  // k_ready[NS]
  static constexpr int NBAR = 8 + 3 * NS;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + kMaxTiles * 8 + 1024;   // misc, tile table, alignment slack
  static_assert(SMEM <= 232448, "over the 227 KiB of shared memory a CTA may opt into");
  static constexpr uint32_t colQ = 0, colDO = 64, colS = 128, colDP = 256, colDQ = 384;
};

template <int D, bool ROPE, bool EPI = false>
__global__ void __launch_bounds__(ROPE ? 384 : 320, 1)
    dq2_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ Bwd2Params p) {
  using C = Dq3Cfg<D>;
  constexpr int NS = C::NS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = tc::smem_u32(smem);
  auto sK = [&](int st) { return sbase + C::OFF_K + st * C::TILE; };
  auto sV = [&](int st) { return sbase + C::OFF_V + st * C::TILE; };
  const uint32_t bar0 = sbase + C::OFF_BAR;
  const uint32_t bar_qdo = bar0, bar_fin = bar0 + 8, bar_s_full = bar0 + 16, bar_dp_full = bar0 + 24,
                 bar_s_free = bar0 + 32, bar_ds_ready = bar0 + 48, bar_dq_done = bar0 + 56;
  auto bar_kv_full = [&](int st) { return bar0 + 64 + 8 * st; };
  auto bar_kv_empty = [&](int st) { return bar0 + 64 + 8 * NS + 8 * st; };
  auto bar_k_ready = [&](int st) { return bar0 + 64 + 16 * NS + 8 * st; };
  auto bar_k_use = [&](int st) { return ROPE ? bar_k_ready(st) : bar_kv_full(st); };   // before S reads K
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
  int *ntiles_slot = reinterpret_cast<int *>(smem + C::OFF_MISC + 12);
  TileEntry *tab = reinterpret_cast<TileEntry *>(smem + C::OFF_MISC + 16);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cp = p.cp, c = p.c, tpc = p.tpc;
  const int bh = blockIdx.x / (2 * cp * tpc);     // heads vary slowest (K/V tiles shared in L2)
  const int bkv = bh / p.group;                   // K/V head of this query head
  const int g = blockIdx.x % (2 * cp * tpc);
  const int kq = 2 * cp - 1 - g / tpc;
  const int qt = tpc - 1 - g % tpc;
  int rq, hq;
  owner_of(kq, cp, rq, hq);
  const int q_pos0 = kq * c + qt * kTile;
  const int q_rows = min(kTile, c - qt * kTile);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NBAR; ++i) {
      const uint32_t b = bar0 + 8 * i;
      const bool by_threads = b == bar_qdo || b == bar_s_free || b == bar_ds_ready;
      uint32_t cnt = by_threads ? 256 : 1;
      if (b >= bar_k_ready(0)) cnt = 64;   // k_ready[]: the two rotation warps
      tc::mbar_init(b, cnt);
    }
    abort_flag[0] = 0;
    abort_flag[1] = 0;
    tc::mbar_fence_init();
  }
  if (warp == 8) {
    tc::tmem_alloc(tc::smem_u32(tmem_slot), 512);
    tc::tmem_relinquish();
    {
      const KvBounds kb = kv_bounds(p.doc_lo, p.doc_hi, p.T, p.T_valid, p.causal, q_pos0, q_pos0 + q_rows - 1);
      const int nt = build_kv_table(tab, cp, c, rq, p.causal, p.T_valid, kb, lane);
      if (lane == 0) *ntiles_slot = nt;
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int ntiles = *ntiles_slot;
  const tc::WaitCtx wc{abort_flag, p.err};
  const tc::WaitCtx drain{abort_flag + 1, p.err};

  TileInfo t;

  if (warp == 8) {
    if (lane == 0) {
      tc::tma_prefetch_desc(&tm_k);
      tc::tma_prefetch_desc(&tm_v);
      int n = 0;
      while (n < ntiles && (decode_tile(tab[n], t), true)) {
        const int st = n % NS;
        if (n >= NS && !tc::mbar_wait(bar_kv_empty(st), ((n / NS) - 1) & 1, wc)) break;
        tc::mbar_arrive_expect_tx(bar_kv_full(st), 2 * C::TILE);
        const int z = bkv * 2 * cp + t.slot;
        for (int blk = 0; blk < D / 64; ++blk) {
          tc::tma_load_3d(sK(st) + blk * kTile * 128, &tm_k, bar_kv_full(st), blk * 64, t.y0, z);
          tc::tma_load_3d(sV(st) + blk * kTile * 128, &tm_v, bar_kv_full(st), blk * 64, t.y0, z);
        }
        ++n;
      }
      for (int m = (n > NS ? n - NS : 0); m < n; ++m) tc::mbar_wait(bar_kv_full(m % NS), (m / NS) & 1, drain);
    }
  } else if (warp == 9) {
    {   // the whole warp runs the issue loop; elect.sync picks the issuing lane
      constexpr uint32_t idS = tc::idesc_bf16(128, 128, false, false);
      constexpr uint32_t idQ = tc::idesc_bf16(128, D, false, true);
      auto issue_s = [&](int st) {
        const uint64_t bk = tc::kdesc0(sK(st));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc::mma_ts_w(tmem + C::colS, tmem + C::colQ + kk * 8, bk + tc::koff(kTile, kk), idS, kk > 0 ? 1u : 0u);
        tc::mma_commit_w(bar_s_full);
      };
      auto issue_dp = [&](int st) {
        const uint64_t bv = tc::kdesc0(sV(st));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc::mma_ts_w(tmem + C::colDP, tmem + C::colDO + kk * 8, bv + tc::koff(kTile, kk), idS, kk > 0 ? 1u : 0u);
        tc::mma_commit_w(bar_dp_full);
      };
      auto wait_all = [&](uint32_t bar, uint32_t par, const tc::WaitCtx &w) {
        return __all_sync(0xffffffffu, tc::mbar_wait(bar, par, w));
      };
      bool ok = wait_all(bar_qdo, 0, wc);
      if (ok && ntiles > 0) {
        ok = wait_all(bar_k_use(0), 0, wc);
        if (ok) {
          tc::tc_fence_after();
          issue_s(0);
          issue_dp(0);
        }
        for (int n = 0; ok; ++n) {
          const bool more = n + 1 < ntiles;
          const int st = n % NS, st1 = (n + 1) % NS;
          if (more) {   // S(n+1) once S(n) has been read
            if (!(ok = wait_all(bar_k_use(st1), ((n + 1) / NS) & 1, wc))) break;
            if (!(ok = wait_all(bar_s_free, n & 1, wc))) break;
            tc::tc_fence_after();
            issue_s(st1);
          }
          if (!(ok = wait_all(bar_ds_ready, n & 1, wc))) break;
          tc::tc_fence_after();
          {   // dQ += dS(n) K(n); dS is 128 keys = 64 packed columns
            const uint64_t bk = tc::mndesc0(sK(st), kTile);
            const uint32_t acc0 = n > 0 ? 1u : 0u;
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)   // dS of keys 0..63 at +0, of keys 64..127 at +64
              tc::mma_ts_w(tmem + C::colDQ, tmem + C::colDP + kk * 8 + (kk >= 4 ? 32 : 0), bk + tc::mnoff(kk), idQ,
                         kk > 0 ? 1u : acc0);
            tc::mma_commit_w(bar_dq_done);
            tc::mma_commit_w(bar_kv_empty(st));
          }
          if (!more) break;
          if (!(ok = wait_all(bar_dq_done, n & 1, wc))) break;   // dP(n+1) overwrites dS(n)
          tc::tc_fence_after();
          issue_dp(st1);
        }
      }
      tc::mma_commit_w(bar_fin);
      wait_all(bar_fin, 0, drain);
    }
  } else if (ROPE && warp >= 10) {
    // ------------------------------------------------ RoPE rotation warps (K tiles)
    tc::RopeRows<D, 64> rr;   // warps 10-11
    rr.init((warp - 10) * 32 + lane, p.theta);
    for (int n = 0; n < ntiles; ++n) {
      decode_tile(tab[n], t);
      const int st = n % NS;
      if (!__all_sync(0xffffffffu, tc::mbar_wait(bar_kv_full(st), (n / NS) & 1, wc))) break;
      rr.rotate(smem + C::OFF_K + st * C::TILE, t.pos0);
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(bar_k_ready(st));
    }
  } else {
    // ---------------------------------------------- softmax warpgroups (key halves)
    const int h = warp >> 2;
    const int row = threadIdx.x & 127;
    const int q_pos = q_pos0 + row;
    const bool valid = row < q_rows;
    const uint32_t t_row = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const long long grow = (long long)bh * p.T + (long long)(2 * c * rq + hq * c + qt * kTile + row);
    const float lse2 = valid ? p.lse[grow] * kLog2eB : INFINITY;
    const float Drow = valid ? p.D[grow] : 0.f;
    {  // this thread's row of Q (warpgroup 0, rotated under ROPE) or dO (warpgroup 1) into TMEM
      const uint4 *src = reinterpret_cast<const uint4 *>((h == 0 ? p.q : p.dO) + grow * D);
      if (ROPE && h == 0) {
        uint32_t r[D / 64][32];
#pragma unroll
        for (int v = 0; v < D / 8; ++v) {
          const uint4 x = valid ? src[v] : make_uint4(0u, 0u, 0u, 0u);
          uint32_t *rv = &r[v / 8][4 * (v % 8)];
          rv[0] = x.x; rv[1] = x.y; rv[2] = x.z; rv[3] = x.w;
        }
        rope_row_words<D, true>(&r[0][0], q_pos, p.theta);
#pragma unroll
        for (int cb = 0; cb < D / 64; ++cb) tc::tmem_st32(t_row + C::colQ + cb * 32, r[cb]);
      } else {
#pragma unroll 1
        for (int cb = 0; cb < D / 64; ++cb) {
          uint32_t r[32];
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const uint4 x = valid ? src[cb * 8 + v] : make_uint4(0u, 0u, 0u, 0u);
            r[4 * v] = x.x; r[4 * v + 1] = x.y; r[4 * v + 2] = x.z; r[4 * v + 3] = x.w;
          }
          tc::tmem_st32(t_row + (h == 0 ? C::colQ : C::colDO) + cb * 32, r);
        }
      }
      tc::tmem_st_wait();
      tc::tc_fence_before();
      tc::mbar_arrive(bar_qdo);
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
        tc::mbar_arrive(bar_s_free);                 // S may now be overwritten by S(n+1)
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
      tc::tc_fence_after();
      uint32_t rd[2][32];
      tc::tmem_ld32(t_row + C::colDP + 64 * h, rd[0]);
      tc::tmem_ld32(t_row + C::colDP + 64 * h + 32, rd[1]);
      tc::tmem_ld_wait();
      const uint64_t nD2 = tc::f2(-Drow, -Drow);
#pragma unroll
      for (int cb = 0; cb < 2; ++cb) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int j = cb * 32 + 2 * e;
          const uint64_t dp = tc::fadd2(tc::f2(__uint_as_float(rd[cb][2 * e]), __uint_as_float(rd[cb][2 * e + 1])), nD2);
          pk[e] = tc::pack_bf16x2_2(tc::fmul2(tc::f2(pr[j], pr[j + 1]), dp));
        }
        tc::tmem_st16(t_row + C::colDP + 64 * h + cb * 16, pk);
      }
      tc::tmem_st_wait();
      tc::tc_fence_before();
      tc::mbar_arrive(bar_ds_ready);
      ++n;
    }
    if (ok && n > 0) {
      ok = __all_sync(0xffffffffu, tc::mbar_wait(bar_dq_done, (n - 1) & 1, wc));
      if (ok) {
        tc::tc_fence_after();
        if (!ROPE && !EPI)
          store_tmem_cols(t_row + C::colDQ, h * (D / 2), D / 64, p.scale, p.dq + grow * D, valid);
        else if (D == 128 || h == 0)   // warpgroup h: frequencies 32h..32h+31 (D = 64: warpgroup 0, all 32)
          store_tmem_pair_rope<D>(t_row + C::colDQ, h, p.scale, q_pos, p.theta, p.dq + grow * D, valid);
      }
    } else if (ok && valid) {   // no key tile at all (rows outside every document)
      uint4 *d4 = reinterpret_cast<uint4 *>(p.dq + grow * D + h * (D / 2));
#pragma unroll 1
      for (int v = 0; v < D / 16; ++v) d4[v] = make_uint4(0u, 0u, 0u, 0u);
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

// ============================================================== dK / dV
// Key-stationary. TMEM: two 128-column regions R0 = [0, 128), R1 = [128, 256)
// that trade roles from tile to tile, dV at 256, dK at 256 + D. Tile n
// writes S^T(n) into R(n & 1) and dP^T(n) into the other region. Warpgroup h
// owns query columns [64h, 64h+64) and packs both of its bf16 operands into
// its own 64 columns of the S^T region: P^T(n) at 64h, dS^T(n) at 64h + 32
// (neither warpgroup waits for the other). Per query tile n:
//   dV(n) as soon as P^T(n) is in TMEM | S^T(n+1), into the region dP^T(n)
//   occupied, once the softmax has loaded dP^T(n) | dK(n) once dS^T(n) is in
//   TMEM | dP^T(n+1), into the region that holds P^T(n) and dS^T(n), once
//   dK(n) (and so dV(n)) has completed.
// S^T(n+1) therefore waits for a TMEM load, not for dV(n) to complete.
// With in-kernel RoPE (ROPE), warps 10-11 rotate the K tile once (k_ready)
// and every Q tile in shared memory (q_ready), and dK leaves through R^T at
// the key's position.
template <int D>
struct Dkdv3Cfg {
  static constexpr int NS = (D == 128) ? 2 : 4;  // Q/dO stages
  static constexpr int TILE = kTile * D * 2;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = TILE;
  static constexpr int OFF_Q = 2 * TILE;
  static constexpr int OFF_DO = OFF_Q + NS * TILE;
  static constexpr int OFF_LD = OFF_DO + NS * TILE;  // per stage: lse*log2e [128], D [128]
  static constexpr int OFF_BAR = OFF_LD + NS * 1024;
  // kv_full, fin, s_full, dp_full, k_ready, (spare), p_ready, ds_ready, dp_free, dk_done, qd_full[NS],
  // qd_empty[NS], q_ready[NS]
  static constexpr int NBAR = 10 + 3 * NS;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + kMaxTiles * 8 + 1024;   // misc, tile table, alignment slack
  static_assert(SMEM <= 232448, "over the 227 KiB of shared memory a CTA may opt into");
  static constexpr uint32_t colDV = 256, colDK = 256 + D;
  // the S^T and dP^T regions of query tile n
  static __device__ __forceinline__ uint32_t colS(int n) { return (n & 1) ? 128u : 0u; }
  static __device__ __forceinline__ uint32_t colDP(int n) { return (n & 1) ? 0u : 128u; }
};

// K/V heads per launch-order group of the dK/dV kernel.
constexpr int kDkdvHeadGroup = 2;

template <int D, bool ROPE, bool EPI = false>
__global__ void __launch_bounds__(ROPE ? 384 : 320, 1)
    dkdv2_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ Bwd2Params p) {
  using C = Dkdv3Cfg<D>;
  constexpr int NS = C::NS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = tc::smem_u32(smem);
  const uint32_t sK = sbase + C::OFF_K, sV = sbase + C::OFF_V;
  auto sQ = [&](int st) { return sbase + C::OFF_Q + st * C::TILE; };
  auto sDO = [&](int st) { return sbase + C::OFF_DO + st * C::TILE; };
  auto ld_lse = [&](int st) { return reinterpret_cast<float *>(smem + C::OFF_LD + st * 1024); };
  auto ld_D = [&](int st) { return reinterpret_cast<float *>(smem + C::OFF_LD + st * 1024 + 512); };
  const uint32_t bar0 = sbase + C::OFF_BAR;
  const uint32_t bar_kv_full = bar0, bar_fin = bar0 + 8, bar_s_full = bar0 + 16, bar_dp_full = bar0 + 24,
                 bar_p_ready = bar0 + 48,
                 bar_ds_ready = bar0 + 56, bar_dp_free = bar0 + 64, bar_dk_done = bar0 + 72;
  auto bar_qd_full = [&](int st) { return bar0 + 80 + 8 * st; };
  auto bar_qd_empty = [&](int st) { return bar0 + 80 + 8 * NS + 8 * st; };
  const uint32_t bar_k_ready = bar0 + 32;
  auto bar_q_ready = [&](int st) { return bar0 + 80 + 16 * NS + 8 * st; };
  // the barriers the MMA issuer waits on before reading K and Q
  const uint32_t bar_k_use = ROPE ? bar_k_ready : bar_kv_full;
  auto bar_q_use = [&](int st) { return ROPE ? bar_q_ready(st) : bar_qd_full(st); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
  int *ntiles_slot = reinterpret_cast<int *>(smem + C::OFF_MISC + 12);
  TileEntry *tab = reinterpret_cast<TileEntry *>(smem + C::OFF_MISC + 16);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cp = p.cp, c = p.c, tpc = p.tpc;
  // K/V head bkv, a few at a time so that the CTAs in flight share their
  // query heads' Q/dO tiles in L2, heaviest CTAs first; its group's query
  // heads are bkv*group + [0, group)
  int bkv, g;
  head_group_order<kDkdvHeadGroup>((int)blockIdx.x, 2 * cp * tpc, (int)gridDim.x / (2 * cp * tpc), bkv, g);
  const int kk_chunk = g / tpc;     // earliest keys first: they are seen by the most queries
  const int kt = g % tpc;
  int rk, hk;
  owner_of(kk_chunk, cp, rk, hk);
  const int k_z = bkv * 2 * cp + 2 * rk + hk;
  const int k_pos0 = kk_chunk * c + kt * kTile;
  const int k_rows = min(kTile, c - kt * kTile);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NBAR; ++i) {
      const uint32_t b = bar0 + 8 * i;
      uint32_t cnt = 1;
      if (b == bar_p_ready || b == bar_ds_ready || b == bar_dp_free) cnt = 256;
      if (b == bar_k_ready) cnt = 64;       // the two rotation warps
      for (int st = 0; st < NS; ++st) {
        if (b == bar_qd_full(st)) cnt = 33;   // expect_tx arrive + 32 producer lanes
        if (b == bar_q_ready(st)) cnt = 64;
      }
      tc::mbar_init(b, cnt);
    }
    abort_flag[0] = 0;
    abort_flag[1] = 0;
    tc::mbar_fence_init();
    tc::fence_proxy_async_smem();
    // the stationary K and V tiles load while the tile table is built
    tc::mbar_arrive_expect_tx(bar_kv_full, 2 * C::TILE);
    for (int blk = 0; blk < D / 64; ++blk) {
      tc::tma_load_3d(sK + blk * kTile * 128, &tm_k, bar_kv_full, blk * 64, kt * kTile, k_z);
      tc::tma_load_3d(sV + blk * kTile * 128, &tm_v, bar_kv_full, blk * 64, kt * kTile, k_z);
    }
  }
  if (warp == 8) {
    tc::tmem_alloc(tc::smem_u32(tmem_slot), 512);
    tc::tmem_relinquish();
    {
      const QBounds qb = q_bounds(p.doc_lo, p.doc_hi, p.T, p.T_valid, p.causal, k_pos0, k_pos0 + k_rows - 1);
      const int nt = build_q_table(tab, cp, c, rk, p.causal, p.T_valid, qb, k_rows < kTile, lane);
      if (lane == 0) *ntiles_slot = nt;
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int ntiles = *ntiles_slot;
  const int ntot = ntiles * p.group;   // the table once per query head of the group
  const tc::WaitCtx wc{abort_flag, p.err};
  const tc::WaitCtx drain{abort_flag + 1, p.err};

  TileInfo t;

  if (warp == 8) {
    if (lane == 0) {
      tc::tma_prefetch_desc(&tm_q);
      tc::tma_prefetch_desc(&tm_do);
    }
    int n = 0, ent = 0, gi = 0;
    while (n < ntot) {
      decode_tile(tab[ent], t);
      const int st = n % NS;
      if (n >= NS && !__all_sync(0xffffffffu, tc::mbar_wait(bar_qd_empty(st), ((n / NS) - 1) & 1, wc))) break;
      const int bq = bkv * p.group + gi;   // query head
      const int z = bq * 2 * cp + t.slot;
      if (lane == 0) {
        tc::mbar_arrive_expect_tx(bar_qd_full(st), 2 * C::TILE);
        for (int blk = 0; blk < D / 64; ++blk) {
          tc::tma_load_3d(sQ(st) + blk * kTile * 128, &tm_q, bar_qd_full(st), blk * 64, t.y0, z);
          tc::tma_load_3d(sDO(st) + blk * kTile * 128, &tm_do, bar_qd_full(st), blk * 64, t.y0, z);
        }
      }
      const long long row0 = (long long)bq * p.T + (long long)t.slot * c + t.y0;
      // All eight loads are issued before any store so their latencies overlap.
      float lv[4], dv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = lane + 32 * i;
        const bool v = r < t.nvalid;
        lv[i] = v ? __ldg(p.lse + row0 + r) * kLog2eB : INFINITY;   // ragged query rows get P = 0
        dv[i] = v ? __ldg(p.D + row0 + r) : 0.f;
      }
      float *sl = ld_lse(st), *sd = ld_D(st);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        sl[lane + 32 * i] = lv[i];
        sd[lane + 32 * i] = dv[i];
      }
      tc::mbar_arrive(bar_qd_full(st));
      ++n;
      if (++ent == ntiles) { ent = 0; ++gi; }
    }
    if (lane == 0) {
      tc::mbar_wait(bar_kv_full, 0, drain);
      for (int m = (n > NS ? n - NS : 0); m < n; ++m) tc::mbar_wait(bar_qd_full(m % NS), (m / NS) & 1, drain);
    }
  } else if (warp == 9) {
    {   // the whole warp runs the issue loop; elect.sync picks the issuing lane
      constexpr uint32_t idS = tc::idesc_bf16(128, 128, false, false);
      constexpr uint32_t idA = tc::idesc_bf16(128, D, false, true);
      const uint64_t ak0 = tc::kdesc0(sK), av0 = tc::kdesc0(sV);
      auto issue_s = [&](int st, int n) {   // S^T(n) into its tile's region
        const uint64_t bq = tc::kdesc0(sQ(st));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc::mma_ss_w(tmem + C::colS(n), ak0 + tc::koff(kTile, kk), bq + tc::koff(kTile, kk), idS, kk > 0 ? 1u : 0u);
        tc::mma_commit_w(bar_s_full);
      };
      auto issue_dp = [&](int st, int n) {   // dP^T(n)
        const uint64_t bo = tc::kdesc0(sDO(st));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc::mma_ss_w(tmem + C::colDP(n), av0 + tc::koff(kTile, kk), bo + tc::koff(kTile, kk), idS, kk > 0 ? 1u : 0u);
        tc::mma_commit_w(bar_dp_full);
      };
      auto wait_all = [&](uint32_t bar, uint32_t par, const tc::WaitCtx &w) {
        return __all_sync(0xffffffffu, tc::mbar_wait(bar, par, w));
      };
      bool ok = wait_all(bar_k_use, 0, wc);
      if (ok && ntot > 0) {
        ok = wait_all(bar_q_use(0), 0, wc);
        if (ok) {
          tc::tc_fence_after();
          issue_s(0, 0);
          issue_dp(0, 0);
        }
        for (int n = 0; ok; ++n) {
          const bool more = n + 1 < ntot;
          const int st = n % NS, st1 = (n + 1) % NS;
          const uint32_t acc0 = n > 0 ? 1u : 0u;
          if (!(ok = wait_all(bar_p_ready, n & 1, wc))) break;
          tc::tc_fence_after();
          {   // dV += P^T(n) dO(n): P^T of warpgroup h at colS(n) + 64h
            const uint64_t bo = tc::mndesc0(sDO(st), kTile);
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              tc::mma_ts_w(tmem + C::colDV, tmem + C::colS(n) + kk * 8 + (kk >= 4 ? 32 : 0), bo + tc::mnoff(kk), idA,
                         kk > 0 ? 1u : acc0);
          }
          // S^T(n+1) goes ahead of dK(n): it starts the next tile's
          // exponentials, the longest phase of a tile, while dK(n) and
          // dP^T(n+1) run. It overwrites dP^T(n), which the softmax has loaded.
          if (more) {
            if (!(ok = wait_all(bar_q_use(st1), ((n + 1) / NS) & 1, wc))) break;
            if (!(ok = wait_all(bar_dp_free, n & 1, wc))) break;
            tc::tc_fence_after();
            issue_s(st1, n + 1);
          }
          if (!(ok = wait_all(bar_ds_ready, n & 1, wc))) break;
          tc::tc_fence_after();
          {   // dK += dS^T(n) Q(n): dS^T of warpgroup h at colS(n) + 64h + 32
            const uint64_t bq = tc::mndesc0(sQ(st), kTile);
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              tc::mma_ts_w(tmem + C::colDK, tmem + C::colS(n) + 32 + kk * 8 + (kk >= 4 ? 32 : 0), bq + tc::mnoff(kk),
                         idA, kk > 0 ? 1u : acc0);
            tc::mma_commit_w(bar_dk_done);
            tc::mma_commit_w(bar_qd_empty(st));
          }
          if (!more) break;
          // dP^T(n+1) overwrites P^T(n) and dS^T(n): after dV(n) and dK(n)
          if (!(ok = wait_all(bar_dk_done, n & 1, wc))) break;
          tc::tc_fence_after();
          issue_dp(st1, n + 1);
        }
      }
      tc::mma_commit_w(bar_fin);
      wait_all(bar_fin, 0, drain);
    }
  } else if (ROPE && warp >= 10) {
    // ------------------------------------------------ RoPE rotation warps (K once, Q tiles)
    tc::RopeRows<D, 64> rr;   // warps 10-11
    rr.init((warp - 10) * 32 + lane, p.theta);
    if (__all_sync(0xffffffffu, tc::mbar_wait(bar_kv_full, 0, wc))) {
      rr.rotate(smem + C::OFF_K, k_pos0);
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(bar_k_ready);
      int n = 0, ent = 0;
      while (n < ntot) {
        decode_tile(tab[ent], t);
        const int st = n % NS;
        if (!__all_sync(0xffffffffu, tc::mbar_wait(bar_qd_full(st), (n / NS) & 1, wc))) break;
        rr.rotate(smem + C::OFF_Q + st * C::TILE, t.pos0);
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(bar_q_ready(st));
        ++n;
        if (++ent == ntiles) ent = 0;
      }
    }
  } else {
    // -------------------------------------------- softmax warpgroups (query halves)
    const int h = warp >> 2;
    const int row = threadIdx.x & 127;     // key row of the tile
    const int k_pos = k_pos0 + row;
    const bool valid = row < k_rows;
    const uint32_t t_row = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const long long grow = (long long)bkv * p.T + (long long)(2 * c * rk + hk * c + kt * kTile + row);
    const float sl2 = p.scale_log2;
    int dlo, dhi;   // this key row's document [dlo, dhi)
    doc_bounds_at(p.doc_lo, p.doc_hi, min(k_pos, p.T - 1), p.T, dlo, dhi);
    int n = 0, ent = 0;
    bool ok = true;
    while (n < ntot) {
      decode_tile(tab[ent], t);
      const int st = n % NS;
      ok = __all_sync(0xffffffffu, tc::mbar_wait(bar_s_full, n & 1, wc));
      if (!ok) break;
      tc::tc_fence_after();
      const uint32_t sl = tc::smem_u32(ld_lse(st)) + 4u * (64 * h), sd = tc::smem_u32(ld_D(st)) + 4u * (64 * h);
      // Queries kept: columns lo <= q < hi: q >= k (causal), dlo <= pos0 + q <
      // dhi (packed documents), none for padding keys; ragged query columns
      // carry LSE = +inf, so their P is 0 already.
      int lo = 0, hi = kTile;
      if (t.need_mask) {
        if (k_pos >= p.T_valid) {
          lo = kTile;
        } else {
          lo = max(p.causal ? k_pos - t.pos0 : 0, dlo - t.pos0);
          hi = dhi - t.pos0;
        }
      }
      lo -= 64 * h;
      hi -= 64 * h;
      float pr[64];
      {
        uint32_t r[2][32];
        tc::tmem_ld32(t_row + C::colS(n) + 64 * h, r[0]);
        tc::tmem_ld32(t_row + C::colS(n) + 64 * h + 32, r[1]);
        tc::tmem_ld_wait();
        const uint64_t sl2x2 = tc::f2(sl2, sl2);
#pragma unroll
        for (int q4 = 0; q4 < 16; ++q4) {
          const float4 l4 = tc::lds_f4(sl + 16u * q4);
          const int q = 4 * q4;
          float x0, x1, x2, x3;
          tc::unf2(tc::ffma2(tc::f2(__uint_as_float(r[q >> 5][q & 31]), __uint_as_float(r[q >> 5][(q & 31) + 1])),
                             sl2x2, tc::f2(-l4.x, -l4.y)), x0, x1);
          tc::unf2(tc::ffma2(tc::f2(__uint_as_float(r[q >> 5][(q & 31) + 2]), __uint_as_float(r[q >> 5][(q & 31) + 3])),
                             sl2x2, tc::f2(-l4.z, -l4.w)), x2, x3);
          pr[q] = tc::ex2(x0);
          pr[q + 1] = tc::ex2(x1);
          pr[q + 2] = tc::ex2(x2);
          pr[q + 3] = tc::ex2(x3);
        }
        if (__any_sync(0xffffffffu, lo > 0 || hi < 64)) {
          const unsigned width = (unsigned)max(hi - lo, 0);
#pragma unroll
          for (int q = 0; q < 64; ++q)
            if ((unsigned)(q - lo) >= width) pr[q] = 0.f;
        }
      }
#pragma unroll
      for (int cb = 0; cb < 2; ++cb) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(pr[cb * 32 + 2 * e], pr[cb * 32 + 2 * e + 1]);
        tc::tmem_st16(t_row + C::colS(n) + 64 * h + cb * 16, pk);   // P^T
      }
      tc::tmem_st_wait();
      tc::tc_fence_before();
      tc::mbar_arrive(bar_p_ready);
      ok = __all_sync(0xffffffffu, tc::mbar_wait(bar_dp_full, n & 1, wc));
      if (!ok) break;
      tc::tc_fence_after();
      {
        uint32_t rd[2][32];
        tc::tmem_ld32(t_row + C::colDP(n) + 64 * h, rd[0]);
        tc::tmem_ld32(t_row + C::colDP(n) + 64 * h + 32, rd[1]);
        tc::tmem_ld_wait();
        tc::tc_fence_before();
        tc::mbar_arrive(bar_dp_free);   // S^T(n+1) may now overwrite dP^T(n)
#pragma unroll
        for (int q4 = 0; q4 < 16; ++q4) {
          const float4 d4 = tc::lds_f4(sd + 16u * q4);
          const int q = 4 * q4;
          const uint64_t a = tc::fmul2(tc::f2(pr[q], pr[q + 1]),
                                       tc::fadd2(tc::f2(__uint_as_float(rd[q >> 5][q & 31]), __uint_as_float(rd[q >> 5][(q & 31) + 1])),
                                                 tc::f2(-d4.x, -d4.y)));
          const uint64_t b = tc::fmul2(tc::f2(pr[q + 2], pr[q + 3]),
                                       tc::fadd2(tc::f2(__uint_as_float(rd[q >> 5][(q & 31) + 2]), __uint_as_float(rd[q >> 5][(q & 31) + 3])),
                                                 tc::f2(-d4.z, -d4.w)));
          tc::unf2(a, pr[q], pr[q + 1]);
          tc::unf2(b, pr[q + 2], pr[q + 3]);
        }
      }
#pragma unroll
      for (int cb = 0; cb < 2; ++cb) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(pr[cb * 32 + 2 * e], pr[cb * 32 + 2 * e + 1]);
        tc::tmem_st16(t_row + C::colS(n) + 64 * h + 32 + cb * 16, pk);   // dS^T
      }
      tc::tmem_st_wait();
      tc::tc_fence_before();
      tc::mbar_arrive(bar_ds_ready);
      ++n;
      if (++ent == ntiles) ent = 0;
    }
    if (ok) {
      __nv_bfloat16 *dst = (h == 0 ? p.dv : p.dk) + grow * D;
      if (n > 0) {
        ok = __all_sync(0xffffffffu, tc::mbar_wait(bar_dk_done, (n - 1) & 1, wc));
        if (ok) {
          tc::tc_fence_after();
          if ((ROPE || EPI) && h == 1) {   // dK = R^T dK' at the key's position
#pragma unroll 1
            for (int a = 0; a < D / 64; ++a)
              store_tmem_pair_rope<D>(t_row + C::colDK, a, p.scale, k_pos, p.theta, dst, valid);
          } else {
            store_tmem_cols(t_row + (h == 0 ? C::colDV : C::colDK), 0, D / 32, h == 0 ? 1.f : p.scale, dst, valid);
          }
        }
      } else if (valid) {   // no query sees these keys (all padding): zero gradients
        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
        for (int v = 0; v < D / 8; ++v) d4[v] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

template <int D, bool ROPE, bool EPI = false>
cpattn_status launch_dkdv2_t(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                             const CUtensorMap &mdo, const Bwd2Params &bp, unsigned grid, cudaStream_t s) {
  constexpr int threads = ROPE ? 384 : 320;
  constexpr int smem = Dkdv3Cfg<D>::SMEM;
  auto kern = dkdv2_tc_kernel<D, ROPE, EPI>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return fail(CPATTN_ERR_CUDA, "cannot set %d bytes of shared memory for the dK/dV kernel", smem);
  kern<<<grid / bp.group, threads, smem, s>>>(mq, mk, mv, mdo, bp);   // one CTA per K/V-head key tile
  return check_launch("tensor-core dK/dV kernel (pipelined)");
}

template <int D, bool ROPE, bool EPI = false>
cpattn_status launch_dq2_t(const CUtensorMap &mk, const CUtensorMap &mv, const Bwd2Params &bp, unsigned grid,
                           cudaStream_t s) {
  constexpr int threads = ROPE ? 384 : 320;
  constexpr int smem = Dq3Cfg<D>::SMEM;
  auto kern = dq2_tc_kernel<D, ROPE, EPI>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return fail(CPATTN_ERR_CUDA, "cannot set %d bytes of shared memory for the dQ kernel", smem);
  kern<<<grid, threads, smem, s>>>(mk, mv, bp);
  return check_launch("tensor-core dQ kernel (pipelined)");
}

}  // namespace

cpattn_status launch_bwd2_bf16(const void *q, const void *k, const void *v, const float *lse,
                               const void *dO, void *dq, void *dk, void *dv, float *D,
                               const Geometry &g, cudaStream_t s) {
  const long long BH = (long long)g.B * g.H;
  const long long n_slots = BH * 2 * g.cp;
  const long long n_kv_slots = (long long)g.B * g.Hkv * 2 * g.cp;
  CUtensorMap mq, mk, mv, mdo;
  if (!make_tile_map(&mq, q, g.d, g.c, n_slots) || !make_tile_map(&mk, k, g.d, g.c, n_kv_slots) ||
      !make_tile_map(&mv, v, g.d, g.c, n_kv_slots) || !make_tile_map(&mdo, dO, g.d, g.c, n_slots))
    return fail(CPATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed (is the driver too old?)");
  Bwd2Params bp;
  bp.q = static_cast<const __nv_bfloat16 *>(q);
  bp.dO = static_cast<const __nv_bfloat16 *>(dO);
  bp.lse = lse;
  bp.D = D;
  bp.dq = static_cast<__nv_bfloat16 *>(dq);
  bp.dk = static_cast<__nv_bfloat16 *>(dk);
  bp.dv = static_cast<__nv_bfloat16 *>(dv);
  bp.err = device_err_flag();
  bp.BH = (int)BH;
  bp.group = g.H / g.Hkv;
  bp.doc_lo = g.doc_lo;
  bp.doc_hi = g.doc_hi;
  bp.T = g.T;
  bp.T_valid = g.T_valid;
  bp.c = g.c;
  bp.cp = g.cp;
  bp.causal = g.causal;
  bp.tpc = (g.c + kTile - 1) / kTile;
  bp.scale = (float)(1.0 / sqrt((double)g.d));
  bp.scale_log2 = (float)(1.4426950408889634 / sqrt((double)g.d));
  make_rope_theta(g.d, &bp.theta, g.rope_cfg);
  const long long grid = BH * 2 * g.cp * bp.tpc;
  if (grid > 0x7fffffffLL) return fail(CPATTN_ERR_SHAPE, "too many tiles");
  const unsigned gr = (unsigned)grid;
  cpattn_status st;
  if (g.o_for_D) {   // the paired dQ kernel computes D (for its rows and for dK/dV) and runs first
    trace_record(4, s);
    if ((st = launch_dq_pair_bf16(q, k, v, lse, dO, dq, D, g, s)) != CPATTN_OK) return st;
    trace_record(5, s);
  }
  trace_record(2, s);
  if (g.d == 128)
    st = g.rope ? launch_dkdv2_t<128, true>(mq, mk, mv, mdo, bp, gr, s)
         : g.rope_epi ? launch_dkdv2_t<128, false, true>(mq, mk, mv, mdo, bp, gr, s)
                      : launch_dkdv2_t<128, false>(mq, mk, mv, mdo, bp, gr, s);
  else
    st = g.rope ? launch_dkdv2_t<64, true>(mq, mk, mv, mdo, bp, gr, s)
         : g.rope_epi ? launch_dkdv2_t<64, false, true>(mq, mk, mv, mdo, bp, gr, s)
                      : launch_dkdv2_t<64, false>(mq, mk, mv, mdo, bp, gr, s);
  if (st != CPATTN_OK) return st;
  trace_record(3, s);
  if (g.o_for_D) return CPATTN_OK;
  // dQ: CTA pairs with two-SM MMAs at d = 128 when q, k arrive rotated (or
  // without RoPE); the one-CTA pipelined kernel otherwise.
  trace_record(4, s);
  if (g.d == 128 && !g.rope) st = launch_dq_pair_bf16(q, k, v, lse, dO, dq, D, g, s);
  else if (g.d == 128) st = launch_dq2_t<128, true>(mk, mv, bp, gr, s);
  else if (g.rope) st = launch_dq2_t<64, true>(mk, mv, bp, gr, s);
  else st = g.rope_epi ? launch_dq2_t<64, false, true>(mk, mv, bp, gr, s) : launch_dq2_t<64, false>(mk, mv, bp, gr, s);
  trace_record(5, s);
  return st;
}

}  // namespace cpattn
