// Ring attention backward on tcgen05 tensor cores, without atomics.
//
// With P = exp(S - LSE) recomputed from the forward's LSE and D = rowsum(dO*O)
// (Claude Logs, 2026-03-24, the D correction):
//   dV = P^T dO,  dS = P * (dO V^T - D),  dK = scale dS^T Q,  dQ = scale dS K.
// Two kernels split the work so that every output tile has one owner:
//  * dkdv_tc_kernel: one CTA per 128-key tile (key-stationary). It visits the
//    query tiles of every rank in ring order -- at step s its K/V sit on rank
//    (j + s) mod cp -- and keeps dK, dV in TMEM across all steps: the ring's
//    travelling dK/dV accumulator that returns to its owner (Claude Logs,
//    2026-06-22, 2026-03-28 "Phase 3"), here never leaving the SM.
//  * dq_tc_kernel: one CTA per 128-query tile (query-stationary), walking the
//    K/V tiles in the forward's ring order and keeping dQ in TMEM. The pages
//    accumulated dQ with atomicAdd (Claude Logs, 2026-04-20); owning the tile
//    instead costs a recomputation of S and dP.
// In both, the softmax warpgroup turns S, dP (fp32, TMEM) into P, dS (bf16),
// written back into TMEM over S / dP, and the next MMAs take them as their A
// operand straight from TMEM.
#include <math.h>

#include "attn_common.cuh"

namespace cpattn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

struct BwdParams {
  const float *lse;  // [BH, T] natural-log LSE, sharded rows
  const float *D;    // [BH, T] rowsum(dO * O)
  __nv_bfloat16 *out0, *out1;  // dkdv: dK, dV ; dq: dQ, unused
  int *err;
  int BH, T, T_valid, c, cp, causal, tpc;
  int group;   // query heads per K/V head
  const int *doc_lo, *doc_hi;   // packed documents: [T] bounds per natural position, or nullptr
  float scale;       // 1/sqrt(d)
  float scale_log2;  // log2(e)/sqrt(d)
  RopeTheta theta;
};

// Epilogue of one accumulator row (D fp32 columns in TMEM at `taddr`):
// x = scale * acc, then m R(pos)^T when ROPE (pairs (i, i + D/2); m the
// RoPE configuration's temperature, 1 for the standard rotation), rounded to
// bf16 and stored at `dst` when `valid`. Columns are taken as pairs of 32-wide
// chunks [32h, 32h+32) and [D/2 + 32h, D/2 + 32h + 32) so each RoPE pair is
// in registers at once. Every lane of the warp must call this (tcgen05.ld).
template <int D, bool ROPE>
__device__ __forceinline__ void epilogue_row(uint32_t taddr, float scale, int pos,
                                             const RopeTheta &th, __nv_bfloat16 *dst, bool valid) {
#pragma unroll 1
  for (int h = 0; h < D / 64; ++h) {
    uint32_t a[32], b[32];
    tc::tmem_ld32(taddr + 32 * h, a);
    tc::tmem_ld32(taddr + D / 2 + 32 * h, b);
    tc::tmem_ld_wait();
    uint32_t pa[16], pb[16];
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      float x0 = __uint_as_float(a[e]) * scale, x1 = __uint_as_float(a[e + 1]) * scale;
      float y0 = __uint_as_float(b[e]) * scale, y1 = __uint_as_float(b[e + 1]) * scale;
      if (ROPE) {
        float s0, c0, s1, c1;
        rope_sincos(pos, th.hi[32 * h + e], th.lo[32 * h + e], s0, c0);
        rope_sincos(pos, th.hi[32 * h + e + 1], th.lo[32 * h + e + 1], s1, c1);
        c0 *= th.mscale; s0 *= th.mscale; c1 *= th.mscale; s1 *= th.mscale;
        const float u0 = fmaf(x0, c0, y0 * s0), w0 = fmaf(y0, c0, -x0 * s0);
        const float u1 = fmaf(x1, c1, y1 * s1), w1 = fmaf(y1, c1, -x1 * s1);
        x0 = u0; y0 = w0; x1 = u1; y1 = w1;
      }
      pa[e / 2] = pack_bf16x2(x0, x1);
      pb[e / 2] = pack_bf16x2(y0, y1);
    }
    if (valid) {
      uint4 *da = reinterpret_cast<uint4 *>(dst + 32 * h);
      uint4 *db = reinterpret_cast<uint4 *>(dst + D / 2 + 32 * h);
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        da[v] = make_uint4(pa[4 * v], pa[4 * v + 1], pa[4 * v + 2], pa[4 * v + 3]);
        db[v] = make_uint4(pb[4 * v], pb[4 * v + 1], pb[4 * v + 2], pb[4 * v + 3]);
      }
    }
  }
}

template <int D>
__device__ __forceinline__ void store_zero_row(__nv_bfloat16 *dst) {
  uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
  for (int v = 0; v < D / 8; ++v) d4[v] = make_uint4(0u, 0u, 0u, 0u);
}

// ============================================================ dK / dV kernel
template <int D>
struct DkdvCfg {
  static constexpr int NS = (D == 128) ? 2 : 4;  // Q/dO pipeline stages
  static constexpr int TILE = kTile * D * 2;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = TILE;
  static constexpr int OFF_Q = 2 * TILE;
  static constexpr int OFF_DO = OFF_Q + NS * TILE;
  static constexpr int OFF_LD = OFF_DO + NS * TILE;        // per stage: lse2[128], D[128]
  static constexpr int OFF_BAR = OFF_LD + NS * 1024;
  // kv_full, k_ready, fin, s_full, p_full, mma_done, qd_full[NS], q_ready[NS], qd_empty[NS]
  static constexpr int NBAR = 6 + 3 * NS;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;
};

template <int D, bool ROPE>
__global__ void __launch_bounds__(ROPE ? 320 : 192, 1)
    dkdv_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                   const __grid_constant__ BwdParams p) {
  using C = DkdvCfg<D>;
  constexpr int NS = C::NS;
  constexpr uint32_t colS = 0, colDP = 128, colDV = 256, colDK = 256 + D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = tc::smem_u32(smem);
  const uint32_t sK = sbase + C::OFF_K, sV = sbase + C::OFF_V;
  auto sQ = [&](int st) { return sbase + C::OFF_Q + st * C::TILE; };
  auto sDO = [&](int st) { return sbase + C::OFF_DO + st * C::TILE; };
  auto ld_lse = [&](int st) { return reinterpret_cast<float *>(smem + C::OFF_LD + st * 1024); };
  auto ld_D = [&](int st) { return reinterpret_cast<float *>(smem + C::OFF_LD + st * 1024 + 512); };
  const uint32_t bar0 = sbase + C::OFF_BAR;
  const uint32_t bar_kv_full = bar0, bar_k_ready = bar0 + 8, bar_fin = bar0 + 16, bar_s_full = bar0 + 24,
                 bar_p_full = bar0 + 32, bar_mma_done = bar0 + 40;
  auto bar_qd_full = [&](int st) { return bar0 + 48 + 8 * st; };
  auto bar_q_ready = [&](int st) { return bar0 + 48 + 8 * NS + 8 * st; };
  auto bar_qd_empty = [&](int st) { return bar0 + 48 + 16 * NS + 8 * st; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cp = p.cp, c = p.c, tpc = p.tpc;
  // Key tile: earliest natural position first (it is seen by the most queries).
  const int BHkv = p.BH / p.group;
  const int bkv = blockIdx.x % BHkv;               // K/V head
  const int g = blockIdx.x / BHkv;
  const int kk_chunk = g / tpc;
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
      if (b == bar_k_ready || b == bar_p_full) cnt = 128;
      for (int st = 0; st < NS; ++st) {
        if (b == bar_q_ready(st)) cnt = 128;
        if (b == bar_qd_full(st)) cnt = 33;   // expect_tx arrive + 32 producer lanes
      }
      tc::mbar_init(b, cnt);
    }
    abort_flag[0] = 0;
    abort_flag[1] = 0;
    tc::mbar_fence_init();
  }
  if (warp == 4) {
    tc::tmem_alloc(tc::smem_u32(tmem_slot), 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const tc::WaitCtx wc{abort_flag, p.err};
  const tc::WaitCtx drain{abort_flag + 1, p.err};

  GroupQSchedule sched;
  {
    const QBounds qb = q_bounds(p.doc_lo, p.doc_hi, p.T, p.T_valid, p.causal, k_pos0, k_pos0 + k_rows - 1);
    sched.init(p.group, cp, c, rk, p.causal, p.T_valid, k_pos0, k_pos0 + k_rows - 1, qb.q_lo, qb.q_hi,
               qb.doc_lo_max, qb.doc_hi_min);
  }
  const int k_ragged = k_rows < kTile;
  TileInfo t;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tc::tma_prefetch_desc(&tm_q);
      tc::tma_prefetch_desc(&tm_do);
      tc::mbar_arrive_expect_tx(bar_kv_full, 2 * C::TILE);
      for (int blk = 0; blk < D / 64; ++blk) {
        tc::tma_load_3d(sK + blk * kTile * 128, &tm_k, bar_kv_full, blk * 64, kt * kTile, k_z);
        tc::tma_load_3d(sV + blk * kTile * 128, &tm_v, bar_kv_full, blk * 64, kt * kTile, k_z);
      }
    }
    int n = 0;
    while (sched.next(t, k_ragged)) {
      const int st = n % NS;
      if (n >= NS && !__all_sync(0xffffffffu, tc::mbar_wait(bar_qd_empty(st), ((n / NS) - 1) & 1, wc))) break;
      const int bq = bkv * p.group + sched.gi;   // query head
      const int z = bq * 2 * cp + t.slot;
      if (lane == 0) {
        tc::mbar_arrive_expect_tx(bar_qd_full(st), 2 * C::TILE);
        for (int blk = 0; blk < D / 64; ++blk) {
          tc::tma_load_3d(sQ(st) + blk * kTile * 128, &tm_q, bar_qd_full(st), blk * 64, t.y0, z);
          tc::tma_load_3d(sDO(st) + blk * kTile * 128, &tm_do, bar_qd_full(st), blk * 64, t.y0, z);
        }
      }
      const long long row0 = (long long)bq * p.T + (long long)t.slot * c + t.y0;
      float lv[4], dv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = lane + 32 * i;
        const bool v = r < t.nvalid;
        lv[i] = v ? __ldg(p.lse + row0 + r) * kLog2e : INFINITY;   // ragged query rows get P = 0
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
    }
    if (lane == 0) {
      tc::mbar_wait(bar_kv_full, 0, drain);
      for (int m = (n > NS ? n - NS : 0); m < n; ++m) tc::mbar_wait(bar_qd_full(m % NS), (m / NS) & 1, drain);
    }
  } else if (warp == 5) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idSS = tc::idesc_bf16(128, 128, false, false);
      constexpr uint32_t idAcc = tc::idesc_bf16(128, D, false, true);
      bool ok = tc::mbar_wait(bar_kv_full, 0, wc) && (!ROPE || tc::mbar_wait(bar_k_ready, 0, wc));
      for (int n = 0; ok && sched.next(t, k_ragged); ++n) {
        const int st = n % NS;
        if (!tc::mbar_wait(bar_qd_full(st), (n / NS) & 1, wc)) break;
        if (ROPE && !tc::mbar_wait(bar_q_ready(st), (n / NS) & 1, wc)) break;
        if (n >= 1 && !tc::mbar_wait(bar_mma_done, (n - 1) & 1, wc)) break;
        tc::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc::mma_ss(tmem + colS, tc::desc_kmajor(sK, kTile, kk), tc::desc_kmajor(sQ(st), kTile, kk), idSS, kk > 0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc::mma_ss(tmem + colDP, tc::desc_kmajor(sV, kTile, kk), tc::desc_kmajor(sDO(st), kTile, kk), idSS, kk > 0);
        tc::mma_commit(bar_s_full);
        if (!tc::mbar_wait(bar_p_full, n & 1, wc)) break;
        tc::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          tc::mma_ts(tmem + colDV, tmem + colS + kk * 8, tc::desc_mnmajor(sDO(st), kTile, kk), idAcc,
                     (n > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          tc::mma_ts(tmem + colDK, tmem + colDP + kk * 8, tc::desc_mnmajor(sQ(st), kTile, kk), idAcc,
                     (n > 0 || kk > 0) ? 1u : 0u);
        tc::mma_commit(bar_mma_done);
        tc::mma_commit(bar_qd_empty(st));
      }
      tc::mma_commit(bar_fin);
      tc::mbar_wait(bar_fin, 0, drain);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------- softmax
    const int row = threadIdx.x;           // key row of the tile
    const int k_pos = k_pos0 + row;
    const uint32_t t_row = tmem + ((uint32_t)(warp * 32) << 16);
    const float sl2 = p.scale_log2;
    int dlo, dhi;   // this key's document [dlo, dhi) (everything without packed documents)
    doc_bounds_at(p.doc_lo, p.doc_hi, min(k_pos, p.T - 1), p.T, dlo, dhi);
    int n = 0;
    bool ok = true;
    while (sched.next(t, k_ragged)) {
      const int st = n % NS;
      ok = __all_sync(0xffffffffu, tc::mbar_wait(bar_s_full, n & 1, wc));
      if (!ok) break;
      tc::tc_fence_after();
      const float *sl = ld_lse(st), *sd = ld_D(st);
#pragma unroll 1
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t rs[32], rd[32];
        tc::tmem_ld32(t_row + colS + cb * 32, rs);
        tc::tmem_ld32(t_row + colDP + cb * 32, rd);
        tc::tmem_ld_wait();
        uint32_t pk[16], dk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float pv[2], dsv[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int q = cb * 32 + 2 * e + h;
            float pr = exp2f(fmaf(__uint_as_float(rs[2 * e + h]), sl2, -sl[q]));
            if (t.need_mask) {
              const int q_pos = t.pos0 + q;
              if ((p.causal && k_pos > q_pos) || k_pos >= p.T_valid || q_pos < dlo || q_pos >= dhi) pr = 0.f;
            }
            pv[h] = pr;
            dsv[h] = pr * (__uint_as_float(rd[2 * e + h]) - sd[q]);
          }
          pk[e] = pack_bf16x2(pv[0], pv[1]);
          dk[e] = pack_bf16x2(dsv[0], dsv[1]);
        }
        tc::tmem_st16(t_row + colS + cb * 16, pk);
        tc::tmem_st16(t_row + colDP + cb * 16, dk);
      }
      tc::tmem_st_wait();
      tc::tc_fence_before();
      tc::mbar_arrive(bar_p_full);
      ++n;
    }
    if (ok) {
      const bool valid = row < k_rows;
      const long long grow = (long long)bkv * p.T + (long long)(2 * c * rk + hk * c + kt * kTile + row);
      if (n > 0) {
        ok = __all_sync(0xffffffffu, tc::mbar_wait(bar_mma_done, (n - 1) & 1, wc));
        if (ok) {
          tc::tc_fence_after();
          epilogue_row<D, false>(t_row + colDV, 1.f, k_pos, p.theta, p.out1 + grow * D, valid);
          epilogue_row<D, ROPE>(t_row + colDK, p.scale, k_pos, p.theta, p.out0 + grow * D, valid);
        }
      } else if (valid) {   // no query sees these keys (all padding): zero gradients
        store_zero_row<D>(p.out0 + grow * D);
        store_zero_row<D>(p.out1 + grow * D);
      }
    }
  } else if (ROPE) {
    // ------------------------------------------------ RoPE transform warps
    const int wid = warp - 6;
    if (tc::mbar_wait(bar_kv_full, 0, wc)) {
      tc::rope_tile<D>(smem + C::OFF_K, k_pos0, wid, lane, p.theta);
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(bar_k_ready);
      int n = 0;
      while (sched.next(t, k_ragged)) {
        const int st = n % NS;
        if (!tc::mbar_wait(bar_qd_full(st), (n / NS) & 1, wc)) break;
        tc::rope_tile<D>(smem + C::OFF_Q + st * C::TILE, t.pos0, wid, lane, p.theta);
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(bar_q_ready(st));
        ++n;
      }
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

// =============================================================== dQ kernel
template <int D>
struct DqCfg {
  static constexpr int NS = (D == 128) ? 2 : 4;  // K/V pipeline stages
  static constexpr int TILE = kTile * D * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = TILE;
  static constexpr int OFF_K = 2 * TILE;
  static constexpr int OFF_V = OFF_K + NS * TILE;
  static constexpr int OFF_BAR = OFF_V + NS * TILE;
  // q_full, q_ready, fin, s_full, p_full, mma_done, kv_full[NS], k_ready[NS], kv_empty[NS]
  static constexpr int NBAR = 6 + 3 * NS;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;
};

template <int D, bool ROPE>
__global__ void __launch_bounds__(ROPE ? 320 : 192, 1)
    dq_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                 const __grid_constant__ BwdParams p) {
  using C = DqCfg<D>;
  constexpr int NS = C::NS;
  constexpr uint32_t colS = 0, colDP = 128, colDQ = 256;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = tc::smem_u32(smem);
  const uint32_t sQ = sbase + C::OFF_Q, sDO = sbase + C::OFF_DO;
  auto sK = [&](int st) { return sbase + C::OFF_K + st * C::TILE; };
  auto sV = [&](int st) { return sbase + C::OFF_V + st * C::TILE; };
  const uint32_t bar0 = sbase + C::OFF_BAR;
  const uint32_t bar_q_full = bar0, bar_q_ready = bar0 + 8, bar_fin = bar0 + 16, bar_s_full = bar0 + 24,
                 bar_p_full = bar0 + 32, bar_mma_done = bar0 + 40;
  auto bar_kv_full = [&](int st) { return bar0 + 48 + 8 * st; };
  auto bar_k_ready = [&](int st) { return bar0 + 48 + 8 * NS + 8 * st; };
  auto bar_kv_empty = [&](int st) { return bar0 + 48 + 16 * NS + 8 * st; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cp = p.cp, c = p.c, tpc = p.tpc;
  const int bh = blockIdx.x % p.BH;
  const int bkv = bh / p.group;                    // K/V head of this query head
  const int g = blockIdx.x / p.BH;
  const int kq = 2 * cp - 1 - g / tpc;
  const int qt = tpc - 1 - g % tpc;
  int rq, hq;
  owner_of(kq, cp, rq, hq);
  const int q_z = bh * 2 * cp + 2 * rq + hq;
  const int q_pos0 = kq * c + qt * kTile;
  const int q_rows = min(kTile, c - qt * kTile);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NBAR; ++i) {
      const uint32_t b = bar0 + 8 * i;
      uint32_t cnt = (b == bar_q_ready || b == bar_p_full) ? 128 : 1;
      for (int st = 0; st < NS; ++st)
        if (b == bar_k_ready(st)) cnt = 128;
      tc::mbar_init(b, cnt);
    }
    abort_flag[0] = 0;
    abort_flag[1] = 0;
    tc::mbar_fence_init();
  }
  if (warp == 4) {
    tc::tmem_alloc(tc::smem_u32(tmem_slot), 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const tc::WaitCtx wc{abort_flag, p.err};
  const tc::WaitCtx drain{abort_flag + 1, p.err};

  KvSchedule sched;
  {
    const KvBounds kb = kv_bounds(p.doc_lo, p.doc_hi, p.T, p.T_valid, p.causal, q_pos0, q_pos0 + q_rows - 1);
    sched.init(cp, c, rq, p.causal, p.T_valid, q_pos0, q_pos0 + q_rows - 1, kb.key_lo, kb.key_hi,
               kb.doc_lo_max, kb.doc_hi_min);
  }
  TileInfo t;

  if (warp == 4) {
    if (lane == 0) {
      tc::tma_prefetch_desc(&tm_k);
      tc::tma_prefetch_desc(&tm_v);
      tc::mbar_arrive_expect_tx(bar_q_full, 2 * C::TILE);
      for (int blk = 0; blk < D / 64; ++blk) {
        tc::tma_load_3d(sQ + blk * kTile * 128, &tm_q, bar_q_full, blk * 64, qt * kTile, q_z);
        tc::tma_load_3d(sDO + blk * kTile * 128, &tm_do, bar_q_full, blk * 64, qt * kTile, q_z);
      }
      int n = 0;
      while (sched.next(t)) {
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
      tc::mbar_wait(bar_q_full, 0, drain);
      for (int m = (n > NS ? n - NS : 0); m < n; ++m) tc::mbar_wait(bar_kv_full(m % NS), (m / NS) & 1, drain);
    }
  } else if (warp == 5) {
    if (lane == 0) {
      constexpr uint32_t idSS = tc::idesc_bf16(128, 128, false, false);
      constexpr uint32_t idAcc = tc::idesc_bf16(128, D, false, true);
      bool ok = tc::mbar_wait(ROPE ? bar_q_ready : bar_q_full, 0, wc);
      for (int n = 0; ok && sched.next(t); ++n) {
        const int st = n % NS;
        if (!tc::mbar_wait(bar_kv_full(st), (n / NS) & 1, wc)) break;
        if (ROPE && !tc::mbar_wait(bar_k_ready(st), (n / NS) & 1, wc)) break;
        if (n >= 1 && !tc::mbar_wait(bar_mma_done, (n - 1) & 1, wc)) break;
        tc::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc::mma_ss(tmem + colS, tc::desc_kmajor(sQ, kTile, kk), tc::desc_kmajor(sK(st), kTile, kk), idSS, kk > 0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc::mma_ss(tmem + colDP, tc::desc_kmajor(sDO, kTile, kk), tc::desc_kmajor(sV(st), kTile, kk), idSS, kk > 0);
        tc::mma_commit(bar_s_full);
        if (!tc::mbar_wait(bar_p_full, n & 1, wc)) break;
        tc::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          tc::mma_ts(tmem + colDQ, tmem + colS + kk * 8, tc::desc_mnmajor(sK(st), kTile, kk), idAcc,
                     (n > 0 || kk > 0) ? 1u : 0u);
        tc::mma_commit(bar_mma_done);
        tc::mma_commit(bar_kv_empty(st));
      }
      tc::mma_commit(bar_fin);
      tc::mbar_wait(bar_fin, 0, drain);
    }
  } else if (warp < 4) {
    const int row = threadIdx.x;
    const int q_pos = q_pos0 + row;
    const bool valid = row < q_rows;
    const long long grow = (long long)bh * p.T + (long long)(2 * c * rq + hq * c + qt * kTile + row);
    const float lse2 = valid ? p.lse[grow] * kLog2e : INFINITY;
    const float Drow = valid ? p.D[grow] : 0.f;
    const uint32_t t_row = tmem + ((uint32_t)(warp * 32) << 16);
    const float sl2 = p.scale_log2;
    int dlo, dhi;   // this row's document [dlo, dhi) (everything without packed documents)
    doc_bounds_at(p.doc_lo, p.doc_hi, min(q_pos, p.T - 1), p.T, dlo, dhi);
    int n = 0;
    bool ok = true;
    while (sched.next(t)) {
      ok = __all_sync(0xffffffffu, tc::mbar_wait(bar_s_full, n & 1, wc));
      if (!ok) break;
      tc::tc_fence_after();
#pragma unroll 1
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t rs[32], rd[32];
        tc::tmem_ld32(t_row + colS + cb * 32, rs);
        tc::tmem_ld32(t_row + colDP + cb * 32, rd);
        tc::tmem_ld_wait();
        uint32_t dk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float dsv[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int j = cb * 32 + 2 * e + h;
            float pr = exp2f(fmaf(__uint_as_float(rs[2 * e + h]), sl2, -lse2));
            if (t.need_mask) {
              const int kp = t.pos0 + j;
              if (j >= t.nvalid || kp >= p.T_valid || (p.causal && kp > q_pos) || kp < dlo || kp >= dhi) pr = 0.f;
            }
            dsv[h] = pr * (__uint_as_float(rd[2 * e + h]) - Drow);
          }
          dk[e] = pack_bf16x2(dsv[0], dsv[1]);
        }
        tc::tmem_st16(t_row + colS + cb * 16, dk);
      }
      tc::tmem_st_wait();
      tc::tc_fence_before();
      tc::mbar_arrive(bar_p_full);
      ++n;
    }
    if (ok && n > 0) {
      ok = __all_sync(0xffffffffu, tc::mbar_wait(bar_mma_done, (n - 1) & 1, wc));
      if (ok) {
        tc::tc_fence_after();
        epilogue_row<D, ROPE>(t_row + colDQ, p.scale, q_pos, p.theta, p.out0 + grow * D, valid);
      }
    } else if (ok && valid) {   // no key tile at all (rows outside every document)
      store_zero_row<D>(p.out0 + grow * D);
    }
  } else if (ROPE) {
    const int wid = warp - 6;
    if (tc::mbar_wait(bar_q_full, 0, wc)) {
      tc::rope_tile<D>(smem + C::OFF_Q, q_pos0, wid, lane, p.theta);
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(bar_q_ready);
      int n = 0;
      while (sched.next(t)) {
        const int st = n % NS;
        if (!tc::mbar_wait(bar_kv_full(st), (n / NS) & 1, wc)) break;
        tc::rope_tile<D>(smem + C::OFF_K + st * C::TILE, t.pos0, wid, lane, p.theta);
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(bar_k_ready(st));
        ++n;
      }
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

template <int D, bool ROPE>
cpattn_status launch_bwd_t(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                           const CUtensorMap &mdo, BwdParams bp, __nv_bfloat16 *dq,
                           __nv_bfloat16 *dk, __nv_bfloat16 *dv, unsigned grid, cudaStream_t s) {
  const int threads = ROPE ? 320 : 192;
  {
    constexpr int smem = DkdvCfg<D>::SMEM;
    auto kern = dkdv_tc_kernel<D, ROPE>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return fail(CPATTN_ERR_CUDA, "cannot set %d bytes of shared memory for the dK/dV kernel", smem);
    bp.out0 = dk;
    bp.out1 = dv;
    trace_record(2, s);
    kern<<<grid / bp.group, threads, smem, s>>>(mq, mk, mv, mdo, bp);   // one CTA per K/V-head key tile
    cpattn_status st = check_launch("tensor-core dK/dV kernel");
    if (st != CPATTN_OK) return st;
    trace_record(3, s);
  }
  {
    constexpr int smem = DqCfg<D>::SMEM;
    auto kern = dq_tc_kernel<D, ROPE>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return fail(CPATTN_ERR_CUDA, "cannot set %d bytes of shared memory for the dQ kernel", smem);
    bp.out0 = dq;
    bp.out1 = nullptr;
    trace_record(4, s);
    kern<<<grid, threads, smem, s>>>(mq, mk, mv, mdo, bp);
    cpattn_status st = check_launch("tensor-core dQ kernel");
    trace_record(5, s);
    return st;
  }
}

}  // namespace

cpattn_status launch_bwd_bf16(const void *q, const void *k, const void *v, const void *o,
                              const float *lse, const void *dO, void *dq, void *dk, void *dv,
                              float *D, const Geometry &g, cudaStream_t s) {
  (void)o;
  // Pipelined kernels with a tile table in shared memory, where the schedule fits it.
  if (2LL * g.cp * ((g.c + kTile - 1) / kTile) <= kMaxTiles)
    return launch_bwd2_bf16(q, k, v, lse, dO, dq, dk, dv, D, g, s);
  const long long BH = (long long)g.B * g.H;
  const long long n_slots = BH * 2 * g.cp;
  const long long n_kv_slots = (long long)g.B * g.Hkv * 2 * g.cp;
  CUtensorMap mq, mk, mv, mdo;
  if (!make_tile_map(&mq, q, g.d, g.c, n_slots) || !make_tile_map(&mk, k, g.d, g.c, n_kv_slots) ||
      !make_tile_map(&mv, v, g.d, g.c, n_kv_slots) || !make_tile_map(&mdo, dO, g.d, g.c, n_slots))
    return fail(CPATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed (is the driver too old?)");
  BwdParams bp;
  bp.lse = lse;
  bp.D = D;
  bp.out0 = bp.out1 = nullptr;
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
  auto *pdq = static_cast<__nv_bfloat16 *>(dq);
  auto *pdk = static_cast<__nv_bfloat16 *>(dk);
  auto *pdv = static_cast<__nv_bfloat16 *>(dv);
  if (g.d == 128)
    return g.rope ? launch_bwd_t<128, true>(mq, mk, mv, mdo, bp, pdq, pdk, pdv, (unsigned)grid, s)
                  : launch_bwd_t<128, false>(mq, mk, mv, mdo, bp, pdq, pdk, pdv, (unsigned)grid, s);
  return g.rope ? launch_bwd_t<64, true>(mq, mk, mv, mdo, bp, pdq, pdk, pdv, (unsigned)grid, s)
                : launch_bwd_t<64, false>(mq, mk, mv, mdo, bp, pdq, pdk, pdv, (unsigned)grid, s);
}

}  // namespace cpattn
