// Ring attention forward on tcgen05 tensor cores (bf16 in, fp32 accumulate).
//
// One CTA owns one 128-row query tile of one (b,h): a tile of virtual rank r's
// head or tail chunk. It walks the K/V tiles the ring would bring to rank r,
// step by step (j = (r - s) mod cp, head then tail chunk), skipping tiles that
// lie wholly above the shifted causal diagonal (Claude Logs, 2026-04-20 and
// 2026-06-17). The online-softmax update at each tile boundary is the
// SDPAMerger rule applied to the running (O, m, l) and the new tile's
// partial, so at every ring-step boundary the running state equals the merge
// of the steps seen so far (Claude Logs, 2026-03-20).
//
// Warp roles (NT threads):
//   warps 0-3  softmax: thread i owns query row i = TMEM lane i. Reads S from
//              TMEM, masks, keeps (m, l), writes P (bf16) back into TMEM over
//              S, rescales O in TMEM when the row max grows by > 2^8, and
//              writes O and LSE at the end.
//   warp 4     TMA producer (lane 0) and TMEM allocator (whole warp).
//   warp 5     MMA issuer (lane 0): S = Q K^T (A, B from smem), O += P V
//              (A = P from TMEM, B = V from smem, MN-major).
//   warps 6-9  (RoPE only) rotate the Q tile once and every K tile in smem.
// TMEM columns: S/P buffer 0 at 0, buffer 1 at 128, O at 256 (512 allocated).
#include <math.h>

#include "attn_common.cuh"

namespace cpattn {
namespace {

struct FwdParams {
  __nv_bfloat16 *o;
  float *lse;
  int *err;
  int BH, T, T_valid, c, cp, causal, tpc;
  int group;   // query heads per K/V head
  const int *doc_lo, *doc_hi;   // packed documents: [T] bounds per natural position, or nullptr
  float scale_log2;  // log2(e) / sqrt(d)
  RopeTheta theta;
};

template <int D>
struct FwdCfg {
  static constexpr int NS = (D == 128) ? 2 : 4;    // K/V pipeline stages
  static constexpr int TILE = kTile * D * 2;       // bytes of one 128 x D bf16 tile
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + TILE;
  static constexpr int OFF_V = OFF_K + NS * TILE;
  static constexpr int OFF_BAR = OFF_V + NS * TILE;
  // barriers: q_full, q_ready, fin, o_done, s_full[2], p_full[2], kv_full[NS], k_ready[NS], kv_empty[NS]
  static constexpr int NBAR = 8 + 3 * NS;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;  // + alignment slack
};

constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256, kTmemCols = 512;

template <int D, bool ROPE>
__global__ void __launch_bounds__(ROPE ? 320 : 192, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ FwdParams p) {
  using C = FwdCfg<D>;
  constexpr int NS = C::NS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = tc::smem_u32(smem);
  const uint32_t sQ = sbase + C::OFF_Q;
  auto sK = [&](int st) { return sbase + C::OFF_K + st * C::TILE; };
  auto sV = [&](int st) { return sbase + C::OFF_V + st * C::TILE; };
  const uint32_t bar0 = sbase + C::OFF_BAR;
  const uint32_t bar_q_full = bar0, bar_q_ready = bar0 + 8, bar_fin = bar0 + 16, bar_o_done = bar0 + 24;
  auto bar_s_full = [&](int b) { return bar0 + 32 + 8 * b; };
  auto bar_p_full = [&](int b) { return bar0 + 48 + 8 * b; };
  auto bar_kv_full = [&](int st) { return bar0 + 64 + 8 * st; };
  auto bar_k_ready = [&](int st) { return bar0 + 64 + 8 * NS + 8 * st; };
  auto bar_kv_empty = [&](int st) { return bar0 + 64 + 16 * NS + 8 * st; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- which query tile: heaviest (latest natural position) first, heads interleaved
  const int cp = p.cp, c = p.c, tpc = p.tpc;
  const int bh = blockIdx.x % p.BH;
  const int bkv = bh / p.group;                   // K/V head of this query head
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
      bool by_threads = b == bar_q_ready || b == bar_p_full(0) || b == bar_p_full(1);
      for (int st = 0; st < NS; ++st) by_threads |= b == bar_k_ready(st);
      tc::mbar_init(b, by_threads ? 128 : 1);
    }
    abort_flag[0] = 0;
    abort_flag[1] = 0;   // never set: lets teardown waits honour only the time limit
    tc::mbar_fence_init();
  }
  if (warp == 4) {
    tc::tmem_alloc(tc::smem_u32(tmem_slot), kTmemCols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const tc::WaitCtx wc{abort_flag, p.err};

  KvSchedule sched;
  {
    const KvBounds kb = kv_bounds(p.doc_lo, p.doc_hi, p.T, p.T_valid, p.causal, q_pos0, q_pos0 + q_rows - 1);
    sched.init(cp, c, rq, p.causal, p.T_valid, q_pos0, q_pos0 + q_rows - 1, kb.key_lo, kb.key_hi,
               kb.doc_lo_max, kb.doc_hi_min);
  }
  TileInfo t;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tc::tma_prefetch_desc(&tm_q);
      tc::tma_prefetch_desc(&tm_k);
      tc::tma_prefetch_desc(&tm_v);
      tc::mbar_arrive_expect_tx(bar_q_full, C::TILE);
      for (int blk = 0; blk < D / 64; ++blk)
        tc::tma_load_3d(sQ + blk * kTile * 128, &tm_q, bar_q_full, blk * 64, qt * kTile, q_z);
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
      // Let every issued copy land before the CTA can exit.
      const tc::WaitCtx drain{abort_flag + 1, p.err};
      tc::mbar_wait(bar_q_full, 0, drain);
      for (int m = (n > NS ? n - NS : 0); m < n; ++m) tc::mbar_wait(bar_kv_full(m % NS), (m / NS) & 1, drain);
    }
  } else if (warp == 5) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = tc::idesc_bf16(128, 128, false, false);
      constexpr uint32_t idPV = tc::idesc_bf16(128, D, false, true);
      bool ok = tc::mbar_wait(ROPE ? bar_q_ready : bar_q_full, 0, wc);
      auto issue_s = [&](int n) -> bool {
        const int st = n % NS;
        if (!tc::mbar_wait(bar_kv_full(st), (n / NS) & 1, wc)) return false;
        if (ROPE && !tc::mbar_wait(bar_k_ready(st), (n / NS) & 1, wc)) return false;
        if (n >= 2 && !tc::mbar_wait(bar_o_done, (n - 2) & 1, wc)) return false;
        tc::tc_fence_after();
        const uint32_t dS = tmem + ((n & 1) ? kColS1 : kColS0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc::mma_ss(dS, tc::desc_kmajor(sQ, kTile, kk), tc::desc_kmajor(sK(st), kTile, kk), idS, kk > 0);
        tc::mma_commit(bar_s_full(n & 1));
        return true;
      };
      if (ok && sched.next(t)) {
        ok = issue_s(0);
        for (int n = 0; ok; ++n) {
          const bool more = sched.next(t);
          if (more && !issue_s(n + 1)) break;
          if (!tc::mbar_wait(bar_p_full(n & 1), (n >> 1) & 1, wc)) break;
          tc::tc_fence_after();
          const uint32_t aP = tmem + ((n & 1) ? kColS1 : kColS0);
          const int st = n % NS;
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            tc::mma_ts(tmem + kColO, aP + kk * 8, tc::desc_mnmajor(sV(st), kTile, kk), idPV,
                       (n > 0 || kk > 0) ? 1u : 0u);
          tc::mma_commit(bar_o_done);
          tc::mma_commit(bar_kv_empty(st));
          if (!more) break;
        }
      }
      // All issued MMAs complete before teardown.
      tc::mma_commit(bar_fin);
      const tc::WaitCtx drain{abort_flag + 1, p.err};
      tc::mbar_wait(bar_fin, 0, drain);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------- softmax
    const int row = threadIdx.x;
    const int q_pos = q_pos0 + row;
    const uint32_t t_row = tmem + ((uint32_t)(warp * 32) << 16);
    const float sl2 = p.scale_log2;
    int dlo, dhi;   // this row's document [dlo, dhi) (everything without packed documents)
    doc_bounds_at(p.doc_lo, p.doc_hi, min(q_pos, p.T - 1), p.T, dlo, dhi);
    float m_run = -INFINITY, l = 0.f;
    int n = 0;
    bool ok = true;
    while (sched.next(t)) {
      const int b = n & 1;
      ok = __all_sync(0xffffffffu, tc::mbar_wait(bar_s_full(b), (n >> 1) & 1, wc));
      if (!ok) break;
      tc::tc_fence_after();
      // Pass 1: masked row max over the tile (S read from TMEM in 32-column chunks).
      const uint32_t t_s = t_row + (b ? kColS1 : kColS0);
      float mt = -INFINITY;
#pragma unroll 1
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t r[32];
        tc::tmem_ld32(t_s + cb * 32, r);
        tc::tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float v = __uint_as_float(r[e]);
          if (t.need_mask) {
            const int j = cb * 32 + e, kp = t.pos0 + j;
            if (!((j < t.nvalid) && (kp < p.T_valid) && (!p.causal || kp <= q_pos) && kp >= dlo && kp < dhi))
              v = -INFINITY;
          }
          mt = fmaxf(mt, v);
        }
      }
      const float m_new = fmaxf(m_run, mt * sl2);
      bool need = m_new > m_run + 8.f;
      if (n == 0) {
        m_run = m_new;
        need = false;
      } else if (__any_sync(0xffffffffu, need)) {
        ok = __all_sync(0xffffffffu, tc::mbar_wait(bar_o_done, (n - 1) & 1, wc));
        if (!ok) break;
        tc::tc_fence_after();
        const float alpha = need ? exp2f(m_run - m_new) : 1.f;
#pragma unroll 1
        for (int cb = 0; cb < D / 32; ++cb) {
          uint32_t r[32];
          tc::tmem_ld32(t_row + kColO + cb * 32, r);
          tc::tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
          tc::tmem_st32(t_row + kColO + cb * 32, r);
        }
        tc::tmem_st_wait();
        if (need) {
          l *= alpha;
          m_run = m_new;
        }
      }
      const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
      // Pass 2: P = 2^(S*scale*log2e - m), rounded to bf16 and written over S.
#pragma unroll 1
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t r[32];
        tc::tmem_ld32(t_s + cb * 32, r);
        tc::tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float v0 = __uint_as_float(r[2 * e]), v1 = __uint_as_float(r[2 * e + 1]);
          if (t.need_mask) {
            const int j = cb * 32 + 2 * e, kp = t.pos0 + j;
            if (!((j < t.nvalid) && (kp < p.T_valid) && (!p.causal || kp <= q_pos) && kp >= dlo && kp < dhi))
              v0 = -INFINITY;
            if (!((j + 1 < t.nvalid) && (kp + 1 < p.T_valid) && (!p.causal || kp + 1 <= q_pos) && kp + 1 >= dlo &&
                  kp + 1 < dhi))
              v1 = -INFINITY;
          }
          pk[e] = pack_bf16x2(exp2f(fmaf(v0, sl2, -m_use)), exp2f(fmaf(v1, sl2, -m_use)));
          l += bf16lo_to_f32(pk[e]) + bf16hi_to_f32(pk[e]);
        }
        tc::tmem_st16(t_s + cb * 16, pk);
      }
      tc::tmem_st_wait();
      tc::tc_fence_before();
      tc::mbar_arrive(bar_p_full(b));
      ++n;
    }
    if (ok && n > 0) {
      ok = __all_sync(0xffffffffu, tc::mbar_wait(bar_o_done, (n - 1) & 1, wc));
      if (ok) {
        tc::tc_fence_after();
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        const bool valid = row < q_rows;
        const long long grow = (long long)bh * p.T + (long long)(2 * c * rq + hq * c + qt * kTile + row);
        uint4 *dst = reinterpret_cast<uint4 *>(p.o + grow * D);
#pragma unroll 1
        for (int cb = 0; cb < D / 32; ++cb) {
          uint32_t r[32];
          tc::tmem_ld32(t_row + kColO + cb * 32, r);
          tc::tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(r[2 * e]) * inv_l, __uint_as_float(r[2 * e + 1]) * inv_l);
          if (valid) {
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
              dst[cb * 4 + v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
          }
        }
        if (valid) p.lse[grow] = l > 0.f ? (m_run + log2f(l)) * 0.693147180559945309f : -INFINITY;
      }
    } else if (ok && row < q_rows) {   // no key tile at all (rows outside every document)
      const long long grow = (long long)bh * p.T + (long long)(2 * c * rq + hq * c + qt * kTile + row);
      uint4 *dst = reinterpret_cast<uint4 *>(p.o + grow * D);
#pragma unroll 1
      for (int v4 = 0; v4 < D / 8; ++v4) dst[v4] = make_uint4(0u, 0u, 0u, 0u);
      p.lse[grow] = -INFINITY;
    }
  } else if (ROPE) {
    // ------------------------------------------------ RoPE transform warps
    const int wid = warp - 6;
    bool ok = tc::mbar_wait(bar_q_full, 0, wc);
    if (ok) {
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
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Paired-tile forward (inputs already rotated, or no RoPE). One CTA owns two
// consecutive 128-row query tiles Q0, Q1 of one chunk and streams each K/V
// tile once for both. Two softmax warpgroups (warps 0-3 for Q0, 4-7 for Q1)
// alternate with the MMA issuer so that while one warpgroup turns S_i into
// P_i, the tensor core works on the other tile:
//   S0(n) S1(n) | PV0(n) S0(n+1) | PV1(n) S1(n+1) | PV0(n+1) ...
// TMEM columns: S0/P0 0, S1/P1 128, O0 256, O1 256 + D (512 allocated).
// Warp 8: TMA producer (lane 0) and TMEM allocator; warp 9: MMA issuer.
// With in-kernel RoPE (ROPE), warps 10-11 rotate Q0, Q1 once and every K
// tile in shared memory between its TMA landing and its first MMA (q_ready,
// k_ready); the issuer waits for those instead of the TMA barriers.
// SAVE (with ROPE) also stores the rotated tiles for the backward: Q0, Q1 to
// q_rot, and the CTA's two diagonal K tiles (the key rows at the positions of
// its own query rows, which every query tile reads) to k_rot -- by the first
// query head of each K/V-head group only -- so that every rotated row is
// written once. A K stage with a store in flight is released by the rotation
// warp once the store has read it (k_empty then counts two arrivals).
template <int D>
struct Fwd2Cfg {
  static constexpr int NS = (D == 128) ? 2 : 4;   // stages of the K ring and of the V ring
  static constexpr int TILE = kTile * D * 2;
  static constexpr int OFF_Q = 0;                 // Q0, Q1
  static constexpr int OFF_K = 2 * TILE;
  static constexpr int OFF_V = OFF_K + NS * TILE;
  static constexpr int OFF_BAR = OFF_V + NS * TILE;
  // q_full, fin, s_full[2], p_full[2], o_done[2], k_full[NS], k_empty[NS], v_full[NS], v_empty[NS],
  // q_ready, k_ready[NS]
  static constexpr int NBAR = 9 + 5 * NS;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 32 + kMaxTiles * 8 + 1024;   // misc, tile table, alignment slack
  static_assert(SMEM <= 232448, "over the 227 KiB of shared memory a CTA may opt into");
};

// Heads per launch-order group of the paired-tile forward.
constexpr int kFwdHeadGroup = 4;

template <int D, bool ROPE, bool SAVE = false>
__global__ void __launch_bounds__(ROPE ? 384 : 320, 1)
    fwd2_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ FwdParams p,
                   const __grid_constant__ CUtensorMap tm_qrot, const __grid_constant__ CUtensorMap tm_krot) {
  static_assert(!SAVE || ROPE, "saving rotated tiles needs the in-kernel rotation");
  using C = Fwd2Cfg<D>;
  constexpr int NS = C::NS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = tc::smem_u32(smem);
  auto sQ = [&](int i) { return sbase + C::OFF_Q + i * C::TILE; };
  auto sK = [&](int st) { return sbase + C::OFF_K + st * C::TILE; };
  auto sV = [&](int st) { return sbase + C::OFF_V + st * C::TILE; };
  const uint32_t bar0 = sbase + C::OFF_BAR;
  const uint32_t bar_q_full = bar0, bar_fin = bar0 + 8;
  auto bar_s_full = [&](int i) { return bar0 + 16 + 8 * i; };
  auto bar_p_full = [&](int i) { return bar0 + 32 + 8 * i; };
  auto bar_o_done = [&](int i) { return bar0 + 48 + 8 * i; };
  auto bar_k_full = [&](int st) { return bar0 + 64 + 8 * st; };
  auto bar_k_empty = [&](int st) { return bar0 + 64 + 8 * NS + 8 * st; };
  auto bar_v_full = [&](int st) { return bar0 + 64 + 16 * NS + 8 * st; };
  auto bar_v_empty = [&](int st) { return bar0 + 64 + 24 * NS + 8 * st; };
  const uint32_t bar_q_ready = bar0 + 64 + 32 * NS;
  auto bar_k_ready = [&](int st) { return bar0 + 72 + 32 * NS + 8 * st; };
  // the barriers the MMA issuer waits on before reading Q and K
  const uint32_t bar_q_use = ROPE ? bar_q_ready : bar_q_full;
  auto bar_k_use = [&](int st) { return ROPE ? bar_k_ready(st) : bar_k_full(st); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
  int *ntiles_slot = reinterpret_cast<int *>(smem + C::OFF_MISC + 12);
  // first output row of the CTA (kept in shared memory: the epilogue reloads it)
  volatile long long *row_base = reinterpret_cast<volatile long long *>(smem + C::OFF_MISC + 16);
  TileEntry *tab = reinterpret_cast<TileEntry *>(smem + C::OFF_MISC + 32);
  constexpr uint32_t colO0 = 256;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cp = p.cp, c = p.c, tpc = p.tpc;
  const int ppc = (tpc + 1) / 2;                  // tile pairs per chunk
  // A few heads at a time (their K/V tiles stay in L2), heaviest CTAs first.
  int bh, g;
  head_group_order<kFwdHeadGroup>((int)blockIdx.x, 2 * cp * ppc, (int)gridDim.x / (2 * cp * ppc), bh, g);
  const int bkv = bh / p.group;                   // K/V head of this query head
  const int kq = 2 * cp - 1 - g / ppc;            // latest chunks first: they carry the most work
  const int pq = ppc - 1 - g % ppc;
  int rq, hq;
  owner_of(kq, cp, rq, hq);
  const int q_z = bh * 2 * cp + 2 * rq + hq;
  const int y0 = pq * 2 * kTile;                  // first row of Q0 inside the chunk
  const int q_pos0 = kq * c + y0;
  const int q_rows = min(2 * kTile, c - y0);      // valid rows of the pair

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NBAR; ++i) {
      const uint32_t b = bar0 + 8 * i;
      uint32_t cnt = (b == bar_p_full(0) || b == bar_p_full(1)) ? 128 : 1;
      if (b >= bar_q_ready) cnt = 64;   // q_ready, k_ready[]: the two rotation warps
      if (SAVE)
        for (int st = 0; st < NS; ++st)
          if (b == bar_k_empty(st)) cnt = 2;   // the issuer's commit and the rotation warp's release
      tc::mbar_init(b, cnt);
    }
    abort_flag[0] = 0;
    abort_flag[1] = 0;
    *row_base = (long long)bh * p.T + (long long)(2 * c * rq + hq * c + y0);
    tc::mbar_fence_init();
    tc::fence_proxy_async_smem();
    // the stationary Q tiles load while the tile table is built
    tc::mbar_arrive_expect_tx(bar_q_full, 2 * C::TILE);
    for (int i = 0; i < 2; ++i)
      for (int blk = 0; blk < D / 64; ++blk)
        tc::tma_load_3d(sQ(i) + blk * kTile * 128, &tm_q, bar_q_full, blk * 64, y0 + i * kTile, q_z);
  }
  if (warp == 8) {
    tc::tmem_alloc(tc::smem_u32(tmem_slot), kTmemCols);
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
        const int z = bkv * 2 * cp + t.slot;
        if (n >= NS && !tc::mbar_wait(bar_k_empty(st), ((n / NS) - 1) & 1, wc)) break;
        tc::mbar_arrive_expect_tx(bar_k_full(st), C::TILE);
        for (int blk = 0; blk < D / 64; ++blk)
          tc::tma_load_3d(sK(st) + blk * kTile * 128, &tm_k, bar_k_full(st), blk * 64, t.y0, z);
        if (n >= NS && !tc::mbar_wait(bar_v_empty(st), ((n / NS) - 1) & 1, wc)) break;
        tc::mbar_arrive_expect_tx(bar_v_full(st), C::TILE);
        for (int blk = 0; blk < D / 64; ++blk)
          tc::tma_load_3d(sV(st) + blk * kTile * 128, &tm_v, bar_v_full(st), blk * 64, t.y0, z);
        ++n;
      }
      tc::mbar_wait(bar_q_full, 0, drain);
      for (int m = (n > NS ? n - NS : 0); m < n; ++m) {
        tc::mbar_wait(bar_k_full(m % NS), (m / NS) & 1, drain);
        tc::mbar_wait(bar_v_full(m % NS), (m / NS) & 1, drain);
      }
    }
  } else if (warp == 9) {
    {   // the whole warp runs the issue loop; elect.sync picks the issuing lane
      constexpr uint32_t idS = tc::idesc_bf16(128, 128, false, false);
      constexpr uint32_t idPV = tc::idesc_bf16(128, D, false, true);
      const uint64_t dq0[2] = {tc::kdesc0(sQ(0)), tc::kdesc0(sQ(1))};
      auto issue_s = [&](int i, int st) {
        const uint64_t a0 = dq0[i], b0 = tc::kdesc0(sK(st));
        const uint32_t d = tmem + i * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc::mma_ss_w(d, a0 + tc::koff(kTile, kk), b0 + tc::koff(kTile, kk), idS, kk > 0 ? 1u : 0u);
        tc::mma_commit_w(bar_s_full(i));
      };
      auto issue_pv = [&](int i, int st, int n) {
        const uint64_t b0 = tc::mndesc0(sV(st), kTile);
        const uint32_t d = tmem + colO0 + i * D, a = tmem + i * 128;
        const uint32_t acc0 = n > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          tc::mma_ts_w(d, a + kk * 8, b0 + tc::mnoff(kk), idPV, kk > 0 ? 1u : acc0);
        tc::mma_commit_w(bar_o_done(i));
      };
      auto wait_all = [&](uint32_t bar, uint32_t par, const tc::WaitCtx &w) {
        return __all_sync(0xffffffffu, tc::mbar_wait(bar, par, w));
      };
      bool ok = wait_all(bar_q_use, 0, wc);
      if (ok && ntiles > 0) {
        ok = wait_all(bar_k_use(0), 0, wc);
        if (ok) {
          tc::tc_fence_after();
          issue_s(0, 0);
          issue_s(1, 0);
          tc::mma_commit_w(bar_k_empty(0));
        }
        for (int n = 0; ok; ++n) {
          const bool more = n + 1 < ntiles;
          const int st = n % NS, st1 = (n + 1) % NS;
          // ---- tile 0: PV0(n), then S0(n+1) once PV0(n) has read P0
          if (!(ok = wait_all(bar_p_full(0), n & 1, wc))) break;
          if (!(ok = wait_all(bar_v_full(st), (n / NS) & 1, wc))) break;
          tc::tc_fence_after();
          issue_pv(0, st, n);
          if (more) {
            if (!(ok = wait_all(bar_k_use(st1), ((n + 1) / NS) & 1, wc))) break;
            if (!(ok = wait_all(bar_o_done(0), n & 1, wc))) break;
            tc::tc_fence_after();
            issue_s(0, st1);
          }
          // ---- tile 1: PV1(n), then S1(n+1)
          if (!(ok = wait_all(bar_p_full(1), n & 1, wc))) break;
          tc::tc_fence_after();
          issue_pv(1, st, n);
          tc::mma_commit_w(bar_v_empty(st));
          if (more) {
            if (!(ok = wait_all(bar_o_done(1), n & 1, wc))) break;
            tc::tc_fence_after();
            issue_s(1, st1);
            tc::mma_commit_w(bar_k_empty(st1));
          }
          if (!more) break;
        }
      }
      tc::mma_commit_w(bar_fin);
      wait_all(bar_fin, 0, drain);
    }
  } else if (ROPE && warp >= 10) {
    // ------------------------------------------------ RoPE rotation warps
    tc::RopeRows<D, 64> rr;   // warps 10-11
    rr.init((warp - 10) * 32 + lane, p.theta);
    const bool storer = SAVE && warp == 10 && lane == 0;
    const int own_slot = 2 * rq + hq;
    const bool kv_writer = (bh % p.group) == 0;     // first query head of its K/V group
    if (__all_sync(0xffffffffu, tc::mbar_wait(bar_q_full, 0, wc))) {
      rr.rotate(smem + C::OFF_Q, q_pos0);
      rr.rotate(smem + C::OFF_Q + C::TILE, q_pos0 + kTile);
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(bar_q_ready);
      if (storer && tc::mbar_wait(bar_q_ready, 0, wc)) {   // both rotation warps are done with Q
        for (int i = 0; i < 2 && y0 + i * kTile < c; ++i)
          for (int blk = 0; blk < D / 64; ++blk)
            tc::tma_store_3d(&tm_qrot, sQ(i) + blk * kTile * 128, blk * 64, y0 + i * kTile, q_z);
        tc::tma_store_commit();
      }
      for (int n = 0; n < ntiles; ++n) {
        decode_tile(tab[n], t);
        const int st = n % NS;
        if (!__all_sync(0xffffffffu, tc::mbar_wait(bar_k_full(st), (n / NS) & 1, wc))) break;
        rr.rotate(smem + C::OFF_K + st * C::TILE, t.pos0);
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(bar_k_ready(st));
        if (storer) {
          const bool diag = kv_writer && t.slot == own_slot && (t.y0 == y0 || t.y0 == y0 + kTile);
          if (diag && tc::mbar_wait(bar_k_ready(st), (n / NS) & 1, wc)) {
            for (int blk = 0; blk < D / 64; ++blk)
              tc::tma_store_3d(&tm_krot, sK(st) + blk * kTile * 128, blk * 64, t.y0, bkv * 2 * cp + t.slot);
            tc::tma_store_commit();
            tc::tma_store_wait_read();                      // the stage may be refilled after this
          }
          tc::mbar_arrive(bar_k_empty(st));
        }
      }
    }
    if (storer) tc::tma_store_wait_all();
  } else {
    // ----------------------------------------------- softmax warpgroups 0, 1
    const int wg = warp >> 2;
    const int row = threadIdx.x & 127;
    const int prow = wg * kTile + row;          // row within the pair
    const int q_pos = q_pos0 + prow;
    const uint32_t t_row = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t t_s = t_row + wg * 128;
    const uint32_t t_o = t_row + colO0 + wg * D;
    const float sl2 = p.scale_log2;
    int dlo, dhi;   // this row's document [dlo, dhi) (everything without packed documents)
    doc_bounds_at(p.doc_lo, p.doc_hi, min(q_pos, p.T - 1), p.T, dlo, dhi);
    float m_run = -INFINITY, l = 0.f;
    int n = 0;
    bool ok = true;
    while (n < ntiles && (decode_tile(tab[n], t), true)) {
      ok = __all_sync(0xffffffffu, tc::mbar_wait(bar_s_full(wg), n & 1, wc));
      if (!ok) break;
      tc::tc_fence_after();
      // The masks of a row keep one interval of key columns j of the tile:
      // j < nvalid (ragged tile), pos0 + j < T_valid (padding), pos0 + j <=
      // q_pos (causal) and dlo <= pos0 + j < dhi (packed documents). Keep
      // lo <= j < lim, tested as one unsigned compare of j - lo with width.
      int lim = kTile, lo = 0;
      if (t.need_mask) {
        lim = min(min(t.nvalid, p.T_valid - t.pos0), dhi - t.pos0);
        if (p.causal) lim = min(lim, q_pos - t.pos0 + 1);
        lo = dlo - t.pos0;
      }
      const bool masked = __any_sync(0xffffffffu, lim < kTile || lo > 0);
      const unsigned width = (unsigned)max(lim - lo, 0);
      // The whole row of S comes out of TMEM in one batch of four loads and
      // one wait; the exponentials then run from registers. On a tile without
      // masks the loads also return the row max of their 32 columns
      // (tcgen05.ld.red); a masked tile takes the max over its kept columns.
      uint32_t r[4][32];
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (masked) {
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) tc::tmem_ld32(t_s + cb * 32, r[cb]);
      } else {
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) tc::tmem_ld32_max(t_s + cb * 32, r[cb], mx[cb]);
      }
      tc::tmem_ld_wait();
      if (masked) {
#pragma unroll
        for (int cb = 0; cb < 4; ++cb)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if ((unsigned)(cb * 32 + e - lo) >= width) r[cb][e] = 0xff800000u;   // -inf
        // row max over the kept columns (three-input max)
#pragma unroll
        for (int cb = 0; cb < 4; ++cb)
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            mx[0] = tc::fmax3(mx[0], __uint_as_float(r[cb][e]), __uint_as_float(r[cb][e + 1]));
            mx[1] = tc::fmax3(mx[1], __uint_as_float(r[cb][e + 2]), __uint_as_float(r[cb][e + 3]));
            mx[2] = tc::fmax3(mx[2], __uint_as_float(r[cb][e + 4]), __uint_as_float(r[cb][e + 5]));
            mx[3] = tc::fmax3(mx[3], __uint_as_float(r[cb][e + 6]), __uint_as_float(r[cb][e + 7]));
          }
      }
      const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      const float m_new = fmaxf(m_run, mt * sl2);
      // The running max moves only when it grows by more than 2^8 (the stale
      // max keeps every P <= 2^8, and l uses the same max, so this is exact).
      bool need = m_new > m_run + 8.f;
      float alpha = 1.f;
      if (n == 0) {
        m_run = m_new;
        need = false;
      } else if (need) {
        alpha = tc::ex2(m_run - m_new);
        l *= alpha;
        m_run = m_new;
      }
      const bool rescale = n > 0 && __any_sync(0xffffffffu, need);
      const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
      // P = 2^(S*scale*log2e - m), rounded to bf16 and written over S; the
      // argument and the row sum use packed fp32 pairs.
      const uint64_t sl2x2 = tc::f2(sl2, sl2), negm2 = tc::f2(-m_use, -m_use);
      uint64_t ls2[2] = {tc::f2(0.f, 0.f), tc::f2(0.f, 0.f)};
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float x0, x1;
          tc::unf2(tc::ffma2(tc::f2(__uint_as_float(r[cb][2 * e]), __uint_as_float(r[cb][2 * e + 1])), sl2x2, negm2),
                   x0, x1);
          const uint64_t p01 = tc::f2(tc::ex2(x0), tc::ex2(x1));
          ls2[e & 1] = tc::fadd2(ls2[e & 1], p01);
          pk[e] = tc::pack_bf16x2_2(p01);
        }
        tc::tmem_st16(t_s + cb * 16, pk);
      }
      float ls[4];
      tc::unf2(ls2[0], ls[0], ls[1]);
      tc::unf2(ls2[1], ls[2], ls[3]);
      l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      // O *= alpha once PV(n-1) has landed, before PV(n) is issued
      if (rescale) {
        ok = __all_sync(0xffffffffu, tc::mbar_wait(bar_o_done(wg), (n - 1) & 1, wc));
        if (!ok) break;
        tc::tc_fence_after();
        uint32_t ro[D / 32][32];
#pragma unroll
        for (int cb = 0; cb < D / 32; ++cb) tc::tmem_ld32(t_o + cb * 32, ro[cb]);
        tc::tmem_ld_wait();
#pragma unroll
        for (int cb = 0; cb < D / 32; ++cb) {
#pragma unroll
          for (int e = 0; e < 32; ++e) ro[cb][e] = __float_as_uint(__uint_as_float(ro[cb][e]) * alpha);
          tc::tmem_st32(t_o + cb * 32, ro[cb]);
        }
      }
      tc::tmem_st_wait();
      tc::tc_fence_before();
      tc::mbar_arrive(bar_p_full(wg));
      ++n;
    }
    if (ok && n > 0) {
      ok = __all_sync(0xffffffffu, tc::mbar_wait(bar_o_done(wg), (n - 1) & 1, wc));
      if (ok) {
        tc::tc_fence_after();
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        const bool valid = prow < q_rows;
        const long long grow = *row_base + prow;
        uint4 *dst = reinterpret_cast<uint4 *>(p.o + grow * D);
#pragma unroll 1
        for (int cb = 0; cb < D / 32; ++cb) {
          uint32_t r[32];
          tc::tmem_ld32(t_o + cb * 32, r);
          tc::tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(r[2 * e]) * inv_l, __uint_as_float(r[2 * e + 1]) * inv_l);
          if (valid) {
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
              dst[cb * 4 + v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
          }
        }
        if (valid) p.lse[grow] = l > 0.f ? (m_run + log2f(l)) * 0.693147180559945309f : -INFINITY;
      }
    } else if (ok && prow < q_rows) {   // no key tile at all (rows outside every document)
      const long long grow = *row_base + prow;
      uint4 *dst = reinterpret_cast<uint4 *>(p.o + grow * D);
#pragma unroll 1
      for (int v4 = 0; v4 < D / 8; ++v4) dst[v4] = make_uint4(0u, 0u, 0u, 0u);
      p.lse[grow] = -INFINITY;
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool make_tile_map(CUtensorMap *m, const void *base, int D, int c, long long n_slots, int box_rows) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)c, (cuuint64_t)n_slots};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)c * D * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

template <int D, bool ROPE, bool SAVE = false>
cpattn_status launch_fwd2_t(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                            const FwdParams &fp, unsigned grid, cudaStream_t s,
                            const CUtensorMap *mqr = nullptr, const CUtensorMap *mkr = nullptr) {
  constexpr int smem = Fwd2Cfg<D>::SMEM;
  auto kern = fwd2_tc_kernel<D, ROPE, SAVE>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return fail(CPATTN_ERR_CUDA, "cannot set %d bytes of shared memory for the forward kernel", smem);
  kern<<<grid, ROPE ? 384 : 320, smem, s>>>(mq, mk, mv, fp, SAVE ? *mqr : mq, SAVE ? *mkr : mk);
  return check_launch("tensor-core forward kernel (paired tiles)");
}

template <int D, bool ROPE>
cpattn_status launch_fwd_t(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                           const FwdParams &fp, unsigned grid, cudaStream_t s) {
  constexpr int smem = FwdCfg<D>::SMEM;
  auto kern = fwd_tc_kernel<D, ROPE>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return fail(CPATTN_ERR_CUDA, "cannot set %d bytes of shared memory for the forward kernel", smem);
  kern<<<grid, ROPE ? 320 : 192, smem, s>>>(mq, mk, mv, fp);
  return check_launch("tensor-core forward kernel");
}

}  // namespace

cpattn_status launch_fwd_bf16(const void *q, const void *k, const void *v, void *o, float *lse,
                              const Geometry &g, cudaStream_t s) {
  const long long BH = (long long)g.B * g.H;
  const long long n_slots = BH * 2 * g.cp;
  const long long n_kv_slots = (long long)g.B * g.Hkv * 2 * g.cp;
  CUtensorMap mq, mk, mv;
  if (!make_tile_map(&mq, q, g.d, g.c, n_slots) || !make_tile_map(&mk, k, g.d, g.c, n_kv_slots) ||
      !make_tile_map(&mv, v, g.d, g.c, n_kv_slots))
    return fail(CPATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed (is the driver too old?)");
  FwdParams fp;
  fp.o = static_cast<__nv_bfloat16 *>(o);
  fp.lse = lse;
  fp.err = device_err_flag();
  fp.BH = (int)BH;
  fp.group = g.H / g.Hkv;
  fp.doc_lo = g.doc_lo;
  fp.doc_hi = g.doc_hi;
  fp.T = g.T;
  fp.T_valid = g.T_valid;
  fp.c = g.c;
  fp.cp = g.cp;
  fp.causal = g.causal;
  fp.tpc = (g.c + kTile - 1) / kTile;
  fp.scale_log2 = (float)(1.4426950408889634 / sqrt((double)g.d));
  make_rope_theta(g.d, &fp.theta, g.rope_cfg);
  // Paired query tiles with a tile table in shared memory (RoPE, if asked
  // for, rotates the tiles in shared memory). Longer schedules take the
  // one-tile kernel below.
  if (2LL * g.cp * fp.tpc <= kMaxTiles) {
    const long long grid2 = BH * 2 * g.cp * ((fp.tpc + 1) / 2);
    if (grid2 > 0x7fffffffLL) return fail(CPATTN_ERR_SHAPE, "too many query tiles");
    if (g.q_rot) {   // in-kernel RoPE that also stores the rotated q, k
      CUtensorMap mqr, mkr;
      if (!g.rope || !make_tile_map(&mqr, g.q_rot, g.d, g.c, n_slots) ||
          !make_tile_map(&mkr, g.k_rot, g.d, g.c, n_kv_slots))
        return fail(CPATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed for the rotated copies");
      return g.d == 128 ? launch_fwd2_t<128, true, true>(mq, mk, mv, fp, (unsigned)grid2, s, &mqr, &mkr)
                        : launch_fwd2_t<64, true, true>(mq, mk, mv, fp, (unsigned)grid2, s, &mqr, &mkr);
    }
    if (g.d == 128)
      return g.rope ? launch_fwd2_t<128, true>(mq, mk, mv, fp, (unsigned)grid2, s)
                    : launch_fwd2_t<128, false>(mq, mk, mv, fp, (unsigned)grid2, s);
    return g.rope ? launch_fwd2_t<64, true>(mq, mk, mv, fp, (unsigned)grid2, s)
                  : launch_fwd2_t<64, false>(mq, mk, mv, fp, (unsigned)grid2, s);
  }
  const long long grid = BH * 2 * g.cp * fp.tpc;
  if (grid > 0x7fffffffLL) return fail(CPATTN_ERR_SHAPE, "too many query tiles");
  if (g.d == 128)
    return g.rope ? launch_fwd_t<128, true>(mq, mk, mv, fp, (unsigned)grid, s)
                  : launch_fwd_t<128, false>(mq, mk, mv, fp, (unsigned)grid, s);
  return g.rope ? launch_fwd_t<64, true>(mq, mk, mv, fp, (unsigned)grid, s)
                : launch_fwd_t<64, false>(mq, mk, mv, fp, (unsigned)grid, s);
}

}  // namespace cpattn
