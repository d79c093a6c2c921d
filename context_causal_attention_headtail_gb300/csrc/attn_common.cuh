// Tile schedule shared by the tensor-core attention kernels: which K/V (or
// Q/dO) tiles a stationary tile meets, in ring order, and which of them need
// an element mask. Tiles never straddle a HeadTail chunk; a chunk of c rows
// has ceil(c/128) tiles and its last one may be ragged.
#pragma once

#include "tc_common.cuh"

namespace cpattn {

constexpr int kTile = 128;

struct TileInfo {
  int slot;       // 2*rank + half: chunk slot within one (b,h) of the sharded tensor
  int y0;         // first row of the tile inside its chunk
  int pos0;       // natural position of that row
  int nvalid;     // rows of the tile inside the chunk (<= 128)
  int need_mask;  // some (query, key) pair of this tile is masked
};

// Enumerates, for a query tile of rank r with natural positions
// [qmin, qmax], the K/V tiles it attends to, in ring order: step s visits
// rank j = (r - s) mod cp (Claude Logs, 2026-03-20 ring; 2026-06-17 shapes),
// its head chunk then its tail chunk. Tiles wholly above the causal diagonal
// or wholly at positions >= T_valid are skipped, and with packed documents
// those wholly outside the keys [key_lo, key_hi] the tile's queries may see;
// a tile reaching before doc_lo_max or past doc_hi_min needs the element mask.
struct KvSchedule {
  int cp, c, tpc, r, causal, T_valid, qmin, qmax;
  int key_lo, key_hi, doc_lo_max, doc_hi_min;
  int s, half, kt;

  __device__ __forceinline__ void init(int cp_, int c_, int r_, int causal_, int T_valid_,
                                       int qmin_, int qmax_, int key_lo_ = 0, int key_hi_ = 0x7fffffff,
                                       int doc_lo_max_ = 0, int doc_hi_min_ = 0x7fffffff) {
    cp = cp_; c = c_; tpc = (c_ + kTile - 1) / kTile; r = r_; causal = causal_;
    T_valid = T_valid_; qmin = qmin_; qmax = qmax_;
    key_lo = key_lo_; key_hi = key_hi_; doc_lo_max = doc_lo_max_; doc_hi_min = doc_hi_min_;
    s = 0; half = 0; kt = -1;
  }
  __device__ __forceinline__ bool next(TileInfo &t) {
    while (true) {
      if (++kt >= tpc) {
        kt = 0;
        if (++half >= 2) { half = 0; ++s; }
      }
      if (s >= cp) return false;
      const int j = (r - s + cp) % cp;
      const int pos0 = chunk_of(j, half, cp) * c + kt * kTile;
      if (pos0 >= T_valid) continue;
      if (causal && pos0 > qmax) continue;
      const int nv = min(kTile, c - kt * kTile);
      if (pos0 > key_hi || pos0 + nv - 1 < key_lo) continue;
      t.slot = 2 * j + half;
      t.y0 = kt * kTile;
      t.pos0 = pos0;
      t.nvalid = nv;
      t.need_mask = (nv < kTile) || (pos0 + nv > T_valid) || (causal && pos0 + nv - 1 > qmin) ||
                    (pos0 < doc_lo_max) || (pos0 + nv > doc_hi_min);
      return true;
    }
  }
};

// The transpose view for key-stationary kernels: for a key tile of rank j
// with natural positions [kmin, kmax], the query tiles that see it, in ring
// order: at step s the K/V of rank j sit on rank (j + s) mod cp (Claude
// Logs, 2026-06-22: the dK/dV accumulator travels with K/V around the ring).
struct QSchedule {
  int cp, c, tpc, j, causal, kmin, kmax, kvalid_max;
  int q_lo, q_hi, doc_lo_max, doc_hi_min;
  int s, half, qt;

  __device__ __forceinline__ void init(int cp_, int c_, int j_, int causal_, int T_valid_,
                                       int kmin_, int kmax_, int q_lo_ = -0x7fffffff, int q_hi_ = 0x7fffffff,
                                       int doc_lo_max_ = 0, int doc_hi_min_ = 0x7fffffff) {
    cp = cp_; c = c_; tpc = (c_ + kTile - 1) / kTile; j = j_; causal = causal_;
    kmin = kmin_; kmax = kmax_;
    kvalid_max = T_valid_;
    q_lo = q_lo_; q_hi = q_hi_; doc_lo_max = doc_lo_max_; doc_hi_min = doc_hi_min_;
    s = 0; half = 0; qt = -1;
  }
  // need_mask is set when any pair of the tile may be masked: causal
  // overlap, a ragged query or key tile, keys at positions >= T_valid, or
  // (packed documents) queries outside the document of some key. Query tiles
  // wholly outside [q_lo, q_hi] see none of the keys and are skipped.
  __device__ __forceinline__ bool next(TileInfo &t, int k_ragged) {
    while (true) {
      if (++qt >= tpc) {
        qt = 0;
        if (++half >= 2) { half = 0; ++s; }
      }
      if (s >= cp) return false;
      const int r = (j + s) % cp;
      const int pos0 = chunk_of(r, half, cp) * c + qt * kTile;
      const int nv = min(kTile, c - qt * kTile);
      if (causal && pos0 + nv - 1 < kmin) continue;   // every query before every key
      if (kmin >= kvalid_max) continue;               // keys all padding
      if (pos0 > q_hi || pos0 + nv - 1 < q_lo) continue;
      t.slot = 2 * r + half;
      t.y0 = qt * kTile;
      t.pos0 = pos0;
      t.nvalid = nv;
      t.need_mask = (nv < kTile) || k_ragged || (kmax >= kvalid_max) || (causal && kmax > pos0) ||
                    (pos0 < doc_lo_max) || (pos0 + nv > doc_hi_min);
      return true;
    }
  }
};

// With grouped K/V heads a key tile is seen by the query tiles of every query
// head of its group: QSchedule's list for each of them, head by head; gi is
// the current head's index inside the group.
struct GroupQSchedule {
  QSchedule q;
  int group, gi;

  __device__ __forceinline__ void init(int group_, int cp_, int c_, int j_, int causal_, int T_valid_,
                                       int kmin_, int kmax_, int q_lo_ = -0x7fffffff, int q_hi_ = 0x7fffffff,
                                       int doc_lo_max_ = 0, int doc_hi_min_ = 0x7fffffff) {
    group = group_;
    gi = 0;
    q.init(cp_, c_, j_, causal_, T_valid_, kmin_, kmax_, q_lo_, q_hi_, doc_lo_max_, doc_hi_min_);
  }
  __device__ __forceinline__ bool next(TileInfo &t, int k_ragged) {
    while (!q.next(t, k_ragged)) {
      if (++gi >= group) return false;
      q.s = 0; q.half = 0; q.qt = -1;
    }
    return true;
  }
};

// ---------------------------------------------------------------------------
// Precomputed schedules. The pipelined kernels build their whole tile list
// once per CTA in shared memory (one warp, lanes in parallel), so the MMA
// issuer and the softmax threads read one 8-byte entry per tile instead of
// re-deriving the ring order. The list is identical to what KvSchedule /
// QSchedule enumerate: groups (step s, half) in ring order, and inside a
// group the live tiles form one contiguous range, found in closed form.
// A kernel that uses a table runs only when 2*cp*tiles_per_chunk <= kMaxTiles,
// so the tile index in its chunk fits in 10 bits (tiles_per_chunk <= 1024)
// and the slot 2r + half in 11 bits (2*cp <= 2048).
constexpr int kMaxTiles = kTableTiles;   // entries per CTA (16 KiB of shared memory)

// Launch order of the pipelined kernels: `heads` heads of `per_head` CTAs
// each (per head, heaviest first), taken in groups of G heads whose CTAs
// interleave (CTA 0 of every head of the group, then CTA 1, ...). Only a
// group's operands are live in L2 at a time, and within a group the heaviest
// CTAs of all its heads start first, so a launch ends on light CTAs instead of
// on the heavy start of its last head. G = 1: heads one after the other.
template <int G>
__device__ __forceinline__ void head_group_order(int idx, int per_head, int heads, int &head, int &unit) {
  const int h0 = idx / (G * per_head) * G;
  const int gs = min(G, heads - h0);
  const int r = idx - h0 * per_head;
  head = h0 + r % gs;
  unit = r / gs;
}

struct TileEntry {
  int pos0;
  uint32_t packed;   // bits 0-9 tile index in chunk, 10-20 slot, 21-27 nvalid-1, 31 need_mask
};

__device__ __forceinline__ void decode_tile(const TileEntry &e, TileInfo &t) {
  t.pos0 = e.pos0;
  t.y0 = (int)(e.packed & 0x3ffu) * kTile;
  t.slot = (int)((e.packed >> 10) & 0x7ffu);
  t.nvalid = (int)((e.packed >> 21) & 0x7fu) + 1;
  t.need_mask = (int)(e.packed >> 31);
}

__device__ __forceinline__ TileEntry encode_tile(int pos0, int kt, int slot, int nv, int need_mask) {
  TileEntry e;
  e.pos0 = pos0;
  e.packed = (uint32_t)kt | ((uint32_t)slot << 10) | ((uint32_t)(nv - 1) << 21) | ((uint32_t)need_mask << 31);
  return e;
}

// Exclusive prefix sum over the warp plus a running base; returns this lane's offset.
__device__ __forceinline__ int warp_offset(int cnt, int lane, int &base) {
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  const int off = base + incl - cnt;
  base += __shfl_sync(0xffffffffu, incl, 31);
  return off;
}

// Tiles [t0, t1] of a chunk that starts at natural position cpos (c rows,
// tpc tiles) and meet the positions [lo, hi]; t1 < t0 when none do.
__device__ __forceinline__ void chunk_tiles(int cpos, int c, int tpc, int lo, int hi, int &t0, int &t1) {
  if (hi < lo || hi < cpos || lo > cpos + c - 1) { t0 = 0; t1 = -1; return; }
  const int x = lo - cpos - (kTile - 1);            // first tile whose last row reaches lo
  t0 = x <= 0 ? 0 : (x + kTile - 1) / kTile;
  t1 = min(tpc - 1, (hi - cpos) / kTile);           // last tile whose first row is <= hi
}

// What a stationary query tile (rows at positions qmin..qmax) may attend to:
// keys in [key_lo, key_hi]. A key tile [p0, p0 + nv) needs an element mask if
// it is ragged, reaches padding, crosses the causal diagonal (p0 + nv - 1 >
// qmin), starts before doc_lo_max (the document start of the last query) or
// ends after doc_hi_min (the document end of the first query). Without packed
// documents doc_lo_max = 0 and doc_hi_min = T.
struct KvBounds {
  int key_lo, key_hi, qmin, doc_lo_max, doc_hi_min;
};

// K/V tiles seen by a query tile of rank r (the KvSchedule order: ring steps,
// head chunk then tail chunk). All 32 lanes call it; returns the tile count.
// Writes one batch of (up to 32) chunk groups into the table: lane L's group
// has cnt tiles t0, t0 + 1, ... at tab[off ...]. A few long groups (the usual
// case: 2cp <= 32 groups of up to c/128 tiles) are written by all lanes, one
// group after the other; many short ones by their own lane each.
template <class Make>
__device__ __forceinline__ void write_groups(TileEntry *tab, int groups, int cnt, int off, int t0, int cpos,
                                             int slot, int lane, Make make) {
  if (__reduce_max_sync(0xffffffffu, cnt) > groups) {
    for (int src = 0; src < groups; ++src) {
      const int n = __shfl_sync(0xffffffffu, cnt, src);
      const int o = __shfl_sync(0xffffffffu, off, src);
      const int s0 = __shfl_sync(0xffffffffu, t0, src);
      const int sp = __shfl_sync(0xffffffffu, cpos, src);
      const int ss = __shfl_sync(0xffffffffu, slot, src);
      for (int i = lane; i < n; i += 32) tab[o + i] = make(sp, s0 + i, ss);
    }
  } else {
    for (int i = 0; i < cnt; ++i) tab[off + i] = make(cpos, t0 + i, slot);
  }
}

__device__ inline int build_kv_table(TileEntry *tab, int cp, int c, int r, int causal, int T_valid,
                                     const KvBounds &kb, int lane) {
  const int tpc = (c + kTile - 1) / kTile;
  auto make = [&](int cpos, int kt, int slot) {
    const int pos0 = cpos + kt * kTile;
    const int nv = min(kTile, c - kt * kTile);
    const int nm = (nv < kTile) || (pos0 + nv > T_valid) || (causal && pos0 + nv - 1 > kb.qmin) ||
                   (pos0 < kb.doc_lo_max) || (pos0 + nv > kb.doc_hi_min);
    return encode_tile(pos0, kt, slot, nv, nm);
  };
  int base = 0;
  for (int g0 = 0; g0 < 2 * cp; g0 += 32) {
    const int g = g0 + lane;
    int cnt = 0, cpos = 0, slot = 0, t0 = 0;
    if (g < 2 * cp) {
      const int s = g >> 1, half = g & 1;
      const int j = (r - s + cp) % cp;
      cpos = chunk_of(j, half, cp) * c;
      slot = 2 * j + half;
      int t1;
      chunk_tiles(cpos, c, tpc, kb.key_lo, kb.key_hi, t0, t1);
      cnt = t1 - t0 + 1;
    }
    const int off = warp_offset(cnt, lane, base);
    write_groups(tab, min(32, 2 * cp - g0), cnt, off, t0, cpos, slot, lane, make);
  }
  return base;
}

// What a stationary key tile (rows at positions kmin..kmax) is seen by:
// queries in [q_lo, q_hi]. A query tile [p0, p0 + nv) needs an element mask
// if it or the key tile is ragged, some key is padding, it crosses the causal
// diagonal (kmax > p0), it starts before doc_lo_max (the document start of
// the last key) or ends after doc_hi_min (the document end of the first key).
struct QBounds {
  int q_lo, q_hi, kmax, doc_lo_max, doc_hi_min;
};

// Query tiles that see a key tile of rank j (the QSchedule order: at step s
// the key tile sits on rank (j + s) mod cp).
__device__ inline int build_q_table(TileEntry *tab, int cp, int c, int j, int causal, int T_valid,
                                    const QBounds &qb, int k_ragged, int lane) {
  const int tpc = (c + kTile - 1) / kTile;
  auto make = [&](int cpos, int qt, int slot) {
    const int pos0 = cpos + qt * kTile;
    const int nv = min(kTile, c - qt * kTile);
    const int nm = (nv < kTile) || k_ragged || (qb.kmax >= T_valid) || (causal && qb.kmax > pos0) ||
                   (pos0 < qb.doc_lo_max) || (pos0 + nv > qb.doc_hi_min);
    return encode_tile(pos0, qt, slot, nv, nm);
  };
  int base = 0;
  for (int g0 = 0; g0 < 2 * cp; g0 += 32) {
    const int g = g0 + lane;
    int cnt = 0, cpos = 0, slot = 0, t0 = 0;
    if (g < 2 * cp) {
      const int s = g >> 1, half = g & 1;
      const int r = (j + s) % cp;
      cpos = chunk_of(r, half, cp) * c;
      slot = 2 * r + half;
      int t1;
      chunk_tiles(cpos, c, tpc, qb.q_lo, qb.q_hi, t0, t1);
      cnt = t1 - t0 + 1;
    }
    const int off = warp_offset(cnt, lane, base);
    write_groups(tab, min(32, 2 * cp - g0), cnt, off, t0, cpos, slot, lane, make);
  }
  return base;
}

// Document bounds [lo, hi) of natural position pos from per-position arrays
// (nullptr: one document covering everything); values are clamped to [0, T]
// so that a malformed array cannot send an index out of range.
__device__ __forceinline__ void doc_bounds_at(const int *doc_lo, const int *doc_hi, int pos, int T,
                                              int &lo, int &hi) {
  if (!doc_lo) { lo = 0; hi = T; return; }
  lo = min(max(__ldg(doc_lo + pos), 0), T);
  hi = min(max(__ldg(doc_hi + pos), 0), T);
}

// The KvBounds of a query tile with rows qmin..qmax.
__device__ __forceinline__ KvBounds kv_bounds(const int *doc_lo, const int *doc_hi, int T, int T_valid,
                                              int causal, int qmin, int qmax) {
  int lo_min, hi_min, lo_max, hi_max;
  doc_bounds_at(doc_lo, doc_hi, qmin, T, lo_min, hi_min);
  doc_bounds_at(doc_lo, doc_hi, qmax, T, lo_max, hi_max);
  KvBounds kb;
  kb.key_lo = lo_min;
  kb.key_hi = min(T_valid - 1, causal ? qmax : hi_max - 1);
  if (causal && doc_lo) kb.key_hi = min(kb.key_hi, hi_max - 1);
  kb.qmin = qmin;
  kb.doc_lo_max = lo_max;
  kb.doc_hi_min = hi_min;
  return kb;
}

// The QBounds of a key tile with rows kmin..kmax (no query when every key is padding).
__device__ __forceinline__ QBounds q_bounds(const int *doc_lo, const int *doc_hi, int T, int T_valid,
                                            int causal, int kmin, int kmax) {
  int lo_min, hi_min, lo_max, hi_max;
  doc_bounds_at(doc_lo, doc_hi, kmin, T, lo_min, hi_min);
  doc_bounds_at(doc_lo, doc_hi, kmax, T, lo_max, hi_max);
  QBounds qb;
  qb.q_lo = causal ? kmin : lo_min;
  qb.q_hi = kmin >= T_valid ? -1 : hi_max - 1;
  qb.kmax = kmax;
  qb.doc_lo_max = lo_max;
  qb.doc_hi_min = hi_min;
  return qb;
}

// Stores scale * m R^T of one pair of 32-column chunks of a TMEM row (m the
// attention temperature of the RoPE configuration, 1 for the standard one): columns
// 32a..32a+31 and their rotation partners D/2 further on (frequencies
// 32a..32a+31), for the key or query at natural position pos, as bf16 at
// dst + the same columns (every lane of the warp must call this).
template <int D>
__device__ __forceinline__ void store_tmem_pair_rope(uint32_t t_col0, int a, float scale, int pos,
                                                     const RopeTheta &th, __nv_bfloat16 *dst, bool valid) {
  uint32_t ra[32], rb[32];
  tc::tmem_ld32(t_col0 + 32 * a, ra);
  tc::tmem_ld32(t_col0 + 32 * a + D / 2, rb);
  tc::tmem_ld_wait();
  uint32_t pa[16], pb[16];
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    float o[2][2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      float sn, cs;
      rope_sincos(pos, th.hi[32 * a + e + u], th.lo[32 * a + e + u], sn, cs);
      sn *= th.mscale;
      cs *= th.mscale;
      const float x = __uint_as_float(ra[e + u]) * scale, y = __uint_as_float(rb[e + u]) * scale;
      o[0][u] = fmaf(x, cs, y * sn);    // R^T: x cos + y sin
      o[1][u] = fmaf(y, cs, -x * sn);   //      y cos - x sin
    }
    pa[e / 2] = pack_bf16x2(o[0][0], o[0][1]);
    pb[e / 2] = pack_bf16x2(o[1][0], o[1][1]);
  }
  if (valid) {
    uint4 *da = reinterpret_cast<uint4 *>(dst + 32 * a), *db = reinterpret_cast<uint4 *>(dst + 32 * a + D / 2);
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      da[v] = make_uint4(pa[4 * v], pa[4 * v + 1], pa[4 * v + 2], pa[4 * v + 3]);
      db[v] = make_uint4(pb[4 * v], pb[4 * v + 1], pb[4 * v + 2], pb[4 * v + 3]);
    }
  }
}

}  // namespace cpattn
