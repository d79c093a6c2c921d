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
// or wholly at positions >= T_valid are skipped.
struct KvSchedule {
  int cp, c, tpc, r, causal, T_valid, qmin, qmax;
  int s, half, kt;

  __device__ __forceinline__ void init(int cp_, int c_, int r_, int causal_, int T_valid_,
                                       int qmin_, int qmax_) {
    cp = cp_; c = c_; tpc = (c_ + kTile - 1) / kTile; r = r_; causal = causal_;
    T_valid = T_valid_; qmin = qmin_; qmax = qmax_;
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
      t.slot = 2 * j + half;
      t.y0 = kt * kTile;
      t.pos0 = pos0;
      t.nvalid = nv;
      t.need_mask = (nv < kTile) || (pos0 + nv > T_valid) || (causal && pos0 + nv - 1 > qmin);
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
  int s, half, qt;

  __device__ __forceinline__ void init(int cp_, int c_, int j_, int causal_, int T_valid_,
                                       int kmin_, int kmax_) {
    cp = cp_; c = c_; tpc = (c_ + kTile - 1) / kTile; j = j_; causal = causal_;
    kmin = kmin_; kmax = kmax_;
    kvalid_max = T_valid_;
    s = 0; half = 0; qt = -1;
  }
  // need_mask is set when any pair of the tile may be masked: causal
  // overlap, a ragged query or key tile, or keys at positions >= T_valid.
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
      t.slot = 2 * r + half;
      t.y0 = qt * kTile;
      t.pos0 = pos0;
      t.nvalid = nv;
      t.need_mask = (nv < kTile) || k_ragged || (kmax >= kvalid_max) || (causal && kmax > pos0);
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
                                       int kmin_, int kmax_) {
    group = group_;
    gi = 0;
    q.init(cp_, c_, j_, causal_, T_valid_, kmin_, kmax_);
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
// so both the tile index and the slot fit in 10 bits.
constexpr int kMaxTiles = 1024;   // entries per CTA (8 KiB of shared memory)

struct TileEntry {
  int pos0;
  uint32_t packed;   // bits 0-9 tile index in chunk, 10-19 slot, 20-26 nvalid-1, 31 need_mask
};

__device__ __forceinline__ void decode_tile(const TileEntry &e, TileInfo &t) {
  t.pos0 = e.pos0;
  t.y0 = (int)(e.packed & 0x3ffu) * kTile;
  t.slot = (int)((e.packed >> 10) & 0x3ffu);
  t.nvalid = (int)((e.packed >> 20) & 0x7fu) + 1;
  t.need_mask = (int)(e.packed >> 31);
}

__device__ __forceinline__ TileEntry encode_tile(int pos0, int kt, int slot, int nv, int need_mask) {
  TileEntry e;
  e.pos0 = pos0;
  e.packed = (uint32_t)kt | ((uint32_t)slot << 10) | ((uint32_t)(nv - 1) << 20) | ((uint32_t)need_mask << 31);
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

// K/V tiles seen by a query tile of rank r with positions [qmin, qmax]
// (the KvSchedule order). All 32 lanes call it; returns the tile count.
__device__ inline int build_kv_table(TileEntry *tab, int cp, int c, int r, int causal, int T_valid,
                                     int qmin, int qmax, int lane) {
  const int tpc = (c + kTile - 1) / kTile;
  int base = 0;
  for (int g0 = 0; g0 < 2 * cp; g0 += 32) {
    const int g = g0 + lane;
    int cnt = 0, cpos = 0, slot = 0;
    if (g < 2 * cp) {
      const int s = g >> 1, half = g & 1;
      const int j = (r - s + cp) % cp;
      cpos = chunk_of(j, half, cp) * c;
      slot = 2 * j + half;
      // tile kt is live iff cpos + 128 kt < T_valid and (not causal or cpos + 128 kt <= qmax)
      const int lim = causal ? min(T_valid - 1, qmax) : T_valid - 1;
      cnt = lim < cpos ? 0 : min(tpc - 1, (lim - cpos) / kTile) + 1;
    }
    const int off = warp_offset(cnt, lane, base);
    for (int kt = 0; kt < cnt; ++kt) {
      const int pos0 = cpos + kt * kTile;
      const int nv = min(kTile, c - kt * kTile);
      const int nm = (nv < kTile) || (pos0 + nv > T_valid) || (causal && pos0 + nv - 1 > qmin);
      tab[off + kt] = encode_tile(pos0, kt, slot, nv, nm);
    }
  }
  return base;
}

// Query tiles that see a key tile of rank j with positions [kmin, kmax]
// (the QSchedule order: at step s the key tile sits on rank (j + s) mod cp).
__device__ inline int build_q_table(TileEntry *tab, int cp, int c, int j, int causal, int T_valid,
                                    int kmin, int kmax, int k_ragged, int lane) {
  const int tpc = (c + kTile - 1) / kTile;
  int base = 0;
  for (int g0 = 0; g0 < 2 * cp; g0 += 32) {
    const int g = g0 + lane;
    int cnt = 0, cpos = 0, slot = 0, qt_lo = 0;
    if (g < 2 * cp && kmin < T_valid) {
      const int s = g >> 1, half = g & 1;
      const int r = (j + s) % cp;
      cpos = chunk_of(r, half, cp) * c;
      slot = 2 * r + half;
      if (!causal) {
        qt_lo = 0;
      } else if (cpos + c - 1 < kmin) {   // every query of the chunk precedes every key
        qt_lo = tpc;
      } else {                             // first tile whose last row reaches kmin
        const int x = kmin - cpos - (kTile - 1);
        qt_lo = x <= 0 ? 0 : (x + kTile - 1) / kTile;
      }
      cnt = tpc - qt_lo;
    }
    const int off = warp_offset(cnt, lane, base);
    for (int i = 0; i < cnt; ++i) {
      const int qt = qt_lo + i;
      const int pos0 = cpos + qt * kTile;
      const int nv = min(kTile, c - qt * kTile);
      const int nm = (nv < kTile) || k_ragged || (kmax >= T_valid) || (causal && kmax > pos0);
      tab[off + i] = encode_tile(pos0, qt, slot, nv, nm);
    }
  }
  return base;
}

}  // namespace cpattn
