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

}  // namespace cpattn
