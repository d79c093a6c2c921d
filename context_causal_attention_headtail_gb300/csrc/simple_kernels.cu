// CUDA-core kernels of libcpattn:
//  * HeadTail shard / unshard (HBM-bound chunk copies),
//  * the backward preprocess D = rowsum(dO * O),
//  * the standalone SDPAMerger over n partial (O, LSE),
//  * the exact-fp32 ring attention forward and backward (the correctness
//    path for fp32 inputs; it follows the ring step by step and merges each
//    step's partial with the SDPAMerger rule, as the pages' ring does).
#include <math.h>

#include "device_common.cuh"

namespace cpattn {

static int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

// ---------------------------------------------------- row permutations ---
// Both layouts that the path permutes between are made of chunks of
// contiguous rows: a chunk of the "natural" tensor lands as a chunk of the
// permuted one. A map gives, for chunk ch, its first row on either side and
// the natural (global) position of its first row, used by RoPE.
//
// HeadTail: chunk (bh, kappa) of c rows; natural row (bh*2cp + kappa)*c, the
// sharded copy at slot 2r+half of that (b,h), position kappa*c.
struct HeadTailMap {
  int cp, c;
  __device__ __forceinline__ int rows() const { return c; }
  __device__ __forceinline__ void at(long long ch, long long &nat, long long &perm, int &pos0) const {
    const int two_cp = 2 * cp;
    const long long bh = ch / two_cp;
    const int kappa = (int)(ch % two_cp);
    int r, half;
    owner_of(kappa, cp, r, half);
    nat = (bh * two_cp + kappa) * (long long)c;
    perm = (bh * two_cp + 2 * r + half) * (long long)c;
    pos0 = kappa * c;
  }
};

// Ulysses all-to-all over P virtual ranks (Tl = T/P tokens, Hl = H/P heads
// per rank): chunk (r, b, h) is rank r's Tl tokens of head h. Its "natural"
// side is the stacked sequence shards [P][B][H][Tl] (row ch*Tl); it lands in
// the stacked head shards [P][B][Hl][T] at rank s = h / Hl, local head
// h % Hl, rows r*Tl..; position r*Tl.
struct UlyssesMap {
  int P, B, H, Tl;
  __device__ __forceinline__ int rows() const { return Tl; }
  __device__ __forceinline__ void at(long long ch, long long &nat, long long &perm, int &pos0) const {
    const int Hl = H / P;
    const long long bh_all = (long long)B * H;
    const int r = (int)(ch / bh_all);
    const long long rem = ch % bh_all;
    const int b = (int)(rem / H), h = (int)(rem % H);
    nat = ch * (long long)Tl;
    perm = (((long long)(h / Hl) * B + b) * Hl + h % Hl) * (long long)Tl * P + (long long)r * Tl;
    pos0 = r * Tl;
  }
};

// Ulysses K/V all-to-all when there are fewer heads than ranks (P = rep * H):
// head shard rank s receives head s / rep, all T tokens, as [P][B][1][T].
// Chunk (s, b, r) is rank r's Tl tokens of that head; chunks are enumerated
// on the receiving side, so a sequence-shard chunk is read once per replica.
// Forward direction only: the adjoint sums replicas (ulysses_kv_reduce_kernel).
struct UlyssesRepMap {
  int P, B, H, Tl;
  __device__ __forceinline__ int rows() const { return Tl; }
  __device__ __forceinline__ void at(long long ch, long long &nat, long long &perm, int &pos0) const {
    const long long per_rank = (long long)B * P;
    const int s = (int)(ch / per_rank);
    const long long rem = ch % per_rank;
    const int b = (int)(rem / P), r = (int)(rem % P);
    nat = (((long long)r * B + b) * H + s / (P / H)) * (long long)Tl;
    perm = ((long long)s * B + b) * (long long)Tl * P + (long long)r * Tl;
    pos0 = r * Tl;
  }
};

// Each grid row (y) takes whole chunks, each x-block a strided slice of the
// chunk's 16-byte words.
template <class Map, bool INVERSE>
__global__ void __launch_bounds__(256) permute_kernel(const uint4 *__restrict__ src,
                                                      uint4 *__restrict__ dst, Map map,
                                                      long long n_chunks, int row_u4) {
  const long long chunk_u4 = (long long)map.rows() * row_u4;
  for (long long ch = blockIdx.y; ch < n_chunks; ch += gridDim.y) {
    long long nat, perm;
    int pos0;
    map.at(ch, nat, perm, pos0);
    const uint4 *s = src + (INVERSE ? perm : nat) * row_u4;
    uint4 *d = dst + (INVERSE ? nat : perm) * row_u4;
    const long long stride = (long long)gridDim.x * blockDim.x;
    long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < chunk_u4; i += 4 * stride) {
      uint4 a = s[i], b = s[i + stride], c = s[i + 2 * stride], e = s[i + 3 * stride];
      d[i] = a; d[i + stride] = b; d[i + 2 * stride] = c; d[i + 3 * stride] = e;
    }
    for (; i < chunk_u4; i += stride) d[i] = s[i];
  }
}

template <class Map>
static cpattn_status launch_permute_t(const void *src, void *dst, const Map &map, int rows,
                                      long long n_chunks, int row_u4, bool inverse, cudaStream_t s) {
  const long long chunk_u4 = (long long)rows * row_u4;
  const long long want_blocks = (long long)sm_count() * 8;
  long long bx = (chunk_u4 + 1023) / 1024;
  long long per_chunk = (want_blocks + n_chunks - 1) / n_chunks;
  if (bx > per_chunk) bx = per_chunk;
  if (bx < 1) bx = 1;
  long long gy = n_chunks < 65535 ? n_chunks : 65535;
  dim3 grid((unsigned)bx, (unsigned)gy);
  if (inverse)
    permute_kernel<Map, true><<<grid, 256, 0, s>>>(static_cast<const uint4 *>(src), static_cast<uint4 *>(dst),
                                                   map, n_chunks, row_u4);
  else
    permute_kernel<Map, false><<<grid, 256, 0, s>>>(static_cast<const uint4 *>(src), static_cast<uint4 *>(dst),
                                                    map, n_chunks, row_u4);
  return check_launch(inverse ? "inverse row permutation kernel" : "row permutation kernel");
}

cpattn_status launch_shard(const void *src, void *dst, const Geometry &g, int elt_bytes,
                           bool inverse, cudaStream_t s) {
  const HeadTailMap map{g.cp, g.c};
  return launch_permute_t(src, dst, map, g.c, (long long)g.B * g.H * 2 * g.cp, g.d * elt_bytes / 16,
                          inverse, s);
}

cpattn_status launch_ulysses(const void *src, void *dst, const Geometry &g, int P, int elt_bytes,
                             bool inverse, cudaStream_t s) {
  if (g.H < P) {   // replication; the inverse direction is a reduction
    if (inverse) return launch_ulysses_kv_reduce(src, dst, g, P, elt_bytes == 4 ? CPATTN_F32 : CPATTN_BF16, false, nullptr, s);
    const UlyssesRepMap map{P, g.B, g.H, g.T / P};
    return launch_permute_t(src, dst, map, g.T / P, (long long)P * g.B * P, g.d * elt_bytes / 16, false, s);
  }
  const UlyssesMap map{P, g.B, g.H, g.T / P};
  return launch_permute_t(src, dst, map, g.T / P, (long long)P * g.B * g.H, g.d * elt_bytes / 16,
                          inverse, s);
}

// ------------------------------------------------------- shard + RoPE ---
// A row permutation (HeadTail shard, Ulysses all-to-all) fused with RoPE, and
// its adjoint fused with the inverse permutation, so that the rotation runs
// inside a pass that already reads and writes every element of q and k. Row
// o of a chunk has position p = pos0 + o.
//   forward  (shard):   dst[sigma(t)] = m R(p) src[t]
//   adjoint  (unshard): dst[t] = m R(p)^T src[sigma(t)]
// (m = 1 and the standard frequencies unless a YaRN configuration is given).
// A lane owns VEC consecutive frequencies f0..f0+VEC-1 (one 16-byte word from
// each half of the row) and walks up to 256/RS rows of one chunk with stride
// RS; its cos/sin are seeded with rope_sincos and advanced by an exact
// angle-addition step of RS rows (error grows ~1 ulp per step, <= 16 steps).
template <typename T>
struct VecOf;
template <>
struct VecOf<__nv_bfloat16> { static constexpr int N = 8; };
template <>
struct VecOf<float> { static constexpr int N = 4; };

template <typename T>
__device__ __forceinline__ void unpack16(const uint4 &u, float *x);
template <>
__device__ __forceinline__ void unpack16<__nv_bfloat16>(const uint4 &u, float *x) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) { x[2 * i] = bf16lo_to_f32(w[i]); x[2 * i + 1] = bf16hi_to_f32(w[i]); }
}
template <>
__device__ __forceinline__ void unpack16<float>(const uint4 &u, float *x) {
  x[0] = __uint_as_float(u.x); x[1] = __uint_as_float(u.y);
  x[2] = __uint_as_float(u.z); x[3] = __uint_as_float(u.w);
}
template <typename T>
__device__ __forceinline__ uint4 pack16(const float *x);
template <>
__device__ __forceinline__ uint4 pack16<__nv_bfloat16>(const float *x) {
  return make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                    pack_bf16x2(x[6], x[7]));
}
template <>
__device__ __forceinline__ uint4 pack16<float>(const float *x) {
  return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                    __float_as_uint(x[3]));
}

constexpr int kRopeRowsPerBlock = 256;

// grid: x = row blocks of 256 rows within a chunk, y = chunks of the map.
// block: 256 threads = (D/2)/VEC frequency groups x the rest as row lanes.
template <typename T, int D, class Map, bool INVERSE>
__global__ void __launch_bounds__(256) shard_rope_kernel(const T *__restrict__ src, T *__restrict__ dst,
                                                         Map map, long long n_chunks, RopeTheta th) {
  constexpr int VEC = VecOf<T>::N;
  constexpr int GROUPS = (D / 2) / VEC;       // frequency groups per row
  constexpr int RS = 256 / GROUPS;            // rows advanced per step
  const int grp = threadIdx.x % GROUPS, lrow = threadIdx.x / GROUPS;
  const int f0 = grp * VEC;
  const int c = map.rows();
  for (long long ch = blockIdx.y; ch < n_chunks; ch += gridDim.y) {
    long long nat0, shd0;                      // first row of the chunk on either side
    int pos0;
    map.at(ch, nat0, shd0, pos0);
    const int row_begin = blockIdx.x * kRopeRowsPerBlock + lrow;
    const int row_end = min(c, (int)(blockIdx.x + 1) * kRopeRowsPerBlock);
    if (row_begin >= row_end) continue;
    float cs[VEC], sn[VEC], cd[VEC], sd[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
      rope_sincos(pos0 + row_begin, th.hi[f0 + v], th.lo[f0 + v], sn[v], cs[v]);
      rope_sincos(RS, th.hi[f0 + v], th.lo[f0 + v], sd[v], cd[v]);
    }
    for (int o = row_begin; o < row_end; o += RS) {
      const T *in = src + ((INVERSE ? shd0 : nat0) + o) * D;
      T *out = dst + ((INVERSE ? nat0 : shd0) + o) * D;
      const uint4 ua = *reinterpret_cast<const uint4 *>(in + f0);
      const uint4 ub = *reinterpret_cast<const uint4 *>(in + f0 + D / 2);
      float x[VEC], y[VEC];
      unpack16<T>(ua, x);
      unpack16<T>(ub, y);
#pragma unroll
      for (int v = 0; v < VEC; ++v) {
        const float s_ = INVERSE ? -sn[v] : sn[v];
        const float xr = fmaf(x[v], cs[v], -y[v] * s_);
        const float yr = fmaf(y[v], cs[v], x[v] * s_);
        x[v] = xr * th.mscale;   // m = 1 (exact) for the standard rotation
        y[v] = yr * th.mscale;
        const float nc = fmaf(cs[v], cd[v], -sn[v] * sd[v]);
        const float ns = fmaf(sn[v], cd[v], cs[v] * sd[v]);
        cs[v] = nc;
        sn[v] = ns;
      }
      *reinterpret_cast<uint4 *>(out + f0) = pack16<T>(x);
      *reinterpret_cast<uint4 *>(out + f0 + D / 2) = pack16<T>(y);
    }
  }
}

template <typename T, int D, class Map>
static void launch_rope_t(const void *src, void *dst, const Map &map, int rows, long long n_chunks,
                          bool inverse, const RopeTheta &th, cudaStream_t s) {
  const unsigned gx = (unsigned)((rows + kRopeRowsPerBlock - 1) / kRopeRowsPerBlock);
  const unsigned gy = (unsigned)(n_chunks < 65535 ? n_chunks : 65535);
  dim3 grid(gx, gy);
  if (inverse)
    shard_rope_kernel<T, D, Map, true><<<grid, 256, 0, s>>>(static_cast<const T *>(src), static_cast<T *>(dst),
                                                            map, n_chunks, th);
  else
    shard_rope_kernel<T, D, Map, false><<<grid, 256, 0, s>>>(static_cast<const T *>(src), static_cast<T *>(dst),
                                                             map, n_chunks, th);
}

template <class Map>
static cpattn_status launch_rope_map(const void *src, void *dst, const Map &map, int rows,
                                     long long n_chunks, int d, cpattn_dtype dt, bool inverse,
                                     const cpattn_rope_cfg *cfg, cudaStream_t s) {
  RopeTheta th;
  make_rope_theta(d, &th, cfg);
  if (dt == CPATTN_BF16) {
    if (d == 128) launch_rope_t<__nv_bfloat16, 128>(src, dst, map, rows, n_chunks, inverse, th, s);
    else launch_rope_t<__nv_bfloat16, 64>(src, dst, map, rows, n_chunks, inverse, th, s);
  } else {
    if (d == 128) launch_rope_t<float, 128>(src, dst, map, rows, n_chunks, inverse, th, s);
    else launch_rope_t<float, 64>(src, dst, map, rows, n_chunks, inverse, th, s);
  }
  return check_launch(inverse ? "inverse permutation + RoPE kernel" : "permutation + RoPE kernel");
}

// ---------------------------------------------- several tensors, one launch ---
// The HeadTail shard (or unshard) of up to kBatchMax tensors of one sequence
// layout in one launch: blockIdx.y walks the chunks of every tensor in turn,
// blockIdx.x the 256-row blocks of a chunk. A tensor with rope set goes
// through the RoPE pass of shard_rope_kernel (R on the way in, R^T on the way
// out), the others through a plain 16-byte copy; one launch instead of one per
// tensor saves the ramp-up and drain of the separate launches.
template <typename T, int D, bool INVERSE>
__global__ void __launch_bounds__(256) shard_batch_kernel(ShardBatch b, HeadTailMap map, RopeTheta th) {
  constexpr int VEC = VecOf<T>::N;
  constexpr int GROUPS = (D / 2) / VEC;       // frequency groups per row
  constexpr int RS = 256 / GROUPS;            // rows advanced per step
  constexpr int ROW_U4 = D * (int)sizeof(T) / 16;
  const int c = map.rows();
  for (long long ch = blockIdx.y; ch < b.n_chunks; ch += gridDim.y) {
    int i = 0;
#pragma unroll 1
    while (i + 1 < b.n && ch >= b.first_chunk[i + 1]) ++i;
    long long nat0, shd0;
    int pos0;
    map.at(ch - b.first_chunk[i], nat0, shd0, pos0);
    const int r_begin = blockIdx.x * kRopeRowsPerBlock;
    const int r_end = min(c, r_begin + kRopeRowsPerBlock);
    if (r_begin >= r_end) continue;
    const T *src = static_cast<const T *>(b.src[i]);
    T *dst = static_cast<T *>(b.dst[i]);
    if (!b.rope[i]) {   // rows [r_begin, r_end) are contiguous on both sides
      const uint4 *s4 = reinterpret_cast<const uint4 *>(src + ((INVERSE ? shd0 : nat0) + r_begin) * D);
      uint4 *d4 = reinterpret_cast<uint4 *>(dst + ((INVERSE ? nat0 : shd0) + r_begin) * D);
      const int n4 = (r_end - r_begin) * ROW_U4;
      int j = threadIdx.x;
      for (; j + 3 * 256 < n4; j += 4 * 256) {
        const uint4 a = s4[j], bb = s4[j + 256], cc = s4[j + 512], e = s4[j + 768];
        d4[j] = a; d4[j + 256] = bb; d4[j + 512] = cc; d4[j + 768] = e;
      }
      for (; j < n4; j += 256) d4[j] = s4[j];
      continue;
    }
    const int grp = threadIdx.x % GROUPS, lrow = threadIdx.x / GROUPS;
    const int f0 = grp * VEC;
    const int row_begin = r_begin + lrow;
    if (row_begin >= r_end) continue;
    float cs[VEC], sn[VEC], cd[VEC], sd[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
      rope_sincos(pos0 + row_begin, th.hi[f0 + v], th.lo[f0 + v], sn[v], cs[v]);
      rope_sincos(RS, th.hi[f0 + v], th.lo[f0 + v], sd[v], cd[v]);
    }
    for (int o = row_begin; o < r_end; o += RS) {
      const T *in = src + ((INVERSE ? shd0 : nat0) + o) * D;
      T *out = dst + ((INVERSE ? nat0 : shd0) + o) * D;
      const uint4 ua = *reinterpret_cast<const uint4 *>(in + f0);
      const uint4 ub = *reinterpret_cast<const uint4 *>(in + f0 + D / 2);
      float x[VEC], y[VEC];
      unpack16<T>(ua, x);
      unpack16<T>(ub, y);
#pragma unroll
      for (int v = 0; v < VEC; ++v) {
        const float s_ = INVERSE ? -sn[v] : sn[v];
        const float xr = fmaf(x[v], cs[v], -y[v] * s_);
        const float yr = fmaf(y[v], cs[v], x[v] * s_);
        x[v] = xr * th.mscale;
        y[v] = yr * th.mscale;
        const float nc = fmaf(cs[v], cd[v], -sn[v] * sd[v]);
        const float ns = fmaf(sn[v], cd[v], cs[v] * sd[v]);
        cs[v] = nc;
        sn[v] = ns;
      }
      *reinterpret_cast<uint4 *>(out + f0) = pack16<T>(x);
      *reinterpret_cast<uint4 *>(out + f0 + D / 2) = pack16<T>(y);
    }
  }
}

template <typename T, int D>
static void launch_shard_batch_t(const ShardBatch &b, const HeadTailMap &map, bool inverse, const RopeTheta &th,
                                 cudaStream_t s) {
  const unsigned gx = (unsigned)((map.c + kRopeRowsPerBlock - 1) / kRopeRowsPerBlock);
  const unsigned gy = (unsigned)(b.n_chunks < 65535 ? b.n_chunks : 65535);
  dim3 grid(gx, gy);
  if (inverse) shard_batch_kernel<T, D, true><<<grid, 256, 0, s>>>(b, map, th);
  else shard_batch_kernel<T, D, false><<<grid, 256, 0, s>>>(b, map, th);
}

cpattn_status launch_shard_batch(const ShardBatch &b, const Geometry &g, cpattn_dtype dt, bool inverse,
                                 const cpattn_rope_cfg *cfg, cudaStream_t s) {
  RopeTheta th;
  make_rope_theta(g.d, &th, cfg);
  const HeadTailMap map{g.cp, g.c};
  if (dt == CPATTN_BF16) {
    if (g.d == 128) launch_shard_batch_t<__nv_bfloat16, 128>(b, map, inverse, th, s);
    else launch_shard_batch_t<__nv_bfloat16, 64>(b, map, inverse, th, s);
  } else {
    if (g.d == 128) launch_shard_batch_t<float, 128>(b, map, inverse, th, s);
    else launch_shard_batch_t<float, 64>(b, map, inverse, th, s);
  }
  return check_launch(inverse ? "batched unshard kernel" : "batched shard kernel");
}

// RoPE of a tensor that is already HeadTail-sharded: chunk ch = (head, slot)
// keeps its rows (nat = perm), its first row sits at natural position
// chunk_of(slot / 2, slot % 2) * c.
struct SlotMap {
  int cp, c;
  __device__ __forceinline__ int rows() const { return c; }
  __device__ __forceinline__ void at(long long ch, long long &nat, long long &perm, int &pos0) const {
    const int slot = (int)(ch % (2 * cp));
    nat = perm = ch * (long long)c;
    pos0 = chunk_of(slot >> 1, slot & 1, cp) * c;
  }
};

// The rotation of shard_rope_kernel on a sharded tensor, without __restrict__:
// dst may equal src (every element is read and then written by one thread).
template <typename T, int D, bool INVERSE>
__global__ void __launch_bounds__(256) rope_sharded_kernel(const T *src, T *dst, SlotMap map, long long n_chunks,
                                                           RopeTheta th) {
  constexpr int VEC = VecOf<T>::N;
  constexpr int GROUPS = (D / 2) / VEC;
  constexpr int RS = 256 / GROUPS;
  const int grp = threadIdx.x % GROUPS, lrow = threadIdx.x / GROUPS;
  const int f0 = grp * VEC;
  const int c = map.rows();
  for (long long ch = blockIdx.y; ch < n_chunks; ch += gridDim.y) {
    long long row0, unused;
    int pos0;
    map.at(ch, row0, unused, pos0);
    const int row_begin = blockIdx.x * kRopeRowsPerBlock + lrow;
    const int row_end = min(c, (int)(blockIdx.x + 1) * kRopeRowsPerBlock);
    if (row_begin >= row_end) continue;
    float cs[VEC], sn[VEC], cd[VEC], sd[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
      rope_sincos(pos0 + row_begin, th.hi[f0 + v], th.lo[f0 + v], sn[v], cs[v]);
      rope_sincos(RS, th.hi[f0 + v], th.lo[f0 + v], sd[v], cd[v]);
    }
    for (int o = row_begin; o < row_end; o += RS) {
      const T *in = src + (row0 + o) * D;
      T *out = dst + (row0 + o) * D;
      const uint4 ua = *reinterpret_cast<const uint4 *>(in + f0);
      const uint4 ub = *reinterpret_cast<const uint4 *>(in + f0 + D / 2);
      float x[VEC], y[VEC];
      unpack16<T>(ua, x);
      unpack16<T>(ub, y);
#pragma unroll
      for (int v = 0; v < VEC; ++v) {
        const float s_ = INVERSE ? -sn[v] : sn[v];
        const float xr = fmaf(x[v], cs[v], -y[v] * s_);
        const float yr = fmaf(y[v], cs[v], x[v] * s_);
        x[v] = xr * th.mscale;
        y[v] = yr * th.mscale;
        const float nc = fmaf(cs[v], cd[v], -sn[v] * sd[v]);
        const float ns = fmaf(sn[v], cd[v], cs[v] * sd[v]);
        cs[v] = nc;
        sn[v] = ns;
      }
      *reinterpret_cast<uint4 *>(out + f0) = pack16<T>(x);
      *reinterpret_cast<uint4 *>(out + f0 + D / 2) = pack16<T>(y);
    }
  }
}

template <typename T, int D>
static void launch_rope_sharded_t(const void *src, void *dst, const SlotMap &map, long long n_chunks, bool inverse,
                                  const RopeTheta &th, cudaStream_t s) {
  const unsigned gx = (unsigned)((map.c + kRopeRowsPerBlock - 1) / kRopeRowsPerBlock);
  const unsigned gy = (unsigned)(n_chunks < 65535 ? n_chunks : 65535);
  dim3 grid(gx, gy);
  if (inverse)
    rope_sharded_kernel<T, D, true><<<grid, 256, 0, s>>>(static_cast<const T *>(src), static_cast<T *>(dst), map,
                                                         n_chunks, th);
  else
    rope_sharded_kernel<T, D, false><<<grid, 256, 0, s>>>(static_cast<const T *>(src), static_cast<T *>(dst), map,
                                                          n_chunks, th);
}

cpattn_status launch_rope_sharded(const void *src, void *dst, const Geometry &g, int heads, cpattn_dtype dt,
                                  bool inverse, const cpattn_rope_cfg *cfg, cudaStream_t s) {
  RopeTheta th;
  make_rope_theta(g.d, &th, cfg);
  const SlotMap map{g.cp, g.c};
  const long long n_chunks = (long long)g.B * heads * 2 * g.cp;
  if (dt == CPATTN_BF16) {
    if (g.d == 128) launch_rope_sharded_t<__nv_bfloat16, 128>(src, dst, map, n_chunks, inverse, th, s);
    else launch_rope_sharded_t<__nv_bfloat16, 64>(src, dst, map, n_chunks, inverse, th, s);
  } else {
    if (g.d == 128) launch_rope_sharded_t<float, 128>(src, dst, map, n_chunks, inverse, th, s);
    else launch_rope_sharded_t<float, 64>(src, dst, map, n_chunks, inverse, th, s);
  }
  return check_launch(inverse ? "RoPE^T kernel (sharded rows)" : "RoPE kernel (sharded rows)");
}

cpattn_status launch_shard_rope(const void *src, void *dst, const Geometry &g, cpattn_dtype dt,
                                bool inverse, const cpattn_rope_cfg *cfg, cudaStream_t s) {
  const HeadTailMap map{g.cp, g.c};
  return launch_rope_map(src, dst, map, g.c, (long long)g.B * g.H * 2 * g.cp, g.d, dt, inverse, cfg, s);
}

cpattn_status launch_ulysses_rope(const void *src, void *dst, const Geometry &g, int P, cpattn_dtype dt,
                                  bool inverse, const cpattn_rope_cfg *cfg, cudaStream_t s) {
  if (g.H < P) {
    if (inverse) return launch_ulysses_kv_reduce(src, dst, g, P, dt, true, cfg, s);
    const UlyssesRepMap map{P, g.B, g.H, g.T / P};
    return launch_rope_map(src, dst, map, g.T / P, (long long)P * g.B * P, g.d, dt, false, cfg, s);
  }
  const UlyssesMap map{P, g.B, g.H, g.T / P};
  return launch_rope_map(src, dst, map, g.T / P, (long long)P * g.B * g.H, g.d, dt, inverse, cfg, s);
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Adjoint of the replicating K/V all-to-all: sequence-shard row (r, b, h, t)
// is the sum, in fp32, of the rep head-shard rows (s, b, 0, r*Tl + t) with
// s / rep = h, rounded once to the storage type; with RoPE the sum is then
// turned by (m R(p))^T at p = r*Tl + t. One thread per (row, rotation pair).
template <typename T, int D, bool ROPE>
__global__ void __launch_bounds__(256) ulysses_kv_reduce_kernel(const T *__restrict__ src, T *__restrict__ dst,
                                                                int P, int B, int H, int Tl, long long rows,
                                                                RopeTheta th) {
  constexpr int HALF = D / 2;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= rows * HALF) return;
  const long long row = idx / HALF;
  const int i = (int)(idx % HALF);
  const int t = (int)(row % Tl);
  const long long rbh = row / Tl;                 // (r*B + b)*H + h
  const int h = (int)(rbh % H);
  const long long rb = rbh / H;
  const int b = (int)(rb % B), r = (int)(rb / B);
  const int rep = P / H;
  float x = 0.f, y = 0.f;
  for (int j = 0; j < rep; ++j) {
    const int s = h * rep + j;
    const T *in = src + (((long long)s * B + b) * (long long)Tl * P + (long long)r * Tl + t) * D;
    x += to_f32(in[i]);
    y += to_f32(in[i + HALF]);
  }
  if (ROPE) {
    float sn, cs;
    rope_sincos(r * Tl + t, th.hi[i], th.lo[i], sn, cs);
    const float xr = fmaf(x, cs, y * sn), yr = fmaf(y, cs, -x * sn);
    x = xr * th.mscale;
    y = yr * th.mscale;
  }
  T *out = dst + row * D;
  out[i] = from_f32<T>(x);
  out[i + HALF] = from_f32<T>(y);
}

cpattn_status launch_ulysses_kv_reduce(const void *src, void *dst, const Geometry &g, int P, cpattn_dtype dt,
                                       bool rope, const cpattn_rope_cfg *cfg, cudaStream_t s) {
  RopeTheta th;
  make_rope_theta(g.d, &th, cfg);
  const long long rows = (long long)P * g.B * g.H * (g.T / P);
  const unsigned blocks = (unsigned)((rows * (g.d / 2) + 255) / 256);
  const int Tl = g.T / P;
#define CPATTN_REDUCE(TT, DD, RR)                                                                         \
  ulysses_kv_reduce_kernel<TT, DD, RR><<<blocks, 256, 0, s>>>(static_cast<const TT *>(src), static_cast<TT *>(dst), \
                                                               P, g.B, g.H, Tl, rows, th)
  if (dt == CPATTN_BF16) {
    if (g.d == 128) { if (rope) CPATTN_REDUCE(__nv_bfloat16, 128, true); else CPATTN_REDUCE(__nv_bfloat16, 128, false); }
    else { if (rope) CPATTN_REDUCE(__nv_bfloat16, 64, true); else CPATTN_REDUCE(__nv_bfloat16, 64, false); }
  } else {
    if (g.d == 128) { if (rope) CPATTN_REDUCE(float, 128, true); else CPATTN_REDUCE(float, 128, false); }
    else { if (rope) CPATTN_REDUCE(float, 64, true); else CPATTN_REDUCE(float, 64, false); }
  }
#undef CPATTN_REDUCE
  return check_launch("Ulysses K/V reduce kernel");
}

// -------------------------------------------------- document bounds ---
// Packed documents: document i holds natural positions [cu[i], cu[i+1]);
// positions >= cu[n] hold padding and get the empty range [cu[n], cu[n]).
// Thread p finds the last i with cu[i] <= p by binary search. Threads
// i < n also check the list (cu[0] = 0, non-decreasing, cu[n] <= T); a bad
// list raises ERR_FLAG_BAD_DOCS and every index stays clamped to [0, T].
__global__ void __launch_bounds__(256) doc_bounds_kernel(const int *__restrict__ cu, int n, int T,
                                                         int *__restrict__ doc_lo,
                                                         int *__restrict__ doc_hi, int *err) {
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  if (p <= n && err) {
    const int x = __ldg(cu + p);
    const bool bad = (p == 0 && x != 0) || (p == n && x > T) || (p < n && x > __ldg(cu + p + 1)) || x < 0;
    if (bad) atomicOr(err, ERR_FLAG_BAD_DOCS);
  }
  if (p >= T) return;
  const int end = min(max(__ldg(cu + n), 0), T);
  int lo = end, hi = end;
  if (p < end) {
    int a = 0, b = n - 1;                      // invariant: the answer is in [a, b]
    while (a < b) {
      const int m = (a + b + 1) >> 1;
      if (__ldg(cu + m) <= p) a = m;
      else b = m - 1;
    }
    lo = min(max(__ldg(cu + a), 0), T);
    hi = min(max(__ldg(cu + a + 1), 0), T);
  }
  doc_lo[p] = lo;
  doc_hi[p] = hi;
}

cpattn_status launch_doc_bounds(const int *cu_seqlens, int n_docs, int T, int *doc_lo, int *doc_hi,
                                cudaStream_t s) {
  const int threads = 256;
  const long long need = (long long)(T > n_docs + 1 ? T : n_docs + 1);
  doc_bounds_kernel<<<(unsigned)((need + threads - 1) / threads), threads, 0, s>>>(
      cu_seqlens, n_docs, T, doc_lo, doc_hi, device_err_flag());
  return check_launch("document bounds kernel");
}

// ------------------------------------------------------------- D = dO.O ---
template <typename T>
__device__ __forceinline__ float ld_f(const T *p);
template <>
__device__ __forceinline__ float ld_f<float>(const float *p) { return *p; }
template <>
__device__ __forceinline__ float ld_f<__nv_bfloat16>(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

// One warp per row; lane l reads elements l, l+32, ... (coalesced rows).
template <typename T>
__global__ void __launch_bounds__(256) preprocess_kernel(const T *__restrict__ o,
                                                         const T *__restrict__ dO,
                                                         float *__restrict__ D, long long rows,
                                                         int d) {
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows;
       row += warps) {
    const T *a = o + row * d, *b = dO + row * d;
    float acc = 0.f;
    for (int e = lane; e < d; e += 32) acc = fmaf(ld_f(a + e), ld_f(b + e), acc);
    for (int off = 16; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) D[row] = acc;
  }
}

// bf16 rows read as 16-byte words: DD/8 lanes share a row (16 for d = 128),
// so a warp covers 32/(DD/8) rows per step and takes two steps per iteration
// (four independent 16-byte loads per lane in flight); the partial dot
// products are summed over the row's lanes with shuffles.
template <int DD>
__global__ void __launch_bounds__(256) preprocess_bf16_kernel(const uint4 *__restrict__ o,
                                                              const uint4 *__restrict__ dO,
                                                              float *__restrict__ D, long long rows) {
  constexpr int LPR = DD / 8;    // lanes per row
  constexpr int RPW = 32 / LPR;  // rows per warp step
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPR, w = lane % LPR;
  const long long gw = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const long long nw = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long base = gw * (2 * RPW); base < rows; base += nw * (2 * RPW)) {
    uint4 a[2], b[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const long long row = base + u * RPW + sub;
      a[u] = row < rows ? o[row * LPR + w] : make_uint4(0u, 0u, 0u, 0u);
      b[u] = row < rows ? dO[row * LPR + w] : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint32_t aw[4] = {a[u].x, a[u].y, a[u].z, a[u].w}, bw[4] = {b[u].x, b[u].y, b[u].z, b[u].w};
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc = fmaf(bf16lo_to_f32(aw[k]), bf16lo_to_f32(bw[k]), acc);
        acc = fmaf(bf16hi_to_f32(aw[k]), bf16hi_to_f32(bw[k]), acc);
      }
#pragma unroll
      for (int off = LPR / 2; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      const long long row = base + u * RPW + sub;
      if (w == 0 && row < rows) D[row] = acc;
    }
  }
}

cpattn_status launch_bwd_preprocess(const void *o, const void *dO, float *D, long long rows,
                                    int d, cpattn_dtype dt, cudaStream_t s) {
  const long long cap = (long long)sm_count() * 16;
  if (dt == CPATTN_F32) {
    long long blocks = (rows + 7) / 8;
    if (blocks > cap) blocks = cap;
    preprocess_kernel<float><<<(unsigned)blocks, 256, 0, s>>>(
        static_cast<const float *>(o), static_cast<const float *>(dO), D, rows, d);
  } else {
    const long long rows_per_block = 8 * 2 * (32 / (d / 8));   // 8 warps, two steps each
    long long blocks = (rows + rows_per_block - 1) / rows_per_block;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (d == 128)
      preprocess_bf16_kernel<128><<<(unsigned)blocks, 256, 0, s>>>(
          static_cast<const uint4 *>(o), static_cast<const uint4 *>(dO), D, rows);
    else
      preprocess_bf16_kernel<64><<<(unsigned)blocks, 256, 0, s>>>(
          static_cast<const uint4 *>(o), static_cast<const uint4 *>(dO), D, rows);
  }
  return check_launch("backward preprocess kernel");
}

// ------------------------------------------------------------------ merge ---
struct MergeParts {
  const float *o[16];
  const float *l[16];
};

// One warp per row. Lane i < n reads L_i; the max, the weights and their sum
// are formed with shuffles and each weight is broadcast from its lane while
// every lane accumulates its d/32-wide slice of O.
template <int D, typename TO>
__global__ void __launch_bounds__(256) merge_kernel(MergeParts parts, int n, TO *__restrict__ o,
                                                    float *__restrict__ lse, long long rows) {
  constexpr int V = D / 32;  // floats per lane (2 or 4)
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows;
       row += warps) {
    float li = lane < n ? parts.l[lane][row] : -INFINITY;
    float m = li;
    for (int off = 16; off; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    const bool empty = !(m > -INFINITY);
    float w = (lane < n && li > -INFINITY) ? expf(li - m) : 0.f;
    float tot = w;
    for (int off = 16; off; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
    float acc[V];
#pragma unroll
    for (int e = 0; e < V; ++e) acc[e] = 0.f;
    for (int i = 0; i < n; ++i) {
      const float wi = __shfl_sync(0xffffffffu, w, i);
      if (empty || wi == 0.f) continue;
      const float *src = parts.o[i] + row * D + lane * V;
      if constexpr (V == 4) {
        float4 x = *reinterpret_cast<const float4 *>(src);
        acc[0] = fmaf(wi, x.x, acc[0]); acc[1] = fmaf(wi, x.y, acc[1]);
        acc[2] = fmaf(wi, x.z, acc[2]); acc[3] = fmaf(wi, x.w, acc[3]);
      } else {
        float2 x = *reinterpret_cast<const float2 *>(src);
        acc[0] = fmaf(wi, x.x, acc[0]); acc[1] = fmaf(wi, x.y, acc[1]);
      }
    }
    const float inv = empty ? 0.f : 1.f / tot;
    TO *dst = o + row * D + lane * V;
#pragma unroll
    for (int e = 0; e < V; ++e) {
      if constexpr (sizeof(TO) == 4) dst[e] = acc[e] * inv;
      else dst[e] = __float2bfloat16_rn(acc[e] * inv);
    }
    if (lane == 0) lse[row] = empty ? -INFINITY : m + logf(tot);
  }
}

cpattn_status launch_merge(const float *const *o_parts, const float *const *lse_parts, int n,
                           void *o, float *lse, long long rows, int d, cpattn_dtype dt,
                           cudaStream_t s) {
  MergeParts p;
  for (int i = 0; i < 16; ++i) {
    p.o[i] = i < n ? o_parts[i] : nullptr;
    p.l[i] = i < n ? lse_parts[i] : nullptr;
  }
  long long blocks = (rows + 7) / 8;
  long long cap = (long long)sm_count() * 16;
  if (blocks > cap) blocks = cap;
  const unsigned gb = (unsigned)blocks;
  if (d == 128) {
    if (dt == CPATTN_F32) merge_kernel<128, float><<<gb, 256, 0, s>>>(p, n, static_cast<float *>(o), lse, rows);
    else merge_kernel<128, __nv_bfloat16><<<gb, 256, 0, s>>>(p, n, static_cast<__nv_bfloat16 *>(o), lse, rows);
  } else {
    if (dt == CPATTN_F32) merge_kernel<64, float><<<gb, 256, 0, s>>>(p, n, static_cast<float *>(o), lse, rows);
    else merge_kernel<64, __nv_bfloat16><<<gb, 256, 0, s>>>(p, n, static_cast<__nv_bfloat16 *>(o), lse, rows);
  }
  return check_launch("merge kernel");
}

// ------------------------------------------------- exact fp32 ring attention ---
// Geometry of sharded row i: rank r = i / 2c, half = (i % 2c) / c; its
// natural position is chunk_of(r, half) * c + i % c.
__device__ __forceinline__ int natural_pos(int i, int c, int cp) {
  const int r = i / (2 * c), l = i % (2 * c);
  return chunk_of(r, l / c, cp) * c + (l % c);
}

// A lane holds elements lane + 32*e of a row (e < D/32); for rotate-half
// RoPE the partner of e is e +- D/64, held by the same lane. Angles are taken
// in double from the frequency pair (hi + lo) of the RoPE configuration, and
// the rotation carries its temperature m (m R, or m R^T for gradients): this
// path is about exactness, not speed.
template <int D>
__device__ __forceinline__ void rope_row_f32(float (&x)[D / 32], int pos, int lane, bool transpose,
                                             const RopeTheta &th) {
  constexpr int V = D / 32, HV = V / 2;
#pragma unroll
  for (int e = 0; e < HV; ++e) {
    const int i = lane + 32 * e;  // frequency index < D/2
    const double theta = (double)th.hi[i] + (double)th.lo[i];
    double sn, cs;
    sincos((double)pos * theta, &sn, &cs);
    const float c = (float)cs * th.mscale, s = (transpose ? -(float)sn : (float)sn) * th.mscale;
    const float a = x[e], b = x[e + HV];
    x[e] = a * c - b * s;
    x[e + HV] = b * c + a * s;
  }
}

template <int D>
__device__ __forceinline__ void load_row(const float *p, int lane, float (&x)[D / 32]) {
#pragma unroll
  for (int e = 0; e < D / 32; ++e) x[e] = p[lane + 32 * e];
}

template <int D>
__device__ __forceinline__ float warp_dot(const float (&a)[D / 32], const float (&b)[D / 32]) {
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < D / 32; ++e) s = fmaf(a[e], b[e], s);
  for (int off = 16; off; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  return s;
}

__device__ __forceinline__ bool pair_allowed(int qp, int kp, const Geometry &g) {
  if (!((!g.causal || kp <= qp) && kp < g.T_valid)) return false;
  if (!g.doc_lo) return true;
  // packed documents: the key must lie in the query's document [lo, hi)
  const int lo = min(max(__ldg(g.doc_lo + qp), 0), g.T), hi = min(max(__ldg(g.doc_hi + qp), 0), g.T);
  return kp >= lo && kp < hi;
}

// Forward: one warp per sharded query row. For ring step s the row's rank r
// holds the K/V of rank j = (r - s) mod cp; the step's partial (O_s, LSE_s)
// is formed over that rank's head and tail chunks and merged into the
// running result with the SDPAMerger rule.
template <int D>
__global__ void __launch_bounds__(128) fwd_f32_kernel(const float *__restrict__ q,
                                                      const float *__restrict__ k,
                                                      const float *__restrict__ v,
                                                      float *__restrict__ o, float *__restrict__ lse,
                                                      Geometry g,
    const __grid_constant__ RopeTheta th) {
  constexpr int V = D / 32;
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= (long long)g.B * g.H * g.T) return;
  const long long bh = row / g.T;
  const int i = (int)(row % g.T);
  const int r = i / (2 * g.c);
  const int qp = natural_pos(i, g.c, g.cp);
  const float scale = 1.f / sqrtf((float)D);
  const long long bkv = bh / (g.H / g.Hkv);   // K/V head of this query head's group
  const float *kb = k + bkv * g.T * D, *vb = v + bkv * g.T * D;
  float qr[V];
  load_row<D>(q + row * D, lane, qr);
  if (g.rope) rope_row_f32<D>(qr, qp, lane, false, th);
  float O[V], L = -INFINITY;
#pragma unroll
  for (int e = 0; e < V; ++e) O[e] = 0.f;
  for (int s = 0; s < g.cp; ++s) {
    const int j = (r - s + g.cp) % g.cp;
    float m_s = -INFINITY, l_s = 0.f, acc[V];
#pragma unroll
    for (int e = 0; e < V; ++e) acc[e] = 0.f;
    for (int half = 0; half < 2; ++half) {
      const int kappa = chunk_of(j, half, g.cp);
      const int row0 = 2 * g.c * j + half * g.c;
      for (int u = 0; u < g.c; ++u) {
        const int kp = kappa * g.c + u;
        if (!pair_allowed(qp, kp, g)) continue;
        float kr[V], vr[V];
        load_row<D>(kb + (long long)(row0 + u) * D, lane, kr);
        if (g.rope) rope_row_f32<D>(kr, kp, lane, false, th);
        load_row<D>(vb + (long long)(row0 + u) * D, lane, vr);
        const float sc = warp_dot<D>(qr, kr) * scale;
        const float m_new = fmaxf(m_s, sc);
        const float alpha = expf(m_s - m_new);  // 0 when m_s = -inf
        const float p = expf(sc - m_new);
        l_s = l_s * alpha + p;
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] = fmaf(p, vr[e], acc[e] * alpha);
        m_s = m_new;
      }
    }
    if (m_s > -INFINITY) {  // merge step partial (acc/l_s, m_s + log l_s) into (O, L)
      const float L_s = m_s + logf(l_s);
      const float m = fmaxf(L, L_s);
      const float wa = (L > -INFINITY) ? expf(L - m) : 0.f, wb = expf(L_s - m);
      const float tot = wa + wb;
#pragma unroll
      for (int e = 0; e < V; ++e) O[e] = (wa * O[e] + wb * (acc[e] / l_s)) / tot;
      L = m + logf(tot);
    }
  }
#pragma unroll
  for (int e = 0; e < V; ++e) o[row * D + lane + 32 * e] = O[e];
  if (lane == 0) lse[row] = L;
}

// dQ: one warp per sharded query row, over every allowed key.
template <int D>
__global__ void __launch_bounds__(128) bwd_dq_f32_kernel(const float *__restrict__ q,
                                                         const float *__restrict__ k,
                                                         const float *__restrict__ v,
                                                         const float *__restrict__ lse,
                                                         const float *__restrict__ dO,
                                                         const float *__restrict__ Dv,
                                                         float *__restrict__ dq, Geometry g,
    const __grid_constant__ RopeTheta th) {
  constexpr int V = D / 32;
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= (long long)g.B * g.H * g.T) return;
  const long long bh = row / g.T;
  const int i = (int)(row % g.T);
  const int r = i / (2 * g.c);
  const int qp = natural_pos(i, g.c, g.cp);
  const float scale = 1.f / sqrtf((float)D);
  const long long bkv = bh / (g.H / g.Hkv);
  const float *kb = k + bkv * g.T * D, *vb = v + bkv * g.T * D;
  float qr[V], dor[V], acc[V];
  load_row<D>(q + row * D, lane, qr);
  if (g.rope) rope_row_f32<D>(qr, qp, lane, false, th);
  load_row<D>(dO + row * D, lane, dor);
  const float L = lse[row], Dt = Dv[row];
#pragma unroll
  for (int e = 0; e < V; ++e) acc[e] = 0.f;
  for (int s = 0; s < g.cp; ++s) {
    const int j = (r - s + g.cp) % g.cp;
    for (int half = 0; half < 2; ++half) {
      const int kappa = chunk_of(j, half, g.cp);
      const int row0 = 2 * g.c * j + half * g.c;
      for (int u = 0; u < g.c; ++u) {
        const int kp = kappa * g.c + u;
        if (!pair_allowed(qp, kp, g)) continue;
        float kr[V], vr[V];
        load_row<D>(kb + (long long)(row0 + u) * D, lane, kr);
        if (g.rope) rope_row_f32<D>(kr, kp, lane, false, th);
        load_row<D>(vb + (long long)(row0 + u) * D, lane, vr);
        const float p = expf(warp_dot<D>(qr, kr) * scale - L);
        const float ds = p * (warp_dot<D>(dor, vr) - Dt);
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] = fmaf(ds, kr[e], acc[e]);
      }
    }
  }
#pragma unroll
  for (int e = 0; e < V; ++e) acc[e] *= scale;
  if (g.rope) rope_row_f32<D>(acc, qp, lane, true, th);
#pragma unroll
  for (int e = 0; e < V; ++e) dq[row * D + lane + 32 * e] = acc[e];
}

// dK, dV: one warp per sharded key row of one K/V head. Its K/V travel the
// ring: at step s they sit on rank (j + s) mod cp, whose queries add their
// contributions; with grouped K/V heads, the group's query heads add theirs
// one after another.
template <int D>
__global__ void __launch_bounds__(128) bwd_dkdv_f32_kernel(const float *__restrict__ q,
                                                           const float *__restrict__ k,
                                                           const float *__restrict__ v,
                                                           const float *__restrict__ lse,
                                                           const float *__restrict__ dO,
                                                           const float *__restrict__ Dv,
                                                           float *__restrict__ dk,
                                                           float *__restrict__ dv, Geometry g,
    const __grid_constant__ RopeTheta th) {
  constexpr int V = D / 32;
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= (long long)g.B * g.Hkv * g.T) return;
  const long long bkv = row / g.T;
  const int i = (int)(row % g.T);
  const int j = i / (2 * g.c);
  const int kp = natural_pos(i, g.c, g.cp);
  const float scale = 1.f / sqrtf((float)D);
  const int group = g.H / g.Hkv;
  float kr[V], vr[V], adk[V], adv[V];
  load_row<D>(k + row * D, lane, kr);
  if (g.rope) rope_row_f32<D>(kr, kp, lane, false, th);
  load_row<D>(v + row * D, lane, vr);
#pragma unroll
  for (int e = 0; e < V; ++e) { adk[e] = 0.f; adv[e] = 0.f; }
  for (int gi = 0; gi < group; ++gi) {
    const long long bh = bkv * group + gi;
    const float *qb = q + bh * g.T * D, *dob = dO + bh * g.T * D;
    const float *lb = lse + bh * g.T, *Db = Dv + bh * g.T;
    for (int s = 0; s < g.cp; ++s) {
      const int r = (j + s) % g.cp;
      for (int half = 0; half < 2; ++half) {
        const int kappa = chunk_of(r, half, g.cp);
        const int row0 = 2 * g.c * r + half * g.c;
        for (int u = 0; u < g.c; ++u) {
          const int qp = kappa * g.c + u;
          if (!pair_allowed(qp, kp, g)) continue;
          const int t = row0 + u;
          float qr[V], dor[V];
          load_row<D>(qb + (long long)t * D, lane, qr);
          if (g.rope) rope_row_f32<D>(qr, qp, lane, false, th);
          load_row<D>(dob + (long long)t * D, lane, dor);
          const float p = expf(warp_dot<D>(qr, kr) * scale - lb[t]);
          const float ds = p * (warp_dot<D>(dor, vr) - Db[t]);
#pragma unroll
          for (int e = 0; e < V; ++e) {
            adv[e] = fmaf(p, dor[e], adv[e]);
            adk[e] = fmaf(ds, qr[e], adk[e]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int e = 0; e < V; ++e) adk[e] *= scale;
  if (g.rope) rope_row_f32<D>(adk, kp, lane, true, th);
#pragma unroll
  for (int e = 0; e < V; ++e) {
    dk[row * D + lane + 32 * e] = adk[e];
    dv[row * D + lane + 32 * e] = adv[e];
  }
}

cpattn_status launch_fwd_f32(const float *q, const float *k, const float *v, float *o, float *lse,
                             const Geometry &g, cudaStream_t s) {
  const long long rows = (long long)g.B * g.H * g.T;
  const unsigned blocks = (unsigned)((rows + 3) / 4);
  RopeTheta th;
  make_rope_theta(g.d, &th, g.rope_cfg);
  if (g.d == 128) fwd_f32_kernel<128><<<blocks, 128, 0, s>>>(q, k, v, o, lse, g, th);
  else fwd_f32_kernel<64><<<blocks, 128, 0, s>>>(q, k, v, o, lse, g, th);
  return check_launch("fp32 forward kernel");
}

cpattn_status launch_bwd_f32(const float *q, const float *k, const float *v, const float *o,
                             const float *lse, const float *dO, float *dq, float *dk, float *dv,
                             float *D, const Geometry &g, cudaStream_t s) {
  (void)o;
  const long long rows = (long long)g.B * g.H * g.T;
  const unsigned blocks = (unsigned)((rows + 3) / 4);
  const unsigned kv_blocks = (unsigned)(((long long)g.B * g.Hkv * g.T + 3) / 4);
  RopeTheta th;
  make_rope_theta(g.d, &th, g.rope_cfg);
  trace_record(2, s);
  if (g.d == 128) bwd_dkdv_f32_kernel<128><<<kv_blocks, 128, 0, s>>>(q, k, v, lse, dO, D, dk, dv, g, th);
  else bwd_dkdv_f32_kernel<64><<<kv_blocks, 128, 0, s>>>(q, k, v, lse, dO, D, dk, dv, g, th);
  trace_record(3, s);
  trace_record(4, s);
  if (g.d == 128) bwd_dq_f32_kernel<128><<<blocks, 128, 0, s>>>(q, k, v, lse, dO, D, dq, g, th);
  else bwd_dq_f32_kernel<64><<<blocks, 128, 0, s>>>(q, k, v, lse, dO, D, dq, g, th);
  trace_record(5, s);
  return check_launch("fp32 backward kernels");
}

}  // namespace cpattn
