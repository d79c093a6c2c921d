// Internal declarations shared by the translation units of libcpattn.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "cpattn.h"

namespace cpattn {

// Records a thread-local message and returns `s`.
cpattn_status fail(cpattn_status s, const char *fmt, ...);
// Turns a pending launch error into CPATTN_ERR_CUDA with a message.
cpattn_status check_launch(const char *what);
// Device address of this device's error flag (set by kernels, read and
// cleared by cpattn_sync_status). nullptr if it could not be resolved.
int *device_err_flag();
// Device address of a file-scope __device__ symbol in the current context,
// cached per context; nullptr on failure.
void *symbol_address(const void *symbol);

// Device error codes written to the flag.
enum : int { ERR_FLAG_TIMEOUT = 1, ERR_FLAG_BAD_DOCS = 2 };

// RoPE frequencies theta_i, i < d/2 (standard: 10000^(-2i/d); YaRN: the
// NTK-by-parts blend of theta_i and theta_i / s), split into two floats
// (hi + lo carries ~48 bits) so that pos * theta can be formed without double
// arithmetic on the device, and the factor m that multiplies cos and sin (1
// for the standard rotation).
struct RopeTheta {
  float hi[64];
  float lo[64];
  float mscale;
};
// cfg = nullptr: the standard rotation, base 10000.
void make_rope_theta(int d, RopeTheta *t, const cpattn_rope_cfg *cfg = nullptr);
// Host validation of a RoPE configuration.
cpattn_status check_rope_cfg(const cpattn_rope_cfg *cfg);

// The pipelined attention kernels keep each CTA's tile schedule in a table of
// this many entries; longer schedules (2*cp*ceil(c/128) above it) take the
// one-tile kernels.
constexpr int kTableTiles = 2048;

// HeadTail geometry of one [B,H,T,d] problem.
struct Geometry {
  int B, H, T, T_valid, d, cp, c;  // c = T / (2 cp)
  int causal, rope;
  int Hkv;                         // K/V heads; query head h reads K/V head h / (H / Hkv)
  // Packed documents: per natural position, its document's [doc_lo, doc_hi)
  // (device int32 [T]); nullptr when the sequence is one document.
  const int *doc_lo = nullptr, *doc_hi = nullptr;
  // In-kernel RoPE frequencies and temperature (host pointer read by the
  // launchers; nullptr: the standard rotation, base 10000).
  const cpattn_rope_cfg *rope_cfg = nullptr;
  // Forward with in-kernel RoPE: also store the rotated q and k here (sharded
  // layout, like q and k); nullptr: do not.
  void *q_rot = nullptr, *k_rot = nullptr;
  // Backward on q, k that are already rotated: the kernels rotate nothing and
  // return dq, dk through R^T (rope must be 0 then).
  bool rope_epi = false;
  // Backward: O of the forward when the dQ kernel computes D = rowsum(dO * O)
  // itself (and writes it for the dK/dV kernel, which then runs after it);
  // nullptr when a separate D pass has run.
  const void *o_for_D = nullptr;
};

// ---- launchers (one per kernel family), all asynchronous on `s` ----------
cpattn_status launch_shard(const void *src, void *dst, const Geometry &g, int elt_bytes,
                           bool inverse, cudaStream_t s);
// doc_lo[p], doc_hi[p] for p < T from cu_seqlens[0..n_docs]; raises
// ERR_FLAG_BAD_DOCS on the device flag if cu_seqlens is not a document list.
cpattn_status launch_doc_bounds(const int *cu_seqlens, int n_docs, int T, int *doc_lo, int *doc_hi,
                                cudaStream_t s);
cpattn_status launch_shard_rope(const void *src, void *dst, const Geometry &g, cpattn_dtype dt,
                                bool inverse, const cpattn_rope_cfg *cfg, cudaStream_t s);
// Ulysses all-to-all of P virtual ranks between the stacked sequence shards
// [P][B][H][T/P][d] and the stacked head shards [P][B][H/P][T][d] (inverse:
// back), optionally fused with RoPE (cfg = nullptr and rope = false: none).
cpattn_status launch_ulysses(const void *src, void *dst, const Geometry &g, int P, int elt_bytes,
                             bool inverse, cudaStream_t s);
cpattn_status launch_ulysses_rope(const void *src, void *dst, const Geometry &g, int P, cpattn_dtype dt,
                                  bool inverse, const cpattn_rope_cfg *cfg, cudaStream_t s);
// With fewer heads than ranks (g.H < P, P a multiple of g.H) the forward
// direction replicates each head to P / g.H ranks and the inverse is this
// reduction over the replicas (fp32 sums; RoPE^T after the sum when rope).
cpattn_status launch_ulysses_kv_reduce(const void *src, void *dst, const Geometry &g, int P, cpattn_dtype dt,
                                       bool rope, const cpattn_rope_cfg *cfg, cudaStream_t s);
cpattn_status launch_fwd_f32(const float *q, const float *k, const float *v, float *o,
                             float *lse, const Geometry &g, cudaStream_t s);
cpattn_status launch_bwd_f32(const float *q, const float *k, const float *v, const float *o,
                             const float *lse, const float *dO, float *dq, float *dk, float *dv,
                             float *D, const Geometry &g, cudaStream_t s);
cpattn_status launch_bwd_preprocess(const void *o, const void *dO, float *D, long long rows,
                                    int d, cpattn_dtype dt, cudaStream_t s);
cpattn_status launch_merge(const float *const *o_parts, const float *const *lse_parts, int n,
                           void *o, float *lse, long long rows, int d, cpattn_dtype dt,
                           cudaStream_t s);
cpattn_status launch_fwd_bf16(const void *q, const void *k, const void *v, void *o, float *lse,
                              const Geometry &g, cudaStream_t s);
cpattn_status launch_bwd_bf16(const void *q, const void *k, const void *v, const void *o,
                              const float *lse, const void *dO, void *dq, void *dk, void *dv,
                              float *D, const Geometry &g, cudaStream_t s);

// Pipelined backward (no in-kernel RoPE): dK/dV and dQ kernels of attn_bwd2_tc.cu.
cpattn_status launch_bwd2_bf16(const void *q, const void *k, const void *v, const float *lse,
                               const void *dO, void *dq, void *dk, void *dv, float *D,
                               const Geometry &g, cudaStream_t s);

// One thread waits on an mbarrier that nothing arrives at, with the given
// limit, so that the bounded wait expires (diagnostics.cu).
cpattn_status launch_wait_probe(unsigned long long limit_ns, cudaStream_t s);

// Tracing events registered by cpattn_set_trace_events for this host thread:
// records event i on stream s if one is registered (no-op otherwise).
void trace_record(int i, cudaStream_t s);

// cuTensorMapEncodeTiled, resolved through the runtime's driver entry point.
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();
// 3-D tensor map over a sharded [B*H*2cp chunk slots][c rows][D] bf16 tensor,
// box {64 columns, box_rows rows, 1 slot}, 128-byte swizzle, zero fill past row c.
bool make_tile_map(CUtensorMap *m, const void *base, int D, int c, long long n_slots, int box_rows = 128);

// dQ of the pipelined backward by CTA pairs (two-SM MMAs), d = 128, inputs
// already rotated (attn_dq_pair.cu); D = rowsum(dO * O) precomputed.
cpattn_status launch_dq_pair_bf16(const void *q, const void *k, const void *v, const float *lse,
                                  const void *dO, void *dq, float *D, const Geometry &g,
                                  cudaStream_t s);
// Up to kBatchMax tensors of one [B, H_i, T, d] layout (H_i per tensor)
// through the HeadTail shard (or unshard) in one launch; tensor i with rope[i]
// set is rotated (R in, R^T out) at natural positions.
constexpr int kBatchMax = 8;
struct ShardBatch {
  const void *src[kBatchMax];
  void *dst[kBatchMax];
  int rope[kBatchMax];
  long long first_chunk[kBatchMax];   // first chunk of tensor i in the launch's chunk order
  int n;
  long long n_chunks;
};
cpattn_status launch_shard_batch(const ShardBatch &b, const Geometry &g, cpattn_dtype dt, bool inverse,
                                 const cpattn_rope_cfg *cfg, cudaStream_t s);
// dst = m R(p) src (inverse: m R(p)^T src) for every row of a HeadTail-sharded
// [B*H, T, d] tensor, p the row's natural position (RoPE configuration cfg,
// nullptr: standard); dst may equal src (each element is read, then written,
// by the same thread).
cpattn_status launch_rope_sharded(const void *src, void *dst, const Geometry &g, int heads, cpattn_dtype dt,
                                  bool inverse, const cpattn_rope_cfg *cfg, cudaStream_t s);

}  // namespace cpattn
