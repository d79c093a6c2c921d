/*
 * cpattn -- HeadTail-balanced ring (context-parallel) causal attention on one
 * GB300 (sm_103a). C ABI: plain pointers, sizes and a CUDA stream; no C++ or
 * framework types cross this boundary.
 *
 * What it computes. A sequence of T tokens is cut into 2*cp chunks of
 * c = T/(2*cp); virtual rank r owns chunk r (head) and chunk 2*cp-1-r (tail)
 * ("BluScriptCP -- docs/Claude Logs.md", entries 2026-05-16 and 2026-06-29;
 * "fix(cp): preserve gradients when sharding VLM inputs - #2931", head-tail
 * chunk pairing). Each rank's queries attend, ring step by ring step, to the
 * K/V chunks of rank j = (r - s) mod cp under the global causal mask
 * (Claude Logs, 2026-04-20: T_q/T_k/q_offset/k_offset masking; 2026-06-17:
 * the three step shapes), and the per-step partials are merged by the
 * log-sum-exp rule (Claude Logs, 2026-03-20: SDPAMerger). The backward
 * recomputes P from the saved LSE and accumulates dQ/dK/dV over all ring
 * steps (Claude Logs, 2026-03-24: D correction; 2026-06-22: dK/dV travel
 * with K/V and return to their owner). Here the ring's K/V rotation is a loop
 * over resident chunks, so the result equals single-pass causal attention.
 *
 * Conventions shared by every call:
 *  - Tensors are dense, contiguous, row-major. [B,H,T,d] tensors passed to
 *    cpattn_fwd / cpattn_bwd are in HeadTail-sharded token order (the output
 *    order of cpattn_shard); LSE and D are [B,H,T] in the same order.
 *  - Device pointers must be 16-byte aligned and must not alias unless
 *    stated. The caller owns every buffer; the library allocates nothing on
 *    the device and keeps no per-call state.
 *  - All work is enqueued on `stream` and is asynchronous. The return value
 *    reports host-detectable errors (arguments, shapes, launch failures). A
 *    device-side error (a bounded wait that timed out) is recorded in a
 *    per-device flag and reported by the next cpattn_sync_status().
 *  - No call aborts, exits or traps; on error nothing is enqueued (or the
 *    launch failed) and cpattn_last_error() describes it.
 *  - softmax scale = 1/sqrt(d). LSE is the natural log of the sum of
 *    exponentials of the scaled scores. RoPE (rope = 1) is the rotate-half
 *    pairing (i, i + d/2) with theta_i = 10000^(-2i/d), applied to q and k at
 *    each token's global (natural) position.
 *  - T_valid <= T real tokens: keys at natural positions >= T_valid (tail
 *    padding, "fix(cp) ... #2931": pad to a multiple of 2*cp at the end) are
 *    masked out.
 */
#ifndef CPATTN_H
#define CPATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *cpattn_stream_t;

typedef enum {
  CPATTN_OK = 0,
  CPATTN_ERR_ARG = 1,         /* null pointer, bad enum, aliasing buffers      */
  CPATTN_ERR_SHAPE = 2,       /* T % (2*cp) != 0, T_valid out of range, d ...  */
  CPATTN_ERR_DTYPE = 3,       /* dtype not supported by this call              */
  CPATTN_ERR_ALIGN = 4,       /* pointer not 16-byte aligned                   */
  CPATTN_ERR_CUDA = 5,        /* a CUDA runtime call or kernel launch failed   */
  CPATTN_ERR_TIMEOUT = 6,     /* a kernel's bounded wait expired (device flag) */
  CPATTN_ERR_UNSUPPORTED = 7  /* valid request the library does not implement  */
} cpattn_status;

typedef enum { CPATTN_F32 = 0, CPATTN_BF16 = 1 } cpattn_dtype;

/* ---------------------------------------------------------------- shard ---
 * HeadTail permutation along T of a [B,H,T,d] tensor (Claude Logs,
 * 2026-05-16, chunk-level HeadTail; 2026-06-29, worked example {0,1,6,7} for
 * N=2). cpattn_shard writes dst[b,h,sigma(t),:] = src[b,h,t,:] with
 *   kappa = t / c, o = t % c,
 *   sigma(t) = 2c*kappa + o            if kappa < cp,
 *            = 2c*(2cp-1-kappa) + c + o otherwise.
 * cpattn_unshard is its inverse. Out of place: src and dst must not overlap.
 * dt selects the element size (4 or 2 bytes); d*elt must be a multiple of 16.
 * Errors: CPATTN_ERR_SHAPE if T % (2*cp) != 0 or any size < 1. */
cpattn_status cpattn_shard(const void *src, void *dst, int B, int H, int T, int d, int cp,
                           cpattn_dtype dt, cpattn_stream_t stream);
cpattn_status cpattn_unshard(const void *src, void *dst, int B, int H, int T, int d, int cp,
                             cpattn_dtype dt, cpattn_stream_t stream);

/* HeadTail shard fused with RoPE, and its adjoint fused with unshard. The
 * rotation (rotate-half pairs (i, i + d/2), theta_i = 10000^(-2i/d)) uses each
 * token's natural position t, the global position the pages require under
 * HeadTail (Claude Logs, 2026-05-07 and 2026-06-05: local positions were a
 * bug; 2026-06-29: cos/sin follow the same permutation as the tokens):
 *   cpattn_shard_rope   : dst[b,h,sigma(t),:] = R(t)   src[b,h,t,:]
 *   cpattn_unshard_rope : dst[b,h,t,:]        = R(t)^T src[b,h,sigma(t),:]
 * With q' = shard_rope(q), k' = shard_rope(k), cpattn_fwd/cpattn_bwd called
 * with rope = 0 on q', k' give the same O and LSE as rope = 1 on the plain
 * shards, and unshard_rope of their dq', dk' gives dq, dk: RoPE then runs in
 * the passes that already read and write q, k and their gradients, and the
 * attention kernels rotate nothing. Same rules as cpattn_shard; d in {64, 128}. */
cpattn_status cpattn_shard_rope(const void *src, void *dst, int B, int H, int T, int d, int cp,
                                cpattn_dtype dt, cpattn_stream_t stream);
cpattn_status cpattn_unshard_rope(const void *src, void *dst, int B, int H, int T, int d, int cp,
                                  cpattn_dtype dt, cpattn_stream_t stream);

/* ---------------------------------------------------- YaRN-scaled RoPE ---
 * cpattn_shard_rope / cpattn_unshard_rope with a RoPE configuration: the
 * YaRN context extension (Claude Logs, 2026-07-09: NTK-by-parts frequency
 * blend over a dimension-index ramp, and an attention temperature multiplied
 * into cos and sin; HANDOFF_H200_32K: the 32k run uses factor 2 over an
 * original 16384 positions). With s = factor and L = original_max_position,
 * pair i of d/2 has theta_i = base^(-2i/d); pair i turns L theta_i / (2 pi)
 * times over L, and the pair index where that count equals n is
 * x(n) = d ln(L / (2 pi n)) / (2 ln base). With lo = max(floor(x(beta_fast)), 0),
 * hi = min(ceil(x(beta_slow)), d - 1) and w_i = clamp((i - lo) / (hi - lo), 0, 1),
 * the rotation uses theta'_i = (1 - w_i) theta_i + w_i theta_i / s and
 * multiplies cos and sin by m (attention_factor, or 0.1 ln(s) + 1 when that
 * is <= 0; 1 when s = 1). The forward stores m R(p) x, the adjoint m R(p)^T g.
 * factor = 1 with base 10000 is exactly cpattn_shard_rope / cpattn_unshard_rope.
 * cfg is read during the call only (host memory, caller-owned). Invalid
 * values (NULL, base <= 1, factor < 1, non-finite fields; for factor > 1
 * original_max_position < 1 or not 0 < beta_slow < beta_fast) give
 * CPATTN_ERR_ARG. Arguments and layouts otherwise as cpattn_shard_rope. */
typedef struct cpattn_rope_cfg {
  double base;                /* 10000 for the standard rotation */
  double factor;              /* YaRN s >= 1; 1 = no extension */
  int original_max_position;  /* L: the length the weights were trained at */
  double beta_fast;           /* usually 32 */
  double beta_slow;           /* usually 1 */
  double attention_factor;    /* m; <= 0 selects 0.1 ln(s) + 1 */
} cpattn_rope_cfg;
cpattn_status cpattn_shard_rope_cfg(const void *src, void *dst, int B, int H, int T, int d, int cp,
                                    cpattn_dtype dt, const cpattn_rope_cfg *cfg,
                                    cpattn_stream_t stream);
cpattn_status cpattn_unshard_rope_cfg(const void *src, void *dst, int B, int H, int T, int d, int cp,
                                      cpattn_dtype dt, const cpattn_rope_cfg *cfg,
                                      cpattn_stream_t stream);

/* Host-only: idx_host[t] = sigma(t) for t in [0, T) (int32, caller-owned,
 * T entries). Launches nothing. */
cpattn_status cpattn_shard_index(int T, int cp, int32_t *idx_host);

/* -------------------------------------------- several tensors at once ---
 * The HeadTail shard (cpattn_shard_batch) or unshard (cpattn_unshard_batch)
 * of n tensors (1 <= n <= 8) in one launch, e.g. q, k, v, dO before the
 * attention and o, dq, dk, dv after it ("Claude Logs", 2026-05-16: the chunk-
 * level HeadTail permutation as one GPU pass):
 *   src[i], dst[i] : device [B, heads[i], T, d] (natural order in, sharded
 *                    out for shard; the reverse for unshard), out of place
 *   rope[i] = 1    : also rotate at the global position, as cpattn_shard_rope
 *                    / cpattn_unshard_rope (R on the way in, R^T on the way
 *                    out; cfg as in cpattn_shard_rope_cfg, NULL = standard)
 * src, dst, heads and rope are host arrays of n entries. The result equals
 * the n single calls. Errors as cpattn_shard / cpattn_shard_rope; a
 * destination that overlaps any other buffer of the batch is CPATTN_ERR_ARG;
 * d must be 64 or 128. */
cpattn_status cpattn_shard_batch(const void *const *src, void *const *dst, const int *heads, const int *rope, int n,
                                 int B, int T, int d, int cp, const cpattn_rope_cfg *cfg, cpattn_dtype dt,
                                 cpattn_stream_t stream);
cpattn_status cpattn_unshard_batch(const void *const *src, void *const *dst, const int *heads, const int *rope, int n,
                                   int B, int T, int d, int cp, const cpattn_rope_cfg *cfg, cpattn_dtype dt,
                                   cpattn_stream_t stream);

/* ------------------------------------------------------------- forward ---
 * Ring attention forward (Claude Logs, 2026-03-20 ring + SDPAMerger;
 * 2026-04-20 global causal masking; 2026-06-17 step shapes).
 *   q, k, v : [B,H,T,d] sharded, dtype dt (read only)
 *   o       : [B,H,T,d] sharded, dtype dt (written)
 *   lse     : [B,H,T]   sharded, fp32     (written)
 * d in {64, 128}. causal in {0,1}, rope in {0,1}, 1 <= T_valid <= T.
 * dt = CPATTN_BF16 runs the tensor-core (tcgen05) kernel; dt = CPATTN_F32 runs
 * the exact-fp32 CUDA-core kernel (a correctness path, not a fast one). */
cpattn_status cpattn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                         int B, int T, int T_valid, int H, int d, int cp, int causal, int rope,
                         cpattn_dtype dt, cpattn_stream_t stream);

/* ------------------------------------------------------------ backward ---
 * Gradient of sum(dO * O) with respect to the q, k, v given to cpattn_fwd
 * (before RoPE), from that call's o and lse (Claude Logs, 2026-03-24 D
 * correction; 2026-06-22 dK/dV accumulate over every ring step; 2026-04-20).
 * With P = exp(S - LSE): dV = P^T dO; D = rowsum(dO * O); dS = P*(dO V^T - D);
 * dQ = scale * dS K; dK = scale * dS^T Q (then R^T when rope = 1).
 *   q, k, v, o, dO : [B,H,T,d] sharded, dtype dt (read only)
 *   lse            : [B,H,T] fp32 (read only, from cpattn_fwd)
 *   dq, dk, dv     : [B,H,T,d] sharded, dtype dt (written; fp32 accumulation)
 *   workspace      : device scratch of at least cpattn_bwd_workspace_bytes()
 *                    bytes, 16-byte aligned, caller-owned; holds D (fp32).
 * dQ is accumulated without atomics: one kernel owns each dQ tile (query
 * stationary) and another each dK/dV tile (key stationary). */
size_t cpattn_bwd_workspace_bytes(int B, int T, int H, int d);
cpattn_status cpattn_bwd(const void *q, const void *k, const void *v, const void *o,
                         const float *lse, const void *dO, void *dq, void *dk, void *dv,
                         void *workspace, int B, int T, int T_valid, int H, int d, int cp,
                         int causal, int rope, cpattn_dtype dt, cpattn_stream_t stream);

/* ------------------------------------------ grouped K/V heads (GQA/MQA) ---
 * cpattn_fwd / cpattn_bwd with H query heads sharing H_kv K/V heads: query
 * head h attends with K/V head h / (H / H_kv), the repeat-interleave grouping
 * (Claude Logs, 2026-06-29: keep GQA-grouped K/V in the ring; 2026-07-01:
 * GQA/MQA as a local broadcast of K/V heads whose backward is a group sum).
 * The gradient of a K/V head is the sum of what its H / H_kv query heads give
 * it. H_kv = H is cpattn_fwd / cpattn_bwd; H_kv = 1 is multi-query attention.
 *   q, o, dO, dq : [B,H,T,d]    sharded, dtype dt
 *   k, v, dk, dv : [B,H_kv,T,d] sharded, dtype dt
 *   lse          : [B,H,T] fp32; workspace as for cpattn_bwd (B*H*T rows)
 * H_kv must divide H, else CPATTN_ERR_SHAPE. Everything else (layouts,
 * validation, ownership, asynchrony, errors) is as for cpattn_fwd/cpattn_bwd. */
cpattn_status cpattn_fwd_gqa(const void *q, const void *k, const void *v, void *o, float *lse,
                             int B, int T, int T_valid, int H, int H_kv, int d, int cp, int causal,
                             int rope, cpattn_dtype dt, cpattn_stream_t stream);
cpattn_status cpattn_bwd_gqa(const void *q, const void *k, const void *v, const void *o,
                             const float *lse, const void *dO, void *dq, void *dk, void *dv,
                             void *workspace, int B, int T, int T_valid, int H, int H_kv, int d,
                             int cp, int causal, int rope, cpattn_dtype dt, cpattn_stream_t stream);

/* ------------------------------------- in-kernel RoPE with a configuration ---
 * cpattn_fwd_gqa / cpattn_bwd_gqa with rope = 1 and the rotation of cfg
 * (standard base, or YaRN: NTK-by-parts frequencies and the attention
 * temperature m; Claude Logs, 2026-07-09) instead of the standard one: the
 * kernels use m R(p) q, m R(p) k, and the gradients leave through (m R(p))^T,
 * so the result equals cpattn_shard_rope_cfg followed by the rope = 0 call.
 * cfg (host, read during the call only) must be valid for
 * cpattn_shard_rope_cfg, else CPATTN_ERR_ARG; NULL is CPATTN_ERR_ARG. */
cpattn_status cpattn_fwd_rope_cfg(const void *q, const void *k, const void *v, void *o, float *lse,
                                  int B, int T, int T_valid, int H, int H_kv, int d, int cp,
                                  int causal, const cpattn_rope_cfg *cfg, cpattn_dtype dt,
                                  cpattn_stream_t stream);
cpattn_status cpattn_bwd_rope_cfg(const void *q, const void *k, const void *v, const void *o,
                                  const float *lse, const void *dO, void *dq, void *dk, void *dv,
                                  void *workspace, int B, int T, int T_valid, int H, int H_kv, int d,
                                  int cp, int causal, const cpattn_rope_cfg *cfg, cpattn_dtype dt,
                                  cpattn_stream_t stream);

/* ------------------------------------------ packed documents (varlen) ---
 * Several documents packed along T (the THD layout of "fix(cp): preserve
 * gradients when sharding VLM inputs - #2931"; Claude Logs, 2026-07-16:
 * training on length-bucketed documents, HANDOFF_H200_32K: 16k-32k
 * documents in a 32k window). A query attends only to keys of its own
 * document, causally when causal = 1; positions past the last document are
 * padding and attend to nothing (O = 0, LSE = -inf, zero gradients).
 *
 * cpattn_doc_bounds turns cu_seqlens (device int32 [n_docs + 1],
 * 0 = cu[0] <= cu[1] <= ... <= cu[n_docs] <= T; document i holds natural
 * positions [cu[i], cu[i+1])) into per-position bounds: doc_lo[p], doc_hi[p]
 * (device int32 [T] each, natural order, caller-owned, 16-byte aligned) are
 * the start and end of p's document, and both equal cu[n_docs] for padding.
 * The list is checked on the device: a bad one makes the next
 * cpattn_sync_status return CPATTN_ERR_ARG (the bounds then stay inside
 * [0, T] but mean nothing). One layout serves every batch row and head.
 *
 * cpattn_fwd_varlen / cpattn_bwd_varlen are cpattn_fwd_gqa / cpattn_bwd_gqa
 * with that same-document condition, rope = 0 (rotate q, k with
 * cpattn_shard_rope: scores inside one document depend only on position
 * differences, so global positions give the per-document result), and
 * T_valid = cu[n_docs] (any T_valid >= it gives the same result). Any
 * schedule length (the bf16 kernels past 2*cp*ceil(T/(2*cp*128)) = 2048 tiles
 * per CTA are the one-tile ones). doc_lo / doc_hi are read during the kernels
 * only. */
cpattn_status cpattn_doc_bounds(const int32_t *cu_seqlens, int n_docs, int T, int32_t *doc_lo,
                                int32_t *doc_hi, cpattn_stream_t stream);
cpattn_status cpattn_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                                int B, int T, int T_valid, int H, int H_kv, int d, int cp, int causal,
                                const int32_t *doc_lo, const int32_t *doc_hi, cpattn_dtype dt,
                                cpattn_stream_t stream);
cpattn_status cpattn_bwd_varlen(const void *q, const void *k, const void *v, const void *o,
                                const float *lse, const void *dO, void *dq, void *dk, void *dv,
                                void *workspace, int B, int T, int T_valid, int H, int H_kv, int d,
                                int cp, int causal, const int32_t *doc_lo, const int32_t *doc_hi,
                                cpattn_dtype dt, cpattn_stream_t stream);

/* ------------------------------- in-kernel RoPE, rotated once per call ---
 * RoPE at global positions applied by the attention calls themselves (Claude
 * Logs, 2026-05-07, 2026-06-05, 2026-06-29: each token's global position), for
 * one document or packed documents, with the rotation done once: the forward
 * rotates q and k as it streams them and also stores the rotated copies,
 *   q_rot = m R(p) q,  k_rot = m R(p) k   (sharded layout, caller-owned,
 *   16-byte aligned, the sizes of q and k; m = 1 and base 10000 when cfg is
 *   NULL, else the YaRN configuration of cpattn_rope_cfg),
 * and the backward takes those copies in place of q and k, runs the kernels
 * that rotate nothing, and returns the gradients with respect to the
 * UNROTATED q and k (dq = m R(p)^T dQ', dk = m R(p)^T dK' in the kernels'
 * epilogues). The results equal cpattn_fwd_rope_cfg / cpattn_bwd_rope_cfg on
 * the same q, k; the backward does not rotate every streamed tile again.
 *   doc_lo, doc_hi : NULL (one sequence) or the per-position document bounds
 *                    of cpattn_doc_bounds (packed documents; RoPE keeps the
 *                    global positions).
 * Other arguments, layouts and errors as cpattn_fwd_gqa / cpattn_bwd_gqa with
 * rope = 1; q_rot and k_rot must not overlap any other buffer. The backward's
 * workspace is cpattn_bwd_workspace_bytes(B, T, H, d). For bf16 inputs whose
 * tile schedule fits the kernels' tables (2*cp*ceil(T/(2cp)/128) <= 2048) the
 * rotation is fused as described; otherwise (fp32, or longer schedules) the
 * forward rotates q and k in one pass before attending and the backward
 * applies R^T in one pass after it, with the same results. */
cpattn_status cpattn_fwd_rope_save(const void *q, const void *k, const void *v, void *o, float *lse,
                                   void *q_rot, void *k_rot, int B, int T, int T_valid, int H, int H_kv,
                                   int d, int cp, int causal, const int32_t *doc_lo, const int32_t *doc_hi,
                                   const cpattn_rope_cfg *cfg, cpattn_dtype dt, cpattn_stream_t stream);
cpattn_status cpattn_bwd_rotated(const void *q_rot, const void *k_rot, const void *v, const void *o,
                                 const float *lse, const void *dO, void *dq, void *dk, void *dv,
                                 void *workspace, int B, int T, int T_valid, int H, int H_kv, int d,
                                 int cp, int causal, const int32_t *doc_lo, const int32_t *doc_hi,
                                 const cpattn_rope_cfg *cfg, cpattn_dtype dt, cpattn_stream_t stream);

/* ----------------------------------------------- Ulysses all-to-all ---
 * The Ulysses (DeepSpeed) variant of sequence parallelism on P virtual
 * ranks (Claude Logs, 2026-06-30: all-to-all layout swaps [B,H,Tl,D] <->
 * [B,Hl,T,D], contiguous shards, one full attention per rank; 2026-07-01:
 * the K/V all-to-all moves only K/V heads). With Tl = T/P and Hl = H/P:
 *   sequence shards  [P][B][H][Tl][d] -- rank r: tokens [r*Tl, (r+1)*Tl) of every head
 *   head shards      [P][B][Hl][T][d] -- rank s: heads [s*Hl, (s+1)*Hl), all T tokens
 * inverse = 0 maps sequence shards to head shards (rank s receives head
 * block s of every rank's tokens, laid out in rank order); inverse = 1 maps
 * back. The head shards are an ordinary [P*B, Hl, T, d] tensor: run
 * cpattn_fwd / cpattn_bwd (or the _gqa forms, with the K/V all-to-all over
 * H_kv heads) on it with B' = P*B, H' = Hl and cp = 1. cpattn_ulysses_a2a_rope
 * also rotates each row at its natural position r*Tl + t (m R(p) forward,
 * (m R(p))^T with inverse = 1), cfg as for cpattn_shard_rope_cfg (NULL:
 * standard RoPE).
 * Fewer heads than ranks (the K/V all-to-all of grouped heads when H_kv < P;
 * Claude Logs, 2026-07-01: replicate by P / n_kv): with H dividing P, rank s
 * receives head s / (P / H) -- head shards [P][B][1][T][d] -- and inverse = 1
 * is the adjoint: the P / H replicas of a head are summed (in fp32, rounded
 * once), then turned by (m R(p))^T for the _rope form. d must then be 64 or 128.
 * P must divide T, and P must divide H or H divide P, else CPATTN_ERR_SHAPE;
 * otherwise as cpattn_shard / cpattn_shard_rope (out of place, 16-byte
 * aligned, d*elt a multiple of 16). */
cpattn_status cpattn_ulysses_a2a(const void *src, void *dst, int B, int H, int T, int d, int P,
                                 int inverse, cpattn_dtype dt, cpattn_stream_t stream);
cpattn_status cpattn_ulysses_a2a_rope(const void *src, void *dst, int B, int H, int T, int d, int P,
                                      int inverse, const cpattn_rope_cfg *cfg, cpattn_dtype dt,
                                      cpattn_stream_t stream);

/* --------------------------------------------- allocation-free backward ---
 * Not from the pages: an addition of this library for callers that cannot
 * allocate device memory when they call it -- for example a plugin inside a
 * host runtime that owns all device memory and gives its plugins no
 * allocator, or a latency-bound loop that forbids cudaMalloc/cudaFree after
 * start-up because those calls can synchronise the device and fragment its
 * memory. Same computation, arguments, layouts and errors as cpattn_bwd, but
 * without `workspace`: the D = rowsum(dO * O) scratch is a file-scope device
 * array of CPATTN_NOALLOC_MAX_ROWS floats (8 MiB) that every GPU loading the
 * library holds until the process exits. The call itself allocates nothing
 * (no cudaMalloc, cudaFree or allocating library routine).
 *  - B*H*T must be <= CPATTN_NOALLOC_MAX_ROWS, else CPATTN_ERR_SHAPE.
 *  - The first call in each CUDA context (per device; again after a device
 *    reset, and in any non-primary context) resolves the array's device
 *    address (cudaGetSymbolAddress, with that device current) and caches it
 *    for that context; make that first call before any stream capture.
 *  - All calls share the one array. Each call overwrites the rows it uses
 *    before reading them, so nothing stale leaks into a result, but calls
 *    whose kernels overlap on the GPU (different streams, or different host
 *    threads on one device) race on it: serialise them. */
#define CPATTN_NOALLOC_MAX_ROWS (1u << 21)
cpattn_status cpattn_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                                 const float *lse, const void *dO, void *dq, void *dk, void *dv,
                                 int B, int T, int T_valid, int H, int d, int cp, int causal,
                                 int rope, cpattn_dtype dt, cpattn_stream_t stream);

/* --------------------------------------------------------------- merge ---
 * Standalone SDPAMerger (Claude Logs, 2026-03-20; 2026-03-26 on keeping P
 * and LSE consistent; 2026-05-20 partial-merge fix): merges n partial
 * results of the same rows,
 *   L = m + log(sum_i exp(L_i - m)), m = max_i L_i;  O = sum_i exp(L_i - L) O_i,
 * with (O_i = 0, L_i = -inf) the identity and an all-empty row giving (0, -inf).
 *   o_parts, lse_parts : host arrays of n device pointers; O_i fp32 [B,H,T,d],
 *                        L_i fp32 [B,H,T]
 *   o   : [B,H,T,d] dtype dt (written);  lse : [B,H,T] fp32 (written)
 * 1 <= n <= 16. Any row order (the merge is row-wise). */
cpattn_status cpattn_merge(const float *const *o_parts, const float *const *lse_parts, int n,
                           void *o, float *lse, int B, int H, int T, int d, cpattn_dtype dt,
                           cpattn_stream_t stream);

/* ----------------------------------------------------------- diagnostics -- */
/* Thread-local description of the last non-OK status ("" if none). */
const char *cpattn_last_error(void);

/* Synchronises `stream`, then reads and clears the current device's error
 * flag: CPATTN_ERR_TIMEOUT if a kernel's bounded wait expired since the last
 * check, CPATTN_ERR_CUDA if the stream reports an error, else CPATTN_OK. */
cpattn_status cpattn_sync_status(cpattn_stream_t stream);

/* Exercises the bounded-wait path on the device ("Fused Linear LogP TP Test
 * Runbook", hang triage: a stuck wait must surface as an error, not a hang).
 * Enqueues one single-thread kernel that waits, with the same bounded wait
 * every attention kernel uses, on an mbarrier that nothing arrives at; after
 * limit_ns nanoseconds (1e3 <= limit_ns <= 1e9, else CPATTN_ERR_ARG) the wait
 * gives up, sets the device error flag and the kernel returns. Nothing else is
 * in flight, so the context stays usable: the next cpattn_sync_status(stream)
 * returns CPATTN_ERR_TIMEOUT and clears the flag, and later calls work as
 * before. The attention kernels wait up to 2 s. */
cpattn_status cpattn_check_wait_timeout(unsigned long long limit_ns, cpattn_stream_t stream);

/* Tracing hook for timing single kernels inside a longer region. Registers
 * up to 8 caller-created CUDA events (cudaEvent_t handles, borrowed, never
 * destroyed here) that later calls from this host thread record on their
 * stream at kernel boundaries:
 *   cpattn_fwd : events[0] before the attention kernel, events[1] after it;
 *   cpattn_bwd : events[0] before its first kernel, events[1] after the
 *                D = rowsum(dO*O) pass (right after events[0] where the dQ
 *                kernel computes D itself), events[2] / events[3] before /
 *                after the dK/dV kernel, events[4] / events[5] before / after
 *                the dQ kernel (the dQ kernel runs first when it computes D);
 *   cpattn_shard / cpattn_unshard : events[0] before, events[1] after.
 * A call records only the events it has (n large enough). n = 0 or
 * events = NULL turns tracing off. Errors: CPATTN_ERR_ARG if n < 0 or n > 8. */
cpattn_status cpattn_set_trace_events(void *const *events, int n);

/* Library version, e.g. "cpattn 0.1 sm_103a". */
const char *cpattn_version(void);

#ifdef __cplusplus
}
#endif
#endif /* CPATTN_H */
