// Blackwell (sm_103a) building blocks written as inline PTX: mbarriers with
// bounded waits, TMA tile loads, tensor-memory allocation and access, and
// tcgen05.mma with shared-memory descriptors for 128-byte-swizzled tiles.
//
// Tile convention used by every tensor-core kernel here. A tile of R rows by
// D bf16 columns (D = 64 or 128) lives in shared memory as D/64 column blocks;
// block b holds columns [64b, 64b+64) of all R rows, 128 bytes per row, in the
// 128-byte swizzle that TMA writes (16-byte chunk index XOR row % 8), and
// each block starts on a 1024-byte boundary. Such a tile is
//  * a K-major operand when its columns are the contraction dimension
//    (Q, K as used in Q K^T): 8-row groups are 1024 bytes apart (SBO); a
//    16-column k-step moves 32 bytes inside the swizzle row or to the next
//    column block;
//  * an MN-major operand when its rows are the contraction dimension (V in
//    P V, dO in P^T dO, Q in dS^T Q, K in dS K): 8-row groups are 1024 bytes
//    apart (SBO), column blocks R*128 bytes apart (LBO), and a 16-row k-step
//    moves 2048 bytes.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "device_common.cuh"

namespace cpattn {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier ---
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
// try_wait may suspend the thread while the phase is incomplete, for a time
// the hardware chooses. Measured on the 32k step: with no suspend-time hint
// every attention kernel is 3-4% faster than with a hint of 20, 100 or 1000 ns
// (the waiting thread resumes sooner once the phase completes); a test_wait
// spin measured slower still (the spinning warp takes issue slots from the
// softmax warps on its sub-partition).
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Shared state for bounded waits: a CTA-wide abort flag in shared memory and
// the device error flag. A wait that has not completed after limit_ns
// (kWaitLimitNs in every attention kernel),
// or that sees another role abort, records the failure and returns false; its
// caller then leaves its loop and the kernel runs its teardown.
struct WaitCtx {
  volatile int *abort;              // shared memory
  int *err;                         // global memory
  uint64_t limit_ns = kWaitLimitNs;
};

static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, WaitCtx w) {
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 256; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*w.abort) return false;
    if (globaltimer_ns() - t0 > w.limit_ns) {
      *w.abort = 1;
      if (w.err) atomicOr(w.err, ERR_FLAG_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, WaitCtx w) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, w);
}

// ---------------------------------------------------------------------- TMA ---
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled load of box {64, rows, 1} at (x, y, z) into 128B-swizzled smem.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// 3-D tiled store of box {64, rows, 1} from 128B-swizzled smem to (x, y, z)
// (rows past the tensor's extent are not written), as one bulk group.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, uint32_t src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void tma_store_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until the committed stores have read their shared-memory source.
__device__ __forceinline__ void tma_store_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Waits until the committed stores are complete.
__device__ __forceinline__ void tma_store_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Generic-proxy shared-memory writes -> visible to the async proxy (MMA, TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------- TMEM ---
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: lane i of the warp gets row
// (warp%4)*32 + i, columns [col, col+32) of the address's lane quarter.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// tmem_ld32 that also reduces what it loads (sm_103a `tcgen05.ld.red`): m is
// the max of the thread's 32 values (checked on the GB300 against a register
// max for every lane, negative and -inf values included). Like the loaded
// values, m is ready only after tmem_ld_wait().
__device__ __forceinline__ void tmem_ld32_max(uint32_t taddr, uint32_t (&r)[32], float &m) {
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, %32, [%33];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=f"(m)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t *r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------------- MMA ---
// Instruction descriptor, kind::f16 with bf16 A/B and fp32 D.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4)                           // D format: f32
         | (1u << 7)                         // A format: bf16
         | (1u << 10)                        // B format: bf16
         | ((a_mn_major ? 1u : 0u) << 15)    // A major-ness (0 = K-major)
         | ((b_mn_major ? 1u : 0u) << 16)    // B major-ness
         | ((uint32_t)(N >> 3) << 17)        // N / 8
         | ((uint32_t)(M >> 4) << 24);       // M / 16
}

// Shared-memory matrix descriptor with 128-byte swizzling.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;   // fixed field of the tcgen05 descriptor format
  d |= (uint64_t)2 << 61;   // swizzle mode: 128 bytes
  return d;
}

// K-major operand: tile of R rows at `base`, k-step kk (16 columns).
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t base, int R, int kk) {
  const uint32_t addr = base + (uint32_t)(kk >> 2) * (uint32_t)R * 128u + (uint32_t)(kk & 3) * 32u;
  return sdesc_sw128(addr, 16u, 1024u);
}
// MN-major operand: tile of R rows (the contraction dim) at `base`, k-step kk
// (16 rows); N runs over the column blocks, R*128 bytes apart.
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t base, int R, int kk) {
  const uint32_t addr = base + (uint32_t)kk * 2048u;
  return sdesc_sw128(addr, (uint32_t)R * 128u, 1024u);
}

// Descriptor of a K-major / MN-major tile at k-step 0. The start address is
// the descriptor's low 14 bits (address >> 4); every k-step offset used here
// keeps it inside shared memory (< 256 KB), so a later k-step's descriptor is
// the base plus a compile-time constant (no carry out of the field).
__device__ __forceinline__ uint64_t kdesc0(uint32_t base) { return sdesc_sw128(base, 16u, 1024u); }
__device__ __forceinline__ uint64_t mndesc0(uint32_t base, int R) { return sdesc_sw128(base, (uint32_t)R * 128u, 1024u); }
__host__ __device__ constexpr uint64_t koff(int R, int kk) {
  return (uint64_t)((((kk >> 2) * R * 128) + (kk & 3) * 32) >> 4);
}
__host__ __device__ constexpr uint64_t mnoff(int kk) { return (uint64_t)((kk * 2048) >> 4); }

// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]; A is M lanes x K bf16, two per 32-bit column.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` when all previously issued tcgen05 ops of this thread finish.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// Warp-wide forms: every lane of a converged warp executes the instruction
// with the same (warp-uniform) operands, and elect.sync picks the one lane
// that issues it. Keeping descriptors warp-uniform lets them live in uniform
// registers instead of being moved there for each MMA of a one-lane branch.
__device__ __forceinline__ void mma_ss_w(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit_w(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}

// Shared-memory load by 32-bit shared address (keeps the access on the
// shared-memory path even when the generic pointer's space is not known).
__device__ __forceinline__ float4 lds_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
  return v;
}

// 2^x with the MUFU.EX2 unit (flush-to-zero; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed fp32 pairs (sm_100+ f32x2 arithmetic: one instruction for two lanes
// of work) and the three-input max.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unf2(uint64_t v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// bf16x2 of a packed pair (round to nearest even; lo in bits 0..15).
__device__ __forceinline__ uint32_t pack_bf16x2_2(uint64_t v) {
  float lo, hi;
  unf2(v, lo, hi);
  return pack_bf16x2(lo, hi);
}

__device__ __forceinline__ uint64_t fsub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// ------------------------------------------------------------- CTA pairs ---
// Two-SM (cta_group::2) forms for kernels launched in clusters of two CTAs.
// The pair's even CTA (cluster rank 0, the leader) issues every MMA; an MMA of
// M = 256 takes rows 0..127 of its A operand and of its result from the
// leader's shared/tensor memory and rows 128..255 from the peer's, at the same
// addresses, and the N columns of B as two halves: 0..N/2-1 from the leader's
// shared memory, N/2..N-1 from the peer's, both at the descriptor's address.
// Tensor memory is allocated by one warp in each CTA of the pair together.

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %cluster_ctarank;" : "=r"(r));
  return r;
}
// Whole-cluster barrier (every thread of both CTAs), release / acquire at cluster scope.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The two halves of cluster_sync_all, for work that needs no ordering with
// the barrier (loads into registers) to run between them.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Shared-memory address of the same variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Arrive on an mbarrier anywhere in the cluster (address from mapa_shared).
// The arrive keeps the default (CTA-scope release) semantics: the hand-offs
// between the pair's softmax warps and its MMA issuer order tensor-memory
// accesses, which the tcgen05 fences around the arrive and the wait already
// do; a release at cluster scope made every arrive a cluster-wide memory
// barrier (measured: the paired dQ kernel took 1.74x as long).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}
// 3-D tiled TMA load into this CTA's shared memory whose completion is
// counted on an mbarrier of either CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap *map, uint32_t cluster_bar,
                                                 int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 "
      "[%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(cluster_bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Warp-wide (elect.sync) pair MMAs and a commit that arrives on the mbarrier
// at the same address in both CTAs of the pair.
__device__ __forceinline__ void mma2_ss_w(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma2_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma2_commit_both_w(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}"
      ::"r"(bar), "h"((uint16_t)3)
      : "memory");
}

// ------------------------------------------------------ swizzled smem access ---
// Byte offset of element (row, col) in a 128B-swizzled tile of R rows.
__device__ __forceinline__ uint32_t sw128_offset(int row, int col, int R) {
  const int blk = col >> 6, cc = col & 63;
  return (uint32_t)blk * (uint32_t)R * 128u + (uint32_t)row * 128u +
         ((uint32_t)((cc >> 3) ^ (row & 7)) << 4) + ((uint32_t)(cc & 7) << 1);
}

// Rotate (rotate-half RoPE) the 128 rows of a swizzled bf16 tile in place;
// row i sits at natural position pos0 + i. Called by
// the four warps of a warpgroup (wid 0..3). A lane owns frequency pair
// (f, f+1) of one row at a time and walks rows with a fixed stride; its
// cos/sin are seeded once with rope_sincos and advanced by an exact
// angle-addition step (error grows by ~1 ulp per step, <= 32 steps).
template <int D>
__device__ __forceinline__ void rope_tile(uint8_t *tile, int pos0, int wid, int lane,
                                          const RopeTheta &th) {
  constexpr int LPR = D / 4;        // lanes per row (each lane: 2 frequencies)
  constexpr int RPI = 32 / LPR;     // rows per warp step
  constexpr int STEP = 4 * RPI;     // row stride of one lane
  const int sub = lane / LPR, f = 2 * (lane % LPR);
  const int row0 = wid * RPI + sub;
  float c0, s0, c1, s1, cd0, sd0, cd1, sd1;
  rope_sincos(pos0 + row0, th.hi[f], th.lo[f], s0, c0);
  rope_sincos(pos0 + row0, th.hi[f + 1], th.lo[f + 1], s1, c1);
  c0 *= th.mscale; s0 *= th.mscale; c1 *= th.mscale; s1 *= th.mscale;   // m R (temperature, YaRN)
  rope_sincos(STEP, th.hi[f], th.lo[f], sd0, cd0);
  rope_sincos(STEP, th.hi[f + 1], th.lo[f + 1], sd1, cd1);
#pragma unroll 4
  for (int row = row0; row < 128; row += STEP) {
    uint32_t *pa = reinterpret_cast<uint32_t *>(tile + sw128_offset(row, f, 128));
    uint32_t *pb = reinterpret_cast<uint32_t *>(tile + sw128_offset(row, f + D / 2, 128));
    const uint32_t a = *pa, b = *pb;
    const float x0 = bf16lo_to_f32(a), x1 = bf16hi_to_f32(a);
    const float y0 = bf16lo_to_f32(b), y1 = bf16hi_to_f32(b);
    *pa = pack_bf16x2(fmaf(x0, c0, -y0 * s0), fmaf(x1, c1, -y1 * s1));
    *pb = pack_bf16x2(fmaf(y0, c0, x0 * s0), fmaf(y1, c1, x1 * s1));
    const float nc0 = fmaf(c0, cd0, -s0 * sd0), ns0 = fmaf(s0, cd0, c0 * sd0);
    const float nc1 = fmaf(c1, cd1, -s1 * sd1), ns1 = fmaf(s1, cd1, c1 * sd1);
    c0 = nc0; s0 = ns0; c1 = nc1; s1 = ns1;
  }
}

// Rotate-half RoPE of a 128-row, 128B-swizzled bf16 tile in place (row i at
// natural position pos0 + i) by NT threads (u = 0..NT-1), 16 bytes at a time.
// Thread u owns one 16-byte chunk c of the first half of every row it visits
// and the matching chunk of the second half: the eight pairs (i, i + D/2),
// i = 8c..8c+7, which sit at the same swizzled column in both halves for
// D = 128 (two 64-column blocks) and four chunks apart for D = 64. It visits
// rows r0, r0 + RS, ... below 128 (RS = NT / chunks per row, a multiple of 8,
// so the swizzle phase r & 7 is fixed); a warp's 32 lanes cover four (D = 128)
// or eight (D = 64) whole consecutive rows per step, which keeps the 16-byte
// accesses free of bank conflicts. cos/sin are seeded per tile at row r0 and
// advanced row to row by the exact angle-addition step of RS * theta_i.
template <int D, int NT>
struct RopeRows {
  static constexpr int kRows = 128;               // rows of a tile
  static constexpr int CPR = (D == 128) ? 8 : 4;  // chunks per row owned (first half)
  static constexpr int RS = NT / CPR;             // row stride of one thread
  static constexpr int NI = kRows / RS;           // rows per thread per tile
  static_assert(NT % (CPR * 8) == 0 && NT % 32 == 0, "row stride must keep the swizzle phase");
  static_assert(kRows % RS == 0, "every thread visits the same number of rows");
  uint32_t xoff, yoff;                            // byte offsets in row r0
  int r0;
  float th_hi[8], th_lo[8];
  float m;                                        // attention temperature (YaRN), 1 otherwise
  uint64_t cd[4], sd[4];                          // cos, sin of RS * theta, frequency pairs

  __device__ __forceinline__ void init(int u, const RopeTheta &th) {
    const int c = u % CPR;
    r0 = u / CPR;
    m = th.mscale;
    const uint32_t sw = (uint32_t)(r0 & 7);
    xoff = (uint32_t)r0 * 128u + (((uint32_t)c ^ sw) << 4);
    yoff = (D == 128) ? (uint32_t)kRows * 128u + xoff : (uint32_t)r0 * 128u + ((((uint32_t)c + 4u) ^ sw) << 4);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      th_hi[e] = th.hi[8 * c + e];
      th_lo[e] = th.lo[8 * c + e];
    }
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      float s0, c0, s1, c1;
      rope_sincos(RS, th_hi[2 * w], th_lo[2 * w], s0, c0);
      rope_sincos(RS, th_hi[2 * w + 1], th_lo[2 * w + 1], s1, c1);
      cd[w] = f2(c0, c1);
      sd[w] = f2(s0, s1);
    }
  }

  __device__ __forceinline__ void rotate(uint8_t *tile, int pos0) const {
    uint64_t C[4], S[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      float s0, c0, s1, c1;
      rope_sincos_fast(pos0 + r0, th_hi[2 * w], th_lo[2 * w], s0, c0);
      rope_sincos_fast(pos0 + r0, th_hi[2 * w + 1], th_lo[2 * w + 1], s1, c1);
      C[w] = f2(m * c0, m * c1);   // m R: the angle step below keeps the factor
      S[w] = f2(m * s0, m * s1);
    }
#pragma unroll 2
    for (int j = 0; j < NI; ++j) {
      uint4 *px = reinterpret_cast<uint4 *>(tile + xoff + (uint32_t)j * (RS * 128));
      uint4 *py = reinterpret_cast<uint4 *>(tile + yoff + (uint32_t)j * (RS * 128));
      const uint4 xv = *px, yv = *py;
      const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, yw[4] = {yv.x, yv.y, yv.z, yv.w};
      uint32_t ox[4], oy[4];
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint64_t X = f2(bf16lo_to_f32(xw[w]), bf16hi_to_f32(xw[w]));
        const uint64_t Y = f2(bf16lo_to_f32(yw[w]), bf16hi_to_f32(yw[w]));
        ox[w] = pack_bf16x2_2(fsub2(fmul2(X, C[w]), fmul2(Y, S[w])));   // x cos - y sin
        oy[w] = pack_bf16x2_2(ffma2(X, S[w], fmul2(Y, C[w])));          // y cos + x sin
      }
      *px = make_uint4(ox[0], ox[1], ox[2], ox[3]);
      *py = make_uint4(oy[0], oy[1], oy[2], oy[3]);
#pragma unroll
      for (int w = 0; w < 4; ++w) {   // advance to row + RS
        const uint64_t nc = fsub2(fmul2(C[w], cd[w]), fmul2(S[w], sd[w]));
        S[w] = ffma2(C[w], sd[w], fmul2(S[w], cd[w]));
        C[w] = nc;
      }
    }
  }
};

}  // namespace tc
}  // namespace cpattn
