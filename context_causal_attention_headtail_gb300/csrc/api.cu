// C-ABI entry points of libcpattn: argument validation and dispatch. Every
// step of the computation runs in the kernels of the other translation units.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "internal.h"

namespace cpattn {

static thread_local char g_msg[512] = "";
static thread_local cudaEvent_t g_trace[8];
static thread_local int g_ntrace = 0;

void trace_record(int i, cudaStream_t s) {
  if (i < g_ntrace && g_trace[i]) cudaEventRecord(g_trace[i], s);
}

cpattn_status fail(cpattn_status s, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return s;
}

cpattn_status check_launch(const char *what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(CPATTN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return CPATTN_OK;
}

// Unique id of the calling thread's current CUDA context (cuCtxGetId: unique
// for the life of the process, so a context created after a device reset, or
// a non-primary context, gets a new one). 0 if it cannot be read.
static unsigned long long current_context_id() {
  typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
  typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);
  static std::once_flag once;
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of a file-scope __device__ symbol in the current context.
// A symbol's name in host code is a host-side stand-in, not a device address,
// so it is resolved with cudaGetSymbolAddress and cached per context (the
// module, and with it the symbol, is loaded again in every new context). When
// the context id cannot be read, the address is resolved on every call.
void *symbol_address(const void *symbol) {
  struct Entry { const void *sym; unsigned long long ctx; void *addr; };
  static std::mutex mu;
  static Entry cache[64];
  static int next = 0;
  std::lock_guard<std::mutex> lock(mu);
  unsigned long long ctx = current_context_id();
  if (ctx)
    for (const Entry &e : cache)
      if (e.sym == symbol && e.ctx == ctx) return e.addr;
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, symbol) != cudaSuccess) return nullptr;
  ctx = current_context_id();        // the runtime has made the device's context current by now
  if (ctx) {
    cache[next] = Entry{symbol, ctx, p};
    next = (next + 1) % 64;
  }
  return p;
}

// One flag per device, written by kernels whose bounded waits expire.
__device__ int g_err_flag;

int *device_err_flag() { return static_cast<int *>(symbol_address(&g_err_flag)); }

void make_rope_theta(int d, RopeTheta *t, const cpattn_rope_cfg *cfg) {
  const double base = cfg ? cfg->base : 10000.0;
  const double s = cfg ? cfg->factor : 1.0;
  // YaRN (NTK-by-parts): pair i keeps theta_i while it turns more than
  // beta_fast times over the trained length L, gets theta_i / s below
  // beta_slow turns, and a linear blend in between, the ramp running over the
  // pair index between the floor and the ceiling of the two crossing indices
  // (a frequency turns n times over L at pair d ln(L / (2 pi n)) / (2 ln base)).
  double ramp_lo = 0.0, ramp_hi = 1.0;
  if (s > 1.0) {
    auto pair_index = [&](double n) {
      return d * log(cfg->original_max_position / (2.0 * M_PI * n)) / (2.0 * log(base));
    };
    ramp_lo = std::max(floor(pair_index(cfg->beta_fast)), 0.0);
    ramp_hi = std::min(ceil(pair_index(cfg->beta_slow)), (double)(d - 1));
    if (ramp_hi == ramp_lo) ramp_hi += 0.001;
  }
  for (int i = 0; i < 64; ++i) {
    double th = (2 * i < d) ? pow(base, -2.0 * i / d) : 0.0;
    if (s > 1.0) {
      const double w = std::min(std::max((i - ramp_lo) / (ramp_hi - ramp_lo), 0.0), 1.0);
      th = th * (1.0 - w) + (th / s) * w;
    }
    float hi = (float)th;
    t->hi[i] = hi;
    t->lo[i] = (float)(th - (double)hi);
  }
  double m = 1.0;
  if (cfg && cfg->attention_factor > 0.0) m = cfg->attention_factor;
  else if (s > 1.0) m = 0.1 * log(s) + 1.0;
  t->mscale = (float)m;
}

cpattn_status check_rope_cfg(const cpattn_rope_cfg *cfg) {
  if (!cfg) return fail(CPATTN_ERR_ARG, "RoPE configuration is NULL");
  if (!std::isfinite(cfg->base) || cfg->base <= 1.0)
    return fail(CPATTN_ERR_ARG, "RoPE base %g must be finite and > 1", cfg->base);
  if (!std::isfinite(cfg->factor) || cfg->factor < 1.0)
    return fail(CPATTN_ERR_ARG, "YaRN factor %g must be finite and >= 1", cfg->factor);
  if (!std::isfinite(cfg->attention_factor))
    return fail(CPATTN_ERR_ARG, "attention_factor must be finite");
  if (cfg->factor > 1.0) {
    if (cfg->original_max_position < 1)
      return fail(CPATTN_ERR_ARG, "original_max_position=%d must be >= 1", cfg->original_max_position);
    if (!(cfg->beta_slow > 0.0) || !(cfg->beta_fast > cfg->beta_slow) || !std::isfinite(cfg->beta_fast))
      return fail(CPATTN_ERR_ARG, "need 0 < beta_slow (%g) < beta_fast (%g)", cfg->beta_slow,
                  cfg->beta_fast);
  }
  return CPATTN_OK;
}

EncodeTiledFn encode_tiled_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace cpattn

using namespace cpattn;

static bool uses_tables(int T, int cp) {
  const long long tpc = ((long long)T / (2 * cp) + 127) / 128;
  return 2LL * cp * tpc <= kTableTiles;
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static cpattn_status check_common(int B, int H, int T, int d, int cp) {
  if (B < 1 || H < 1 || T < 1 || d < 1 || cp < 1)
    return fail(CPATTN_ERR_SHAPE, "sizes must be >= 1 (B=%d H=%d T=%d d=%d cp=%d)", B, H, T, d, cp);
  if (T % (2 * cp) != 0)
    return fail(CPATTN_ERR_SHAPE, "T=%d is not a multiple of 2*cp=%d (pad the tail first)", T, 2 * cp);
  if ((long long)B * H * T > (1LL << 31) - 1)
    return fail(CPATTN_ERR_SHAPE, "B*H*T too large");
  return CPATTN_OK;
}

static cpattn_status check_attn(int B, int T, int T_valid, int H, int d, int cp, int causal,
                                int rope, cpattn_dtype dt) {
  cpattn_status st = check_common(B, H, T, d, cp);
  if (st != CPATTN_OK) return st;
  if (d != 64 && d != 128) return fail(CPATTN_ERR_SHAPE, "d=%d: only 64 and 128 are supported", d);
  if (T_valid < 1 || T_valid > T)
    return fail(CPATTN_ERR_SHAPE, "T_valid=%d must be in [1, T=%d]", T_valid, T);
  if ((causal != 0 && causal != 1) || (rope != 0 && rope != 1))
    return fail(CPATTN_ERR_ARG, "causal and rope must be 0 or 1");
  if (dt != CPATTN_F32 && dt != CPATTN_BF16) return fail(CPATTN_ERR_DTYPE, "unknown dtype %d", (int)dt);
  if (T > (1 << 24)) return fail(CPATTN_ERR_SHAPE, "T=%d exceeds 2^24", T);
  return CPATTN_OK;
}

static Geometry geometry(int B, int H, int T, int T_valid, int d, int cp, int causal, int rope,
                         int Hkv = 0) {
  Geometry g;
  g.B = B; g.H = H; g.T = T; g.T_valid = T_valid; g.d = d; g.cp = cp;
  g.c = T / (2 * cp); g.causal = causal; g.rope = rope;
  g.Hkv = Hkv > 0 ? Hkv : H;
  return g;
}

static cpattn_status check_heads(int H, int H_kv) {
  if (H_kv < 1 || H_kv > H || H % H_kv != 0)
    return fail(CPATTN_ERR_SHAPE, "H_kv=%d must divide H=%d", H_kv, H);
  return CPATTN_OK;
}

static bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
  uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

extern "C" {

const char *cpattn_last_error(void) { return g_msg; }

const char *cpattn_version(void) { return "cpattn 0.1 sm_103a"; }

cpattn_status cpattn_set_trace_events(void *const *events, int n) {
  g_msg[0] = 0;
  if (n < 0 || n > 8) return fail(CPATTN_ERR_ARG, "n=%d must be in [0, 8]", n);
  if (!events) n = 0;
  for (int i = 0; i < 8; ++i) g_trace[i] = i < n ? static_cast<cudaEvent_t>(events[i]) : nullptr;
  g_ntrace = n;
  return CPATTN_OK;
}

cpattn_status cpattn_sync_status(cpattn_stream_t stream) {
  g_msg[0] = 0;
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(CPATTN_ERR_CUDA, "stream: %s", cudaGetErrorString(e));
  int *flag = device_err_flag();
  if (!flag) return fail(CPATTN_ERR_CUDA, "cannot resolve the device error flag");
  int v = 0;
  if (cudaMemcpy(&v, flag, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return fail(CPATTN_ERR_CUDA, "reading the device error flag failed");
  if (v != 0) {
    int zero = 0;
    cudaMemcpy(flag, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (v & ERR_FLAG_TIMEOUT)
      return fail(CPATTN_ERR_TIMEOUT, "a kernel's bounded wait expired (flag=%d)", v);
    if (v & ERR_FLAG_BAD_DOCS)
      return fail(CPATTN_ERR_ARG, "cu_seqlens is not a document list (0 = cu[0] <= ... <= cu[n] <= T)");
    return fail(CPATTN_ERR_CUDA, "device error flag=%d", v);
  }
  return CPATTN_OK;
}

cpattn_status cpattn_check_wait_timeout(unsigned long long limit_ns, cpattn_stream_t stream) {
  g_msg[0] = 0;
  if (limit_ns < 1000ull || limit_ns > 1000000000ull)
    return fail(CPATTN_ERR_ARG, "limit_ns=%llu must be in [1e3, 1e9]", limit_ns);
  return launch_wait_probe(limit_ns, reinterpret_cast<cudaStream_t>(stream));
}

cpattn_status cpattn_shard_index(int T, int cp, int32_t *idx_host) {
  g_msg[0] = 0;
  if (!idx_host) return fail(CPATTN_ERR_ARG, "idx_host is NULL");
  cpattn_status st = check_common(1, 1, T, 1, cp);
  if (st != CPATTN_OK) return st;
  const int c = T / (2 * cp);
  for (int t = 0; t < T; ++t) {
    int kappa = t / c, o = t % c;
    idx_host[t] = kappa < cp ? 2 * c * kappa + o : 2 * c * (2 * cp - 1 - kappa) + c + o;
  }
  return CPATTN_OK;
}

static cpattn_status shard_common(const void *src, void *dst, int B, int H, int T, int d, int cp,
                                  cpattn_dtype dt, cpattn_stream_t stream, bool inverse,
                                  bool rope = false, const cpattn_rope_cfg *cfg = nullptr) {
  g_msg[0] = 0;
  if (!src || !dst) return fail(CPATTN_ERR_ARG, "null pointer");
  if (cfg && check_rope_cfg(cfg) != CPATTN_OK) return CPATTN_ERR_ARG;
  cpattn_status st = check_common(B, H, T, d, cp);
  if (st != CPATTN_OK) return st;
  if (dt != CPATTN_F32 && dt != CPATTN_BF16) return fail(CPATTN_ERR_DTYPE, "unknown dtype %d", (int)dt);
  const int elt = dt == CPATTN_F32 ? 4 : 2;
  if ((d * elt) % 16 != 0) return fail(CPATTN_ERR_ALIGN, "row of d*elt=%d bytes is not a multiple of 16", d * elt);
  if (!aligned16(src) || !aligned16(dst)) return fail(CPATTN_ERR_ALIGN, "pointers must be 16-byte aligned");
  const size_t bytes = (size_t)B * H * T * d * elt;
  if (overlaps(src, bytes, dst, bytes)) return fail(CPATTN_ERR_ARG, "src and dst overlap");
  if (rope && d != 64 && d != 128) return fail(CPATTN_ERR_SHAPE, "d=%d: RoPE needs d in {64, 128}", d);
  if (rope && T > (1 << 24)) return fail(CPATTN_ERR_SHAPE, "T=%d exceeds 2^24", T);
  Geometry g = geometry(B, H, T, T, d, cp, 1, rope ? 1 : 0);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  trace_record(0, s);
  st = rope ? launch_shard_rope(src, dst, g, dt, inverse, cfg, s) : launch_shard(src, dst, g, elt, inverse, s);
  trace_record(1, s);
  return st;
}

cpattn_status cpattn_shard(const void *src, void *dst, int B, int H, int T, int d, int cp,
                           cpattn_dtype dt, cpattn_stream_t stream) {
  return shard_common(src, dst, B, H, T, d, cp, dt, stream, false);
}

cpattn_status cpattn_unshard(const void *src, void *dst, int B, int H, int T, int d, int cp,
                             cpattn_dtype dt, cpattn_stream_t stream) {
  return shard_common(src, dst, B, H, T, d, cp, dt, stream, true);
}

cpattn_status cpattn_shard_rope(const void *src, void *dst, int B, int H, int T, int d, int cp,
                                cpattn_dtype dt, cpattn_stream_t stream) {
  return shard_common(src, dst, B, H, T, d, cp, dt, stream, false, true);
}

cpattn_status cpattn_unshard_rope(const void *src, void *dst, int B, int H, int T, int d, int cp,
                                  cpattn_dtype dt, cpattn_stream_t stream) {
  return shard_common(src, dst, B, H, T, d, cp, dt, stream, true, true);
}

cpattn_status cpattn_shard_rope_cfg(const void *src, void *dst, int B, int H, int T, int d, int cp,
                                    cpattn_dtype dt, const cpattn_rope_cfg *cfg,
                                    cpattn_stream_t stream) {
  g_msg[0] = 0;
  if (!cfg) return fail(CPATTN_ERR_ARG, "RoPE configuration is NULL");
  return shard_common(src, dst, B, H, T, d, cp, dt, stream, false, true, cfg);
}

cpattn_status cpattn_unshard_rope_cfg(const void *src, void *dst, int B, int H, int T, int d, int cp,
                                      cpattn_dtype dt, const cpattn_rope_cfg *cfg,
                                      cpattn_stream_t stream) {
  g_msg[0] = 0;
  if (!cfg) return fail(CPATTN_ERR_ARG, "RoPE configuration is NULL");
  return shard_common(src, dst, B, H, T, d, cp, dt, stream, true, true, cfg);
}

static cpattn_status shard_batch_common(const void *const *src, void *const *dst, const int *heads, const int *rope,
                                        int n, int B, int T, int d, int cp, const cpattn_rope_cfg *cfg,
                                        cpattn_dtype dt, cpattn_stream_t stream, bool inverse) {
  g_msg[0] = 0;
  if (!src || !dst || !heads || !rope) return fail(CPATTN_ERR_ARG, "null pointer");
  if (n < 1 || n > kBatchMax) return fail(CPATTN_ERR_ARG, "n=%d must be in [1, %d]", n, kBatchMax);
  if (cfg && check_rope_cfg(cfg) != CPATTN_OK) return CPATTN_ERR_ARG;
  if (dt != CPATTN_F32 && dt != CPATTN_BF16) return fail(CPATTN_ERR_DTYPE, "unknown dtype %d", (int)dt);
  const int elt = dt == CPATTN_F32 ? 4 : 2;
  if (d != 64 && d != 128) return fail(CPATTN_ERR_SHAPE, "d=%d: only 64 and 128 are supported", d);
  if (T > (1 << 24)) return fail(CPATTN_ERR_SHAPE, "T=%d exceeds 2^24", T);
  ShardBatch b;
  b.n = n;
  long long chunks = 0;
  size_t bytes[kBatchMax];
  for (int i = 0; i < n; ++i) {
    cpattn_status st = check_common(B, heads[i], T, d, cp);
    if (st != CPATTN_OK) return st;
    if (!src[i] || !dst[i]) return fail(CPATTN_ERR_ARG, "null pointer for tensor %d", i);
    if (!aligned16(src[i]) || !aligned16(dst[i])) return fail(CPATTN_ERR_ALIGN, "pointers must be 16-byte aligned");
    if (rope[i] != 0 && rope[i] != 1) return fail(CPATTN_ERR_ARG, "rope[%d] must be 0 or 1", i);
    bytes[i] = (size_t)B * heads[i] * T * d * elt;
    b.src[i] = src[i];
    b.dst[i] = dst[i];
    b.rope[i] = rope[i];
    b.first_chunk[i] = chunks;
    chunks += (long long)B * heads[i] * 2 * cp;
  }
  for (int i = 0; i < n; ++i)
    for (int j = 0; j < n; ++j)
      if (overlaps(dst[i], bytes[i], src[j], bytes[j]) || (i != j && overlaps(dst[i], bytes[i], dst[j], bytes[j])))
        return fail(CPATTN_ERR_ARG, "a destination overlaps another buffer of the batch");
  b.n_chunks = chunks;
  Geometry g = geometry(B, 1, T, T, d, cp, 1, 0);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  trace_record(0, s);
  cpattn_status st = launch_shard_batch(b, g, dt, inverse, cfg, s);
  trace_record(1, s);
  return st;
}

cpattn_status cpattn_shard_batch(const void *const *src, void *const *dst, const int *heads, const int *rope, int n,
                                 int B, int T, int d, int cp, const cpattn_rope_cfg *cfg, cpattn_dtype dt,
                                 cpattn_stream_t stream) {
  return shard_batch_common(src, dst, heads, rope, n, B, T, d, cp, cfg, dt, stream, false);
}

cpattn_status cpattn_unshard_batch(const void *const *src, void *const *dst, const int *heads, const int *rope, int n,
                                   int B, int T, int d, int cp, const cpattn_rope_cfg *cfg, cpattn_dtype dt,
                                   cpattn_stream_t stream) {
  return shard_batch_common(src, dst, heads, rope, n, B, T, d, cp, cfg, dt, stream, true);
}

static cpattn_status ulysses_common(const void *src, void *dst, int B, int H, int T, int d, int P,
                                    int inverse, bool rope, const cpattn_rope_cfg *cfg,
                                    cpattn_dtype dt, cpattn_stream_t stream) {
  g_msg[0] = 0;
  if (!src || !dst) return fail(CPATTN_ERR_ARG, "null pointer");
  if (B < 1 || H < 1 || T < 1 || d < 1 || P < 1)
    return fail(CPATTN_ERR_SHAPE, "sizes must be >= 1 (B=%d H=%d T=%d d=%d P=%d)", B, H, T, d, P);
  if (T % P != 0 || (H % P != 0 && (H > P || P % H != 0)))
    return fail(CPATTN_ERR_SHAPE, "P=%d must divide T=%d, and P must divide H=%d or H divide P", P, T, H);
  if ((long long)B * (H < P ? P : H) * T > (1LL << 31) - 1) return fail(CPATTN_ERR_SHAPE, "B*H*T too large");
  if (inverse != 0 && inverse != 1) return fail(CPATTN_ERR_ARG, "inverse must be 0 or 1");
  if (dt != CPATTN_F32 && dt != CPATTN_BF16) return fail(CPATTN_ERR_DTYPE, "unknown dtype %d", (int)dt);
  if (cfg && check_rope_cfg(cfg) != CPATTN_OK) return CPATTN_ERR_ARG;
  const int elt = dt == CPATTN_F32 ? 4 : 2;
  if ((d * elt) % 16 != 0) return fail(CPATTN_ERR_ALIGN, "row of d*elt=%d bytes is not a multiple of 16", d * elt);
  if (!aligned16(src) || !aligned16(dst)) return fail(CPATTN_ERR_ALIGN, "pointers must be 16-byte aligned");
  const size_t seq_bytes = (size_t)B * H * T * d * elt;                    // sequence shards
  const size_t head_bytes = H < P ? (size_t)P * B * T * d * elt : seq_bytes;   // head shards (replicated)
  if (overlaps(src, inverse ? head_bytes : seq_bytes, dst, inverse ? seq_bytes : head_bytes))
    return fail(CPATTN_ERR_ARG, "src and dst overlap");
  if ((rope || H < P) && d != 64 && d != 128)
    return fail(CPATTN_ERR_SHAPE, "d=%d: RoPE and replication need d in {64, 128}", d);
  if (rope && T > (1 << 24)) return fail(CPATTN_ERR_SHAPE, "T=%d exceeds 2^24", T);
  Geometry g = geometry(B, H, T, T, d, 1, 1, rope ? 1 : 0);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  trace_record(0, s);
  cpattn_status st = rope ? launch_ulysses_rope(src, dst, g, P, dt, inverse != 0, cfg, s)
                          : launch_ulysses(src, dst, g, P, elt, inverse != 0, s);
  trace_record(1, s);
  return st;
}

cpattn_status cpattn_ulysses_a2a(const void *src, void *dst, int B, int H, int T, int d, int P,
                                 int inverse, cpattn_dtype dt, cpattn_stream_t stream) {
  return ulysses_common(src, dst, B, H, T, d, P, inverse, false, nullptr, dt, stream);
}

cpattn_status cpattn_ulysses_a2a_rope(const void *src, void *dst, int B, int H, int T, int d, int P,
                                      int inverse, const cpattn_rope_cfg *cfg, cpattn_dtype dt,
                                      cpattn_stream_t stream) {
  return ulysses_common(src, dst, B, H, T, d, P, inverse, true, cfg, dt, stream);
}

cpattn_status cpattn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                         int B, int T, int T_valid, int H, int d, int cp, int causal, int rope,
                         cpattn_dtype dt, cpattn_stream_t stream) {
  return cpattn_fwd_gqa(q, k, v, o, lse, B, T, T_valid, H, H, d, cp, causal, rope, dt, stream);
}

static cpattn_status fwd_impl(const void *q, const void *k, const void *v, void *o, float *lse,
                              int B, int T, int T_valid, int H, int H_kv, int d, int cp, int causal,
                              int rope, const int *doc_lo, const int *doc_hi, cpattn_dtype dt,
                              cpattn_stream_t stream, const cpattn_rope_cfg *rope_cfg = nullptr,
                              void *q_rot = nullptr, void *k_rot = nullptr);

cpattn_status cpattn_fwd_gqa(const void *q, const void *k, const void *v, void *o, float *lse,
                             int B, int T, int T_valid, int H, int H_kv, int d, int cp, int causal,
                             int rope, cpattn_dtype dt, cpattn_stream_t stream) {
  return fwd_impl(q, k, v, o, lse, B, T, T_valid, H, H_kv, d, cp, causal, rope, nullptr, nullptr, dt,
                  stream);
}

cpattn_status cpattn_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                                int B, int T, int T_valid, int H, int H_kv, int d, int cp, int causal,
                                const int32_t *doc_lo, const int32_t *doc_hi, cpattn_dtype dt,
                                cpattn_stream_t stream) {
  g_msg[0] = 0;
  if (!doc_lo || !doc_hi) return fail(CPATTN_ERR_ARG, "document bounds are NULL");
  return fwd_impl(q, k, v, o, lse, B, T, T_valid, H, H_kv, d, cp, causal, 0, doc_lo, doc_hi, dt, stream);
}

cpattn_status cpattn_fwd_rope_cfg(const void *q, const void *k, const void *v, void *o, float *lse,
                                  int B, int T, int T_valid, int H, int H_kv, int d, int cp,
                                  int causal, const cpattn_rope_cfg *cfg, cpattn_dtype dt,
                                  cpattn_stream_t stream) {
  g_msg[0] = 0;
  cpattn_status st = check_rope_cfg(cfg);
  if (st != CPATTN_OK) return st;
  return fwd_impl(q, k, v, o, lse, B, T, T_valid, H, H_kv, d, cp, causal, 1, nullptr, nullptr, dt, stream,
                  cfg);
}

static cpattn_status fwd_impl(const void *q, const void *k, const void *v, void *o, float *lse,
                              int B, int T, int T_valid, int H, int H_kv, int d, int cp, int causal,
                              int rope, const int *doc_lo, const int *doc_hi, cpattn_dtype dt,
                              cpattn_stream_t stream, const cpattn_rope_cfg *rope_cfg, void *q_rot,
                              void *k_rot) {
  g_msg[0] = 0;
  if (!q || !k || !v || !o || !lse) return fail(CPATTN_ERR_ARG, "null pointer");
  cpattn_status st = check_attn(B, T, T_valid, H, d, cp, causal, rope, dt);
  if (st != CPATTN_OK) return st;
  if ((st = check_heads(H, H_kv)) != CPATTN_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return fail(CPATTN_ERR_ALIGN, "pointers must be 16-byte aligned");
  const size_t elt = dt == CPATTN_F32 ? 4 : 2;
  const size_t tb = (size_t)B * H * T * d * elt;
  const size_t tkv = (size_t)B * H_kv * T * d * elt;
  if (overlaps(o, tb, q, tb) || overlaps(o, tb, k, tkv) || overlaps(o, tb, v, tkv) ||
      overlaps(lse, (size_t)B * H * T * 4, o, tb))
    return fail(CPATTN_ERR_ARG, "outputs overlap inputs");
  Geometry g = geometry(B, H, T, T_valid, d, cp, causal, rope, H_kv);
  g.doc_lo = doc_lo;
  g.doc_hi = doc_hi;
  g.rope_cfg = rope_cfg;
  g.q_rot = q_rot;
  g.k_rot = k_rot;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  trace_record(0, s);
  if (dt == CPATTN_F32)
    st = launch_fwd_f32(static_cast<const float *>(q), static_cast<const float *>(k),
                        static_cast<const float *>(v), static_cast<float *>(o), lse, g, s);
  else
    st = launch_fwd_bf16(q, k, v, o, lse, g, s);
  trace_record(1, s);
  return st;
}

size_t cpattn_bwd_workspace_bytes(int B, int T, int H, int d) {
  (void)d;
  if (B < 1 || T < 1 || H < 1) return 0;
  size_t rows = (size_t)B * H * T;
  return ((rows * sizeof(float) + 255) / 256) * 256;   // D = rowsum(dO * O), fp32
}

cpattn_status cpattn_bwd(const void *q, const void *k, const void *v, const void *o,
                         const float *lse, const void *dO, void *dq, void *dk, void *dv,
                         void *workspace, int B, int T, int T_valid, int H, int d, int cp,
                         int causal, int rope, cpattn_dtype dt, cpattn_stream_t stream) {
  return cpattn_bwd_gqa(q, k, v, o, lse, dO, dq, dk, dv, workspace, B, T, T_valid, H, H, d, cp,
                        causal, rope, dt, stream);
}

static cpattn_status bwd_impl(const void *q, const void *k, const void *v, const void *o,
                              const float *lse, const void *dO, void *dq, void *dk, void *dv,
                              void *workspace, int B, int T, int T_valid, int H, int H_kv, int d,
                              int cp, int causal, int rope, const int *doc_lo, const int *doc_hi,
                              cpattn_dtype dt, cpattn_stream_t stream,
                              const cpattn_rope_cfg *rope_cfg = nullptr, bool rope_epi = false);

cpattn_status cpattn_bwd_gqa(const void *q, const void *k, const void *v, const void *o,
                             const float *lse, const void *dO, void *dq, void *dk, void *dv,
                             void *workspace, int B, int T, int T_valid, int H, int H_kv, int d,
                             int cp, int causal, int rope, cpattn_dtype dt, cpattn_stream_t stream) {
  return bwd_impl(q, k, v, o, lse, dO, dq, dk, dv, workspace, B, T, T_valid, H, H_kv, d, cp, causal,
                  rope, nullptr, nullptr, dt, stream);
}

cpattn_status cpattn_bwd_varlen(const void *q, const void *k, const void *v, const void *o,
                                const float *lse, const void *dO, void *dq, void *dk, void *dv,
                                void *workspace, int B, int T, int T_valid, int H, int H_kv, int d,
                                int cp, int causal, const int32_t *doc_lo, const int32_t *doc_hi,
                                cpattn_dtype dt, cpattn_stream_t stream) {
  g_msg[0] = 0;
  if (!doc_lo || !doc_hi) return fail(CPATTN_ERR_ARG, "document bounds are NULL");
  return bwd_impl(q, k, v, o, lse, dO, dq, dk, dv, workspace, B, T, T_valid, H, H_kv, d, cp, causal, 0,
                  doc_lo, doc_hi, dt, stream);
}

cpattn_status cpattn_bwd_rope_cfg(const void *q, const void *k, const void *v, const void *o,
                                  const float *lse, const void *dO, void *dq, void *dk, void *dv,
                                  void *workspace, int B, int T, int T_valid, int H, int H_kv, int d,
                                  int cp, int causal, const cpattn_rope_cfg *cfg, cpattn_dtype dt,
                                  cpattn_stream_t stream) {
  g_msg[0] = 0;
  cpattn_status st = check_rope_cfg(cfg);
  if (st != CPATTN_OK) return st;
  return bwd_impl(q, k, v, o, lse, dO, dq, dk, dv, workspace, B, T, T_valid, H, H_kv, d, cp, causal, 1,
                  nullptr, nullptr, dt, stream, cfg);
}

cpattn_status cpattn_doc_bounds(const int32_t *cu_seqlens, int n_docs, int T, int32_t *doc_lo,
                                int32_t *doc_hi, cpattn_stream_t stream) {
  g_msg[0] = 0;
  if (!cu_seqlens || !doc_lo || !doc_hi) return fail(CPATTN_ERR_ARG, "null pointer");
  if (n_docs < 1 || T < 1) return fail(CPATTN_ERR_SHAPE, "n_docs=%d and T=%d must be >= 1", n_docs, T);
  if (!aligned16(doc_lo) || !aligned16(doc_hi) || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u))
    return fail(CPATTN_ERR_ALIGN, "doc_lo, doc_hi must be 16-byte aligned, cu_seqlens 4-byte aligned");
  const size_t tb = (size_t)T * 4;
  if (overlaps(doc_lo, tb, doc_hi, tb) || overlaps(cu_seqlens, (size_t)(n_docs + 1) * 4, doc_lo, tb) ||
      overlaps(cu_seqlens, (size_t)(n_docs + 1) * 4, doc_hi, tb))
    return fail(CPATTN_ERR_ARG, "cu_seqlens, doc_lo and doc_hi must not overlap");
  return launch_doc_bounds(cu_seqlens, n_docs, T, doc_lo, doc_hi, reinterpret_cast<cudaStream_t>(stream));
}

static cpattn_status bwd_impl(const void *q, const void *k, const void *v, const void *o,
                              const float *lse, const void *dO, void *dq, void *dk, void *dv,
                              void *workspace, int B, int T, int T_valid, int H, int H_kv, int d,
                              int cp, int causal, int rope, const int *doc_lo, const int *doc_hi,
                              cpattn_dtype dt, cpattn_stream_t stream, const cpattn_rope_cfg *rope_cfg,
                              bool rope_epi) {
  g_msg[0] = 0;
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv || !workspace)
    return fail(CPATTN_ERR_ARG, "null pointer");
  cpattn_status st = check_attn(B, T, T_valid, H, d, cp, causal, rope, dt);
  if (st != CPATTN_OK) return st;
  if ((st = check_heads(H, H_kv)) != CPATTN_OK) return st;
  const void *ptrs[] = {q, k, v, o, lse, dO, dq, dk, dv, workspace};
  for (const void *p : ptrs)
    if (!aligned16(p)) return fail(CPATTN_ERR_ALIGN, "pointers must be 16-byte aligned");
  const size_t elt = dt == CPATTN_F32 ? 4 : 2;
  const size_t tq = (size_t)B * H * T * d * elt;
  const size_t tkv = (size_t)B * H_kv * T * d * elt;
  const size_t wb = cpattn_bwd_workspace_bytes(B, T, H, d);
  const void *outs[] = {dq, dk, dv};
  const size_t out_b[] = {tq, tkv, tkv};
  const void *ins[] = {q, k, v, o, dO};
  const size_t in_b[] = {tq, tkv, tkv, tq, tq};
  for (int i = 0; i < 3; ++i) {
    for (int j = 0; j < 5; ++j)
      if (overlaps(outs[i], out_b[i], ins[j], in_b[j]))
        return fail(CPATTN_ERR_ARG, "gradient outputs overlap inputs");
    for (int j = 0; j < 3; ++j)
      if (i != j && overlaps(outs[i], out_b[i], outs[j], out_b[j]))
        return fail(CPATTN_ERR_ARG, "gradient outputs overlap");
    if (overlaps(outs[i], out_b[i], workspace, wb)) return fail(CPATTN_ERR_ARG, "workspace overlaps outputs");
  }
  Geometry g = geometry(B, H, T, T_valid, d, cp, causal, rope, H_kv);
  g.doc_lo = doc_lo;
  g.doc_hi = doc_hi;
  g.rope_cfg = rope_cfg;
  g.rope_epi = rope_epi;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  float *D = static_cast<float *>(workspace);
  // The paired dQ kernel (bf16, d = 128, q and k not rotated in-kernel, tile
  // tables) computes D = rowsum(dO * O) for its own rows and runs first;
  // every other path runs the D pass before its kernels.
  const bool d_in_dq = dt == CPATTN_BF16 && d == 128 && !rope && uses_tables(T, cp);
  trace_record(0, s);
  if (d_in_dq) {
    g.o_for_D = o;
  } else {
    st = launch_bwd_preprocess(o, dO, D, (long long)B * H * T, d, dt, s);
    if (st != CPATTN_OK) return st;
  }
  trace_record(1, s);
  if (dt == CPATTN_F32)
    st = launch_bwd_f32(static_cast<const float *>(q), static_cast<const float *>(k),
                          static_cast<const float *>(v), static_cast<const float *>(o), lse,
                          static_cast<const float *>(dO), static_cast<float *>(dq),
                          static_cast<float *>(dk), static_cast<float *>(dv), D, g, s);
  else
    st = launch_bwd_bf16(q, k, v, o, lse, dO, dq, dk, dv, D, g, s);
  return st;
}

// ------------------------------------------- in-kernel RoPE, rotated once
cpattn_status cpattn_fwd_rope_save(const void *q, const void *k, const void *v, void *o, float *lse, void *q_rot,
                                   void *k_rot, int B, int T, int T_valid, int H, int H_kv, int d, int cp,
                                   int causal, const int32_t *doc_lo, const int32_t *doc_hi,
                                   const cpattn_rope_cfg *cfg, cpattn_dtype dt, cpattn_stream_t stream) {
  g_msg[0] = 0;
  if (!q_rot || !k_rot) return fail(CPATTN_ERR_ARG, "q_rot and k_rot must not be NULL");
  if ((doc_lo == nullptr) != (doc_hi == nullptr)) return fail(CPATTN_ERR_ARG, "give both document bounds or neither");
  if (cfg && check_rope_cfg(cfg) != CPATTN_OK) return CPATTN_ERR_ARG;
  cpattn_status st = check_attn(B, T, T_valid, H, d, cp, causal, 1, dt);
  if (st != CPATTN_OK) return st;
  if ((st = check_heads(H, H_kv)) != CPATTN_OK) return st;
  if (!aligned16(q_rot) || !aligned16(k_rot)) return fail(CPATTN_ERR_ALIGN, "pointers must be 16-byte aligned");
  const size_t elt = dt == CPATTN_F32 ? 4 : 2;
  const size_t tq = (size_t)B * H * T * d * elt, tkv = (size_t)B * H_kv * T * d * elt;
  const void *bufs[] = {q, k, v, o, lse, q_rot, k_rot};
  const size_t sizes[] = {tq, tkv, tkv, tq, (size_t)B * H * T * 4, tq, tkv};
  for (int i = 5; i < 7; ++i)
    for (int j = 0; j < 7; ++j)
      if (i != j && bufs[j] && overlaps(bufs[i], sizes[i], bufs[j], sizes[j]))
        return fail(CPATTN_ERR_ARG, "q_rot and k_rot must not overlap each other, the inputs or the outputs");
  if (dt == CPATTN_BF16 && uses_tables(T, cp))   // rotated tiles stored by the attention kernel itself
    return fwd_impl(q, k, v, o, lse, B, T, T_valid, H, H_kv, d, cp, causal, 1, doc_lo, doc_hi, dt, stream, cfg,
                    q_rot, k_rot);
  // fp32, or a schedule past the tile tables: rotate first, then attend with rope = 0
  Geometry g = geometry(B, H, T, T, d, cp, 1, 1, H_kv);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((st = launch_rope_sharded(q, q_rot, g, H, dt, false, cfg, s)) != CPATTN_OK) return st;
  if ((st = launch_rope_sharded(k, k_rot, g, H_kv, dt, false, cfg, s)) != CPATTN_OK) return st;
  return fwd_impl(q_rot, k_rot, v, o, lse, B, T, T_valid, H, H_kv, d, cp, causal, 0, doc_lo, doc_hi, dt, stream);
}

cpattn_status cpattn_bwd_rotated(const void *q_rot, const void *k_rot, const void *v, const void *o,
                                 const float *lse, const void *dO, void *dq, void *dk, void *dv, void *workspace,
                                 int B, int T, int T_valid, int H, int H_kv, int d, int cp, int causal,
                                 const int32_t *doc_lo, const int32_t *doc_hi, const cpattn_rope_cfg *cfg,
                                 cpattn_dtype dt, cpattn_stream_t stream) {
  g_msg[0] = 0;
  if ((doc_lo == nullptr) != (doc_hi == nullptr)) return fail(CPATTN_ERR_ARG, "give both document bounds or neither");
  if (cfg && check_rope_cfg(cfg) != CPATTN_OK) return CPATTN_ERR_ARG;
  cpattn_status st = check_attn(B, T, T_valid, H, d, cp, causal, 1, dt);   // RoPE needs d in {64, 128}
  if (st != CPATTN_OK) return st;
  if (dt == CPATTN_BF16 && uses_tables(T, cp))   // R^T in the dQ and dK epilogues
    return bwd_impl(q_rot, k_rot, v, o, lse, dO, dq, dk, dv, workspace, B, T, T_valid, H, H_kv, d, cp, causal, 0,
                    doc_lo, doc_hi, dt, stream, cfg, true);
  // fp32, or a schedule past the tile tables: dq', dk' from the rope = 0 kernels, then R^T in place
  st = bwd_impl(q_rot, k_rot, v, o, lse, dO, dq, dk, dv, workspace, B, T, T_valid, H, H_kv, d, cp, causal, 0,
                doc_lo, doc_hi, dt, stream);
  if (st != CPATTN_OK) return st;
  Geometry g = geometry(B, H, T, T, d, cp, 1, 1, H_kv);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((st = launch_rope_sharded(dq, dq, g, H, dt, true, cfg, s)) != CPATTN_OK) return st;
  return launch_rope_sharded(dk, dk, g, H_kv, dt, true, cfg, s);
}

// --------------------------------------------------- allocation-free backward
// D = rowsum(dO * O) for cpattn_bwd_noalloc lives in this file-scope array
// instead of a caller workspace. Every GPU that loads the library holds it
// (CPATTN_NOALLOC_MAX_ROWS floats) until the process exits.
static __device__ __align__(256) float g_noalloc_scratch[CPATTN_NOALLOC_MAX_ROWS];

// Device address of the current context's copy of the array. Host code must
// not pass the symbol itself to a kernel (on the host it names a stand-in, not
// device memory), so the address is resolved with the device current, checked,
// and cached per context (symbol_address).
static float *noalloc_scratch() { return static_cast<float *>(symbol_address(g_noalloc_scratch)); }

cpattn_status cpattn_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                                 const float *lse, const void *dO, void *dq, void *dk, void *dv,
                                 int B, int T, int T_valid, int H, int d, int cp, int causal,
                                 int rope, cpattn_dtype dt, cpattn_stream_t stream) {
  g_msg[0] = 0;
  if (B < 1 || H < 1 || T < 1) return fail(CPATTN_ERR_SHAPE, "sizes must be >= 1");
  const long long rows = (long long)B * H * T;
  if (rows > (long long)CPATTN_NOALLOC_MAX_ROWS)
    return fail(CPATTN_ERR_SHAPE, "B*H*T=%lld exceeds the static scratch of %u rows", rows,
                (unsigned)CPATTN_NOALLOC_MAX_ROWS);
  float *scratch = noalloc_scratch();
  if (!scratch) return fail(CPATTN_ERR_CUDA, "cannot resolve the device address of the static scratch");
  return cpattn_bwd(q, k, v, o, lse, dO, dq, dk, dv, scratch, B, T, T_valid, H, d, cp, causal, rope,
                    dt, stream);
}

cpattn_status cpattn_merge(const float *const *o_parts, const float *const *lse_parts, int n,
                           void *o, float *lse, int B, int H, int T, int d, cpattn_dtype dt,
                           cpattn_stream_t stream) {
  g_msg[0] = 0;
  if (!o_parts || !lse_parts || !o || !lse) return fail(CPATTN_ERR_ARG, "null pointer");
  if (n < 1 || n > 16) return fail(CPATTN_ERR_ARG, "n=%d must be in [1, 16]", n);
  if (B < 1 || H < 1 || T < 1) return fail(CPATTN_ERR_SHAPE, "sizes must be >= 1");
  if (d != 64 && d != 128) return fail(CPATTN_ERR_SHAPE, "d=%d: only 64 and 128 are supported", d);
  if (dt != CPATTN_F32 && dt != CPATTN_BF16) return fail(CPATTN_ERR_DTYPE, "unknown dtype %d", (int)dt);
  for (int i = 0; i < n; ++i) {
    if (!o_parts[i] || !lse_parts[i]) return fail(CPATTN_ERR_ARG, "null partial pointer %d", i);
    if (!aligned16(o_parts[i]) || !aligned16(lse_parts[i]))
      return fail(CPATTN_ERR_ALIGN, "partial %d not 16-byte aligned", i);
  }
  if (!aligned16(o) || !aligned16(lse)) return fail(CPATTN_ERR_ALIGN, "outputs must be 16-byte aligned");
  return launch_merge(o_parts, lse_parts, n, o, lse, (long long)B * H * T, d, dt,
                      reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
