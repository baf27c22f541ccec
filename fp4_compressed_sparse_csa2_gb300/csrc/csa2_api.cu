// csa2_api.cu -- the C ABI of libcsa2 (declared in include/csa2.h).
//
// Host side only: argument validation, workspace carving, launch configuration,
// mode orchestration (Full = pack + index + top-k + attention; Reindex = index +
// top-k + attention on a shared cache; Reuse = attention on given indices), a launch
// counter and optional per-kernel CUDA-event timing.
#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>
#include <vector>

#include "csa2_kernels.cuh"

using namespace csa2;

namespace csa2 {

cudaError_t smem_limit_once(const void* kernel, size_t bytes, std::atomic<int>* cache) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cached = dev >= 0 && dev < kMaxDevices;
  if (cached && cache[dev].load(std::memory_order_acquire) >= static_cast<int>(bytes)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess && cached) cache[dev].store(static_cast<int>(bytes), std::memory_order_release);
  return e;
}

std::atomic<uint64_t> g_wait_ns{0};  // 0: the default bound

uint64_t pipeline_wait_ns() {
  const uint64_t v = g_wait_ns.load(std::memory_order_relaxed);
  return v ? v : kWaitLimitNs;
}

}  // namespace csa2

namespace {

thread_local std::string g_last_error;
std::atomic<int64_t> g_launches{0};

csa2_status fail(csa2_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

csa2_status cuda_fail(cudaError_t e, const char* what) {
  return fail(CSA2_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// ------------------------------------------------------------------ tracing
enum Kind {
  kPack = 0, kIndex = 1, kTopkHist = 2, kTopkSel = 3, kTopkFinal = 4, kAttn = 5, kTopk = 6, kPool = 7, kGather = 8,
  kMap = 9, kPoolBmax = 10, kPackWindow = 12, kKinds = 13
};
constexpr int kTraceCap = 4096;

struct Trace {
  std::mutex mu;
  bool on = false;
  std::vector<cudaEvent_t> ev;  // 2 per record
  std::vector<int> kind;
  int n = 0;
  int pending_kind = -1;
} g_trace;

void trace_begin(int kind, cudaStream_t s) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  std::lock_guard<std::mutex> lk(g_trace.mu);
  if (!g_trace.on || g_trace.n >= kTraceCap) return;
  cudaEventRecord(g_trace.ev[2 * g_trace.n], s);
  g_trace.pending_kind = kind;
}

void trace_end(int kind, cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_trace.mu);
  if (!g_trace.on || g_trace.n >= kTraceCap || g_trace.pending_kind != kind) return;
  cudaEventRecord(g_trace.ev[2 * g_trace.n + 1], s);
  g_trace.kind[g_trace.n] = kind;
  ++g_trace.n;
  g_trace.pending_kind = -1;
}

int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

// ------------------------------------------------------------------ workspace
constexpr size_t kHeader = 256;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
  size_t qpack, scores, topk, apart, total;
  int64_t ld;
  // candidate pool (hierarchical indexer)
  size_t bkey, compact, pscores, plen, preq, pslots;
  int64_t nb_cap;
};

int64_t ws_ld(int64_t t_max) { return ((t_max + 127) / 128) * 128; }

WsLayout ws_layout(int64_t n_q, int32_t heads_I, int64_t t_max, int32_t scores_in_ws, bool pool = false) {
  WsLayout L{};
  size_t off = kHeader;
  const size_t nq = static_cast<size_t>(n_q);
  L.qpack = off;
  off = align256(off + nq * (static_cast<size_t>(heads_I) * 64 + 1024));
  L.ld = ws_ld(t_max);
  L.scores = off;
  if (scores_in_ws) off = align256(off + nq * static_cast<size_t>(L.ld) * 4);
  L.topk = off;
  off = align256(off + topk_ws_bytes(n_q));
  L.apart = off;  // partial outputs of the attention's key splits (small batches)
  off = align256(off + attn_split_ws_bytes(n_q, sm_count()));
  if (pool) {
    L.nb_cap = (t_max + CSA2_POOL_BLOCK - 1) / CSA2_POOL_BLOCK;
    L.bkey = off;
    off = align256(off + nq * static_cast<size_t>(L.nb_cap) * 4);
    L.compact = off;  // 128 pages per query, sized for the larger (72-byte) format
    off = align256(off + nq * (CSA2_POOL / kPage) * static_cast<size_t>(kIdxPageBytes));
    L.pscores = off;
    off = align256(off + nq * CSA2_POOL * 4);
    L.plen = off;
    off = align256(off + nq * 4);
    L.preq = off;
    off = align256(off + nq * 4);
    L.pslots = off;
    off = align256(off + nq * CSA2_TOPK * 4);
  }
  L.total = off;
  return L;
}

csa2_status check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (ws == nullptr || !aligned(ws, 256)) return fail(CSA2_ERR_WORKSPACE, "workspace must be a 256-byte aligned device pointer");
  if (ws_bytes < need) return fail(CSA2_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu needed", ws_bytes, need);
  return CSA2_OK;
}

csa2_status check_cache(const csa2_cache* c, bool need_kv, bool need_idx) {
  if (c == nullptr) return fail(CSA2_ERR_INVALID_ARG, "cache is NULL");
  if (need_kv && (c->kv == nullptr || !aligned(c->kv, 256)))
    return fail(CSA2_ERR_INVALID_ARG, "cache.kv must be a 256-byte aligned device pointer");
  if (need_idx && (c->idx == nullptr || !aligned(c->idx, 256)))
    return fail(CSA2_ERR_INVALID_ARG, "cache.idx must be a 256-byte aligned device pointer");
  if (c->max_pages <= 0 || c->n_pages <= 0) return fail(CSA2_ERR_INVALID_ARG, "cache.max_pages and cache.n_pages must be positive");
  if (c->idx_format != CSA2_IDX_E4M3_16 && c->idx_format != CSA2_IDX_MXFP4)
    return fail(CSA2_ERR_INVALID_ARG, "cache.idx_format must be CSA2_IDX_E4M3_16 or CSA2_IDX_MXFP4 (got %d)", c->idx_format);
  return CSA2_OK;
}

// Bytes of one packed indexer-query group of N rows: the nibbles, then the scale atoms
// (two of E4M3 per 16 channels, or one of E8M0 per 32 channels for MXFP4).
int32_t grp_bytes(int32_t N, const csa2_cache& c) {
  return N * 64 + (c.idx_format == CSA2_IDX_MXFP4 ? 512 : 1024);
}

int32_t* err_word(void* ws) { return reinterpret_cast<int32_t*>(ws); }

// ------------------------------------------------------------------ steps
csa2_status run_pack(const void* latent, const void* idx_key, const int32_t* req, const int64_t* pos, int64_t n,
                     const csa2_cache& cache, const void* q_idx, int64_t n_q, int32_t heads_I, int32_t G, uint8_t* qpack,
                     int32_t* err, cudaStream_t stream) {
  PackArgs a{};
  a.latent = static_cast<const __nv_bfloat16*>(latent);
  a.idx_key = static_cast<const __nv_bfloat16*>(idx_key);
  a.new_req = req;
  a.new_pos = pos;
  a.n_new = n;
  a.cache = cache;
  a.q_idx = static_cast<const __nv_bfloat16*>(q_idx);
  a.n_q = q_idx ? n_q : 0;
  a.heads_I = heads_I;
  a.G = G;
  a.N = G * heads_I;
  a.grp_bytes = grp_bytes(a.N, cache);
  a.n_groups = q_idx ? (n_q + G - 1) / G : 0;
  a.qpack = qpack;
  a.err = err;
  if (a.n_new == 0 && a.n_groups == 0) return CSA2_OK;
  trace_begin(kPack, stream);
  const cudaError_t e = launch_pack(a, stream);
  trace_end(kPack, stream);
  return e == cudaSuccess ? CSA2_OK : cuda_fail(e, "pack kernel");
}

csa2_status run_index(const csa2_cache& cache, const uint8_t* qpack, const float* w, int32_t heads_I, const int32_t* req,
                      const int32_t* n_visible, int64_t n_q, int32_t G, int64_t t_max, float* scores, int64_t ld,
                      int32_t* err, cudaStream_t stream, bool early = false, const int32_t* new_req = nullptr,
                      const int64_t* new_pos = nullptr, int64_t n_new = 0) {
  if (n_q == 0 || t_max == 0) return CSA2_OK;
  IndexArgs a{};
  a.idx_pages = cache.idx;
  a.cache = cache;
  a.qpack = qpack;
  a.heads_I = heads_I;
  a.G = G;
  a.N = G * heads_I;
  a.grp_bytes = grp_bytes(a.N, cache);
  a.w = w;
  a.req = req;
  a.n_visible = n_visible;
  a.scores = scores;
  a.ld = ld;
  a.n_q = n_q;
  a.n_groups = (n_q + G - 1) / G;
  a.tpg = static_cast<int32_t>((t_max + kPage - 1) / kPage);
  a.err = err;
  a.stages = 16;
  a.tmem_cols = 512u;
  a.wait_ns = pipeline_wait_ns();
  // early page copies: the previous kernel is this call's own pack kernel (see IndexArgs);
  // the scan of the new entries stays short (decode-sized steps only)
  a.early = early && n_new <= 256 ? 1 : 0;
  a.new_req = new_req;
  a.new_pos = new_pos;
  a.n_new = a.early ? n_new : 0;
  const int64_t total = a.n_groups * a.tpg;
  const int64_t slots = static_cast<int64_t>(sm_count());  // one persistent CTA per SM
  const int grid = static_cast<int>(total < slots ? total : slots);
  trace_begin(kIndex, stream);
  const cudaError_t e = launch_index(a, grid, stream);
  trace_end(kIndex, stream);
  return e == cudaSuccess ? CSA2_OK : cuda_fail(e, "index kernel");
}

csa2_status run_topk(const float* scores, int64_t ld, const int32_t* n_visible, int64_t n_q, int64_t t_max, int32_t k,
                     int32_t* out, uint8_t* tk_ws, int32_t* err, cudaStream_t stream) {
  if (n_q == 0) return CSA2_OK;
  TopkArgs a{};
  a.scores = scores;
  a.ld = ld;
  a.n_visible = n_visible;
  a.n_q = n_q;
  a.k = k;
  a.out = out;
  a.t_max = t_max;
  a.err = err;
  topk_carve(tk_ws, n_q, a);
  const cudaError_t e = launch_topk(a, stream, kTopkHist, kTopkSel, kTopkFinal, trace_begin, trace_end);
  return e == cudaSuccess ? CSA2_OK : cuda_fail(e, "top-k kernels");
}

// One launch, one thread-block cluster per row (no scratch memory).
csa2_status run_topk_cluster(const float* scores, int64_t ld, const int32_t* n_visible, int64_t n_q, int64_t t_max,
                             int32_t k, int32_t* out, int32_t* err, cudaStream_t stream) {
  if (n_q == 0) return CSA2_OK;
  TopkArgs a{};
  a.scores = scores;
  a.ld = ld;
  a.n_visible = n_visible;
  a.n_q = n_q;
  a.k = k;
  a.out = out;
  a.t_max = t_max;
  a.err = err;
  trace_begin(kTopk, stream);
  const cudaError_t e = launch_topk_cluster(a, sm_count(), stream);
  trace_end(kTopk, stream);
  return e == cudaSuccess ? CSA2_OK : cuda_fail(e, "top-k kernel");
}

csa2_status run_pool(const float* scores, int64_t ld, const int32_t* n_visible, int64_t n_q, int64_t t_max,
                     const WsLayout& L, uint8_t* base, int32_t* pool, int32_t* err, cudaStream_t stream) {
  if (n_q == 0) return CSA2_OK;
  PoolArgs a{};
  a.scores = scores;
  a.ld = ld;
  a.n_visible = n_visible;
  a.n_q = n_q;
  a.bkey = reinterpret_cast<uint32_t*>(base + L.bkey);
  a.nb_cap = L.nb_cap;
  a.t_max = L.nb_cap * CSA2_POOL_BLOCK < t_max ? L.nb_cap * CSA2_POOL_BLOCK : t_max;
  a.pool = pool;
  a.pool_len = reinterpret_cast<int32_t*>(base + L.plen);
  a.err = err;
  trace_begin(kPoolBmax, stream);
  cudaError_t e = launch_pool_bmax(a, stream);
  trace_end(kPoolBmax, stream);
  if (e != cudaSuccess) return cuda_fail(e, "block-maximum kernel");
  trace_begin(kPool, stream);
  e = launch_pool(a, stream);
  trace_end(kPool, stream);
  return e == cudaSuccess ? CSA2_OK : cuda_fail(e, "pool kernel");
}

// Reindex over a candidate pool: gather the pool's indexer entries into compact pages,
// score them with the packed query, take the top-512 of the pool slots, map the slots
// back to cache positions.
csa2_status run_pool_reindex(const csa2_step* s, const WsLayout& L, uint8_t* base, int32_t* err,
                             cudaStream_t stream) {
  if (s->n_q == 0) return CSA2_OK;
  GatherArgs g{};
  g.cache = s->cache;
  g.pool = s->pool;
  g.req = s->req;
  g.n_visible = s->n_visible;
  g.n_q = s->n_q;
  g.compact = base + L.compact;
  g.pool_len = reinterpret_cast<int32_t*>(base + L.plen);
  g.req_q = reinterpret_cast<int32_t*>(base + L.preq);
  g.err = err;
  trace_begin(kGather, stream);
  cudaError_t e = launch_gather(g, stream);
  trace_end(kGather, stream);
  if (e != cudaSuccess) return cuda_fail(e, "pool gather kernel");
  csa2_cache cc{};
  cc.kv = s->cache.kv;
  cc.idx = base + L.compact;
  cc.block_table = nullptr;
  cc.max_pages = CSA2_POOL / kPage;
  cc.n_pages = static_cast<int32_t>(s->n_q * (CSA2_POOL / kPage));
  cc.idx_format = s->cache.idx_format;
  float* sc = s->scores ? s->scores : reinterpret_cast<float*>(base + L.pscores);
  const int64_t ld = s->scores ? s->ld : CSA2_POOL;
  csa2_status st = run_index(cc, base + L.qpack, s->w, s->heads_I, g.req_q, g.pool_len, s->n_q, 1, CSA2_POOL, sc, ld,
                             err, stream);
  if (st != CSA2_OK) return st;
  int32_t* slots = reinterpret_cast<int32_t*>(base + L.pslots);
  st = run_topk_cluster(sc, ld, g.pool_len, s->n_q, CSA2_POOL, s->topk, slots, err, stream);
  if (st != CSA2_OK) return st;
  trace_begin(kMap, stream);
  e = launch_map(slots, s->pool, s->topk_idx, s->n_q, stream);
  trace_end(kMap, stream);
  return e == cudaSuccess ? CSA2_OK : cuda_fail(e, "pool map kernel");
}

csa2_status run_attn(const csa2_step& s, uint8_t* base, const WsLayout& L, int32_t* err, cudaStream_t stream) {
  if (s.n_q == 0) return CSA2_OK;
  AttnArgs a{};
  a.q = static_cast<const __nv_bfloat16*>(s.q);
  a.topk_idx = s.topk_idx;
  a.n_visible = s.n_visible;
  a.req = s.req;
  a.window = static_cast<const __nv_bfloat16*>(s.window);
  a.win_start = s.win_start;
  a.win_len = s.win_len;
  a.cache = s.cache;
  const float scale = s.softmax_scale > 0.0f ? s.softmax_scale : 0.04419417382415922f;  // 512^-0.5
  a.scale_log2 = scale * 1.4426950408889634f;
  a.out = static_cast<__nv_bfloat16*>(s.out);
  a.lse = s.lse;
  a.n_q = s.n_q;
  a.err = err;
  a.sinks = s.sinks;
  a.rope_cos = s.rope_cos;
  a.rope_sin = s.rope_sin;
  a.win_ring = s.win_ring;
  a.win_ring_reqs = s.win_ring_reqs;
  a.wait_ns = pipeline_wait_ns();
  // small batches split each query's key tiles over a cluster of CTAs
  const bool ext = s.sinks != nullptr || s.rope_cos != nullptr || s.win_ring != nullptr;
  a.splits = attn_splits_for(s.n_q, sm_count(), ext);
  if (a.splits > 1) {
    a.opart = reinterpret_cast<float*>(base + L.apart);
    a.mpart = a.opart + static_cast<size_t>(s.n_q) * a.splits * CSA2_HEADS * CSA2_D;
  }
  trace_begin(kAttn, stream);
  const cudaError_t e = launch_attn(a, stream);
  trace_end(kAttn, stream);
  if (e != cudaSuccess) return cuda_fail(e, "attention kernel");
  return CSA2_OK;
}

enum Mode { kFull, kReindex, kReuse };

csa2_status check_step(const csa2_step* s, Mode mode) {
  if (s == nullptr) return fail(CSA2_ERR_INVALID_ARG, "step is NULL");
  if (s->n_q < 0) return fail(CSA2_ERR_INVALID_ARG, "n_q must be >= 0");
  if (s->heads != CSA2_HEADS) return fail(CSA2_ERR_UNSUPPORTED, "heads must be 64 (got %d)", s->heads);
  if (s->topk != CSA2_TOPK) return fail(CSA2_ERR_UNSUPPORTED, "topk must be 512 (got %d)", s->topk);
  if (s->n_q > 0) {
    if (!s->q || !aligned(s->q, 16)) return fail(CSA2_ERR_INVALID_ARG, "q must be a 16-byte aligned device pointer");
    if (!s->out) return fail(CSA2_ERR_INVALID_ARG, "out is NULL");
    if (!s->req || !s->n_visible) return fail(CSA2_ERR_INVALID_ARG, "req and n_visible are required");
    if (!s->win_start || !s->win_len) return fail(CSA2_ERR_INVALID_ARG, "win_start and win_len are required");
    if (s->win_ring == nullptr && (!s->window || !aligned(s->window, 16)))
      return fail(CSA2_ERR_INVALID_ARG, "window rows (16-byte aligned) are required without a window ring");
    if (s->win_ring != nullptr && (!aligned(s->win_ring, 16) || s->win_ring_reqs <= 0))
      return fail(CSA2_ERR_INVALID_ARG, "win_ring must be 16-byte aligned with win_ring_reqs > 0");
    if (!s->topk_idx) return fail(CSA2_ERR_INVALID_ARG, "topk_idx is NULL");
    if ((s->rope_cos == nullptr) != (s->rope_sin == nullptr))
      return fail(CSA2_ERR_INVALID_ARG, "rope_cos and rope_sin go together");
  }
  if (s->t_max < 0 || s->t_max > static_cast<int64_t>(s->cache.max_pages) * kPage)
    return fail(CSA2_ERR_INVALID_ARG, "t_max %lld outside [0, max_pages*128]", static_cast<long long>(s->t_max));
  if (mode != kReuse) {
    if (s->heads_I != 64 && s->heads_I != 32) return fail(CSA2_ERR_UNSUPPORTED, "heads_I must be 64 or 32");
    if (s->group != 1 && s->group != 2) return fail(CSA2_ERR_UNSUPPORTED, "group must be 1 or 2");
    if (s->n_q > 0 && (!s->q_idx || !aligned(s->q_idx, 16) || !s->w))
      return fail(CSA2_ERR_INVALID_ARG, "q_idx (16-byte aligned) and w are required");
    const bool pool_scores = mode == kReindex && s->pool != nullptr;  // scores of the pool slots
    const int64_t need_ld = pool_scores ? CSA2_POOL : s->t_max;
    if (s->scores && (s->ld < need_ld || s->ld % 4 != 0 || !aligned(s->scores, 16)))
      return fail(CSA2_ERR_INVALID_ARG, "scores needs ld >= %s, ld %% 4 == 0 and 16-byte alignment",
                  pool_scores ? "16384 (pool slots)" : "t_max");
    if (s->pool != nullptr && !aligned(s->pool, 16))
      return fail(CSA2_ERR_INVALID_ARG, "pool must be a 16-byte aligned device pointer");
    if (pool_scores && s->group != 1) return fail(CSA2_ERR_UNSUPPORTED, "a pool-restricted Reindex needs group 1");
  }
  if (mode == kFull && s->n_new > 0) {
    if (!s->new_latent || !s->new_idx_key || !aligned(s->new_latent, 16) || !aligned(s->new_idx_key, 16) ||
        !s->new_req || !s->new_pos)
      return fail(CSA2_ERR_INVALID_ARG, "new_latent/new_idx_key (16-byte aligned), new_req and new_pos are required");
  }
  return check_cache(&s->cache, true, mode != kReuse);
}

csa2_status run_step(const csa2_step* s, Mode mode, void* ws, size_t ws_bytes, cudaStream_t stream) {
  csa2_status st = check_step(s, mode);
  if (st != CSA2_OK) return st;
  const int32_t heads_I = mode == kReuse ? 64 : s->heads_I;
  const bool pool = mode != kReuse && s->pool != nullptr;
  const WsLayout L = ws_layout(s->n_q, heads_I, s->t_max, mode != kReuse && s->scores == nullptr, pool);
  if ((st = check_ws(ws, ws_bytes, L.total)) != CSA2_OK) return st;
  uint8_t* base = static_cast<uint8_t*>(ws);
  int32_t* err = err_word(ws);
  if (pool && mode == kReindex) {
    st = run_pack(nullptr, nullptr, nullptr, nullptr, 0, s->cache, s->q_idx, s->n_q, heads_I, 1, base + L.qpack, err,
                  stream);
    if (st != CSA2_OK) return st;
    if ((st = run_pool_reindex(s, L, base, err, stream)) != CSA2_OK) return st;
    return run_attn(*s, base, L, err, stream);
  }
  if (mode != kReuse) {
    float* scores = s->scores ? s->scores : reinterpret_cast<float*>(base + L.scores);
    const int64_t ld = s->scores ? s->ld : L.ld;
    st = run_pack(s->new_latent, s->new_idx_key, s->new_req, s->new_pos, mode == kFull ? s->n_new : 0, s->cache,
                  s->q_idx, s->n_q, heads_I, s->group, base + L.qpack, err, stream);
    if (st != CSA2_OK) return st;
    st = run_index(s->cache, base + L.qpack, s->w, heads_I, s->req, s->n_visible, s->n_q, s->group, s->t_max, scores,
                   ld, err, stream, true, s->new_req, s->new_pos, mode == kFull ? s->n_new : 0);
    if (st != CSA2_OK) return st;
    st = run_topk_cluster(scores, ld, s->n_visible, s->n_q, s->t_max, s->topk, s->topk_idx, err, stream);
    if (st != CSA2_OK) return st;
    if (pool) {  // attention first; the pool serves later layers
      if ((st = run_attn(*s, base, L, err, stream)) != CSA2_OK) return st;
      return run_pool(scores, ld, s->n_visible, s->n_q, s->t_max, L, base, s->pool, err, stream);
    }
  }
  return run_attn(*s, base, L, err, stream);
}

}  // namespace

extern "C" {

const char* csa2_last_error(void) { return g_last_error.c_str(); }

size_t csa2_workspace_bytes(int64_t n_q, int32_t heads_I, int64_t t_max, int32_t scores_in_ws) {
  if (n_q < 0 || t_max < 0) return 0;
  return ws_layout(n_q, heads_I > 0 ? heads_I : 64, t_max, scores_in_ws).total;
}

size_t csa2_workspace_bytes_pool(int64_t n_q, int32_t heads_I, int64_t t_max, int32_t scores_in_ws) {
  if (n_q < 0 || t_max < 0) return 0;
  return ws_layout(n_q, heads_I > 0 ? heads_I : 64, t_max, scores_in_ws, true).total;
}

csa2_status csa2_pack_kv(const void* latent, const void* idx_key, const int32_t* req, const int64_t* pos, int64_t n,
                         const csa2_cache* cache, void* ws, size_t ws_bytes, csa2_stream_t stream) {
  if (n < 0) return fail(CSA2_ERR_INVALID_ARG, "n must be >= 0");
  csa2_status st = check_cache(cache, true, true);
  if (st != CSA2_OK) return st;
  if ((st = check_ws(ws, ws_bytes, kHeader)) != CSA2_OK) return st;
  if (n == 0) return CSA2_OK;
  if (!latent || !idx_key || !aligned(latent, 16) || !aligned(idx_key, 16) || !req || !pos)
    return fail(CSA2_ERR_INVALID_ARG, "latent/idx_key (16-byte aligned), req and pos are required");
  return run_pack(latent, idx_key, req, pos, n, *cache, nullptr, 0, 64, 1, nullptr, err_word(ws),
                  reinterpret_cast<cudaStream_t>(stream));
}

csa2_status csa2_pack_window(const void* rows, const int32_t* req, const int64_t* pos, int64_t n, uint8_t* ring,
                             int32_t n_ring, void* ws, size_t ws_bytes, csa2_stream_t stream) {
  if (n < 0) return fail(CSA2_ERR_INVALID_ARG, "n must be >= 0");
  csa2_status st = check_ws(ws, ws_bytes, kHeader);
  if (st != CSA2_OK) return st;
  if (n == 0) return CSA2_OK;
  if (!rows || !aligned(rows, 16) || !req || !pos) return fail(CSA2_ERR_INVALID_ARG, "rows (16-byte aligned), req and pos are required");
  if (!ring || !aligned(ring, 16) || n_ring <= 0) return fail(CSA2_ERR_INVALID_ARG, "ring must be 16-byte aligned with n_ring > 0");
  WinPackArgs a{};
  a.rows = static_cast<const __nv_bfloat16*>(rows);
  a.req = req;
  a.pos = pos;
  a.n = n;
  a.ring = ring;
  a.n_ring = n_ring;
  a.err = err_word(ws);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  trace_begin(kPackWindow, s);
  const cudaError_t e = launch_pack_window(a, s);
  trace_end(kPackWindow, s);
  return e == cudaSuccess ? CSA2_OK : cuda_fail(e, "window pack kernel");
}

csa2_status csa2_index_score(const void* q_idx, const float* w, int32_t heads_I, const int32_t* req,
                             const int32_t* n_visible, int64_t n_q, int32_t group, int64_t t_max,
                             const csa2_cache* cache, float* scores, int64_t ld, void* ws, size_t ws_bytes,
                             csa2_stream_t stream) {
  if (n_q < 0) return fail(CSA2_ERR_INVALID_ARG, "n_q must be >= 0");
  if (heads_I != 64 && heads_I != 32) return fail(CSA2_ERR_UNSUPPORTED, "heads_I must be 64 or 32");
  if (group != 1 && group != 2) return fail(CSA2_ERR_UNSUPPORTED, "group must be 1 or 2");
  csa2_status st = check_cache(cache, false, true);
  if (st != CSA2_OK) return st;
  if (t_max < 0 || t_max > static_cast<int64_t>(cache->max_pages) * kPage)
    return fail(CSA2_ERR_INVALID_ARG, "t_max outside [0, max_pages*128]");
  if (n_q > 0 && (!q_idx || !aligned(q_idx, 16) || !w || !req || !n_visible))
    return fail(CSA2_ERR_INVALID_ARG, "q_idx (16-byte aligned), w, req and n_visible are required");
  if (n_q > 0 && (!scores || ld < t_max || ld % 4 != 0 || !aligned(scores, 16)))
    return fail(CSA2_ERR_INVALID_ARG, "scores needs ld >= t_max, ld %% 4 == 0 and 16-byte alignment");
  const WsLayout L = ws_layout(n_q, heads_I, t_max, 0);
  if ((st = check_ws(ws, ws_bytes, L.total)) != CSA2_OK) return st;
  uint8_t* base = static_cast<uint8_t*>(ws);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  st = run_pack(nullptr, nullptr, nullptr, nullptr, 0, *cache, q_idx, n_q, heads_I, group, base + L.qpack,
                err_word(ws), s);
  if (st != CSA2_OK) return st;
  return run_index(*cache, base + L.qpack, w, heads_I, req, n_visible, n_q, group, t_max, scores, ld, err_word(ws), s,
                   true);
}

csa2_status csa2_topk(const float* scores, int64_t ld, const int32_t* n_visible, int64_t n_q, int64_t t_max,
                      int32_t k, int32_t* out_idx, void* ws, size_t ws_bytes, csa2_stream_t stream) {
  if (n_q < 0 || t_max < 0) return fail(CSA2_ERR_INVALID_ARG, "n_q and t_max must be >= 0");
  if (k != CSA2_TOPK) return fail(CSA2_ERR_UNSUPPORTED, "k must be 512 (got %d)", k);
  if (n_q > 0 && (!scores || !n_visible || !out_idx || ld < t_max || ld % 4 != 0 || !aligned(scores, 16)))
    return fail(CSA2_ERR_INVALID_ARG, "scores (16-byte aligned, ld >= t_max, ld %% 4 == 0), n_visible and out_idx are required");
  const WsLayout L = ws_layout(n_q, 64, t_max, 0);
  csa2_status st = check_ws(ws, ws_bytes, L.total);
  if (st != CSA2_OK) return st;
  return run_topk_cluster(scores, ld, n_visible, n_q, t_max, k, out_idx, err_word(ws),
                          reinterpret_cast<cudaStream_t>(stream));
}

csa2_status csa2_sparse_attn_full(const csa2_step* step, void* ws, size_t ws_bytes, csa2_stream_t stream) {
  return run_step(step, kFull, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

csa2_status csa2_sparse_attn_reindex(const csa2_step* step, void* ws, size_t ws_bytes, csa2_stream_t stream) {
  return run_step(step, kReindex, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

csa2_status csa2_sparse_attn_reuse(const csa2_step* step, void* ws, size_t ws_bytes, csa2_stream_t stream) {
  return run_step(step, kReuse, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

csa2_status csa2_check(void* ws, csa2_stream_t stream, int32_t* info) {
  if (ws == nullptr) return fail(CSA2_ERR_WORKSPACE, "workspace is NULL");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t h[2] = {0, 0};
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpy(h, ws, sizeof(h), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(ws, 0, sizeof(h));
  if (e != cudaSuccess) return cuda_fail(e, "csa2_check");
  if (info) *info = h[1];
  if (h[0] == 0) return CSA2_OK;
  return static_cast<csa2_status>(h[0]) == CSA2_ERR_TIMEOUT
             ? fail(CSA2_ERR_TIMEOUT, "a device-side wait ran out (info %d)", h[1])
             : fail(CSA2_ERR_DEVICE, "a device-side limit check failed (info %d)", h[1]);
}

int64_t csa2_launch_count(void) { return g_launches.load(); }

csa2_status csa2_debug_set_wait_limit(uint64_t ns) {
  g_wait_ns.store(ns, std::memory_order_relaxed);
  return CSA2_OK;
}

csa2_status csa2_probe_mma(int32_t kind, int32_t n, int32_t iters, int32_t issuers, int32_t n_ctas, int64_t* cycles,
                           csa2_stream_t stream) {
  if (kind != 0 && kind != 1) return fail(CSA2_ERR_INVALID_ARG, "kind must be 0 (f16) or 1 (NVFP4)");
  if (n != 64 && n != 128 && n != 256) return fail(CSA2_ERR_INVALID_ARG, "n must be 64, 128 or 256");
  if (issuers < 1 || issuers > 4 || issuers * n > 448)
    return fail(CSA2_ERR_INVALID_ARG, "issuers must be 1..4 with issuers * n <= 448");
  if (iters < 1 || iters > (1 << 22)) return fail(CSA2_ERR_INVALID_ARG, "iters must be in [1, 2^22]");
  if (n_ctas < 1 || cycles == nullptr || !aligned(cycles, 8))
    return fail(CSA2_ERR_INVALID_ARG, "n_ctas >= 1 and an 8-byte aligned cycles array are required");
  const cudaError_t e = launch_probe_mma(kind, n, iters, issuers, n_ctas, reinterpret_cast<long long*>(cycles),
                                         reinterpret_cast<cudaStream_t>(stream));
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return e == cudaSuccess ? CSA2_OK : cuda_fail(e, "probe kernel");
}

csa2_status csa2_trace_enable(int32_t on) {
  std::lock_guard<std::mutex> lk(g_trace.mu);
  if (on && !g_trace.on) {
    if (g_trace.ev.empty()) {
      g_trace.ev.resize(2 * kTraceCap);
      g_trace.kind.resize(kTraceCap);
      for (auto& ev : g_trace.ev) {
        const cudaError_t e = cudaEventCreate(&ev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreate");
      }
    }
    g_trace.n = 0;
    g_trace.on = true;
  } else if (!on) {
    g_trace.on = false;
    g_trace.n = 0;
  }
  return CSA2_OK;
}

csa2_status csa2_trace_read(int32_t kind, double* total_ms, int64_t* count) {
  std::lock_guard<std::mutex> lk(g_trace.mu);
  double sum = 0.0;
  int64_t n = 0;
  for (int i = 0; i < g_trace.n; ++i) {
    if (g_trace.kind[i] != kind) continue;
    cudaError_t e = cudaEventSynchronize(g_trace.ev[2 * i + 1]);
    float ms = 0.0f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, g_trace.ev[2 * i], g_trace.ev[2 * i + 1]);
    if (e != cudaSuccess) return cuda_fail(e, "csa2_trace_read");
    sum += ms;
    ++n;
  }
  if (total_ms) *total_ms = sum;
  if (count) *count = n;
  return CSA2_OK;
}

}  // extern "C"

// ----------------------------------------------------------------------------
// csa2_topk_noalloc: the top-k of csa2_topk with its scratch in a fixed device array
// inside the library instead of a caller workspace, for callers that cannot allocate
// device memory.  It allocates nothing.
extern "C" csa2_status csa2_topk_noalloc(const float* scores, int64_t ld, const int32_t* n_visible, int64_t n_q,
                                         int64_t t_max, int32_t k, int32_t* out_idx, csa2_stream_t stream) {
  if (n_q < 0 || t_max < 0) return fail(CSA2_ERR_INVALID_ARG, "n_q and t_max must be >= 0");
  if (n_q > kStaticTopkRows)
    return fail(CSA2_ERR_WORKSPACE, "csa2_topk_noalloc handles at most %lld rows per call (got %lld)",
                static_cast<long long>(kStaticTopkRows), static_cast<long long>(n_q));
  if (k != CSA2_TOPK) return fail(CSA2_ERR_UNSUPPORTED, "k must be 512 (got %d)", k);
  if (n_q > 0 && (!scores || !n_visible || !out_idx || ld < t_max || ld % 4 != 0 || !aligned(scores, 16)))
    return fail(CSA2_ERR_INVALID_ARG, "scores (16-byte aligned, ld >= t_max, ld %% 4 == 0), n_visible and out_idx are required");
  uint8_t* scratch = nullptr;
  size_t scratch_bytes = 0;
  cudaError_t e = topk_static_scratch(&scratch, &scratch_bytes);
  if (e != cudaSuccess) return cuda_fail(e, "csa2_topk_noalloc scratch lookup");
  if (scratch_bytes < kHeader + topk_ws_bytes(n_q)) return fail(CSA2_ERR_WORKSPACE, "static top-k scratch too small");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the error word starts clear on every call; the histograms are cleared by the launch
  e = cudaMemsetAsync(scratch, 0, kHeader, s);
  if (e != cudaSuccess) return cuda_fail(e, "csa2_topk_noalloc");
  return run_topk(scores, ld, n_visible, n_q, t_max, k, out_idx, scratch + kHeader, err_word(scratch), s);
}

// Reads and clears the error word of the fixed array behind csa2_topk_noalloc, after the
// stream has finished: the same report as csa2_check gives for a caller workspace.  It
// allocates nothing (a synchronous 8-byte copy and clear of the library's own array).
extern "C" csa2_status csa2_topk_noalloc_check(csa2_stream_t stream, int32_t* info) {
  uint8_t* scratch = nullptr;
  size_t scratch_bytes = 0;
  cudaError_t e = topk_static_scratch(&scratch, &scratch_bytes);
  if (e != cudaSuccess) return cuda_fail(e, "csa2_topk_noalloc_check scratch lookup");
  return csa2_check(scratch, stream, info);
}
