// csa2_kernels.cuh -- argument blocks and launchers of the CSA2 kernels.
#pragma once

#include "csa2_dev.cuh"

#include <atomic>

namespace csa2 {

struct PackArgs {
  // new cache entries
  const __nv_bfloat16* latent;   // [n_new][512]
  const __nv_bfloat16* idx_key;  // [n_new][128]
  const int32_t* new_req;
  const int64_t* new_pos;
  int64_t n_new;
  csa2_cache cache;
  // indexer query groups
  const __nv_bfloat16* q_idx;  // [n_q][heads_I][128]
  int64_t n_q;
  int32_t heads_I;
  int32_t G;           // queries per group
  int32_t N;           // G * heads_I rows per group (<= 128)
  int32_t grp_bytes;   // N*64 + 1024
  int64_t n_groups;
  uint8_t* qpack;      // [n_groups][grp_bytes]
  int32_t* err;
};

struct IndexArgs {
  const uint8_t* idx_pages;
  csa2_cache cache;
  const uint8_t* qpack;
  int32_t grp_bytes;
  const float* w;
  const int32_t* req;
  const int32_t* n_visible;
  float* scores;
  int64_t ld;
  int64_t n_q;
  int32_t heads_I;
  int32_t G;
  int32_t N;
  int64_t n_groups;
  int32_t tpg;     // tiles (pages) per group
  int32_t stages;  // smem ring depth
  uint32_t tmem_cols;
  int32_t* err;
  uint64_t wait_ns;  // bound of each pipeline wait (csa2_debug_set_wait_limit)
  // early != 0: the previous kernel is this call's pack kernel, which starts the next
  // kernel only after everything before it has completed and writes only the cache
  // entries (new_req[i], new_pos[i]), i < n_new, and the packed queries; the producer may
  // then copy the first pages of its range that hold none of those entries before
  // griddepcontrol.wait
  const int32_t* new_req;
  const int64_t* new_pos;
  int64_t n_new;
  int32_t early;
};

struct TopkArgs {
  const float* scores;
  int64_t ld;
  const int32_t* n_visible;
  int64_t n_q;
  int32_t k;
  int32_t* out;
  uint32_t* hist;  // [n_q][kBins]
  uint32_t* cnt;   // [n_q][2]  selection count, candidate count
  int32_t* sel;    // [n_q][k]
  uint2* cand;     // [n_q][kCandCap]  (key, index)
  int64_t t_max;
  int32_t* err;
};

struct AttnArgs {
  const __nv_bfloat16* q;  // [n_q][64][512]
  const int32_t* topk_idx; // [n_q][512]
  const int32_t* n_visible;
  const int32_t* req;
  const __nv_bfloat16* window;
  const int64_t* win_start;
  const int32_t* win_len;
  csa2_cache cache;
  float scale_log2;  // softmax scale * log2(e)
  __nv_bfloat16* out;
  float* lse;
  int64_t n_q;
  int32_t* err;
  const float* sinks;     // [64] natural-log sink logits or nullptr
  const float* rope_cos;  // [n_q][32] or nullptr (then rope_sin too)
  const float* rope_sin;
  const uint8_t* win_ring;  // FP8 window ring [win_ring_reqs][128][528] or nullptr
  int32_t win_ring_reqs;
  // key splits: `splits` CTAs per query (one thread-block cluster) each take a run of the
  // tile list [window, selected 0..3]; they write raw partial outputs and per-head (max,
  // sum) to the workspace and combine them after a cluster barrier; 1 = one CTA per query
  int32_t splits;
  float* opart;  // [n_q * splits][64][512] (splits > 1)
  float* mpart;  // [n_q * splits][2][64]
  uint64_t wait_ns;  // bound of each pipeline wait (csa2_debug_set_wait_limit)
};

// Upper bound on the key splits of one query (its five 128-key tiles).
constexpr int kAttnMaxSplits = 5;
// Key splits that keep n_q queries' CTAs in one wave on sm_count SMs (before the cluster
// occupancy check), and the workspace bytes of their partials.
inline int attn_wave_splits(int64_t n_q, int sm_count) {
  if (n_q <= 0) return 1;
  const int64_t s = sm_count / n_q;
  return static_cast<int>(s < 1 ? 1 : (s > kAttnMaxSplits ? kAttnMaxSplits : s));
}
inline size_t attn_split_ws_bytes(int64_t n_q, int sm_count) {
  const int s = attn_wave_splits(n_q, sm_count);
  return s > 1 ? static_cast<size_t>(n_q) * s * 64 * (512 + 2) * sizeof(float) : 0;
}

struct WinPackArgs {
  const __nv_bfloat16* rows;  // [n][512]
  const int32_t* req;
  const int64_t* pos;
  int64_t n;
  uint8_t* ring;  // [n_ring][128][528]
  int32_t n_ring;
  int32_t* err;
};

struct PoolArgs {
  const float* scores;  // [n_q][ld] a Full layer's index scores
  int64_t ld;
  const int32_t* n_visible;
  int64_t n_q;
  uint32_t* bkey;  // [n_q][nb_cap] scratch: block-maximum keys
  int64_t nb_cap;  // ceil(t_max / 8)
  int64_t t_max;   // n_visible[] is clamped to it
  int32_t stage;   // set by the launcher: dynamic shared memory holds min(nb_cap, 32768) keys
  int32_t* pool;   // [n_q][16384] out: positions ascending, -1 padded
  int32_t* pool_len;  // [n_q] out
  int32_t* err;
};

struct GatherArgs {
  csa2_cache cache;  // the layer's cache (source pages)
  const int32_t* pool;  // [n_q][16384]
  const int32_t* req;
  const int32_t* n_visible;
  int64_t n_q;
  uint8_t* compact;   // [n_q][128 pages] compact indexer pages, same format as the cache
  int32_t* pool_len;  // [n_q] out: listed positions
  int32_t* req_q;     // [n_q] out: q (each query owns its compact pages)
  int32_t* err;
};

using TraceFn = void (*)(int, cudaStream_t);

// Launches `kernel` so that it may start while the previous kernel on the stream
// drains (programmatic stream serialization); the kernel must call pdl_wait() before
// touching the previous kernel's outputs or anything it reads.  extra: an optional
// further launch attribute (a cluster shape).
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       const cudaLaunchAttribute* extra, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int n = 1;
  if (extra != nullptr) attr[n++] = *extra;
  cfg.attrs = attr;
  cfg.numAttrs = static_cast<unsigned>(n);
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

cudaError_t launch_pack(const PackArgs& a, cudaStream_t stream);
size_t index_smem_bytes(int stages);
cudaError_t launch_index(const IndexArgs& a, int grid, cudaStream_t stream);
size_t topk_ws_bytes(int64_t n_q);
void topk_carve(uint8_t* base, int64_t n_q, TopkArgs& a);
cudaError_t launch_topk(const TopkArgs& a, cudaStream_t stream, int kind_hist, int kind_sel, int kind_final,
                        TraceFn trace_begin, TraceFn trace_end);
// No-allocation top-k: rows held by the fixed scratch, and its device address on the
// current device (looked up on first use per device).
constexpr int64_t kStaticTopkRows = 128;
constexpr int kMaxDevices = 64;

// Raises `kernel`'s dynamic shared-memory limit to `bytes` once per device; `cache` holds
// kMaxDevices entries of the limit already set.  cudaFuncSetAttribute on every launch
// leaves the GPU idle between back-to-back launches.
cudaError_t smem_limit_once(const void* kernel, size_t bytes, std::atomic<int>* cache);
// The pipeline-wait bound the kernels are launched with (csa2_debug_set_wait_limit; the
// default about 2 s).
uint64_t pipeline_wait_ns();
cudaError_t topk_static_scratch(uint8_t** ptr, size_t* bytes);
cudaError_t launch_topk_cluster(const TopkArgs& a, int sm_count, cudaStream_t stream);
size_t attn_smem_bytes();
// Key splits per query for n_q queries on sm_count SMs: the most (up to 5) that keep all CTAs
// in one wave and that the device can hold as one cluster (ext: the optional-feature kernel).
int attn_splits_for(int64_t n_q, int sm_count, bool ext);
cudaError_t launch_attn(const AttnArgs& a, cudaStream_t stream);
cudaError_t launch_pack_window(const WinPackArgs& a, cudaStream_t stream);
cudaError_t launch_probe_mma(int32_t kind, int32_t n, int32_t iters, int32_t issuers, int32_t n_ctas,
                             long long* cycles, cudaStream_t stream);
cudaError_t launch_pool_bmax(const PoolArgs& a, cudaStream_t stream);  // block maxima (first)
cudaError_t launch_pool(const PoolArgs& a, cudaStream_t stream);       // the selection
cudaError_t launch_gather(const GatherArgs& a, cudaStream_t stream);
cudaError_t launch_map(const int32_t* slots, const int32_t* pool, int32_t* out, int64_t n_q, cudaStream_t stream);

}  // namespace csa2
