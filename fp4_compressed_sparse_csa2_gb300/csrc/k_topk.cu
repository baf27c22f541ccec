// k_topk.cu -- top-k selection over index scores.
//
// "DeepSeek's Attention and KV Cache - From MLA to CSA2", "DeepSeek-V3.2": selection is
// a top-k over the index scores; "DeepSeek-V4.1": k = 512.  "From MLA to DSA to
// HCA/CSA", "CSA: two changes to HCA": fewer than k visible entries leave -1 sentinels.
//
// Scores become order-preserving 32-bit keys (+0 and -0 equal).  Three launches, no
// inter-CTA waiting:
//   hist    (chunks x rows CTAs): 2048-bin histogram of the key's top 11 bits, smem
//           atomics, merged into a per-row global histogram;
//   select  (chunks x rows CTAs): every CTA derives the threshold bin b* (the bin that
//           holds the k-th largest key) from the row histogram, appends indices with a
//           higher bin to the row's selection and (key, index) pairs of bin b* to the
//           row's candidate list (warp-aggregated atomics);
//   final   (one CTA per row): sorts the candidates by (key desc, index asc), takes
//           the k - |selection| first, merges, sorts the k indices ascending, pads -1.
//           A row whose threshold bin overflows the candidate buffer (massive ties) is
//           resolved by exact radix refinement over the whole row instead.
// The result is unique: the k largest keys, equal keys by lower index.
#include <mutex>

#include "csa2_kernels.cuh"

namespace csa2 {

constexpr int kBins = 2048;
constexpr int kChunk = 8192;  // score entries per CTA in the hist and select passes
constexpr int kCandCap = 4096;
constexpr int kTopkThreads = 512;


__device__ __forceinline__ int64_t row_visible(const TopkArgs& a, int64_t q) {
  int64_t nv = __ldg(a.n_visible + q);
  if (nv < 0) nv = 0;
  if (nv > a.t_max) nv = a.t_max;
  return nv;
}

__global__ void __launch_bounds__(kTopkThreads) topk_hist_kernel(const TopkArgs a) {
  __shared__ uint32_t h[kBins];
  const int64_t q = blockIdx.y;
  const int64_t nv = row_visible(a, q);
  if (nv <= a.k) return;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kChunk;
  if (c0 >= nv) return;
  const int64_t c1 = c0 + kChunk < nv ? c0 + kChunk : nv;
  for (int b = threadIdx.x; b < kBins; b += kTopkThreads) h[b] = 0;
  __syncthreads();
  const float* row = a.scores + q * a.ld;
  if (c1 - c0 == kChunk) {  // full chunk: 4 float4 per thread, all loads in flight together
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = __ldg(reinterpret_cast<const float4*>(row + c0) + threadIdx.x + u * kTopkThreads);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      atomicAdd(&h[order_key(v[u].x) >> 21], 1u);
      atomicAdd(&h[order_key(v[u].y) >> 21], 1u);
      atomicAdd(&h[order_key(v[u].z) >> 21], 1u);
      atomicAdd(&h[order_key(v[u].w) >> 21], 1u);
    }
  } else {
    for (int64_t i = c0 + threadIdx.x; i < c1; i += kTopkThreads) atomicAdd(&h[order_key(__ldg(row + i)) >> 21], 1u);
  }
  __syncthreads();
  uint32_t* gh = a.hist + q * kBins;
  for (int b = threadIdx.x; b < kBins; b += kTopkThreads)
    if (h[b]) atomicAdd(gh + b, h[b]);
}

// The bin holding the k-th largest key and the number of keys in higher bins.
// h: smem histogram; 512 threads.  Thread t owns bins 4t .. 4t+3; suffix sums run over
// a warp with shuffles, then over the 16 warp totals in warp 0.
__device__ void threshold_bin(const uint32_t* h, uint32_t k, int* s_bin, uint32_t* s_above, uint32_t* s_warp) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  if (t == 0) {  // defaults when no bin reaches k (a histogram of fewer than k keys)
    *s_bin = 0;
    *s_above = 0;
  }
  const uint32_t loc = h[4 * t] + h[4 * t + 1] + h[4 * t + 2] + h[4 * t + 3];
  uint32_t x = loc;  // inclusive suffix within the warp
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t v = __shfl_down_sync(0xffffffffu, x, off);
    if (lane + off < 32) x += v;
  }
  if (lane == 0) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {  // exclusive suffix over the warp totals: keys in the warps above
    constexpr int kW = kTopkThreads / 32;
    const uint32_t tot = lane < kW ? s_warp[lane] : 0u;
    uint32_t y = tot;
#pragma unroll
    for (int off = 1; off < kW; off <<= 1) {
      const uint32_t v = __shfl_down_sync(0xffffffffu, y, off);
      if (lane + off < kW) y += v;
    }
    __syncwarp();
    if (lane < kW) s_warp[kW + lane] = y - tot;
  }
  __syncthreads();
  uint32_t running = x - loc + s_warp[kTopkThreads / 32 + warp];  // keys in bins above 4t+3
  for (int b = 4 * t + 3; b >= 4 * t; --b) {
    if (running < k && running + h[b] >= k) {
      *s_bin = b;
      *s_above = running;
    }
    running += h[b];
  }
  __syncthreads();
}

__device__ __forceinline__ void append(uint32_t* counter, bool pred, uint32_t& slot) {
  const uint32_t m = __ballot_sync(0xffffffffu, pred);
  if (m == 0) return;
  const int lane = threadIdx.x & 31;
  const int leader = __ffs(m) - 1;
  uint32_t base = 0;
  if (lane == leader) base = atomicAdd(counter, static_cast<uint32_t>(__popc(m)));
  base = __shfl_sync(0xffffffffu, base, leader);
  slot = base + __popc(m & ((1u << lane) - 1u));
}

__global__ void __launch_bounds__(kTopkThreads) topk_select_kernel(const TopkArgs a) {
  __shared__ uint32_t h[kBins];
  __shared__ uint32_t s_warp[32];
  __shared__ int s_bin;
  __shared__ uint32_t s_above;
  const int64_t q = blockIdx.y;
  const int64_t nv = row_visible(a, q);
  if (nv <= a.k) return;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kChunk;
  if (c0 >= nv) return;
  const int64_t c1 = c0 + kChunk < nv ? c0 + kChunk : nv;
  const uint32_t* gh = a.hist + q * kBins;
  for (int b = threadIdx.x; b < kBins; b += kTopkThreads) h[b] = gh[b];
  __syncthreads();
  threshold_bin(h, static_cast<uint32_t>(a.k), &s_bin, &s_above, s_warp);
  const uint32_t bstar = static_cast<uint32_t>(s_bin);
  const float* row = a.scores + q * a.ld;
  int32_t* sel = a.sel + q * a.k;
  uint2* cand = a.cand + q * kCandCap;
  // all of this thread's loads go out together (16 keys per thread for a full chunk);
  // the warp votes below see every lane
  constexpr int kU = kChunk / (4 * kTopkThreads);
  float4 v[kU];
#pragma unroll
  for (int u = 0; u < kU; ++u) {
    const int64_t i0 = c0 + (static_cast<int64_t>(u) * kTopkThreads + threadIdx.x) * 4;
    if (i0 + 3 < c1) {
      v[u] = __ldg(reinterpret_cast<const float4*>(row + i0));
    } else {
      v[u].x = i0 + 0 < c1 ? __ldg(row + i0 + 0) : 0.0f;
      v[u].y = i0 + 1 < c1 ? __ldg(row + i0 + 1) : 0.0f;
      v[u].z = i0 + 2 < c1 ? __ldg(row + i0 + 2) : 0.0f;
      v[u].w = i0 + 3 < c1 ? __ldg(row + i0 + 3) : 0.0f;
    }
  }
#pragma unroll
  for (int u = 0; u < kU; ++u) {
    const int64_t i0 = c0 + (static_cast<int64_t>(u) * kTopkThreads + threadIdx.x) * 4;
    const uint32_t key[4] = {order_key(v[u].x), order_key(v[u].y), order_key(v[u].z), order_key(v[u].w)};
    bool in[4], any = false;
    uint32_t bin[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      in[j] = i0 + j < c1;
      bin[j] = key[j] >> 21;
      any |= in[j] && bin[j] >= bstar;
    }
    if (!__any_sync(0xffffffffu, any)) continue;  // the common case: nothing to keep here
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t slot;
      const bool hi = in[j] && bin[j] > bstar;
      append(&a.cnt[2 * q], hi, slot);
      if (hi && slot < static_cast<uint32_t>(a.k)) sel[slot] = static_cast<int32_t>(i0 + j);
      const bool eq = in[j] && bin[j] == bstar;
      append(&a.cnt[2 * q + 1], eq, slot);
      if (eq && slot < kCandCap) cand[slot] = make_uint2(key[j], static_cast<uint32_t>(i0 + j));
    }
  }
}

// Bitonic sort, ascending, of n (power of two) elements in shared memory.
template <typename T>
__device__ void bitonic_sort(T* v, int n) {
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n / 2; i += blockDim.x) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool up = ((lo & size) == 0);
        const T x = v[lo], y = v[hi];
        if ((x > y) == up) {
          v[lo] = y;
          v[hi] = x;
        }
      }
      __syncthreads();
    }
  }
}

// Exact selection over a whole row by radix refinement (rows whose threshold bin
// holds more than kCandCap keys).  Appends the chosen indices (beyond those already in
// `picked[0..n_picked)`, which hold every index of a bin above b*) to `picked`.
__device__ void refine_row(const TopkArgs& a, int64_t q, int64_t nv, uint32_t bstar, uint32_t need, uint32_t* h,
                           uint32_t* s_warp, int32_t* picked, uint32_t* n_picked) {
  __shared__ int s_bin;
  __shared__ uint32_t s_above;
  __shared__ uint32_t s_cnt;
  const float* row = a.scores + q * a.ld;
  uint32_t prefix = bstar, prefix_bits = 11;
  // levels: bits [10, 21) then [0, 10) of the key below the 11-bit prefix
  const int shifts[2] = {10, 0};
  const int widths[2] = {11, 10};
  for (int lv = 0; lv < 2; ++lv) {
    const int sh = shifts[lv], wd = widths[lv];
    for (int b = threadIdx.x; b < kBins; b += kTopkThreads) h[b] = 0;
    __syncthreads();
    for (int64_t i = threadIdx.x; i < nv; i += kTopkThreads) {
      const uint32_t key = order_key(__ldg(row + i));
      if ((key >> (32 - prefix_bits)) == prefix) atomicAdd(&h[(key >> sh) & ((1u << wd) - 1u)], 1u);
    }
    __syncthreads();
    threshold_bin(h, need, &s_bin, &s_above, s_warp);
    need -= s_above;
    prefix = (prefix << wd) | static_cast<uint32_t>(s_bin);
    prefix_bits += wd;
  }
  const uint32_t vstar = prefix;  // exact key of the k-th largest
  // keys above vstar that are inside bin b* (higher bins are already picked)
  for (int64_t base = 0; base < nv; base += kTopkThreads) {
    const int64_t i = base + threadIdx.x;
    const uint32_t key = i < nv ? order_key(__ldg(row + i)) : 0u;
    const bool take = i < nv && (key >> 21) == bstar && key > vstar;
    uint32_t slot;
    append(n_picked, take, slot);
    if (take && slot < static_cast<uint32_t>(a.k)) picked[slot] = static_cast<int32_t>(i);
  }
  // the `need` lowest indices whose key equals vstar, in index order
  if (threadIdx.x == 0) s_cnt = 0;
  __syncthreads();
  for (int64_t base = 0; base < nv; base += kTopkThreads) {
    const int64_t i = base + threadIdx.x;
    const bool eq = i < nv && order_key(__ldg(row + i)) == vstar;
    const uint32_t m = __ballot_sync(0xffffffffu, eq);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) s_warp[warp] = __popc(m);
    __syncthreads();
    uint32_t before = s_cnt;
    for (int w = 0; w < warp; ++w) before += s_warp[w];
    const uint32_t rank = before + __popc(m & ((1u << lane) - 1u));
    if (eq && rank < need) {
      const uint32_t slot = atomicAdd(n_picked, 1u);
      if (slot < static_cast<uint32_t>(a.k)) picked[slot] = static_cast<int32_t>(i);
    }
    __syncthreads();
    if (threadIdx.x == 0)
      for (int w = 0; w < kTopkThreads / 32; ++w) s_cnt += s_warp[w];
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kTopkThreads) topk_final_kernel(const TopkArgs a) {
  extern __shared__ __align__(16) uint8_t tk_smem[];
  uint64_t* cs = reinterpret_cast<uint64_t*>(tk_smem);                 // kCandCap composites
  uint32_t* h = reinterpret_cast<uint32_t*>(cs + kCandCap);            // kBins
  int32_t* picked = reinterpret_cast<int32_t*>(h + kBins);             // k (<= 512)
  __shared__ uint32_t s_warp[32];
  __shared__ int s_bin;
  __shared__ uint32_t s_above;
  __shared__ uint32_t n_picked;
  const int64_t q = blockIdx.x;
  const int64_t nv = row_visible(a, q);
  int32_t* out = a.out + q * a.k;
  if (nv <= a.k) {
    for (int i = threadIdx.x; i < a.k; i += kTopkThreads) out[i] = i < nv ? i : -1;
    return;
  }
  for (int b = threadIdx.x; b < kBins; b += kTopkThreads) h[b] = a.hist[q * kBins + b];
  __syncthreads();
  threshold_bin(h, static_cast<uint32_t>(a.k), &s_bin, &s_above, s_warp);
  const uint32_t bstar = static_cast<uint32_t>(s_bin), above = s_above;
  const uint32_t nc = h[bstar];
  const uint32_t need = static_cast<uint32_t>(a.k) - above;
  if (threadIdx.x == 0) {
    if (a.cnt[2 * q] != above || a.cnt[2 * q + 1] != nc) report(a.err, CSA2_ERR_DEVICE, kInfoTopkIdx);
    n_picked = above;
  }
  for (uint32_t i = threadIdx.x; i < above; i += kTopkThreads) picked[i] = a.sel[q * a.k + i];
  __syncthreads();
  if (nc <= 1024) {
    // rank each candidate among all candidates by (key desc, index asc): no sort stages
    const uint2* cand = a.cand + q * kCandCap;
    for (uint32_t i = threadIdx.x; i < nc; i += kTopkThreads) {
      const uint2 c = cand[i];
      cs[i] = (static_cast<uint64_t>(0xFFFFFFFFu - c.x) << 32) | c.y;
    }
    __syncthreads();
    for (uint32_t i = threadIdx.x; i < nc; i += kTopkThreads) {
      const uint64_t me = cs[i];
      uint32_t rank = 0;
      for (uint32_t j = 0; j < nc; ++j) rank += cs[j] < me;
      if (rank < need) picked[above + rank] = static_cast<int32_t>(me & 0xFFFFFFFFu);
    }
    __syncthreads();
  } else if (nc <= kCandCap) {
    int p2 = 1;
    while (p2 < static_cast<int>(nc)) p2 <<= 1;
    const uint2* cand = a.cand + q * kCandCap;
    for (int i = threadIdx.x; i < p2; i += kTopkThreads) {
      if (i < static_cast<int>(nc)) {
        const uint2 c = cand[i];
        cs[i] = (static_cast<uint64_t>(0xFFFFFFFFu - c.x) << 32) | c.y;
      } else {
        cs[i] = ~0ull;
      }
    }
    __syncthreads();
    bitonic_sort(cs, p2);
    for (uint32_t i = threadIdx.x; i < need; i += kTopkThreads) picked[above + i] = static_cast<int32_t>(cs[i] & 0xFFFFFFFFu);
    __syncthreads();
  } else {
    refine_row(a, q, nv, bstar, need, h, s_warp, picked, &n_picked);
    __syncthreads();
  }
  // ascending order of the k chosen (distinct) indices: each index's rank is the number
  // of smaller ones
  for (int i = threadIdx.x; i < a.k; i += kTopkThreads) {
    const int32_t me = picked[i];
    int rank = 0;
    for (int j = 0; j < a.k; ++j) rank += picked[j] < me;
    out[rank] = me;
  }
}

size_t topk_final_smem() { return kCandCap * sizeof(uint64_t) + kBins * sizeof(uint32_t) + 512 * sizeof(int32_t); }

size_t topk_ws_bytes(int64_t n_q) {
  return static_cast<size_t>(n_q) * (kBins * 4 + 8 + 512 * 4 + kCandCap * 8);
}

void topk_carve(uint8_t* base, int64_t n_q, TopkArgs& a) {
  a.hist = reinterpret_cast<uint32_t*>(base);
  a.cnt = a.hist + n_q * kBins;
  a.sel = reinterpret_cast<int32_t*>(a.cnt + 2 * n_q);
  a.cand = reinterpret_cast<uint2*>(a.sel + 512 * n_q);
}

size_t topk_zero_bytes(int64_t n_q) { return static_cast<size_t>(n_q) * (kBins * 4 + 8); }

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t stream, int kind_hist, int kind_sel, int kind_final,
                        TraceFn trace_begin, TraceFn trace_end) {
  if (a.n_q == 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(a.hist, 0, topk_zero_bytes(a.n_q), stream);
  if (e != cudaSuccess) return e;
  const int chunks = static_cast<int>((a.t_max + kChunk - 1) / kChunk);
  if (chunks > 0) {
    const dim3 grid(chunks, static_cast<unsigned>(a.n_q));
    trace_begin(kind_hist, stream);
    topk_hist_kernel<<<grid, kTopkThreads, 0, stream>>>(a);
    trace_end(kind_hist, stream);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    trace_begin(kind_sel, stream);
    topk_select_kernel<<<grid, kTopkThreads, 0, stream>>>(a);
    trace_end(kind_sel, stream);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const size_t smem = topk_final_smem();
  static std::atomic<int> limit_set[kMaxDevices];
  e = smem_limit_once(reinterpret_cast<const void*>(topk_final_kernel), smem, limit_set);
  if (e != cudaSuccess) return e;
  trace_begin(kind_final, stream);
  topk_final_kernel<<<static_cast<unsigned>(a.n_q), kTopkThreads, smem, stream>>>(a);
  trace_end(kind_final, stream);
  return cudaGetLastError();
}

}  // namespace csa2

// ----------------------------------------------------------------------------
// Fixed scratch for the no-allocation top-k entry point (csa2_topk_noalloc).
// A file-scope device array: every GPU that loads the library holds it until the
// process exits.  Host code cannot pass the array's name to a kernel (on the host it
// is only a stand-in symbol), so the device address is looked up once per device with
// cudaGetSymbolAddress and cached.
namespace csa2 {

constexpr size_t kStaticScratchBytes = 256 + static_cast<size_t>(kStaticTopkRows) * (kBins * 4 + 8 + 512 * 4 + kCandCap * 8);
static __device__ __align__(256) uint8_t g_topk_scratch[kStaticScratchBytes];

cudaError_t topk_static_scratch(uint8_t** ptr, size_t* bytes) {
  static std::mutex mu;
  static uint8_t* addr[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_topk_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = static_cast<uint8_t*>(p);
  }
  *ptr = addr[dev];
  *bytes = kStaticScratchBytes;
  return cudaSuccess;
}

}  // namespace csa2

// ----------------------------------------------------------------------------
// Cluster top-k: one launch, one thread-block cluster of C CTAs per score row.
// Each CTA histograms its chunk; the cluster sums the histograms through distributed
// shared memory; each CTA re-reads its chunk and appends the indices above the
// threshold bin and the candidates inside it to the leader CTA's shared memory; the
// leader resolves the threshold bin exactly and writes the row.  No workspace, no
// polling: the only waits are hardware cluster barriers.
namespace csa2 {

constexpr int kClCandCap = 4096;   // leader: candidates of the threshold bin
constexpr int kClLocalCap = 4096;  // per CTA: staged candidates (long rows on 2-CTA clusters stage ~1.5 K)
constexpr int kClBlockCap = 4352;  // per CTA: block maxima (32-entry blocks) of the chunk (133,120-entry chunks fit)

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t dsmem_map(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ uint32_t dsmem_atom_add(uint32_t addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ uint4 dsmem_ld4(uint32_t addr) {  // 16-byte aligned
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ void dsmem_st(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void dsmem_st2(uint32_t addr, uint32_t x, uint32_t y) {
  asm volatile("st.shared::cluster.v2.u32 [%0], {%1, %2};" ::"r"(addr), "r"(x), "r"(y) : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}


// Sorts the k = 512 distinct indices in v (one per thread; padding INT_MAX) ascending
// and writes the first k to out: each warp sorts its 32 with a shuffle network, then an
// element's position is the number of smaller elements over all 16 sorted runs (binary
// searches), so only one block barrier is needed.
__device__ void sort_indices_out(int32_t v, int32_t* runs, int32_t* out, int k) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const int32_t o = __shfl_xor_sync(0xffffffffu, v, stride);
      const bool up = (lane & size) == 0 || size == 32;
      const bool low = (lane & stride) == 0;
      v = (low == up) ? min(v, o) : max(v, o);
    }
  }
  runs[threadIdx.x] = v;
  __syncthreads();
  int pos = lane;  // smaller elements of this warp's run
  int lo[kTopkThreads / 32];  // the 15 searches are independent: run them side by side
#pragma unroll
  for (int w = 0; w < kTopkThreads / 32; ++w) lo[w] = 0;
#pragma unroll
  for (int step = 16; step > 0; step >>= 1) {
#pragma unroll
    for (int w = 0; w < kTopkThreads / 32; ++w)
      if (runs[32 * w + lo[w] + step - 1] < v) lo[w] += step;
  }
#pragma unroll
  for (int w = 0; w < kTopkThreads / 32; ++w)
    if (w != warp) pos += lo[w] + (runs[32 * w + lo[w]] < v ? 1 : 0);
  if (pos < k && v != INT_MAX) out[pos] = v;
}


// Exact selection among candidate (key, index) pairs that contain the `need` largest
// keys: v* = the need-th largest key, found by radix selection on the key relative to
// the candidates' smallest key, 8 bits a level from the top of that range (about 3
// levels: a 256-bin histogram, then one warp finds the digit where the count from the
// top reaches the remaining need); keys above v* are taken, then the lowest indices
// among keys equal to v*.  Appends to sel starting at *n_picked.  h: 512 bins scratch
// (two histograms); ties: kBins scratch.  Returns false (nothing written) when the ties
// at v* do not fit.
__device__ bool select_candidates(const uint2* cand, uint32_t nc, uint32_t need, uint32_t* h, int32_t* ties,
                                  int32_t* sel, uint32_t* n_picked, uint32_t* n_ties_ctr) {
  __shared__ uint32_t s_lo, s_hi, s_digit, s_above;
  constexpr int kPer = kClCandCap / kTopkThreads;  // candidates per thread
  const uint32_t lane = threadIdx.x & 31;
  uint32_t key[kPer];
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const uint32_t i = threadIdx.x + j * kTopkThreads;
    key[j] = i < nc ? cand[i].x : 0u;
    if (i < nc) {
      kmin = min(kmin, key[j]);
      kmax = max(kmax, key[j]);
    }
  }
  if (threadIdx.x == 0) {
    s_lo = 0xFFFFFFFFu;
    s_hi = 0u;
  }
  for (uint32_t b = threadIdx.x; b < 512u; b += kTopkThreads) h[b] = 0u;  // both level histograms
  __syncthreads();
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if (lane == 0) {
    atomicMin(&s_lo, kmin);
    atomicMax(&s_hi, kmax);
  }
  __syncthreads();
  const uint32_t base = s_lo, span = s_hi - s_lo;  // relative keys d = key - base lie in [0, span]
  const int levels = span ? (32 - __clz(span) + 7) / 8 : 0;
  uint32_t prefix = 0, need_l = need;
  for (int lv = levels - 1; lv >= 0; --lv) {
    const int sh = 8 * lv;
    uint32_t* hc = h + 256 * (lv & 1);                  // this level's histogram (cleared before)
    uint32_t* hn = h + 256 * ((lv & 1) ^ 1);            // the next level's
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const uint32_t d = key[j] - base;
      const bool in = threadIdx.x + j * kTopkThreads < nc && (sh + 8 >= 32 || (d >> (sh + 8)) == prefix);
      if (in) atomicAdd(&hc[(d >> sh) & 255u], 1u);
    }
    if (threadIdx.x == 0) {  // defaults when no digit reaches need_l (inconsistent counts)
      s_digit = 0;
      s_above = 0;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // lane l owns digits 8l .. 8l+7; counts from the top of the range
      uint32_t c[8], loc = 0;
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        c[b] = hc[8 * lane + b];
        loc += c[b];
      }
      uint32_t x = loc;  // inclusive suffix over lanes
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t v = __shfl_down_sync(0xffffffffu, x, off);
        if (lane + off < 32) x += v;
      }
      uint32_t running = x - loc;  // keys with a larger digit
#pragma unroll
      for (int b = 7; b >= 0; --b) {
        if (running < need_l && running + c[b] >= need_l) {
          s_digit = 8 * lane + static_cast<uint32_t>(b);
          s_above = running;
        }
        running += c[b];
      }
    } else if (threadIdx.x < 32 + 256) {
      hn[threadIdx.x - 32] = 0u;
    }
    __syncthreads();
    prefix = (prefix << 8) | s_digit;
    need_l -= s_above;
  }
  const uint32_t vstar = base + prefix;
  const uint32_t start = *n_picked;
  if (threadIdx.x == 0) *n_ties_ctr = 0;
  __syncthreads();
  // appends with one shared atomic per warp and list (a per-thread atomic on one counter
  // serialises hundreds of updates)
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const uint32_t i = threadIdx.x + j * kTopkThreads;
    const bool hi = i < nc && key[j] > vstar, eq = i < nc && key[j] == vstar;
    uint32_t slot = 0;
    append(n_picked, hi, slot);
    if (hi && slot < static_cast<uint32_t>(CSA2_TOPK)) sel[slot] = static_cast<int32_t>(cand[i].y);
    append(n_ties_ctr, eq, slot);
    if (eq && slot < static_cast<uint32_t>(kBins)) ties[slot] = static_cast<int32_t>(cand[i].y);
  }
  __syncthreads();
  const uint32_t n_ties = *n_ties_ctr;
  __syncthreads();
  if (n_ties > static_cast<uint32_t>(kBins)) return false;  // block-uniform
  if (n_ties > 1) {
    int p2 = 1;
    while (p2 < static_cast<int>(n_ties)) p2 <<= 1;
    for (int i = static_cast<int>(n_ties) + threadIdx.x; i < p2; i += kTopkThreads) ties[i] = 0x7FFFFFFF;
    __syncthreads();
    bitonic_sort(ties, p2);
  }
  const uint32_t taken = start + (need - need_l);  // keys above v*
  const uint32_t n_take = need_l < n_ties ? need_l : n_ties;
  for (uint32_t i = threadIdx.x; i < n_take; i += kTopkThreads)
    if (taken + i < static_cast<uint32_t>(CSA2_TOPK)) sel[taken + i] = ties[i];
  __syncthreads();
  if (threadIdx.x == 0) *n_picked = start + need;
  __syncthreads();
  return true;
}

// Exact top-k of a whole row by one CTA (inputs whose candidates overflow the buffers):
// the row's 11-bit histogram, the entries of higher bins, then refine_row.
__device__ void full_row_select(const TopkArgs& a, int64_t q, int64_t nv, uint32_t* h, uint32_t* s_warp, int32_t* sel,
                                uint32_t* n_picked) {
  __shared__ int s_bin;
  __shared__ uint32_t s_above;
  const float* row = a.scores + q * a.ld;
  for (int b = threadIdx.x; b < kBins; b += kTopkThreads) h[b] = 0;
  __syncthreads();
  for (int64_t i = threadIdx.x; i < nv; i += kTopkThreads) atomicAdd(&h[order_key(__ldg(row + i)) >> 21], 1u);
  __syncthreads();
  threshold_bin(h, static_cast<uint32_t>(a.k), &s_bin, &s_above, s_warp);
  const uint32_t bstar = static_cast<uint32_t>(s_bin), above = s_above;
  if (threadIdx.x == 0) *n_picked = 0;
  __syncthreads();
  for (int64_t base = 0; base < nv; base += kTopkThreads) {
    const int64_t i = base + threadIdx.x;
    const bool take = i < nv && (order_key(__ldg(row + i)) >> 21) > bstar;
    uint32_t slot = 0;
    append(n_picked, take, slot);
    if (take && slot < static_cast<uint32_t>(a.k)) sel[slot] = static_cast<int32_t>(i);
  }
  __syncthreads();
  refine_row(a, q, nv, bstar, static_cast<uint32_t>(a.k) - above, h, s_warp, sel, n_picked);
  __syncthreads();
}

// Adds the lanes' entries flagged in msk (bit 4u + j = entry j of float4 u) to a
// shared list with one packed warp scan and one shared atomic per warp.
template <typename Emit>
__device__ __forceinline__ void warp_append(uint32_t msk, uint32_t* counter, Emit emit) {
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t mine = static_cast<uint32_t>(__popc(msk));
  uint32_t incl = mine;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= static_cast<uint32_t>(off)) incl += o;
  }
  uint32_t b = 0;
  if (lane == 31 && incl) b = atomicAdd(counter, incl);
  b = __shfl_sync(0xffffffffu, b, 31);
  uint32_t slot = b + incl - mine;
  while (msk) {
    const uint32_t bit = __ffs(msk) - 1;
    emit(bit, slot);
    ++slot;
    msk &= msk - 1u;
  }
}

// Stages the keys of bin >= bstar from the listed 32-entry blocks of row[c0, c1): 8
// lanes per block, 4 blocks per warp and kRounds such groups of loads in flight per lane;
// (key, index) pairs go to cand[0, cap) through one packed warp scan per append
// (*counter counts every pair, also those beyond cap).
template <uint32_t kRounds>
__device__ __forceinline__ void gather_block_candidates(const float* row, int64_t c0, int64_t c1, const uint32_t* blist,
                                                        uint32_t nbl, uint32_t bstar, uint2* cand, uint32_t cap,
                                                        uint32_t* counter) {
  const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5, grp = lane >> 3;
  constexpr uint32_t kStride = 4 * (kTopkThreads / 32);
  for (uint32_t r0 = warp * 4; r0 < nbl; r0 += kRounds * kStride) {
    float4 v[kRounds];
    int64_t i0[kRounds];
    bool ok[kRounds];
#pragma unroll
    for (uint32_t u = 0; u < kRounds; ++u) {
      const uint32_t r = r0 + u * kStride + grp;
      ok[u] = r < nbl;
      i0[u] = c0 + static_cast<int64_t>(ok[u] ? blist[r] : 0u) * 32 + (lane & 7u) * 4;
      v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (ok[u] && i0[u] + 3 < c1) {
        v[u] = __ldg(reinterpret_cast<const float4*>(row + i0[u]));
      } else if (ok[u]) {
        v[u].x = i0[u] + 0 < c1 ? __ldg(row + i0[u] + 0) : 0.0f;
        v[u].y = i0[u] + 1 < c1 ? __ldg(row + i0[u] + 1) : 0.0f;
        v[u].z = i0[u] + 2 < c1 ? __ldg(row + i0[u] + 2) : 0.0f;
        v[u].w = i0[u] + 3 < c1 ? __ldg(row + i0[u] + 3) : 0.0f;
      }
    }
    // kRounds <= 8: 4 entries per round fit the 32-bit mask; bin >= b* is a plain float
    // comparison with the bin's lower edge
    const float lo = key_floor(bstar << 21);
    uint32_t msk = 0;
#pragma unroll
    for (uint32_t u = 0; u < kRounds; ++u) {
      const float vv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) msk |= (ok[u] && i0[u] + j < c1 && vv[j] >= lo) ? (1u << (4 * u + j)) : 0u;
    }
    if (!__any_sync(0xffffffffu, msk != 0)) continue;
    warp_append(msk, counter, [&](uint32_t bit, uint32_t slot) {
      const uint32_t u = bit >> 2, j = bit & 3u;
      float4 w = v[0];
      int64_t b = i0[0];
#pragma unroll
      for (uint32_t x = 1; x < kRounds; ++x)
        if (u == x) {
          w = v[x];
          b = i0[x];
        }
      const float e = j == 0 ? w.x : (j == 1 ? w.y : (j == 2 ? w.z : w.w));
      if (slot < cap) cand[slot] = make_uint2(order_key(e), static_cast<uint32_t>(b + j));
    });
  }
}

__global__ void __launch_bounds__(kTopkThreads, 2) topk_cluster_kernel(const TopkArgs a, int64_t chunk) {
  extern __shared__ __align__(16) uint8_t tc_smem[];
  uint32_t* h = reinterpret_cast<uint32_t*>(tc_smem);  // [2][kBins] histograms (lane parity); [1] later: block list
  uint32_t* hsum = h + 2 * kBins;                      // [kBins] row histogram
  uint32_t* ctr = hsum + kBins;                        // [4] leader: selected, candidates, picked, overflow
  uint32_t* lctr = ctr + 4;                            // [4] this CTA: staged selected, candidates, blocks, ties
  int32_t* sel = reinterpret_cast<int32_t*>(lctr + 4);  // [512] leader: chosen indices
  int32_t* lsel = sel + 512;                            // [512] this CTA: indices above the threshold bin
  uint2* cand = reinterpret_cast<uint2*>(lsel + 512);   // [kClCandCap] leader: (key, index)
  uint2* lcand = cand + kClCandCap;                     // [kClLocalCap] this CTA: (key, index)
  uint32_t* bm = reinterpret_cast<uint32_t*>(lcand + kClLocalCap);  // [kClBlockCap] block maxima of the chunk
  __shared__ uint32_t s_warp[32];
  __shared__ int s_bin;
  __shared__ uint32_t s_above;
  __shared__ uint32_t s_base[2];
  pdl_trigger();
  pdl_wait();  // the score rows come from the previous kernel
  const uint32_t rank = cluster_rank();
  const uint32_t csize = gridDim.x;  // one cluster spans the x dimension
  const uint32_t lane = threadIdx.x & 31;
  const int64_t q = blockIdx.y;
  const int64_t nv = row_visible(a, q);
  int32_t* out = a.out + q * a.k;
  if (nv <= a.k) {  // the whole row is selected (uniform across the cluster)
    if (rank == 0)
      for (int i = threadIdx.x; i < a.k; i += kTopkThreads) out[i] = i < nv ? i : -1;
    return;
  }
  const int64_t c0 = static_cast<int64_t>(rank) * chunk;
  const int64_t c1 = c0 + chunk < nv ? c0 + chunk : nv;
  // Long rows go by 32-entry block maxima: the k-th largest block maximum bounds the
  // k-th largest key from below (k blocks each hold a key at least that large), so only
  // blocks reaching the bound are read again.  That pays when the row has many more
  // blocks than k (with about k blocks the bound is the smallest block maximum and every
  // block is read again); shorter rows histogram every key.
  const bool by_blocks = (nv + 31) / 32 >= 4 * a.k && chunk / 32 <= kClBlockCap;  // uniform across the cluster
  for (int b = threadIdx.x; b < 2 * kBins; b += kTopkThreads) h[b] = 0;
  if (threadIdx.x < 8) ctr[threadIdx.x] = 0;  // ctr and lctr
  __syncthreads();
  const float* row = a.scores + q * a.ld;
  uint32_t* hl = h + (threadIdx.x & 1) * kBins;  // two copies halve the atomic contention on busy bins
  // ---- pass 1: histogram of the top 11 key bits of every key, or of every block maximum
  // (8 float4 per thread per round, all loads issued before the first is used; offsets
  // relative to the chunk in 32 bits, and full rounds without per-element bounds checks)
  {
    const int32_t len = c1 > c0 ? static_cast<int32_t>(c1 - c0) : 0;
    const float* crow = row + c0;
    for (int32_t base = 0; base < len; base += 32 * kTopkThreads) {
      float4 v[8];
      const bool full = base + 32 * kTopkThreads <= len;
      if (full) {
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = __ldg(reinterpret_cast<const float4*>(crow + base) + u * kTopkThreads + threadIdx.x);
      } else {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int32_t i0 = base + (u * kTopkThreads + static_cast<int32_t>(threadIdx.x)) * 4;
          if (i0 + 3 < len) {
            v[u] = __ldg(reinterpret_cast<const float4*>(crow + i0));
          } else {
            v[u].x = i0 + 0 < len ? __ldg(crow + i0 + 0) : NAN;
            v[u].y = i0 + 1 < len ? __ldg(crow + i0 + 1) : NAN;
            v[u].z = i0 + 2 < len ? __ldg(crow + i0 + 2) : NAN;
            v[u].w = i0 + 3 < len ? __ldg(crow + i0 + 3) : NAN;
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int32_t i0 = base + (u * kTopkThreads + static_cast<int32_t>(threadIdx.x)) * 4;
        const uint32_t k0 = full || i0 + 0 < len ? order_key(v[u].x) : 0u;
        const uint32_t k1 = full || i0 + 1 < len ? order_key(v[u].y) : 0u;
        const uint32_t k2 = full || i0 + 2 < len ? order_key(v[u].z) : 0u;
        const uint32_t k3 = full || i0 + 3 < len ? order_key(v[u].w) : 0u;
        if (by_blocks) {
          // lanes 8g .. 8g + 7 hold the 32 entries of one block
          uint32_t m = max(max(k0, k1), max(k2, k3));
          m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
          m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
          m = max(m, __shfl_xor_sync(0xffffffffu, m, 4));
          if ((lane & 7u) == 0 && i0 < len) {
            bm[i0 >> 5] = m;
            atomicAdd(&h[m >> 21], 1u);
          }
        } else {
          if (full || i0 + 0 < len) atomicAdd(&hl[k0 >> 21], 1u);
          if (full || i0 + 1 < len) atomicAdd(&hl[k1 >> 21], 1u);
          if (full || i0 + 2 < len) atomicAdd(&hl[k2 >> 21], 1u);
          if (full || i0 + 3 < len) atomicAdd(&hl[k3 >> 21], 1u);
        }
      }
    }
  }
  __syncthreads();
  for (int b = threadIdx.x; b < kBins; b += kTopkThreads) h[b] += h[kBins + b];
  cluster_sync_all();  // every CTA's histogram and the leader's counters are ready
  {
    static_assert(kBins == 4 * kTopkThreads, "one 16-byte histogram slice per thread");
    uint4 sum = make_uint4(0u, 0u, 0u, 0u);
    for (uint32_t r = 0; r < csize; ++r) {
      const uint4 v = dsmem_ld4(dsmem_map(&h[4 * threadIdx.x], r));
      sum.x += v.x;
      sum.y += v.y;
      sum.z += v.z;
      sum.w += v.w;
    }
    *reinterpret_cast<uint4*>(&hsum[4 * threadIdx.x]) = sum;
  }
  __syncthreads();
  threshold_bin(hsum, static_cast<uint32_t>(a.k), &s_bin, &s_above, s_warp);
  const uint32_t bstar = static_cast<uint32_t>(s_bin);
  if (by_blocks) {
    // ---- pass 2 (blocks): list the chunk's blocks whose maximum reaches bin b*, then
    // stage their keys of bin >= b* (8 lanes per block, 4 blocks per warp in flight)
    uint32_t* blist = h + kBins;  // the second histogram copy is free now
    // CTAs whose chunk starts past the row's end (c1 < c0) have no blocks
    const uint32_t nb = c1 > c0 ? static_cast<uint32_t>((c1 - c0 + 31) >> 5) : 0u;
    for (uint32_t base = 0; base < nb; base += kTopkThreads) {
      const uint32_t i = base + threadIdx.x;
      const bool take = i < nb && (bm[i] >> 21) >= bstar;
      uint32_t slot = 0;
      append(&lctr[2], take, slot);
      if (take && slot < kBins) blist[slot] = i;
    }
    __syncthreads();
    const uint32_t nbl = lctr[2] < static_cast<uint32_t>(kBins) ? lctr[2] : static_cast<uint32_t>(kBins);
    gather_block_candidates<6>(row, c0, c1, blist, nbl, bstar, lcand, kClLocalCap, &lctr[1]);
  } else {
    // ---- pass 2 (keys): stage this chunk's entries above / in the threshold bin (the
    // chunk is mostly still in L2)
    for (int64_t base = c0; base < c1; base += 16 * kTopkThreads) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t i0 = base + (static_cast<int64_t>(u) * kTopkThreads + threadIdx.x) * 4;
        if (i0 + 3 < c1) {
          v[u] = __ldg(reinterpret_cast<const float4*>(row + i0));
        } else {
          v[u].x = i0 + 0 < c1 ? __ldg(row + i0 + 0) : 0.0f;
          v[u].y = i0 + 1 < c1 ? __ldg(row + i0 + 1) : 0.0f;
          v[u].z = i0 + 2 < c1 ? __ldg(row + i0 + 2) : 0.0f;
          v[u].w = i0 + 3 < c1 ? __ldg(row + i0 + 3) : 0.0f;
        }
      }
      uint32_t mhi = 0, meq = 0;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t i0 = base + (static_cast<int64_t>(u) * kTopkThreads + threadIdx.x) * 4;
        const float vv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t bin = order_key(vv[j]) >> 21;
          const bool in = i0 + j < c1;
          mhi |= (in && bin > bstar) ? (1u << (4 * u + j)) : 0u;
          meq |= (in && bin == bstar) ? (1u << (4 * u + j)) : 0u;
        }
      }
      if (!__any_sync(0xffffffffu, (mhi | meq) != 0)) continue;
      auto entry = [&](uint32_t bit, float& x) {
        const int u = static_cast<int>(bit >> 2), j = static_cast<int>(bit & 3u);
        const float4 w = u == 0 ? v[0] : (u == 1 ? v[1] : (u == 2 ? v[2] : v[3]));
        x = j == 0 ? w.x : (j == 1 ? w.y : (j == 2 ? w.z : w.w));
        return base + (static_cast<int64_t>(u) * kTopkThreads + threadIdx.x) * 4 + j;
      };
      warp_append(mhi, &lctr[0], [&](uint32_t bit, uint32_t slot) {
        float x;
        const int64_t idx = entry(bit, x);
        if (slot < static_cast<uint32_t>(a.k)) lsel[slot] = static_cast<int32_t>(idx);
      });
      warp_append(meq, &lctr[1], [&](uint32_t bit, uint32_t slot) {
        float x;
        const int64_t idx = entry(bit, x);
        if (slot < kClLocalCap) lcand[slot] = make_uint2(order_key(x), static_cast<uint32_t>(idx));
      });
    }
  }
  __syncthreads();
  // ---- hand the staged lists to the leader (one shared-cluster atomic per list)
  const uint32_t l_ctr = dsmem_map(&ctr[0], 0), l_sel = dsmem_map(sel, 0), l_cand = dsmem_map(cand, 0);
  const uint32_t n_hi = lctr[0] < static_cast<uint32_t>(a.k) ? lctr[0] : static_cast<uint32_t>(a.k);
  const uint32_t n_eq = lctr[1];
  if (threadIdx.x == 0) {
    s_base[0] = n_hi ? dsmem_atom_add(l_ctr, n_hi) : 0u;
    s_base[1] = n_eq ? dsmem_atom_add(l_ctr + 4u, n_eq) : 0u;
    if (n_eq > kClLocalCap || lctr[2] > static_cast<uint32_t>(kBins))
      dsmem_st(l_ctr + 12u, 1u);  // a staged list overflowed: the leader selects over the whole row
  }
  __syncthreads();
  for (uint32_t i = threadIdx.x; i < n_hi; i += kTopkThreads)
    if (s_base[0] + i < static_cast<uint32_t>(a.k)) dsmem_st(l_sel + 4u * (s_base[0] + i), static_cast<uint32_t>(lsel[i]));
  const uint32_t n_eq_st = n_eq < kClLocalCap ? n_eq : kClLocalCap;
  for (uint32_t i = threadIdx.x; i < n_eq_st; i += kTopkThreads)
    if (s_base[1] + i < kClCandCap) dsmem_st2(l_cand + 8u * (s_base[1] + i), lcand[i].x, lcand[i].y);
  cluster_sync_all();  // every hand-off has landed in the leader
  if (rank != 0) return;
  // ---- leader: exact selection among the candidates
  const uint32_t above = by_blocks ? 0u : s_above;
  const uint32_t nc = ctr[1];
  if (!by_blocks && threadIdx.x == 0 && (ctr[0] != above || nc != hsum[bstar])) report(a.err, CSA2_ERR_DEVICE, kInfoTopkIdx);
  bool done = false;
  if (ctr[3] == 0 && nc <= static_cast<uint32_t>(kClCandCap)) {
    if (threadIdx.x == 0) ctr[2] = above;  // entries of higher bins are already in sel[0, above)
    __syncthreads();
    done = select_candidates(cand, nc, static_cast<uint32_t>(a.k) - above, h, reinterpret_cast<int32_t*>(hsum), sel,
                             &ctr[2], &lctr[3]);
  }
  if (!done) full_row_select(a, q, nv, h, s_warp, sel, &ctr[2]);
  // ascending output: a shuffle sort per warp, then each index's rank from binary searches
  // in the 16 sorted runs (one block barrier)
  __syncthreads();
  sort_indices_out(threadIdx.x < a.k ? sel[threadIdx.x] : INT_MAX, reinterpret_cast<int32_t*>(hsum), out, a.k);
}

size_t topk_cluster_smem() {
  return 3 * kBins * sizeof(uint32_t) + 8 * sizeof(uint32_t) + 2 * 512 * sizeof(int32_t) +
         (kClCandCap + kClLocalCap) * sizeof(uint2) + kClBlockCap * sizeof(uint32_t);
}

cudaError_t launch_topk_cluster(const TopkArgs& a, int sm_count, cudaStream_t stream) {
  if (a.n_q == 0) return cudaSuccess;
  const size_t smem = topk_cluster_smem();
  static std::atomic<int> limit_set[kMaxDevices];
  cudaError_t e = smem_limit_once(reinterpret_cast<const void*>(topk_cluster_kernel), smem, limit_set);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kTopkThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // Cluster size: the largest of 8, 4, 2, 1 whose clusters for all rows are resident at
  // once (one wave), with chunks of at least 8K entries; the resident-cluster counts are
  // queried once per device.
  static std::atomic<int> active[kMaxDevices][4];
  int dev = 0;
  cudaGetDevice(&dev);
  const int64_t by_len = (a.t_max + 8191) / 8192;
  int64_t c = 1;
  for (int lg = 3; lg >= 0; --lg) {
    const int64_t cc = int64_t(1) << lg;
    if (cc > by_len && cc > 1) continue;
    int n_act = (dev >= 0 && dev < kMaxDevices) ? active[dev][lg].load(std::memory_order_relaxed) : 0;
    if (n_act == 0) {
      cfg.gridDim = dim3(static_cast<unsigned>(cc), 1, 1);
      attr[0].val.clusterDim.x = static_cast<unsigned>(cc);
      if (cudaOccupancyMaxActiveClusters(&n_act, topk_cluster_kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n_act = -1;
      }
      if (dev >= 0 && dev < kMaxDevices) active[dev][lg].store(n_act == 0 ? -1 : n_act, std::memory_order_relaxed);
    }
    if (n_act > 0 && n_act >= a.n_q) {
      c = cc;
      break;
    }
  }
  if (c == 1) {
    // no size holds every row in one wave (many rows, e.g. a prefill chunk): take the
    // smallest cluster whose chunks fit the block-maximum path, which reads each long row
    // about once instead of histogramming every key and re-reading the row
    for (int64_t cc = 1; cc <= 8 && cc <= by_len; cc *= 2) {
      const int64_t ch = (((a.t_max + cc - 1) / cc + 2047) / 2048) * 2048;
      if (ch / 32 <= kClBlockCap) {
        c = cc;
        break;
      }
    }
  }
  (void)sm_count;
  int64_t chunk = (a.t_max + c - 1) / c;
  chunk = ((chunk + 2047) / 2048) * 2048;
  attr[0].val.clusterDim.x = static_cast<unsigned>(c);
  return launch_pdl(topk_cluster_kernel, dim3(static_cast<unsigned>(c), static_cast<unsigned>(a.n_q), 1),
                    dim3(kTopkThreads), smem, stream, &attr[0], a, chunk);
}


}  // namespace csa2
