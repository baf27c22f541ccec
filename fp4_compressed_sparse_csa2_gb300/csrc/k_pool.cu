// k_pool.cu -- hierarchical sparse indexer: a Full layer's candidate pool, and the
// compact indexer pages that a pool-restricted Reindex layer scores.
//
// "DeepSeek's Attention and KV Cache - From MLA to CSA2", "The hierarchical indexer";
// "From First Principles: DeepSeek-V4.1-Flash Inference", "The Hierarchical Sparse
// Indexer": the Full layer gives each block of 8 positions the maximum score inside it,
// keeps the 2,048 highest-scoring blocks and publishes their positions (at most 16,384)
// as a pool; each Reindex layer scores only the pool and takes its own top-512 from it,
// so its cost no longer grows with the context.
//
// bmax_kernel     block maxima of the score rows as order-preserving keys (scratch),
//                 2,048 blocks per 256-thread CTA, 8 independent blocks per thread.
// pool_kernel     one 1024-thread CTA per row over the keys only: exact radix selection
//                 of the 2,048th largest key (11 + 11 + 10 bits), then an ordered pass
//                 (warp ballots, warp-range prefix sums) that keeps the blocks above it
//                 plus the lowest-index blocks equal to it and writes their positions
//                 ascending.
// gather_kernel   one warp per 4 pooled blocks of 8 entries: each block's 512-byte nibble
//                 group and its scale bytes move from the cache page into a compact
//                 per-query page in the same operand layout, so the indexer kernel runs
//                 on the pool unchanged.
// map_kernel      the Reindex top-512 over pool slots back to cache positions (the pool
//                 is ascending, so the output stays ascending).
#include <algorithm>

#include "csa2_kernels.cuh"

namespace csa2 {

constexpr int kPoolThreads = 1024;
constexpr int kPoolWarps = kPoolThreads / 32;

// Exclusive prefix over the CTA's threads in thread order; *total gets the sum.
// s: 33 words of shared memory; every thread must call it.
__device__ __forceinline__ uint32_t cta_scan_excl(uint32_t v, uint32_t* s, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += n;
  }
  __syncthreads();  // s may still be read by a previous call
  if (lane == 31) s[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const uint32_t w = s[lane];
    uint32_t wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t n = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += n;
    }
    s[lane] = wi - w;
    if (lane == 31) s[32] = wi;
  }
  __syncthreads();
  *total = s[32];
  return s[warp] + incl - v;
}

// Bin b* of a histogram of n_bins (1 .. 2048) counts, read from the top bin down, where
// the K-th largest item falls: sum(bins > b*) < K <= sum(bins >= b*).  Sets *bin and
// *above = sum(bins > b*).  Every thread must call it; thread t reads bins
// n_bins - 1 - 2t and n_bins - 2 - 2t.
__device__ __forceinline__ void pool_threshold(const uint32_t* h, int n_bins, uint32_t K, uint32_t* s_scan,
                                               uint32_t* bin, uint32_t* above) {
  const int hi = n_bins - 1 - 2 * static_cast<int>(threadIdx.x);
  const uint32_t c0 = hi >= 0 ? h[hi] : 0u, c1 = hi >= 1 ? h[hi - 1] : 0u;
  uint32_t tot;
  const uint32_t ex = cta_scan_excl(c0 + c1, s_scan, &tot);
  if (hi >= 0 && ex < K && ex + c0 >= K) {
    *bin = static_cast<uint32_t>(hi);
    *above = ex;
  } else if (hi >= 1 && ex + c0 < K && ex + c0 + c1 >= K) {
    *bin = static_cast<uint32_t>(hi - 1);
    *above = ex + c0;
  }
  __syncthreads();
}

// Visible entries of row q, clamped to t_max (scores exist for s < t_max only).
__device__ __forceinline__ int64_t pool_visible(const PoolArgs& a, int64_t q, bool report_err) {
  int64_t nv = a.n_visible[q];
  if (nv < 0) nv = 0;
  if (nv > a.t_max) {
    if (report_err) report(a.err, CSA2_ERR_DEVICE, kInfoPos);
    nv = a.t_max;
  }
  return nv;
}

constexpr int kBmaxThreads = 256, kBmaxPer = 8;  // 2,048 blocks per CTA

__global__ void __launch_bounds__(kBmaxThreads) bmax_kernel(const PoolArgs a) {
  pdl_trigger();
  pdl_wait();  // the scores come from the previous kernel
  const int64_t q = blockIdx.y;
  const int64_t nv = pool_visible(a, q, false);
  const int64_t nb = (nv + CSA2_POOL_BLOCK - 1) / CSA2_POOL_BLOCK;
  if (nb <= CSA2_POOL_BLOCKS) return;  // the select kernel lists every visible position
  const float* row = a.scores + q * a.ld;
  uint32_t* key = a.bkey + q * a.nb_cap;
  const int64_t j0 = static_cast<int64_t>(blockIdx.x) * kBmaxThreads * kBmaxPer + threadIdx.x;
  float4 u[kBmaxPer], v[kBmaxPer];
#pragma unroll
  for (int i = 0; i < kBmaxPer; ++i) {  // all loads first
    const int64_t j = j0 + i * kBmaxThreads;
    if (8 * j + 8 <= nv) {
      const float4* p = reinterpret_cast<const float4*>(row + 8 * j);
      u[i] = __ldg(p);
      v[i] = __ldg(p + 1);
    }
  }
#pragma unroll
  for (int i = 0; i < kBmaxPer; ++i) {
    const int64_t j = j0 + i * kBmaxThreads;
    if (j >= nb) break;
    float m;
    if (8 * j + 8 <= nv) {
      m = fmaxf(fmaxf(fmaxf(u[i].x, u[i].y), fmaxf(u[i].z, u[i].w)),
                fmaxf(fmaxf(v[i].x, v[i].y), fmaxf(v[i].z, v[i].w)));
    } else {  // the partial last block
      m = row[8 * j];
      for (int64_t s = 8 * j + 1; s < nv; ++s) m = fmaxf(m, row[s]);
    }
    key[j] = order_key(m);  // a real score never has key 0
  }
}

constexpr int64_t kPoolStage = 32768;  // block keys staged in shared memory (128 KB)
constexpr uint32_t kPoolList = 2048;    // keys still in play kept for the last radix level
constexpr int kKeyUnroll = 8;          // independent key loads in flight per thread

// f(j, key) for every j < nb, each thread 8 keys a round with all loads issued first.
template <typename F>
__device__ __forceinline__ void for_keys(const uint32_t* key, int64_t nb, F f) {
  for (int64_t j0 = threadIdx.x; j0 < nb; j0 += kKeyUnroll * kPoolThreads) {
    uint32_t k[kKeyUnroll];
#pragma unroll
    for (int u = 0; u < kKeyUnroll; ++u) {
      const int64_t j = j0 + static_cast<int64_t>(u) * kPoolThreads;
      k[u] = j < nb ? key[j] : 0u;
    }
#pragma unroll
    for (int u = 0; u < kKeyUnroll; ++u) {
      const int64_t j = j0 + static_cast<int64_t>(u) * kPoolThreads;
      if (j < nb) f(j, k[u]);
    }
  }
}

__global__ void __launch_bounds__(kPoolThreads, 1) pool_kernel(const PoolArgs a) {
  extern __shared__ __align__(16) uint32_t stage[];  // [kPoolStage] when the launch provides it
  __shared__ uint32_t h[2048];
  __shared__ uint32_t s_scan[33];
  __shared__ uint32_t s_gt[kPoolWarps], s_tie[kPoolWarps], s_tbase[kPoolWarps], s_sbase[kPoolWarps];
  __shared__ uint32_t s_bin, s_above, s_lcnt;
  __shared__ uint32_t s_list[kPoolList];  // keys in play (radix levels), then the kept block ids
  pdl_trigger();
  pdl_wait();  // the scores come from the previous kernel
  const int64_t q = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t nv = pool_visible(a, q, true);
  const int64_t nb = (nv + CSA2_POOL_BLOCK - 1) / CSA2_POOL_BLOCK;
  int32_t* out = a.pool + q * CSA2_POOL;
  if (nb <= CSA2_POOL_BLOCKS) {  // every visible position
    for (int i = threadIdx.x; i < CSA2_POOL; i += kPoolThreads) out[i] = i < nv ? i : -1;
    if (threadIdx.x == 0) a.pool_len[q] = static_cast<int32_t>(nv);
    return;
  }
  const uint32_t* gkey = a.bkey + q * a.nb_cap;  // block-maximum keys from bmax_kernel
  const bool staged = a.stage && nb <= kPoolStage;
  // the keys' range [lo, hi]: radix digits over it (block maxima crowd into a narrow
  // range, where fixed top-bit digits would pile into a few bins); the keys move to
  // shared memory on the way when they fit
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
  for_keys(gkey, nb, [&](int64_t j, uint32_t k) {
    lo = min(lo, k);
    hi = max(hi, k);
    if (staged) stage[j] = k;
  });
  const uint32_t* key = staged ? stage : gkey;
  lo = __reduce_min_sync(0xffffffffu, lo);
  hi = __reduce_max_sync(0xffffffffu, hi);
  if (lane == 0) {
    s_gt[warp] = lo;
    s_tie[warp] = hi;
  }
  __syncthreads();
  lo = __reduce_min_sync(0xffffffffu, s_gt[lane]);
  hi = __reduce_max_sync(0xffffffffu, s_tie[lane]);
  __syncthreads();
  // exact K-th largest key, K = 2048: digits of (key - lo), at most 11 bits a level,
  // from the top of the range; a key stays in play while (key - lo) >> m_shift == m_val
  const uint32_t K = CSA2_POOL_BLOCKS;
  const uint32_t span = hi - lo;
  uint32_t m_shift = span ? 32u - static_cast<uint32_t>(__clz(span)) : 0u, m_val = 0u, above = 0u;
  // a level whose keys in play fit the list copies them there on its pass over the row,
  // so the levels after it scan only the list
  uint32_t in_play = static_cast<uint32_t>(nb), list_n = 0;
  bool from_list = false;
  while (m_shift > 0u) {
    const uint32_t c_shift = m_shift > 11u ? m_shift - 11u : 0u;
    const uint32_t width = m_shift - c_shift;
    const bool collect = !from_list && c_shift > 0u && in_play <= kPoolList;
    for (int b = threadIdx.x; b < 2048; b += kPoolThreads) h[b] = 0u;
    if (threadIdx.x == 0) s_lcnt = 0u;
    __syncthreads();
    auto visit = [&](uint32_t k) {
      const uint32_t d = k - lo;
      if ((static_cast<uint64_t>(d) >> m_shift) == m_val) {
        atomicAdd(&h[(d >> c_shift) & ((1u << width) - 1u)], 1u);
        if (collect) s_list[atomicAdd(&s_lcnt, 1u)] = k;  // at most in_play <= kPoolList keys
      }
    };
    if (from_list) {
      for (uint32_t i = threadIdx.x; i < list_n; i += kPoolThreads) visit(s_list[i]);
    } else {
      for_keys(key, nb, [&](int64_t, uint32_t k) { visit(k); });
    }
    __syncthreads();
    pool_threshold(h, 1 << width, K - above, s_scan, &s_bin, &s_above);
    in_play = h[s_bin];
    if (collect) {
      from_list = true;
      list_n = s_lcnt;
    }
    m_val = (m_val << width) | s_bin;
    above += s_above;
    m_shift = c_shift;
    __syncthreads();  // h, s_bin and s_lcnt are read above before the next level resets them
  }
  const uint32_t vstar = lo + m_val;
  const uint32_t need = K - above;  // blocks equal to v* to keep, lowest index first
  // ordered pass: warp w owns blocks [w*R, (w+1)*R), R a multiple of 32
  const int64_t R = ((nb + kPoolWarps * 32 - 1) / (kPoolWarps * 32)) * 32;
  const int64_t w0 = warp * R, w1 = w0 + R < nb ? w0 + R : nb;
  uint32_t gt = 0, tie = 0;
  for (int64_t j0 = w0; j0 < w1; j0 += 32 * kKeyUnroll) {
    uint32_t k[kKeyUnroll];
#pragma unroll
    for (int u = 0; u < kKeyUnroll; ++u) {
      const int64_t j = j0 + 32 * u + lane;
      k[u] = j < w1 ? key[j] : 0u;
    }
#pragma unroll
    for (int u = 0; u < kKeyUnroll; ++u) {
      gt += __popc(__ballot_sync(0xffffffffu, k[u] > vstar));
      tie += __popc(__ballot_sync(0xffffffffu, k[u] == vstar));
    }
  }
  if (lane == 0) {
    s_gt[warp] = gt;
    s_tie[warp] = tie;
  }
  __syncthreads();
  if (warp == 0) {
    const uint32_t t = s_tie[lane];
    uint32_t ti = t;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t n = __shfl_up_sync(0xffffffffu, ti, off);
      if (lane >= off) ti += n;
    }
    const uint32_t tb = ti - t;
    const uint32_t take = tb >= need ? 0u : (need - tb < t ? need - tb : t);
    const uint32_t sel = s_gt[lane] + take;
    uint32_t si = sel;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t n = __shfl_up_sync(0xffffffffu, si, off);
      if (lane >= off) si += n;
    }
    s_tbase[lane] = tb;
    s_sbase[lane] = si - sel;
  }
  __syncthreads();
  uint32_t tr = s_tbase[warp], sr = s_sbase[warp];
  const uint32_t lt = (1u << lane) - 1u;
  for (int64_t j0 = w0; j0 < w1; j0 += 32) {
    const int64_t j = j0 + lane;
    const uint32_t k = j < w1 ? key[j] : 0u;  // (staged keys, or a second read from L2)
    const uint32_t tmask = __ballot_sync(0xffffffffu, k == vstar);
    const bool sel = k > vstar || (k == vstar && tr + __popc(tmask & lt) < need);
    const uint32_t smask = __ballot_sync(0xffffffffu, sel);
    if (sel) {
      const uint32_t slot = sr + __popc(smask & lt);
      if (slot < K) s_list[slot] = static_cast<uint32_t>(j);  // kept blocks in ascending order
    }
    tr += __popc(tmask);
    sr += __popc(smask);
  }
  __syncthreads();
  // positions of the kept blocks, ascending: plain coalesced stores
  for (int i = threadIdx.x; i < CSA2_POOL; i += kPoolThreads) {
    const int64_t p = 8 * static_cast<int64_t>(s_list[i >> 3]) + (i & 7);
    out[i] = p < nv ? static_cast<int32_t>(p) : -1;
  }
  if (threadIdx.x == 0) {  // only the last block can be partial, and it is kept last
    const int64_t part = nv % CSA2_POOL_BLOCK;
    const bool last = s_list[K - 1] == static_cast<uint32_t>(nb - 1);
    a.pool_len[q] = static_cast<int32_t>(CSA2_POOL - (last && part ? CSA2_POOL_BLOCK - part : 0));
  }
}

// One warp per 4 consecutive pooled blocks of 8 entries (one coalesced 128-byte read of
// their pool entries, then every copy's load issued before its store); 8 warps per CTA.
constexpr int kGatherSlots = 4;

template <bool kMx>
__global__ void __launch_bounds__(256) gather_kernel(const GatherArgs a) {
  constexpr uint32_t kPg = kMx ? kIdxMxPageBytes : kIdxPageBytes;
  constexpr int kAtoms = kMx ? 1 : 2;  // scale atoms per page: E8M0 per 32, or E4M3 per 16
  pdl_trigger();
  pdl_wait();  // the pool may come from the previous kernel
  const int lane = threadIdx.x & 31, sub = lane >> 3, i = lane & 7;
  constexpr int64_t kPerQ = CSA2_POOL_BLOCKS / kGatherSlots;
  const int64_t wid = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (wid >= a.n_q * kPerQ) return;
  const int64_t q = wid / kPerQ;
  const int32_t r0 = static_cast<int32_t>(wid % kPerQ) * kGatherSlots;
  const int32_t* pl = a.pool + q * CSA2_POOL + 8 * r0;
  const int32_t p = pl[lane];  // block slot r0 + sub, entry i
  const int32_t nxt = (lane == 0 && r0 + kGatherSlots < CSA2_POOL_BLOCKS) ? pl[8 * kGatherSlots] : -1;
  const int32_t p0 = __shfl_sync(0xffffffffu, p, lane & ~7);
  // a slot lists 8j .. 8j + c - 1 then -1s; the pool is a prefix of such slots, ascending
  const uint32_t valid = __ballot_sync(0xffffffffu, p >= 0);
  const uint32_t vs = (valid >> (8 * sub)) & 0xFFu;
  const int cnt = __popc(vs);
  const int32_t nx_in = __shfl_sync(0xffffffffu, p, ((sub + 1) & 3) * 8);
  const int32_t nx_out = __shfl_sync(0xffffffffu, nxt, 0);
  const int32_t pn = sub < kGatherSlots - 1 ? nx_in : nx_out;  // first entry of the following slot
  bool form = p == -1 || (p0 >= 0 && (p0 & 7) == 0 && p == p0 + i);
  form = form && ((vs + 1u) & vs) == 0u && !(cnt < 8 && pn >= 0) && !(cnt == 8 && pn >= 0 && pn <= p0);
  if (r0 == 0 && lane == 0) a.req_q[q] = static_cast<int32_t>(q);
  if (__ballot_sync(0xffffffffu, !form) != 0u) {
    if (lane == 0) report(a.err, CSA2_ERR_DEVICE, kInfoPool);
    return;
  }
  const int32_t r = r0 + sub;
  if (i == 0 && (cnt > 0 || r == 0) && (cnt < 8 || pn < 0)) a.pool_len[q] = 8 * r + cnt;  // the last block
  // source page of this lane's slot
  bool ok = cnt > 0;
  int64_t page = 0;
  if (ok) {
    const int32_t rq = a.req[q];
    if (p0 + cnt > a.n_visible[q] || p0 + cnt > a.cache.max_pages * kPage) {
      if (i == 0) report(a.err, CSA2_ERR_DEVICE, kInfoPool);
      ok = false;
    } else {
      page = page_id(a.cache, rq, p0);
      if (page < 0 || page >= a.cache.n_pages) {
        if (i == 0) report(a.err, CSA2_ERR_DEVICE, kInfoPage);
        ok = false;
      }
    }
  }
  uint8_t* cbase = a.compact + q * (CSA2_POOL / kPage) * static_cast<int64_t>(kPg);
  // nibbles: each slot's 8 entries are one 512-byte group of the operand layout
  uint4 nib[kGatherSlots];
#pragma unroll
  for (int t = 0; t < kGatherSlots; ++t) {
    const int64_t pg_t = __shfl_sync(0xffffffffu, page, 8 * t);
    const int32_t p0_t = __shfl_sync(0xffffffffu, p0, 8 * t);
    if (__shfl_sync(0xffffffffu, ok, 8 * t))
      nib[t] = reinterpret_cast<const uint4*>(a.cache.idx + pg_t * kPg + ((p0_t % kPage) >> 3) * 512)[lane];
  }
  // scales: 4 bytes per entry and atom; lane = (slot sub, entry i)
  uint32_t sc[kAtoms];
  const uint32_t e = static_cast<uint32_t>(p0 % kPage) + i;
  if (ok) {
#pragma unroll
    for (int at = 0; at < kAtoms; ++at)
      sc[at] = *reinterpret_cast<const uint32_t*>(a.cache.idx + page * kPg + kIdxNibBytes + at * 512u +
                                                  (e & 31u) * 16u + (e >> 5) * 4u);
  }
#pragma unroll
  for (int t = 0; t < kGatherSlots; ++t) {
    if (__shfl_sync(0xffffffffu, ok, 8 * t)) {
      const int32_t rt = r0 + t;
      uint8_t* dst = cbase + ((8 * rt) / kPage) * static_cast<int64_t>(kPg);
      reinterpret_cast<uint4*>(dst + (((8 * rt) % kPage) >> 3) * 512)[lane] = nib[t];
    }
  }
  if (ok) {
    const uint32_t n = static_cast<uint32_t>((8 * r) % kPage) + i;
    uint8_t* dst = cbase + ((8 * r) / kPage) * static_cast<int64_t>(kPg);
#pragma unroll
    for (int at = 0; at < kAtoms; ++at)
      *reinterpret_cast<uint32_t*>(dst + kIdxNibBytes + at * 512u + (n & 31u) * 16u + (n >> 5) * 4u) = sc[at];
  }
}

__global__ void __launch_bounds__(512) map_kernel(const int32_t* slots, const int32_t* pool, int32_t* out) {
  pdl_trigger();
  pdl_wait();  // the slots come from the previous kernel
  const int64_t q = blockIdx.x;
  const int32_t s = slots[q * CSA2_TOPK + threadIdx.x];
  out[q * CSA2_TOPK + threadIdx.x] = (s >= 0 && s < CSA2_POOL) ? pool[q * CSA2_POOL + s] : -1;
}

cudaError_t launch_pool_bmax(const PoolArgs& a, cudaStream_t stream) {
  const int64_t per_cta = kBmaxThreads * kBmaxPer;
  const int64_t gx = (a.nb_cap + per_cta - 1) / per_cta;
  if (a.n_q == 0 || gx == 0) return cudaSuccess;
  return launch_pdl(bmax_kernel, dim3(static_cast<unsigned>(gx), static_cast<unsigned>(a.n_q)), dim3(kBmaxThreads),
                    0, stream, nullptr, a);
}

cudaError_t launch_pool(const PoolArgs& a, cudaStream_t stream) {
  if (a.n_q == 0) return cudaSuccess;
  static std::atomic<int> limit_set[kMaxDevices];
  PoolArgs b = a;
  b.stage = a.nb_cap > CSA2_POOL_BLOCKS ? 1 : 0;  // rows of at most 2,048 blocks need no keys
  const size_t smem = b.stage ? static_cast<size_t>(std::min<int64_t>(a.nb_cap, kPoolStage)) * 4 : 0;
  if (smem > 0) {
    const cudaError_t e = smem_limit_once(reinterpret_cast<const void*>(pool_kernel), smem, limit_set);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(pool_kernel, dim3(static_cast<unsigned>(a.n_q)), dim3(kPoolThreads), smem, stream, nullptr, b);
}

cudaError_t launch_gather(const GatherArgs& a, cudaStream_t stream) {
  if (a.n_q == 0) return cudaSuccess;
  const int64_t blocks = a.n_q * (CSA2_POOL_BLOCKS / kGatherSlots) / 8;
  auto* k = a.cache.idx_format == CSA2_IDX_MXFP4 ? gather_kernel<true> : gather_kernel<false>;
  return launch_pdl(k, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, nullptr, a);
}

cudaError_t launch_map(const int32_t* slots, const int32_t* pool, int32_t* out, int64_t n_q, cudaStream_t stream) {
  if (n_q == 0) return cudaSuccess;
  return launch_pdl(map_kernel, dim3(static_cast<unsigned>(n_q)), dim3(CSA2_TOPK), 0, stream, nullptr, slots, pool,
                    out);
}

}  // namespace csa2
