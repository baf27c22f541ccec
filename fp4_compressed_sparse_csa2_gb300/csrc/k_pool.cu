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
// pool_kernel     one 1024-thread CTA per score row: block maxima as order-preserving
//                 keys (written to scratch) with an 11-bit histogram, exact radix
//                 selection of the 2,048th largest key (11 + 11 + 10 bits), then an
//                 ordered pass (warp ballots, warp-range prefix sums) that keeps the
//                 blocks above it plus the lowest-index blocks equal to it and writes
//                 their positions ascending.
// gather_kernel   one warp per pooled block of 8 entries: the entries' 512-byte nibble
//                 group and their scale bytes move from the cache page into a compact
//                 per-query page in the same operand layout, so the indexer kernel runs
//                 on the pool unchanged.
// map_kernel      the Reindex top-512 over pool slots back to cache positions (the pool
//                 is ascending, so the output stays ascending).
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

// Bin b* of a histogram of n_bins (2048 or 1024) counts, read from the top bin down,
// where the K-th largest item falls: sum(bins > b*) < K <= sum(bins >= b*).  Sets
// *bin and *above = sum(bins > b*).  Every thread must call it.
__device__ __forceinline__ void pool_threshold(const uint32_t* h, int n_bins, uint32_t K, uint32_t* s_scan,
                                               uint32_t* bin, uint32_t* above) {
  const int per = n_bins / kPoolThreads;  // 2 or 1 bins per thread, from the top
  const int hi = n_bins - 1 - per * static_cast<int>(threadIdx.x);
  uint32_t c[2] = {h[hi], per == 2 ? h[hi - 1] : 0u};
  uint32_t tot;
  const uint32_t ex = cta_scan_excl(c[0] + c[1], s_scan, &tot);
  if (ex < K && ex + c[0] >= K) {
    *bin = static_cast<uint32_t>(hi);
    *above = ex;
  } else if (per == 2 && ex + c[0] < K && ex + c[0] + c[1] >= K) {
    *bin = static_cast<uint32_t>(hi - 1);
    *above = ex + c[0];
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kPoolThreads, 1) pool_kernel(const PoolArgs a) {
  __shared__ uint32_t h[2048];
  __shared__ uint32_t s_scan[33];
  __shared__ uint32_t s_gt[kPoolWarps], s_tie[kPoolWarps], s_tbase[kPoolWarps], s_sbase[kPoolWarps];
  __shared__ uint32_t s_bin, s_above, s_last;
  pdl_trigger();
  pdl_wait();  // the scores come from the previous kernel
  const int64_t q = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t nv = a.n_visible[q];
  if (nv < 0) nv = 0;
  if (nv > a.t_max) {  // scores exist for s < t_max only
    report(a.err, CSA2_ERR_DEVICE, kInfoPos);
    nv = a.t_max;
  }
  const int64_t nb = (nv + CSA2_POOL_BLOCK - 1) / CSA2_POOL_BLOCK;
  int32_t* out = a.pool + q * CSA2_POOL;
  if (nb <= CSA2_POOL_BLOCKS) {  // every visible position
    for (int i = threadIdx.x; i < CSA2_POOL; i += kPoolThreads) out[i] = i < nv ? i : -1;
    if (threadIdx.x == 0) a.pool_len[q] = static_cast<int32_t>(nv);
    return;
  }
  const float* row = a.scores + q * a.ld;
  uint32_t* key = a.bkey + q * a.nb_cap;
  for (int b = threadIdx.x; b < 2048; b += kPoolThreads) h[b] = 0u;
  __syncthreads();
  // block maxima as order keys (a real score never has key 0)
  for (int64_t j = threadIdx.x; j < nb; j += kPoolThreads) {
    float m;
    if (8 * j + 8 <= nv) {
      const float4* p = reinterpret_cast<const float4*>(row + 8 * j);
      const float4 u = p[0], v = p[1];
      m = fmaxf(fmaxf(fmaxf(u.x, u.y), fmaxf(u.z, u.w)), fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
    } else {
      m = row[8 * j];
      for (int64_t s = 8 * j + 1; s < nv; ++s) m = fmaxf(m, row[s]);
    }
    const uint32_t k = order_key(m);
    key[j] = k;
    atomicAdd(&h[k >> 21], 1u);
  }
  __syncthreads();
  // exact K-th largest key, K = 2048, by three radix levels
  const uint32_t K = CSA2_POOL_BLOCKS;
  pool_threshold(h, 2048, K, s_scan, &s_bin, &s_above);
  const uint32_t b1 = s_bin, a1 = s_above;
  for (int b = threadIdx.x; b < 2048; b += kPoolThreads) h[b] = 0u;
  __syncthreads();
  for (int64_t j = threadIdx.x; j < nb; j += kPoolThreads) {
    const uint32_t k = key[j];
    if ((k >> 21) == b1) atomicAdd(&h[(k >> 10) & 2047u], 1u);
  }
  __syncthreads();
  pool_threshold(h, 2048, K - a1, s_scan, &s_bin, &s_above);
  const uint32_t b2 = s_bin, a2 = s_above;
  const uint32_t pre = (b1 << 11) | b2;
  for (int b = threadIdx.x; b < 1024; b += kPoolThreads) h[b] = 0u;
  __syncthreads();
  for (int64_t j = threadIdx.x; j < nb; j += kPoolThreads) {
    const uint32_t k = key[j];
    if ((k >> 10) == pre) atomicAdd(&h[k & 1023u], 1u);
  }
  __syncthreads();
  pool_threshold(h, 1024, K - a1 - a2, s_scan, &s_bin, &s_above);
  const uint32_t vstar = (pre << 10) | s_bin;
  const uint32_t need = K - a1 - a2 - s_above;  // blocks equal to v* to keep, lowest index first
  // ordered pass: warp w owns blocks [w*R, (w+1)*R), R a multiple of 32
  const int64_t R = ((nb + kPoolWarps * 32 - 1) / (kPoolWarps * 32)) * 32;
  const int64_t w0 = warp * R, w1 = w0 + R < nb ? w0 + R : nb;
  uint32_t gt = 0, tie = 0;
  for (int64_t j0 = w0; j0 < w1; j0 += 32) {
    const int64_t j = j0 + lane;
    const uint32_t k = j < w1 ? key[j] : 0u;
    gt += __popc(__ballot_sync(0xffffffffu, k > vstar));
    tie += __popc(__ballot_sync(0xffffffffu, k == vstar));
  }
  if (lane == 0) {
    s_gt[warp] = gt;
    s_tie[warp] = tie;
  }
  if (threadIdx.x == 0) s_last = 0u;
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
    const uint32_t k = j < w1 ? key[j] : 0u;
    const uint32_t tmask = __ballot_sync(0xffffffffu, k == vstar);
    const bool sel = k > vstar || (k == vstar && tr + __popc(tmask & lt) < need);
    const uint32_t smask = __ballot_sync(0xffffffffu, sel);
    if (sel) {
      const uint32_t slot = sr + __popc(smask & lt);
      if (slot < K) {
        int32_t v[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) v[t] = 8 * j + t < nv ? static_cast<int32_t>(8 * j + t) : -1;
        int4* dst = reinterpret_cast<int4*>(out + 8 * static_cast<int64_t>(slot));
        dst[0] = make_int4(v[0], v[1], v[2], v[3]);
        dst[1] = make_int4(v[4], v[5], v[6], v[7]);
        if (j == nb - 1) s_last = 1u;
      }
    }
    tr += __popc(tmask);
    sr += __popc(smask);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const int64_t part = nv % CSA2_POOL_BLOCK;
    a.pool_len[q] = static_cast<int32_t>(CSA2_POOL - (s_last && part ? CSA2_POOL_BLOCK - part : 0));
  }
}

// One warp per pooled block of 8 entries; 8 warps per CTA.
template <bool kMx>
__global__ void __launch_bounds__(256) gather_kernel(const GatherArgs a) {
  constexpr uint32_t kPg = kMx ? kIdxMxPageBytes : kIdxPageBytes;
  pdl_trigger();
  pdl_wait();  // the pool may come from the previous kernel
  const int lane = threadIdx.x & 31;
  const int64_t item = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (item >= a.n_q * CSA2_POOL_BLOCKS) return;
  const int64_t q = item / CSA2_POOL_BLOCKS;
  const int32_t r = static_cast<int32_t>(item % CSA2_POOL_BLOCKS);
  const int32_t* pl = a.pool + q * CSA2_POOL + 8 * r;
  const int32_t p = lane < 8 ? pl[lane] : 0;
  const int32_t p0 = __shfl_sync(0xffffffffu, p, 0);
  // a block slot lists 8j .. 8j + c - 1 then -1s; the pool is a prefix of such slots
  const bool form = lane >= 8 || (p == -1 ? true : (p0 >= 0 && (p0 & 7) == 0 && p == p0 + lane));
  const uint32_t valid = __ballot_sync(0xffffffffu, lane < 8 && p >= 0);
  const bool ok_form = __all_sync(0xffffffffu, form) && ((valid + 1u) & valid) == 0u;
  const int32_t cnt = __popc(valid);
  if (r == 0 && lane == 0) a.req_q[q] = static_cast<int32_t>(q);
  if (!ok_form) {
    if (lane == 0) report(a.err, CSA2_ERR_DEVICE, kInfoPool);
    return;
  }
  const int32_t nxt = (r + 1 < CSA2_POOL_BLOCKS && lane == 0) ? pl[8] : -1;
  if (lane == 0 && ((cnt < 8 && nxt >= 0) || (cnt == 8 && nxt >= 0 && nxt <= p0))) {
    report(a.err, CSA2_ERR_DEVICE, kInfoPool);  // a hole in the pool, or positions not ascending
    return;
  }
  if (lane == 0 && (cnt > 0 || r == 0) && (cnt < 8 || nxt < 0)) a.pool_len[q] = 8 * r + cnt;  // the last block
  if (cnt == 0) return;
  const int32_t rq = a.req[q];
  const int32_t nvq = a.n_visible[q];
  if (p0 + cnt > nvq || p0 + cnt > a.cache.max_pages * kPage) {
    if (lane == 0) report(a.err, CSA2_ERR_DEVICE, kInfoPool);
    return;
  }
  const int64_t page = page_id(a.cache, rq, p0);
  if (page < 0 || page >= a.cache.n_pages) {
    if (lane == 0) report(a.err, CSA2_ERR_DEVICE, kInfoPage);
    return;
  }
  const uint8_t* src = a.cache.idx + page * kPg;
  uint8_t* dst = a.compact + (q * (CSA2_POOL / kPage) + (8 * r) / kPage) * static_cast<int64_t>(kPg);
  const uint32_t e0 = static_cast<uint32_t>(p0 % kPage), n0 = static_cast<uint32_t>((8 * r) % kPage);
  // nibbles: the 8 entries form one 512-byte group of the operand layout
  reinterpret_cast<uint4*>(dst + (n0 >> 3) * 512u)[lane] = reinterpret_cast<const uint4*>(src + (e0 >> 3) * 512u)[lane];
  // scales: 4 bytes per entry and scale atom (two atoms of E4M3 per 16, one of E8M0 per 32)
  constexpr int kAtoms = kMx ? 1 : 2;
  if (lane < 8 * kAtoms) {
    const uint32_t i = lane & 7u, at = lane >> 3;
    const uint32_t e = e0 + i, n = n0 + i;
    const uint32_t so = kIdxNibBytes + at * 512u + (e & 31u) * 16u + (e >> 5) * 4u;
    const uint32_t d_o = kIdxNibBytes + at * 512u + (n & 31u) * 16u + (n >> 5) * 4u;
    *reinterpret_cast<uint32_t*>(dst + d_o) = *reinterpret_cast<const uint32_t*>(src + so);
  }
}

__global__ void __launch_bounds__(512) map_kernel(const int32_t* slots, const int32_t* pool, int32_t* out) {
  pdl_trigger();
  pdl_wait();  // the slots come from the previous kernel
  const int64_t q = blockIdx.x;
  const int32_t s = slots[q * CSA2_TOPK + threadIdx.x];
  out[q * CSA2_TOPK + threadIdx.x] = (s >= 0 && s < CSA2_POOL) ? pool[q * CSA2_POOL + s] : -1;
}

cudaError_t launch_pool(const PoolArgs& a, cudaStream_t stream) {
  if (a.n_q == 0) return cudaSuccess;
  return launch_pdl(pool_kernel, dim3(static_cast<unsigned>(a.n_q)), dim3(kPoolThreads), 0, stream, nullptr, a);
}

cudaError_t launch_gather(const GatherArgs& a, cudaStream_t stream) {
  if (a.n_q == 0) return cudaSuccess;
  const int64_t blocks = a.n_q * CSA2_POOL_BLOCKS / 8;
  auto* k = a.cache.idx_format == CSA2_IDX_MXFP4 ? gather_kernel<true> : gather_kernel<false>;
  return launch_pdl(k, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, nullptr, a);
}

cudaError_t launch_map(const int32_t* slots, const int32_t* pool, int32_t* out, int64_t n_q, cudaStream_t stream) {
  if (n_q == 0) return cudaSuccess;
  return launch_pdl(map_kernel, dim3(static_cast<unsigned>(n_q)), dim3(CSA2_TOPK), 0, stream, nullptr, slots, pool,
                    out);
}

}  // namespace csa2
