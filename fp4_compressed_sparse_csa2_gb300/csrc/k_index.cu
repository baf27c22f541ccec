// k_index.cu -- lightning-indexer scores on the block-scaled FP4 tensor cores.
//
// "DeepSeek's Attention and KV Cache - From MLA to CSA2", "DeepSeek-V3.2: Sparse
// Attention With a Learned Indexer": I[t,s] = sum_j w[t,j] ReLU(q^I[t,j] . k^I[s]),
// one shared key per cached entry; "DeepSeek-V4": the indexer's query-key product
// multiplies entirely in FP4.  "From MLA to DSA to HCA/CSA", "CSA: two changes to
// HCA": the scorer takes ReLU(q . k) * 128^-0.5, weights it per head and sums heads.
//
// Design (one CTA = 6 warps, persistent over a contiguous range of key tiles):
//   warp 0      producer: one 9216-byte bulk copy per 128-entry indexer page (the
//               page is stored in the MMA's operand layout), and one per packed
//               query group, into an mbarrier-tracked smem ring;
//   warp 1      TMEM allocator and MMA issuer: tcgen05.cp of the E4M3 scale atoms
//               into TMEM, then two tcgen05.mma kind::mxf4nvf4 (K = 64 each) per tile:
//               D[128 keys][N = G*heads_I] in fp32 TMEM, double buffered;
//   warps 2..5  epilogue: tcgen05.ld a TMEM row per thread (thread = key), ReLU,
//               head weights, head sum, 128^-0.5, coalesced fp32 score stores.
// Every wait is bounded; a timeout sets the workspace error word and the CTA drains
// its copies and MMAs, frees TMEM and returns.
#include "csa2_kernels.cuh"

namespace csa2 {

constexpr int kIdxThreads = 192;
constexpr float kInvSqrtDI = 0.08838834764831845f;  // 128^-0.5

struct TileInfo {
  int64_t g;
  int32_t t;
  int32_t r;
  bool active;
  bool page_ok;
  int64_t page;
};

__device__ __forceinline__ TileInfo tile_info(const IndexArgs& a, int64_t flat) {
  TileInfo ti;
  ti.g = flat / a.tpg;
  ti.t = static_cast<int32_t>(flat % a.tpg);
  const int64_t q0 = ti.g * a.G;
  const int32_t qn = static_cast<int32_t>(a.n_q - q0 < a.G ? a.n_q - q0 : a.G);
  ti.r = __ldg(a.req + q0);
  int32_t vis = 0;
  for (int i = 0; i < qn; ++i) vis = max(vis, __ldg(a.n_visible + q0 + i));
  vis = min(vis, a.cache.max_pages * kPage);
  ti.active = static_cast<int64_t>(ti.t) * kPage < vis;
  ti.page = ti.active ? page_id(a.cache, ti.r, static_cast<int64_t>(ti.t) * kPage) : -1;
  ti.page_ok = ti.page >= 0 && ti.page < a.cache.n_pages;
  return ti;
}

__global__ void __launch_bounds__(kIdxThreads, 2) index_kernel(const IndexArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = a.stages;
  uint8_t* ring = smem;                                   // S x 9216
  uint8_t* qslot = ring + static_cast<size_t>(S) * kIdxPageBytes;  // 2 x 9216
  float* sw_all = reinterpret_cast<float*>(qslot + 2 * kIdxPageBytes);  // 4 warps x 128 head weights
  uint64_t* bars = reinterpret_cast<uint64_t*>(sw_all + 4 * 128);
  uint64_t* full = bars;           // [S]
  uint64_t* empty = full + S;      // [S]
  uint64_t* acc_full = empty + S;  // [2]
  uint64_t* acc_empty = acc_full + 2;  // [2]
  uint64_t* q_full = acc_empty + 2;    // [2]
  uint64_t* q_empty = q_full + 2;      // [2]
  uint64_t* drain = q_empty + 2;       // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int32_t* abort = reinterpret_cast<volatile int32_t*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 128);
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
    }
    mbar_init(drain, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, a.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int64_t total = a.n_groups * a.tpg;
  const int64_t begin = total * blockIdx.x / gridDim.x;
  const int64_t end = total * (blockIdx.x + 1) / gridDim.x;
  const uint32_t N = static_cast<uint32_t>(a.N);
  const uint32_t nib_q = N * 64u;
  const uint32_t acc_col[2] = {0u, N};
  const uint32_t sfa_col[2] = {2u * N, 2u * N + 8u};
  const uint32_t sfb_col[2] = {2u * N + 16u, 2u * N + 24u};

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int64_t n = 0, m = 0, prev_g = -1;
      bool ok = true;
      for (int64_t flat = begin; flat < end && ok; ++flat) {
        const TileInfo ti = tile_info(a, flat);
        if (!ti.active) continue;
        if (ti.g != prev_g) {
          const int slot = static_cast<int>(m & 1);
          ok = mbar_wait(&q_empty[slot], static_cast<uint32_t>(((m >> 1) & 1) ^ 1), abort);
          if (!ok) break;
          mbar_arrive_expect_tx(&q_full[slot], static_cast<uint32_t>(a.grp_bytes));
          bulk_g2s(qslot + slot * kIdxPageBytes, a.qpack + ti.g * a.grp_bytes, static_cast<uint32_t>(a.grp_bytes),
                   &q_full[slot]);
          ++m;
          prev_g = ti.g;
        }
        const int s = static_cast<int>(n % S);
        ok = mbar_wait(&empty[s], static_cast<uint32_t>(((n / S) & 1) ^ 1), abort);
        if (!ok) break;
        if (ti.page_ok) {
          mbar_arrive_expect_tx(&full[s], kIdxPageBytes);
          bulk_g2s_hint(ring + static_cast<size_t>(s) * kIdxPageBytes, a.idx_pages + ti.page * kIdxPageBytes,
                        kIdxPageBytes, &full[s], pol);
        } else {
          report(a.err, CSA2_ERR_DEVICE, kInfoPage);
          mbar_arrive(&full[s]);
        }
        ++n;
      }
      if (!ok) {
        *abort = 1;
        report(a.err, CSA2_ERR_TIMEOUT, kInfoWait);
      }
      // drain: the last copies issued into each slot have landed before exit
      for (int64_t k = (n > S ? n - S : 0); k < n; ++k) mbar_wait(&full[k % S], static_cast<uint32_t>((k / S) & 1), nullptr);
      for (int64_t k = (m > 2 ? m - 2 : 0); k < m; ++k) mbar_wait(&q_full[k & 1], static_cast<uint32_t>((k >> 1) & 1), nullptr);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_nvf4(128, a.N);
      int64_t n = 0, m = 0, prev_g = -1;
      int cur = 0;
      bool ok = true;
      for (int64_t flat = begin; flat < end && ok; ++flat) {
        const TileInfo ti = tile_info(a, flat);
        if (!ti.active) continue;
        if (ti.g != prev_g) {
          if (m > 0) mma_commit(&q_empty[(m - 1) & 1]);
          cur = static_cast<int>(m & 1);
          ok = mbar_wait(&q_full[cur], static_cast<uint32_t>((m >> 1) & 1), abort);
          if (!ok) break;
          tc_fence_after();
          const uint32_t qs = smem_u32(qslot + cur * kIdxPageBytes);
          tmem_cp_sf(tmem + sfb_col[cur], sdesc(qs + nib_q, 128, 128));
          tmem_cp_sf(tmem + sfb_col[cur] + 4, sdesc(qs + nib_q + 512, 128, 128));
          ++m;
          prev_g = ti.g;
        }
        const int s = static_cast<int>(n % S);
        const int ab = static_cast<int>(n & 1);
        ok = mbar_wait(&full[s], static_cast<uint32_t>((n / S) & 1), abort);
        if (!ok) break;
        ok = mbar_wait(&acc_empty[ab], static_cast<uint32_t>(((n >> 1) & 1) ^ 1), abort);
        if (!ok) break;
        tc_fence_after();
        const uint32_t st = smem_u32(ring + static_cast<size_t>(s) * kIdxPageBytes);
        const uint32_t qs = smem_u32(qslot + cur * kIdxPageBytes);
        tmem_cp_sf(tmem + sfa_col[ab], sdesc(st + kIdxNibBytes, 128, 128));
        tmem_cp_sf(tmem + sfa_col[ab] + 4, sdesc(st + kIdxNibBytes + 512, 128, 128));
#pragma unroll
        for (uint32_t kk = 0; kk < 2; ++kk) {
          mma_nvf4(tmem + acc_col[ab], sdesc(st + kk * 256u, 128, 512), sdesc(qs + kk * 256u, 128, 512), idesc,
                   tmem + sfa_col[ab] + 4u * kk, tmem + sfb_col[cur] + 4u * kk, kk);
        }
        mma_commit(&empty[s]);
        mma_commit(&acc_full[ab]);
        ++n;
      }
      if (!ok) {
        *abort = 1;
        report(a.err, CSA2_ERR_TIMEOUT, kInfoWait);
      }
      mma_commit(drain);
      mbar_wait(drain, 0, nullptr);
    }
  } else {
    // epilogue: 4 warps, thread = TMEM lane = key within the tile
    const int quarter = warp & 3;
    const uint32_t row = static_cast<uint32_t>(quarter * 32 + lane);
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    float* sw = sw_all + quarter * 128;  // this warp's copy of the group's head weights
    int64_t n = 0, prev_g = -1;
    bool ok = true;
    for (int64_t flat = begin; flat < end && ok; ++flat) {
      const TileInfo ti = tile_info(a, flat);
      if (!ti.active) continue;
      const int ab = static_cast<int>(n & 1);
      ok = mbar_wait(&acc_full[ab], static_cast<uint32_t>((n >> 1) & 1), abort);
      if (!ok) break;
      tc_fence_after();
      const int64_t q0 = ti.g * a.G;
      if (ti.g != prev_g) {
        __syncwarp();
        for (int i = lane; i < a.N; i += 32) {
          const int64_t q = q0 + i / a.heads_I;
          sw[i] = q < a.n_q ? __ldg(a.w + q * a.heads_I + i % a.heads_I) : 0.0f;
          if (q < a.n_q && __ldg(a.req + q) != ti.r) report(a.err, CSA2_ERR_DEVICE, kInfoGroup);
        }
        __syncwarp();
        prev_g = ti.g;
      }
      const int64_t key = static_cast<int64_t>(ti.t) * kPage + row;
      for (int gq = 0; gq < a.G; ++gq) {
        const int64_t q = q0 + gq;
        if (q >= a.n_q) break;
        float acc = 0.0f;
        for (int c0 = 0; c0 < a.heads_I; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_base + acc_col[ab] + static_cast<uint32_t>(gq * a.heads_I + c0), r);
          tmem_ld_wait();
          const float4* w4 = reinterpret_cast<const float4*>(sw + gq * a.heads_I + c0);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 wv = w4[i];
            acc = fmaf(wv.x, fmaxf(__uint_as_float(r[4 * i + 0]), 0.0f), acc);
            acc = fmaf(wv.y, fmaxf(__uint_as_float(r[4 * i + 1]), 0.0f), acc);
            acc = fmaf(wv.z, fmaxf(__uint_as_float(r[4 * i + 2]), 0.0f), acc);
            acc = fmaf(wv.w, fmaxf(__uint_as_float(r[4 * i + 3]), 0.0f), acc);
          }
        }
        if (ti.page_ok && key < __ldg(a.n_visible + q)) a.scores[q * a.ld + key] = acc * kInvSqrtDI;
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[ab]);
      ++n;
    }
    if (!ok) {
      *abort = 1;
      report(a.err, CSA2_ERR_TIMEOUT, kInfoWait);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, a.tmem_cols);
}

size_t index_smem_bytes(int stages) {
  return 1024 + static_cast<size_t>(stages + 2) * kIdxPageBytes + 4 * 128 * sizeof(float) +
         (2 * stages + 9) * sizeof(uint64_t) + 16;
}

cudaError_t launch_index(const IndexArgs& a, int grid, cudaStream_t stream) {
  const size_t smem = index_smem_bytes(a.stages);
  cudaError_t e = cudaFuncSetAttribute(index_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  index_kernel<<<grid, kIdxThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace csa2
