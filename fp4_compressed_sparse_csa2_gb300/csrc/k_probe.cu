// k_probe.cu -- tensor-core throughput probe: the measured peak the indexer's FP4 work
// and the attention's f16 work are judged against.
//
// "DeepSeek's Attention and KV Cache - From MLA to CSA2", "A Precision Primer": the FP4
// (block-scaled E2M1) tensor-core rate is a multiple of the bf16 rate on Blackwell parts;
// this kernel measures the rate the indexer's own instruction shapes reach instead of
// deriving it from a nominal ratio.
//
// One CTA per SM.  `issuers` threads (lane 0 of warps 0..issuers-1) each issue `iters`
// back-to-back tcgen05.mma of the requested kind (f16, or block-scaled NVFP4: E2M1 with
// an E4M3 scale per 16, the indexer's default key format) and N into their own TMEM accumulator
// (M = 128; operands in shared memory, zeroed; their values do not change the rate);
// each then commits and waits.  Thread 0 records the clock cycles from its first issue
// to the completion of every issuer's MMAs.
#include "csa2_kernels.cuh"

namespace csa2 {

constexpr int kProbeThreads = 128;
constexpr uint32_t kProbeSmem = 96 * 1024;  // operands: A at 0 (32 KB), B at 32 KB (64 KB)

__global__ void __launch_bounds__(kProbeThreads, 1) probe_mma_kernel(int32_t kind, int32_t n, int32_t iters,
                                                                     int32_t issuers, long long* cycles) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ uint64_t bars[5];  // one per issuer, one for the scale copies
  __shared__ uint32_t tmem_slot;
  __shared__ long long t_start;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < static_cast<int>(kProbeSmem / 16); i += kProbeThreads)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
  if (tid == 0)
    for (int i = 0; i < 5; ++i) mbar_init(&bars[i], 1);
  fence_mbar_init();
  fence_proxy_async_smem();
  if (warp == 0) {
    tmem_alloc(&tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t a0 = smem_u32(smem), b0 = smem_u32(smem + 32 * 1024);
  constexpr uint32_t kSf = 448;  // scale-factor columns (block-scaled kinds)
  if (kind == 1 && warp == 0) {  // scale factors: zeros from shared memory into TMEM
    if (lane == 0) {
      tmem_cp_sf(tmem + kSf, sdesc(a0, 128, 128));
      tmem_cp_sf(tmem + kSf + 4, sdesc(a0, 128, 128));
      tmem_cp_sf(tmem + kSf + 8, sdesc(a0, 128, 128));
      tmem_cp_sf(tmem + kSf + 12, sdesc(a0, 128, 128));
      mma_commit(&bars[4]);  // the copies land before any issuer reads the columns
      mbar_drain_wait(&bars[4], 0);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (lane == 0 && warp < issuers) {
    const uint32_t d = tmem + static_cast<uint32_t>(warp * n);
    long long t0 = clock64();
    if (warp == 0) t_start = t0;
    if (kind == 0) {
      // f16, K-major A [128][128] and B [n][128]: row groups of 8 at 2048 B, K steps at 256 B
      const uint32_t idesc = idesc_f16(128, n, 0, 0);
      const uint64_t da = sdesc(a0, 128, 2048), db = sdesc(b0, 128, 2048);
      for (int i = 0; i < iters; ++i) {
        const uint64_t k = static_cast<uint64_t>(16 * (i & 7));
        mma_f16(d, da + k, db + k, idesc, i > 0 ? 1u : 0u);
      }
    } else {
      // FP4, K-major A [128][256] and B [n][256]: row groups of 8 at 1024 B, K steps of 64
      // elements at 256 B (the indexer page's operand layout)
      const uint64_t da = sdesc(a0, 128, 1024), db = sdesc(b0, 128, 1024);
      const uint32_t idesc = idesc_nvf4(128, n);
      for (int i = 0; i < iters; ++i) {
        const uint64_t k = static_cast<uint64_t>(16 * (i & 3));
        mma_nvf4(d, da + k, db + k, idesc, tmem + kSf, tmem + kSf + 8, i > 0 ? 1u : 0u);
      }
    }
    mma_commit(&bars[warp]);
    mbar_drain_wait(&bars[warp], 0);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) cycles[blockIdx.x] = clock64() - t_start;
  if (warp == 0) tmem_dealloc(tmem, 512);
}

cudaError_t launch_probe_mma(int32_t kind, int32_t n, int32_t iters, int32_t issuers, int32_t n_ctas,
                             long long* cycles, cudaStream_t stream) {
  static std::atomic<int> limit_set[kMaxDevices];
  cudaError_t e = smem_limit_once(reinterpret_cast<const void*>(probe_mma_kernel), kProbeSmem, limit_set);
  if (e != cudaSuccess) return e;
  probe_mma_kernel<<<n_ctas, kProbeThreads, kProbeSmem, stream>>>(kind, n, iters, issuers, cycles);
  return cudaGetLastError();
}

}  // namespace csa2
