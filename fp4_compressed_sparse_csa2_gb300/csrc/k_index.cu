// k_index.cu -- lightning-indexer scores on the block-scaled FP4 tensor cores.
//
// "DeepSeek's Attention and KV Cache - From MLA to CSA2", "DeepSeek-V3.2: Sparse
// Attention With a Learned Indexer": I[t,s] = sum_j w[t,j] ReLU(q^I[t,j] . k^I[s]),
// one shared key per cached entry; "DeepSeek-V4": the indexer's query-key product
// multiplies entirely in FP4.  "From MLA to DSA to HCA/CSA", "CSA: two changes to
// HCA": the scorer takes ReLU(q . k) * 128^-0.5, weights it per head and sums heads.
//
// Design: one persistent CTA per SM (16 warps for N <= 64, 19 for N = 128) over a
// contiguous range of 128-key tiles (one indexer page each):
//   warp 0      producer: a 16-page mbarrier ring of bulk copies (147 KB in flight per
//               SM; the page is stored in the MMA's operand layout), one copy per stage of
//               adjacent pages, plus one per packed query group;
//   issuers     one thread on each of the next three (N <= 64) or two (N = 128) warps,
//               warp 1 also allocating TMEM: tcgen05.cp of the page's scale atoms into
//               TMEM slots as soon as a page lands, then, once the accumulator is free,
//               two tcgen05.mma kind::mxf4nvf4 (K = 64 each; MX scale_vec::2X with E8M0
//               scales per 32 for MXFP4 pages, 4X with E4M3 per 16 otherwise) into one of
//               6 (N <= 64) or 2 (N = 128) fp32 TMEM accumulators D[128 keys][N];
//   epilogue    three warpgroups (N <= 64), each alternating between two accumulators so
//               that it reads one while the other's MMAs run, or four warpgroups in pairs
//               (N = 128): tcgen05.ld of one TMEM row per thread (thread = key), 32
//               columns at a time; the accumulator goes back to its issuer as soon as the
//               last columns are in registers.  ReLU, head weights (held in registers for
//               N <= 64, read from shared memory for N = 128) and head sum use packed
//               fp32x2 FMAs over four partial sums, then x 128^-0.5 and coalesced fp32
//               stores.
// Every wait is bounded; a timeout sets the workspace error word, and the CTA drains
// its copies and MMAs, frees TMEM and returns.
#include "csa2_kernels.cuh"


namespace csa2 {

constexpr uint32_t kIssuers = 4;    // upper bound on MMA issuers (drain-barrier space)
constexpr uint32_t kEpiGroups = 4;  // upper bound on epilogue warpgroups (head-weight space)
// MMA issuers (one warp each) and epilogue warpgroups of the N <= 64 and N = 128
// variants; the CTA is the producer warp, the issuer warps and the epilogue warpgroups
__host__ __device__ constexpr uint32_t idx_issuers(bool split) { return split ? 2u : 3u; }
__host__ __device__ constexpr uint32_t idx_epi_groups(bool split) { return split ? 4u : 3u; }
__host__ __device__ constexpr int idx_threads(bool split) {
  return 32 * (1 + static_cast<int>(idx_issuers(split)) + 4 * static_cast<int>(idx_epi_groups(split)));
}
constexpr int kLgStages = 4;
constexpr int kIdxStages = 1 << kLgStages;  // ring capacity in pages (147 KB); a stage holds n_iss pages
constexpr float kInvSqrtDI = 0.08838834764831845f;  // 128^-0.5

// The CTA's range [begin, end) of the flat (group, tile) space, walked as group
// segments: a segment is the run of tiles of one group inside the range, cut at the
// group's last visible tile.  Group-level values are loaded once per segment, so the
// per-tile loops of the single-thread roles stay short.
struct Segment {
  int64_t g;
  int32_t t0, t1;  // tiles [t0, t1) of group g
  int32_t r;       // request of the group
  int32_t nv0, nv1;
  int64_t page_base;
  const int32_t* bt_row;
};

__device__ __forceinline__ bool segment(const IndexArgs& a, int64_t g, int64_t begin, int64_t end, Segment& sg) {
  const int64_t lo = g * a.tpg;
  sg.g = g;
  sg.t0 = static_cast<int32_t>(begin > lo ? begin - lo : 0);
  const int64_t hi = end - lo;
  const int64_t q0 = g * a.G;
  sg.r = __ldg(a.req + q0);
  sg.nv0 = __ldg(a.n_visible + q0);
  sg.nv1 = (a.G > 1 && q0 + 1 < a.n_q) ? __ldg(a.n_visible + q0 + 1) : 0;
  const int32_t vis = min(max(sg.nv0, sg.nv1), a.cache.max_pages * kPage);
  const int32_t n_tiles = (max(vis, 0) + kPage - 1) / kPage;
  const int64_t cap = hi < a.tpg ? hi : a.tpg;
  sg.t1 = static_cast<int32_t>(cap < n_tiles ? cap : n_tiles);
  sg.page_base = static_cast<int64_t>(sg.r) * a.cache.max_pages;
  sg.bt_row = a.cache.block_table ? a.cache.block_table + sg.page_base : nullptr;
  return sg.t0 < sg.t1;
}

// Named barrier over `count` threads that also ANDs a predicate across them.
__device__ __forceinline__ bool named_bar_and(uint32_t id, uint32_t count, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "barrier.cta.red.and.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// kSplit: N = 128 (two queries of 64 heads per group), handled by warpgroup pairs.
// kMx: MXFP4 pages (8704 B, one E8M0 scale per 32 channels, MX block-scaled MMA);
// otherwise 9216-byte pages with one E4M3 scale per 16 channels.
template <bool kSplit, bool kMx>
__global__ void __launch_bounds__(idx_threads(kSplit), 1) index_kernel(const IndexArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int S = kIdxStages;
  constexpr uint32_t kPg = kMx ? kIdxMxPageBytes : kIdxPageBytes;  // bytes per page
  uint8_t* ring = smem;                                                 // S x kPg
  uint8_t* qslot = ring + static_cast<size_t>(S) * kPg;                 // 2 x 9216
  float* sw_all = reinterpret_cast<float*>(qslot + 2 * kIdxPageBytes);  // per epilogue warp: 128 head weights
  uint64_t* bars = reinterpret_cast<uint64_t*>(sw_all + 4 * kEpiGroups * 128);
  uint64_t* full = bars;               // [S]
  uint64_t* empty = full + S;          // [S]
  uint64_t* acc_full = empty + S;      // [8]
  uint64_t* acc_empty = acc_full + 8;  // [8]
  uint64_t* q_full = acc_empty + 8;    // [2]
  uint64_t* q_empty = q_full + 2;      // [2]
  uint64_t* drain = q_empty + 2;       // [kIssuers]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + kIssuers);
  volatile int32_t* abort = reinterpret_cast<volatile int32_t*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t N = static_cast<uint32_t>(a.N);
  // TMEM accumulators.  Accumulator b serves tiles n with n % kAcc == b.  Each
  // accumulator must always be handled by the same issuer and the same epilogue
  // warpgroup, so that no waiter can run two barrier phases ahead (parity waits would
  // alias): the active issuer and warpgroup counts divide kAcc.
  //   N <= 64: six accumulators of N <= 64 columns (0..383); three issuers, issuer i and
  //     warpgroup i serving accumulators i and i + 3, so the warpgroup reads one
  //     accumulator while the MMAs of the other one are in flight.  Key scales at
  //     384..455: each issuer's tiles rotate over three 8-column slots (when tile j's
  //     scales are copied, only its tiles j - 1 and j - 2 can still be in the tensor
  //     pipe: the issuer has seen tile j - 3's accumulator released).  Query scales at
  //     456..503.
  //   N = 128 (two queries of 64 heads): two accumulators (0..255), key scales at
  //     256..319, query scales at 320..383; the four warpgroups pair up, warpgroup w
  //     reads the 64 columns (one query) w >> 1 of accumulator w & 1.
  constexpr uint32_t kAcc = kSplit ? 2u : 6u;
  constexpr uint32_t kSfA = kSplit ? 256u : 384u, kSfB = kSplit ? 320u : 456u;
  constexpr uint32_t n_iss = idx_issuers(kSplit);
  constexpr uint32_t n_st = kIdxStages / n_iss;  // ring stages of n_iss pages
  constexpr bool split_cols = kSplit;
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);       // the producer's one arrive per stage (plus the copies' bytes)
      mbar_init(&empty[i], n_iss);  // one commit per issuer (one page each)
    }
    for (uint32_t i = 0; i < kAcc; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], split_cols ? 256 : 128);  // every reader of the accumulator
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], n_iss);  // released by every active MMA issuer
    }
    for (uint32_t i = 0; i < kIssuers; ++i) mbar_init(&drain[i], 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  pdl_trigger();
  // griddepcontrol.wait (the packed query groups and the new cache entries come from the
  // previous kernel) sits in each role: the producer may copy its first pages before it
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int64_t total = a.n_groups * a.tpg;
  const int64_t begin = total * blockIdx.x / gridDim.x;
  const int64_t end = total * (blockIdx.x + 1) / gridDim.x;
  const uint32_t nib_q = N * 64u;

  const int64_t g_first = begin / a.tpg;
  const int64_t g_last = end > begin ? (end - 1) / a.tpg : g_first - 1;

  if (warp == 0) {
    // -------------------------------------------------------------- producer (one warp)
    // Stage k holds the pages of CTA-local tiles k*n_iss .. k*n_iss + n_iss - 1 (one per
    // issuer).  Without a block table a request's pages are adjacent, so lane 0 moves a
    // stage's pages of one group with a single bulk copy; with a block table each lane
    // looks up and copies one page, so the lookups overlap.  The per-stage work of this
    // warp is kept to a few dozen instructions: it bounds the rate at which the ring refills.
    const uint64_t pol = policy_evict_first();
    uint32_t k = 0, ph = 0, n = 0, n_stages = 0, m = 0;
    bool ok = true;
    Segment sg;
    // Tiles [t, t_end) of segment sg into the ring (the copies of a stage of adjacent
    // pages go as one bulk copy without a block table).
    auto copy_tiles = [&](int32_t& t, int32_t t_end) {
      while (t < t_end) {
        const uint32_t in_st = n % n_iss;
        const int32_t left = t_end - t;
        const int32_t cnt = left < static_cast<int32_t>(n_iss - in_st) ? left : static_cast<int32_t>(n_iss - in_st);
        if (in_st == 0) {
          if (lane == 0) ok = mbar_wait(&empty[k], ph ^ 1u, abort, a.wait_ns);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) return;
        }
        uint8_t* dst = ring + (k * n_iss + in_st) * kPg;
        if (sg.bt_row == nullptr) {
          if (lane == 0) {
            const int64_t page = sg.page_base + t;
            if (page >= 0 && page + cnt <= a.cache.n_pages) {
              const uint32_t bytes = static_cast<uint32_t>(cnt) * kPg;
              mbar_expect_tx(&full[k], bytes);
              bulk_g2s_hint(dst, a.idx_pages + page * kPg, bytes, &full[k], pol);
            } else {
              report(a.err, CSA2_ERR_DEVICE, kInfoPage);
            }
          }
        } else if (lane < cnt) {
          const int64_t page = __ldg(sg.bt_row + t + lane);
          if (page >= 0 && page < a.cache.n_pages) {
            mbar_expect_tx(&full[k], kPg);
            bulk_g2s_hint(dst + lane * kPg, a.idx_pages + page * kPg, kPg, &full[k], pol);
          } else {
            report(a.err, CSA2_ERR_DEVICE, kInfoPage);
          }
        }
        __syncwarp();
        t += cnt;
        n += static_cast<uint32_t>(cnt);
        if (n % n_iss == 0) {
          if (lane == 0) mbar_arrive(&full[k]);
          ++n_stages;
          if (++k == n_st) {
            k = 0;
            ph ^= 1u;
          }
        }
      }
    };
    // The first pages of the CTA's range go before griddepcontrol.wait (early), up to the
    // ring's capacity and short of the first page holding an entry the pack kernel writes
    // for the segment's request.  Only without a block table: a request's pages are then its
    // own (page = request * max_pages + tile), so the pack kernel's writes are known by
    // (request, tile) alone.
    bool waited = false;
    if (a.early == 0 || a.cache.block_table != nullptr) {
      pdl_wait();
      waited = true;
    }
    for (int64_t g = g_first; ok && g <= g_last; ++g) {
      if (!segment(a, g, begin, end, sg)) continue;
      int32_t t = sg.t0;
      if (!waited) {
        int32_t first_new = sg.t1;  // first tile of this request written by the pack kernel
        for (int64_t i = lane; i < a.n_new; i += 32)
          if (__ldg(a.new_req + i) == sg.r) {
            const int64_t tp = __ldg(a.new_pos + i) / kPage;
            if (tp >= sg.t0 && tp < first_new) first_new = static_cast<int32_t>(tp);
          }
        first_new = __reduce_min_sync(0xffffffffu, first_new);
        int32_t t_end = sg.t0 + static_cast<int32_t>(n_st * n_iss);
        t_end = t_end < first_new ? t_end : first_new;
        copy_tiles(t, t_end);
        pdl_wait();
        waited = true;
      }
      if (!ok) break;
      if (lane == 0) {
        const uint32_t slot = m & 1u;
        ok = mbar_wait(&q_empty[slot], ((m >> 1) & 1u) ^ 1u, abort, a.wait_ns);
        if (ok) {
          mbar_arrive_expect_tx(&q_full[slot], static_cast<uint32_t>(a.grp_bytes));
          bulk_g2s(qslot + slot * kIdxPageBytes, a.qpack + g * a.grp_bytes, static_cast<uint32_t>(a.grp_bytes),
                   &q_full[slot]);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      ++m;
      copy_tiles(t, sg.t1);
    }
    if (!waited) pdl_wait();  // no segment at all
    if (lane == 0) {
      // a partial last stage (also one left open when a wait ran out at a group boundary:
      // its copies are in flight) is closed, so that the drain below waits for it too
      if (n % n_iss != 0) {
        mbar_arrive(&full[k]);
        ++n_stages;
      }
      if (!ok) {
        *abort = 1;
        report(a.err, CSA2_ERR_TIMEOUT, kInfoWait);
      }
      // the copies of the last stages land before the CTA exits
      for (uint32_t j = (n_stages > n_st ? n_stages - n_st : 0); j < n_stages; ++j)
        mbar_drain_wait(&full[j % n_st], (j / n_st) & 1u);
      for (uint32_t j = (m > 2 ? m - 2 : 0); j < m; ++j) mbar_drain_wait(&q_full[j & 1u], (j >> 1) & 1u);
    }
  } else if (warp >= 1 && warp <= static_cast<int>(n_iss)) {
    if (lane == 0 && static_cast<uint32_t>(warp - 1) < n_iss) {
      // ------------------------------------------------------------ MMA issuers
      pdl_wait();
      // issuer i takes the tiles n with n % n_iss == i: a single thread pays ~130 cycles per
      // dependent tcgen05 op, so the issuers (three, or two for N = 128) sit on different
      // warps to keep the tensor pipe and the copy ring moving
      const uint32_t me = static_cast<uint32_t>(warp - 1);
      const uint32_t idesc = idesc_nvf4(128, a.N);
      const uint32_t idesc_mx[2] = {idesc_mxf4(128, a.N, 0u), idesc_mxf4(128, a.N, 2u)};
      uint32_t n = 0, m = 0, cur = 0, j = 0;
      bool ok = true;
      Segment sg;
      for (int64_t g = g_first; ok && g <= g_last; ++g) {
        if (!segment(a, g, begin, end, sg)) continue;
        if (m > 0) mma_commit(&q_empty[(m - 1) & 1u]);  // previous query slot is free once its MMAs finish
        cur = m & 1u;
        ok = mbar_wait(&q_full[cur], (m >> 1) & 1u, abort, a.wait_ns);
        if (!ok) break;
        tc_fence_after();
        const uint32_t qs = smem_u32(qslot + cur * kIdxPageBytes);
        const uint32_t sfb = tmem + kSfB + 16u * me + 8u * cur;
        tmem_cp_sf(sfb, sdesc(qs + nib_q, 128, 128));
        if (!kMx) tmem_cp_sf(sfb + 4, sdesc(qs + nib_q + 512, 128, 128));
        ++m;
        // CTA-local tiles n .. n + len - 1 belong to this segment; this issuer's are the
        // ones with nn % n_iss == me
        const uint32_t len = static_cast<uint32_t>(sg.t1 - sg.t0);
        for (uint32_t nn = n + (me + n_iss - n % n_iss) % n_iss; nn < n + len; nn += n_iss, ++j) {
          const uint32_t kst = nn / n_iss;
          const uint32_t s = kst % n_st, ph = (kst / n_st) & 1u;
          const uint32_t b = nn % kAcc, bph = (nn / kAcc) & 1u;
          ok = mbar_wait(&full[s], ph, abort, a.wait_ns);
          if (!ok) break;
          tc_fence_after();
          const uint32_t st = smem_u32(ring + (s * n_iss + me) * kPg);
          const uint32_t sfa = tmem + (kSplit ? kSfA + 16u * b + 8u * bph : kSfA + 24u * me + 8u * (j % 3u));
          tmem_cp_sf(sfa, sdesc(st + kIdxNibBytes, 128, 128));
          if (!kMx) tmem_cp_sf(sfa + 4, sdesc(st + kIdxNibBytes + 512, 128, 128));
          ok = mbar_wait(&acc_empty[b], bph ^ 1u, abort, a.wait_ns);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (uint32_t kk = 0; kk < 2; ++kk) {
            if (kMx)  // one scale column per row; the two K halves use its bytes 0-1 and 2-3
              mma_mxf4(tmem + b * N, sdesc(st + kk * 256u, 128, 512), sdesc(qs + kk * 256u, 128, 512),
                       idesc_mx[kk], sfa, sfb, kk);
            else
              mma_nvf4(tmem + b * N, sdesc(st + kk * 256u, 128, 512), sdesc(qs + kk * 256u, 128, 512), idesc,
                       sfa + 4u * kk, sfb + 4u * kk, kk);
          }
          mma_commit(&empty[s]);
          mma_commit(&acc_full[b]);
        }
        n += len;
      }
      if (!ok) {
        *abort = 1;
        report(a.err, CSA2_ERR_TIMEOUT, kInfoWait);
      }
      mma_commit(&drain[me]);
      mbar_drain_wait(&drain[me], 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    pdl_wait();
    // thread = TMEM lane = key.  N <= 64: warpgroup wg takes the tiles with n % 3 == wg
    // and every column; N = 128: the tiles with n % 2 == wg % 2 and the 64 columns (the
    // query) wg / 2.
    const uint32_t wg = static_cast<uint32_t>(warp - 1 - static_cast<int>(n_iss)) >> 2;
    constexpr uint32_t wg_step = split_cols ? 2u : 3u;
    const uint32_t wg_res = split_cols ? (wg & 1u) : wg;
    const uint32_t c_lo = split_cols ? 64u * (wg >> 1) : 0u, c_hi = split_cols ? c_lo + 64u : N;
    const int quarter = warp & 3;
    // one leader warp per warpgroup polls the accumulator barrier; the other three park
    // on a named barrier and cost no issue slots while they wait
    const bool leader = static_cast<uint32_t>(quarter) == ((wg + 1u) & 3u);
    const uint32_t row = static_cast<uint32_t>(quarter * 32 + lane);
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    float* sw = sw_all + (warp - 1 - static_cast<int>(n_iss)) * 128;  // this warp's copy of the group's head weights
    float wr[kSplit ? 1 : 64];  // N <= 64: the group's head weights, one per accumulator column
    uint32_t n = 0;
    bool ok = true;
    Segment sg;
    for (int64_t g = g_first; ok && g <= g_last; ++g) {
      if (!segment(a, g, begin, end, sg)) continue;
      const int64_t q0 = g * a.G;
      __syncwarp();
      for (int i = lane; i < a.N; i += 32) {
        const int64_t q = q0 + i / a.heads_I;
        sw[i] = q < a.n_q ? __ldg(a.w + q * a.heads_I + i % a.heads_I) : 0.0f;
        if (q < a.n_q && __ldg(a.req + q) != sg.r) report(a.err, CSA2_ERR_DEVICE, kInfoGroup);
      }
      __syncwarp();
      if constexpr (!kSplit) {
#pragma unroll
        for (int i = 0; i < 64; ++i) wr[i] = static_cast<uint32_t>(i) < N ? sw[i] : 0.0f;
      }
      const int nq = static_cast<int>(a.n_q - q0 < a.G ? a.n_q - q0 : a.G);
      const uint32_t len = static_cast<uint32_t>(sg.t1 - sg.t0);
      // this warpgroup's first tile of the segment; its accumulator, phase and tile index
      // then advance by wg_step tiles per iteration
      const uint32_t nn0 = n + (wg_res + wg_step - n % wg_step) % wg_step;
      uint32_t ab = nn0 % kAcc, ap = (nn0 / kAcc) & 1u;
      int32_t t = sg.t0 + static_cast<int32_t>(nn0 - n);
      float* const srow = a.scores + q0 * a.ld;  // the group's first score row
      // without a block table the segment's pages are adjacent: checked once here
      const bool seg_pages_ok =
          sg.bt_row != nullptr || (sg.page_base + sg.t0 >= 0 && sg.page_base + sg.t1 <= a.cache.n_pages);
      for (uint32_t nn = nn0; nn < n + len; nn += wg_step, t += static_cast<int32_t>(wg_step)) {
        const uint32_t bb = ab, bp = ap;
        ab += wg_step;
        if (ab >= kAcc) {
          ab -= kAcc;
          ap ^= 1u;
        }
        bool page_ok = seg_pages_ok;
        if (sg.bt_row != nullptr) {
          const int64_t page = __ldg(sg.bt_row + t);
          page_ok = page >= 0 && page < a.cache.n_pages;
        }
        // the leader warp waits for the accumulator; the barrier hands its result to the
        // other three warps (which wait there without issuing)
        const bool got = leader ? mbar_wait(&acc_full[bb], bp, abort, a.wait_ns) : true;
        if (!named_bar_and(1u + wg, 128u, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int32_t key = t * kPage + static_cast<int32_t>(row);
        const uint32_t hmask = static_cast<uint32_t>(a.heads_I) - 1u;
        const uint32_t lg_h = a.heads_I == 64 ? 6u : 5u;
        float2 acc01 = make_float2(0.0f, 0.0f), acc23 = make_float2(0.0f, 0.0f);
        if constexpr (!kSplit) {
          // head weights from registers (loaded once per group), two 32-column chunks
#pragma unroll
          for (uint32_t cc = 0; cc < 2; ++cc) {
            if (cc == 1 && N <= 32u) break;
            uint32_t r[32];
            tmem_ld32(tmem + lane_base + bb * N + 32u * cc, r);
            tmem_ld_wait();
            if (cc == 1 || N <= 32u) {
              tc_fence_before();
              mbar_arrive(&acc_empty[bb]);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              fma2(acc01, make_float2(wr[32 * cc + 4 * i + 0], wr[32 * cc + 4 * i + 1]),
                   make_float2(fmaxf(__uint_as_float(r[4 * i + 0]), 0.0f), fmaxf(__uint_as_float(r[4 * i + 1]), 0.0f)));
              fma2(acc23, make_float2(wr[32 * cc + 4 * i + 2], wr[32 * cc + 4 * i + 3]),
                   make_float2(fmaxf(__uint_as_float(r[4 * i + 2]), 0.0f), fmaxf(__uint_as_float(r[4 * i + 3]), 0.0f)));
            }
            if (((32u * cc + 32u) & hmask) == 0) {
              const int gq = static_cast<int>((32u * cc) >> lg_h);
              if (gq < nq && page_ok && key < (gq == 0 ? sg.nv0 : sg.nv1))
                (gq == 0 ? srow : srow + a.ld)[key] = ((acc01.x + acc01.y) + (acc23.x + acc23.y)) * kInvSqrtDI;
              acc01 = acc23 = make_float2(0.0f, 0.0f);
            }
          }
        } else {  // N = 128: weights from shared memory (the 19-warp CTA has no registers for them)
          for (uint32_t c = c_lo; c < c_hi; c += 32u) {
            uint32_t r[32];
            tmem_ld32(tmem + lane_base + bb * N + c, r);
            tmem_ld_wait();
            if (c + 32u >= c_hi) {
              tc_fence_before();
              mbar_arrive(&acc_empty[bb]);
            }
            const float4* w4 = reinterpret_cast<const float4*>(sw + c);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 wv = w4[i];
              fma2(acc01, make_float2(wv.x, wv.y),
                   make_float2(fmaxf(__uint_as_float(r[4 * i + 0]), 0.0f), fmaxf(__uint_as_float(r[4 * i + 1]), 0.0f)));
              fma2(acc23, make_float2(wv.z, wv.w),
                   make_float2(fmaxf(__uint_as_float(r[4 * i + 2]), 0.0f), fmaxf(__uint_as_float(r[4 * i + 3]), 0.0f)));
            }
            if (((c + 32u) & hmask) == 0) {
              const int gq = static_cast<int>(c >> lg_h);
              if (gq < nq && page_ok && key < (gq == 0 ? sg.nv0 : sg.nv1))
                (gq == 0 ? srow : srow + a.ld)[key] = ((acc01.x + acc01.y) + (acc23.x + acc23.y)) * kInvSqrtDI;
              acc01 = acc23 = make_float2(0.0f, 0.0f);
            }
          }
        }
      }
      n += len;
    }
    if (!ok) {
      *abort = 1;
      report(a.err, CSA2_ERR_TIMEOUT, kInfoWait);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

size_t index_smem_bytes(int stages) {
  (void)stages;
  return 1024 + static_cast<size_t>(kIdxStages + 2) * kIdxPageBytes + 4 * kEpiGroups * 128 * sizeof(float) +
         (2 * kIdxStages + 20 + kIssuers) * sizeof(uint64_t) + 16 + 4 * 2;
}

cudaError_t launch_index(const IndexArgs& a, int grid, cudaStream_t stream) {
  const size_t smem = index_smem_bytes(a.stages);
  static std::atomic<int> limit_set[4][kMaxDevices];
  const bool split = a.N == 128, mx = a.cache.idx_format == CSA2_IDX_MXFP4;
  auto* kernel = mx ? (split ? index_kernel<true, true> : index_kernel<false, true>)
                    : (split ? index_kernel<true, false> : index_kernel<false, false>);
  cudaError_t e =
      smem_limit_once(reinterpret_cast<const void*>(kernel), smem, limit_set[(split ? 1 : 0) + (mx ? 2 : 0)]);
  if (e != cudaSuccess) return e;
  return launch_pdl(kernel, dim3(static_cast<unsigned>(grid)), dim3(static_cast<unsigned>(idx_threads(split))), smem,
                    stream, nullptr, a);
}

}  // namespace csa2
