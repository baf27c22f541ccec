// k_attn.cu -- shared-KV MQA over the selected FP4 entries plus the sliding window.
//
// "DeepSeek's Attention and KV Cache - From MLA to CSA2", "DeepSeek-V4": a query
// attends to the top-512 selected entries concatenated with the 128 window entries;
// each entry is one 512-wide vector serving as both key and value.  "DeepSeek-V4.1":
// the FP4 entries are dequantised before attention.  "From MLA to DSA to HCA/CSA",
// "What replaced MLA": attention(q, kv, kv) with K and V the same tensor.
//
// Design: one CTA of 16 warps per (query, key split), all 64 heads, so every selected
// record is dequantised once.  A query's key tiles are [window, selected 0..3] (128 keys
// each); S CTAs of a thread-block cluster take consecutive runs of them and merge their
// partial outputs through L2 after a cluster barrier (S = 1 needs no merge).
//   operands  f16: the dequantised entries (e2m1 x e4m3 products are exact in f16), the
//             window rows and the queries (bf16 -> f16 is exact in f16's range), and the
//             probabilities P (8 more bits than bf16);
//   tile      one f16 K = V buffer [128 keys][512] in the core-matrix layout, seen as four
//             128-channel chunks.  The O MMAs of tile t free the chunks one by one, and
//             tile t+1 is dequantised into each freed chunk (its records were loaded into
//             registers one tile ahead) while the later O chunks and the S MMAs of the
//             chunks already built run on the tensor pipe;
//   S^T      tcgen05.mma kind::f16, M = 128 keys, N = 64 heads, K = 512, as two partial sums
//             over alternate channel chunks (TMEM cols 256..383);
//   softmax  thread = key, 16 heads per thread: a block-wide vote finds whether any score
//             exceeds its head's reference maximum by 2^8; only then are the reference
//             maxima raised (warp max reductions) and O^T and the running sums rescaled;
//   O^T      += V^T P^T: 4 output chunks of 128 channels x 64 heads (TMEM cols 0..255)
//             reading the same tile as an MN-major operand (K == V);
//   epilogue O = O^T / l per head -> bf16 and lse; with S > 1 the CTAs write their raw
//             partials and (max, sum) per head to the workspace and one cluster barrier
//             orders them: with S = 2 the second CTA adds the first one's partial to its
//             own accumulator as it writes the output, with S > 2 each CTA of the
//             cluster combines one slice of the heads.
// Optional, from "From MLA to DSA to HCA/CSA": per-head attention sinks (a logit that
// joins the softmax denominator and has no value; section "The sliding window") and
// the partial RoPE of "What replaced MLA" (the queries' trailing 64 channels rotated
// before the first S^T MMA; the output's rotated back with the negated angle before it
// is rounded to bf16), and windows read from the FP8 ring.
#include "csa2_kernels.cuh"

namespace csa2 {

constexpr int kComputeWarps = 16;  // softmax, tile build, epilogue; lane 0 of warps 0..3 issues MMAs
constexpr int kComputeThreads = 32 * kComputeWarps;
constexpr int kAttnThreads = kComputeThreads;
constexpr int kHeads = 64;
constexpr uint32_t kKtBytes = 128 * 512 * 2;  // f16 key/value tile
constexpr uint32_t kQsBytes = 64 * 512 * 2;   // f16 queries, all heads
constexpr uint32_t kPsBytes = 128 * 64 * 2;   // f16 P^T
constexpr uint32_t kSCol = 256;               // TMEM: O^T chunk c at columns 64c.., S^T partial i at 256 + 64i
constexpr float kRescaleThreshold = 8.0f;     // log2 units
// shared memory map (bytes)
constexpr uint32_t kOffQs = kKtBytes;
constexpr uint32_t kOffPs = kOffQs + kQsBytes;
constexpr uint32_t kOffRec = kOffPs + kPsBytes;     // int32 [512] record ids (page * 128 + slot), -1 = none
constexpr uint32_t kOffCnt = kOffRec + 512 * 4;     // int32 [4] valid entries per selected tile
constexpr uint32_t kOffAlpha = kOffCnt + 16;        // f32 [64] per-head factor
constexpr uint32_t kOffRef = kOffAlpha + 64 * 4;    // f32 [64] reference maximum (log2 units)
constexpr uint32_t kOffMl = kOffRef + 64 * 4;       // f32 [2][64] (max, sum) published to the cluster
constexpr uint32_t kOffBar = kOffMl + 128 * 4;      // u64 s_bar, o_bar[4], drain
constexpr uint32_t kOffMisc = kOffBar + 6 * 8;      // u32 tmem slot, i32 abort flag, 2 spare
constexpr uint32_t kAttnSmem = kOffMisc + 16;

// Offset of element (row, col) in a [rows][512] 16-bit operand tile stored as 8x8 core
// matrices: row groups of 8 at 8192-byte stride, 8-column chunks at 128-byte stride.
__device__ __forceinline__ uint32_t tile_off(uint32_t row, uint32_t col) {
  return (row >> 3) * 8192u + (col >> 3) * 128u + (row & 7u) * 16u + (col & 7u) * 2u;
}

// Work item c of a [rows][64 chunks of 16 bytes] tile -> (row, chunk).  A warp's 32
// items cover 8 consecutive rows x 4 consecutive chunks: each group of 8 lanes writes
// one 128-byte line of the core-matrix layout (no bank conflicts), and each row's 4
// chunks are 64 contiguous bytes of the source row (whole 32-byte sectors).
__device__ __forceinline__ void tile_item(uint32_t c, uint32_t rows, uint32_t& row, uint32_t& chunk) {
  const uint32_t rg = rows >> 3;  // row groups
  row = (c & 7u) | (((c >> 5) % rg) << 3);
  chunk = ((c >> 3) & 3u) | ((c >> 5) / rg << 2);
}

__device__ __forceinline__ void cp_async16(uint32_t sdst, const void* gsrc, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(sdst), "l"(gsrc), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// Barrier over every thread of the cluster; release/acquire orders the partials each CTA
// wrote to global memory before it.
__device__ __forceinline__ void attn_cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Per-head sum of the four lane quarters' partial sums ([4][64] in shared memory).
__device__ __forceinline__ float lred_sum(const float* lred, int h) {
  return lred[h] + lred[64 + h] + lred[128 + h] + lred[192 + h];
}

// 2^x by the hardware approximation (PTX ex2.approx, at most 2 ulp from the exact value),
// denormal results flushed to zero: the softmax's P values are rounded to f16 next, whose
// smallest subnormal (2^-24) lies far above the flushed range.
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Named barrier 1 over the CTA's 512 threads, and its OR-reduction form.
__device__ __forceinline__ void cbar_sync() { asm volatile("bar.sync 1, 512;" ::: "memory"); }
__device__ __forceinline__ bool cbar_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "barrier.cta.red.or.pred p, 1, 512, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v))
      : "memory");
  return r != 0;
}

// kExt: the optional features (sinks, partial RoPE, FP8 window ring) are compiled in;
// the plain instance carries none of their code.
template <bool kExt>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_kernel(const AttnArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* Kt = smem;
  uint8_t* Qs = smem + kOffQs;
  uint8_t* Ps = smem + kOffPs;
  int32_t* recid = reinterpret_cast<int32_t*>(smem + kOffRec);
  int32_t* tile_cnt = reinterpret_cast<int32_t*>(smem + kOffCnt);
  float* alpha = reinterpret_cast<float*>(smem + kOffAlpha);
  float* ref_s = reinterpret_cast<float*>(smem + kOffRef);
  float* ml = reinterpret_cast<float*>(smem + kOffMl);
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(smem + kOffBar);  // S of a tile complete
  uint64_t* o_bar = s_bar + 1;                                     // [4] O chunk c complete
  uint64_t* drain = s_bar + 5;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int32_t* abort = reinterpret_cast<volatile int32_t*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Two MMA-issuing threads, lane 0 of warps 0 and 1 (one thread issues a dependent MMA
  // about every 66 cycles, two keep the tensor pipe busy): issuer i owns the 128-channel
  // chunks c with c % 2 == i (their S^T partial i and their O^T chunks).  Building warps
  // hand each built chunk over with a non-blocking barrier arrival and only the chunk's
  // issuer warp waits there, so an MMA issue that stalls on a full tensor-core queue holds
  // up that warp alone.
  const bool issuer = warp < 2 && lane == 0;
  const int qd = warp & 3;   // TMEM lane quarter of this warp
  const int hg = warp >> 2;  // head group: heads [16 hg, 16 hg + 16) in the softmax, O chunk hg
  const int S = a.splits;    // CTAs per query (one cluster)
  const int64_t qi = blockIdx.x / S;
  const int sp = static_cast<int>(blockIdx.x % S);  // rank in the cluster
  // this CTA's run [t_lo, t_hi) of the tile list [window, selected 0, 1, 2, 3]
  const int t_lo = sp * 5 / S, t_hi = (sp + 1) * 5 / S;
  const bool has_win = t_lo == 0;
  const int sel_lo = has_win ? 0 : t_lo - 1, sel_hi = t_hi - 1;  // selected tiles [sel_lo, sel_hi)
  const int32_t nv = __ldg(a.n_visible + qi);
  const int32_t wl = has_win ? max(0, min(CSA2_WIN, __ldg(a.win_len + qi))) : 0;
  const bool ring = kExt && a.win_ring != nullptr;
  const bool rope = kExt && a.rope_cos != nullptr;
  const bool win_tile = has_win && wl > 0;  // an empty window is no tile

  if (tid == 0) {
    mbar_init(s_bar, 2);  // one commit per issuer and tile, after its last S^T chunk
    for (int i = 0; i < 4; ++i) mbar_init(&o_bar[i], 1);
    mbar_init(drain, 2);  // one commit per issuer
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  pdl_trigger();
  // The queries go to registers and the window's bf16 rows (for the window's CTA) to the
  // key tile with cp.async: both are this call's inputs, so the loads overlap the previous
  // kernel's tail.  The f16 conversion follows (the window's chunk by chunk, in place).
  uint4 qv[8];
  {
    const __nv_bfloat16* qg = a.q + qi * kHeads * CSA2_D;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t h, ch;
      tile_item(static_cast<uint32_t>(tid + kComputeThreads * i), kHeads, h, ch);
      qv[i] = __ldg(reinterpret_cast<const uint4*>(qg + h * CSA2_D + ch * 8));
    }
    if (win_tile && !ring) {
      const __nv_bfloat16* wg = a.window + __ldg(a.win_start + qi) * CSA2_D;
      for (int c = tid; c < 128 * 64; c += kComputeThreads) {
        uint32_t r, ch;
        tile_item(static_cast<uint32_t>(c), 128, r, ch);
        const bool ok = static_cast<int32_t>(r) < wl;
        cp_async16(smem_u32(Kt + tile_off(r, ch * 8)),
                   ok ? static_cast<const void*>(wg + r * CSA2_D + ch * 8) : static_cast<const void*>(a.window),
                   ok ? 16u : 0u);
      }
      cp_async_commit();
    }
  }
  // the selected indices (and in Full mode the new entries, or the window ring) come from
  // earlier kernels
  pdl_wait();
  const int tsel = tid >> 7;  // 512 compute threads: one selected slot each
  const bool mine = tsel >= sel_lo && tsel < sel_hi;
  const int32_t e_sel = mine ? __ldg(a.topk_idx + qi * CSA2_TOPK + tid) : -1;
  if (tid < 4) tile_cnt[tid] = 0;
  auto cvt16 = [](uint4 v) {  // 8 bf16 -> 8 f16
    return make_uint4(f16x2_sat(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u)),
                      f16x2_sat(__uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u)),
                      f16x2_sat(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xFFFF0000u)),
                      f16x2_sat(__uint_as_float(v.w << 16), __uint_as_float(v.w & 0xFFFF0000u)));
  };
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t h, ch;
    tile_item(static_cast<uint32_t>(tid + kComputeThreads * i), kHeads, h, ch);
    *reinterpret_cast<uint4*>(Qs + tile_off(h, ch * 8)) = cvt16(qv[i]);
  }
  __syncthreads();  // tile_cnt cleared
  {
    int32_t rid = -1;
    if (e_sel >= 0) {
      const int64_t pg = e_sel < nv ? page_id(a.cache, __ldg(a.req + qi), e_sel) : -1;
      if (pg >= 0 && pg < a.cache.n_pages && pg < (int64_t(1) << 24))
        rid = static_cast<int32_t>(pg * kPage + e_sel % kPage);
      else
        report(a.err, CSA2_ERR_DEVICE, kInfoTopkIdx);
    }
    recid[tid] = rid;
    if (rid >= 0) atomicAdd(&tile_cnt[tsel], 1);
  }
  if (kExt && win_tile && ring) {
    // FP8 window ring: row i of the tile is the entry of position newest - i; E4M3 -> f16 in
    // hardware (exact), times the block's 2^e in fp32, -> f16
    const int64_t newest = __ldg(a.win_start + qi);
    const int32_t r = __ldg(a.req + qi);
    const bool ring_ok = r >= 0 && r < a.win_ring_reqs && newest - wl + 1 >= 0;
    if (!ring_ok && tid == 0) report(a.err, CSA2_ERR_DEVICE, kInfoPos);
#pragma unroll 1
    for (int i = 0; i < 4; ++i) {
      const uint32_t task = static_cast<uint32_t>(tid + kComputeThreads * i);
      const uint32_t row = (task & 7u) | (((task >> 5) & 15u) << 3);
      const uint32_t j = ((task >> 3) & 3u) | ((task >> 9) << 2);  // 32-channel block
      uint8_t* dst = Kt + tile_off(row, 32 * j);
      if (!ring_ok || static_cast<int32_t>(row) >= wl) {  // no entry: zeros (masked)
#pragma unroll
        for (int m = 0; m < 4; ++m) *reinterpret_cast<uint4*>(dst + m * 128) = make_uint4(0, 0, 0, 0);
        continue;
      }
      const int64_t pos = newest - row;
      const uint8_t* rec = a.win_ring + (static_cast<int64_t>(r) * CSA2_WIN + pos % CSA2_WIN) * CSA2_WIN_BYTES;
      const uint4 c0 = __ldg(reinterpret_cast<const uint4*>(rec + 32 * j));
      const uint4 c1 = __ldg(reinterpret_cast<const uint4*>(rec + 32 * j + 16));
      const float sc = ldexpf(1.0f, static_cast<int>(__ldg(rec + 512 + j)) - 127);
      const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 f = __half22float2(e4m3x2_f16x2((cw[2 * m + (k >> 1)] >> (16 * (k & 1))) & 0xFFFFu));
          o[k] = f16x2_sat(f.x * sc, f.y * sc);
        }
        *reinterpret_cast<uint4*>(dst + m * 128) = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
  if (tid < kHeads) ref_s[tid] = ml[tid] = -INFINITY;  // ml[0..63]: the vote's bound ref + 2^8 during the tiles
  tc_fence_before();
  __syncthreads();  // record ids, tile counts, converted queries (and the ring window)
  tc_fence_after();
  if (rope) {
    // q = q cos + rotate_half(q) sin on channels 448 + i / 480 + i (angle i), in f16 after
    // the conversion (one rounding of the fp32 rotation of the exact inputs)
    for (int p = tid; p < kHeads * 32; p += kAttnThreads) {
      const uint32_t h = static_cast<uint32_t>(p) >> 5, i = static_cast<uint32_t>(p) & 31u;
      const float c = __ldg(a.rope_cos + qi * 32 + i), sn = __ldg(a.rope_sin + qi * 32 + i);
      __half* pa = reinterpret_cast<__half*>(Qs + tile_off(h, 448u + i));
      __half* pb = reinterpret_cast<__half*>(Qs + tile_off(h, 480u + i));
      const float x = __half2float(*pa), y = __half2float(*pb);
      const uint32_t two = f16x2_sat(x * c - y * sn, y * c + x * sn);
      *reinterpret_cast<uint16_t*>(pa) = static_cast<uint16_t>(two & 0xFFFFu);
      *reinterpret_cast<uint16_t*>(pb) = static_cast<uint16_t>(two >> 16);
    }
    __syncthreads();
  }
  const uint32_t tmem = *tmem_slot;

  auto next_sel = [&](int t) {  // first selected tile of this run after t with an entry, or -1
    int u = t + 1;
    while (u < sel_hi && tile_cnt[u] == 0) ++u;
    return u < sel_hi ? u : -1;
  };
  const int first = win_tile ? 4 : next_sel(sel_lo - 1);  // 4: the window tile; -1: none
  auto after = [&](int t) { return t == 4 ? next_sel(sel_lo - 1) : next_sel(t); };  // the tile after t

  bool ok = true;
  bool o_started = false;
  uint32_t oph = 0;  // parity of the next O completion
  const uint32_t idesc_s = idesc_f16(128, kHeads, 0, 0);
  const uint32_t idesc_o = idesc_f16(128, kHeads, 1, 1);
  // S^T partial (c % 2) += K_c Q_c^T over the channels of chunk c (its issuer, once the
  // chunk is built); both partials are complete after chunks 2 and 3
  auto issue_s = [&](int c) {
    if (issuer && warp == (c & 1)) {
      const uint64_t dK0 = sdesc(smem_u32(Kt), 128, 8192), dQ0 = sdesc(smem_u32(Qs), 128, 8192);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        mma_f16(tmem + kSCol + 64u * static_cast<uint32_t>(c & 1), dK0 + static_cast<uint64_t>(16 * (8 * c + k)),
                dQ0 + static_cast<uint64_t>(16 * (8 * c + k)), idesc_s, (c > 1 || k > 0) ? 1u : 0u);
      if (c > 1) mma_commit(s_bar);
    }
  };
  // O^T chunks (issuer i: i, then i + 2; after the block barrier that follows the P
  // stores); o_bar[c] completes when chunk c has been computed
  auto issue_o = [&]() {
    if (issuer) {
      const uint64_t dV0 = sdesc(smem_u32(Kt), 8192, 128), dP0 = sdesc(smem_u32(Ps), 1024, 128);
#pragma unroll
      for (uint32_t j = 0; j < 2; ++j) {
        const uint32_t c = static_cast<uint32_t>(warp) + 2u * j;
#pragma unroll
        for (uint32_t kk = 0; kk < 8; ++kk)
          mma_f16(tmem + 64u * c, dV0 + static_cast<uint64_t>(128u * c + 1024u * kk),
                  dP0 + static_cast<uint64_t>(128u * kk), idesc_o, (o_started || kk > 0) ? 1u : 0u);
        mma_commit(&o_bar[c]);
      }
    }
  };
  {
    // ================================================================ the tiles
    // register prefetch of a selected tile: thread = (key 8 warp + lane % 8, 32-channel
    // piece lane / 8 of each 128-channel chunk); per chunk 16 bytes of nibbles.  The
    // record's 32 scale bytes are loaded once per tile, 16 bytes by each of the key's
    // lanes with piece 0 and 1 (chunks 0-1 and 2-3), and handed to the other lanes by
    // shuffles: the narrow per-chunk scale loads doubled the load instructions that the
    // memory pipeline accepts only slowly for scattered records.
    const uint32_t bkey = static_cast<uint32_t>(8 * warp + (lane & 7));
    const uint32_t bj = static_cast<uint32_t>(lane >> 3);
    uint4 pn[4];
    uint4 sq = make_uint4(0u, 0u, 0u, 0u);
    // chunk c of selected tile ts (ts < 0 or 4: nothing); c == 3 also loads the scales (the
    // current tile's are no longer needed once its last chunk is dequantised)
    auto prefetch_chunk = [&](int ts, int c) {
      const int32_t rid = (ts < 0 || ts == 4) ? -1 : recid[ts * 128 + static_cast<int>(bkey)];
      if (rid >= 0) {
        const uint8_t* rec = a.cache.kv + static_cast<int64_t>(rid) * kKvBytes;
        pn[c] = __ldg(reinterpret_cast<const uint4*>(rec + 64 * c + 16 * bj));
        if (c == 3 && bj < 2u) sq = __ldg(reinterpret_cast<const uint4*>(rec + 256 + 16 * bj));
      } else {  // no entry: zeros (masked below)
        pn[c] = make_uint4(0u, 0u, 0u, 0u);
        if (c == 3) sq = make_uint4(0u, 0u, 0u, 0u);
      }
    };
    uint32_t dq[16];
    auto dequant_chunk = [&](int c) {  // registers -> 32 f16 values of this thread's piece
      // scale bytes 8c + 2bj, 8c + 2bj + 1 of the record: word 2 (c % 2) + bj / 2, half
      // bj % 2 of the 16 bytes held by the key's lane with piece c / 2
      const uint32_t src = (static_cast<uint32_t>(lane) & 7u) + 8u * static_cast<uint32_t>(c >> 1);
      const uint32_t w0 = __shfl_sync(0xffffffffu, (c & 1) ? sq.z : sq.x, static_cast<int>(src));
      const uint32_t w1 = __shfl_sync(0xffffffffu, (c & 1) ? sq.w : sq.y, static_cast<int>(src));
      const uint32_t wsel = (bj >> 1) ? w1 : w0;
      const uint32_t sc2 = e4m3x2_f16x2_bits((bj & 1u) ? (wsel >> 16) : (wsel & 0xFFFFu));
      const uint32_t s0 = prmt(sc2, sc2, 0x1010u), s1 = prmt(sc2, sc2, 0x3232u);
      const uint32_t wds[4] = {pn[c].x, pn[c].y, pn[c].z, pn[c].w};
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        uint32_t o[4];
        dequant8_f16(wds[m], m < 2 ? s0 : s1, o);
#pragma unroll
        for (int k = 0; k < 4; ++k) dq[4 * m + k] = o[k];
      }
    };
    auto store_chunk = [&](int c) {
#pragma unroll
      for (int m = 0; m < 4; ++m)
        *reinterpret_cast<uint4*>(Kt + tile_off(bkey, 128u * c + 32u * bj + 8u * m)) =
            make_uint4(dq[4 * m], dq[4 * m + 1], dq[4 * m + 2], dq[4 * m + 3]);
    };
    // chunk c is in place (and every S load is done): the chunk's issuer warp waits for
    // every warp's part and issues its S MMAs; the other warps arrive and go on
    auto chunk_done = [&](int c) {
      fence_proxy_async_smem();
      tc_fence_before();
      if (warp == (c & 1)) {
        named_bar_sync(2u + static_cast<uint32_t>(c), 512u);
        tc_fence_after();
        issue_s(c);
      } else {
        named_bar_arrive(2u + static_cast<uint32_t>(c), 512u);
      }
    };

    int cur = first;
#pragma unroll
    for (int c = 0; c < 4; ++c) prefetch_chunk(cur == 4 ? after(4) : cur, c);
    // ---- the first tile: the window (converted to f16 chunk by chunk) or a selected tile
    if (cur == 4) {
      if (!ring) {
        cp_async_wait_all();
        cbar_sync();  // every thread's window pieces have landed
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (!ring) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {  // 128 rows x 16 pieces of channels [128 c, 128 c + 128)
            const uint32_t t = static_cast<uint32_t>(tid + kComputeThreads * i);
            uint8_t* p = Kt + tile_off((t & 7u) | (((t >> 5) & 15u) << 3), 128u * c + 8u * (((t >> 3) & 3u) | ((t >> 9) << 2)));
            *reinterpret_cast<uint4*>(p) = cvt16(*reinterpret_cast<const uint4*>(p));
          }
        }
        chunk_done(c);
      }
    } else if (cur >= 0) {
      const int nx = after(cur);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        dequant_chunk(c);
        prefetch_chunk(nx, c);  // the registers of chunk c are free again: the next tile's
        store_chunk(c);
        chunk_done(c);
      }
    }

    float lsum[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) lsum[i] = 0.0f;
    uint32_t sph = 0;
    const uint32_t key = static_cast<uint32_t>(32 * qd + lane);  // softmax: TMEM lane = key
    const uint32_t lane_base = static_cast<uint32_t>(32 * qd) << 16;
    const int h0 = 16 * hg;

    while (cur >= 0) {
      // ---------------------------------------------------------------- S^T of tile cur
      const bool w_ok = mbar_wait(s_bar, sph, abort, a.wait_ns);
      sph ^= 1u;
      if (cbar_or(!(ok && w_ok))) {
        ok = false;
        break;
      }
      tc_fence_after();
      // ---------------------------------------------------------------- softmax
      const bool kv_ok = cur == 4 ? static_cast<int32_t>(key) < wl : recid[cur * 128 + key] >= 0;
      float x[16];
      {  // the two partial sums
        uint32_t r[2][16];
        tmem_ld16(tmem + lane_base + kSCol + static_cast<uint32_t>(h0), r[0]);
        tmem_ld16(tmem + lane_base + kSCol + 64u + static_cast<uint32_t>(h0), r[1]);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i)
          x[i] = kv_ok ? (__uint_as_float(r[0][i]) + __uint_as_float(r[1][i])) * a.scale_log2 : -INFINITY;
      }
      // the reference maxima live in shared memory (ref_s, and ref + 2^8 in ml), read as
      // broadcasts
      bool need = false, rescale = false;
#pragma unroll
      for (int i = 0; i < 16; ++i) need |= x[i] > ml[h0 + i];
      if (cbar_or(need)) {
        // raise the reference maxima of the heads whose scores exceed them by 2^8
        float* tmax = reinterpret_cast<float*>(Ps);  // [4][64] scratch: P is rewritten below
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float m = redux_max(x[i]);
          if (lane == i) tmax[qd * kHeads + h0 + i] = m;
        }
        cbar_sync();
        bool ch = false;
        if (tid < kHeads) {  // one thread per head decides (every reader of ref_s has passed the vote)
          const float mt = fmaxf(fmaxf(tmax[tid], tmax[kHeads + tid]), fmaxf(tmax[2 * kHeads + tid], tmax[3 * kHeads + tid]));
          const float old = ref_s[tid];
          const float nw = (mt > old + kRescaleThreshold || (old == -INFINITY && mt != -INFINITY)) ? mt : old;
          const float al = nw == old ? 1.0f : (old == -INFINITY ? 0.0f : exp2f(old - nw));
          alpha[tid] = al;
          ref_s[tid] = nw;
          ml[tid] = nw + kRescaleThreshold;
          ch = al != 1.0f;
        }
        rescale = cbar_or(ch) && o_started;  // alpha and ref_s are visible
#pragma unroll
        for (int i = 0; i < 16; ++i) lsum[i] *= alpha[h0 + i];
      }
      // P = exp2(x - ref) -> f16, P^T tile (MN-major: 8 heads x 2 bytes per core row); the
      // running sums add the rounded values, so that numerator and denominator agree
      {
        uint32_t pk[8];
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
          // a masked key (x = -inf) gives 2^-inf = 0, also against a head whose reference
          // is still -inf (the NaN of -inf - -inf is replaced by -inf)
          const float p0 = ex2_ftz(fmaxf(x[i] - ref_s[h0 + i], -INFINITY));
          const float p1 = ex2_ftz(fmaxf(x[i + 1] - ref_s[h0 + i + 1], -INFINITY));
          const __half2 ph = __floats2half2_rn(p0, p1);
          const float2 pr = __half22float2(ph);
          lsum[i] += pr.x;
          lsum[i + 1] += pr.y;
          pk[i / 2] = *reinterpret_cast<const uint32_t*>(&ph);
        }
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          const uint32_t off = (key >> 3) * 1024u + static_cast<uint32_t>(2 * hg + g) * 128u + (key & 7u) * 16u;
          *reinterpret_cast<uint4*>(Ps + off) = make_uint4(pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
        }
      }
      if (rescale) {
        // O^T chunk hg, TMEM lanes of this quarter: every head column times its factor
        // (after P, so that the scores' registers are free)
#pragma unroll 1
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t r[16];
          const uint32_t addr = tmem + lane_base + static_cast<uint32_t>(64 * hg + 16 * q4);
          tmem_ld16(addr, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha[16 * q4 + i]);
          tmem_st16(addr, r);
        }
        tmem_st_wait();
      }
      fence_proxy_async_smem();
      tc_fence_before();  // the rescaled O^T columns (TMEM stores) before the O MMAs
      cbar_sync();
      tc_fence_after();
      issue_o();
      o_started = true;
      // ---------------------------------------------------------------- the next tile
      const int nt = after(cur);
      if (nt < 0) break;
      const int nx = after(nt);
      // chunk c of the buffer is free once O chunk c has read it; the issuer runs the S MMAs
      // of the chunks already in place while the later ones are built, and the records of
      // the tile after next are loaded as each chunk's registers free up (unrolled: the
      // prefetched registers are indexed by c)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        dequant_chunk(c);
        prefetch_chunk(nx, c);
        const bool c_ok = mbar_wait(&o_bar[c], oph, abort, a.wait_ns);
        if (c_ok) store_chunk(c);
        ok = ok && c_ok;
        chunk_done(c);
      }
      oph ^= 1u;
      cur = nt;
    }
    // the last tile's O chunks complete before the epilogue reads O^T
    if (ok && o_started) {
      bool w_ok = true;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) w_ok &= mbar_wait(&o_bar[c], oph, abort, a.wait_ns);
      ok = ok && w_ok;
    }
    if (!ok || *abort) {
      ok = false;
      *abort = 1;
      if (tid == 0) report(a.err, CSA2_ERR_TIMEOUT, kInfoWait);
      if (issuer) {  // every MMA this issuer started completes before TMEM is freed
        mma_commit(drain);
        mbar_drain_wait(drain, 0);
      }
    }
    // ---- per-head sums over the 128 key lanes
    float* lred = reinterpret_cast<float*>(Ps);  // [4][64]
    cbar_sync();  // every warp is past its last P use
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float v = lsum[i];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == i) lred[qd * kHeads + h0 + i] = v;
    }
  }
  tc_fence_before();
  __syncthreads();  // per-head sums are in place
  tc_fence_after();
  const bool have_o = !*abort && o_started;
  if (tid < kHeads) {
    const float l = lred_sum(reinterpret_cast<const float*>(Ps), tid);
    ml[tid] = ref_s[tid];
    ml[kHeads + tid] = have_o ? l : 0.0f;
  }

  // ---------------------------------------------------------------- epilogue
  const uint32_t d = static_cast<uint32_t>(128 * hg + 32 * qd + lane);  // output channel (O^T lane)
  const uint32_t lane_base = static_cast<uint32_t>(32 * qd) << 16;
  // One CTA per query, or the second of a pair: it writes the output itself, the second
  // of a pair adding the first one's partial (written to the workspace before the pair's
  // cluster barrier) instead of both writing partials and splitting the heads.
  if (S == 1 || (S == 2 && sp == 1)) {
    const float* part0 = a.opart + static_cast<int64_t>(qi) * 2 * kHeads * CSA2_D;  // rank 0's [64][512]
    if (S == 2) attn_cluster_sync();  // rank 0's partial and (max, sum) are written and visible
    __syncthreads();
    if (tid < kHeads) {
      // O = (2^(m1 - M) O1^T + 2^(m0 - M) O0) / L with L = sum over the parts (and the sink)
      // of l 2^(m - M), relative to the largest maximum M of the non-empty parts
      const float l1 = ml[kHeads + tid], m1 = ml[tid];
      const float l0 = S == 2 ? __ldcg(a.mpart + qi * 2 * 2 * kHeads + kHeads + tid) : 0.0f;
      const float m0 = S == 2 ? __ldcg(a.mpart + qi * 2 * 2 * kHeads + tid) : -INFINITY;
      const float sk = (kExt && a.sinks != nullptr) ? __ldg(a.sinks + tid) * 1.4426950408889634f : -INFINITY;
      float M = sk;
      if (l1 > 0.0f) M = fmaxf(M, m1);
      if (l0 > 0.0f) M = fmaxf(M, m0);
      float lse2 = -INFINITY, w1 = 0.0f, w0 = 0.0f;  // log2 sum-exp and the parts' weights
      if (M != -INFINITY) {
        const float e1 = l1 > 0.0f ? exp2f(m1 - M) : 0.0f, e0 = l0 > 0.0f ? exp2f(m0 - M) : 0.0f;
        const float L = l1 * e1 + l0 * e0 + (sk != -INFINITY ? exp2f(sk - M) : 0.0f);
        lse2 = M + log2f(L);
        w1 = e1 / L;
        w0 = e0 / L;
      }
      if (a.lse) a.lse[qi * kHeads + tid] = lse2 * 0.6931471805599453f;
      alpha[tid] = w1;
      ref_s[tid] = w0;  // the reference maxima are in ml now
    }
    __syncthreads();
    // O^T (TMEM lane = channel, column = head) -> bf16 straight to the output: for each
    // head a warp writes 32 consecutive channels (64 bytes)
    __nv_bfloat16* og = a.out + qi * kHeads * CSA2_D;
    float* otail = reinterpret_cast<float*>(Ps);  // [64 heads][64] fp32 rotated channels (RoPE)
    {
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint32_t r[32];
        if (have_o) {
          tmem_ld32(tmem + lane_base + static_cast<uint32_t>(64 * hg + 32 * half), r);
          tmem_ld_wait();
        }
        float p0[32];  // rank 0's partial for these heads (S == 2), all loads issued first
#pragma unroll
        for (int i = 0; i < 32; ++i) p0[i] = S == 2 ? __ldcg(part0 + (32 * half + i) * CSA2_D + d) : 0.0f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int h = 32 * half + i;
          const float o = (have_o ? __uint_as_float(r[i]) * alpha[h] : 0.0f) + (S == 2 ? p0[i] * ref_s[h] : 0.0f);
          if (rope && d >= 448u)
            otail[h * 64 + (d - 448u)] = o;
          else
            og[h * CSA2_D + d] = __float2bfloat16_rn(o);
        }
      }
    }
    if (rope) {
      // o = o cos - rotate_half(o) sin: the rotation the values carried, undone at the
      // query's position
      __syncthreads();
      for (int p = tid; p < kHeads * 32; p += kAttnThreads) {
        const int h = p >> 5, i = p & 31;
        const float c = __ldg(a.rope_cos + qi * 32 + i), sn = __ldg(a.rope_sin + qi * 32 + i);
        const float x = otail[h * 64 + i], y = otail[h * 64 + 32 + i];
        og[h * CSA2_D + 448 + i] = __float2bfloat16_rn(x * c + y * sn);
        og[h * CSA2_D + 480 + i] = __float2bfloat16_rn(y * c - x * sn);
      }
    }
  } else {
    // ---- merge of the cluster's partials through L2: every CTA writes its raw O^T
    // (relative to its own reference maxima) and its (max, sum) per head to the workspace;
    // after one cluster barrier rank r combines heads [64 r / S, 64 (r + 1) / S) (S > 2; with
    // S == 2 rank 0 only writes, see above).  Every CTA reaches the barrier, also after a
    // failed wait (its partial then counts as empty).
    float* opart = a.opart + static_cast<int64_t>(blockIdx.x) * kHeads * CSA2_D;  // [64][512]
    float* mpart = a.mpart + static_cast<int64_t>(blockIdx.x) * 2 * kHeads;       // [2][64]
    {
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint32_t r[32];
        if (have_o) {
          tmem_ld32(tmem + lane_base + static_cast<uint32_t>(64 * hg + 32 * half), r);
          tmem_ld_wait();
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) opart[(32 * half + i) * CSA2_D + d] = have_o ? __uint_as_float(r[i]) : 0.0f;
      }
    }
    if (tid < kHeads) {
      mpart[tid] = ml[tid];
      mpart[kHeads + tid] = ml[kHeads + tid];
    }
    attn_cluster_sync();  // every partial of the cluster is written and visible
    if (S > 2) {  // rank 0 of a pair is done: rank 1 adds its partial
      const int hlo = kHeads * sp / S, hhi = kHeads * (sp + 1) / S;
      const float* opart0 = a.opart + static_cast<int64_t>(qi) * S * kHeads * CSA2_D;
      const float* mpart0 = a.mpart + static_cast<int64_t>(qi) * S * 2 * kHeads;
      float* fs = reinterpret_cast<float*>(Ps);  // [S][64] weight of each rank's partial
      float* otail = fs + kAttnMaxSplits * kHeads;  // [owned heads][64] fp32 rotated channels (RoPE)
      if (tid >= hlo && tid < hhi) {
        float mr[kAttnMaxSplits], lr[kAttnMaxSplits];
        float M = -INFINITY;
#pragma unroll
        for (int r = 0; r < kAttnMaxSplits; ++r) {
          mr[r] = r < S ? __ldcg(mpart0 + r * 2 * kHeads + tid) : -INFINITY;
          lr[r] = r < S ? __ldcg(mpart0 + r * 2 * kHeads + kHeads + tid) : 0.0f;
          if (lr[r] > 0.0f) M = fmaxf(M, mr[r]);
        }
        float sk = -INFINITY;
        if (kExt && a.sinks != nullptr) sk = __ldg(a.sinks + tid) * 1.4426950408889634f;
        const float M2 = fmaxf(M, sk);
        float L = sk != -INFINITY ? exp2f(sk - M2) : 0.0f;
#pragma unroll
        for (int r = 0; r < kAttnMaxSplits; ++r)
          if (lr[r] > 0.0f) L += lr[r] * exp2f(mr[r] - M2);
#pragma unroll
        for (int r = 0; r < kAttnMaxSplits; ++r)
          if (r < S) fs[r * kHeads + tid] = (lr[r] > 0.0f && L > 0.0f) ? exp2f(mr[r] - M2) / L : 0.0f;
        if (a.lse) a.lse[qi * kHeads + tid] = L > 0.0f ? (M2 + log2f(L)) * 0.6931471805599453f : -INFINITY;
      }
      __syncthreads();
      // items of 4 channels of one owned head: the S partials with 16-byte loads, weighted,
      // -> bf16 (with RoPE the last 64 channels go through otail and are rotated below).  A
      // thread's items are at most 8 (32 heads x 128 groups / 512 threads); all of their loads
      // are issued before the first is used.
      const int items = (hhi - hlo) * (CSA2_D / 4);
      float4 accs[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) accs[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int r = 0; r < S; ++r) {
        float4 v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int it = tid + kComputeThreads * k;
          const int h = hlo + it / (CSA2_D / 4), g = it % (CSA2_D / 4);
          v[k] = it < items ? __ldcg(reinterpret_cast<const float4*>(opart0 + (static_cast<int64_t>(r) * kHeads + h) * CSA2_D) + g)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int it = tid + kComputeThreads * k;
          const int h = hlo + (it < items ? it / (CSA2_D / 4) : 0);
          const float f = fs[r * kHeads + h];
          accs[k].x += f * v[k].x;
          accs[k].y += f * v[k].y;
          accs[k].z += f * v[k].z;
          accs[k].w += f * v[k].w;
        }
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int it = tid + kComputeThreads * k;
        if (it >= items) break;
        const int h = hlo + it / (CSA2_D / 4), g = it % (CSA2_D / 4);
        const float4 acc = accs[k];
        if (rope && g >= 112) {
          float* t = otail + (h - hlo) * 64 + (4 * g - 448);
          t[0] = acc.x;
          t[1] = acc.y;
          t[2] = acc.z;
          t[3] = acc.w;
        } else {
          const __nv_bfloat162 b0 = __floats2bfloat162_rn(acc.x, acc.y), b1 = __floats2bfloat162_rn(acc.z, acc.w);
          *reinterpret_cast<uint2*>(a.out + (qi * kHeads + h) * CSA2_D + 4 * g) =
              make_uint2(*reinterpret_cast<const uint32_t*>(&b0), *reinterpret_cast<const uint32_t*>(&b1));
        }
      }
      if (rope) {
        __syncthreads();
        for (int p = tid; p < (hhi - hlo) * 32; p += kAttnThreads) {
          const int hh = p >> 5, i = p & 31;
          const float c = __ldg(a.rope_cos + qi * 32 + i), sn = __ldg(a.rope_sin + qi * 32 + i);
          const float x = otail[hh * 64 + i], y = otail[hh * 64 + 32 + i];
          __nv_bfloat16* dst = a.out + (qi * kHeads + hlo + hh) * CSA2_D;
          dst[448 + i] = __float2bfloat16_rn(x * c + y * sn);
          dst[480 + i] = __float2bfloat16_rn(y * c - x * sn);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

size_t attn_smem_bytes() { return kAttnSmem; }

// Splits per query for this launch: the most (up to the 5 tiles) that keep every CTA of a
// batch in one wave, reduced while the device cannot hold a cluster of that size with this
// kernel's shared memory (queried once per device and size).
int attn_splits_for(int64_t n_q, int sm_count, bool ext) {
  static std::atomic<int> fits[2][kMaxDevices][kAttnMaxSplits + 1];
  int dev = 0;
  cudaGetDevice(&dev);
  int S = attn_wave_splits(n_q, sm_count);
  for (; S > 1; --S) {
    int v = (dev >= 0 && dev < kMaxDevices) ? fits[ext][dev][S].load(std::memory_order_relaxed) : 0;
    if (v == 0) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(S), 1, 1);
      cfg.blockDim = dim3(kAttnThreads, 1, 1);
      cfg.dynamicSmemBytes = kAttnSmem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = static_cast<unsigned>(S);
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n_act = 0;
      auto* kernel = ext ? attn_kernel<true> : attn_kernel<false>;
      static std::atomic<int> limit_set[2][kMaxDevices];
      cudaError_t e = smem_limit_once(reinterpret_cast<const void*>(kernel), kAttnSmem, limit_set[ext]);
      if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&n_act, kernel, &cfg);
      if (e != cudaSuccess) {
        cudaGetLastError();
        n_act = 0;
      }
      v = n_act > 0 ? 1 : -1;
      if (dev >= 0 && dev < kMaxDevices) fits[ext][dev][S].store(v, std::memory_order_relaxed);
    }
    if (v > 0) break;
  }
  return S;
}

cudaError_t launch_attn(const AttnArgs& a, cudaStream_t stream) {
  if (a.n_q == 0) return cudaSuccess;
  static std::atomic<int> limit_set[2][kMaxDevices];
  const bool ext = a.sinks != nullptr || a.rope_cos != nullptr || a.win_ring != nullptr;
  auto* kernel = ext ? attn_kernel<true> : attn_kernel<false>;
  cudaError_t e = smem_limit_once(reinterpret_cast<const void*>(kernel), kAttnSmem, limit_set[ext ? 1 : 0]);
  if (e != cudaSuccess) return e;
  const int S = a.splits;
  cudaLaunchAttribute cl;
  cl.id = cudaLaunchAttributeClusterDimension;
  cl.val.clusterDim.x = static_cast<unsigned>(S);
  cl.val.clusterDim.y = 1;
  cl.val.clusterDim.z = 1;
  return launch_pdl(kernel, dim3(static_cast<unsigned>(a.n_q * S)), dim3(kAttnThreads), kAttnSmem, stream,
                    S > 1 ? &cl : nullptr, a);
}

}  // namespace csa2
