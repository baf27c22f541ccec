// k_attn.cu -- shared-KV MQA over the selected FP4 entries plus the sliding window.
//
// "DeepSeek's Attention and KV Cache - From MLA to CSA2", "DeepSeek-V4": a query
// attends to the top-512 selected entries concatenated with the 128 window entries;
// each entry is one 512-wide vector serving as both key and value.  "DeepSeek-V4.1":
// the FP4 entries are dequantised before attention.  "From MLA to DSA to HCA/CSA",
// "What replaced MLA": attention(q, kv, kv) with K and V the same tensor.
//
// Design: two CTAs of 8 warps per query, each owning 32 of the 64 heads (heads are
// independent, so the halves exchange nothing); 5 key tiles of 128 keys, the window
// tile first:
//   prefetch the 288-byte records of the next selected tile go to a raw staging buffer
//            with cp.async while the current tile is processed; the window rows (bf16)
//            are copied straight into the key tile at the start;
//   build    all warps dequantise the staged records (byte-permute lookups, exact bf16
//            products) into the bf16 key tile in the tensor-core operand layout;
//   S^T      two threads issue 32 tcgen05.mma kind::f16 (M = 128 keys, N = 32 heads,
//            K = 512) into four partial TMEM sums;
//   softmax  thread = key, 16 heads per thread: warp max reductions, a per-head
//            reference max that only moves when a tile exceeds it by 2^8 (then the
//            TMEM accumulator and the running sums are rescaled), exp2, bf16 P^T to
//            shared memory;
//   O^T      32 tcgen05.mma (4 M-tiles of 128 output channels, N = 32 heads, K = 128
//            keys) reading the SAME bf16 tile as an MN-major operand (K == V);
//   epilogue O = O^T / l per head -> bf16, lse = ln(sum exp).
// Optional, from "From MLA to DSA to HCA/CSA": per-head attention sinks (a logit that
// joins the softmax denominator and has no value; section "The sliding window") and
// the partial RoPE of "What replaced MLA" (the queries' trailing 64 channels rotated
// in shared memory before the first S^T MMA; the output's rotated back with the
// negated angle before it is rounded to bf16).
#include "csa2_kernels.cuh"

namespace csa2 {

constexpr int kAttnThreads = 256;
constexpr int kHeads = 64;                          // query heads
constexpr int kHH = 32;                             // heads per CTA
constexpr uint32_t kKtBytes = 128 * 512 * 2;        // bf16 key tile
constexpr uint32_t kQsBytes = kHH * 512 * 2;        // bf16 queries of this CTA's heads
constexpr uint32_t kPsBytes = 128 * kHH * 2;        // bf16 P^T
constexpr uint32_t kRawBytes = 128 * kKvBytes;      // staged FP4 records of one tile
constexpr uint32_t kOCols = 0, kSCols = 256;        // TMEM columns: O^T 4 x 32, S^T 4 partial sums x 32
constexpr float kRescaleThreshold = 8.0f;      // log2 units

// Offset of element (row, col) in a [rows][512] bf16 operand tile stored as 8x8 core
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
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }


// E4M3 code -> bf16 (exact: 4 significant bits, range 2^-9 .. 448), both halves.
__device__ __forceinline__ __nv_bfloat162 e4m3_bf16x2(uint32_t code) {
  const uint32_t e = (code >> 3) & 15u, m = code & 7u;
  uint32_t bits = e ? (((e + 120u) << 7) | (m << 4)) : (__float_as_uint(static_cast<float>(m) * 0.001953125f) >> 16);
  bits |= (code & 0x80u) << 8;
  const uint32_t both = bits | (bits << 16);
  return *reinterpret_cast<const __nv_bfloat162*>(&both);
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_newest_pending() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// kExt: the optional features (sinks, partial RoPE, FP8 window ring) are compiled in;
// the plain instance carries none of their code.  kSplit (plain path only): a.splits CTAs
// per (query, head half) each take a run of the key tiles and write a partial.
template <bool kExt, bool kSplit>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_kernel(const AttnArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* Kt = smem;
  uint8_t* Qs = Kt + kKtBytes;
  uint8_t* Ps = Qs + kQsBytes;
  uint8_t* Raw = Ps + kPsBytes;
  float* ref = reinterpret_cast<float*>(Raw + kRawBytes);  // [32] reference max (log2 units)
  float* alpha = ref + kHH;                                 // [32]
  float* tmax = alpha + kHH;                                // [4][32]
  float* lred = tmax + 4 * kHH;                             // [4][32]
  int64_t* recoff = reinterpret_cast<int64_t*>(lred + 4 * kHH);        // [512] record byte offsets, -1 = none
  int32_t* tile_cnt = reinterpret_cast<int32_t*>(recoff + CSA2_TOPK);  // [4] valid entries per selected tile
  uint64_t* mma_bar = reinterpret_cast<uint64_t*>(tile_cnt + 4);  // [2] one per MMA issuer
  uint64_t* drain = mma_bar + 2;                                    // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 2);
  int32_t* flags = reinterpret_cast<int32_t*>(tmem_slot + 1);  // [0] abort, [1] rescale

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = kSplit ? a.splits : 1;  // CTAs per (query, head half), each over a run of tiles
  const int64_t qi = blockIdx.x / (2 * S);
  const int sp = static_cast<int>((blockIdx.x >> 1) % S);
  const int h0 = (blockIdx.x & 1) * kHH;  // first head of this CTA
  // this CTA's run [t_lo, t_hi) of the tile list [window, selected 0, 1, 2, 3]
  const int t_lo = sp * 5 / S, t_hi = (sp + 1) * 5 / S;
  const bool has_win = t_lo == 0;
  const int sel_lo = t_lo == 0 ? 0 : t_lo - 1, sel_hi = t_hi - 1;  // selected tiles [sel_lo, sel_hi)
  const int32_t nv = __ldg(a.n_visible + qi);
  const int32_t wl = max(0, min(CSA2_WIN, __ldg(a.win_len + qi)));

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&mma_bar[i], 1);
      mbar_init(&drain[i], 1);
    }
    flags[0] = 0;
    flags[1] = 0;
    fence_mbar_init();
  }
  if (tid < kHH) ref[tid] = -INFINITY;
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  pdl_trigger();
  // queries of this CTA's heads, then the window rows, -> shared memory (operand
  // layout, K-major over the 512 channels); two cp.async groups
  {
    const __nv_bfloat16* qg = a.q + (qi * kHeads + h0) * CSA2_D;
    for (int c = tid; c < kHH * 64; c += kAttnThreads) {
      uint32_t h, ch;
      tile_item(static_cast<uint32_t>(c), kHH, h, ch);
      cp_async16(smem_u32(Qs + tile_off(h, ch * 8)), qg + h * CSA2_D + ch * 8, 16);
    }
    cp_async_commit();
    const __nv_bfloat16* wg = a.window + __ldg(a.win_start + qi) * CSA2_D;
    const bool bf16_rows = (!kExt || a.win_ring == nullptr) && has_win;
    for (int c = tid; bf16_rows && c < 128 * 64; c += kAttnThreads) {  // bf16 window rows
      uint32_t r, ch;
      tile_item(static_cast<uint32_t>(c), 128, r, ch);
      const bool ok = static_cast<int32_t>(r) < wl;
      cp_async16(smem_u32(Kt + tile_off(r, ch * 8)), ok ? static_cast<const void*>(wg + r * CSA2_D + ch * 8)
                                                         : static_cast<const void*>(a.window),
                 ok ? 16u : 0u);
    }
    cp_async_commit();
  }
  // The copies above read only this call's inputs, so they overlap the previous kernel's
  // tail; the selected indices (and in Full mode the new entries) come from earlier kernels.
  pdl_wait();
  // offsets of the 512 selected records (one round trip for all indices)
  if (tid < 4) tile_cnt[tid] = 0;
  __syncthreads();
  {
    const int32_t r = __ldg(a.req + qi);
    for (int i = tid; i < CSA2_TOPK; i += kAttnThreads) {
      const int32_t e = __ldg(a.topk_idx + qi * CSA2_TOPK + i);
      int64_t off = -1;
      if (e >= 0) {
        const int64_t pg = e < nv ? page_id(a.cache, r, e) : -1;
        if (pg >= 0 && pg < a.cache.n_pages)
          off = pg * kKvPageBytes + static_cast<int64_t>(e % kPage) * kKvBytes;
        else
          report(a.err, CSA2_ERR_DEVICE, kInfoTopkIdx);
      }
      recoff[i] = off;
      if (off >= 0) atomicAdd(&tile_cnt[i >> 7], 1);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t idesc_s = idesc_bf16(128, kHH, 0, 0);
  const uint32_t idesc_o = idesc_bf16(128, kHH, 1, 1);

  // Stages the records of selected tile t (16-byte pieces; a missing record reads as zeros).
  auto prefetch = [&](int t) {
    for (int c = tid; c < 128 * (kKvBytes / 16); c += kAttnThreads) {
      const int slot = c / (kKvBytes / 16), j = c - slot * (kKvBytes / 16);
      const int64_t off = recoff[t * 128 + slot];
      cp_async16(smem_u32(Raw + slot * kKvBytes + j * 16), a.cache.kv + (off >= 0 ? off + j * 16 : 0),
                 off >= 0 ? 16u : 0u);
    }
    cp_async_commit();
  };
  auto next_selected = [&](int t) {  // first selected tile of this run after t with any entry, or 4
    int u = t + 1;
    while (u < sel_hi && tile_cnt[u] == 0) ++u;
    return u < sel_hi ? u : 4;
  };
  int staged = next_selected(sel_lo - 1);
  if (staged < 4) prefetch(staged);

  float lsum[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) lsum[i] = 0.0f;
  uint32_t phase = 0;
  bool o_started = false;
  const int hb = (warp >> 2) * 16;                  // this thread's 16 heads (of the CTA's 32)
  const uint32_t key_row = (warp & 3) * 32 + lane;  // TMEM lane = key (softmax) / channel (epilogue)
  const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;

  for (int it = 0; it < 5; ++it) {
    // ---------------------------------------------------------------- the key tile
    const bool win_turn = it == 0 && has_win;
    const int t = win_turn ? 4 : staged;  // the window first, then the selected tiles in order
    if (t == 4 && !win_turn) break;       // no selected tile left
    if (t == 4) {
      if (staged < 4) cp_async_wait_newest_pending();  // queries and window landed; records may still fly
      else cp_async_wait_all();
      if (kExt && a.rope_cos != nullptr) {
        // q = q cos + rotate_half(q) sin on channels 448 + i / 480 + i (angle i), in place
        __syncthreads();  // every thread's query pieces have landed
        for (int p = tid; p < kHH * 32; p += kAttnThreads) {
          const uint32_t h = static_cast<uint32_t>(p) >> 5, i = static_cast<uint32_t>(p) & 31u;
          const float c = __ldg(a.rope_cos + qi * 32 + i), sn = __ldg(a.rope_sin + qi * 32 + i);
          __nv_bfloat16* pa = reinterpret_cast<__nv_bfloat16*>(Qs + tile_off(h, 448u + i));
          __nv_bfloat16* pb = reinterpret_cast<__nv_bfloat16*>(Qs + tile_off(h, 480u + i));
          const float x = __bfloat162float(*pa), y = __bfloat162float(*pb);
          *pa = __float2bfloat16_rn(x * c - y * sn);
          *pb = __float2bfloat16_rn(y * c + x * sn);
        }
      }
      if (kExt && a.win_ring != nullptr) {
        // FP8 window ring: row i of the tile is the entry of position newest - i, read
        // after the wait on the previous kernel (the ring is written by an earlier call);
        // E4M3 -> f16 in hardware, times the block's 2^e, -> bf16 (exact)
        const int64_t newest = __ldg(a.win_start + qi);
        const int32_t r = __ldg(a.req + qi);
        const bool ring_ok = r >= 0 && r < a.win_ring_reqs && newest - wl + 1 >= 0;
        if (!ring_ok && wl > 0 && tid == 0) report(a.err, CSA2_ERR_DEVICE, kInfoPos);
#pragma unroll 2
        for (int i = 0; i < 8; ++i) {
          const uint32_t task = static_cast<uint32_t>(tid + kAttnThreads * i);
          const uint32_t row = (task & 7u) | (((task >> 5) & 15u) << 3);
          const uint32_t j = ((task >> 3) & 3u) | ((task >> 9) << 2);
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
              const __nv_bfloat162 bv = __floats2bfloat162_rn(f.x * sc, f.y * sc);
              o[k] = *reinterpret_cast<const uint32_t*>(&bv);
            }
            *reinterpret_cast<uint4*>(dst + m * 128) = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
      }
    } else {
      cp_async_wait_all();
      __syncthreads();  // every thread's pieces of the staged records are visible
      // item = (entry slot, 32-channel block j); a warp takes 8 slots x 4 blocks so that
      // its 16-byte tile stores fill whole 128-byte lines
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t task = static_cast<uint32_t>(tid + kAttnThreads * i);
        const uint32_t slot = (task & 7u) | (((task >> 5) & 15u) << 3);
        const uint32_t j = ((task >> 3) & 3u) | ((task >> 9) << 2);
        const uint8_t* rec = Raw + slot * kKvBytes;
        const uint4 nib = *reinterpret_cast<const uint4*>(rec + j * 16);
        const uint32_t scw = *reinterpret_cast<const uint16_t*>(rec + 256 + j * 2);
        const __nv_bfloat162 s0 = e4m3_bf16x2(scw & 0xFFu), s1 = e4m3_bf16x2(scw >> 8);
        const uint32_t wds[4] = {nib.x, nib.y, nib.z, nib.w};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          uint32_t o[4];
          dequant8_bf16(wds[m], m < 2 ? s0 : s1, o);
          *reinterpret_cast<uint4*>(Kt + tile_off(slot, 32 * j + 8 * m)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (t != 4) {  // the staging buffer is free again: fetch the next selected tile
      staged = next_selected(t);
      if (staged < 4) prefetch(staged);
    }

    // ---------------------------------------------------------------- S^T = K Q^T
    // two issuing threads (warps 0 and 1): issuer i takes K-steps kk = i, i+2, ... into
    // partial sums i and i + 2, so neither thread waits on the other's MMA latency
    if (lane == 0 && warp < 2) {
      const uint32_t me = static_cast<uint32_t>(warp);
      const uint32_t kb = smem_u32(Kt), qb = smem_u32(Qs);
#pragma unroll 4
      for (uint32_t kk = me; kk < 32; kk += 2)
        mma_bf16(tmem + kSCols + (kk & 3u) * kHH, sdesc(kb + kk * 256u, 128, 8192), sdesc(qb + kk * 256u, 128, 8192),
                 idesc_s, kk >= 4 ? 1u : 0u);
      mma_commit(&mma_bar[me]);
      if (!mbar_wait(&mma_bar[me], phase, nullptr)) {
        flags[0] = 1;
        report(a.err, CSA2_ERR_TIMEOUT, kInfoWait);
      }
    }
    phase ^= 1;
    __syncthreads();
    tc_fence_after();
    if (flags[0]) break;

    // ---------------------------------------------------------------- softmax
    const bool kv_ok = t == 4 ? static_cast<int32_t>(key_row) < wl : recoff[t * 128 + key_row] >= 0;
    float x[16];
    {
      uint32_t r[16];
      tmem_ld16(tmem + lane_base + kSCols + static_cast<uint32_t>(hb), r);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = __uint_as_float(r[i]);
#pragma unroll
      for (uint32_t pp = 1; pp < 4; ++pp) {
        tmem_ld16(tmem + lane_base + kSCols + pp * kHH + static_cast<uint32_t>(hb), r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] += __uint_as_float(r[i]);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = kv_ok ? x[i] * a.scale_log2 : -INFINITY;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float m = redux_max(x[i]);
      if (lane == i) tmax[(warp & 3) * kHH + hb + i] = m;
    }
    if (tid == 0) flags[1] = 0;
    __syncthreads();
    if (tid < kHH) {
      const float mt = fmaxf(fmaxf(tmax[tid], tmax[kHH + tid]), fmaxf(tmax[2 * kHH + tid], tmax[3 * kHH + tid]));
      const float old = ref[tid];
      float nw = old;
      if (mt > old + kRescaleThreshold || (old == -INFINITY && mt != -INFINITY)) nw = mt;
      alpha[tid] = (old == -INFINITY) ? 0.0f : exp2f(old - nw);
      ref[tid] = nw;
      if (nw != old && old != -INFINITY) flags[1] = 1;
    }
    __syncthreads();
    if (flags[1] && o_started) {
      // rescale O^T columns (heads) and the running sums by alpha
#pragma unroll
      for (int i = 0; i < 16; ++i) lsum[i] *= alpha[hb + i];
      for (int c = (warp >> 2) * 2; c < (warp >> 2) * 2 + 2; ++c) {
        uint32_t r[32];
        const uint32_t addr = tmem + lane_base + kOCols + static_cast<uint32_t>(c * kHH);
        tmem_ld32(addr, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha[i]);
        tmem_st32(addr, r);
      }
      tmem_st_wait();
    }
    // P = exp2(x - ref) -> bf16, P^T tile (MN-major: 8 heads x 2 bytes per core row)
    {
      uint32_t pk[8];
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        const float r0 = ref[hb + i], r1 = ref[hb + i + 1];
        const float p0 = (r0 == -INFINITY) ? 0.0f : exp2f(x[i] - r0);
        const float p1 = (r1 == -INFINITY) ? 0.0f : exp2f(x[i + 1] - r1);
        const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
        lsum[i] += __low2float(pb);
        lsum[i + 1] += __high2float(pb);
        pk[i / 2] = *reinterpret_cast<const uint32_t*>(&pb);
      }
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const uint32_t off = (key_row >> 3) * (kHH * 16u) + static_cast<uint32_t>((hb >> 3) + c) * 128u +
                             (key_row & 7u) * 16u;
        *reinterpret_cast<uint4*>(Ps + off) = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---------------------------------------------------------------- O^T += V^T P^T
    // issuer i accumulates output tiles 2i and 2i+1 (channels [256 i, 256 i + 256))
    if (lane == 0 && warp < 2) {
      const uint32_t me = static_cast<uint32_t>(warp);
      const uint32_t kb = smem_u32(Kt), pb = smem_u32(Ps);
      for (uint32_t kk = 0; kk < 8; ++kk) {
#pragma unroll
        for (uint32_t c = 2 * me; c < 2 * me + 2; ++c)
          mma_bf16(tmem + kOCols + c * kHH, sdesc(kb + c * 2048u + kk * 16384u, 8192, 128),
                   sdesc(pb + kk * (2u * kHH * 16u), kHH * 16u, 128), idesc_o, (o_started || kk > 0) ? 1u : 0u);
      }
      mma_commit(&mma_bar[me]);
      if (!mbar_wait(&mma_bar[me], phase, nullptr)) {
        flags[0] = 1;
        report(a.err, CSA2_ERR_TIMEOUT, kInfoWait);
      }
    }
    phase ^= 1;
    o_started = true;
    __syncthreads();
    tc_fence_after();
    if (flags[0]) break;
  }
  cp_async_wait_all();  // no copy may land after the CTA is gone

  // ---------------------------------------------------------------- epilogue
  if (!flags[0]) {
    // row sums: reduce the 128 key slots of each head
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float v = lsum[i];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == i) lred[(warp & 3) * kHH + hb + i] = v;
    }
    __syncthreads();
    if (tid < kHH) {
      const float l = lred[tid] + lred[kHH + tid] + lred[2 * kHH + tid] + lred[3 * kHH + tid];
      float lse2 = -INFINITY, inv = 0.0f;  // log2 sum-exp; O = O^T * inv
      if (kSplit) {  // a partial over this CTA's tiles, merged by attn_combine_kernel
        if (l > 0.0f) {
          lse2 = ref[tid] + log2f(l);
          inv = 1.0f / l;
        }
        a.lpart[(qi * S + sp) * kHeads + h0 + tid] = lse2;
      } else if (!kExt || a.sinks == nullptr) {
        if (l > 0.0f) {
          lse2 = ref[tid] + log2f(l);
          inv = 1.0f / l;
        }
      } else {
        // the sink joins the denominator: O = O^T / (l + 2^(sink - ref)), taken relative
        // to the larger of the two maxima so that nothing overflows
        const float sk = __ldg(a.sinks + h0 + tid) * 1.4426950408889634f;
        if (l > 0.0f || sk != -INFINITY) {
          const float m2 = l > 0.0f ? fmaxf(ref[tid], sk) : sk;
          const float lt = (l > 0.0f ? l * exp2f(ref[tid] - m2) : 0.0f) + exp2f(sk - m2);
          lse2 = m2 + log2f(lt);
          inv = l > 0.0f ? exp2f(ref[tid] - m2) / lt : 0.0f;
        }
      }
      if (a.lse && !kSplit) a.lse[qi * kHeads + h0 + tid] = lse2 * 0.6931471805599453f;
      alpha[tid] = inv;  // reuse: the output scale per head
    }
    __syncthreads();
    // O^T (TMEM lane = channel, column = head) -> bf16 [32][512] staged in the free key
    // tile, then written out with 16-byte coalesced stores
    __nv_bfloat16* ostage = reinterpret_cast<__nv_bfloat16*>(Kt);
    float* otail = reinterpret_cast<float*>(Ps);  // [32 heads][64] fp32 rotated channels (RoPE)
    const bool rope = kExt && a.rope_cos != nullptr;
    if (kSplit) {
      // the normalised partial in fp32 [32][512], staged in the free key tile, then 16-byte
      // coalesced stores
      float* fstage = reinterpret_cast<float*>(Kt);
      for (int c = (warp >> 2) * 2; c < (warp >> 2) * 2 + 2; ++c) {
        const uint32_t d = static_cast<uint32_t>(c) * 128u + key_row;
        uint32_t r[32];
        if (o_started) {
          tmem_ld32(tmem + lane_base + kOCols + static_cast<uint32_t>(c * kHH), r);
          tmem_ld_wait();
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) fstage[i * CSA2_D + d] = o_started ? __uint_as_float(r[i]) * alpha[i] : 0.0f;
      }
      __syncthreads();
      uint4* pg = reinterpret_cast<uint4*>(a.opart + ((qi * S + sp) * kHeads + h0) * CSA2_D);
      const uint4* fs = reinterpret_cast<const uint4*>(fstage);
      for (int i = tid; i < kHH * CSA2_D / 4; i += kAttnThreads) pg[i] = fs[i];
    }
    for (int c = (warp >> 2) * 2; c < (warp >> 2) * 2 + 2 && !kSplit; ++c) {
      const uint32_t d = static_cast<uint32_t>(c) * 128u + key_row;
      uint32_t r[32];
      if (o_started) {
        tmem_ld32(tmem + lane_base + kOCols + static_cast<uint32_t>(c * kHH), r);
        tmem_ld_wait();
      }
      if (rope && d >= 448u) {  // rotated back below, in fp32
#pragma unroll
        for (int i = 0; i < 32; ++i) otail[i * 64 + (d - 448u)] = o_started ? __uint_as_float(r[i]) * alpha[i] : 0.0f;
        continue;
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float o = o_started ? __uint_as_float(r[i]) * alpha[i] : 0.0f;
        ostage[i * CSA2_D + d] = __float2bfloat16_rn(o);
      }
    }
    if (rope) {
      // o = o cos - rotate_half(o) sin: the rotation the values carried, undone at the
      // query's position
      __syncthreads();
      for (int p = tid; p < kHH * 32; p += kAttnThreads) {
        const int h = p >> 5, i = p & 31;
        const float c = __ldg(a.rope_cos + qi * 32 + i), sn = __ldg(a.rope_sin + qi * 32 + i);
        const float x = otail[h * 64 + i], y = otail[h * 64 + 32 + i];
        ostage[h * CSA2_D + 448 + i] = __float2bfloat16_rn(x * c + y * sn);
        ostage[h * CSA2_D + 480 + i] = __float2bfloat16_rn(y * c - x * sn);
      }
    }
    __syncthreads();
    uint4* og = reinterpret_cast<uint4*>(a.out + (qi * kHeads + h0) * CSA2_D);
    const uint4* os = reinterpret_cast<const uint4*>(ostage);
    for (int i = tid; i < kHH * CSA2_D / 8 && !kSplit; i += kAttnThreads) og[i] = os[i];
  }
  // drain outstanding MMAs, then free TMEM
  if (lane == 0 && warp < 2) {
    mma_commit(&drain[warp]);
    mbar_wait(&drain[warp], 0, nullptr);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

size_t attn_smem_bytes() {
  return 1024 + kKtBytes + kQsBytes + kPsBytes + kRawBytes + (2 + 8) * kHH * sizeof(float) + CSA2_TOPK * 8 + 16 +
         4 * sizeof(uint64_t) + 16;
}

// Merge of the key-tile splits: one warp per (query, head).  The total log2 sum-exp is
// L = log2(sum_s 2^L_s) and O = sum_s 2^(L_s - L) O_s (each O_s already normalised by
// its own sum); lanes take 16 channels each.
__global__ void __launch_bounds__(256) attn_combine_kernel(const AttnArgs a) {
  pdl_trigger();
  pdl_wait();  // the partials come from the attention kernel
  const int lane = threadIdx.x & 31;
  const int64_t item = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (item >= a.n_q * kHeads) return;
  const int64_t qi = item / kHeads;
  const int h = static_cast<int>(item % kHeads);
  const int S = a.splits;
  float ls[kAttnMaxSplits];
  float m = -INFINITY;
#pragma unroll
  for (int s = 0; s < kAttnMaxSplits; ++s) {
    ls[s] = s < S ? __ldg(a.lpart + (qi * S + s) * kHeads + h) : -INFINITY;
    m = fmaxf(m, ls[s]);
  }
  float tot = 0.0f;
#pragma unroll
  for (int s = 0; s < kAttnMaxSplits; ++s) tot += ls[s] == -INFINITY ? 0.0f : exp2f(ls[s] - m);
  const float lse2 = m == -INFINITY ? -INFINITY : m + log2f(tot);
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
#pragma unroll
  for (int s = 0; s < kAttnMaxSplits; ++s) {
    if (ls[s] == -INFINITY) continue;
    const float wgt = exp2f(ls[s] - lse2);
    const float4* src = reinterpret_cast<const float4*>(a.opart + ((qi * S + s) * kHeads + h) * CSA2_D + 16 * lane);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float4 v = __ldg(src + k);
      acc[4 * k + 0] += wgt * v.x;
      acc[4 * k + 1] += wgt * v.y;
      acc[4 * k + 2] += wgt * v.z;
      acc[4 * k + 3] += wgt * v.w;
    }
  }
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    o[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
  uint4* dst = reinterpret_cast<uint4*>(a.out + (qi * kHeads + h) * CSA2_D + 16 * lane);
  dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
  dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  if (lane == 0 && a.lse) a.lse[qi * kHeads + h] = lse2 * 0.6931471805599453f;
}

cudaError_t launch_attn(const AttnArgs& a, cudaStream_t stream) {
  if (a.n_q == 0) return cudaSuccess;
  const size_t smem = attn_smem_bytes();
  static std::atomic<int> limit_set[3][kMaxDevices];
  const bool ext = a.sinks != nullptr || a.rope_cos != nullptr || a.win_ring != nullptr;
  const int S = ext ? 1 : a.splits;
  auto* kernel = ext ? attn_kernel<true, false> : (S > 1 ? attn_kernel<false, true> : attn_kernel<false, false>);
  cudaError_t e = smem_limit_once(reinterpret_cast<const void*>(kernel), smem, limit_set[ext ? 2 : (S > 1 ? 1 : 0)]);
  if (e != cudaSuccess) return e;
  return launch_pdl(kernel, dim3(static_cast<unsigned>(2 * a.n_q * S)), dim3(kAttnThreads), smem, stream, nullptr,
                    a);
}

cudaError_t launch_attn_combine(const AttnArgs& a, cudaStream_t stream) {
  if (a.n_q == 0) return cudaSuccess;
  const int64_t blocks = (a.n_q * kHeads + 7) / 8;
  return launch_pdl(attn_combine_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, nullptr, a);
}

}  // namespace csa2
