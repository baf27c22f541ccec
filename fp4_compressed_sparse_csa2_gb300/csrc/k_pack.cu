// k_pack.cu -- FP4 packing of new cache entries and of the indexer query.
//
// "DeepSeek's Attention and KV Cache - From MLA to CSA2", "DeepSeek-V4.1 ... Four bits
// for the main KV": E2M1 elements with one E4M3 scale per 16 channels, the scale
// mapping the block maximum onto 6, no tensor-level scale; 288 B per 512-channel
// entry.  "DeepSeek-V4.1-Flash and the 890-byte KV cache", section 3: the 128-channel
// indexer key in the same format, 72 B.  "DeepSeek-V4: ... The indexer in four bits":
// the indexer query-key product runs entirely in FP4, so the query is packed with the
// same codec.  Alternatively ("A Precision Primer", MX formats and E8M0; "What's in a
// cell" of "From First Principles: DeepSeek-V4.1-Flash Inference") the indexer key and
// query take MXFP4, one power-of-two E8M0 scale per 32 channels, 68 B per key.
//
// One thread per 16-channel block: two 16-byte loads, one fp32 division for the
// scale, 16 for the codes (hardware RN/satfinite conversions), an 8-byte nibble
// store and a 1-byte scale store.  An MXFP4 block of 32 channels takes one thread:
// its exponent, 32 exact power-of-two quotients, two 8-byte stores and a scale byte.
#include "csa2_kernels.cuh"

namespace csa2 {

__device__ __forceinline__ void load16(const __nv_bfloat16* src, float (&x)[16]) {
  const uint4* p = reinterpret_cast<const uint4*>(src);
  const uint4 a = __ldg(p), b = __ldg(p + 1);
  const uint32_t u[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = __uint_as_float(u[i] << 16);
    x[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
}

// Items [0, n_new*40) pack cache entries (32 main-KV blocks + 8 indexer blocks per
// entry); items [n_new*40, +n_groups*128*8) pack indexer-query rows (rows >= N of a
// group only clear their scale bytes).
__global__ void __launch_bounds__(256) pack_kernel(PackArgs a) {
  pdl_wait();  // the previous step's kernels may still read the cache slots written here
  // the next kernel (the indexer) starts only now: every kernel before this one has
  // completed, so it may read the cache pages this kernel does not write before its wait
  pdl_trigger();
  const int64_t item = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t n_pack = a.n_new * 40;
  if (item < n_pack) {
    const int64_t i = item / 40;
    const int b = static_cast<int>(item % 40);
    const int32_t r = a.new_req[i];
    const int64_t s = a.new_pos[i];
    if (r < 0 || s < 0 || s >= static_cast<int64_t>(a.cache.max_pages) * kPage) {
      report(a.err, CSA2_ERR_DEVICE, kInfoPos);
      return;
    }
    const int64_t p = page_id(a.cache, r, s);
    if (p < 0 || p >= a.cache.n_pages) {
      report(a.err, CSA2_ERR_DEVICE, kInfoPage);
      return;
    }
    const uint32_t e = static_cast<uint32_t>(s % kPage);
    float x[16];
    uint32_t lo, hi;
    if (b < 32) {
      load16(a.latent + i * kD + 16 * b, x);
      const uint32_t sc = quant_block16(x, lo, hi);
      uint8_t* rec = a.cache.kv + p * kKvPageBytes + static_cast<int64_t>(e) * kKvBytes;
      *reinterpret_cast<uint2*>(rec + 8 * b) = make_uint2(lo, hi);
      rec[256 + b] = static_cast<uint8_t>(sc);
    } else if (a.cache.idx_format == CSA2_IDX_MXFP4) {
      const int bb = b - 32;  // items 32..35: one 32-channel MXFP4 block each
      if (bb >= 4) return;
      float x32[32];
      load16(a.idx_key + i * kDI + 32 * bb, *reinterpret_cast<float(*)[16]>(&x32[0]));
      load16(a.idx_key + i * kDI + 32 * bb + 16, *reinterpret_cast<float(*)[16]>(&x32[16]));
      uint32_t nib[4];
      const uint32_t sc = quant_block32_mx(x32, nib);
      uint8_t* pg = a.cache.idx + p * kIdxMxPageBytes;
      *reinterpret_cast<uint2*>(pg + idx_nib_off(e, 2 * bb)) = make_uint2(nib[0], nib[1]);
      *reinterpret_cast<uint2*>(pg + idx_nib_off(e, 2 * bb + 1)) = make_uint2(nib[2], nib[3]);
      pg[idx_mx_sf_off(kIdxNibBytes, e, bb)] = static_cast<uint8_t>(sc);
    } else {
      const int bb = b - 32;
      load16(a.idx_key + i * kDI + 16 * bb, x);
      const uint32_t sc = quant_block16(x, lo, hi);
      uint8_t* pg = a.cache.idx + p * kIdxPageBytes;
      *reinterpret_cast<uint2*>(pg + idx_nib_off(e, bb)) = make_uint2(lo, hi);
      pg[idx_sf_off(kIdxNibBytes, e, bb)] = static_cast<uint8_t>(sc);
    }
    return;
  }
  const int64_t qi = item - n_pack;
  if (qi >= a.n_groups * 128 * 8) return;
  const int64_t g = qi / (128 * 8);
  const uint32_t n = static_cast<uint32_t>((qi / 8) % 128);
  const uint32_t bb = static_cast<uint32_t>(qi % 8);
  uint8_t* gp = a.qpack + g * a.grp_bytes;
  const uint32_t nib_bytes = static_cast<uint32_t>(a.N) * 64u;
  if (a.cache.idx_format == CSA2_IDX_MXFP4) {  // items bb < 4: one 32-channel block each
    if (bb >= 4) return;
    if (n >= static_cast<uint32_t>(a.N)) {
      gp[idx_mx_sf_off(nib_bytes, n, bb)] = 0;
      return;
    }
    const int64_t q = g * a.G + n / a.heads_I;
    const int32_t j = static_cast<int32_t>(n % a.heads_I);
    uint32_t nib[4] = {0u, 0u, 0u, 0u}, sc = 0;
    if (q < a.n_q) {
      float x32[32];
      const __nv_bfloat16* src = a.q_idx + (q * a.heads_I + j) * kDI + 32 * bb;
      load16(src, *reinterpret_cast<float(*)[16]>(&x32[0]));
      load16(src + 16, *reinterpret_cast<float(*)[16]>(&x32[16]));
      sc = quant_block32_mx(x32, nib);
    }
    *reinterpret_cast<uint2*>(gp + idx_nib_off(n, 2 * bb)) = make_uint2(nib[0], nib[1]);
    *reinterpret_cast<uint2*>(gp + idx_nib_off(n, 2 * bb + 1)) = make_uint2(nib[2], nib[3]);
    gp[idx_mx_sf_off(nib_bytes, n, bb)] = static_cast<uint8_t>(sc);
    return;
  }
  if (n >= static_cast<uint32_t>(a.N)) {  // unused scale slots of a short group
    gp[idx_sf_off(nib_bytes, n, bb)] = 0;
    return;
  }
  const int64_t q = g * a.G + n / a.heads_I;
  const int32_t j = static_cast<int32_t>(n % a.heads_I);
  uint32_t lo = 0, hi = 0, sc = 0;
  if (q < a.n_q) {
    float x[16];
    load16(a.q_idx + (q * a.heads_I + j) * kDI + 16 * bb, x);
    sc = quant_block16(x, lo, hi);
  }
  *reinterpret_cast<uint2*>(gp + idx_nib_off(n, bb)) = make_uint2(lo, hi);
  gp[idx_sf_off(nib_bytes, n, bb)] = static_cast<uint8_t>(sc);
}

// FP8 window ring ("Four bits for the main KV, eight for the window": 512 E4M3 bytes
// plus 16 E8M0 scales per entry; "Definition and the bounded cache": position i in slot
// i mod 128).  One thread per 32-channel block: four 16-byte loads, the block's
// power-of-two scale, 32 E4M3 conversions of exact quotients, two 16-byte stores and a
// scale byte.
__global__ void __launch_bounds__(256) pack_window_kernel(WinPackArgs a) {
  pdl_trigger();
  pdl_wait();  // earlier kernels may still read the slots written here
  const int64_t item = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (item >= a.n * 16) return;
  const int64_t i = item >> 4;
  const int b = static_cast<int>(item & 15);
  const int32_t r = a.req[i];
  const int64_t p = a.pos[i];
  if (r < 0 || r >= a.n_ring || p < 0) {
    report(a.err, CSA2_ERR_DEVICE, kInfoPos);
    return;
  }
  float x[32];
  load16(a.rows + i * kD + 32 * b, *reinterpret_cast<float(*)[16]>(&x[0]));
  load16(a.rows + i * kD + 32 * b + 16, *reinterpret_cast<float(*)[16]>(&x[16]));
  float amax = 0.0f;
#pragma unroll
  for (int c = 0; c < 32; ++c) amax = fmaxf(amax, fabsf(x[c]));
  const int e = e8m0_exponent(amax);
  uint32_t w[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    uint32_t v = 0;
#pragma unroll
    for (int m = 0; m < 4; ++m) v |= cvt_e4m3(ldexpf(x[4 * k + m], -e)) << (8 * m);  // exact quotient
    w[k] = v;
  }
  uint8_t* rec = a.ring + (static_cast<int64_t>(r) * CSA2_WIN + p % CSA2_WIN) * CSA2_WIN_BYTES;
  uint4* dst = reinterpret_cast<uint4*>(rec + 32 * b);
  dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
  dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
  rec[512 + b] = static_cast<uint8_t>(e + 127);
}

cudaError_t launch_pack_window(const WinPackArgs& a, cudaStream_t stream) {
  if (a.n == 0) return cudaSuccess;
  const int64_t blocks = (a.n * 16 + 255) / 256;
  return launch_pdl(pack_window_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, nullptr, a);
}

cudaError_t launch_pack(const PackArgs& a, cudaStream_t stream) {
  const int64_t items = a.n_new * 40 + a.n_groups * 128 * 8;
  if (items == 0) return cudaSuccess;
  const int64_t blocks = (items + 255) / 256;
  return launch_pdl(pack_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, nullptr, a);
}

}  // namespace csa2
