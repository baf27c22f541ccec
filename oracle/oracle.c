/*
 * CSA2 CPU oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct CPU restatement of what one CSA2 attention
 * layer of DeepSeek-V4.1-Flash computes at decode and chunked prefill.  It is
 * used only by the test suite, by the smoke check and by the CPU-baseline leg of
 * the benchmark; the product library never links or calls it.  It shares no
 * code, header, table or constant generator with the CUDA path.
 *
 * Sources (page title, section):
 *   [P1] "DeepSeek's Attention and KV Cache - From MLA to CSA2, From First
 *        Principles": "A Precision Primer" (E4M3, E2M1, block scaling),
 *        "DeepSeek-V3.2: Sparse Attention With a Learned Indexer" (index score,
 *        top-k), "DeepSeek-V4" (window concatenated with the selected entries,
 *        shared-KV MQA), "DeepSeek-V4.1 ... Four bits for the main KV" (E2M1
 *        with one E4M3 scale per 16 channels, no global scale, 288 B entry,
 *        numpy quantizer check).
 *   [P2] "From MLA to DSA to HCA/CSA: DeepSeek V3.2 and V4 Attention":
 *        "The indexer" (ReLU score, head sum, fp32 scoring path),
 *        "CSA: two changes to HCA" (-1 sentinel when fewer than k are
 *        visible), "What replaced MLA" (K and V are the same tensor).
 *   [P3] "DeepSeek-V4.1-Flash and the 890-byte KV cache", section 3
 *        (indexer key in the main-KV format: 72 B per entry).
 *   [P4] "From First Principles: DeepSeek-V4.1-Flash Inference", "What's in a
 *        cell" (the MXFP4 indexer key: 64 B of nibbles + four E8M0 scales, 68 B;
 *        see the MXFP4 section at the end of this file).
 *
 * Precision: codecs decide integer codes in fp32 (the kernel's precision);
 * every dot product, score, softmax and output accumulation is fp64.
 *
 * Cache layout (the pages give entry sizes only; the layout is this build's
 * reading and is restated here from its definition, independently of the GPU
 * code):
 *   page = 128 entries.  Page id of (request r, page j) is bt[r*max_pages+j],
 *   or r*max_pages+j when bt == NULL.
 *   main-KV page: 128 * 288 B.  Entry e at e*288: bytes [0,256) hold channel
 *     pairs (2i, 2i+1) as low/high nibble of byte i; bytes [256,288) hold the
 *     32 block scales in block order.
 *   indexer-K page: 9216 B = 128 * 72 B.  Nibbles of entry e, channel c at
 *     (e/8)*512 + (c/32)*128 + (e%8)*16 + (c%32)/2 (low nibble = even c);
 *     scale of entry e, block b at 8192 + (b/4)*512 + (e%32)*16 + (e/32)*4 + b%4.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_D 512
#define OR_DI 128
#define OR_PAGE 128
#define OR_KV_BYTES 288
#define OR_IDX_BYTES 72
#define OR_KV_PAGE_BYTES (OR_PAGE * OR_KV_BYTES)
#define OR_IDX_PAGE_BYTES (OR_PAGE * OR_IDX_BYTES)

/* ---------------------------------------------------------------- bf16 */

static float bf16_to_float(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* ------------------------------------------------------------ E4M3 [P1]
 * E4M3 (FN variant): 1 sign, 4 exponent bits with bias 7, 3 mantissa bits.
 * Exponent field 0 is subnormal (m * 2^-9); the all-ones pattern 0x7F/0xFF is
 * the single NaN; there is no infinity; the largest finite value is 448.
 */
double or_e4m3_decode(uint8_t c) {
  int s = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

/* Round-to-nearest-even onto the E4M3 grid, saturating to +-448 (satfinite).
 * x is an fp32 value; all arithmetic below is exact in double. */
uint8_t or_e4m3_encode(float xf) {
  double x = (double)xf;
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs(x);
  if (isnan(x)) return 0x7F;
  if (a >= 448.0) return sign | 0x7E; /* satfinite */
  if (a < ldexp(1.0, -6)) {
    /* subnormal range: a = q * 2^-9, q in [0, 8) */
    double q = ldexp(a, 9);
    double fl = floor(q), fr = q - fl;
    int qi = (int)fl;
    if (fr > 0.5 || (fr == 0.5 && (qi & 1))) qi += 1;
    /* qi == 8 becomes the smallest normal: field (e=1, m=0) = 0x08 */
    return sign | (uint8_t)qi;
  }
  int e2;
  double fr = frexp(a, &e2); /* a = fr * 2^e2, fr in [0.5, 1) */
  int e = e2 - 1;            /* a = (2*fr) * 2^e, 2*fr in [1, 2) */
  double mant = (2.0 * fr - 1.0) * 8.0; /* in [0, 8) */
  double fl = floor(mant), rem = mant - fl;
  int mi = (int)fl;
  if (rem > 0.5 || (rem == 0.5 && (mi & 1))) mi += 1;
  if (mi == 8) { mi = 0; e += 1; }
  int field = e + 7;
  /* a < 448 so the rounded value is at most 448 = (field 15, m 6) */
  return sign | (uint8_t)((field << 3) | mi);
}

/* ------------------------------------------------------------ E2M1 [P1]
 * E2M1: 1 sign, 2 exponent bits, 1 mantissa bit.  Magnitudes of codes 0..7 are
 * 0, 0.5, 1, 1.5, 2, 3, 4, 6; bit 3 is the sign; no infinity, no NaN.
 */
static const double e2m1_mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double or_e2m1_decode(uint8_t c) {
  double v = e2m1_mag[c & 7];
  return (c & 8) ? -v : v;
}

/* Nearest magnitude, ties to the even code (mantissa bit 0), |y| > 6 -> 6.
 * The sign bit is kept even when the magnitude rounds to 0. */
uint8_t or_e2m1_encode(float yf) {
  double y = (double)yf;
  uint8_t sign = signbit(y) ? 8 : 0;
  double a = fabs(y);
  if (a >= 6.0) return sign | 7;
  int best = 0;
  for (int c = 1; c < 8; ++c) {
    double dc = fabs(a - e2m1_mag[c]), db = fabs(a - e2m1_mag[best]);
    if (dc < db || (dc == db && (c & 1) == 0 && (best & 1) == 1)) best = c;
  }
  return sign | (uint8_t)best;
}

/* ---------------------------------------------------- block of 16 [P1]
 * One E4M3 scale per 16 channels mapping the block maximum onto 6; the
 * second-level tensor scale of NVFP4 is omitted.  amax/6 and x/s are
 * correctly rounded fp32 divisions; a zero scale encodes the block as +0. */
void or_quant_block16(const float* x, uint8_t* codes, uint8_t* scale_code) {
  float amax = 0.0f;
  for (int i = 0; i < 16; ++i) {
    float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  volatile float ratio = amax / 6.0f; /* fp32 division */
  uint8_t sc = or_e4m3_encode(ratio);
  *scale_code = sc;
  float s = (float)or_e4m3_decode(sc);
  for (int i = 0; i < 16; ++i) {
    if (s == 0.0f) {
      codes[i] = 0;
    } else {
      volatile float y = x[i] / s; /* fp32 division */
      codes[i] = or_e2m1_encode(y);
    }
  }
}

/* ---------------------------------------------------------- cache layout */

static int64_t page_of(const int32_t* bt, int32_t max_pages, int32_t r, int64_t s) {
  int64_t j = s / OR_PAGE;
  return bt ? (int64_t)bt[(int64_t)r * max_pages + j] : (int64_t)r * max_pages + j;
}

static int64_t idx_nib_off(int64_t e, int64_t c) {
  return (e / 8) * 512 + (c / 32) * 128 + (e % 8) * 16 + (c % 32) / 2;
}

static int64_t idx_sf_off(int64_t e, int64_t b) {
  return 8192 + (b / 4) * 512 + (e % 32) * 16 + (e / 32) * 4 + (b % 4);
}

/* Write one 512-channel main-KV entry and one 128-channel indexer-K entry. */
static void write_entry(const float* lat, const float* key, uint8_t* kv_pages, uint8_t* idx_pages,
                        int64_t page, int64_t e) {
  uint8_t* rec = kv_pages + page * OR_KV_PAGE_BYTES + e * OR_KV_BYTES;
  for (int b = 0; b < 32; ++b) {
    uint8_t codes[16], sc;
    or_quant_block16(lat + 16 * b, codes, &sc);
    for (int i = 0; i < 8; ++i) rec[b * 8 + i] = (uint8_t)(codes[2 * i] | (codes[2 * i + 1] << 4));
    rec[256 + b] = sc;
  }
  uint8_t* pg = idx_pages + page * OR_IDX_PAGE_BYTES;
  for (int b = 0; b < 8; ++b) {
    uint8_t codes[16], sc;
    or_quant_block16(key + 16 * b, codes, &sc);
    for (int i = 0; i < 16; i += 2) {
      int64_t c = 16 * b + i;
      pg[idx_nib_off(e, c)] = (uint8_t)(codes[i] | (codes[i + 1] << 4));
    }
    pg[idx_sf_off(e, b)] = sc;
  }
}

/* Pack n new entries (bf16 latents [n][512], bf16 indexer keys [n][128]) at
 * positions pos[i] of requests req[i]. */
void or_pack_kv(const uint16_t* latent, const uint16_t* idx_key, const int32_t* req,
                const int64_t* pos, int64_t n, uint8_t* kv_pages, uint8_t* idx_pages,
                const int32_t* bt, int32_t max_pages) {
  float lat[OR_D], key[OR_DI];
  for (int64_t i = 0; i < n; ++i) {
    for (int c = 0; c < OR_D; ++c) lat[c] = bf16_to_float(latent[i * OR_D + c]);
    for (int c = 0; c < OR_DI; ++c) key[c] = bf16_to_float(idx_key[i * OR_DI + c]);
    int64_t page = page_of(bt, max_pages, req[i], pos[i]);
    write_entry(lat, key, kv_pages, idx_pages, page, pos[i] % OR_PAGE);
  }
}

/* Pack fp32 vectors (used by the quantizer check on an fp32 latent). */
void or_quant_vector(const float* x, int64_t nblocks, uint8_t* codes, uint8_t* scales) {
  for (int64_t b = 0; b < nblocks; ++b) or_quant_block16(x + 16 * b, codes + 16 * b, scales + b);
}

/* Dequantised values of one cached entry: v = e2m1(code) * e4m3(scale). */
void or_read_main(const uint8_t* kv_pages, const int32_t* bt, int32_t max_pages, int32_t r,
                  int64_t s, double* out) {
  const uint8_t* rec = kv_pages + page_of(bt, max_pages, r, s) * OR_KV_PAGE_BYTES +
                       (s % OR_PAGE) * OR_KV_BYTES;
  for (int c = 0; c < OR_D; ++c) {
    uint8_t byte = rec[c / 2];
    uint8_t code = (c % 2) ? (byte >> 4) : (byte & 15);
    out[c] = or_e2m1_decode(code) * or_e4m3_decode(rec[256 + c / 16]);
  }
}

void or_read_idx(const uint8_t* idx_pages, const int32_t* bt, int32_t max_pages, int32_t r,
                 int64_t s, double* out) {
  const uint8_t* pg = idx_pages + page_of(bt, max_pages, r, s) * OR_IDX_PAGE_BYTES;
  int64_t e = s % OR_PAGE;
  for (int c = 0; c < OR_DI; ++c) {
    uint8_t byte = pg[idx_nib_off(e, c)];
    uint8_t code = (c % 2) ? (byte >> 4) : (byte & 15);
    out[c] = or_e2m1_decode(code) * or_e4m3_decode(pg[idx_sf_off(e, c / 16)]);
  }
}

/* ----------------------------------------------------- index score [P1][P2]
 * I[t,s] = sum_j w[t,j] * ReLU( qhat[t,j] . khat[s] * 128^-0.5 ), for
 * s in [s0, s1).  qhat is the indexer query quantised with the same block
 * codec (the query-key product is taken entirely in FP4).  M[t,s] is the same
 * sum with |w| (the scale for the score tolerance).  All in fp64. */
void or_index_score(const uint16_t* q_idx, const float* w, int32_t heads, const uint8_t* idx_pages,
                    const int32_t* bt, int32_t max_pages, int32_t r, int64_t s0, int64_t s1,
                    double* I, double* M) {
  double* qh = (double*)malloc(sizeof(double) * heads * OR_DI);
  for (int j = 0; j < heads; ++j) {
    for (int b = 0; b < 8; ++b) {
      float x[16];
      uint8_t codes[16], sc;
      for (int i = 0; i < 16; ++i) x[i] = bf16_to_float(q_idx[(int64_t)j * OR_DI + 16 * b + i]);
      or_quant_block16(x, codes, &sc);
      for (int i = 0; i < 16; ++i)
        qh[j * OR_DI + 16 * b + i] = or_e2m1_decode(codes[i]) * or_e4m3_decode(sc);
    }
  }
  const double scale = 1.0 / sqrt(128.0);
  double k[OR_DI];
  for (int64_t s = s0; s < s1; ++s) {
    or_read_idx(idx_pages, bt, max_pages, r, s, k);
    double acc = 0.0, accm = 0.0;
    for (int j = 0; j < heads; ++j) {
      double dot = 0.0;
      for (int c = 0; c < OR_DI; ++c) dot += qh[j * OR_DI + c] * k[c];
      double relu = dot * scale > 0.0 ? dot * scale : 0.0;
      acc += (double)w[j] * relu;
      accm += fabs((double)w[j]) * relu;
    }
    I[s - s0] = acc;
    M[s - s0] = accm;
  }
  free(qh);
}

/* --------------------------------------------------------------- top-k [P2]
 * The k largest scores among the n visible entries; equal scores are ordered
 * by the lower index first; -0 and +0 are equal.  The chosen indices are
 * returned in ascending order, padded with -1 when n < k. */
typedef struct { float v; int64_t i; } or_pair;

static int cmp_pair(const void* a, const void* b) {
  const or_pair* x = (const or_pair*)a;
  const or_pair* y = (const or_pair*)b;
  if (x->v > y->v) return -1;
  if (x->v < y->v) return 1;
  return (x->i < y->i) ? -1 : (x->i > y->i);
}

static int cmp_i32(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

void or_topk(const float* scores, int64_t n, int32_t k, int32_t* out) {
  or_pair* p = (or_pair*)malloc(sizeof(or_pair) * (n > 0 ? n : 1));
  for (int64_t i = 0; i < n; ++i) {
    float v = scores[i];
    p[i].v = (v == 0.0f) ? 0.0f : v; /* -0 -> +0 */
    p[i].i = i;
  }
  qsort(p, (size_t)n, sizeof(or_pair), cmp_pair);
  int64_t take = n < k ? n : k;
  for (int64_t i = 0; i < take; ++i) out[i] = (int32_t)p[i].i;
  qsort(out, (size_t)take, sizeof(int32_t), cmp_i32);
  for (int64_t i = take; i < k; ++i) out[i] = -1;
  free(p);
}

/* ------------------------------------------------ sparse + window MQA [P1][P2]
 * Keys = the dequantised entries named by idx (entries < 0 are skipped) followed
 * by the win_len bf16 window rows; no de-duplication.  Each key is both key and
 * value.  For each head h: S = scale * q_h . key, P = softmax(S), O_h = P . keys,
 * lse_h = log(sum exp S).  Two passes, fp64.  With no keys, O = 0, lse = -inf. */
void or_attention(const uint16_t* q, int32_t heads, const int32_t* idx, int32_t k,
                  const uint8_t* kv_pages, const int32_t* bt, int32_t max_pages, int32_t r,
                  const uint16_t* win, int32_t win_len, double scale, double* O, double* lse) {
  int32_t nk = 0;
  for (int i = 0; i < k; ++i) nk += idx[i] >= 0;
  nk += win_len;
  double* keys = (double*)malloc(sizeof(double) * (nk > 0 ? nk : 1) * OR_D);
  int32_t t = 0;
  for (int i = 0; i < k; ++i)
    if (idx[i] >= 0) or_read_main(kv_pages, bt, max_pages, r, idx[i], keys + (int64_t)(t++) * OR_D);
  for (int i = 0; i < win_len; ++i, ++t)
    for (int c = 0; c < OR_D; ++c) keys[(int64_t)t * OR_D + c] = bf16_to_float(win[(int64_t)i * OR_D + c]);
  double* S = (double*)malloc(sizeof(double) * (nk > 0 ? nk : 1));
  double qd[OR_D];
  for (int h = 0; h < heads; ++h) {
    for (int c = 0; c < OR_D; ++c) qd[c] = bf16_to_float(q[(int64_t)h * OR_D + c]);
    double* o = O + (int64_t)h * OR_D;
    for (int c = 0; c < OR_D; ++c) o[c] = 0.0;
    if (nk == 0) { lse[h] = -INFINITY; continue; }
    double mx = -INFINITY;
    for (int j = 0; j < nk; ++j) {
      double dot = 0.0;
      for (int c = 0; c < OR_D; ++c) dot += qd[c] * keys[(int64_t)j * OR_D + c];
      S[j] = scale * dot;
      if (S[j] > mx) mx = S[j];
    }
    double sum = 0.0;
    for (int j = 0; j < nk; ++j) { S[j] = exp(S[j] - mx); sum += S[j]; }
    for (int j = 0; j < nk; ++j) {
      double p = S[j] / sum;
      for (int c = 0; c < OR_D; ++c) o[c] += p * keys[(int64_t)j * OR_D + c];
    }
    lse[h] = mx + log(sum);
  }
  free(S);
  free(keys);
}

/* ------------------------------------------------ sinks and partial RoPE [P2]
 * "From MLA to DSA to HCA/CSA", section "What replaced MLA" (partial RoPE and its
 * inverse on the output): the trailing 64 channels of the query are rotated at the
 * query's position, q = q cos + rotate_half(q) sin, and the output is rotated back
 * with the negated angle, o = o cos - rotate_half(o) sin, where rotate_half pairs
 * channel 448 + i with 480 + i: rotate_half(x)[448 + i] = -x[480 + i] and
 * rotate_half(x)[480 + i] = x[448 + i] (i < 32, both halves share angle i).  The
 * cached entries are rotated before they are packed, so keys are used as given.
 * Section "The sliding window" (attention sinks): one logit per head is appended to
 * each score row before the softmax and dropped after it; it has no value vector, so
 * the weights of the real keys sum to 1 - p_sink.
 * sinks: natural-log logits [heads] or NULL; cos/sin: [32] or NULL (no rotation).
 * With no keys: O = 0 and lse = the sink (or -inf without sinks). */
static void or_rotate_tail(double* x, const double* cos_, const double* sin_, double sign) {
  for (int i = 0; i < 32; ++i) {
    const double a = x[OR_D - 64 + i], b = x[OR_D - 32 + i];
    x[OR_D - 64 + i] = a * cos_[i] - sign * b * sin_[i];
    x[OR_D - 32 + i] = b * cos_[i] + sign * a * sin_[i];
  }
}

/* S, softmax (with the sink) and the output over nk fp64 keys; q rotated first and the
 * output rotated back when cos_ is given. */
static void or_attend(const uint16_t* q, int32_t heads, const double* keys, int32_t nk, double scale,
                      const double* sinks, const double* cos_, const double* sin_, double* O, double* lse) {
  double* S = (double*)malloc(sizeof(double) * (nk > 0 ? nk : 1));
  double qd[OR_D];
  for (int h = 0; h < heads; ++h) {
    for (int c = 0; c < OR_D; ++c) qd[c] = bf16_to_float(q[(int64_t)h * OR_D + c]);
    if (cos_) or_rotate_tail(qd, cos_, sin_, 1.0);
    double* o = O + (int64_t)h * OR_D;
    for (int c = 0; c < OR_D; ++c) o[c] = 0.0;
    double mx = sinks ? sinks[h] : -INFINITY;
    for (int j = 0; j < nk; ++j) {
      double dot = 0.0;
      for (int c = 0; c < OR_D; ++c) dot += qd[c] * keys[(int64_t)j * OR_D + c];
      S[j] = scale * dot;
      if (S[j] > mx) mx = S[j];
    }
    if (mx == -INFINITY) { lse[h] = -INFINITY; continue; }  /* no key and no sink */
    double sum = sinks ? exp(sinks[h] - mx) : 0.0;
    for (int j = 0; j < nk; ++j) { S[j] = exp(S[j] - mx); sum += S[j]; }
    for (int j = 0; j < nk; ++j) {
      double p = S[j] / sum;
      for (int c = 0; c < OR_D; ++c) o[c] += p * keys[(int64_t)j * OR_D + c];
    }
    if (cos_) or_rotate_tail(o, cos_, sin_, -1.0);
    lse[h] = mx + log(sum);
  }
  free(S);
}

void or_attention_ext(const uint16_t* q, int32_t heads, const int32_t* idx, int32_t k,
                      const uint8_t* kv_pages, const int32_t* bt, int32_t max_pages, int32_t r,
                      const uint16_t* win, int32_t win_len, double scale, const double* sinks,
                      const double* cos_, const double* sin_, double* O, double* lse) {
  int32_t nk = 0;
  for (int i = 0; i < k; ++i) nk += idx[i] >= 0;
  nk += win_len;
  double* keys = (double*)malloc(sizeof(double) * (nk > 0 ? nk : 1) * OR_D);
  int32_t t = 0;
  for (int i = 0; i < k; ++i)
    if (idx[i] >= 0) or_read_main(kv_pages, bt, max_pages, r, idx[i], keys + (int64_t)(t++) * OR_D);
  for (int i = 0; i < win_len; ++i, ++t)
    for (int c = 0; c < OR_D; ++c) keys[(int64_t)t * OR_D + c] = bf16_to_float(win[(int64_t)i * OR_D + c]);
  or_attend(q, heads, keys, nk, scale, sinks, cos_, sin_, O, lse);
  free(keys);
}

/* ------------------------------------------------ FP8 window ring [P1]
 * "DeepSeek's Attention and KV Cache - From MLA to CSA2", "Four bits for the main KV,
 * eight for the window": a window entry is 512 E4M3 bytes (RoPE channels included)
 * plus 16 E8M0 scales, 528 bytes, one scale per 32 channels.  "Definition and the
 * bounded cache": the entry of position i lives in slot i mod W of a W-slot ring
 * (W = 128).  Scale (the pages are silent): the smallest power of two 2^e with
 * amax <= 448 * 2^e, so that no element clips, e clamped to the E8M0 range [-127, 127];
 * an all-zero block takes e = -127.  Element: E4M3 round-to-nearest-even of x / 2^e
 * (an exact division).  Record: bytes [0, 512) the codes in channel order, then the
 * 16 E8M0 codes e + 127 in block order. */
#define OR_WIN 128
#define OR_WIN_BYTES 528

int32_t or_e8m0_exponent(double amax) {
  if (!(amax > 0.0)) return -127;
  int E;
  frexp(amax, &E); /* amax in [2^(E-1), 2^E); 448 * 2^(E-10) < 2^(E-1) <= amax < 448 * 2^(E-8) */
  int e = amax <= ldexp(448.0, E - 9) ? E - 9 : E - 8;
  if (e < -127) e = -127;
  if (e > 127) e = 127;
  return e;
}

void or_pack_window(const uint16_t* rows, const int32_t* req, const int64_t* pos, int64_t n, uint8_t* ring) {
  for (int64_t i = 0; i < n; ++i) {
    uint8_t* rec = ring + ((int64_t)req[i] * OR_WIN + pos[i] % OR_WIN) * OR_WIN_BYTES;
    for (int b = 0; b < OR_D / 32; ++b) {
      double amax = 0.0;
      for (int c = 0; c < 32; ++c) {
        double v = fabs((double)bf16_to_float(rows[i * OR_D + 32 * b + c]));
        if (v > amax) amax = v;
      }
      int e = or_e8m0_exponent(amax);
      for (int c = 0; c < 32; ++c) {
        double x = (double)bf16_to_float(rows[i * OR_D + 32 * b + c]);
        rec[32 * b + c] = or_e4m3_encode((float)ldexp(x, -e)); /* exact: |x / 2^e| <= 448 */
      }
      rec[OR_D + b] = (uint8_t)(e + 127);
    }
  }
}

void or_read_window(const uint8_t* ring, int32_t r, int64_t p, double* out) {
  const uint8_t* rec = ring + ((int64_t)r * OR_WIN + p % OR_WIN) * OR_WIN_BYTES;
  for (int c = 0; c < OR_D; ++c) out[c] = or_e4m3_decode(rec[c]) * ldexp(1.0, (int)rec[OR_D + c / 32] - 127);
}

/* Attention whose window keys are the ring entries of positions win_pos - win_len + 1
 * .. win_pos of request r (the selected entries as in or_attention_ext). */
void or_attention_ring(const uint16_t* q, int32_t heads, const int32_t* idx, int32_t k,
                       const uint8_t* kv_pages, const int32_t* bt, int32_t max_pages, int32_t r,
                       const uint8_t* ring, int64_t win_pos, int32_t win_len, double scale, const double* sinks,
                       const double* cos_, const double* sin_, double* O, double* lse) {
  int32_t nk = 0;
  for (int i = 0; i < k; ++i) nk += idx[i] >= 0;
  nk += win_len;
  double* keys = (double*)malloc(sizeof(double) * (nk > 0 ? nk : 1) * OR_D);
  int32_t t = 0;
  for (int i = 0; i < k; ++i)
    if (idx[i] >= 0) or_read_main(kv_pages, bt, max_pages, r, idx[i], keys + (int64_t)(t++) * OR_D);
  for (int i = 0; i < win_len; ++i, ++t) or_read_window(ring, r, win_pos - i, keys + (int64_t)t * OR_D);
  or_attend(q, heads, keys, nk, scale, sinks, cos_, sin_, O, lse);
  free(keys);
}

/* ------------------------------------------- MXFP4 indexer key [P1][P3][P4]
 * "DeepSeek's Attention and KV Cache", "A Precision Primer" (block scaling: MX
 * formats and E8M0): an MX block is k = 32 elements sharing one E8M0 scale, a pure
 * power of two 2^-127 .. 2^127, decoded as v_i = X * P_i; MXFP4 takes E2M1 elements
 * (4 + 8/32 = 4.25 bits each).  "DeepSeek-V4 ... the indexer in four bits" and "From
 * First Principles: DeepSeek-V4.1-Flash Inference", "What's in a cell": the indexer
 * key is MXFP4, 64 bytes of nibbles plus four E8M0 scales, 68 bytes.
 * Scale (the pages fix the format, not the rule): the primer's worked example has a
 * block maximum of 3 + delta take the scale 1, since E8M0 must round the ideal
 * (3 + delta)/6 up; so the scale is the smallest power of two 2^e with amax <= 6 * 2^e
 * (no element clips), e clamped to [-127, 127], e = -127 for an all-zero block.
 * Element: E2M1 round-to-nearest-even of the exact quotient x / 2^e.
 * Indexer-K page in this format: 8704 B = 128 * 68: the nibbles of entry e, channel c
 * where the 72-byte format has them, (e/8)*512 + (c/32)*128 + (e%8)*16 + (c%32)/2;
 * the E8M0 code e + 127 of entry e, block b (channels [32b, 32b+32)) at
 * 8192 + (e%32)*16 + (e/32)*4 + b. */
#define OR_IDX_MX_BYTES 68
#define OR_IDX_MX_PAGE_BYTES (OR_PAGE * OR_IDX_MX_BYTES)

int32_t or_mx_exponent(double amax) {
  if (!(amax > 0.0)) return -127;
  int E;
  frexp(amax, &E); /* amax in [2^(E-1), 2^E): 6 * 2^(E-4) < 2^(E-1) <= amax < 6 * 2^(E-2) */
  int e = amax <= ldexp(6.0, E - 3) ? E - 3 : E - 2;
  if (e < -127) e = -127;
  if (e > 127) e = 127;
  return e;
}

/* One 32-element block: E2M1 codes and the E8M0 code e + 127. */
void or_mx_quant_block32(const float* x, uint8_t* codes, uint8_t* scale_code) {
  double amax = 0.0;
  for (int i = 0; i < 32; ++i) {
    double a = fabs((double)x[i]);
    if (a > amax) amax = a;
  }
  int e = or_mx_exponent(amax);
  for (int i = 0; i < 32; ++i) codes[i] = or_e2m1_encode((float)ldexp((double)x[i], -e));
  *scale_code = (uint8_t)(e + 127);
}

static int64_t idx_mx_sf_off(int64_t e, int64_t b) { return 8192 + (e % 32) * 16 + (e / 32) * 4 + b; }

/* Pack n indexer keys (bf16 [n][128]) in the MXFP4 format at positions pos[i] of
 * requests req[i]. */
void or_pack_idx_mx(const uint16_t* idx_key, const int32_t* req, const int64_t* pos, int64_t n,
                    uint8_t* idx_pages, const int32_t* bt, int32_t max_pages) {
  for (int64_t i = 0; i < n; ++i) {
    uint8_t* pg = idx_pages + page_of(bt, max_pages, req[i], pos[i]) * OR_IDX_MX_PAGE_BYTES;
    int64_t e = pos[i] % OR_PAGE;
    for (int b = 0; b < 4; ++b) {
      float x[32];
      uint8_t codes[32], sc;
      for (int c = 0; c < 32; ++c) x[c] = bf16_to_float(idx_key[i * OR_DI + 32 * b + c]);
      or_mx_quant_block32(x, codes, &sc);
      for (int c = 0; c < 32; c += 2) pg[idx_nib_off(e, 32 * b + c)] = (uint8_t)(codes[c] | (codes[c + 1] << 4));
      pg[idx_mx_sf_off(e, b)] = sc;
    }
  }
}

void or_read_idx_mx(const uint8_t* idx_pages, const int32_t* bt, int32_t max_pages, int32_t r, int64_t s,
                    double* out) {
  const uint8_t* pg = idx_pages + page_of(bt, max_pages, r, s) * OR_IDX_MX_PAGE_BYTES;
  int64_t e = s % OR_PAGE;
  for (int c = 0; c < OR_DI; ++c) {
    uint8_t byte = pg[idx_nib_off(e, c)];
    uint8_t code = (c % 2) ? (byte >> 4) : (byte & 15);
    out[c] = or_e2m1_decode(code) * ldexp(1.0, (int)pg[idx_mx_sf_off(e, c / 32)] - 127);
  }
}

/* Index score over MXFP4 keys with the query quantised to MXFP4 too (the query-key
 * path is FP4 end to end): the same sum as or_index_score, fp64. */
void or_index_score_mx(const uint16_t* q_idx, const float* w, int32_t heads, const uint8_t* idx_pages,
                       const int32_t* bt, int32_t max_pages, int32_t r, int64_t s0, int64_t s1, double* I,
                       double* M) {
  double* qh = (double*)malloc(sizeof(double) * heads * OR_DI);
  for (int j = 0; j < heads; ++j) {
    for (int b = 0; b < 4; ++b) {
      float x[32];
      uint8_t codes[32], sc;
      for (int i = 0; i < 32; ++i) x[i] = bf16_to_float(q_idx[(int64_t)j * OR_DI + 32 * b + i]);
      or_mx_quant_block32(x, codes, &sc);
      for (int i = 0; i < 32; ++i) qh[j * OR_DI + 32 * b + i] = or_e2m1_decode(codes[i]) * ldexp(1.0, (int)sc - 127);
    }
  }
  const double scale = 1.0 / sqrt(128.0);
  double k[OR_DI];
  for (int64_t s = s0; s < s1; ++s) {
    or_read_idx_mx(idx_pages, bt, max_pages, r, s, k);
    double acc = 0.0, accm = 0.0;
    for (int j = 0; j < heads; ++j) {
      double dot = 0.0;
      for (int c = 0; c < OR_DI; ++c) dot += qh[j * OR_DI + c] * k[c];
      double relu = dot * scale > 0.0 ? dot * scale : 0.0;
      acc += (double)w[j] * relu;
      accm += fabs((double)w[j]) * relu;
    }
    I[s - s0] = acc;
    M[s - s0] = accm;
  }
  free(qh);
}

/* ----------------------------------------- hierarchical sparse indexer [P1][P4]
 * "DeepSeek's Attention and KV Cache", "The hierarchical indexer", and "From First
 * Principles: DeepSeek-V4.1-Flash Inference", "The Hierarchical Sparse Indexer": the
 * Full layer, besides its own top-512, gives every block of 8 consecutive positions the
 * maximum score inside it, keeps at most the 2,048 highest-scoring blocks and publishes
 * their positions (at most 2,048 x 8 = 16,384) as a candidate pool; the Reindex layers
 * score only the pool and take their own top-512 from inside it.
 * Readings (the pages are silent): block j covers positions [8j, 8j + 8) that are
 * visible (s < n_visible); equal block maxima prefer the lower block (the top-k's
 * lower-index rule), -0 equals +0; the pool lists the positions in ascending order,
 * -1 after the last. */
typedef struct {
  double v;
  int64_t j;
} or_blk;

static int cmp_blk(const void* a, const void* b) {
  const or_blk* x = (const or_blk*)a;
  const or_blk* y = (const or_blk*)b;
  if (x->v != y->v) return x->v > y->v ? -1 : 1;
  return x->j < y->j ? -1 : (x->j > y->j);
}

/* pool: [keep * block] positions ascending, -1 padded; returns the number listed. */
int64_t or_block_pool(const float* scores, int64_t nv, int32_t block, int32_t keep, int32_t* pool) {
  int64_t nb = (nv + block - 1) / block;
  or_blk* b = (or_blk*)malloc(sizeof(or_blk) * (nb > 0 ? nb : 1));
  for (int64_t j = 0; j < nb; ++j) {
    double m = -INFINITY;
    for (int64_t s = j * block; s < (j + 1) * block && s < nv; ++s)
      if ((double)scores[s] > m) m = (double)scores[s];
    b[j].v = m == 0.0 ? 0.0 : m; /* -0 -> +0 */
    b[j].j = j;
  }
  qsort(b, (size_t)nb, sizeof(or_blk), cmp_blk);
  int64_t take = nb < keep ? nb : keep;
  uint8_t* sel = (uint8_t*)calloc((size_t)(nb > 0 ? nb : 1), 1);
  for (int64_t i = 0; i < take; ++i) sel[b[i].j] = 1;
  int64_t n = 0;
  for (int64_t j = 0; j < nb; ++j)
    if (sel[j])
      for (int64_t s = j * block; s < (j + 1) * block && s < nv; ++s) pool[n++] = (int32_t)s;
  for (int64_t i = n; i < (int64_t)keep * block; ++i) pool[i] = -1;
  free(sel);
  free(b);
  return n;
}

/* Index scores at the listed positions (n of them, each < the request's cache length)
 * of request r; mx selects the MXFP4 key format.  The same sums as or_index_score. */
void or_index_score_at(const uint16_t* q_idx, const float* w, int32_t heads, const uint8_t* idx_pages,
                       const int32_t* bt, int32_t max_pages, int32_t r, const int32_t* pos, int64_t n, int32_t mx,
                       double* I, double* M) {
  for (int64_t i = 0; i < n; ++i) {
    if (mx)
      or_index_score_mx(q_idx, w, heads, idx_pages, bt, max_pages, r, pos[i], pos[i] + 1, I + i, M + i);
    else
      or_index_score(q_idx, w, heads, idx_pages, bt, max_pages, r, pos[i], pos[i] + 1, I + i, M + i);
  }
}

/* ------------------------------------- bf16 reference of the index score [P1]
 * "DeepSeek's Attention and KV Cache", "DeepSeek-V4 ... the indexer in four bits": with
 * the query and key in FP4 the V4 report keeps 99.7 % recall of the top-k.  This is the
 * same score from the unquantised bf16 query and key, fp64 throughout, for measuring
 * the recall of the FP4 selection (a reported figure, not a pin). */
void or_index_score_bf16(const uint16_t* q_idx, const float* w, int32_t heads, const uint16_t* keys, int64_t n,
                         double* I) {
  const double scale = 1.0 / sqrt(128.0);
  for (int64_t s = 0; s < n; ++s) {
    double acc = 0.0;
    for (int j = 0; j < heads; ++j) {
      double dot = 0.0;
      for (int c = 0; c < OR_DI; ++c)
        dot += (double)bf16_to_float(q_idx[(int64_t)j * OR_DI + c]) * (double)bf16_to_float(keys[s * OR_DI + c]);
      double relu = dot * scale > 0.0 ? dot * scale : 0.0;
      acc += (double)w[j] * relu;
    }
    I[s] = acc;
  }
}
