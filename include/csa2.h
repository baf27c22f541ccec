/*
 * csa2.h -- C ABI of libcsa2: one CSA2 attention layer (DeepSeek-V4.1-Flash) over an
 * FP4 KV cache, at decode and chunked prefill, on one NVIDIA GB300 (sm_103a).
 *
 * Sources (page title, section):
 *   [P1] "DeepSeek's Attention and KV Cache - From MLA to CSA2, From First Principles":
 *        "A Precision Primer", "DeepSeek-V3.2: Sparse Attention With a Learned Indexer",
 *        "DeepSeek-V4: Compress the Sequence, Then Sparsify",
 *        "DeepSeek-V4.1: Reuse Across Layers, Project Across Halves, Store in Four Bits".
 *   [P2] "From MLA to DSA to HCA/CSA: DeepSeek V3.2 and V4 Attention":
 *        "The indexer", "What replaced MLA", "The sliding window", "CSA: two changes to HCA".
 *   [P3] "DeepSeek-V4.1-Flash and the 890-byte KV cache", sections 2 and 3.
 *   [P4] "From First Principles: DeepSeek-V4.1-Flash Inference":
 *        "Two branches", "What's in a cell", "CSA2: four layers keep their own copy".
 *
 * Conventions for every entry point:
 *   - Pointers named here are DEVICE pointers owned by the caller, unless stated.
 *     The library allocates nothing; scratch memory is the caller's workspace `ws`
 *     of `ws_bytes` bytes (see csa2_workspace_bytes), 256-byte aligned.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  Argument validation is synchronous: a bad argument returns
 *     CSA2_ERR_INVALID_ARG / CSA2_ERR_UNSUPPORTED / CSA2_ERR_WORKSPACE before anything
 *     is launched, and csa2_last_error() gives a message.  A failed launch returns
 *     CSA2_ERR_CUDA.  Limit breaches found on the device (a page id outside the cache,
 *     a position beyond a request's pages, an index beyond the visible prefix, a
 *     pipeline wait that ran out) skip the offending access and set an error word in
 *     the workspace that csa2_check() reports (CSA2_ERR_DEVICE / CSA2_ERR_TIMEOUT).
 *   - bf16 tensors are passed as `const void*` holding IEEE bfloat16 bit patterns.
 *   - All device pointers must be 16-byte aligned; cache page arrays and the
 *     workspace 256-byte aligned.
 */
#ifndef CSA2_H_
#define CSA2_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* csa2_stream_t; /* = cudaStream_t */

typedef enum csa2_status {
  CSA2_OK = 0,
  CSA2_ERR_INVALID_ARG = 1, /* a pointer, size or stride is invalid             */
  CSA2_ERR_UNSUPPORTED = 2, /* a valid but unimplemented shape (e.g. k != 512) */
  CSA2_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed            */
  CSA2_ERR_TIMEOUT = 4,     /* a device-side bounded wait ran out              */
  CSA2_ERR_WORKSPACE = 5,   /* ws is NULL, misaligned or smaller than needed   */
  CSA2_ERR_DEVICE = 6       /* a device-side limit check failed (see csa2_check) */
} csa2_status;

/* Sizes fixed by the pages.
 *   CSA2_D      main-KV latent width, 512 [P1 "DeepSeek-V4.1"; P2 "What replaced MLA"]
 *   CSA2_DI     indexer key/query width, 128 [P1 "DeepSeek-V3.2"; P2 "The indexer"]
 *   CSA2_BLOCK  channels per E4M3 scale, 16 [P1 "DeepSeek-V4.1": E2M1 with one E4M3
 *               scale per 16 channels, NVFP4 without its global scale]
 *   CSA2_KV_BYTES  256 B of nibbles + 32 scale bytes = 288 [P1 "DeepSeek-V4.1"]
 *   CSA2_IDX_BYTES 64 B of nibbles + 8 scale bytes = 72 [P3 section 3]
 *   CSA2_TOPK   selected entries per query, 512 [P1 "DeepSeek-V4.1"; P3 section 2]
 *   CSA2_WIN    sliding-window entries, 128 [P1 "DeepSeek-V4"; P4 "Two branches"]
 *   CSA2_HEADS  attention query heads sharing one KV entry, 64 [P2 "Part 2"; P4]
 *   CSA2_WIN_BYTES FP8 window entry: 512 E4M3 bytes + 16 E8M0 scales = 528 [P1 "Four
 *               bits for the main KV, eight for the window"]
 * Layout choice of this library (the pages give entry sizes only):
 *   CSA2_PAGE   entries per cache page, 128. */
enum {
  CSA2_D = 512,
  CSA2_DI = 128,
  CSA2_BLOCK = 16,
  CSA2_KV_BYTES = 288,
  CSA2_IDX_BYTES = 72,
  CSA2_TOPK = 512,
  CSA2_WIN = 128,
  CSA2_HEADS = 64,
  CSA2_PAGE = 128,
  CSA2_KV_PAGE_BYTES = 36864,  /* 128 x 288 */
  CSA2_IDX_PAGE_BYTES = 9216,  /* 128 x 72  */
  CSA2_WIN_BYTES = 528,
  CSA2_IDX_MX_BYTES = 68,        /* MXFP4 indexer key: 64 B of nibbles + 4 E8M0 scales */
  CSA2_IDX_MX_PAGE_BYTES = 8704, /* 128 x 68 */
  CSA2_POOL_BLOCK = 8,           /* positions per block of the hierarchical indexer  */
  CSA2_POOL_BLOCKS = 2048,       /* blocks kept in a candidate pool                  */
  CSA2_POOL = 16384              /* positions in a full candidate pool (2048 x 8)    */
};

/* Indexer-K formats (csa2_cache.idx_format).
 *   CSA2_IDX_E4M3_16  E2M1 with one E4M3 scale per 16 channels, 72 B per entry: the
 *                     main-KV format [P3 section 3].
 *   CSA2_IDX_MXFP4    MXFP4: E2M1 with one E8M0 (power-of-two) scale per 32 channels,
 *                     68 B per entry [P1 "A Precision Primer", MX formats and E8M0;
 *                     P1 "DeepSeek-V4", the indexer in four bits; P4 "What's in a cell"].
 *                     Scale 2^e with e the smallest exponent such that the block maximum
 *                     is <= 6 * 2^e (no element clips; the primer's worked example has a
 *                     maximum of 3 + delta take the scale 1), clamped to [-127, 127], -127
 *                     for an all-zero block; code_i = E2M1_rn(x_i / 2^e), exact quotient.
 *                     The indexer query is quantised in the same format, and the product
 *                     runs on the MX block-scaled FP4 tensor cores. */
enum { CSA2_IDX_E4M3_16 = 0, CSA2_IDX_MXFP4 = 1 };

/* The global cache of one CSA2 Full layer: a paged main-KV cache and a paged
 * indexer-K cache sharing one block table [P1 "DeepSeek-V4": compressed entries are a
 * classical paged cache; P4 "What's in a cell": main KV + indexer K per entry].
 *
 * Entry s of request r lives in page p = block_table[r*max_pages + s/128] (or
 * p = r*max_pages + s/128 when block_table is NULL), slot e = s % 128.
 *
 * Main-KV page (36864 B): entry e occupies bytes [288e, 288e+288): byte i < 256 holds
 *   channel 2i in its low nibble and channel 2i+1 in its high nibble (E2M1 codes:
 *   bit 3 sign, bits 0-2 magnitude index of 0,.5,1,1.5,2,3,4,6); bytes 256..287 hold
 *   the E4M3 scale of channels [16b, 16b+16) at byte 256+b.
 * Indexer-K page (9216 B = 128 x 72): the nibble of entry e, channel c sits at byte
 *   (e/8)*512 + (c/32)*128 + (e%8)*16 + (c%32)/2 (low nibble = even c): eight entries
 *   form a 512-byte group of four 128-byte core blocks, the operand layout of the
 *   block-scaled tensor-core MMA, so a page feeds the MMA without reshuffling.  The
 *   E4M3 scale of entry e, block b sits at byte 8192 + (b/4)*512 + (e%32)*16 +
 *   (e/32)*4 + b%4, the scale-factor layout the MMA reads.
 * Each entry still costs exactly 288 + 72 bytes.
 * MXFP4 indexer-K page (idx_format = CSA2_IDX_MXFP4; 8704 B = 128 x 68): the nibbles as
 *   above; the E8M0 code e + 127 of entry e, block b (channels [32b, 32b+32)) at byte
 *   8192 + (e%32)*16 + (e/32)*4 + b.  Each entry costs 288 + 68 bytes. */
typedef struct csa2_cache {
  uint8_t* kv;                /* main-KV pages [n_pages][36864]                     */
  uint8_t* idx;               /* indexer-K pages [n_pages][9216], or [n_pages][8704]
                                 with idx_format = CSA2_IDX_MXFP4                  */
  const int32_t* block_table; /* [n_req][max_pages] page ids, or NULL (contiguous)  */
  int32_t max_pages;          /* pages per request (row length of block_table)      */
  int32_t n_pages;            /* pages allocated in kv and idx (bounds check)       */
  int32_t idx_format;         /* CSA2_IDX_E4M3_16 (0, default) or CSA2_IDX_MXFP4    */
} csa2_cache;

/* One CSA2 layer step for n_q queries [P1 "DeepSeek-V4.1" three modes; P3 section 2;
 * P4 "CSA2"].  Query q belongs to request req[q], sees entries [0, n_visible[q]) of
 * that request's cache, and attends to the topk selected entries plus its window
 * rows window[(win_start[q] + i) * 512 ...] for i < win_len[q] (<= 128). */
typedef struct csa2_step {
  int64_t n_q;               /* number of queries (decode: one per request)            */
  int32_t heads;             /* attention heads, must be 64                            */
  int32_t heads_I;           /* indexer heads: 64 or 32                                */
  int32_t topk;              /* must be 512                                            */
  int32_t group;             /* indexer query group: 1, or 2 when consecutive queries
                                share one request (chunked prefill)                    */
  int64_t t_max;             /* host-known upper bound of n_visible[] (grid sizing)    */
  const void* q;             /* bf16 [n_q][heads][512] attention queries: post-RoPE, or
                                pre-RoPE when rope_cos / rope_sin are given           */
  const void* q_idx;         /* bf16 [n_q][heads_I][128] indexer queries (Full/Reindex)*/
  const float* w;            /* fp32 [n_q][heads_I] indexer head weights               */
  const int32_t* req;        /* [n_q] request of each query                            */
  const int32_t* n_visible;  /* [n_q] visible cache entries of each query              */
  const void* window;        /* bf16 window rows [*][512]                              */
  const int64_t* win_start;  /* [n_q] first window row of each query                   */
  const int32_t* win_len;    /* [n_q] window rows of each query, 0..128                */
  int64_t n_new;             /* Full mode: entries to pack before scoring (may be 0)   */
  const void* new_latent;    /* bf16 [n_new][512] main-KV latents (post-RoPE)          */
  const void* new_idx_key;   /* bf16 [n_new][128] indexer keys                         */
  const int32_t* new_req;    /* [n_new] request of each new entry                      */
  const int64_t* new_pos;    /* [n_new] position of each new entry in its request      */
  csa2_cache cache;          /* the (possibly shared) global cache                     */
  int32_t* topk_idx;         /* [n_q][topk]: output (Full, Reindex) or input (Reuse);
                                ascending entry indices, -1 padded                     */
  float* scores;             /* optional fp32 [n_q][ld] index scores out; NULL = keep
                                them in the workspace                                  */
  int64_t ld;                /* row stride of scores (elements, multiple of 4) or 0    */
  float softmax_scale;       /* <= 0 selects 512^-0.5                                  */
  void* out;                 /* bf16 [n_q][heads][512] attention output                */
  float* lse;                /* optional fp32 [n_q][heads] natural-log sum-exp         */
  /* Attention sinks [P2 "From MLA to DSA to HCA/CSA", "The sliding window"]: one logit
   * per head joins every score row of the softmax and has no value vector, so the
   * weights of the real keys sum to 1 - p_sink; lse includes it. */
  const float* sinks;        /* optional fp32 [heads] natural-log sink logits; NULL = none */
  /* Partial RoPE [P2 "What replaced MLA"]: the trailing 64 channels of q are rotated at
   * the query's position, q = q cos + rotate_half(q) sin with rotate_half pairing
   * channel 448 + i with 480 + i (angle i < 32), and the output is rotated back with the
   * negated angle.  Cached entries are rotated before they are packed, as before. */
  const float* rope_cos;     /* optional fp32 [n_q][32] cos of the query position's angles;
                                NULL (with rope_sin) = q post-RoPE, O returned as is    */
  const float* rope_sin;     /* optional fp32 [n_q][32] sin of the same angles           */
  /* FP8 window ring (see csa2_pack_window).  When win_ring is set, the window of query
   * q is the ring entries of positions win_start[q] - win_len[q] + 1 .. win_start[q] of
   * request req[q] (win_start is then the newest window position) and `window` is not
   * read; NULL = bf16 window rows as above. */
  const uint8_t* win_ring;   /* optional [win_ring_reqs][128][528]                      */
  int32_t win_ring_reqs;     /* requests in win_ring (bounds check)                    */
  /* Hierarchical sparse indexer [P1 "The hierarchical indexer"; P4 "The Hierarchical
   * Sparse Indexer"]: a candidate pool per query, int32 [n_q][16384], the positions of
   * up to 2,048 blocks of 8 in ascending order, -1 after the last.
   *   Full mode:    when set, the call also publishes its pool here: every block of 8
   *                 positions [8j, 8j+8) (visible ones only) gets the maximum of its
   *                 index scores, the 2,048 largest blocks are kept (equal maxima prefer
   *                 the lower block, -0 equals +0; all blocks when there are fewer).
   *   Reindex mode: when set, the call scores only the pool's positions and takes its own
   *                 top-512 among them (ties to the lower position); `scores`, when
   *                 given, receives the pool-slot scores [n_q][ld >= 16384], slot i
   *                 scoring position pool[q][i].  A pool that is not ascending blocks of 8
   *                 visible positions sets the error word (info 6).  group must be 1.
   * Either mode needs csa2_workspace_bytes_pool() bytes of workspace; Reuse mode ignores
 * the pool. */
  int32_t* pool;
} csa2_step;

/* Message describing the last failed call on this host thread ("" if none). */
const char* csa2_last_error(void);

/* Workspace bytes needed by every call below for n_q queries of up to t_max visible
 * entries with heads_I indexer heads; scores_in_ws != 0 when the caller does not
 * provide a score array (the scores then live in the workspace).  For small batches
 * (n_q < 76 on 152 SMs) it includes the attention's partial outputs: each query's key tiles
 * are then split over a cluster of 2 to 5 CTAs that merge their fp32 partials through the
 * workspace (n_q * S * 64 * 514 * 4 bytes for S CTAs per query, at most about 20 MB).
 * Bytes [0, 8) of the workspace are the error word (csa2_check); after a call that scores
 * (csa2_index_score, Full, Reindex) bytes [256, 256 + ceil(n_q / group) * (N * 64 + 1024))
 * hold the quantised indexer query, N = group * heads_I rows per group in the
 * indexer page's operand layout with the scale atoms after the nibbles (N * 64 + 512 with
 * MXFP4 keys); row n is head n % heads_I of query group * g + n / heads_I.
 * Host-only. */
size_t csa2_workspace_bytes(int64_t n_q, int32_t heads_I, int64_t t_max, int32_t scores_in_ws);

/* Workspace bytes for the same calls with a candidate pool (csa2_step.pool set): adds
 * the block-maximum keys of a Full layer (4 B per 8 entries per query) and, for a
 * pool-restricted Reindex, the compact indexer pages of each query's pool (128 pages),
 * its scores and its top-512 slots.  Host-only. */
size_t csa2_workspace_bytes_pool(int64_t n_q, int32_t heads_I, int64_t t_max, int32_t scores_in_ws);

/* Pack n new entries into the cache [P1 "DeepSeek-V4.1", Four bits for the main KV;
 * P3 section 3].  For each 16-channel block: amax = max|x|, scale =
 * E4M3_rn_satfinite(amax / 6) (fp32 division), code_i = E2M1_rn_satfinite(x_i / scale)
 * (fp32 division; a zero scale gives +0 codes).  latent: bf16 [n][512]; idx_key: bf16
 * [n][128]; req/pos: [n].  Entries at the same (req, pos) must not repeat in one call.
 * With cache->idx_format = CSA2_IDX_MXFP4 the indexer key takes the MXFP4 format
 * (see CSA2_IDX_MXFP4); the main-KV entry is unchanged. */
csa2_status csa2_pack_kv(const void* latent, const void* idx_key, const int32_t* req,
                         const int64_t* pos, int64_t n, const csa2_cache* cache, void* ws,
                         size_t ws_bytes, csa2_stream_t stream);

/* FP8 window ring [P1 "Four bits for the main KV, eight for the window": a window
 * entry is 512 E4M3 bytes plus 16 E8M0 scales, 528 bytes; P1 "Definition and the
 * bounded cache": position i lives in slot i mod 128 of its request's ring].
 * ring: [n_ring][128][528] bytes, 16-byte aligned; entry layout: bytes [0, 512) the
 * E4M3 codes in channel order, [512, 528) the E8M0 codes e + 127 of the 16 blocks of 32
 * channels.  For each block: e = the smallest exponent with amax <= 448 * 2^e (no
 * element clips), clamped to [-127, 127] (all-zero block: -127); code_i =
 * E4M3_rn(x_i / 2^e).  rows: bf16 [n][512]; req/pos: [n] with 0 <= req < n_ring and
 * pos >= 0 (device-side violations set the error word).  Entries of one call must not
 * share a slot. */
csa2_status csa2_pack_window(const void* rows, const int32_t* req, const int64_t* pos, int64_t n, uint8_t* ring,
                             int32_t n_ring, void* ws, size_t ws_bytes, csa2_stream_t stream);

/* Lightning-indexer scores [P1 "DeepSeek-V3.2" index score, "DeepSeek-V4" the indexer
 * in four bits; P2 "The indexer", "CSA" scorer]:
 *   scores[q*ld + s] = sum_j w[q][j] * ReLU( qhat[q][j] . khat[s] * 128^-0.5 )
 * for s < n_visible[q], where qhat is q_idx quantised in-call with the same E2M1/E4M3
 * block codec and khat the cached indexer key (the product runs on the block-scaled
 * FP4 tensor cores, fp32 accumulation).  Entries s >= n_visible[q] are not written.
 * With cache->idx_format = CSA2_IDX_MXFP4, qhat and khat are MXFP4 (E8M0 scale per 32
 * channels) and the product runs as the MX block-scaled MMA.
 * group = 1 or 2 consecutive queries of one request per MMA tile. */
csa2_status csa2_index_score(const void* q_idx, const float* w, int32_t heads_I,
                             const int32_t* req, const int32_t* n_visible, int64_t n_q,
                             int32_t group, int64_t t_max, const csa2_cache* cache,
                             float* scores, int64_t ld, void* ws, size_t ws_bytes,
                             csa2_stream_t stream);

/* Top-k selection [P1 "DeepSeek-V3.2" top-k, "DeepSeek-V4.1" top-512; P2 "CSA" -1
 * sentinel]: for each row q the k largest of scores[q*ld + s], s < n_visible[q];
 * equal scores prefer the lower index, -0 equals +0; out_idx[q][0..k) lists the chosen
 * indices in ascending order, padded with -1 when n_visible[q] < k.  k must be 512. */
csa2_status csa2_topk(const float* scores, int64_t ld, const int32_t* n_visible, int64_t n_q,
                      int64_t t_max, int32_t k, int32_t* out_idx, void* ws, size_t ws_bytes,
                      csa2_stream_t stream);

/* No-allocation variant of csa2_topk (the pages have no counterpart to this entry point).
 * Some callers cannot call cudaMalloc: a serving engine that hands all device memory to
 * its KV-cache pool at start-up, or a host thread that must not stall, since
 * cudaMalloc and cudaFree can synchronise the device.  This call takes no workspace:
 * its scratch is a fixed device array inside the library, sized for at most 128 rows
 * (n_q <= 128, about 5.5 MB, held on every GPU that loads the library until the
 * process exits).  It allocates nothing and calls no allocating routine.
 *   - Same arguments and result as csa2_topk; n_q > 128 returns CSA2_ERR_WORKSPACE.
 *   - The first call on a device looks up the array's device address (once per device,
 *     with that device current); make that first call before any stream capture.
 *   - Every call on a device shares the one array and leaves its contents behind (the
 *     parts that must start at zero are cleared by each call): calls whose work
 *     overlaps on the GPU (different streams, or different host threads) race and
 *     must be serialised by the caller.
 *   - Device-side checks write the array's own error word, not a caller workspace, so
 *     csa2_check does not report them. */
csa2_status csa2_topk_noalloc(const float* scores, int64_t ld, const int32_t* n_visible, int64_t n_q,
                              int64_t t_max, int32_t k, int32_t* out_idx, csa2_stream_t stream);

/* Error word of the last csa2_topk_noalloc call (no counterpart on the pages): synchronises
 * `stream`, reads and clears the fixed array's error word and reports it as csa2_check
 * does for a workspace (CSA2_OK, or CSA2_ERR_DEVICE with *info = 3 when a row's counts
 * disagree between the passes, which overlapping calls on the shared array can cause).
 * Allocates nothing. */
csa2_status csa2_topk_noalloc_check(csa2_stream_t stream, int32_t* info);

/* Full mode [P3 section 2 "Full Mode"; P4 "CSA2"]: pack the step's new entries, score
 * the cache with the step's own indexer query, select its own top-512, then run the
 * shared-KV MQA over the 512 selected (dequantised) entries plus the window rows:
 *   for each head h: S = scale * Q_h . K^T over keys K = [selected ; window] (K == V),
 *   O_h = softmax(S) K, lse_h = log sum exp S   [P1 "DeepSeek-V4"; P2 "What replaced MLA"].
 * Window and selection may overlap; nothing is de-duplicated. */
csa2_status csa2_sparse_attn_full(const csa2_step* step, void* ws, size_t ws_bytes,
                                  csa2_stream_t stream);

/* Reindex mode [P3 section 2 "Reindex Mode"]: as Full mode on a cache written by
 * another layer (no packing): its own indexer query, its own top-512, then attention. */
csa2_status csa2_sparse_attn_reindex(const csa2_step* step, void* ws, size_t ws_bytes,
                                     csa2_stream_t stream);

/* Reuse mode [P3 section 2 "Reuse Mode"]: attention only, over step->topk_idx given by a
 * preceding Full or Reindex layer plus the window rows; no indexer work. */
csa2_status csa2_sparse_attn_reuse(const csa2_step* step, void* ws, size_t ws_bytes,
                                   csa2_stream_t stream);

/* Synchronise `stream`, read and clear the workspace error word.  Returns CSA2_OK,
 * CSA2_ERR_DEVICE or CSA2_ERR_TIMEOUT; *info (may be NULL) receives a code naming the
 * check that failed (1 page id, 2 position, 3 top-k index, 4 group request, 5 wait,
 * 6 candidate pool). */
csa2_status csa2_check(void* ws, csa2_stream_t stream, int32_t* info);

/* Tensor-core throughput probe (a measurement utility; the pages have no counterpart):
 * n_ctas CTAs (one per SM when n_ctas is the SM count) each run `iters` back-to-back
 * tcgen05.mma of M = 128 and the given N, issued by `issuers` threads into separate TMEM
 * accumulators, with zeroed shared-memory operands; cycles[i] (device, int64) receives CTA
 * i's clock cycles from the first issue to the completion of the last MMA.
 *   kind 0: kind::f16, f16 x f16 -> fp32, K = 16 per MMA
 *   kind 1: kind::mxf4nvf4 scale_vec::4X (E2M1 x E2M1, E4M3 scale per 16), K = 64
 * FLOPs per MMA = 2 * 128 * n * K.  n in {64, 128, 256}; issuers in 1..4 with
 * issuers * n <= 448; iters in [1, 2^22].  "A Precision Primer" of "DeepSeek's Attention
 * and KV Cache" quotes the FP4 rate as a multiple of bf16 on Blackwell; this measures it. */
csa2_status csa2_probe_mma(int32_t kind, int32_t n, int32_t iters, int32_t issuers, int32_t n_ctas, int64_t* cycles,
                           csa2_stream_t stream);

/* Failure-path testing (the pages have no counterpart): sets the bound of every pipeline
 * wait of the indexer and attention kernels launched afterwards by this process (default
 * about 2 s; ns = 0 restores it).  A wait that runs out makes the kernel record
 * CSA2_ERR_TIMEOUT with info 5 in the workspace error word, wait (with the fixed 2 s bound)
 * for the copies and MMAs it has in flight, free its tensor memory and return; csa2_check
 * then reports it, and the outputs of that call are undefined.  Not thread-safe with
 * respect to concurrent launches from other host threads. */
csa2_status csa2_debug_set_wait_limit(uint64_t ns);

/* Number of kernels this library has launched in this process. */
int64_t csa2_launch_count(void);

/* Per-kernel device timing with CUDA events recorded on the launching stream.
 * csa2_trace_enable(1) starts recording (at most 4096 launches are kept);
 * csa2_trace_read(kind, &ms, &n) synchronises and returns the summed duration and count
 * of kernel `kind` (0 pack/quantise, 1 index score, 2/3/4 histogram, select and final
 * passes of the workspace top-k, 5 attention, 6 cluster top-k, 7 candidate-pool
 * selection, 8 pool gather, 9 pool slot map, 10 pool block maxima, 11 attention split
 * combine, 12 FP8 window pack); csa2_trace_enable(0) stops and clears. */
csa2_status csa2_trace_enable(int32_t on);
csa2_status csa2_trace_read(int32_t kind, double* total_ms, int64_t* count);

#ifdef __cplusplus
}
#endif

#endif /* CSA2_H_ */
