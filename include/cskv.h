/*
 * cskv - compressed sparse attention KV: DeepSeek-V4-style compressed-KV decode
 * attention for NVIDIA GB300 (sm_103a).
 *
 * C ABI of libcskv.so.  Every pointer argument named "device" is CUDA device
 * memory owned by the caller; the library never allocates, frees or keeps a
 * pointer past the call.  Every call is asynchronous on the given stream
 * (a cudaStream_t passed as void*, NULL = legacy default stream) and never
 * synchronises, except cskv_device_status().
 *
 * Errors: arguments are checked on the host before anything is launched; a
 * failed check returns CSKV_ERR_INVALID (or CSKV_ERR_UNSUPPORTED) and launches
 * nothing.  A failed launch returns CSKV_ERR_CUDA.  Problems that only the
 * device can see (a block-table entry outside the pool, a context longer than
 * the table, a bounded wait that ran out) never fault: the kernel skips the
 * offending access and sets a sticky error word, which cskv_device_status()
 * reports and clears.
 *
 * Layout conventions (all row-major):
 *  - a cache "row" is one 512-d compressed entry / window token (main lane) or
 *    one 128-d index key, stored in a cskv_format;
 *  - caches are paged: 64 rows per page, a per-request block table maps a
 *    request's logical page p (rows 64p .. 64p+63) to a physical page of a
 *    shared pool;
 *  - the sliding-window ring of request b is 128 rows, row (b*128 + pos % 128).
 *
 * The operations follow "DeepSeek-V4 deep dive" (gangliao.me): section 4 for
 * the compressor, section 5.2 for the indexer, sections 3.3-3.4 and 5.3 for the
 * attention; the cache formats follow the "DeepSeek-V4-Flash" model record
 * (528 B FP8 rows) and the "DeepSeek-V4.1-Flash" KV-compression diagram
 * (MXFP4 with an E4M3 scale per 16 channels).
 */
#ifndef CSKV_H
#define CSKV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define CSKV_API __attribute__((visibility("default")))
#else
#define CSKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CSKV_OK = 0,
  CSKV_ERR_INVALID = 1,     /* bad argument; nothing launched */
  CSKV_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. > 64 indexer heads) */
  CSKV_ERR_CUDA = 3,        /* a CUDA call failed */
  CSKV_ERR_TIMEOUT = 4,     /* device: a bounded wait gave up (see cskv_set_spin_limit) */
  CSKV_ERR_BOUNDS = 5       /* device: an index outside its table or pool was skipped */
} cskv_status;

typedef enum {
  /* dim bf16 values: 2*dim bytes (1024 B at 512). */
  CSKV_FMT_BF16 = 0,
  /* dim float8_e4m3 codes, then dim/32 float8_e8m0 scale bytes (scale j covers
   * channels 32j..32j+31): dim + dim/32 bytes, 528 B at 512, inline per row.
   * "DeepSeek-V4-Flash" model record, engine kernel constraint (2). */
  CSKV_FMT_FP8_E4M3_E8M0_B32 = 1,
  /* dim/2 bytes of packed float4_e2m1 (channel 2i in the low nibble of byte i),
   * then dim/16 float8_e4m3 scale codes (scale j covers channels 16j..16j+15):
   * 288 B at 512, inline per row.  "DeepSeek-V4.1-Flash" diagram, MXFP4. */
  CSKV_FMT_FP4_E2M1_E4M3_B16 = 2,
  /* index keys: dim float8_e4m3 codes with one scale for the whole row, stored
   * as the fp32 value of a power of two (the rounding rules of format 1 with a
   * block of dim values): dim + 4 bytes, 132 B per 128-d key (the size of the
   * V3.2 index key).  Each 64-row page stores its 64 code rows first (dim bytes
   * each), then its 64 fp32 scales: 8,448 B per page.  Index keys only. */
  CSKV_FMT_FP8_E4M3_ROWSCALE_PAGESPLIT = 3,
  /* index keys rotated and coded in FP4 ("DeepSeek-V4 deep dive", section 5.2:
   * the indexer's keys and queries go through a Hadamard rotation, then FP4
   * rounding with block size 32; "DeepSeek-V4.1 Flash", section 10.4: MXFP4).
   * A written row is rotated by H / sqrt(dim) (H the Sylvester Hadamard matrix,
   * H[i][j] = (-1)^popcount(i & j)) in a fixed fp32 order - butterflies of
   * stride 1, 2, ..., dim/2, each (a, b) -> (a + b, a - b), then one product by
   * fp32(1 / sqrt(dim)) - then coded as dim/2 bytes of packed float4_e2m1
   * (channel 2i in the low nibble of byte i) and dim/32 float8_e8m0 scales (scale
   * j covers channels 32j..32j+31: the smallest 2^e with amax <= 6 * 2^e; codes
   * RNE(x * 2^-e)): 68 B per 128-d key.  Each 64-row page stores its 64 code rows
   * first (dim/2 bytes each), then its 64 scale rows (dim/32 bytes each): 4,352 B
   * per page.  The indexer rotates and codes its queries the same way and keeps
   * its scores in bf16.  Index keys only (dim 128). */
  CSKV_FMT_FP4_E2M1_E8M0_HADAMARD_PAGESPLIT = 4
} cskv_format;

/* A paged cache (or, with block_table == NULL, a flat array of rows in which
 * row r lives in page r/64 at slot r%64). */
typedef struct cskv_paged {
  void* pool;                 /* device, 16-byte aligned: num_pages pages, page_bytes apart */
  const int32_t* block_table; /* device [batch, max_pages] logical page -> physical page, or NULL */
  int64_t page_bytes;         /* bytes from one page to the next: >= 64*row_bytes, multiple of 16 */
  int32_t num_pages;          /* pages in the pool; table entries outside [0, num_pages) are errors */
  int32_t max_pages;          /* row stride of block_table = most pages one request may own */
  int32_t fmt;                /* cskv_format */
  int32_t dim;                /* 512 (main entries and window) or 128 (index keys) */
} cskv_paged;

/* Bytes of one row of format fmt at dimension dim (528, 288, 1024, 132 ...);
 * 0 for an invalid pair. */
CSKV_API size_t cskv_row_bytes(int32_t fmt, int32_t dim);

/* Static description of a status code. */
CSKV_API const char* cskv_status_string(int32_t status);

/* Library version (major*10000 + minor*100 + patch). */
CSKV_API int32_t cskv_version(void);

/* Synchronises `stream`, then returns and clears the sticky device error word
 * (CSKV_OK if no kernel reported a problem since the last call).  The only call
 * that blocks. */
CSKV_API int32_t cskv_device_status(void* stream);

/* Process-wide state.  The library keeps no per-call state between calls; two
 * settings are the exceptions, both process-wide (every device, every thread):
 * the spin limit below and the measurement hook cskv_set_timing_events.  Set them
 * before launching work from several threads; changing them while other threads
 * launch is safe (each launch reads them once) but the launch may see either value. */

/* Upper bound, in SM clock cycles, of every spin-wait on an mbarrier inside the
 * library's kernels (default 2^31, about one second).  A wait that runs out sets
 * CSKV_ERR_TIMEOUT, drains the copies its block has in flight and returns.
 * 0 restores the default.  Applies to launches made after the call.
 * Process-wide. */
CSKV_API void cskv_set_spin_limit(uint64_t cycles);

/* Measurement hook.  With both non-NULL (cudaEvent_t handles passed as void*),
 * every later cskv_index_topk call records `begin` when the kernel before its
 * score kernel (the query prep) completes, and `end` when the score kernel - the
 * pass that streams the index keys - completes.  Both are recorded on a
 * library-owned branch stream forked from the call's stream, so each kernel on the
 * call's stream still depends on the one before it alone and may overlap it as a
 * programmatic dependent launch (the score kernel's set-up overlaps the prep; the
 * attention's set-up overlaps the score kernel's tail).  Inside a stream capture both become external
 * event-record nodes, so a replayed CUDA graph records them on every replay.
 * NULL, NULL turns the hook off and joins the branch back into the stream of the
 * last timed call: under stream capture, turn it off before the capture ends.
 * Turning it on creates the branch stream for the current device: do that
 * outside any stream capture.  Process-wide; meant for benchmarks, not for
 * concurrent use. */
CSKV_API void cskv_set_timing_events(void* begin, void* end);

/* ------------------------------------------------------------------------
 * cskv_rope_table: the (cos, sin) table that the kernels take as their RoPE
 * input ("DeepSeek-V4 deep dive", section 3.3 "Partial RoPE and the inverse
 * rotation on the output": the last 64 dims are 32 adjacent pairs (2k, 2k+1),
 * pair k turning by position * f_k with f_k = theta^(-2k/64); compressed layers
 * use theta = 160,000; section 9.1 "Positions to 1M": YaRN, factor 16 over
 * 65,536 original positions, betas 32 and 1).  Host code, no GPU needed.
 *   out[i, k, 0] = (float) cos(positions[i] * f_k), out[i, k, 1] = (float) sin(...),
 * angles and functions in double precision, rounded to float once.
 * With yarn_factor > 1 the frequencies are YaRN-blended over the pair index:
 * low = floor(kb(beta_fast)), high = ceil(kb(beta_slow)), kb(beta) =
 * 64 ln(yarn_original / (2 pi beta)) / (2 ln theta), both kept in [0, 31];
 * ramp_k = clamp((k - low) / max(high - low, 0.001), 0, 1);
 * f_k <- f_k / yarn_factor * ramp_k + f_k * (1 - ramp_k).  yarn_factor <= 1:
 * plain frequencies (the other YaRN arguments are ignored).
 * positions: host int64 [n] (any value); out: host float [n, 32, 2]; n >= 0.
 * Errors: CSKV_ERR_INVALID for NULL pointers with n > 0, n < 0, theta <= 1, or
 * YaRN arguments that are not positive.
 * ------------------------------------------------------------------------ */
CSKV_API int32_t cskv_rope_table(const int64_t* positions, int32_t n, double theta, double yarn_factor,
                                 double yarn_original, double beta_fast, double beta_slow, float* out);

/* ------------------------------------------------------------------------
 * cskv_encode_rows: code rows of values into a cache.
 * Row i of src (fp32 or bf16, [n, dim] row-major) is coded in dst.fmt and
 * written as row dst_row[i] (or i if dst_row is NULL) of request dst_req[i]
 * (or 0 if dst_req is NULL) of the paged cache dst.  Codes follow the block
 * rules of cskv_compress (same bits for the same fp32 values).
 * src: device, 16-byte aligned; n >= 0; dim in {128, 512}.
 * ------------------------------------------------------------------------ */
CSKV_API int32_t cskv_encode_rows(const void* src, int32_t src_is_bf16, int32_t n, int32_t dim,
                         const int32_t* dst_req, const int32_t* dst_row,
                         cskv_paged dst, void* stream);

/* ------------------------------------------------------------------------
 * cskv_compress: the KV compressor ("DeepSeek-V4 deep dive", section 4.1
 * "Idea: average, but let the model choose the weights per channel" and
 * section 4.2 "Ratio 4 (CSA) overlaps; ratio 128 (HCA) does not").
 *
 * S independent sequences, each a chunk of T tokens (T a multiple of ratio)
 * of projected values kv and gate scores gate, both bf16 [S, T, coff, dim]
 * (coff = 2 with overlap, 1 without).  Entry i of sequence s pools, for every
 * channel c, the softmax over its slots of (gate + ape[slot position]) times kv:
 *   - no overlap: slots = tokens ratio*i .. ratio*i + ratio-1, channel half 0;
 *   - overlap (ratio <= 8): 2*ratio slots; the first ratio are the previous
 *     block's tokens through channel half 0 with ape[:, :dim], the last ratio
 *     the entry's own tokens through half 1 with ape[:, dim:].  The block before
 *     a chunk's first block comes from prev_kv / prev_gate ([S, ratio, 2, dim]
 *     bf16); NULL means the chunk starts the sequence (value 0, score -inf).
 * then RMSNorm over dim with weight norm_w ([dim] fp32; NULL = no norm) and
 * eps, then RoPE on the last 64 dims with the table rope_cs ([S, T/ratio, 32, 2]
 * fp32 (cos, sin) per entry, pair k = dims (dim-64+2k, dim-64+2k+1); NULL = no
 * RoPE), then coding in out.fmt.  Entry i of sequence s is written as row
 * first_entry[s] + i of request req[s] of `out`.
 *
 * Arithmetic: bit-exact fp32 in a fixed order (no fused multiply-add): slot
 * scores s = gate + ape; m = max; e = exp_own(s - m) (Cody-Waite reduction and a
 * degree-7 Taylor polynomial); numerator and denominator summed in slot order;
 * division; RMSNorm with a pairwise (recursive halves) sum of squares,
 * 1/sqrt(ss/dim + eps); rotation y0*c - y1*s, y0*s + y1*c.
 * ape: [ratio, coff*dim] fp32, or NULL for no slot bias (the same bits as a
 * zero table): the V4.1 compressor of "DeepSeek-V4.1 Flash" (section 1.1,
 * the sequence dimension) and the deep dive's implementation notes to section
 * 4 drop both the overlap and the slot bias, and pool 2 adjacent positions
 * (ratio 2) in the encoder or keep one entry per position (ratio 1) in the
 * decoder.  req, first_entry: device int32 [S].
 * Alignment: kv, gate, prev_* 8 bytes; ape, norm_w, rope_cs 16 bytes.
 * ------------------------------------------------------------------------ */
CSKV_API int32_t cskv_compress(const void* kv, const void* gate,
                      const void* prev_kv, const void* prev_gate,
                      const float* ape, const float* norm_w, float eps,
                      const float* rope_cs,
                      int32_t S, int32_t T, int32_t ratio, int32_t overlap, int32_t dim,
                      const int32_t* req, const int32_t* first_entry,
                      cskv_paged out, void* stream);

/* ------------------------------------------------------------------------
 * cskv_compress_many: several compressor jobs in one launch, e.g. the entry of
 * the main cache and the entry of the index-key cache that a decode step's
 * completed block produces ("DeepSeek-V4 deep dive", section 4.1 for the
 * computation; one launch instead of two is a deployment choice, the pages
 * have no counterpart).  Each job holds the arguments of one cskv_compress call,
 * is checked the same way and gives the same bits; jobs must not write the same
 * rows.  njobs in [1, 4].  Errors: CSKV_ERR_INVALID for a bad job (nothing is
 * launched), else as cskv_compress.
 * ------------------------------------------------------------------------ */
typedef struct {
  const void* kv;
  const void* gate;
  const void* prev_kv;
  const void* prev_gate;
  const float* ape;
  const float* norm_w;
  float eps;
  const float* rope_cs;
  int32_t S, T, ratio, overlap, dim;
  const int32_t* req;
  const int32_t* first_entry;
  cskv_paged out;
} cskv_compress_job;
CSKV_API int32_t cskv_compress_many(const cskv_compress_job* jobs, int32_t njobs, void* stream);

/* ------------------------------------------------------------------------
 * cskv_decode_append: the state update of one decode step ("DeepSeek-V4 deep
 * dive", section 4.3 "What is cached" and its implementation notes to section
 * 4: every compressor keeps the projected tokens of its unfinished block, and of
 * the block before it when it overlaps, in a fixed-size per-request state; the
 * window keeps the last 128 tokens as a ring).
 *
 * For each job and each request b with pos[b] >= 0 (the position p of the
 * request's new token; pos[b] < 0 = no token for b this step):
 *   - ratio > 1: the token's kv and gate ([B, coff, dim] bf16, coff = 2 with
 *     overlap) go into slot (overlap ? ratio : 0) + p % ratio of the request's
 *     state ring state_kv / state_gate ([B, nblk * ratio, coff, dim] bf16,
 *     nblk = 2 with overlap: the previous block, then the one being filled;
 *     else 1).  If p + 1 is a multiple of ratio the block is complete: its
 *     entry is pooled exactly as cskv_compress pools entry 1 of a 2-block
 *     sequence (overlap) or entry 0 of a 1-block one, and written as row
 *     (p + 1) / ratio - 1 of request b of `out`; with overlap the completed
 *     block then moves into the previous-block slots.  A fresh request's ring
 *     holds kv 0 and gate -inf (bf16 0xFF80) in every slot: the first block
 *     then sees an empty previous block, as in cskv_compress.
 *   - ratio 1 (no pooling; state_* unused and may be NULL, gate may be NULL):
 *     the entry is the token itself, RMSNorm-ed, rotated and coded; it is
 *     written to row p, or, with ring_rows > 0, to row p % ring_rows (the
 *     window ring: give it the 128-row window as a paged cache of two 64-row
 *     pages per request).
 * RMSNorm (norm_w, eps), RoPE and coding are those of cskv_compress; rope_cs
 * ([B, 32, 2] fp32, NULL = none) holds, per request, (cos, sin) at the
 * position of the row it writes this step: p + 1 - ratio (the block's first
 * token) for ratio > 1, p for ratio 1.  Rows of requests that complete
 * nothing are ignored.
 * Arithmetic: bit-exact with cskv_compress (same contract).  Up to 8 jobs
 * (e.g. the main and index-key compressors of a CSA layer and the window) in
 * one launch.  pos: device int32 [B].  Alignment: kv, gate, state_* 8 bytes;
 * ape, norm_w, rope_cs 16 bytes.  Errors: CSKV_ERR_INVALID for bad arguments;
 * a row outside the block table or the pool sets CSKV_ERR_BOUNDS on the
 * device (the row is skipped).
 * ------------------------------------------------------------------------ */
typedef struct {
  const void* kv;
  const void* gate;
  void* state_kv;
  void* state_gate;
  const float* ape;
  const float* norm_w;
  float eps;
  const float* rope_cs;
  int32_t ratio, overlap, dim, ring_rows;
  cskv_paged out;
} cskv_decode_job;
CSKV_API int32_t cskv_decode_append(const cskv_decode_job* jobs, int32_t njobs, const int32_t* pos, int32_t B,
                                    void* stream);

/* ------------------------------------------------------------------------
 * cskv_index_topk: the lightning indexer and top-k ("DeepSeek-V4 deep dive",
 * section 5.2 "What is different from V3.2's indexer"):
 *   I_{b,j} = sum_h w[b,h] * ReLU(q[b,h,:] . k_{b,j})   for j < n_b,
 *   n_b = floor(ctx_len[b] / ratio) visible entries (the query sits at
 *   position ctx_len[b]-1),
 * and topk_idx[b, :] = the min(k, n_b) entries with the largest I (ties: the
 * smaller entry index), in ascending entry order, -1 after them.
 * q_idx: bf16 [B, Hi, 128] device (post-RoPE).  w: fp32 [B, Hi] device (final
 * head weights, any scale included).  keys: 128-d index keys, format
 * FP8_E4M3_ROWSCALE_PAGESPLIT (queries are then coded e4m3 with one power-of-two
 * scale per head, the products run on the FP8 tensor cores and each key's scale
 * multiplies its weighted sum) or BF16.  ctx_len: int32 [B]
 * device, each <= max_ctx_len.  Hi in [1, 64]; k in [1, 2048].
 * topk_score: optional fp32 [B, k] (NULL to skip): the kernel's fp32 score of
 * each selected entry (-inf after the selection).
 * workspace: device, >= cskv_index_topk_workspace_size(...) bytes, 256-byte
 * aligned; its contents need no initialisation and are garbage afterwards.
 * ------------------------------------------------------------------------ */
CSKV_API size_t cskv_index_topk_workspace_size(int32_t B, int32_t max_ctx_len, int32_t ratio,
                                      int32_t Hi, int32_t k);
CSKV_API int32_t cskv_index_topk(const void* q_idx, const float* w, cskv_paged keys,
                        const int32_t* ctx_len, int32_t B, int32_t Hi, int32_t ratio,
                        int32_t k, int32_t max_ctx_len,
                        int32_t* topk_idx, float* topk_score,
                        void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * cskv_index_topk_noalloc: cskv_index_topk for callers that cannot allocate
 * device memory.  The paper has no counterpart: this is a deployment variant.
 * Same arguments, results and bits as cskv_index_topk, minus the workspace.
 * Some callers cannot call cudaMalloc: code that runs while a stream is being
 * captured into a CUDA graph (allocation is not a stream operation and may
 * synchronise the device), plugins inside hosts that own every byte of device
 * memory and expose no allocator, and latency-critical threads that must never
 * block on the driver.  They get the workspace from a fixed array inside the
 * library instead: CSKV_NOALLOC_SCRATCH_BYTES (32 MiB) of device memory that
 * every GPU which loads the library holds until the process exits.  The limit:
 * a call is accepted when cskv_index_topk_workspace_size(B, max_ctx_len, ratio,
 * Hi, k) <= CSKV_NOALLOC_SCRATCH_BYTES, i.e. about 12.1 bytes per entry of
 * B * ceil(max_ctx_len / ratio) (every request is sized at the batch's longest
 * context) plus about 38 KB per request - e.g. 8 requests at 1M tokens (ratio 4)
 * or 1 request at 11M.  Larger sizes are rejected with CSKV_ERR_INVALID before
 * anything is launched.  The array's device address is looked up in the current
 * context on every call (cudaGetSymbolAddress; it allocates nothing), so a
 * cudaDeviceReset between calls is harmless.  The first call on a device may also
 * load the library's device code there (lazy module loading): make it before any
 * stream capture.  Every call uses the same array and leaves its last contents
 * behind; each call clears what must start at zero itself, but calls whose
 * kernels overlap on the GPU (different streams, or graphs replayed
 * concurrently) race on the array and give wrong results.  The call allocates
 * nothing: no cudaMalloc, no cudaFree.
 * ------------------------------------------------------------------------ */
#define CSKV_NOALLOC_SCRATCH_BYTES (32u << 20)
CSKV_API int32_t cskv_index_topk_noalloc(const void* q_idx, const float* w, cskv_paged keys,
                                         const int32_t* ctx_len, int32_t B, int32_t Hi,
                                         int32_t ratio, int32_t k, int32_t max_ctx_len,
                                         int32_t* topk_idx, float* topk_score, void* stream);

/* ------------------------------------------------------------------------
 * cskv_sparse_decode_attn: shared-KV decode attention over the sliding window
 * and the compressed entries in one softmax with a sink ("DeepSeek-V4 deep
 * dive", section 3.1 "K = V, one head", section 3.3 partial RoPE with the
 * inverse rotation, section 3.4 Eq. 27, section 5.3 index list; section 6.1
 * for HCA).
 * For request b with query position t = ctx_len[b] - 1 and every head h:
 *   q' = q[b,h] with its last 64 dims rotated by angle(t) (q_rope_cs[b]),
 *   keys = window rows of positions max(0, t-127) .. t (ring slot pos % 128 of
 *          `swa`), then the compressed entries topk_idx[b, 0..k) (-1 skipped,
 *          duplicates kept) or, if topk_idx is NULL, every visible entry
 *          j < floor(ctx_len[b] / ratio) (HCA),
 *   z_j = (q' . c_j) * softmax_scale,
 *   o   = sum_j exp(z_j) c_j / (sum_j exp(z_j) + exp(sink[h])),
 *   out[b,h] = o with its last 64 dims rotated back by -angle(t).
 * q: bf16 [B, H, 512] device (pre-RoPE).  main_kv: 512-d entries, format FP8,
 * FP4 or BF16.  swa: device [B, 128, row_bytes(swa_fmt, 512)], swa_fmt FP8 or
 * BF16.  sink: fp32 [H] or NULL (no sink).  q_rope_cs: fp32 [B, 32, 2] (cos,
 * sin) of each query position.  out: bf16 [B, H, 512] device.  H in [1, 128].
 * Dequantised keys and values are exact in bf16; products run as tcgen05
 * bf16 MMAs with fp32 accumulation; the query is rounded to bf16 after RoPE;
 * each 128-key tile's partial output is kept as O / l in bf16 (with its fp32
 * max and sum) until the tiles are merged in fp32.
 * workspace: >= cskv_sparse_decode_attn_workspace_size(...) bytes, 256-byte
 * aligned, no initialisation needed.
 * ------------------------------------------------------------------------ */
CSKV_API size_t cskv_sparse_decode_attn_workspace_size(int32_t B, int32_t H, int32_t max_ctx_len,
                                              int32_t ratio, int32_t k);
CSKV_API int32_t cskv_sparse_decode_attn(const void* q, cskv_paged main_kv,
                                const void* swa, int32_t swa_fmt,
                                const int32_t* ctx_len, const int32_t* topk_idx, int32_t k,
                                int32_t ratio, int32_t max_ctx_len,
                                const float* sink, float softmax_scale,
                                const float* q_rope_cs, int32_t B, int32_t H,
                                void* out, void* workspace, size_t workspace_bytes,
                                void* stream);

/* ------------------------------------------------------------------------
 * cskv_sparse_prefill_attn: the same attention for many queries of a prompt
 * ("DeepSeek-V4 deep dive", section 5.3: in prefill the buffer is [all raw-token
 * keys of the prompt ; its compressed entries] and each query's index list is
 * its window positions t-127 .. t, those below 0 masked, then its selected
 * entries; section 5.2: a query sees the entries j < floor((t + 1) / ratio)).
 * Query i (of T) belongs to request req_of[i] (NULL: request i) and sits at
 * position t = pos1[i] - 1; it attends exactly as cskv_sparse_decode_attn's
 * request with ctx_len = pos1[i], except that its window rows are rows
 * max(0, t-127) .. t of its request in `window` (a paged cache of the raw rows
 * by position, FP8 or BF16, 512-d) and its compressed entries come from its
 * request's rows of main_kv.  q: bf16 [T, H, 512]; topk_idx: int32 [T, k] (each
 * query's own selection, e.g. from cskv_index_topk run with one row per query;
 * NULL: every visible entry); q_rope_cs: fp32 [T, 32, 2] at each query's
 * position; out: bf16 [T, H, 512].  max_ctx_len >= every pos1[i].  Workspace:
 * cskv_sparse_decode_attn_workspace_size(T, H, max_ctx_len, ratio, k) bytes.
 * Errors as cskv_sparse_decode_attn; a window row outside the block table or
 * the pool sets CSKV_ERR_BOUNDS on the device and is skipped.
 * ------------------------------------------------------------------------ */
CSKV_API int32_t cskv_sparse_prefill_attn(const void* q, cskv_paged main_kv, cskv_paged window,
                                          const int32_t* req_of, const int32_t* pos1,
                                          const int32_t* topk_idx, int32_t k, int32_t ratio,
                                          int32_t max_ctx_len, const float* sink, float softmax_scale,
                                          const float* q_rope_cs, int32_t T, int32_t H, void* out,
                                          void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * cskv_decode_layer: one decode step of one compressed-attention layer, from
 * host memory to host memory ("DeepSeek-V4 deep dive", section 4.1 for the
 * entries a step completes, section 5.2 for the indexer, sections 3.4 and 5.3
 * for the attention; section 6.1: an HCA layer has no indexer).  In stream
 * order, on `stream`:
 *   1. in_bytes bytes from h_in (host) to d_in (device), if in_bytes > 0;
 *   2. cskv_compress_many(jobs, njobs), if njobs > 0 (the entries whose blocks
 *      complete at this step; written before they are read below);
 *   3. cskv_index_topk(q_idx, w, keys, ctx_len, B, Hi, ratio, k, max_ctx_len,
 *      topk_idx, NULL, index_workspace, ...), if q_idx != NULL (CSA); with
 *      q_idx == NULL (HCA) the attention reads every visible entry;
 *   4. cskv_sparse_decode_attn(q, main_kv, swa, swa_fmt, ctx_len, topk_idx or
 *      NULL, k, ratio, max_ctx_len, sink, softmax_scale, q_rope_cs, B, H, out,
 *      attn_workspace, ...);
 *   5. out_bytes bytes from out (device) to h_out (host), if out_bytes > 0
 *      (at most B * H * 512 * 2, the bf16 output).
 * The device pointers of steps 2-4 may point into d_in: the copy of step 1 is
 * ordered before every kernel that reads them.  Each stage takes exactly the
 * arguments, layouts, results and bits of its own entry point above.
 * Copies: page-locked host memory (cudaHostAlloc / cudaMallocHost /
 * cudaHostRegister) is read or written by a copy kernel on the SMs through its
 * device alias, and a page-locked h_out of the whole output's size is written
 * by the attention's last kernel itself, beside `out`; any other host memory
 * goes through cudaMemcpyAsync (synchronous for pageable memory, and not
 * capturable into a CUDA graph).  Two kinds of input may also be page-locked
 * host memory outside h_in, read in place through their device alias, so that
 * their transfer is off the step's critical path: `q`, which the attention reads
 * before it waits for its selection, and a job's kv, gate, prev_kv, prev_gate and
 * rope_cs, which the compressor reads while the score kernel streams the older
 * keys (its other arrays, and every other pointer of steps 2-4, are device
 * memory).
 * Ownership: every buffer is the caller's; h_in must hold in_bytes bytes, d_in at
 * least as many, h_out out_bytes.  The call returns once everything is enqueued;
 * h_out holds the output after the stream has synchronised.  Host memory that the
 * kernels read in place (q, the jobs' per-step inputs) and h_in must stay unchanged
 * until then: a CUDA graph that captured the call reads them again at every replay.
 * Errors: the arguments of every stage are checked before anything is
 * enqueued (CSKV_ERR_INVALID / CSKV_ERR_UNSUPPORTED as the stage's own entry
 * point would return, and CSKV_ERR_INVALID for a NULL h_in / d_in / h_out with
 * a non-zero byte count or an out_bytes above the output's size); a CUDA error
 * while enqueueing returns CSKV_ERR_CUDA and leaves the later stages unqueued.
 * ------------------------------------------------------------------------ */
typedef struct {
  const cskv_compress_job* jobs; /* njobs entries (0..4); NULL when njobs == 0 */
  int32_t njobs;
  const void* q_idx;             /* bf16 [B, Hi, 128]; NULL: HCA (no indexer) */
  const float* w;                /* fp32 [B, Hi] */
  cskv_paged keys;               /* index keys (read only when q_idx != NULL) */
  int32_t Hi, k;                 /* indexer heads; entries selected (and read) per query */
  int32_t* topk_idx;             /* int32 [B, k] device, the selection (written) */
  void* index_workspace;
  size_t index_workspace_bytes;
  const void* q;                 /* bf16 [B, H, 512] device, or page-locked host memory */
  cskv_paged main_kv;
  const void* swa;               /* [B, 128, row_bytes(swa_fmt, 512)] window ring */
  int32_t swa_fmt;
  const int32_t* ctx_len;        /* int32 [B] */
  int32_t ratio, max_ctx_len;
  const float* sink;             /* fp32 [H] or NULL */
  float softmax_scale;
  const float* q_rope_cs;        /* fp32 [B, 32, 2] */
  int32_t B, H;
  void* out;                     /* bf16 [B, H, 512] device */
  void* attn_workspace;
  size_t attn_workspace_bytes;
  const void* h_in;              /* host source of step 1 */
  void* d_in;                    /* device destination of step 1 */
  size_t in_bytes;
  void* h_out;                   /* host destination of step 5 */
  size_t out_bytes;
} cskv_decode_layer_args;
CSKV_API int32_t cskv_decode_layer(const cskv_decode_layer_args* args, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* CSKV_H */
