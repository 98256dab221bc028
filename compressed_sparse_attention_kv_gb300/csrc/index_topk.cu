// Lightning indexer + top-k (cskv_index_topk).
//
// "DeepSeek-V4 deep dive", section 5.2: I_{b,j} = sum_h w_h ReLU(q_h . k_j) over
// the visible entries j < floor(ctx_len / ratio), one 128-d key shared by all
// indexer heads; the selector keeps min(k, n) entries (section 5.3).
//
// GB300 design (HBM-bound: at 1M context the keys are 34.6 MB per query):
//  1. index_prep_kernel   codes each request's queries into the image of the score
//     kernel's shared-memory query tile (FP8 keys: e4m3 with one e8m0 scale per
//     head, the scale folded into the head weight since ReLU(c x) = c ReLU(x) for
//     c > 0; FP4 keys: rotated like the keys, then e2m1 with an e8m0 scale per 32;
//     bf16: as they are), clears the request's histogram, counters, flags and queue
//     slot, and puts what the score kernel reads first (context lengths, block-table
//     rows) into L2.
//  2. index_score_kernel  persistent, one block per SM (all 512 TMEM columns),
//     warp-specialised:
//       warp 11    the scheduler: takes chunks of four tiles from the requests' work
//                  counters (the block's first chunk without an atomic, its page ids
//                  requested before the set-up barrier) and writes one record per
//                  tile - request, tile, two page ids - into an 8-record ring;
//       warps 0-1  two TMA producers on alternate records, each with its own stage
//                  ring (one TMA-issuing thread per SM cannot keep enough copies in
//                  flight): 64-row key pages by 3-D TMA (tensor map over the page
//                  pool, 128-byte swizzle; FP4: 64-byte), the pages' scales by bulk
//                  copies, all L2 evict-first;
//       warp 2     issues tcgen05 MMAs: M = 128 entries, N = heads, K = 128 (FP8:
//                  four K = 32 e4m3 x e4m3 steps, the key's single scale applied
//                  afterwards; FP4: two K = 64 block-scaled e2m1 steps with the
//                  scale factors copied into TMEM; bf16: eight K = 16 steps) into
//                  one fp32 TMEM accumulator, up to eight in flight;
//       warps 3-10 two epilogue groups on alternate tiles: tcgen05.ld (one TMEM
//                  lane = one entry), ReLU and the head weights, the heads summed
//                  inside one thread, times the key's scale, the score written
//                  (FP4: rounded to bf16), its order-preserving key binned into the
//                  group's 4,096-bin shared histogram (with 256 coarse bins of 16)
//                  and per 32-entry segment the largest key, its lane and the bin
//                  of the runner-up kept.
//     Streaming (batches of at most 64 requests of at most 262,144 entries): a group
//     that leaves a request adds its tile count to the request's counter; the count
//     that completes it queues the request, and a block done with its stream takes it
//     from the queue: the threshold bin T (the bin holding the k-th score), the
//     candidates (a segment with one key in a bin >= T gives it from the metadata,
//     one with more has its scores read), the exact cut among the keys of bin T
//     (ties -> smaller index), the k entries in entry order and the request's ready
//     flag, on which the attention's tiles of that request start.
//     LARGE (more or longer requests; a cooperative launch): behind one bounded grid
//     barrier every request's tiles are split over a run of blocks: each finds T,
//     reads again only the segments whose largest key reaches T and writes the
//     entries in bins >= T as 64-bit (score, ~index) keys in entry order; the block
//     that finishes a request's last slice radix-selects the cut among the keys of
//     bin T and writes the k entries in entry order, so the output needs no sort.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>

#include "codec.cuh"
#include "internal.h"

namespace cskv {

namespace {

constexpr int kHistBits = 12;
constexpr int kHistBins = 1 << kHistBits;
constexpr int kCoarseBins = 256;                      // sums of 16 fine bins (the top 8 key bits)
constexpr int kHistStride = kHistBins + kCoarseBins;  // per request in the workspace
constexpr int kTileRows = 128;
constexpr int kProducers = 2;        // TMA-issuing warps, each with its own stage ring
constexpr int kGroups = 2;           // epilogue groups of 4 warps (one per TMEM lane quarter)
constexpr int kStagesFp8 = 4;        // per producer, 16 KiB stages
constexpr int kStagesBf16 = 2;       // per producer, 32 KiB stages
constexpr int kStagesFp4 = 8;        // per producer, 9 KiB stages
constexpr int kStagesMax = 8;
constexpr int kAccsMax = 8;          // TMEM accumulators in flight (8 x 64 columns)
constexpr int kScaleSlots = 16;      // ring of per-tile scale rows (2 pages x 64 fp32)
constexpr int kRecSlots = 8;         // tile records in flight from the scheduler to the producers (two chunks:
                                     // a deeper lookahead commits work to a block too early)
constexpr int kChunkTiles = 4;       // tiles per grab from a request's work counter
constexpr int kWarpMma = kProducers;
constexpr int kWarpEpi = kProducers + 1;
constexpr int kWarpSched = kWarpEpi + 4 * kGroups;
constexpr int kScoreThreads = 32 * (kProducers + 1 + 4 * kGroups + 1);   // 384
// three groups (15 warps) put four warps on a scheduler partition: 128 registers each
constexpr int kLaunchBound = kGroups >= 3 ? 512 : kScoreThreads;
constexpr int kCandCap = 4096;       // per-block staging of threshold-bin candidates
constexpr int kQImageFp8 = 8192;     // e4m3 [64 rows][128 B]
constexpr int kQImageBf16 = 16384;   // bf16 [2 chunks][64 rows][128 B]
constexpr int kQImageFp4 = 4608;     // e2m1 [64 rows][64 B], then the heads' scale factors [32][16 B]

// Key formats of the score kernel (its template parameter KF) and what they size.
constexpr int kKfBf16 = 0, kKfFp8 = 1, kKfFp4 = 2;
template <int KF>
struct KeyFmt {
  // one stage holds a tile of 128 keys: FP4 = 8 KiB of codes, their 512 scale bytes and
  // the same bytes in the scale-factor copy's layout
  static constexpr int kStageBytes = KF == kKfFp8 ? kTileRows * 128 : KF == kKfBf16 ? kTileRows * 256 : kTileRows * 64 + 1024;
  static constexpr int kStages = KF == kKfFp8 ? kStagesFp8 : KF == kKfBf16 ? kStagesBf16 : kStagesFp4;
  static constexpr int kQImage = KF == kKfFp8 ? kQImageFp8 : KF == kKfBf16 ? kQImageBf16 : kQImageFp4;
  static constexpr int kQBuf = 2 * kQImage > 16384 ? 2 * kQImage : 16384;   // the selection reuses 16 KiB of it
  // FP4: six accumulators (384 columns), their keys' scale factors (4 columns each) and
  // the two query buffers' (4 each) in one 512-column allocation
  static constexpr int kAccs = KF == kKfFp4 ? 6 : 8;
};
constexpr int kSfaCol = 384;         // FP4: first TMEM column of the keys' scale factors
constexpr int kQSlot = 16384;        // per request in the workspace

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

constexpr int kMaxGrid = 1024;       // bound of the per-block counters' table
constexpr int kSeg = 32;             // entries per segment (one epilogue warp's rows of a tile)
constexpr int kSelSegs = 8192;       // segments per selection pass (262,144 entries)
constexpr int kReqCache = 64;        // requests whose visible count is kept in shared memory
constexpr int kFastN = 2048;         // LARGE: requests of at most this many entries are selected by one warp
constexpr int kScratch16 = kSelSegs + 64 - kScaleSlots * kTileRows * 2;   // u16 words after the scale ring

struct WsLayout {
  size_t scores, segmax, segmeta, cand, qimg, wq, hist, ctr, slc, gbar, done, ready, fresh, queue, total;
  int n_pad;
};

__host__ __device__ inline WsLayout ws_layout(int B, int n_max, int k) {
  WsLayout L;
  L.n_pad = (n_max + kTileRows - 1) / kTileRows * kTileRows;
  if (L.n_pad == 0) L.n_pad = kTileRows;
  size_t o = 0;
  L.scores = o; o = align256(o + size_t(B) * L.n_pad * 4);
  L.segmax = o; o = align256(o + size_t(B) * (L.n_pad / kSeg) * 4);
  // streaming mode: per segment (max key << 32) | (bin of the second largest key << 8) | lane of the max
  L.segmeta = o; o = align256(o + size_t(B) * (L.n_pad / kSeg) * 8);
  L.cand = o;   o = align256(o + size_t(B) * L.n_pad * 8);
  L.qimg = o;   o = align256(o + size_t(B) * kQSlot);
  L.wq = o;     o = align256(o + size_t(B) * 64 * 4);
  L.hist = o;   o = align256(o + size_t(B) * kHistStride * 4);
  L.ctr = o;    o = align256(o + size_t(B) * 4 * 4);
  L.slc = o;    o = align256(o + size_t(B) * kMaxGrid * 4);
  L.gbar = o;   o = align256(o + 16);
  L.done = o;   o = align256(o + size_t(B) * 4);   // per request: tiles scored and flushed
  L.ready = o;  o = align256(o + size_t(B) * 4);   // per request: 1 once its selection is written
  L.fresh = o;  o = align256(o + size_t(B) * 4);   // per request: first entry the kernel before may write
  // selection queue: [0] slots claimed, [1] slots filled, then B requests in completion order (-1: not yet)
  L.queue = o;  o = align256(o + size_t(B + 2) * 4);
  L.total = o;
  return L;
}

// order-preserving map of an fp32 score to uint32 (larger score -> larger key)
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float from_order_key(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

struct IndexArgs {
  const uint8_t* q;          // bf16 [B, Hi, 128]
  const float* w;            // [B, Hi]
  cskv_paged keys;
  const int32_t* ctx_len;
  int B, Hi, N, ratio, k, n_max;
  int kfmt;                  // key format: 0 bf16, 1 page-split FP8, 2 page-split rotated FP4
  int grid;                  // blocks of the score kernel
  int32_t* topk_idx;
  float* topk_score;
  uint8_t* ws;
  WsLayout L;
  unsigned long long spin;
  // Streaming mode (batches of at most kReqCache requests): no grid barrier; the block
  // that completes a request's last tile selects it and raises ready[b].  With
  // wait_fresh, the kernel before the score kernel in the stream (the compressor of a
  // fused decode step) may still be writing index keys: tiles holding entries at or
  // after fresh[b] are read only after it has completed; nothing else waits for it.
  int wait_fresh;
  int fused;                       // the prep waits for the kernel before it first (its queries may come from it)
  int nfresh;                      // jobs that write this step's index keys (prep input)
  const int32_t* fresh_req[4];     // [S] request of each sequence of the job
  const int32_t* fresh_first[4];   // [S] first entry the sequence writes
  int fresh_S[4];
};

// Phase-1 work distribution: block blk starts at its home request blk * B / G and
// takes chunk r of it without an atomic (r = its rank among the blocks of that
// home); the request's counter starts after those chunks.
__device__ __forceinline__ int home_request(int blk, int B, int G) {
  return static_cast<int>((static_cast<long long>(blk) * B) / G);
}
__device__ __forceinline__ int first_home_block(int b, int B, int G) {   // smallest blk with home b
  return static_cast<int>((static_cast<long long>(b) * G + B - 1) / B);
}

__device__ __forceinline__ int visible(const IndexArgs& a, int b) {
  long long c = a.ctx_len[b];
  long long n = c / a.ratio;
  if (c < 0 || n > a.n_max) {
    set_err(CSKV_ERR_BOUNDS);
    n = c < 0 ? 0 : a.n_max;
  }
  return static_cast<int>(n);
}

// The page ids of tiles t0 .. t0 + kChunkTiles - 1 of request b (n_b visible entries),
// two per tile; -2: no page (past the request's entries, or b < 0), -3: outside the
// block table.  All loads are issued before any is used.
template <int kChunk>
__device__ __forceinline__ void chunk_page_ids(const IndexArgs& a, int b, int n_b, int t0, int (&ids)[2 * kChunk]) {
  const int32_t* bt = a.keys.block_table + static_cast<long long>(b < 0 ? 0 : b) * a.keys.max_pages;
#pragma unroll
  for (int u = 0; u < 2 * kChunk; ++u) {
    const long long lp = static_cast<long long>(t0) * 2 + u;
    ids[u] = (b < 0 || lp * kPageRows >= n_b) ? -2 : (lp >= a.keys.max_pages ? -3 : bt[lp]);
  }
}

// ---------------------------------------------------------------------------
// 1. prep: query image, folded head weights, histogram / counters / barrier cleared
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) index_prep_kernel(const IndexArgs a) {
  const int b = blockIdx.x;
  uint8_t* img = a.ws + a.L.qimg + size_t(b) * kQSlot;
  float* wq = reinterpret_cast<float*>(a.ws + a.L.wq) + b * 64;
  uint32_t* hist = reinterpret_cast<uint32_t*>(a.ws + a.L.hist) + size_t(b) * kHistStride;
  uint32_t* ctr = reinterpret_cast<uint32_t*>(a.ws + a.L.ctr) + b * 4;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // in a fused decode step the queries may come from the kernel before (a staging copy)
  if (a.fused) grid_dep_wait();
  // the score kernel (a programmatic dependent of this one) may start its set-up now
  grid_dep_launch();
  // what that set-up and its first chunks read, into L2 (no load waits on it here): the
  // requests' context lengths and request b's block-table row
  if (threadIdx.x == 0) prefetch_l2(a.ctx_len + b);
  if (a.keys.block_table != nullptr) {
    const int pages = min(a.keys.max_pages, static_cast<int>((a.n_max + kPageRows - 1) / kPageRows));
    const int32_t* row = a.keys.block_table + static_cast<long long>(b) * a.keys.max_pages;
    for (int x = threadIdx.x * 32; x < pages; x += blockDim.x * 32) prefetch_l2(row + x);
  }
  // warp w owns heads w, w+8, ... (N <= 64); lane l holds dims 4l .. 4l+3.  All loads first.
  uint2 raw[8];
  float wv[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int h = warp + 8 * i;
    const bool real = h < a.Hi;
    raw[i] = real ? *reinterpret_cast<const uint2*>(a.q + (size_t(b) * a.Hi + h) * 256 + lane * 8)
                  : make_uint2(0u, 0u);
    wv[i] = real ? a.w[size_t(b) * a.Hi + h] : 0.f;
  }
  if (a.wait_fresh && warp == 0) {
    // the first index key of request b that this step's compressor writes (none:
    // INT_MAX); its loads overlap the queries'.  (A fused step waited above for the
    // kernels before it, so the workspace word is free.)
    int fr = 0x7FFFFFFF;
    for (int j = 0; j < a.nfresh; ++j)
      for (int q = lane; q < a.fresh_S[j]; q += 32)
        if (a.fresh_req[j][q] == b) fr = min(fr, a.fresh_first[j][q]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) fr = min(fr, __shfl_xor_sync(0xFFFFFFFFu, fr, o));
    if (lane == 0) reinterpret_cast<int32_t*>(a.ws + a.L.fresh)[b] = fr;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int h = warp + 8 * i;
    if (h >= a.N) break;
    if (a.kfmt == kKfFp4) {
      // rotated like the keys, then e2m1 with an e8m0 scale per 32 (8 lanes); row h of the
      // 64-byte swizzled image (16-byte chunk c of row h at chunk c ^ ((h >> 1) & 3)), the
      // scale bytes in the scale-factor copy's layout after the image (row h % 32, word h / 32)
      float y[4] = {bf16lo(raw[i].x), bf16hi(raw[i].x), bf16lo(raw[i].y), bf16hi(raw[i].y)};
      hadamard128_x4(y, lane);
      float am = fmaxf(fmaxf(fabsf(y[0]), fabsf(y[1])), fmaxf(fabsf(y[2]), fabsf(y[3])));
      am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
      am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 2));
      am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 4));
      const int e = e8m0_exponent_fp4(am);
      const uint32_t codes = e2m1x4_scaled(y, e);
      *reinterpret_cast<uint16_t*>(img + h * 64 + ((((lane >> 3) ^ ((h >> 1) & 3))) << 4) + ((2 * lane) & 15)) =
          static_cast<uint16_t>(codes);
      if ((lane & 7) == 0) img[4096 + 16 * (h & 31) + 4 * (h >> 5) + (lane >> 3)] = static_cast<uint8_t>(e + 127);
      if (lane == 0) wq[h] = wv[i];
    } else if (a.kfmt == kKfFp8) {
      const float4 v = make_float4(bf16lo(raw[i].x), bf16hi(raw[i].x), bf16lo(raw[i].y), bf16hi(raw[i].y));
      float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
      const int e = e8m0_exponent(amax);
      const float inv = exp2i(-e);
      const uint32_t codes = e4m3x2(__fmul_rn(v.x, inv), __fmul_rn(v.y, inv)) |
                             (e4m3x2(__fmul_rn(v.z, inv), __fmul_rn(v.w, inv)) << 16);
      // row h, byte 4*lane of 128: chunk lane/4, byte (lane%4)*4 inside it
      *reinterpret_cast<uint32_t*>(img + sw128_offset(h, lane >> 2) + (lane & 3) * 4) = codes;
      if (lane == 0) wq[h] = __fmul_rn(wv[i], exp2i(e));
    } else {
      // bf16: dims 0..63 in chunk 0, 64..127 in chunk 1; lane l -> chunk l/16, byte (l%16)*8
      uint8_t* base = img + (lane >> 4) * (a.N * 128);
      const int byte = (lane & 15) * 8;
      *reinterpret_cast<uint2*>(base + sw128_offset(h, byte >> 4) + (byte & 15)) = raw[i];
      if (lane == 0) wq[h] = wv[i];
    }
  }
  // This kernel may run beside the kernel before it in the stream (it is launched as
  // a programmatic dependent: that kernel writes the keys this indexer reads, not its
  // queries).  The workspace words that an earlier indexer launch on the same
  // workspace may still be using are cleared only after the wait, and finishing
  // after the wait makes the next kernel see the previous one complete.
  grid_dep_wait();
  for (int i = threadIdx.x; i < kHistStride; i += blockDim.x) hist[i] = 0;
  if (threadIdx.x < 4)
    ctr[threadIdx.x] = threadIdx.x == 0 ? static_cast<uint32_t>(first_home_block(b + 1, a.B, a.grid) -
                                                             first_home_block(b, a.B, a.grid)) * kChunkTiles
                                        : 0u;
  if (b == 0 && threadIdx.x < 2) reinterpret_cast<uint32_t*>(a.ws + a.L.gbar)[threadIdx.x] = 0;
  if (threadIdx.x == 0) {
    reinterpret_cast<uint32_t*>(a.ws + a.L.done)[b] = 0;
    reinterpret_cast<uint32_t*>(a.ws + a.L.ready)[b] = 0;
    reinterpret_cast<int32_t*>(a.ws + a.L.queue)[2 + b] = -1;
    if (b == 0) reinterpret_cast<uint32_t*>(a.ws + a.L.queue)[0] = reinterpret_cast<uint32_t*>(a.ws + a.L.queue)[1] = 0;
  }
}

// ---------------------------------------------------------------------------
// 2. score kernel (+ fused selection)
// ---------------------------------------------------------------------------
// One request of this block's selection work: tiles [lo, hi) of request b, whose run
// of blocks starts at fb and has nbk blocks of `per` tiles.
struct WorkItem {
  long long lo, hi, per;
  int b, fb, nbk, pad;
};
constexpr int kWorkItems = 16;

struct ScoreSmem {
  uint64_t full[kProducers][kStagesMax], empty[kProducers][kStagesMax];
  uint64_t accfull[kAccsMax], accempty[kAccsMax];
  uint64_t qfull[2], qempty[2];
  uint64_t sfull[kScaleSlots], sempty[kScaleSlots];
  uint64_t rfull[kRecSlots], rempty[kRecSlots];     // tile records from the scheduler
  uint64_t drain;
  uint64_t hbar[kGroups];          // an epilogue group's warps meet here at a request switch
  int4 rec[kRecSlots];             // (request, tile, page id, page id) of local tile i at i % kRecSlots; request -1 = the end
  int2 tinfo[kScaleSlots];         // (request, tile) of each tile in flight; request -1 = the end
  uint32_t tmem_base;
  volatile int abort;
  int smask[kScaleSlots];          // per tile: bit p = page p of the tile was loaded
  __align__(16) float wq[kGroups][64];   // folded head weights of each group's current request
  // selection phases
  uint32_t cnt[2];
  uint32_t base[2];
  uint32_t nlist;
  int nbv[kReqCache];              // visible entries of the first kReqCache requests
  uint32_t wcnt[16];               // streaming-mode selection: per-warp selected counts
  uint32_t d256[256];              // 8-bit digit histogram of the cut
  int qreq;                        // streaming mode: the request this block selects next (-1: none)
  int fresh[kReqCache];            // streaming mode: first entry of each request the compressor may write
  WorkItem work[kWorkItems];       // this block's selection work, found before the scores
  int nwork;                       // -1: more than kWorkItems (found again after the barrier)
  int T, cbin;
  uint32_t above, inT;
  uint32_t need, done, out;
  int last;
  unsigned long long prefix, mask;
  uint32_t part[256];
  uint32_t dh[256];
};

__device__ __forceinline__ bool role_wait(ScoreSmem* sm, uint64_t* bar, uint32_t parity,
                                          unsigned long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (sm->abort) return false;
    if (clock64() - t0 > limit) {
      set_err(CSKV_ERR_TIMEOUT);
      sm->abort = 1;
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// All blocks of the (cooperatively launched, hence co-resident) grid meet here.
// Bounded: a wait that runs out sets CSKV_ERR_TIMEOUT and the block carries on
// with abort set, so nothing hangs.
__device__ __forceinline__ void grid_barrier(ScoreSmem* sm, uint32_t* counter, uint32_t target, unsigned long long limit) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(counter, 1u);
    const unsigned long long t0 = clock64();
    while (ld_acquire(counter) < target) {
      if (clock64() - t0 > limit) {
        set_err(CSKV_ERR_TIMEOUT);
        sm->abort = 1;
        break;
      }
      __nanosleep(64);
    }
    __threadfence();
  }
  __syncthreads();
}

// T = the largest histogram bin with (entries in bins >= T) >= k; above = entries in
// bins > T; inT = entries in bin T; T = -1 if the histogram holds fewer than k
// entries.  Whole block (warp 0 works): the 256 coarse bins (sums of 16 fine bins),
// then the 16 fine bins of the coarse bin that crosses k, read from s_fine: the
// request's 4,096 fine bins, whose cp.async copies the caller issued beside the
// coarse loads (this function waits for every copy the thread has in flight).
// newest_pending: the caller's copies form two groups, the fine bins first; only that
// group is awaited (the newer one lands meanwhile).  Otherwise every copy is awaited.
__device__ __forceinline__ void threshold_bin(ScoreSmem* sm, const uint32_t* gh, int k, const uint32_t* s_fine,
                                              bool newest_pending = false) {
  const int lane = threadIdx.x;
  if (lane < 32) {
    // lane l owns coarse bins 255-8l .. 248-8l (from the top): two 16-byte loads
    const uint4 c0 = __ldcg(reinterpret_cast<const uint4*>(gh + kHistBins + 248 - 8 * lane));
    const uint4 c1 = __ldcg(reinterpret_cast<const uint4*>(gh + kHistBins + 252 - 8 * lane));
    const uint32_t loc[8] = {c1.w, c1.z, c1.y, c1.x, c0.w, c0.z, c0.y, c0.x};   // top first
    uint32_t sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) sum += loc[i];
    uint32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t x = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += x;
    }
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, incl >= static_cast<uint32_t>(k));
    if (hit == 0) {
      if (lane == 0) { sm->T = -1; sm->above = 0; sm->inT = 0; sm->cbin = -1; }
    } else if (lane == __ffs(hit) - 1) {
      uint32_t acc = incl - sum;
      int u = 255 - 8 * lane - 7;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (acc + loc[i] >= static_cast<uint32_t>(k)) { u = 255 - 8 * lane - i; break; }
        acc += loc[i];
      }
      sm->cbin = u;   // the coarse bin that crosses k
      sm->above = acc;
    }
  }
  if (newest_pending) cp_async_wait_prior1();
  else cp_async_wait_all();
  __syncthreads();
  if (threadIdx.x < 32 && sm->cbin >= 0) {
    // the 16 fine bins of coarse bin u, lane l = fine bin 15 - l (from the top): the
    // first whose running count reaches k is T
    const int u = sm->cbin;
    const uint32_t acc0 = sm->above;
    const uint32_t f = lane < 16 ? s_fine[u * 16 + 15 - lane] : 0u;
    uint32_t incl = f;
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) {
      const uint32_t x = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += x;
    }
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, lane < 16 && acc0 + incl >= static_cast<uint32_t>(k));
    if (hit != 0) {
      if (lane == __ffs(hit) - 1) {
        sm->T = u * 16 + 15 - lane;
        sm->above = acc0 + incl - f;
        sm->inT = f;
      }
    } else if (lane == 15) {   // inconsistent tables (only after an earlier error)
      sm->T = u * 16;
      sm->above = acc0 + incl;
      sm->inT = s_fine[u * 16];
    }
  }
  __syncthreads();
}

// Exclusive scan, in place, of n 16-bit counters in shared memory (whole block;
// the sums stay below 65,536).
__device__ __forceinline__ void block_exclusive_scan16(ScoreSmem* sm, uint16_t* x, int n) {
  const int per = (n + kScoreThreads - 1) / kScoreThreads;
  const int lo = min(n, static_cast<int>(threadIdx.x) * per), hi = min(n, lo + per);
  uint32_t sum = 0;
#pragma unroll 1
  for (int i = lo; i < hi; ++i) sum += x[i];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) sm->part[warp] = incl;
  __syncthreads();
  uint32_t run = incl - sum;
#pragma unroll 1
  for (int w = 0; w < warp; ++w) run += sm->part[w];
#pragma unroll 1
  for (int i = lo; i < hi; ++i) {
    const uint32_t v = x[i];
    x[i] = static_cast<uint16_t>(run);
    run += v;
  }
  __syncthreads();
}

// The selection splits every request's tiles over a run of consecutive blocks, in
// proportion to its share of all tiles (a request too small for a block of its own
// shares block fb with its neighbours), so that few blocks work on two requests.
// For request b, whose tiles are [C, C + tb) of the total: whether block blk holds
// tiles [lo, hi) of it; the run's first block fb, its length nbk and tiles per block.
// An empty request belongs to block fb, so that its output is still written.
__device__ __forceinline__ bool block_range(int blk, int G, long long C, long long tb, long long total,
                                            long long& lo, long long& hi, int& fb, int& nbk,
                                            long long& per) {
  // 32-bit arithmetic while (C + tb) * G fits (every realistic batch), 64-bit beyond
  if (total * G < (1ll << 32)) {
    const uint32_t t32 = static_cast<uint32_t>(total), g32 = static_cast<uint32_t>(G);
    const uint32_t c32 = static_cast<uint32_t>(C), b32 = static_cast<uint32_t>(tb);
    const uint32_t f = t32 ? min(g32 - 1, c32 * g32 / t32) : 0u;
    fb = static_cast<int>(f);
    if (b32 == 0) {   // an empty request: its run is block fb alone, with no tiles
      nbk = 1;
      per = 1;
      lo = hi = 0;
      return blk == fb;
    }
    uint32_t e = (c32 + b32) * g32 / t32;
    if (e <= f) e = f + 1;
    const uint32_t p = (b32 + (e - f) - 1) / (e - f);
    per = p;
    nbk = static_cast<int>((b32 + p - 1) / p);
    if (blk < fb || blk >= fb + nbk) return false;
    lo = static_cast<long long>(static_cast<uint32_t>(blk - fb) * p);
    hi = min(tb, lo + p);
    return true;
  }
  fb = static_cast<int>(min(static_cast<long long>(G - 1), C * G / total));
  if (tb <= 0) {
    nbk = 1;
    per = 1;
    lo = hi = 0;
    return blk == fb;
  }
  int eb = static_cast<int>(((C + tb) * G) / total);
  if (eb <= fb) eb = fb + 1;
  per = (tb + (eb - fb) - 1) / (eb - fb);
  nbk = static_cast<int>((tb + per - 1) / per);
  if (blk < fb || blk >= fb + nbk) return false;
  lo = (blk - fb) * per;
  hi = min(tb, lo + per);
  return true;
}

// The indices q in [0, n) with pred(q), in increasing order, into list (whole
// block; pred is evaluated twice and must not change in between).  Returns the count.
template <class Pred>
__device__ uint32_t ordered_list(ScoreSmem* sm, int n, Pred pred, uint16_t* list) {
  const int per = (n + kScoreThreads - 1) / kScoreThreads;
  const int lo = min(n, static_cast<int>(threadIdx.x) * per), hi = min(n, lo + per);
  uint32_t cnt = 0;
#pragma unroll 1
  for (int q = lo; q < hi; ++q) cnt += pred(q) ? 1u : 0u;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) sm->part[warp] = incl;
  __syncthreads();
  uint32_t pos = incl - cnt, tot = 0;
#pragma unroll 1
  for (int w = 0; w < kScoreThreads / 32; ++w) {
    const uint32_t x = sm->part[w];
    if (w < warp) pos += x;
    tot += x;
  }
#pragma unroll 1
  for (int q = lo; q < hi; ++q)
    if (pred(q)) list[pos++] = static_cast<uint16_t>(q);
  __syncthreads();
  return tot;
}

// Exclusive scan of one 32-bit value per thread over the whole block; tot = the sum.
__device__ __forceinline__ uint32_t block_scan_excl(ScoreSmem* sm, uint32_t v, uint32_t& tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t x = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) sm->part[warp] = incl;
  __syncthreads();
  uint32_t pos = incl - v;
  tot = 0;
#pragma unroll 1
  for (int w = 0; w < kScoreThreads / 32; ++w) {
    const uint32_t x = sm->part[w];
    if (w < warp) pos += x;
    tot += x;
  }
  __syncthreads();
  return pos;
}

// The score kernel's shared memory, 1024-byte aligned, derived from the extern array by
// pointer arithmetic so that every access stays a shared-memory access (an integer
// round trip would make them generic).  The selection, which runs out of line, carves
// the same layout from the same array.
struct ScoreCarve {
  uint8_t* stages;     // kProducers x kStages stage tiles
  uint8_t* qbuf;       // 2 query images
  uint32_t* hist;      // kGroups x 4,096 bins
  float* sring;        // kScaleSlots x 128 fp32 key scales
  uint16_t* scratch;   // kScratch16
  ScoreSmem* sm;
};
template <int KF>
__device__ __forceinline__ ScoreCarve score_carve() {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  using F = KeyFmt<KF>;
  ScoreCarve c;
  c.stages = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  c.qbuf = c.stages + kProducers * F::kStages * F::kStageBytes;
  c.hist = reinterpret_cast<uint32_t*>(c.qbuf + F::kQBuf);
  c.sring = reinterpret_cast<float*>(c.hist + kGroups * kHistBins);
  c.scratch = reinterpret_cast<uint16_t*>(c.sring + kScaleSlots * kTileRows);
  c.sm = reinterpret_cast<ScoreSmem*>(c.scratch + kScratch16);
  return c;
}

__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_s32(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Appends request b to the selection queue (its scores, bins and metadata are complete
// and were acquired by this thread).
__device__ __forceinline__ void queue_push(const IndexArgs& a, int b) {
  uint32_t* qctl = reinterpret_cast<uint32_t*>(a.ws + a.L.queue);
  const uint32_t slot = atomicAdd(qctl + 1, 1u);
  if (slot < static_cast<uint32_t>(a.B)) st_release(reinterpret_cast<uint32_t*>(qctl + 2 + slot), static_cast<uint32_t>(b));
}

constexpr int kSelCand = 8192;    // candidates kept in shared memory (64 KiB of the stage ring)
constexpr int kHitRound = 512;    // general path: hit segments whose scores are copied in at once (64 KiB)
constexpr int kMetaSegs = 8192;   // fast path: segments whose metadata fits in shared memory (64 KiB)
constexpr int kMulti = 256;       // fast path: segments with two or more entries at the threshold (32 KiB)

// Exclusive prefix sums, in place, of n <= 1024 counters (whole block; warp 0 works,
// each lane a contiguous run of up to 32); returns the total.
template <class C>
__device__ __forceinline__ uint32_t scan_rows(ScoreSmem* sm, C* x, int n) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int per = (n + 31) / 32;
    const int lo = min(n, lane * per), hi = min(n, lo + per);
    uint32_t sum = 0;
#pragma unroll 1
    for (int i = lo; i < hi; ++i) sum += x[i];
    uint32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    uint32_t run = incl - sum;
#pragma unroll 1
    for (int i = lo; i < hi; ++i) {
      const uint32_t v = x[i];
      x[i] = static_cast<C>(run);
      run += v;
    }
    if (lane == 31) sm->cnt[0] = incl;
  }
  __syncthreads();
  return sm->cnt[0];
}

// The cut among the candidates (each a 64-bit key: order key << 32 | ~entry, so that
// larger keys are larger scores and, on a tie, smaller entries) and the output, in entry
// order (the candidates are in entry order): `above` candidates lie in bins above T and
// are all taken; among those of bin T the need-th largest key is found by 12-bit radix
// digits (bits 51-40, 39-28, 27-16, 15-4, then 3-0); selected <=> (key & mask) >= prefix.
// Every pass over an array goes by rows of 32 (a warp per row, a lane per element), so
// the shared-memory accesses are conflict-free.
__device__ __forceinline__ void cut_and_write(const IndexArgs& a, ScoreSmem* sm, const unsigned long long* cand, uint32_t nkt,
                              int T, uint32_t above, uint32_t* dh, uint32_t* rows, int32_t* out_idx, float* out_sc) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int nwarps = kScoreThreads / 32;
  const uint32_t lt_mask = (1u << lane) - 1u;
  if (threadIdx.x == 0) {
    sm->need = min(static_cast<uint32_t>(a.k) - above, nkt > above ? nkt - above : 0u);
    sm->done = 0;
    sm->mask = ~0ull << 52;
    sm->prefix = static_cast<unsigned long long>(T) << 52;
  }
  __syncthreads();
#pragma unroll 1
  for (int shift = 40; shift >= 0; shift = shift >= 12 ? shift - 12 : (shift > 0 ? 0 : -1)) {
    if (sm->done || sm->need == 0) break;
    const int width = shift >= 4 ? 12 : 4;
    const int nd = 1 << width;
    const unsigned long long dmask = static_cast<unsigned long long>(nd - 1) << shift;
#pragma unroll 1
    for (int x = threadIdx.x; x < nd; x += blockDim.x) dh[x] = 0;
    __syncthreads();
    const unsigned long long pm = sm->mask, pp = sm->prefix;
#pragma unroll 1
    for (uint32_t x = threadIdx.x; x < nkt; x += blockDim.x) {
      const unsigned long long key = cand[x];
      if ((key & pm) == pp) atomicAdd(&dh[(key & dmask) >> shift], 1u);
    }
    __syncthreads();
    // digit rows of 32 from the top: row i holds digits nd-1-32i .. nd-32-32i
    const int nrow = (nd + 31) / 32;
#pragma unroll 1
    for (int r = warp; r < nrow; r += nwarps) {
      const int d = nd - 1 - (32 * r + lane);
      const uint32_t v = d >= 0 ? dh[d] : 0u;
      const uint32_t tot = __reduce_add_sync(0xFFFFFFFFu, v);
      if (lane == 0) rows[r] = tot;
    }
    __syncthreads();
    if (warp == 0) {
      // the row that holds the need-th key (from the top), then the digit in it
      const uint32_t need = sm->need;
      uint32_t acc = 0;
      int rr = nrow - 1;
#pragma unroll 1
      for (int r0 = 0; r0 < nrow; r0 += 32) {
        const uint32_t v = r0 + lane < nrow ? rows[r0 + lane] : 0u;
        uint32_t incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += y;
        }
        const unsigned hit = __ballot_sync(0xFFFFFFFFu, acc + incl >= need);
        if (hit) {
          const int l = __ffs(hit) - 1;
          rr = r0 + l;
          acc += __shfl_sync(0xFFFFFFFFu, incl - v, l);
          break;
        }
        acc += __shfl_sync(0xFFFFFFFFu, incl, 31);
      }
      const int d = nd - 1 - (32 * rr + lane);
      const uint32_t v = d >= 0 ? dh[d] : 0u;
      uint32_t incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned hit = __ballot_sync(0xFFFFFFFFu, acc + incl >= need);
      const int l = hit ? __ffs(hit) - 1 : 31;
      const uint32_t before = acc + __shfl_sync(0xFFFFFFFFu, incl - v, l);
      const uint32_t dv = __shfl_sync(0xFFFFFFFFu, v, l);
      if (lane == 0) {
        const int dd = nd - 1 - (32 * rr + l);
        sm->need = need - before;
        sm->prefix = pp | (static_cast<unsigned long long>(dd) << shift);
        sm->mask = pm | dmask;
        if (dv == need - before) sm->done = 1;
      }
    }
    __syncthreads();
    if (shift == 0) break;
  }
  // the output, in entry order: selected candidates counted per row of 32, rows scanned
  // (in chunks of 1,024 rows)
  const unsigned long long pm = sm->mask, pp = sm->prefix;
  uint32_t nsel = 0;
#pragma unroll 1
  for (uint32_t c0 = 0; c0 < nkt; c0 += 32768u) {
    const uint32_t cn = min(nkt - c0, 32768u);
    const int nrow = static_cast<int>((cn + 31) / 32);
#pragma unroll 1
    for (int r = warp; r < nrow; r += nwarps) {
      const uint32_t x = c0 + 32u * r + lane;
      const bool sel = x < nkt && (cand[x] & pm) >= pp;
      const unsigned m = __ballot_sync(0xFFFFFFFFu, sel);
      if (lane == 0) rows[r] = static_cast<uint32_t>(__popc(m));
    }
    __syncthreads();
    const uint32_t tot = scan_rows(sm, rows, nrow);
#pragma unroll 1
    for (int r = warp; r < nrow; r += nwarps) {
      const uint32_t x = c0 + 32u * r + lane;
      const unsigned long long key = x < nkt ? cand[x] : 0ull;
      const bool sel = x < nkt && (key & pm) >= pp;
      const unsigned m = __ballot_sync(0xFFFFFFFFu, sel);
      const uint32_t pos = nsel + rows[r] + __popc(m & lt_mask);
      if (sel && pos < static_cast<uint32_t>(a.k)) {
        out_idx[pos] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(key));
        if (out_sc) out_sc[pos] = from_order_key(static_cast<uint32_t>(key >> 32));
      }
    }
    nsel += tot;
    __syncthreads();
  }
  // fewer than k selected (only after an error): -1 after them
#pragma unroll 1
  for (uint32_t j = min(nsel, static_cast<uint32_t>(a.k)) + threadIdx.x; j < static_cast<uint32_t>(a.k);
       j += blockDim.x) {
    out_idx[j] = -1;
    if (out_sc) out_sc[j] = -INFINITY;
  }
}

// Streaming mode (batches of at most kReqCache requests; no grid barrier).  This block
// selects every request whose last tile it scored - all of that request's tiles are
// scored and their bins flushed - then the requests without entries that fall to it
// (b % gridDim.x), and raises ready[b] after each.  For request b:
//  - T, the histogram bin holding the k-th score, with `above` entries in bins > T and
//    inT in bin T (the request's 4,096 fine and 256 coarse bins in the workspace);
//  - the candidates, every entry in a bin >= T, in entry order, as 64-bit keys.  Fast
//    path (the usual case): the segment metadata the epilogue kept (each 32-entry
//    segment's largest key, its lane, and the bin of the second largest key) is read
//    with the histogram; a segment whose largest key is in a bin >= T and whose second
//    is not gives its one candidate straight from the metadata, and only segments with
//    two or more such entries have their scores read again.  General path (bin T too
//    full, too many segments): the scores of every segment whose largest key reaches T
//    are read again, in rounds, and the candidates may spill to the workspace;
//  - cut_and_write: the exact cut in bin T and the k entries in entry order.
// It runs once per request from a cold instruction cache: loops stay rolled.
template <int KF>
__device__ __noinline__ void select_completed(const IndexArgs& a) {
  const ScoreCarve cv = score_carve<KF>();
  ScoreSmem* sm = cv.sm;
  uint8_t* stages = cv.stages;
  uint8_t* qbuf = cv.qbuf;
  uint32_t* hist = cv.hist;
  uint16_t* scratch = cv.scratch;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int nwarps = kScoreThreads / 32;
  const uint32_t lt_mask = (1u << lane) - 1u;
  const float* scores_all = reinterpret_cast<const float*>(a.ws + a.L.scores);
  const uint64_t* segmeta_all = reinterpret_cast<const uint64_t*>(a.ws + a.L.segmeta);
  const uint32_t* ghist = reinterpret_cast<const uint32_t*>(a.ws + a.L.hist);
  uint32_t* ready = reinterpret_cast<uint32_t*>(a.ws + a.L.ready);
  const int segs_pad = a.L.n_pad / kSeg;
  // The threads that saw a request's count complete read it with an acquire-release
  // atomic; this fence and barrier order every read below after it for the whole block.
  __threadfence();
  // In a fused step the attention reads the main entries this step's compressor writes
  // as soon as a ready flag is up: raise none before that kernel has completed.
  if (a.wait_fresh && threadIdx.x == 0) grid_dep_wait();
  __syncthreads();
  auto raise_ready = [&](int b) {
    __threadfence();   // this thread's output, before the flag
    __syncthreads();
    if (threadIdx.x == 0) st_release(ready + b, 1u);
  };
  auto pad_out = [&](int b, int from) {
    int32_t* out_idx = a.topk_idx + size_t(b) * a.k;
    float* out_sc = a.topk_score ? a.topk_score + size_t(b) * a.k : nullptr;
#pragma unroll 1
    for (int j = from + threadIdx.x; j < a.k; j += blockDim.x) {
      out_idx[j] = -1;
      if (out_sc) out_sc[j] = -INFINITY;
    }
  };
  // Requests come from the selection queue, in completion order: a block that is done
  // streaming claims the next slot and waits (bounded) for the request that fills it, so
  // the selections of a batch run on as many blocks as there are requests, each starting
  // as soon as its request is complete.
  uint32_t* qctl = reinterpret_cast<uint32_t*>(a.ws + a.L.queue);
  const int32_t* qslot = reinterpret_cast<const int32_t*>(qctl + 2);
#pragma unroll 1
  for (;;) {
    if (threadIdx.x == 0) {
      int q = -1;
      const uint32_t slot = atomicAdd(qctl, 1u);
      if (slot < static_cast<uint32_t>(a.B)) {
        q = ld_acquire_s32(qslot + slot);
        if (q < 0) {
          const unsigned long long t0 = clock64();
          while ((q = ld_acquire_s32(qslot + slot)) < 0) {
            if (clock64() - t0 > a.spin) {
              set_err(CSKV_ERR_TIMEOUT);
              break;
            }
            __nanosleep(64);
          }
        }
      }
      sm->qreq = q;
    }
    __threadfence();
    __syncthreads();
    const int b = sm->qreq;
    __syncthreads();
    if (b < 0) break;
    const int nb = sm->nbv[b];
    const float* sc = scores_all + size_t(b) * a.L.n_pad;
    const uint64_t* meta = segmeta_all + size_t(b) * segs_pad;
    int32_t* out_idx = a.topk_idx + size_t(b) * a.k;
    float* out_sc = a.topk_score ? a.topk_score + size_t(b) * a.k : nullptr;
    if (nb <= a.k) {
      // every visible entry is selected, in order
#pragma unroll 1
      for (int j = threadIdx.x; j < nb; j += blockDim.x) {
        out_idx[j] = j;
        if (out_sc) out_sc[j] = __ldcg(sc + j);
      }
      pad_out(b, nb);
      raise_ready(b);
      continue;
    }
    const int nseg = (nb + kSeg - 1) / kSeg;
    const bool meta_fits = nseg <= kMetaSegs;
    // ---- threshold bin; the segment metadata comes in beside the fine bins
    uint64_t* s_meta = reinterpret_cast<uint64_t*>(stages);   // [0, 64 KiB)
    const uint32_t* ghb = ghist + size_t(b) * kHistStride;
    uint32_t* s_fine = hist;
#pragma unroll 1
    for (int x = threadIdx.x; x < kHistBins / 4; x += blockDim.x) cp_async16(s_fine + 4 * x, ghb + 4 * x);
    cp_async_commit();
    if (meta_fits) {
#pragma unroll 1
      for (int x = threadIdx.x; x < (nseg + 1) / 2; x += blockDim.x) cp_async16(s_meta + 2 * x, meta + 2 * x);
    }
    cp_async_commit();
    threshold_bin(sm, ghb, a.k, s_fine, true);   // waits for the fine bins; the metadata lands meanwhile
    const int T = sm->T;
    const uint32_t above = sm->above;
    if (T < 0) {   // fewer than k binned entries (an earlier error dropped some)
      cp_async_wait_all();   // the metadata copies land before the next request reuses their place
      pad_out(b, 0);
      raise_ready(b);
      continue;
    }
    const uint32_t nexp = above + sm->inT;
    // ---- fast path (the usual case).  Thread t owns the kOwn consecutive segments from
    // kOwn * t, so its candidates are consecutive and in entry order once the threads'
    // counts are scanned; it visits them in an order rotated by t, so that a warp's
    // metadata loads spread over the banks.  single = largest key in a bin >= T and the
    // second not: its one candidate comes from the metadata, written by the owner.
    // multi = both (rare): the owner lists the segment and copies its 32 scores into
    // shared memory (up to kMulti in the block); a warp per listed segment counts and
    // writes its entries (a lane per entry).
    constexpr int kGrp = 8;   // shared-memory loads issued together in the passes below
    constexpr int kOwn = ((kMetaSegs + kScoreThreads - 1) / kScoreThreads + kGrp - 1) / kGrp * kGrp;
    static_assert(kOwn <= 32, "a thread's segments fit a 32-bit mask");
    const bool fast = meta_fits && nexp <= static_cast<uint32_t>(kSelCand);
    if (fast) {
      unsigned long long* s_cand = reinterpret_cast<unsigned long long*>(stages + kMetaSegs * 8);
      float* s_msc = reinterpret_cast<float*>(hist);         // [kMulti][32] scores of the multi segments
      uint16_t* s_mseg = scratch;                            // [kMulti] their segments
      uint16_t* s_mc = scratch + kMulti;                     // [kMulti] their candidate counts
      uint32_t* s_mbits = reinterpret_cast<uint32_t*>(qbuf);   // [kMulti] their candidates' lanes
      uint32_t* s_mpos = s_mbits + kMulti;                   // [kMulti] position of their first candidate
      const int q0 = min(nseg, static_cast<int>(threadIdx.x) * kOwn);
      const int no = min(nseg - q0, kOwn);
      const int rot = static_cast<int>(threadIdx.x) % kOwn;
      if (threadIdx.x == 0) sm->cnt[1] = 0;
      cp_async_wait_all();   // the segment metadata
      __syncthreads();
      // The loops below issue their shared-memory loads in groups of eight before any use
      // (the latency of one load, not of eight, per group).
      static_assert(kOwn % kGrp == 0, "whole groups");
      uint32_t smask = 0, mmask = 0;   // bit i: segment q0 + i is single / multi
#pragma unroll 1
      for (int g0 = 0; g0 < kOwn; g0 += kGrp) {
        uint64_t mv[kGrp];
#pragma unroll
        for (int u = 0; u < kGrp; ++u) {
          const int i = (g0 + u + rot) % kOwn;
          mv[u] = i < no ? s_meta[q0 + i] : 0ull;
        }
#pragma unroll
        for (int u = 0; u < kGrp; ++u) {
          const int i = (g0 + u + rot) % kOwn;
          const int b1 = static_cast<int>(mv[u] >> (64 - kHistBits));
          const int b2 = static_cast<int>((mv[u] >> 8) & (kHistBins - 1));
          if (i < no && b1 >= T) {
            if (b2 < T) smask |= 1u << i;
            else mmask |= 1u << i;
          }
        }
      }
      const uint32_t nm = static_cast<uint32_t>(__popc(mmask));
      const uint32_t mslot = nm ? atomicAdd(&sm->cnt[1], nm) : 0u;
      if (nm != 0 && mslot + nm <= static_cast<uint32_t>(kMulti)) {
        uint32_t h = mslot;
#pragma unroll 1
        for (uint32_t mb = mmask; mb != 0; mb &= mb - 1, ++h) {
          const int q = q0 + __ffs(mb) - 1;
          s_mseg[h] = static_cast<uint16_t>(q);
          const float* src = sc + static_cast<long long>(q) * kSeg;
#pragma unroll
          for (int x = 0; x < kSeg / 4; ++x) cp_async16(s_msc + h * kSeg + 4 * x, src + 4 * x);
        }
      }
      cp_async_wait_all();
      __syncthreads();
      const uint32_t nmulti = sm->cnt[1];
      if (nmulti <= static_cast<uint32_t>(kMulti)) {   // uniform
        // the multi segments' entries in bins >= T: a warp per segment
#pragma unroll 1
        for (uint32_t h = warp; h < nmulti; h += nwarps) {
          const long long j = static_cast<long long>(s_mseg[h]) * kSeg + lane;
          const bool f = j < nb && static_cast<int>(order_key(s_msc[h * kSeg + lane]) >> (32 - kHistBits)) >= T;
          const unsigned fm = __ballot_sync(0xFFFFFFFFu, f);
          if (lane == 0) {
            s_mbits[h] = fm;
            s_mc[h] = static_cast<uint16_t>(__popc(fm));
          }
        }
        __syncthreads();
        uint32_t c = static_cast<uint32_t>(__popc(smask));
#pragma unroll 1
        for (uint32_t r = 0; r < nm; ++r) c += s_mc[mslot + r];
        uint32_t total;
        const uint32_t pos = block_scan_excl(sm, c, total);
        if (total <= static_cast<uint32_t>(kSelCand)) {   // uniform; only an earlier error breaks it
          // singles by their owners (a visit per candidate segment, not per segment); each
          // multi segment's first position noted.  The candidates of the thread's first two
          // multi segments come in by selects, more (rare) by a loop.
          const uint32_t mb1 = mmask & (0u - mmask);   // lowest multi bit (0: none)
          const uint32_t mrest = mmask & ~mb1;
          const uint32_t mb2 = mrest & (0u - mrest);   // second lowest
          const uint32_t mc1 = nm > 0 ? s_mc[mslot] : 0u;
          const uint32_t mc2 = nm > 1 ? s_mc[mslot + 1] : 0u;
#pragma unroll 1
          for (uint32_t rem = smask | mmask; rem != 0; rem &= rem - 1u) {
            const int i = __ffs(rem) - 1;
            const uint32_t bit = 1u << i;
            uint32_t p = pos + static_cast<uint32_t>(__popc(smask & (bit - 1u))) + (mb1 != 0u && mb1 < bit ? mc1 : 0u) +
                         (mb2 != 0u && mb2 < bit ? mc2 : 0u);
            const uint32_t nbefore = static_cast<uint32_t>(__popc(mmask & (bit - 1u)));
#pragma unroll 1
            for (uint32_t r = 2; r < nbefore; ++r) p += s_mc[mslot + r];
            if (smask & bit) {
              const uint64_t m = s_meta[q0 + i];
              const uint32_t j = static_cast<uint32_t>(q0 + i) * kSeg + static_cast<uint32_t>(m & 31u);
              s_cand[p] = (m & 0xFFFFFFFF00000000ull) | (0xFFFFFFFFu - j);
            } else {
              s_mpos[mslot + nbefore] = p;
            }
          }
          __syncthreads();
#pragma unroll 1
          for (uint32_t h = warp; h < nmulti; h += nwarps) {
            const uint32_t fm = s_mbits[h];
            if ((fm >> lane) & 1u) {
              const uint32_t j = static_cast<uint32_t>(s_mseg[h]) * kSeg + static_cast<uint32_t>(lane);
              s_cand[s_mpos[h] + __popc(fm & lt_mask)] =
                  (static_cast<unsigned long long>(order_key(s_msc[h * kSeg + lane])) << 32) | (0xFFFFFFFFu - j);
            }
          }
          __syncthreads();
        // ---- the cut among bin T's keys by 8-bit digits (bits 51-44, 43-36, ..., 11-4, 3-0);
        // keys above bin T never match the prefix and are all taken
        if (threadIdx.x == 0) {
          sm->need = min(static_cast<uint32_t>(a.k) - above, total > above ? total - above : 0u);
          sm->done = 0;
          sm->mask = ~0ull << 52;
          sm->prefix = static_cast<unsigned long long>(T) << 52;
        }
        __syncthreads();
#pragma unroll 1
        for (int shift = 44; shift >= 0; shift = shift >= 8 ? shift - 8 : (shift > 0 ? 0 : -1)) {
          if (sm->done || sm->need == 0) break;
          const int nd = shift >= 4 ? 256 : 16;
          const unsigned long long dmask = static_cast<unsigned long long>(nd - 1) << shift;
          if (threadIdx.x < 256) sm->d256[threadIdx.x] = 0;
          __syncthreads();
          const unsigned long long pm = sm->mask, pp = sm->prefix;
#pragma unroll 1
          for (uint32_t x = threadIdx.x; x < total; x += blockDim.x) {
            const unsigned long long key = s_cand[x];
            if ((key & pm) == pp) atomicAdd(&sm->d256[(key & dmask) >> shift], 1u);
          }
          __syncthreads();
          if (warp == 0) {
            // lane l owns digits nd-1-8l .. nd-8-8l (from the top)
            const uint32_t need = sm->need;
            uint32_t v[8], sum = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int d = nd - 1 - 8 * lane - i;
              v[i] = d >= 0 ? sm->d256[d] : 0u;
              sum += v[i];
            }
            uint32_t incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
              if (lane >= o) incl += y;
            }
            const unsigned hit = __ballot_sync(0xFFFFFFFFu, incl >= need);
            if (hit != 0 && lane == __ffs(hit) - 1) {
              uint32_t acc = incl - sum, dv = v[7];
              int di = 7;
              bool got = false;
#pragma unroll
              for (int i = 0; i < 8; ++i) {   // unrolled: v stays in registers
                if (!got) {
                  if (acc + v[i] >= need) {
                    got = true;
                    di = i;
                    dv = v[i];
                  } else {
                    acc += v[i];
                  }
                }
              }
              const int d = nd - 1 - 8 * lane - di;
              sm->need = need - acc;
              sm->prefix = pp | (static_cast<unsigned long long>(d) << shift);
              sm->mask = pm | dmask;
              if (dv == need - acc) sm->done = 1;
            }
          }
          __syncthreads();
          if (shift == 0) break;
        }
        // ---- the output: selected <=> (key & mask) >= prefix; each warp a contiguous
        // range of the candidates, in order
        const unsigned long long pm = sm->mask, pp = sm->prefix;
        const uint32_t off = static_cast<uint32_t>((static_cast<unsigned long long>(total) * warp) / nwarps);
        const uint32_t end = static_cast<uint32_t>((static_cast<unsigned long long>(total) * (warp + 1)) / nwarps);
        uint32_t nsel_w = 0;
#pragma unroll 1
        for (uint32_t x0 = off; x0 < end; x0 += 32) {
          const uint32_t x = x0 + lane;
          const bool sel = x < end && (s_cand[x] & pm) >= pp;
          nsel_w += __popc(__ballot_sync(0xFFFFFFFFu, sel));
        }
        if (lane == 0) sm->wcnt[warp] = nsel_w;
        __syncthreads();
        uint32_t opos = 0, nsel = 0;
#pragma unroll 1
        for (int w2 = 0; w2 < nwarps; ++w2) {
          opos += w2 < warp ? sm->wcnt[w2] : 0u;
          nsel += sm->wcnt[w2];
        }
#pragma unroll 1
        for (uint32_t x0 = off; x0 < end; x0 += 32) {
          const uint32_t x = x0 + lane;
          const unsigned long long key = x < end ? s_cand[x] : 0ull;
          const bool sel = x < end && (key & pm) >= pp;
          const unsigned m = __ballot_sync(0xFFFFFFFFu, sel);
          const uint32_t p = opos + __popc(m & lt_mask);
          if (sel && p < static_cast<uint32_t>(a.k)) {
            out_idx[p] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(key));
            if (out_sc) out_sc[p] = from_order_key(static_cast<uint32_t>(key >> 32));
          }
          opos += __popc(m);
        }
        pad_out(b, static_cast<int>(min(nsel, static_cast<uint32_t>(a.k))));   // only after an error
        raise_ready(b);
        continue;
        }
      }
      __syncthreads();   // too many multi segments: every thread is past the counts before the general path
    }
    // ---- general path: every segment whose largest key reaches T is read again, in rounds
    cp_async_wait_all();   // the metadata copies (unused here) land before the stage ring is reused
    __syncthreads();
    unsigned long long* cand = nexp <= static_cast<uint32_t>(kSelCand)
                                   ? reinterpret_cast<unsigned long long*>(stages + kMetaSegs * 8)
                                   : reinterpret_cast<unsigned long long*>(a.ws + a.L.cand) + size_t(b) * a.L.n_pad;
    float* s_score = reinterpret_cast<float*>(stages);   // [0, 64 KiB): the metadata is not needed here
    uint16_t* s_list = reinterpret_cast<uint16_t*>(qbuf);
    uint16_t* g_cnt = scratch;
    uint32_t nk = 0;
#pragma unroll 1
    for (int gc = 0; gc < nseg; gc += kSelSegs) {
      const int ns = min(kSelSegs, nseg - gc);
      // the hit segments of [gc, gc + ns), in order: thread t owns segments 24t .. 24t+23
      uint32_t nhit;
      {
        constexpr int kOwn = 24;
        static_assert(kOwn * kScoreThreads >= kSelSegs, "every segment of a pass has an owner");
        const int q0 = threadIdx.x * kOwn;
        uint32_t m = 0;
#pragma unroll
        for (int u = 0; u < kOwn / 2; ++u) {
          const int q = q0 + 2 * u;
          if (q < ns) {   // the table's rows are padded to a multiple of 4 segments
            const uint4 x = __ldcg(reinterpret_cast<const uint4*>(meta + gc + q));
            m |= (static_cast<int>(x.y >> (32 - kHistBits)) >= T ? 1u : 0u) << (2 * u);
            m |= (static_cast<int>(x.w >> (32 - kHistBits)) >= T ? 2u : 0u) << (2 * u);
          }
        }
        if (ns - q0 < kOwn) m &= ns > q0 ? (1u << (ns - q0)) - 1u : 0u;
        uint32_t pos = block_scan_excl(sm, __popc(m), nhit);
#pragma unroll 1
        while (m) {
          const int q = __ffs(m) - 1;
          m &= m - 1;
          s_list[pos++] = static_cast<uint16_t>(q0 + q);
        }
        __syncthreads();
      }
#pragma unroll 1
      for (uint32_t h0 = 0; h0 < nhit; h0 += kHitRound) {
        const uint32_t nh = min(nhit - h0, static_cast<uint32_t>(kHitRound));
#pragma unroll 1
        for (uint32_t x = threadIdx.x; x < nh * 8; x += blockDim.x)
          cp_async16(s_score + (x >> 3) * kSeg + (x & 7) * 4,
                     sc + (static_cast<long long>(gc) + s_list[h0 + (x >> 3)]) * kSeg + (x & 7) * 4);
        cp_async_wait_all();
        __syncthreads();
        // per hit segment (a warp, a lane per entry): how many of its entries are in bins >= T
        constexpr int kU = 4;
#pragma unroll 1
        for (uint32_t hb = warp * kU; hb < nh; hb += nwarps * kU) {
#pragma unroll
          for (int u = 0; u < kU; ++u) {
            const uint32_t h = min(hb + u, nh - 1);
            const long long j = (static_cast<long long>(gc) + s_list[h0 + h]) * kSeg + lane;
            const bool f = hb + u < nh && j < nb &&
                           static_cast<int>(order_key(s_score[h * kSeg + lane]) >> (32 - kHistBits)) >= T;
            const unsigned mm = __ballot_sync(0xFFFFFFFFu, f);
            if (lane == 0 && hb + u < nh) g_cnt[hb + u] = static_cast<uint16_t>(__popc(mm));
          }
        }
        if (threadIdx.x == 0) g_cnt[nh] = 0;
        __syncthreads();
        block_exclusive_scan16(sm, g_cnt, static_cast<int>(nh) + 1);
#pragma unroll 1
        for (uint32_t hb = warp * kU; hb < nh; hb += nwarps * kU) {
#pragma unroll
          for (int u = 0; u < kU; ++u) {
            const uint32_t h = min(hb + u, nh - 1);
            const long long j = (static_cast<long long>(gc) + s_list[h0 + h]) * kSeg + lane;
            const uint32_t key = order_key(s_score[h * kSeg + lane]);
            const bool f = hb + u < nh && j < nb && static_cast<int>(key >> (32 - kHistBits)) >= T;
            const unsigned mm = __ballot_sync(0xFFFFFFFFu, f);
            const uint32_t at = nk + g_cnt[h] + __popc(mm & lt_mask);
            if (f && at < nexp)   // at most the binned count (guards a histogram short of the scores)
              cand[at] = (static_cast<unsigned long long>(key) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(j));
          }
        }
        nk += g_cnt[nh];
        __syncthreads();
      }
    }
    cut_and_write(a, sm, cand, min(nk, nexp), T, above, reinterpret_cast<uint32_t*>(hist),
                  reinterpret_cast<uint32_t*>(qbuf + 1024), out_idx, out_sc);
    raise_ready(b);
  }
}

// LARGE (batches of more than kReqCache requests, e.g. one request per prompt query in
// prefill): the scheduler also counts the tiles handed out, so that a block that finds
// its requests exhausted stops as soon as every tile has an owner instead of visiting
// every request (one atomic each) before it concludes there is no work left.
template <int KF, bool LARGE>
__global__ void __launch_bounds__(kLaunchBound, 1)
    index_score_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ IndexArgs a) {
  constexpr int kStageBytes = KeyFmt<KF>::kStageBytes;
  constexpr int kStages = KeyFmt<KF>::kStages;   // per producer
  constexpr int kQImage = KeyFmt<KF>::kQImage;
  constexpr int kAccs = KeyFmt<KF>::kAccs;
  constexpr bool FP8 = KF == kKfFp8;
  constexpr bool FP4 = KF == kKfFp4;
  // With as many accumulators as stages (FP8), tile i's stage and accumulator are
  // released by the same event - its MMAs completing - so the MMA warp commits once per
  // tile (to accfull[i % kAccs]) and the producers wait on that barrier for the stage.
  constexpr bool kMerged = kAccs == kProducers * kStages;
  const ScoreCarve cv = score_carve<KF>();
  uint8_t* stages = cv.stages;
  uint8_t* qbuf = cv.qbuf;
  uint32_t* hist = cv.hist;
  float* sring = cv.sring;
  uint16_t* scratch = cv.scratch;
  ScoreSmem* sm = cv.sm;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = a.N;
  float* scores_all = reinterpret_cast<float*>(a.ws + a.L.scores);
  uint32_t* segmax_all = reinterpret_cast<uint32_t*>(a.ws + a.L.segmax);
  uint32_t* ghist = reinterpret_cast<uint32_t*>(a.ws + a.L.hist);
  uint32_t* ctr_all = reinterpret_cast<uint32_t*>(a.ws + a.L.ctr);
  uint32_t* gbar = reinterpret_cast<uint32_t*>(a.ws + a.L.gbar);

  // tiles of all requests; for small batches every thread sums them here, for large
  // ones the block does, after the set-up barrier
  long long total = 0;
  if (a.B <= kReqCache) {
#pragma unroll 1
    for (int b = 0; b < a.B; ++b) {
      const int v = visible(a, b);
      total += (v + kTileRows - 1) / kTileRows;
      if (threadIdx.x == 0) sm->nbv[b] = v;   // read after the set-up barrier
    }
  }

  if constexpr (!LARGE) {
    // requests without a visible entry have no tile to complete: block 0 queues them
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      if (!a.wait_fresh) grid_dep_wait();   // the prep cleared the queue
      for (int b = 0; b < a.B; ++b)
        if (sm->nbv[b] == 0) queue_push(a, b);
    }
    // the prep (complete before this kernel starts) wrote the fresh bounds
    if (a.wait_fresh && threadIdx.x < a.B) sm->fresh[threadIdx.x] = reinterpret_cast<const int32_t*>(a.ws + a.L.fresh)[threadIdx.x];
  }
  if (threadIdx.x == 0) {
    for (int p = 0; p < kProducers; ++p)
      for (int s = 0; s < kStages; ++s) { mbar_init(&sm->full[p][s], 1); mbar_init(&sm->empty[p][s], 1); }
    for (int c = 0; c < kAccs; ++c) { mbar_init(&sm->accfull[c], 1); mbar_init(&sm->accempty[c], 4); }
    for (int c = 0; c < 2; ++c) { mbar_init(&sm->qfull[c], 1); mbar_init(&sm->qempty[c], 1); }
    for (int s = 0; s < kScaleSlots; ++s) { mbar_init(&sm->sfull[s], 1); mbar_init(&sm->sempty[s], 4); }
    for (int s = 0; s < kRecSlots; ++s) { mbar_init(&sm->rfull[s], 1); mbar_init(&sm->rempty[s], 1); }
    mbar_init(&sm->drain, 1);
    for (int g = 0; g < kGroups; ++g) mbar_init(&sm->hbar[g], 4);
    sm->abort = 0;
    fence_mbar_init();
  }
  // The scheduler's first chunk - chunk r of its home request, r = its rank among that
  // request's home blocks, taken without an atomic - has its page ids requested here,
  // so that their loads overlap the set-up (block tables are inputs); and the home
  // request's block-table row goes to L2 (the scheduler reads it next), each of its home
  // blocks prefetching a share of the row's 128-byte lines.
  const int home = home_request(blockIdx.x, a.B, gridDim.x);
  int first_ids[2 * kChunkTiles];   // before the request's visible count is known: masked below
  if (warp == kWarpSched && lane == 0) {
    const int r0 = blockIdx.x - first_home_block(home, a.B, gridDim.x);
    chunk_page_ids<kChunkTiles>(a, home, 0x7FFFFFFF, r0 * kChunkTiles, first_ids);
  }
  if constexpr (!LARGE) {
    const int f0 = first_home_block(home, a.B, gridDim.x);
    const int nh = first_home_block(home + 1, a.B, gridDim.x) - f0;
    const int pages = min(a.keys.max_pages, static_cast<int>((a.n_max + kPageRows - 1) / kPageRows));
    const int32_t* row = a.keys.block_table + static_cast<long long>(home) * a.keys.max_pages;
    if (a.keys.block_table != nullptr) {
#pragma unroll 1
      for (int x = static_cast<int>(blockIdx.x) - f0 + nh * static_cast<int>(threadIdx.x); 32 * x < pages;
           x += nh * static_cast<int>(blockDim.x))
        prefetch_l2(row + 32 * x);
    }
  }
  for (int i = threadIdx.x; i < kGroups * kHistBins; i += blockDim.x) hist[i] = 0;
  uint32_t ncols = 32;
  while (ncols < static_cast<uint32_t>(kAccs * N)) ncols <<= 1;
  if (FP4) ncols = 512;   // the scale factors sit above the accumulators
  if (warp == kWarpMma) tmem_alloc(&sm->tmem_base, ncols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  // The kernel is a programmatic dependent of the query prep, which is one of the
  // compressor that writes this step's keys: the set-up above overlaps them, and no
  // thread reads what they write (keys, query images, weights, counters) before
  // this wait.  The scheduling producer first requests its first chunk's page ids
  // (block tables are inputs) and waits after that.
  const bool sched_thread = warp == kWarpSched && lane == 0;
  // Streaming mode reads its predecessor's output (query images, counters) only after
  // waiting for it, unless that predecessor is the compressor of a fused step (the
  // prep before it has completed; only tiles with fresh keys wait, below).
  const bool wait_at_start = LARGE || !a.wait_fresh;
  // In a fused step the next kernel is the attention, which touches nothing of the
  // indexer's workspace: it may be scheduled as soon as SMs free up.
  if (!LARGE && a.wait_fresh) grid_dep_launch();
  if constexpr (LARGE) {
    // Large batches: the requests' tile counts, their total, and this block's selection
    // work are found by the whole block (each thread a contiguous range of requests,
    // block scans for the prefixes), so the cost grows with the batch divided by the
    // block, not with the batch.
    const int per = (a.B + kScoreThreads - 1) / kScoreThreads;
    const int rb0 = min(a.B, static_cast<int>(threadIdx.x) * per), rb1 = min(a.B, rb0 + per);
    uint32_t cnt = 0;
#pragma unroll 1
    for (int b = rb0; b < rb1; ++b) {
      const int v = visible(a, b);
      cnt += static_cast<uint32_t>((v + kTileRows - 1) / kTileRows);
      if (b < kReqCache) sm->nbv[b] = v;
    }
    uint32_t tot;
    const uint32_t c0 = block_scan_excl(sm, cnt, tot);
    total = tot;
    long long C = c0;
    uint32_t nmine = 0;
#pragma unroll 1
    for (int b = rb0; b < rb1; ++b) {
      const long long tb = (visible(a, b) + kTileRows - 1) / kTileRows;
      WorkItem wi;
      nmine += block_range(blockIdx.x, gridDim.x, C, tb, total, wi.lo, wi.hi, wi.fb, wi.nbk, wi.per) ? 1u : 0u;
      C += tb;
    }
    uint32_t nw;
    uint32_t pos = block_scan_excl(sm, nmine, nw);
    if (nmine) {
      C = c0;
#pragma unroll 1
      for (int b = rb0; b < rb1; ++b) {
        const long long tb = (visible(a, b) + kTileRows - 1) / kTileRows;
        WorkItem wi;
        if (block_range(blockIdx.x, gridDim.x, C, tb, total, wi.lo, wi.hi, wi.fb, wi.nbk, wi.per)) {
          wi.b = b;
          if (pos < static_cast<uint32_t>(kWorkItems)) sm->work[pos] = wi;
          ++pos;
        }
        C += tb;
      }
    }
    if (threadIdx.x == 0) sm->nwork = nw <= static_cast<uint32_t>(kWorkItems) ? static_cast<int>(nw) : -1;
    __syncthreads();
  }
  if (!sched_thread && wait_at_start) grid_dep_wait();
  // visible entries of request b: the first kReqCache requests' counts were kept in
  // shared memory by the set-up (a global load and a 64-bit division fewer on the
  // scheduler's path)
  auto nvis = [&](int b) { return b < kReqCache ? sm->nbv[b] : visible(a, b); };

  // ======================================================= phase 1: scores
  // Tiles are handed out dynamically, in chunks of kChunkTiles consecutive tiles of
  // one request: the scheduler warp grabs a chunk from the request's counter (starting
  // at a home request spread over the grid, moving on when it is exhausted), loads its
  // page ids and writes one record per tile of the request into a ring that runs up to
  // kRecSlots tiles ahead of the copies, so that neither its atomics nor its
  // block-table loads hold up a tile.  Block-local tile i goes through producer i % 2
  // (stage (i / 2) % kStages of its ring), accumulator i % kAccs, epilogue group i % 2
  // and slot i % 16 of the scale and tile-info rings; request -1 ends the sequence
  // (one end record per producer).
  if (warp < kProducers) {
    // ------------------------------------------------------------ producers
    const int pw = warp;
    if (lane == 0) {
      prefetch_tmap(&tmap);
      // the keys are read once: evict-first, so the stream does not push the scores,
      // segment maxima and histograms that the selection reads back out of L2
      const uint64_t pol = l2_evict_first();
      long long np = 0;       // tiles this producer posted (the end marker included)
      bool waited = wait_at_start;   // this thread has seen the kernel before complete
      // post local tile i = (request b, tile t) with its two page ids (-2: no page,
      // -3: page outside the block table); b < 0 posts the end marker
      auto post = [&](long long i, int b, int t, int id0, int id1) -> bool {
        const int s = static_cast<int>(np % kStages);
        const long long round = np / kStages;
        if (round > 0 && !role_wait(sm, kMerged ? &sm->accfull[i % kAccs] : &sm->empty[pw][s], (round - 1) & 1, a.spin))
          return false;
        const int ss = static_cast<int>(i % kScaleSlots);
        const long long su = i / kScaleSlots;
        if (su > 0 && !role_wait(sm, &sm->sempty[ss], (su - 1) & 1, a.spin)) return false;
        if (!waited && b >= 0) {
          // a tile holding entries the compressor before this kernel may still write
          if (static_cast<long long>(t + 1) * kTileRows > sm->fresh[b]) {
            grid_dep_wait();
            fence_proxy_async_global();   // its generic-proxy writes, before the tensor copies read them
            waited = true;
          }
        }
        uint8_t* dst = stages + (pw * kStages + s) * kStageBytes;
        uint32_t bytes = 0;
        int pages[2] = {b >= 0 ? id0 : -2, b >= 0 ? id1 : -2};
        for (int pg = 0; pg < 2; ++pg) {
          if (pages[pg] == -2) continue;
          if (pages[pg] < 0 || pages[pg] >= a.keys.num_pages) {
            set_err(CSKV_ERR_BOUNDS);
            pages[pg] = -2;
            continue;
          }
          bytes += FP8 ? 64 * 128 : FP4 ? 64 * 64 + 256 : 64 * 256;
        }
        sm->tinfo[ss] = make_int2(b, t);
        sm->smask[ss] = (pages[0] >= 0 ? 1 : 0) | (pages[1] >= 0 ? 2 : 0);
        mbar_expect_tx(&sm->full[pw][s], bytes);
        mbar_expect_tx(&sm->sfull[ss], FP8 ? (pages[0] >= 0 ? 256u : 0u) + (pages[1] >= 0 ? 256u : 0u) : 0u);
        for (int pg = 0; pg < 2; ++pg) {
          if (pages[pg] < 0) continue;
          if (FP4) {
            // the page's 64 code rows (64-byte swizzle) and its 64 rows of 4 scale bytes
            const uint8_t* pgp = static_cast<const uint8_t*>(a.keys.pool) + size_t(pages[pg]) * a.keys.page_bytes;
            tma_load_3d_hint(dst + pg * 4096, &tmap, 0, 0, pages[pg], &sm->full[pw][s], pol);
            bulk_g2s_hint(dst + 8192 + pg * 256, pgp + kPageRows * 64, 256, &sm->full[pw][s], pol);
            continue;
          }
          tma_load_3d_hint(dst + pg * 8192, &tmap, 0, 0, pages[pg], &sm->full[pw][s], pol);
          if (!FP8) tma_load_3d_hint(dst + 16384 + pg * 8192, &tmap, 64, 0, pages[pg], &sm->full[pw][s], pol);
          if (FP8) {
            const uint8_t* pgp = static_cast<const uint8_t*>(a.keys.pool) + size_t(pages[pg]) * a.keys.page_bytes;
            bulk_g2s_hint(sring + ss * kTileRows + pg * kPageRows, pgp + kPageRows * 128, 256, &sm->sfull[ss],
                          pol);
          }
        }
        ++np;
        return true;
      };
      for (long long i = pw;; i += kProducers) {
        const int rs = static_cast<int>(i % kRecSlots);
        if (!role_wait(sm, &sm->rfull[rs], (i / kRecSlots) & 1, a.spin)) break;
        const int4 r = sm->rec[rs];
        mbar_arrive(&sm->rempty[rs]);
        if (!post(i, r.x, r.y, r.z, r.w) || r.x < 0) break;
      }
      // drain: every copy this producer issued must land before the block moves on
      for (int s = 0; s < kStages && s < np; ++s) {
        const long long uses = (np - s + kStages - 1) / kStages;
        mbar_wait(&sm->full[pw][s], (uses - 1) & 1, kDefaultSpinLimit);
      }
      for (int r = 0; r < kScaleSlots / 2 && r < np; ++r) {   // slot 2r + pw: its tiles are m = r mod 8
        const long long uses = (np - r + kScaleSlots / 2 - 1) / (kScaleSlots / 2);
        mbar_wait(&sm->sfull[2 * r + pw], (uses - 1) & 1, kDefaultSpinLimit);
      }
    }
  } else if (warp == kWarpSched) {
    // ------------------------------------------------------------ scheduler
    if (lane == 0) {
      int nreq = 0;   // query images loaded
      auto tiles_of = [&](int b) { return (nvis(b) + kTileRows - 1) / kTileRows; };
      // the chunk's 2 x kChunkTiles page ids, all loads in flight
      auto chunk_ids = [&](int b, int t0, int (&ids)[2 * kChunkTiles]) {
        chunk_page_ids<kChunkTiles>(a, b, b >= 0 ? nvis(b) : 0, t0, ids);
      };
      int req = home;
      uint32_t pending = 0;   // the next grab (one in flight: the record ring hides its latency)
      auto grab = [&]() { return atomicAdd(&ctr_all[req * 4], static_cast<uint32_t>(kChunkTiles)); };
      uint32_t* handed = gbar + 1;   // LARGE: tiles handed out so far (cleared by the prep)
      // the next chunk: (request, first tile) from the pending grab; request -1 = none left
      auto resolve = [&](int& b, int& t0) {
        int tiles = tiles_of(req);
        int fails = 0;
        uint32_t seen = 0;   // LARGE: the handed-out count read during the previous step
        while (pending >= static_cast<uint32_t>(tiles) && ++fails < a.B) {
          if constexpr (LARGE) {
            if (seen >= static_cast<uint32_t>(total)) break;
          }
          req = (req + 1) % a.B;
          tiles = tiles_of(req);
          if constexpr (LARGE) seen = *reinterpret_cast<volatile uint32_t*>(handed);
          pending = grab();
        }
        if (pending >= static_cast<uint32_t>(tiles)) {
          b = -1;
          t0 = 0;
        } else {
          b = req;
          t0 = static_cast<int>(pending);
          if constexpr (LARGE) atomicAdd(handed, static_cast<uint32_t>(min(kChunkTiles, tiles - t0)));
          pending = grab();
        }
      };
      // record of local tile i (waits for its slot to be free)
      auto emit = [&](long long i, int b, int t, int id0, int id1) -> bool {
        const int rs = static_cast<int>(i % kRecSlots);
        const long long u = i / kRecSlots;
        if (u > 0 && !role_wait(sm, &sm->rempty[rs], (u - 1) & 1, a.spin)) return false;
        sm->rec[rs] = make_int4(b, t, id0, id1);
        mbar_arrive(&sm->rfull[rs]);
        return true;
      };
      int cb = -1, ct = 0;
      int ids[2 * kChunkTiles];
      const int r0 = blockIdx.x - first_home_block(req, a.B, gridDim.x);
      const bool static_first = static_cast<long long>(r0) * kChunkTiles < tiles_of(req);
      if (static_first) {
        cb = req;   // the block's first chunk, assigned without an atomic (page ids requested above)
        ct = r0 * kChunkTiles;
        const int n_b = nvis(req);
#pragma unroll
        for (int u = 0; u < 2 * kChunkTiles; ++u)
          ids[u] = (static_cast<long long>(ct) * 2 + u) * kPageRows >= n_b ? -2 : first_ids[u];
      }
      if (wait_at_start) grid_dep_wait();
      if constexpr (LARGE) {
        if (static_first) atomicAdd(handed, static_cast<uint32_t>(min(kChunkTiles, tiles_of(cb) - ct)));
      }
      pending = grab();
      if (!static_first) {
        resolve(cb, ct);
        chunk_ids(cb, ct, ids);
      }
      int q_b = -1;
      long long i = 0;   // records written
      bool ok = true;
      while (ok && cb >= 0) {
        if (cb != q_b) {
          // query image of the new request into buffer nreq % 2
          const int qb = nreq & 1;
          if (nreq >= 2 && !role_wait(sm, &sm->qempty[qb], ((nreq >> 1) - 1) & 1, a.spin)) break;
          mbar_expect_tx(&sm->qfull[qb], kQImage);
          bulk_g2s(qbuf + qb * kQImage, a.ws + a.L.qimg + size_t(cb) * kQSlot, kQImage, &sm->qfull[qb]);
          ++nreq;
          q_b = cb;
        }
        // the next chunk is resolved and its page ids requested before this one's records
        // (after them for the block's first chunk, whose records go out at once: the
        // ring is empty, and resolving waits for a grab's round trip)
        int nb2 = -1, nt = 0;
        int nids[2 * kChunkTiles];
        const bool first = i == 0;
        if (!first) {
          resolve(nb2, nt);
          chunk_ids(nb2, nt, nids);
        }
        const int tiles = tiles_of(cb);
#pragma unroll
        for (int u = 0; u < kChunkTiles; ++u) {
          if (ct + u < tiles && !emit(i++, cb, ct + u, ids[2 * u], ids[2 * u + 1])) {
            ok = false;
            break;
          }
        }
        if (first) {
          resolve(nb2, nt);
          chunk_ids(nb2, nt, nids);
        }
        cb = nb2;
        ct = nt;
#pragma unroll
        for (int u = 0; u < 2 * kChunkTiles; ++u) ids[u] = nids[u];
      }
      // one end record per producer
      if (ok) ok = emit(i, -1, 0, -2, -2);
      if (ok) emit(i + 1, -1, 0, -2, -2);
      for (int qb = 0; qb < 2 && qb < nreq; ++qb) {
        const int uses = (nreq - qb + 1) / 2;
        mbar_wait(&sm->qfull[qb], (uses - 1) & 1, kDefaultSpinLimit);
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if constexpr (FP4) {
      // The whole warp: per tile it first lays the keys' scale bytes out for the
      // scale-factor copy (lane r: the words of keys r, r + 32, r + 64, r + 96), then
      // lane 0 copies them to TMEM and issues the two K = 64 block-scaled MMAs.
      const uint32_t id0 = make_idesc_mxf4(128, 0, 0) | (static_cast<uint32_t>(N >> 3) << 17);
      const uint32_t id1 = make_idesc_mxf4(128, 0, 2) | (static_cast<uint32_t>(N >> 3) << 17);
      int nreq = 0, qb = 0, cur = -1;
      for (long long i = 0;; ++i) {
        const int pw = static_cast<int>(i & 1);
        const long long ip = i >> 1;
        const int s = static_cast<int>(ip % kStages);
        // every lane waits (each reads the landed bytes); a give-up is taken by all
        if (!__all_sync(0xFFFFFFFFu, role_wait(sm, &sm->full[pw][s], (ip / kStages) & 1, a.spin))) break;
        const int2 ti = sm->tinfo[i % kScaleSlots];
        if (ti.x < 0) break;
        uint8_t* st = stages + (pw * kStages + s) * kStageBytes;
        {
          const uint32_t* raw = reinterpret_cast<const uint32_t*>(st + 8192);
          const uint4 v = make_uint4(raw[lane], raw[lane + 32], raw[lane + 64], raw[lane + 96]);
          *reinterpret_cast<uint4*>(st + 8704 + 16 * lane) = v;
        }
        fence_proxy_async_smem();   // generic-proxy writes, before the copy reads them
        __syncwarp();
        const bool sw = ti.x != cur;
        if (sw) {
          if (cur >= 0 && lane == 0) mma_commit(&sm->qempty[qb]);
          qb = nreq & 1;
          if (!__all_sync(0xFFFFFFFFu, role_wait(sm, &sm->qfull[qb], (nreq >> 1) & 1, a.spin))) break;
          ++nreq;
          cur = ti.x;
        }
        const int c = static_cast<int>(i % kAccs);
        const long long use = i / kAccs;
        if (use > 0 && !__all_sync(0xFFFFFFFFu, role_wait(sm, &sm->accempty[c], (use - 1) & 1, a.spin))) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a_addr = smem_u32(st);
          const uint32_t b_addr = smem_u32(qbuf + qb * kQImage);
          const uint32_t sfa = tmem + kSfaCol + 4 * c;
          const uint32_t sfb = tmem + kSfaCol + 4 * kAccs + 4 * qb;
          if (sw) tmem_cp_32x128b_x4(sfb, smem_desc_plain(b_addr + 4096, 16, 128));
          tmem_cp_32x128b_x4(sfa, smem_desc_plain(smem_u32(st + 8704), 16, 128));
          const uint32_t d = tmem + c * N;
          const uint64_t da = smem_desc_sw64(a_addr, 512), db = smem_desc_sw64(b_addr, 512);
          mma_mxf4(d, da, db, id0, sfa, sfb, 0);
          mma_mxf4(d, da + 2, db + 2, id1, sfa, sfb, 1);   // K step of 32 bytes
          mma_commit(&sm->empty[pw][s]);
          mma_commit(&sm->accfull[c]);
        }
        __syncwarp();
      }
      if (lane == 0) {
        // drain: all issued MMAs complete before TMEM is released
        mma_commit(&sm->drain);
        mbar_wait(&sm->drain, 0, kDefaultSpinLimit);
      }
    } else if (lane == 0) {
      constexpr uint32_t idesc = FP8 ? make_idesc(0, 0, 0, 0, 128, 0) : make_idesc(1, 1, 0, 0, 128, 0);
      const uint32_t id = idesc | (static_cast<uint32_t>(N >> 3) << 17);
      int nreq = 0, qb = 0, cur = -1;
      for (long long i = 0;; ++i) {
        const int pw = static_cast<int>(i & 1);
        const long long ip = i >> 1;
        const int s = static_cast<int>(ip % kStages);
        if (!role_wait(sm, &sm->full[pw][s], (ip / kStages) & 1, a.spin)) break;
        const int2 ti = sm->tinfo[i % kScaleSlots];
        if (ti.x < 0) break;
        if (ti.x != cur) {
          if (cur >= 0) mma_commit(&sm->qempty[qb]);
          qb = nreq & 1;
          if (!role_wait(sm, &sm->qfull[qb], (nreq >> 1) & 1, a.spin)) break;
          ++nreq;
          cur = ti.x;
        }
        const int c = static_cast<int>(i % kAccs);
        const long long use = i / kAccs;
        if (use > 0 && !role_wait(sm, &sm->accempty[c], (use - 1) & 1, a.spin)) break;
        tc_fence_after();
        const uint32_t a_addr = smem_u32(stages + (pw * kStages + s) * kStageBytes);
        const uint32_t b_addr = smem_u32(qbuf + qb * kQImage);
        const uint32_t d = tmem + c * N;
        // the descriptors' start-address field counts 16-byte units: a 32-byte K step
        // within the swizzle atom adds 2 (the fields never carry: shared memory < 256 KiB)
        const uint64_t da = smem_desc_sw128(a_addr, 16, 1024), db = smem_desc_sw128(b_addr, 16, 1024);
        if (FP8) {
#pragma unroll
          for (int kb = 0; kb < 4; ++kb) mma_f8(d, da + 2 * kb, db + 2 * kb, id, kb > 0);
        } else {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const int ch = kk >> 2, o = (kk & 3) * 2;
            mma_f16(d, da + ch * (16384 >> 4) + o, db + ch * ((N * 128) >> 4) + o, id, kk > 0);
          }
        }
        if (!kMerged) mma_commit(&sm->empty[pw][s]);
        mma_commit(&sm->accfull[c]);
      }
      // drain: all issued MMAs complete before TMEM is released
      mma_commit(&sm->drain);
      mbar_wait(&sm->drain, 0, kDefaultSpinLimit);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int e = warp - kWarpEpi;               // 0 .. 4 * kGroups - 1
    const int grp = e >> 2;
    const int sub = warp & 3;                    // TMEM lane quarter of this warp
    const int row = sub * 32 + lane;             // entry within the tile
    const int gtid = (e & 3) * 32 + lane;        // 0..127 within the group
    uint32_t* ghs = hist + grp * kHistBins;      // this group's histogram
    float* wq_s = sm->wq[grp];
    const float* wq_all = reinterpret_cast<const float*>(a.ws + a.L.wq);
    int cur_b = -1, n_b = 0, tiles_b = 0;
    uint32_t tcount = 0;                         // streaming mode: real tiles of cur_b since the last flush
    uint32_t* done_all = reinterpret_cast<uint32_t*>(a.ws + a.L.done);
    uint64_t* segmeta_all = reinterpret_cast<uint64_t*>(a.ws + a.L.segmeta);
    // the count published at the last switch: its result is looked at one switch later,
    // so the atomic's round trip does not hold up the group
    int pend_b = -1;
    uint32_t pend_old = 0, pend_cnt = 0, pend_tiles = 0;
    uint32_t hphase = 0;
    float wr[64];   // the current request's head weights (query scales folded in)
    // the group's four warps meet (bounded: an aborted pass falls through)
    auto grp_sync = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm->hbar[grp]);
      role_wait(sm, &sm->hbar[grp], hphase & 1, a.spin);
      ++hphase;
    };
    // streaming mode: the group's tiles of request b are scored and flushed; the group
    // whose count completes the request hands it to its block's selection
    auto settle = [&]() {
      if (gtid == 0 && pend_b >= 0) {
        if (pend_old + pend_cnt == pend_tiles) queue_push(a, pend_b);
        pend_b = -1;
      }
    };
    // The group's tiles of b are scored and its bins flushed (its four warps met after
    // that): one thread adds their count with release semantics, which orders the whole
    // group's stores and bin atomics before it.  The group whose count completes the
    // request hands it to its block's selection.
    auto publish = [&](int b) {
      if (gtid == 0 && tcount > 0) {
        settle();
        uint32_t old;
        asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(done_all + b), "r"(tcount) : "memory");
        pend_b = b;
        pend_old = old;
        pend_cnt = tcount;
        pend_tiles = static_cast<uint32_t>(tiles_b);
      }
      tcount = 0;
    };
    auto flush = [&](int b) {
      uint32_t* gh = ghist + size_t(b) * kHistStride;
      // coarse bins c = gtid, gtid + 128: the sums of fine bins 16c .. 16c+15 (rotated
      // start, so the lanes of a warp spread over the banks)
#pragma unroll 1
      for (int c = gtid; c < kCoarseBins; c += 128) {
        uint32_t sum = 0;
#pragma unroll
        for (int q = 0; q < 16; ++q) sum += ghs[16 * c + ((q + c) & 15)];
        if (sum) atomicAdd(gh + kHistBins + c, sum);
      }
#pragma unroll 1
      for (int x = gtid; x < kHistBins; x += 128) {
        const uint32_t cnt = ghs[x];
        if (cnt) { atomicAdd(gh + x, cnt); ghs[x] = 0; }
      }
    };
    for (long long i = grp;; i += kGroups) {
      const int ss = static_cast<int>(i % kScaleSlots);
      if (!role_wait(sm, &sm->sfull[ss], (i / kScaleSlots) & 1, a.spin)) break;
      const int2 ti = sm->tinfo[ss];
      const int pmask = sm->smask[ss];
      const float ks = FP8 ? sring[ss * kTileRows + row] : 1.0f;   // FP4: inside the MMA
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm->sempty[ss]);   // one arrival per warp
      if (ti.x < 0) break;
      if (ti.x != cur_b) {
        // request switch: the group is done with the previous request's tiles
        grp_sync();
        if (cur_b >= 0) flush(cur_b);
        if constexpr (!LARGE) {
          grp_sync();
          if (cur_b >= 0) publish(cur_b);
        }
        cur_b = ti.x;
        n_b = cur_b < kReqCache ? sm->nbv[cur_b] : visible(a, cur_b);
        tiles_b = (n_b + kTileRows - 1) / kTileRows;
        if (gtid < 64) wq_s[gtid] = gtid < N ? wq_all[cur_b * 64 + gtid] : 0.f;
        grp_sync();
#pragma unroll
        for (int h = 0; h < 64; ++h) wr[h] = wq_s[h];
      }
      const long long j = static_cast<long long>(ti.y) * kTileRows + row;
      const bool real = ti.y < tiles_b;
      if constexpr (!LARGE) tcount += real ? 1u : 0u;
      const bool valid = real && j < n_b && ((pmask >> (row >> 6)) & 1);
      const int c = static_cast<int>(i % kAccs);
      if (!role_wait(sm, &sm->accfull[c], (i / kAccs) & 1, a.spin)) break;
      tc_fence_after();
      const uint32_t tb = tmem + (static_cast<uint32_t>(sub * 32) << 16) + c * N;
      // Heads 0-31, then 32-63: half the logits in registers at a time (the weights stay
      // in registers for the whole request).  Four independent accumulation chains, two
      // per packed fma (the epilogue's instruction count and latency set part of the
      // streaming pace).
      float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
      float P[32];
      auto release_acc = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->accempty[c]);   // this warp's TMEM reads are done
      };
      if (N >= 32) {
        tmem_ld32(tb, P);
      } else {
        tmem_ld16(tb, *reinterpret_cast<float(*)[16]>(P));
      }
      tmem_wait_ld();
      if (N <= 32) release_acc();
#pragma unroll
      for (int h = 0; h < 32; h += 4) {
        if (h < N) {
          fma2(s0, s1, wr[h], wr[h + 1], fmaxf(P[h], 0.f), fmaxf(P[h + 1], 0.f));
          fma2(s2, s3, wr[h + 2], wr[h + 3], fmaxf(P[h + 2], 0.f), fmaxf(P[h + 3], 0.f));
        }
      }
      if (N > 32) {
        if (N == 64) {
          tmem_ld32(tb + 32, P);
        } else {
          tmem_ld16(tb + 32, *reinterpret_cast<float(*)[16]>(P));
        }
        tmem_wait_ld();
        release_acc();
#pragma unroll
        for (int h = 0; h < 32; h += 4) {
          if (32 + h < N) {
            fma2(s0, s1, wr[32 + h], wr[33 + h], fmaxf(P[h], 0.f), fmaxf(P[h + 1], 0.f));
            fma2(s2, s3, wr[34 + h], wr[35 + h], fmaxf(P[h + 2], 0.f), fmaxf(P[h + 3], 0.f));
          }
        }
      }
      float I = ((s0 + s1) + (s2 + s3)) * ks;   // the key's scale is a positive power of two
      // FP4 index keys keep their scores in bf16 ("DeepSeek-V4.1 Flash", section 10.4)
      if (FP4) I = __bfloat162float(__float2bfloat16_rn(I));
      const uint32_t key = valid ? order_key(I) : 0u;
      if (valid) {
        scores_all[size_t(cur_b) * a.L.n_pad + j] = I;
        atomicAdd(&ghs[key >> (32 - kHistBits)], 1u);
      }
      // largest key of this warp's 32 entries: the selection re-reads only
      // segments that can hold a selected entry
      const uint32_t kmax = __reduce_max_sync(0xFFFFFFFFu, key);
      if constexpr (LARGE) {
        if (lane == 0 && real) segmax_all[size_t(cur_b) * (a.L.n_pad / kSeg) + (j >> 5)] = kmax;
      } else {
        // streaming mode keeps the max with its lane and the bin of the runner-up: a
        // segment with one entry at the threshold needs no second look at its scores
        const int l1 = __ffs(__ballot_sync(0xFFFFFFFFu, key == kmax)) - 1;
        const uint32_t k2 = __reduce_max_sync(0xFFFFFFFFu, lane == l1 ? 0u : key);
        if (lane == 0 && real)
          segmeta_all[size_t(cur_b) * (a.L.n_pad / kSeg) + (j >> 5)] =
              (static_cast<uint64_t>(kmax) << 32) | ((k2 >> (32 - kHistBits)) << 8) | static_cast<uint32_t>(l1);
      }
    }
    grp_sync();
    if (cur_b >= 0) flush(cur_b);
    if constexpr (!LARGE) {
      grp_sync();
      if (cur_b >= 0) publish(cur_b);
      settle();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
  if constexpr (!LARGE) {
    // plain call: this block reads no more query images; once every block is past its
    // stream, the next kernel may start (a following prep waits before clearing)
    if (!a.wait_fresh) grid_dep_launch();
    select_completed<KF>(a);
    if (a.wait_fresh && threadIdx.x == 0) grid_dep_wait();   // complete only after the compressor
    return;
  }

  // ======================================================= phase 2: selection
  // After every request's histogram is complete (the one grid barrier), each request
  // is selected in two steps:
  //  - every block of the request's run takes a slice of its tiles: the threshold bin
  //    T (the bin holding the k-th score) from the request's histogram, the slice's
  //    "hit" segments (largest key in a bin >= T, about one in nine) from the segment
  //    table, their scores copied into shared memory with cp.async, and every entry
  //    in a bin >= T written as a 64-bit (score key, ~index) key, in entry order, to
  //    the slice's own area of the request's key buffer;
  //  - the block that finishes its slice last (a per-request counter) gathers the
  //    slices' keys, radix-selects the exact cut among the keys of bin T (ties ->
  //    smaller index) and writes the selected entries in entry order.
  // This code runs once per launch; its loops stay rolled.
  grid_barrier(sm, gbar, gridDim.x, a.spin);
  const bool aborted = sm->abort;   // uniform: only thread 0 sets it, before the barrier's sync
  grid_dep_launch();   // the next kernel (attention) may be scheduled as blocks retire
  {
    float* s_cache = reinterpret_cast<float*>(stages);                       // the stage ring, 32 fp32 per hit
    uint16_t* s_list = reinterpret_cast<uint16_t*>(qbuf);                     // kSelSegs
    unsigned long long* s_cand = reinterpret_cast<unsigned long long*>(hist);   // kCandCap
    uint16_t* s_cnt = reinterpret_cast<uint16_t*>(sring);                    // kSelSegs + 64
    uint32_t* s_pre = reinterpret_cast<uint32_t*>(sring);                    // slice offsets (final step)
    const int segs_pad = a.L.n_pad / kSeg;
    const int nwarps = kScoreThreads / 32;
    const uint32_t lt_mask = (1u << lane) - 1u;
    const int kCache = kProducers * kStages * kStageBytes / (kSeg * 4);   // hit segments per round
    uint32_t* slc_all = reinterpret_cast<uint32_t*>(a.ws + a.L.slc);
    // block-wide placement: each thread's count -> its exclusive offset; the total
    auto place = [&](uint32_t cnt, uint32_t& tot) -> uint32_t {
      uint32_t incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
      }
      if (lane == 31) sm->part[warp] = incl;
      __syncthreads();
      uint32_t pos = incl - cnt;
      tot = 0;
#pragma unroll 1
      for (int w = 0; w < kScoreThreads / 32; ++w) {
        const uint32_t x = sm->part[w];
        if (w < warp) pos += x;
        tot += x;
      }
      __syncthreads();
      return pos;
    };
    const int nwork = sm->nwork;
    long long C = 0;
    int bnext = 0;
#pragma unroll 1
    for (int w = 0; !aborted; ++w) {
      int b = -1, fb, nbk;
      long long lo, hi, per_b;
      if (nwork >= 0) {
        if (w >= nwork) break;
        const WorkItem wi = sm->work[w];
        b = wi.b;
        lo = wi.lo;
        hi = wi.hi;
        per_b = wi.per;
        fb = wi.fb;
        nbk = wi.nbk;
      } else {
        // more requests than the list holds: the next one whose run holds this block
#pragma unroll 1
        while (bnext < a.B) {
          const int bb = bnext++;
          const long long tb = (visible(a, bb) + kTileRows - 1) / kTileRows;
          const bool mine = block_range(blockIdx.x, gridDim.x, C, tb, total, lo, hi, fb, nbk, per_b);
          C += tb;
          if (mine) {
            b = bb;
            break;
          }
          if (fb > static_cast<int>(blockIdx.x)) bnext = a.B;   // the runs only move further right
        }
        if (b < 0) break;
      }
      const int nb = b < kReqCache ? sm->nbv[b] : visible(a, b);
      const int slice = blockIdx.x - fb;
      const float* sc = scores_all + size_t(b) * a.L.n_pad;
      int32_t* out_idx = a.topk_idx + size_t(b) * a.k;
      float* out_sc = a.topk_score ? a.topk_score + size_t(b) * a.k : nullptr;
      if (nb <= a.k) {
        // every visible entry is selected, in order; the run's first block pads with -1
        const long long jhi = min(hi * kTileRows, static_cast<long long>(nb));
#pragma unroll 1
        for (long long j = lo * kTileRows + threadIdx.x; j < jhi; j += blockDim.x) {
          out_idx[j] = static_cast<int32_t>(j);
          if (out_sc) out_sc[j] = __ldcg(sc + j);
        }
        if (slice == 0) {
#pragma unroll 1
          for (int j = nb + threadIdx.x; j < a.k; j += blockDim.x) {
            out_idx[j] = -1;
            if (out_sc) out_sc[j] = -INFINITY;
          }
        }
        continue;
      }
      if constexpr (LARGE) {
        if (nb <= kFastN) continue;   // one warp selects it, after this loop
      }
      const uint32_t* smx = segmax_all + size_t(b) * segs_pad;
      unsigned long long* kbuf = reinterpret_cast<unsigned long long*>(a.ws + a.L.cand) + size_t(b) * a.L.n_pad;
      const int nseg = (nb + kSeg - 1) / kSeg;
      const long long gs0 = lo * 4, gs1 = min(hi * 4, static_cast<long long>(nseg));
      // the slice's segment table into shared memory, in flight with the threshold loads
      uint32_t* s_seg32 = hist;   // free: the selection keys use it only in the final step
      const bool pre = gs1 - gs0 <= kSelSegs;
      if (pre) {
#pragma unroll 1
        for (long long x = threadIdx.x; x < (gs1 - gs0 + 3) / 4; x += blockDim.x)
          cp_async16(s_seg32 + 4 * x, smx + gs0 + 4 * x);
      }
      // the request's fine histogram into the (free) stage ring, in flight with the
      // coarse loads; threshold_bin waits for both tables
      uint32_t* s_fine = reinterpret_cast<uint32_t*>(stages);
      const uint32_t* ghb = ghist + size_t(b) * kHistStride;
#pragma unroll 1
      for (int x = threadIdx.x; x < kHistBins / 4; x += blockDim.x) cp_async16(s_fine + 4 * x, ghb + 4 * x);
      threshold_bin(sm, ghb, a.k, s_fine);
      const int T = sm->T;
      const uint32_t above = sm->above;
      if (T < 0) {
        // fewer than k binned entries (an earlier error dropped some): no selection
        if (slice == 0) {
#pragma unroll 1
          for (int j = threadIdx.x; j < a.k; j += blockDim.x) {
            out_idx[j] = -1;
            if (out_sc) out_sc[j] = -INFINITY;
          }
        }
        continue;
      }
      // the hit segments of [g0, g0 + ns) (g0 a multiple of 4) into s_list, in order:
      // thread t owns segments 24t .. 24t+23 (six 16-byte loads of the segment table)
      auto hit_list = [&](long long g0, int ns) -> uint32_t {
        constexpr int kOwn = 24;
        static_assert(kOwn * kScoreThreads >= kSelSegs, "every segment of a pass has an owner");
        const int q0 = threadIdx.x * kOwn;
        uint32_t m = 0;
#pragma unroll
        for (int u = 0; u < kOwn / 4; ++u) {
          const int q = q0 + 4 * u;
          if (q < ns) {   // the table's rows are padded to a multiple of 4 segments
            const uint4 x = pre ? *reinterpret_cast<const uint4*>(s_seg32 + (g0 - gs0) + q)
                                : __ldcg(reinterpret_cast<const uint4*>(smx + g0 + q));
            m |= (static_cast<int>(x.x >> (32 - kHistBits)) >= T ? 1u : 0u) << (4 * u);
            m |= (static_cast<int>(x.y >> (32 - kHistBits)) >= T ? 2u : 0u) << (4 * u);
            m |= (static_cast<int>(x.z >> (32 - kHistBits)) >= T ? 4u : 0u) << (4 * u);
            m |= (static_cast<int>(x.w >> (32 - kHistBits)) >= T ? 8u : 0u) << (4 * u);
          }
        }
        if (ns - q0 < kOwn) m &= ns > q0 ? (1u << (ns - q0)) - 1u : 0u;
        uint32_t tot;
        uint32_t pos = place(__popc(m), tot);
#pragma unroll 1
        while (m) {
          const int q = __ffs(m) - 1;
          m &= m - 1;
          s_list[pos++] = static_cast<uint16_t>(q0 + q);
        }
        __syncthreads();
        return tot;
      };
      // ---- the slice: every entry in a bin >= T as a key, in entry order, into
      // kbuf[lo * 128 + ...] (the slice's tiles bound its count).  A warp per hit
      // segment, one entry per lane, four segments per step with their loads first.
      unsigned long long* kout = kbuf + lo * kTileRows;
      uint32_t nk = 0;
#pragma unroll 1
      for (long long gc = gs0; gc < gs1; gc += kSelSegs) {
        const int ns = static_cast<int>(min(static_cast<long long>(kSelSegs), gs1 - gc));
        const uint32_t nhit = hit_list(gc, ns);
#pragma unroll 1
        for (uint32_t h0 = 0; h0 < nhit; h0 += kCache) {
          const uint32_t nh = min(nhit - h0, static_cast<uint32_t>(kCache));
#pragma unroll 1
          for (uint32_t x = threadIdx.x; x < nh * 8; x += blockDim.x)
            cp_async16(s_cache + (x >> 3) * kSeg + (x & 7) * 4,
                       sc + (gc + s_list[h0 + (x >> 3)]) * kSeg + (x & 7) * 4);
          cp_async_wait_all();
          __syncthreads();
          constexpr int kU = 4;
#pragma unroll 1
          for (uint32_t hb = warp * kU; hb < nh; hb += nwarps * kU) {
            float v[kU];
            long long j[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
              const uint32_t h = min(hb + u, nh - 1);
              j[u] = (gc + static_cast<long long>(s_list[h0 + h])) * kSeg + lane;
              v[u] = s_cache[h * kSeg + lane];
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
              const bool f = hb + u < nh && j[u] < nb &&
                             static_cast<int>(order_key(v[u]) >> (32 - kHistBits)) >= T;
              const unsigned m = __ballot_sync(0xFFFFFFFFu, f);
              if (lane == 0 && hb + u < nh) s_cnt[hb + u] = static_cast<uint16_t>(__popc(m));
            }
          }
          if (threadIdx.x == 0) s_cnt[nh] = 0;
          __syncthreads();
          block_exclusive_scan16(sm, s_cnt, static_cast<int>(nh) + 1);
#pragma unroll 1
          for (uint32_t hb = warp * kU; hb < nh; hb += nwarps * kU) {
            float v[kU];
            long long j[kU];
            uint32_t base[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
              const uint32_t h = min(hb + u, nh - 1);
              j[u] = (gc + static_cast<long long>(s_list[h0 + h])) * kSeg + lane;
              v[u] = s_cache[h * kSeg + lane];
              base[u] = s_cnt[h];
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
              const uint32_t key = order_key(v[u]);
              const bool f = hb + u < nh && j[u] < nb && static_cast<int>(key >> (32 - kHistBits)) >= T;
              const unsigned m = __ballot_sync(0xFFFFFFFFu, f);
              if (f)
                kout[nk + base[u] + __popc(m & lt_mask)] =
                    (static_cast<unsigned long long>(key) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(j[u]));
            }
          }
          nk += s_cnt[nh];
          __syncthreads();
        }
      }
      // publish the slice; the block that completes the request's last slice goes on
      __threadfence();   // this thread's key writes, before the count and the arrival
      __syncthreads();
      if (threadIdx.x == 0) {
        slc_all[size_t(b) * kMaxGrid + slice] = nk;
        __threadfence();
        sm->last = atomicAdd(&ctr_all[b * 4 + 1], 1u) == static_cast<uint32_t>(nbk - 1);
        __threadfence();
      }
      __syncthreads();
      if (!sm->last) continue;
      // ---- the final step of request b: slice offsets (a block scan over the run)
      uint32_t tot = 0;
      {
        const int per = (nbk + kScoreThreads - 1) / kScoreThreads;
        const int s0 = min(nbk, static_cast<int>(threadIdx.x) * per), s1 = min(nbk, s0 + per);
        uint32_t cnt = 0;
#pragma unroll 1
        for (int q = s0; q < s1; ++q) cnt += __ldcg(slc_all + size_t(b) * kMaxGrid + q);
        uint32_t pos = place(cnt, tot);
#pragma unroll 1
        for (int q = s0; q < s1; ++q) {
          s_pre[q] = pos;
          pos += __ldcg(slc_all + size_t(b) * kMaxGrid + q);
        }
        if (threadIdx.x == 0) s_pre[nbk] = tot;
        __syncthreads();
      }
      const uint32_t nkt = tot;
      // the first kCandCap keys into shared memory (8-byte cp.async, all in flight)
#pragma unroll 1
      for (int q = 0; q < nbk; ++q) {
        const uint32_t p0 = s_pre[q], n = s_pre[q + 1] - p0;
        if (p0 >= static_cast<uint32_t>(kCandCap)) break;
        const unsigned long long* src = kbuf + q * per_b * kTileRows;
#pragma unroll 1
        for (uint32_t i = threadIdx.x; i < n && p0 + i < static_cast<uint32_t>(kCandCap); i += blockDim.x)
          cp_async8(s_cand + p0 + i, src + i);
      }
      cp_async_wait_all();
      __syncthreads();
      // key x of the request, in entry order (past kCandCap: found in its slice's area)
      auto key_at = [&](uint32_t x) -> unsigned long long {
        if (x < static_cast<uint32_t>(kCandCap)) return s_cand[x];
        int l = 0, r = nbk - 1;   // the slice q with s_pre[q] <= x < s_pre[q + 1]
        while (l < r) {
          const int m = (l + r + 1) >> 1;
          if (s_pre[m] <= x) l = m; else r = m - 1;
        }
        return __ldcg(kbuf + l * per_b * kTileRows + (x - s_pre[l]));
      };
      // ---- the cut: the need-th largest key in bin T, by 12-bit digits (bits 51-40,
      // 39-28, 27-16, 15-4, then 3-0; with a few hundred keys in bin T the first digit
      // usually decides).  Keys above T never match the prefix, so only bin T's keys
      // are counted.  The digit histogram uses the stage ring (free by now).
      uint32_t* dh = reinterpret_cast<uint32_t*>(stages);   // 4,096 bins
      if (threadIdx.x == 0) {
        sm->need = min(static_cast<uint32_t>(a.k) - above, nkt > above ? nkt - above : 0u);
        sm->done = 0;
        sm->mask = ~0ull << 52;
        sm->prefix = static_cast<unsigned long long>(T) << 52;
      }
      __syncthreads();
#pragma unroll 1
      for (int shift = 40; shift >= 0; shift = shift >= 12 ? shift - 12 : (shift > 0 ? 0 : -1)) {
        if (sm->done || sm->need == 0) break;
        const int width = shift >= 4 ? 12 : 4;
        const int nd = 1 << width;
        const unsigned long long dmask = static_cast<unsigned long long>(nd - 1) << shift;
#pragma unroll 1
        for (int x = threadIdx.x; x < nd; x += blockDim.x) dh[x] = 0;
        __syncthreads();
        const unsigned long long pm = sm->mask, pp = sm->prefix;
#pragma unroll 1
        for (uint32_t x = threadIdx.x; x < nkt; x += blockDim.x) {
          const unsigned long long key = key_at(x);
          if ((key & pm) == pp) atomicAdd(&dh[(key & dmask) >> shift], 1u);
        }
        __syncthreads();
        // thread t owns digits nd-1-per*t .. (from the top); the one whose run holds
        // the need-th key walks it
        const int per = (nd + kScoreThreads - 1) / kScoreThreads;
        const int d0 = nd - 1 - per * static_cast<int>(threadIdx.x);
        uint32_t sum = 0;
#pragma unroll 1
        for (int q = 0; q < per && d0 - q >= 0; ++q) sum += dh[d0 - q];
        // read before place(): its barriers order every thread's read before the
        // owning thread's update below, so no thread can see the updated count
        const uint32_t need = sm->need;
        uint32_t tot;
        const uint32_t before = place(sum, tot);
        if (sum > 0 && before < need && before + sum >= need) {
          uint32_t accd = before;
          int d = d0;
#pragma unroll 1
          for (int q = 0; q < per && d0 - q >= 0; ++q) {
            const uint32_t y = dh[d0 - q];
            if (accd + y >= need) { d = d0 - q; break; }
            accd += y;
          }
          sm->need = need - accd;
          sm->prefix = pp | (static_cast<unsigned long long>(d) << shift);
          sm->mask = pm | dmask;
          if (dh[d] == need - accd) sm->done = 1;
        }
        __syncthreads();
        if (shift == 0) break;
      }
      // ---- the output: selected  <=>  (key64 & pm) >= pp, in entry order
      {
        const unsigned long long pm = sm->mask, pp = sm->prefix;
        const uint32_t per = (nkt + kScoreThreads - 1) / kScoreThreads;
        const uint32_t x0 = min(nkt, threadIdx.x * per), x1 = min(nkt, x0 + per);
        uint32_t cnt = 0;
#pragma unroll 1
        for (uint32_t x = x0; x < x1; ++x) cnt += (key_at(x) & pm) >= pp ? 1u : 0u;
        uint32_t nsel;
        uint32_t pos = place(cnt, nsel);
#pragma unroll 1
        for (uint32_t x = x0; x < x1; ++x) {
          const unsigned long long key = key_at(x);
          if ((key & pm) < pp) continue;
          if (pos < static_cast<uint32_t>(a.k)) {
            out_idx[pos] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(key));
            if (out_sc) out_sc[pos] = from_order_key(static_cast<uint32_t>(key >> 32));
          }
          ++pos;
        }
        // fewer than k selected (only after an error): -1 after them
#pragma unroll 1
        for (uint32_t x = nsel + threadIdx.x; x < static_cast<uint32_t>(a.k); x += blockDim.x) {
          out_idx[x] = -1;
          if (out_sc) out_sc[x] = -INFINITY;
        }
      }
      __syncthreads();
    }
    if constexpr (LARGE) {
      // Requests of more than k and at most kFastN visible entries (e.g. one prompt query
      // each in prefill): one warp selects each from its scores in the workspace, the
      // block's such requests taken by its warps in turn (a request belongs to the first
      // block of its run).  Radix select on the order keys, four 8-bit digits from the
      // top: the k-th largest key K and how many of the entries equal to K are taken (the
      // ones of smallest index); then every entry above K and those, in entry order.
      __syncthreads();   // the stage ring is free
      uint32_t* wkeys = reinterpret_cast<uint32_t*>(stages) + warp * (kFastN + 256);
      uint32_t* whist = wkeys + kFastN;
      const unsigned full = 0xFFFFFFFFu;
      int f = 0;
      long long C2 = 0;
      int bnext2 = 0;
#pragma unroll 1
      for (int w = 0; !aborted; ++w) {
        int b = -1, fb = 0, nbk = 0;
        long long lo = 0, hi = 0, per_b = 0;
        if (nwork >= 0) {
          if (w >= nwork) break;
          const WorkItem wi = sm->work[w];
          b = wi.b;
          fb = wi.fb;
        } else {
#pragma unroll 1
          while (bnext2 < a.B) {
            const int bb = bnext2++;
            const long long tb = (visible(a, bb) + kTileRows - 1) / kTileRows;
            const bool mine = block_range(blockIdx.x, gridDim.x, C2, tb, total, lo, hi, fb, nbk, per_b);
            C2 += tb;
            if (mine) {
              b = bb;
              break;
            }
            if (fb > static_cast<int>(blockIdx.x)) bnext2 = a.B;
          }
          if (b < 0) break;
        }
        const int nb = b < kReqCache ? sm->nbv[b] : visible(a, b);
        if (nb <= a.k || nb > kFastN || fb != static_cast<int>(blockIdx.x)) continue;
        if ((f++ % nwarps) != warp) continue;
        const float* sc = scores_all + size_t(b) * a.L.n_pad;
        int32_t* out_idx = a.topk_idx + size_t(b) * a.k;
        float* out_sc = a.topk_score ? a.topk_score + size_t(b) * a.k : nullptr;
#pragma unroll 1
        for (int j = lane; j < nb; j += 32) wkeys[j] = order_key(__ldcg(sc + j));
        uint32_t prefix = 0, pmask = 0, need = static_cast<uint32_t>(a.k);
#pragma unroll 1
        for (int shift = 24; shift >= 0; shift -= 8) {
#pragma unroll
          for (int x = lane; x < 256; x += 32) whist[x] = 0;
          __syncwarp();
#pragma unroll 1
          for (int j = lane; j < nb; j += 32) {
            const uint32_t key = wkeys[j];
            if ((key & pmask) == prefix) atomicAdd(&whist[(key >> shift) & 255u], 1u);
          }
          __syncwarp();
          // lane l owns digits 255 - 8l down to 248 - 8l
          uint32_t sum = 0;
#pragma unroll
          for (int q = 0; q < 8; ++q) sum += whist[255 - 8 * lane - q];
          uint32_t incl = sum;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const uint32_t x = __shfl_up_sync(full, incl, o);
            if (lane >= o) incl += x;
          }
          // never empty: the keys under the prefix number at least need
          const unsigned hit = __ballot_sync(full, incl >= need);
          const int src = __ffs(hit) - 1;
          uint32_t d = 0, acc = incl - sum;
          if (lane == src) {
#pragma unroll 1
            for (int q = 0; q < 8; ++q) {
              const uint32_t c = whist[255 - 8 * lane - q];
              if (acc + c >= need) {
                d = static_cast<uint32_t>(255 - 8 * lane - q);
                break;
              }
              acc += c;
            }
          }
          d = __shfl_sync(full, d, src);
          acc = __shfl_sync(full, acc, src);
          need -= acc;
          prefix |= d << shift;
          pmask |= 255u << shift;
          __syncwarp();
        }
        uint32_t pos = 0, eq_seen = 0;
#pragma unroll 1
        for (int base = 0; base < nb; base += 32) {
          const int j = base + lane;
          const uint32_t key = j < nb ? wkeys[j] : 0u;
          const bool eq = j < nb && key == prefix;
          const unsigned em = __ballot_sync(full, eq);
          const bool take = (j < nb && key > prefix) || (eq && eq_seen + __popc(em & lt_mask) < need);
          const unsigned tm = __ballot_sync(full, take);
          if (take) {
            const uint32_t p = pos + __popc(tm & lt_mask);
            out_idx[p] = j;
            if (out_sc) out_sc[p] = from_order_key(key);
          }
          pos += __popc(tm);
          eq_seen += __popc(em);
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// host helpers
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

template <int KF>
size_t score_smem_bytes() {
  using F = KeyFmt<KF>;
  static_assert(kSelSegs * 2 <= F::kQBuf, "the hit list reuses the query images");
  static_assert(kCandCap * 8 <= kGroups * kHistBins * 4, "the candidates reuse the histograms");
  static_assert(kProducers * F::kStages * F::kStageBytes >= kMetaSegs * 8 + kSelCand * 8,
                "the selection's metadata and candidates reuse the stage ring");
  return 1024 + kProducers * F::kStages * F::kStageBytes + F::kQBuf + kGroups * kHistBins * 4 +
         kScaleSlots * kTileRows * 4 + kScratch16 * 2 + sizeof(ScoreSmem);
}

// Cooperative launch of the score kernel: the selection phases meet at grid
// barriers, so the grid is the number of blocks that fit on the GPU at once.
template <int KF, bool LARGE>
cudaError_t launch_score(const CUtensorMap& tmap, const IndexArgs& a, cudaStream_t stream) {
  const size_t smem = score_smem_bytes<KF>();
  cudaError_t e = cudaFuncSetAttribute(index_score_kernel<KF, LARGE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, index_score_kernel<KF, LARGE>, kScoreThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  // one block per SM: it allocates all 512 TMEM columns and most of shared memory
  const int grid = a.grid;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kScoreThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  if constexpr (!LARGE) {
    // streaming mode: no grid barrier, so no co-residency is needed; blocks are placed
    // as SMs free up (beside a compressor that is still running, in a fused step)
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, index_score_kernel<KF, LARGE>, tmap, a);
  }
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  // A cooperative launch that is also a programmatic dependent: whether the runtime
  // takes the pair is learnt from the first launch made outside a stream capture
  // (a failed launch inside one could end the capture); until then, and if it
  // refuses, the launch is cooperative only.
  static std::atomic<int> pdl_ok{-1};
  int ok = pdl_ok.load(std::memory_order_relaxed);
  if (ok < 0) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) ok = 0;
  }
  if (ok != 0) {
    cfg.numAttrs = 2;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, index_score_kernel<KF, LARGE>, tmap, a);
    if (e == cudaSuccess) {
      pdl_ok.store(1, std::memory_order_relaxed);
      return e;
    }
    if (ok == 1) return e;   // the pair was taken before: a real failure
    cudaGetLastError();      // the refused pair: clear it and launch cooperative only
    pdl_ok.store(0, std::memory_order_relaxed);
  }
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, index_score_kernel<KF, LARGE>, tmap, a);
}

}  // namespace

size_t index_workspace_bytes(int B, int n_max, int Hi, int k) {
  (void)Hi;
  return ws_layout(B, n_max, k).total;
}

namespace {

struct IndexLaunch {
  IndexArgs a;
  CUtensorMap tmap;
};

cudaError_t index_setup(IndexLaunch& L, const void* q_idx, const float* w, const cskv_paged& keys,
                        const int32_t* ctx_len, int B, int Hi, int ratio, int k, int max_ctx_len,
                        int32_t* topk_idx, float* topk_score, void* workspace) {
  IndexArgs& a = L.a;
  a = IndexArgs{};
  a.q = static_cast<const uint8_t*>(q_idx);
  a.w = w;
  a.keys = keys;
  a.ctx_len = ctx_len;
  a.B = B;
  a.Hi = Hi;
  a.N = Hi <= 16 ? 16 : (Hi + 15) / 16 * 16;
  a.ratio = ratio;
  a.k = k;
  a.n_max = max_ctx_len / ratio;
  a.kfmt = keys.fmt == CSKV_FMT_FP8_E4M3_ROWSCALE_PAGESPLIT          ? kKfFp8
           : keys.fmt == CSKV_FMT_FP4_E2M1_E8M0_HADAMARD_PAGESPLIT ? kKfFp4
                                                                    : kKfBf16;
  a.topk_idx = topk_idx;
  a.topk_score = topk_score;
  a.ws = static_cast<uint8_t*>(workspace);
  a.L = ws_layout(B, a.n_max, k);
  a.spin = spin_limit();
  a.grid = sm_count();   // the score kernel runs one block per SM
  if (a.grid > kMaxGrid) a.grid = kMaxGrid;

  auto enc = encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  cuuint64_t dims[3], strides[2];
  cuuint32_t box[3], estr[3] = {1, 1, 1};
  CUtensorMapDataType dt;
  CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B;
  if (a.kfmt == kKfFp8) {
    dims[0] = 128; strides[0] = 128;
    box[0] = 128;
    dt = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  } else if (a.kfmt == kKfFp4) {
    dims[0] = 64; strides[0] = 64;   // 64 code bytes per key
    box[0] = 64;
    dt = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    swz = CU_TENSOR_MAP_SWIZZLE_64B;
  } else {
    dims[0] = 128; strides[0] = 256;
    box[0] = 64;
    dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  }
  dims[1] = 64;
  dims[2] = static_cast<cuuint64_t>(keys.num_pages);
  strides[1] = static_cast<cuuint64_t>(keys.page_bytes);
  box[1] = 64;
  box[2] = 1;
  CUresult r = enc(&L.tmap, dt, 3, keys.pool, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t index_launch_prep(const IndexLaunch& L, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.a.B);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, index_prep_kernel, L.a);
}

// Streaming mode (per-request selection as requests complete, no grid barrier) needs
// the batch's visible counts in shared memory and each request's segment table in the
// fast selection's shared-memory area; larger batches or requests take the cooperative
// kernel.
bool streaming_mode(const IndexArgs& a) {
  return a.B <= kReqCache && static_cast<long long>(a.n_max) <= static_cast<long long>(kMetaSegs) * kSeg;
}

cudaError_t index_launch_score(const IndexLaunch& L, cudaStream_t stream) {
  const IndexArgs& a = L.a;
  // streaming mode for batches of at most kReqCache requests of at most kMetaSegs
  // segments each (the fast selection keeps a request's segment table in shared memory);
  // the cooperative kernel (grid barrier, selection sliced over the grid) otherwise
  // (grid barrier, sliced selection) above that, whatever the key format
  if (!streaming_mode(a)) {
    if (a.kfmt == kKfFp8) return launch_score<kKfFp8, true>(L.tmap, a, stream);
    if (a.kfmt == kKfFp4) return launch_score<kKfFp4, true>(L.tmap, a, stream);
    return launch_score<kKfBf16, true>(L.tmap, a, stream);
  }
  if (a.kfmt == kKfFp8) return launch_score<kKfFp8, false>(L.tmap, a, stream);
  if (a.kfmt == kKfFp4) return launch_score<kKfFp4, false>(L.tmap, a, stream);
  return launch_score<kKfBf16, false>(L.tmap, a, stream);
}

}  // namespace

cudaError_t launch_index_topk(const void* q_idx, const float* w, const cskv_paged& keys,
                              const int32_t* ctx_len, int B, int Hi, int ratio, int k,
                              int max_ctx_len, int32_t* topk_idx, float* topk_score,
                              void* workspace, cudaStream_t stream) {
  IndexLaunch L;
  cudaError_t e = index_setup(L, q_idx, w, keys, ctx_len, B, Hi, ratio, k, max_ctx_len, topk_idx, topk_score,
                              workspace);
  if (e != cudaSuccess) return e;
  e = index_launch_prep(L, stream);
  if (e != cudaSuccess) return e;
  cudaEvent_t ev_begin, ev_end;
  timing_events(&ev_begin, &ev_end);
  record_timing_branch(ev_begin, stream);
  e = index_launch_score(L, stream);
  record_timing_branch(ev_end, stream);
  return e;
}

cudaError_t launch_index_topk_fused(const void* q_idx, const float* w, const cskv_paged& keys,
                                    const int32_t* ctx_len, int B, int Hi, int ratio, int k, int max_ctx_len,
                                    int32_t* topk_idx, float* topk_score, void* workspace,
                                    const cskv_compress_job* jobs, int njobs, cudaStream_t stream,
                                    const uint32_t** ready) {
  IndexLaunch L;
  cudaError_t e = index_setup(L, q_idx, w, keys, ctx_len, B, Hi, ratio, k, max_ctx_len, topk_idx, topk_score,
                              workspace);
  if (e != cudaSuccess) return e;
  const bool streaming = streaming_mode(L.a);
  L.a.fused = 1;
  if (streaming) {
    // the score kernel overlaps the compressor: it waits for it only before the index
    // keys that the jobs writing into this key cache produce
    L.a.wait_fresh = 1;
    for (int j = 0; j < njobs; ++j) {
      if (jobs[j].out.pool != keys.pool || L.a.nfresh >= 4) continue;
      L.a.fresh_req[L.a.nfresh] = jobs[j].req;
      L.a.fresh_first[L.a.nfresh] = jobs[j].first_entry;
      L.a.fresh_S[L.a.nfresh] = jobs[j].S;
      ++L.a.nfresh;
    }
  }
  // prep, compressor (a programmatic dependent of the prep), score kernel (of the compressor)
  e = index_launch_prep(L, stream);
  if (e != cudaSuccess) return e;
  cudaEvent_t ev_begin, ev_end;
  timing_events(&ev_begin, &ev_end);
  record_timing_branch(ev_begin, stream);
  if (njobs > 0) {
    e = launch_compress_many(jobs, njobs, stream, true);
    if (e != cudaSuccess) return e;
  }
  e = index_launch_score(L, stream);
  record_timing_branch(ev_end, stream);
  if (ready) *ready = streaming ? reinterpret_cast<const uint32_t*>(L.a.ws + L.a.L.ready) : nullptr;
  return e;
}

unsigned int take_err_index() { return take_dev_err(); }

// ---------------------------------------------------------------------------
// Scratch for cskv_index_topk_noalloc: callers that cannot allocate device
// memory get the indexer's workspace from this fixed array instead.  It lives
// in every GPU context that loads the library, for the life of the process.
// ---------------------------------------------------------------------------
static __device__ __align__(256) uint8_t g_noalloc_scratch[CSKV_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch in the current device's context.  Host code
// must not use the symbol itself (it is a host-side stand-in, not a device address).
// The address is looked up on every call, with the call's device current: the lookup
// allocates nothing, and a cached address would outlive a cudaDeviceReset, after
// which the context (and the array's place in it) is new.
static void* noalloc_scratch_address(cudaError_t* err) {
  void* p = nullptr;
  *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  return *err == cudaSuccess ? p : nullptr;
}

cudaError_t launch_index_topk_noalloc(const void* q_idx, const float* w, const cskv_paged& keys,
                                      const int32_t* ctx_len, int B, int Hi, int ratio, int k,
                                      int max_ctx_len, int32_t* topk_idx, float* topk_score,
                                      cudaStream_t stream) {
  cudaError_t err = cudaSuccess;
  void* scratch = noalloc_scratch_address(&err);
  if (scratch == nullptr) return err;
  return launch_index_topk(q_idx, w, keys, ctx_len, B, Hi, ratio, k, max_ctx_len, topk_idx, topk_score,
                           scratch, stream);
}

}  // namespace cskv
