// Lightning indexer + top-k (cskv_index_topk).
//
// "DeepSeek-V4 deep dive", section 5.2: I_{b,j} = sum_h w_h ReLU(q_h . k_j) over
// the visible entries j < floor(ctx_len / ratio), one 128-d key shared by all
// indexer heads; the selector keeps min(k, n) entries (section 5.3).
//
// GB300 design (HBM-bound: at 1M context the keys are 34.6 MB per query):
//  1. index_prep_kernel   codes each request's queries (e4m3, one e8m0 scale per
//     head) into the image of a 128-byte-swizzled shared-memory tile, folds the
//     head scale into the head weight (ReLU(c x) = c ReLU(x) for c > 0) and
//     clears the request's histogram, counters and the grid-barrier word.
//  2. index_score_kernel  persistent and cooperative, two blocks per SM (one
//     TMA-issuing thread per block cannot keep enough copies in flight on its
//     own; two per SM can), warp-specialised:
//       warp 0     streams the 64-row key pages with TMA (3-D tensor map over
//                  the page pool, 128-byte swizzle) into a 4-stage ring, and
//                  their fp32 row scales with bulk copies into a ring that the
//                  epilogue releases;
//       warp 1     issues tcgen05 MMAs: M = 128 entries, N = heads, K = 128 in
//                  four K = 32 e4m3 x e4m3 steps into one fp32 TMEM
//                  accumulator (the key's single scale is applied afterwards),
//                  four accumulators in flight;
//       warps 2-5  read the accumulator with tcgen05.ld (one TMEM lane = one
//                  entry), apply ReLU and the head weights, sum the heads
//                  inside one thread, multiply by the key's scale, write the
//                  fp32 score and bin its order-preserving key into a
//                  4,096-bin shared histogram.
//     Then, behind a bounded grid barrier, every block finds each request's
//     threshold bin (the bin holding the k-th score), emits its own entries
//     above it and stages the ones in it; behind a second barrier the block
//     owning request b radix-selects the remainder among those 64-bit
//     (score, ~index) keys (ties -> smaller index), sorts the k indices and
//     writes indices and scores.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "codec.cuh"
#include "internal.h"

namespace cskv {

namespace {

constexpr int kHistBits = 12;
constexpr int kHistBins = 1 << kHistBits;
constexpr int kTileRows = 128;
constexpr int kStagesFp8 = 4;        // 16 KiB stages
constexpr int kStagesBf16 = 2;       // 32 KiB stages
constexpr int kAccs = 4;             // TMEM accumulators in flight
constexpr int kScaleSlots = 8;       // ring of per-tile scale rows (2 pages x 64 fp32)
constexpr int kScoreThreads = 192;   // warp 0 producer, warp 1 MMA, warps 2-5 epilogue
constexpr int kCandCap = 4096;       // per-block staging of threshold-bin candidates
constexpr int kMaxK = 2048;
constexpr int kQImageFp8 = 8192;     // e4m3 [64 rows][128 B]
constexpr int kQImageBf16 = 16384;   // bf16 [2 chunks][64 rows][128 B]
constexpr int kQSlot = 16384;        // per request in the workspace

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
  size_t scores, cand, qimg, wq, hist, ctr, sel, gbar, total;
  int n_pad;
};

__host__ __device__ inline WsLayout ws_layout(int B, int n_max, int k) {
  WsLayout L;
  L.n_pad = (n_max + kTileRows - 1) / kTileRows * kTileRows;
  if (L.n_pad == 0) L.n_pad = kTileRows;
  size_t o = 0;
  L.scores = o; o = align256(o + size_t(B) * L.n_pad * 4);
  L.cand = o;   o = align256(o + size_t(B) * L.n_pad * 8);
  L.qimg = o;   o = align256(o + size_t(B) * kQSlot);
  L.wq = o;     o = align256(o + size_t(B) * 64 * 4);
  L.hist = o;   o = align256(o + size_t(B) * kHistBins * 4);
  L.ctr = o;    o = align256(o + size_t(B) * 4 * 4);
  L.sel = o;    o = align256(o + size_t(B) * k * 4);
  L.gbar = o;   o = align256(o + 16);
  L.total = o;
  return L;
}

// order-preserving map of an fp32 score to uint32 (larger score -> larger key)
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct IndexArgs {
  const uint8_t* q;          // bf16 [B, Hi, 128]
  const float* w;            // [B, Hi]
  cskv_paged keys;
  const int32_t* ctx_len;
  int B, Hi, N, ratio, k, n_max;
  int fp8;                   // 1: page-split FP8 keys, 0: bf16 keys
  int32_t* topk_idx;
  float* topk_score;
  uint8_t* ws;
  WsLayout L;
  unsigned long long spin;
};

__device__ __forceinline__ int visible(const IndexArgs& a, int b) {
  long long c = a.ctx_len[b];
  long long n = c / a.ratio;
  if (c < 0 || n > a.n_max) {
    set_err(CSKV_ERR_BOUNDS);
    n = c < 0 ? 0 : a.n_max;
  }
  return static_cast<int>(n);
}

// ---------------------------------------------------------------------------
// 1. prep: query image, folded head weights, histogram / counters / barrier cleared
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) index_prep_kernel(const IndexArgs a) {
  const int b = blockIdx.x;
  uint8_t* img = a.ws + a.L.qimg + size_t(b) * kQSlot;
  float* wq = reinterpret_cast<float*>(a.ws + a.L.wq) + b * 64;
  uint32_t* hist = reinterpret_cast<uint32_t*>(a.ws + a.L.hist) + size_t(b) * kHistBins;
  uint32_t* ctr = reinterpret_cast<uint32_t*>(a.ws + a.L.ctr) + b * 4;
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) hist[i] = 0;
  if (threadIdx.x < 4) ctr[threadIdx.x] = 0;
  if (b == 0 && threadIdx.x == 0) *reinterpret_cast<uint32_t*>(a.ws + a.L.gbar) = 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int h = warp + 8 * i;
    if (h >= a.N) break;
    if (a.fp8) {
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
}

// ---------------------------------------------------------------------------
// 2. score kernel (+ fused selection)
// ---------------------------------------------------------------------------
struct ScoreSmem {
  uint64_t full[kStagesFp8], empty[kStagesFp8];
  uint64_t accfull[kAccs], accempty[kAccs];
  uint64_t qfull[2], qempty[2];
  uint64_t sfull[kScaleSlots], sempty[kScaleSlots];
  uint64_t drain;
  uint64_t hbar;                   // epilogue warps meet here at a request switch
  uint32_t tmem_base;
  volatile int abort;
  int smask[kScaleSlots];          // per tile: bit p = page p of the tile was loaded
  int ptab[64];                    // producer's prefetched page ids of its current request
  __align__(16) float wq[64];      // folded head weights of the epilogue's current request
  // selection phases
  uint32_t cnt[2];
  uint32_t base[2];
  int T;
  uint32_t above;
  uint32_t need, done, out;
  unsigned long long prefix, mask;
  uint32_t part[256];
  uint32_t dh[256];
};

// Walks the global tile sequence [start, end) over requests (tiles of request b
// are ceil(n_b / 128)); every role keeps its own walker.
struct TileWalker {
  int b, t, tiles_b, n_b;
  long long g, end;
  __device__ void init(const IndexArgs& a, long long start, long long end_) {
    g = start;
    end = end_;
    long long acc = 0;
    t = 0;
    n_b = 0;
    tiles_b = 0;
    for (b = 0; b < a.B; ++b) {
      n_b = visible(a, b);
      tiles_b = (n_b + kTileRows - 1) / kTileRows;
      if (start < acc + tiles_b) { t = static_cast<int>(start - acc); return; }
      acc += tiles_b;
    }
  }
  __device__ bool valid() const { return g < end; }
  // advance; returns true if the request changed
  __device__ bool next(const IndexArgs& a) {
    ++g;
    if (g >= end) return false;
    if (++t < tiles_b) return false;
    t = 0;
    do {
      ++b;
      n_b = visible(a, b);
      tiles_b = (n_b + kTileRows - 1) / kTileRows;
    } while (tiles_b == 0 && b < a.B - 1);
    return true;
  }
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
__device__ void grid_barrier(ScoreSmem* sm, uint32_t* counter, uint32_t target, unsigned long long limit) {
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
// bins > T; T = -1 if the histogram holds fewer than k entries.  Whole block.
__device__ void threshold_bin(ScoreSmem* sm, const uint32_t* ghist, int k) {
  for (int t = threadIdx.x; t < 256; t += blockDim.x) {
    uint32_t hb[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) hb[i] = __ldcg(ghist + t * 16 + i);
    uint32_t loc = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) loc += hb[i];
    sm->part[t] = loc;
  }
  __syncthreads();
  const int lane = threadIdx.x;
  if (lane < 32) {
    // lane l owns parts 255-8l .. 248-8l (from the top)
    uint32_t loc[8], sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) { loc[i] = sm->part[255 - 8 * lane - i]; sum += loc[i]; }
    uint32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    const uint32_t excl = incl - sum;
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, incl >= static_cast<uint32_t>(k));
    if (hit == 0) {
      if (lane == 0) { sm->T = -1; sm->above = 0; }
    } else if (lane == __ffs(hit) - 1) {
      uint32_t acc = excl;
      int u = 255 - 8 * lane - 7;
      for (int i = 0; i < 8; ++i) {
        if (acc + loc[i] >= static_cast<uint32_t>(k)) { u = 255 - 8 * lane - i; break; }
        acc += loc[i];
      }
      uint32_t hb[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) hb[i] = __ldcg(ghist + u * 16 + i);   // one round trip
      int T = u * 16;
#pragma unroll
      for (int i = 15; i >= 0; --i) {
        if (acc + hb[i] >= static_cast<uint32_t>(k)) { T = u * 16 + i; break; }
        acc += hb[i];
      }
      sm->T = T;
      sm->above = acc;
    }
  }
  __syncthreads();
}

template <int FP8>
__global__ void __launch_bounds__(kScoreThreads, 2)
    index_score_kernel(const __grid_constant__ CUtensorMap tmap, const IndexArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned carve-up
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int kStageBytes = FP8 ? kTileRows * 128 : kTileRows * 256;
  constexpr int kStages = FP8 ? kStagesFp8 : kStagesBf16;
  constexpr int kQImage = FP8 ? kQImageFp8 : kQImageBf16;
  uint8_t* stages = base;
  uint8_t* qbuf = stages + kStages * kStageBytes;                         // 2 x kQImage
  uint32_t* hist = reinterpret_cast<uint32_t*>(qbuf + 2 * kQImage);      // 4096 bins
  float* sring = reinterpret_cast<float*>(hist + kHistBins);             // kScaleSlots x 128 fp32
  ScoreSmem* sm = reinterpret_cast<ScoreSmem*>(sring + kScaleSlots * kTileRows);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = a.N;
  float* scores_all = reinterpret_cast<float*>(a.ws + a.L.scores);
  uint32_t* ghist = reinterpret_cast<uint32_t*>(a.ws + a.L.hist);
  uint32_t* ctr_all = reinterpret_cast<uint32_t*>(a.ws + a.L.ctr);
  uint32_t* gbar = reinterpret_cast<uint32_t*>(a.ws + a.L.gbar);

  // work range of this block
  long long total = 0;
  for (int b = 0; b < a.B; ++b) total += (visible(a, b) + kTileRows - 1) / kTileRows;
  const long long per = (total + gridDim.x - 1) / gridDim.x;
  const long long start = min(total, per * blockIdx.x);
  const long long end = min(total, start + per);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) { mbar_init(&sm->full[s], 1); mbar_init(&sm->empty[s], 1); }
    for (int c = 0; c < kAccs; ++c) { mbar_init(&sm->accfull[c], 1); mbar_init(&sm->accempty[c], 4); }
    for (int c = 0; c < 2; ++c) { mbar_init(&sm->qfull[c], 1); mbar_init(&sm->qempty[c], 1); }
    for (int s = 0; s < kScaleSlots; ++s) { mbar_init(&sm->sfull[s], 1); mbar_init(&sm->sempty[s], 4); }
    mbar_init(&sm->drain, 1);
    mbar_init(&sm->hbar, 4);
    sm->abort = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) hist[i] = 0;
  uint32_t ncols = 32;
  while (ncols < static_cast<uint32_t>(kAccs * N)) ncols <<= 1;
  if (warp == 1) tmem_alloc(&sm->tmem_base, ncols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;

  // ======================================================= phase 1: scores
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && start < end) {
      prefetch_tmap(&tmap);
      TileWalker tw;
      tw.init(a, start, end);
      long long issued = 0;
      int nreq = 0;
      bool need_q = true;
      int pt_b = -1;           // request and first logical page of sm->ptab
      long long pt_lp = 0;
      while (tw.valid()) {
        if (need_q) {
          // query image of the new request into buffer nreq % 2
          const int qb = nreq & 1;
          if (nreq >= 2 && !role_wait(sm, &sm->qempty[qb], ((nreq >> 1) - 1) & 1, a.spin)) break;
          mbar_expect_tx(&sm->qfull[qb], kQImage);
          bulk_g2s(qbuf + qb * kQImage, a.ws + a.L.qimg + size_t(tw.b) * kQSlot, kQImage, &sm->qfull[qb]);
          ++nreq;
          need_q = false;
        }
        const int s = static_cast<int>(issued % kStages);
        const long long round = issued / kStages;
        if (round > 0 && !role_wait(sm, &sm->empty[s], (round - 1) & 1, a.spin)) break;
        const int ss = static_cast<int>(issued % kScaleSlots);
        const long long su = issued / kScaleSlots;
        if (su > 0 && !role_wait(sm, &sm->sempty[ss], (su - 1) & 1, a.spin)) break;
        uint8_t* dst = stages + s * kStageBytes;
        uint32_t bytes = 0;
        int pages[2] = {-1, -1};
        const long long lp0 = static_cast<long long>(tw.t) * 2;
        if (tw.b != pt_b || lp0 < pt_lp || lp0 + 1 >= pt_lp + 64) {
          // refill: 64 page ids of this request, two batches of 32 loads in flight
          pt_b = tw.b;
          pt_lp = lp0;
          const int32_t* bt = a.keys.block_table + static_cast<long long>(tw.b) * a.keys.max_pages;
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            int ids[32];
#pragma unroll
            for (int u = 0; u < 32; ++u) {
              const long long lp = lp0 + 32 * h2 + u;
              ids[u] = (lp * kPageRows < tw.n_b && lp < a.keys.max_pages) ? bt[lp] : -2;
            }
#pragma unroll
            for (int u = 0; u < 32; ++u) sm->ptab[32 * h2 + u] = ids[u];
          }
        }
        for (int pg = 0; pg < 2; ++pg) {
          const long long lp = lp0 + pg;
          if (lp * kPageRows >= tw.n_b) continue;
          if (lp >= a.keys.max_pages) { set_err(CSKV_ERR_BOUNDS); continue; }
          const int pid = sm->ptab[lp - pt_lp];
          if (pid < 0 || pid >= a.keys.num_pages) { set_err(CSKV_ERR_BOUNDS); continue; }
          pages[pg] = pid;
          bytes += FP8 ? 64 * 128 : 64 * 256;
        }
        sm->smask[ss] = (pages[0] >= 0 ? 1 : 0) | (pages[1] >= 0 ? 2 : 0);
        mbar_expect_tx(&sm->full[s], bytes);
        mbar_expect_tx(&sm->sfull[ss], FP8 ? (pages[0] >= 0 ? 256u : 0u) + (pages[1] >= 0 ? 256u : 0u) : 0u);
        for (int pg = 0; pg < 2; ++pg) {
          if (pages[pg] < 0) continue;
          tma_load_3d(dst + pg * 8192, &tmap, 0, 0, pages[pg], &sm->full[s]);
          if (!FP8) tma_load_3d(dst + 16384 + pg * 8192, &tmap, 64, 0, pages[pg], &sm->full[s]);
          if (FP8) {
            const uint8_t* pgp = static_cast<const uint8_t*>(a.keys.pool) + size_t(pages[pg]) * a.keys.page_bytes;
            bulk_g2s(sring + ss * kTileRows + pg * kPageRows, pgp + kPageRows * 128, 256, &sm->sfull[ss]);
          }
        }
        ++issued;
        if (tw.next(a)) need_q = true;
      }
      // drain: every copy this producer issued must land before the block moves on
      for (int s = 0; s < kStages && s < issued; ++s) {
        const long long uses = (issued - s + kStages - 1) / kStages;
        mbar_wait(&sm->full[s], (uses - 1) & 1, kDefaultSpinLimit);
      }
      for (int s = 0; s < kScaleSlots && s < issued; ++s) {
        const long long uses = (issued - s + kScaleSlots - 1) / kScaleSlots;
        mbar_wait(&sm->sfull[s], (uses - 1) & 1, kDefaultSpinLimit);
      }
      for (int qb = 0; qb < 2 && qb < nreq; ++qb) {
        const int uses = (nreq - qb + 1) / 2;
        mbar_wait(&sm->qfull[qb], (uses - 1) & 1, kDefaultSpinLimit);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && start < end) {
      constexpr uint32_t idesc = FP8 ? make_idesc(0, 0, 0, 0, 128, 0) : make_idesc(1, 1, 0, 0, 128, 0);
      const uint32_t id = idesc | (static_cast<uint32_t>(N >> 3) << 17);
      TileWalker tw;
      tw.init(a, start, end);
      long long it = 0;
      int nreq = 0, qb = 0;
      bool need_q = true;
      while (tw.valid()) {
        if (need_q) {
          qb = nreq & 1;
          if (!role_wait(sm, &sm->qfull[qb], (nreq >> 1) & 1, a.spin)) break;
          ++nreq;
          need_q = false;
        }
        const int s = static_cast<int>(it % kStages);
        const int c = static_cast<int>(it % kAccs);
        const long long use = it / kAccs;
        if (!role_wait(sm, &sm->full[s], (it / kStages) & 1, a.spin)) break;
        if (use > 0 && !role_wait(sm, &sm->accempty[c], (use - 1) & 1, a.spin)) break;
        tc_fence_after();
        const uint32_t a_addr = smem_u32(stages + s * kStageBytes);
        const uint32_t b_addr = smem_u32(qbuf + qb * kQImage);
        const uint32_t d = tmem + c * N;
        if (FP8) {
#pragma unroll
          for (int kb = 0; kb < 4; ++kb) {
            mma_f8(d, smem_desc_sw128(a_addr + kb * 32, 16, 1024), smem_desc_sw128(b_addr + kb * 32, 16, 1024),
                   id, kb > 0);
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const int ch = kk >> 2, o = (kk & 3) * 32;
            mma_f16(d, smem_desc_sw128(a_addr + ch * 16384 + o, 16, 1024),
                    smem_desc_sw128(b_addr + ch * (N * 128) + o, 16, 1024), id, kk > 0);
          }
        }
        mma_commit(&sm->empty[s]);
        mma_commit(&sm->accfull[c]);
        ++it;
        if (tw.next(a)) {
          mma_commit(&sm->qempty[qb]);
          need_q = true;
        }
      }
      // drain: all issued MMAs complete before TMEM is released
      mma_commit(&sm->drain);
      mbar_wait(&sm->drain, 0, kDefaultSpinLimit);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int sub = warp & 3;                      // TMEM sub-partition of this warp
    const int row = sub * 32 + lane;               // entry within the tile
    const int tid = threadIdx.x - 64;              // 0..127
    const float* wq_all = reinterpret_cast<const float*>(a.ws + a.L.wq);
    if (start < end) {
      TileWalker tw;
      tw.init(a, start, end);
      long long it = 0;
      int cur_b = -1;
      uint32_t hphase = 0;
      // the four epilogue warps meet (bounded: an aborted pass falls through)
      auto wg_sync = [&]() {
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->hbar);
        role_wait(sm, &sm->hbar, hphase & 1, a.spin);
        ++hphase;
      };
      while (tw.valid()) {
        if (tw.b != cur_b) {
          // request switch: every warp is done with the previous request's tiles
          wg_sync();
          if (cur_b >= 0) {
            for (int i = tid; i < kHistBins; i += 128) {
              const uint32_t cnt = hist[i];
              if (cnt) { atomicAdd(ghist + size_t(cur_b) * kHistBins + i, cnt); hist[i] = 0; }
            }
          }
          cur_b = tw.b;
          if (tid < 64) sm->wq[tid] = tid < N ? wq_all[cur_b * 64 + tid] : 0.f;
          wg_sync();
        }
        const long long j = static_cast<long long>(tw.t) * kTileRows + row;
        const int ss = static_cast<int>(it % kScaleSlots);
        if (!role_wait(sm, &sm->sfull[ss], (it / kScaleSlots) & 1, a.spin)) break;
        const int pmask = sm->smask[ss];
        const bool valid = j < tw.n_b && ((pmask >> (row >> 6)) & 1);
        const float ks = FP8 ? sring[ss * kTileRows + row] : 1.0f;
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->sempty[ss]);   // one arrival per warp
        const int c = static_cast<int>(it % kAccs);
        if (!role_wait(sm, &sm->accfull[c], (it / kAccs) & 1, a.spin)) break;
        tc_fence_after();
        const uint32_t tb = tmem + (static_cast<uint32_t>(sub * 32) << 16) + c * N;
        float P[64];
        if (N == 64) {
          tmem_ld32(tb, *reinterpret_cast<float(*)[32]>(P));
          tmem_ld32(tb + 32, *reinterpret_cast<float(*)[32]>(P + 32));
        } else {
#pragma unroll
          for (int c0 = 0; c0 < 64; c0 += 16)
            if (c0 < N) tmem_ld16(tb + c0, *reinterpret_cast<float(*)[16]>(P + c0));
        }
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->accempty[c]);   // this warp's TMEM reads are done
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int h = 0; h < 64; h += 4) {
          if (h < N) {
            const float4 w4 = *reinterpret_cast<const float4*>(&sm->wq[h]);
            s0 = fmaf(w4.x, fmaxf(P[h], 0.f), s0);
            s1 = fmaf(w4.y, fmaxf(P[h + 1], 0.f), s1);
            s0 = fmaf(w4.z, fmaxf(P[h + 2], 0.f), s0);
            s1 = fmaf(w4.w, fmaxf(P[h + 3], 0.f), s1);
          }
        }
        const float I = (s0 + s1) * ks;   // the key's scale is a positive power of two
        if (valid) {
          scores_all[size_t(tw.b) * a.L.n_pad + j] = I;
          atomicAdd(&hist[order_key(I) >> (32 - kHistBits)], 1u);
        }
        ++it;
        tw.next(a);
      }
      wg_sync();
      for (int i = tid; i < kHistBins; i += 128) {
        const uint32_t cnt = hist[i];
        if (cnt) atomicAdd(ghist + size_t(cur_b) * kHistBins + i, cnt);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }

  // ======================================================= phase 2: split by threshold
  grid_barrier(sm, gbar, gridDim.x, a.spin);
  const bool aborted2 = sm->abort;   // uniform: only thread 0 sets it, before the barrier's sync
  int32_t* s_above = reinterpret_cast<int32_t*>(stages);                                   // kMaxK
  unsigned long long* s_cand = reinterpret_cast<unsigned long long*>(stages + 4 * kMaxK);  // kCandCap
  {
    long long acc = 0;
    for (int b = 0; b < a.B && acc < end && !aborted2; ++b) {
      const int nb = visible(a, b);
      const long long tb = (nb + kTileRows - 1) / kTileRows;
      const long long s0 = max(start, acc), s1 = min(end, acc + tb);
      const long long first = acc;
      acc += tb;
      if (s0 >= s1) continue;
      const long long j0 = (s0 - first) * kTileRows;
      const long long j1 = min((s1 - first) * kTileRows, static_cast<long long>(nb));
      const float* sc = scores_all + size_t(b) * a.L.n_pad;
      if (nb <= a.k) {
        // every visible entry is selected, in order
        for (long long j = j0 + threadIdx.x; j < j1; j += blockDim.x) {
          a.topk_idx[size_t(b) * a.k + j] = static_cast<int32_t>(j);
          if (a.topk_score) a.topk_score[size_t(b) * a.k + j] = sc[j];
        }
        continue;
      }
      threshold_bin(sm, ghist + size_t(b) * kHistBins, a.k);
      const int T = sm->T;
      if (T < 0) continue;   // inconsistent histogram (an aborted pass)
      if (threadIdx.x == 0) { sm->cnt[0] = 0; sm->cnt[1] = 0; }
      __syncthreads();
      uint32_t* ctr = ctr_all + b * 4;
      unsigned long long* cand = reinterpret_cast<unsigned long long*>(a.ws + a.L.cand) + size_t(b) * a.L.n_pad;
      for (long long jb = j0 + threadIdx.x; jb < j1; jb += 8 * blockDim.x) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const long long j = jb + static_cast<long long>(u) * blockDim.x;
          v[u] = j < j1 ? sc[j] : -INFINITY;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const long long j = jb + static_cast<long long>(u) * blockDim.x;
          if (j >= j1) break;
          const uint32_t key = order_key(v[u]);
          const int bin = static_cast<int>(key >> (32 - kHistBits));
          if (bin > T) {
            const uint32_t pos = atomicAdd(&sm->cnt[0], 1u);
            if (pos < kMaxK) s_above[pos] = static_cast<int32_t>(j);
          } else if (bin == T) {
            const unsigned long long k64 =
                (static_cast<unsigned long long>(key) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(j));
            const uint32_t pos = atomicAdd(&sm->cnt[1], 1u);
            if (pos < kCandCap) {
              s_cand[pos] = k64;
            } else {
              const uint32_t gp = atomicAdd(&ctr[1], 1u);   // rare: many ties in one bin
              if (gp < static_cast<uint32_t>(a.L.n_pad)) cand[gp] = k64;
            }
          }
        }
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        const uint32_t na = min(sm->cnt[0], static_cast<uint32_t>(kMaxK));
        const uint32_t nc = min(sm->cnt[1], static_cast<uint32_t>(kCandCap));
        sm->cnt[0] = na;
        sm->cnt[1] = nc;
        sm->base[0] = na ? atomicAdd(&ctr[0], na) : 0;
        sm->base[1] = nc ? atomicAdd(&ctr[1], nc) : 0;
      }
      __syncthreads();
      int32_t* sel = reinterpret_cast<int32_t*>(a.ws + a.L.sel) + size_t(b) * a.k;
      for (uint32_t i = threadIdx.x; i < sm->cnt[0]; i += blockDim.x)
        if (sm->base[0] + i < static_cast<uint32_t>(a.k)) sel[sm->base[0] + i] = s_above[i];
      for (uint32_t i = threadIdx.x; i < sm->cnt[1]; i += blockDim.x)
        if (sm->base[1] + i < static_cast<uint32_t>(a.L.n_pad)) cand[sm->base[1] + i] = s_cand[i];
      __syncthreads();
    }
  }

  // ======================================================= phase 3: finish each request
  grid_barrier(sm, gbar, 2 * gridDim.x, a.spin);
  const bool aborted3 = sm->abort;
  int32_t* s_sorted = reinterpret_cast<int32_t*>(stages);                                // kMaxK
  unsigned long long* s_c = reinterpret_cast<unsigned long long*>(stages + 4 * kMaxK);   // kCandCap
  for (int b = blockIdx.x; b < a.B && !aborted3; b += gridDim.x) {
    const int nb = visible(a, b);
    const float* sc = scores_all + size_t(b) * a.L.n_pad;
    if (nb <= a.k) {
      for (int j = nb + threadIdx.x; j < a.k; j += blockDim.x) {
        a.topk_idx[size_t(b) * a.k + j] = -1;
        if (a.topk_score) a.topk_score[size_t(b) * a.k + j] = -INFINITY;
      }
      continue;
    }
    uint32_t* ctr = ctr_all + b * 4;
    int32_t* sel = reinterpret_cast<int32_t*>(a.ws + a.L.sel) + size_t(b) * a.k;
    const unsigned long long* gcand =
        reinterpret_cast<const unsigned long long*>(a.ws + a.L.cand) + size_t(b) * a.L.n_pad;
    const uint32_t above = min(ld_acquire(&ctr[0]), static_cast<uint32_t>(a.k));
    const uint32_t c = min(ld_acquire(&ctr[1]), static_cast<uint32_t>(a.L.n_pad));
    const bool in_smem = c <= static_cast<uint32_t>(kCandCap);
    if (in_smem)
      for (uint32_t i = threadIdx.x; i < c; i += blockDim.x) s_c[i] = __ldcg(gcand + i);
    const unsigned long long* cp = in_smem ? s_c : gcand;
    if (threadIdx.x == 0) {
      sm->need = min(static_cast<uint32_t>(a.k) - above, c);
      sm->done = 0;
      sm->out = 0;
      sm->mask = c > 0 ? (~0ull << 52) : 0;   // the 12 histogram bits are shared
      sm->prefix = c > 0 ? (__ldcg(gcand) & sm->mask) : 0;
    }
    __syncthreads();
    // radix passes over the remaining 52 key bits (8-bit digits, a last 4-bit one)
    for (int shift = 44; shift >= 0; shift = shift >= 8 ? shift - 8 : (shift > 0 ? 0 : -1)) {
      if (sm->done || sm->need == 0) break;
      const int width = shift >= 4 ? 8 : 4;
      const unsigned long long dmask = ((1ull << width) - 1) << shift;
      for (int i = threadIdx.x; i < 256; i += blockDim.x) sm->dh[i] = 0;
      __syncthreads();
      const unsigned long long pm = sm->mask, pp = sm->prefix;
      for (uint32_t i = threadIdx.x; i < c; i += blockDim.x) {
        const unsigned long long key = in_smem ? cp[i] : __ldcg(cp + i);
        if ((key & pm) == pp) atomicAdd(&sm->dh[(key & dmask) >> shift], 1u);
      }
      __syncthreads();
      if (threadIdx.x < 32) {
        // lane l owns digits (from the top) nd-1-8l .. nd-8-8l; find the digit holding the need-th key
        const int nd = 1 << width;
        uint32_t loc[8], sum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int dg = nd - 1 - 8 * lane - i;
          loc[i] = dg >= 0 ? sm->dh[dg] : 0;
          sum += loc[i];
        }
        uint32_t incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += v;
        }
        const uint32_t need = sm->need;
        const unsigned hit = __ballot_sync(0xFFFFFFFFu, incl >= need);
        const int Ln = hit ? __ffs(hit) - 1 : 31;
        if (lane == Ln) {
          uint32_t accd = incl - sum;
          int d = 0;
          for (int i = 0; i < 8; ++i) {
            const int dg = nd - 1 - 8 * lane - i;
            if (dg < 0) break;
            if (accd + loc[i] >= need || dg == 0) { d = dg; break; }
            accd += loc[i];
          }
          sm->need = need - accd;
          sm->prefix = pp | (static_cast<unsigned long long>(d) << shift);
          sm->mask = pm | dmask;
          if (sm->dh[d] == need - accd) sm->done = 1;
        }
      }
      __syncthreads();
      if (shift == 0) break;
    }
    {
      const unsigned long long pm = sm->mask, pp = sm->prefix;
      const uint32_t room = static_cast<uint32_t>(a.k) - above;
      for (uint32_t i = threadIdx.x; i < c; i += blockDim.x) {
        const unsigned long long key = in_smem ? cp[i] : __ldcg(cp + i);
        if ((key & pm) >= pp) {
          const uint32_t pos = atomicAdd(&sm->out, 1u);
          if (pos < room) sel[above + pos] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(key));
        }
      }
    }
    __syncthreads();
    // ascending order of the k selected entries (bitonic; padded with INT_MAX)
    int P = 1;
    while (P < a.k) P <<= 1;
    const uint32_t filled = min(static_cast<uint32_t>(a.k), above + sm->out);
    for (int i = threadIdx.x; i < P; i += blockDim.x)
      s_sorted[i] = (i < static_cast<int>(filled)) ? __ldcg(sel + i) : 0x7FFFFFFF;
    __syncthreads();
    for (int size = 2; size <= P; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int i = threadIdx.x; i < P / 2; i += blockDim.x) {
          const int lo = 2 * i - (i & (stride - 1));
          const int hi = lo + stride;
          const bool up = (lo & size) == 0;
          const int x = s_sorted[lo], y = s_sorted[hi];
          if ((x > y) == up) { s_sorted[lo] = y; s_sorted[hi] = x; }
        }
        __syncthreads();
      }
    }
    for (int i = threadIdx.x; i < a.k; i += blockDim.x) {
      const int v = s_sorted[i];
      const bool ok = v != 0x7FFFFFFF && v >= 0 && v < nb;
      a.topk_idx[size_t(b) * a.k + i] = ok ? v : -1;
      if (a.topk_score) a.topk_score[size_t(b) * a.k + i] = ok ? __ldcg(sc + v) : -INFINITY;
    }
    __syncthreads();
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

template <int FP8>
size_t score_smem_bytes() {
  constexpr int kStageBytes = FP8 ? kTileRows * 128 : kTileRows * 256;
  constexpr int kStages = FP8 ? kStagesFp8 : kStagesBf16;
  constexpr int kQImage = FP8 ? kQImageFp8 : kQImageBf16;
  return 1024 + kStages * kStageBytes + 2 * kQImage + kHistBins * 4 + kScaleSlots * kTileRows * 4 +
         sizeof(ScoreSmem);
}

// Cooperative launch of the score kernel: the selection phases meet at grid
// barriers, so the grid is the number of blocks that fit on the GPU at once.
template <int FP8>
cudaError_t launch_score(const CUtensorMap& tmap, const IndexArgs& a, cudaStream_t stream) {
  const size_t smem = score_smem_bytes<FP8>();
  cudaError_t e = cudaFuncSetAttribute(index_score_kernel<FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, index_score_kernel<FP8>, kScoreThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  per_sm = per_sm > 2 ? 2 : per_sm;   // TMEM: two blocks of at most 256 columns per SM
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sm_count() * per_sm);
  cfg.blockDim = dim3(kScoreThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, index_score_kernel<FP8>, tmap, a);
}

}  // namespace

size_t index_workspace_bytes(int B, int n_max, int Hi, int k) {
  (void)Hi;
  return ws_layout(B, n_max, k).total;
}

cudaError_t launch_index_topk(const void* q_idx, const float* w, const cskv_paged& keys,
                              const int32_t* ctx_len, int B, int Hi, int ratio, int k,
                              int max_ctx_len, int32_t* topk_idx, float* topk_score,
                              void* workspace, cudaStream_t stream) {
  IndexArgs a;
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
  a.fp8 = keys.fmt == CSKV_FMT_FP8_E4M3_ROWSCALE_PAGESPLIT;
  a.topk_idx = topk_idx;
  a.topk_score = topk_score;
  a.ws = static_cast<uint8_t*>(workspace);
  a.L = ws_layout(B, a.n_max, k);
  a.spin = spin_limit();

  CUtensorMap tmap;
  auto enc = encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  {
    cuuint64_t dims[3], strides[2];
    cuuint32_t box[3], estr[3] = {1, 1, 1};
    CUtensorMapDataType dt;
    if (a.fp8) {
      dims[0] = 128; strides[0] = 128;
      box[0] = 128;
      dt = CU_TENSOR_MAP_DATA_TYPE_UINT8;
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
    CUresult r = enc(&tmap, dt, 3, keys.pool, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }

  index_prep_kernel<<<B, 256, 0, stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  cudaEvent_t ev_begin, ev_end;
  timing_events(&ev_begin, &ev_end);
  record_timing_event(ev_begin, stream);
  e = a.fp8 ? launch_score<1>(tmap, a, stream) : launch_score<0>(tmap, a, stream);
  record_timing_event(ev_end, stream);
  return e;
}

unsigned int take_err_index() { return take_dev_err(); }

// ---------------------------------------------------------------------------
// Scratch for cskv_index_topk_noalloc: callers that cannot allocate device
// memory get the indexer's workspace from this fixed array instead.  It lives
// in every GPU context that loads the library, for the life of the process.
// ---------------------------------------------------------------------------
static __device__ __align__(256) uint8_t g_noalloc_scratch[CSKV_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch on the current device.  Host code must not
// use the symbol itself (it is a host-side stand-in, not a device address); the
// address is looked up once per device, with that device current, and cached.
static void* noalloc_scratch_address(cudaError_t* err) {
  static std::mutex mu;
  static void* addr[256] = {};
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 256) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (*err != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
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
