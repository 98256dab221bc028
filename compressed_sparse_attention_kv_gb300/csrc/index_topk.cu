// Lightning indexer + top-k (cskv_index_topk).
//
// "DeepSeek-V4 deep dive", section 5.2: I_{b,j} = sum_h w_h ReLU(q_h . k_j) over
// the visible entries j < floor(ctx_len / ratio), one 128-d key shared by all
// indexer heads; the selector keeps min(k, n) entries (section 5.3).
//
// GB300 design (HBM-bound: at 1M context the keys are 34.6 MB per query):
//  1. index_prep_kernel   codes each request's queries (e4m3, one e8m0 scale per
//     head) into the image of a 128-byte-swizzled shared-memory tile, folds the
//     head scale into the head weight (ReLU(c x) = c ReLU(x) for c > 0), and
//     clears the request's histogram.
//  2. index_score_kernel  persistent, one block per SM, warp-specialised:
//     warp 0 streams 64-row key pages with TMA (3-D tensor map over the page
//     pool, 128-byte swizzle) into a 6-stage ring; warp 1 issues tcgen05 MMAs
//     (M = 128 entries, N = heads, K = 32 per instruction, e4m3 x e4m3, one
//     fp32 TMEM accumulator per 32-dim scale block); warps 2-9 (two
//     warpgroups, alternating tiles and TMEM accumulators) read TMEM, apply the
//     key scales, ReLU, the head weights, sum over heads inside one thread (one
//     TMEM lane = one entry), write the fp32 score and build a 4096-bin
//     histogram of the top 12 bits of its order-preserving key.
//  3. index_select1_kernel  finds the histogram bin that holds the k-th score,
//     emits every entry above it and collects the entries in it.
//  4. index_select2_kernel  radix-selects the remainder among the collected
//     64-bit (score, ~index) keys (ties -> smaller index), sorts the k
//     selected indices ascending and writes indices and scores.
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
constexpr int kStagesFp8 = 6;     // 16 KiB stages
constexpr int kStagesBf16 = 3;    // 32 KiB stages
constexpr int kScoreThreads = 320;     // 10 warps
constexpr int kQImageBytes = 16384;    // per request: bf16 [2 chunks][64 rows][128 B] or e4m3 [64][128 B]

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
  size_t scores, cand, qimg, wq, hist, ctr, sel, total;
  int n_pad;
};

__host__ __device__ inline WsLayout ws_layout(int B, int n_max, int k) {
  WsLayout L;
  L.n_pad = (n_max + kTileRows - 1) / kTileRows * kTileRows;
  if (L.n_pad == 0) L.n_pad = kTileRows;
  size_t o = 0;
  L.scores = o; o = align256(o + size_t(B) * L.n_pad * 4);
  L.cand = o;   o = align256(o + size_t(B) * L.n_pad * 8);
  L.qimg = o;   o = align256(o + size_t(B) * kQImageBytes);
  L.wq = o;     o = align256(o + size_t(B) * 64 * 4);
  L.hist = o;   o = align256(o + size_t(B) * kHistBins * 4);
  L.ctr = o;    o = align256(o + size_t(B) * 4 * 4);
  L.sel = o;    o = align256(o + size_t(B) * k * 4);
  L.total = o;
  return L;
}

// order-preserving map of an fp32 score to uint32 (larger score -> larger key)
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_to_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
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
// 1. prep: query image, folded head weights, histogram and counters cleared
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) index_prep_kernel(const IndexArgs a) {
  const int b = blockIdx.x;
  uint8_t* img = a.ws + a.L.qimg + size_t(b) * kQImageBytes;
  float* wq = reinterpret_cast<float*>(a.ws + a.L.wq) + b * 64;
  uint32_t* hist = reinterpret_cast<uint32_t*>(a.ws + a.L.hist) + size_t(b) * kHistBins;
  uint32_t* ctr = reinterpret_cast<uint32_t*>(a.ws + a.L.ctr) + b * 4;
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) hist[i] = 0;
  if (threadIdx.x < 4) ctr[threadIdx.x] = 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // one warp per head, lane l holds dims 4l .. 4l+3
  for (int h = warp; h < a.N; h += 8) {
    const bool real = h < a.Hi;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (real) v = load_bf16x4(a.q + (size_t(b) * a.Hi + h) * 256 + lane * 8);
    if (a.fp8) {
      float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
      const int e = e8m0_exponent(amax);
      const float inv = exp2i(-e);
      const uint32_t codes = e4m3x2(__fmul_rn(v.x, inv), __fmul_rn(v.y, inv)) |
                             (e4m3x2(__fmul_rn(v.z, inv), __fmul_rn(v.w, inv)) << 16);
      // row h, byte 4*lane of 128: chunk lane/4, byte (lane%4)*4 inside it
      *reinterpret_cast<uint32_t*>(img + sw128_offset(h, lane >> 2) + (lane & 3) * 4) = codes;
      if (lane == 0) wq[h] = real ? __fmul_rn(a.w[size_t(b) * a.Hi + h], exp2i(e)) : 0.f;
    } else {
      // bf16: dims 0..63 in chunk 0, 64..127 in chunk 1; lane l -> chunk l/16, byte (l%16)*8
      uint2 u = make_uint2(0u, 0u);
      if (real) u = *reinterpret_cast<const uint2*>(a.q + (size_t(b) * a.Hi + h) * 256 + lane * 8);
      uint8_t* base = img + (lane >> 4) * (a.N * 128);
      const int byte = (lane & 15) * 8;
      *reinterpret_cast<uint2*>(base + sw128_offset(h, byte >> 4) + (byte & 15)) = u;
      if (lane == 0) wq[h] = real ? a.w[size_t(b) * a.Hi + h] : 0.f;
    }
  }
}

// ---------------------------------------------------------------------------
// 2. score kernel
// ---------------------------------------------------------------------------
struct ScoreSmem {
  uint64_t full[kStagesFp8], empty[kStagesFp8];
  uint64_t accfull[2], accempty[2];
  uint64_t qfull[2], qempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  volatile int abort;
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
    b = 0;
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

template <int FP8>
__global__ void __launch_bounds__(kScoreThreads, 1)
    index_score_kernel(const __grid_constant__ CUtensorMap tmap, const IndexArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned carve-up
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int kStageBytes = FP8 ? kTileRows * 128 : kTileRows * 256;
  constexpr int kStages = FP8 ? kStagesFp8 : kStagesBf16;
  uint8_t* stages = base;
  uint8_t* qbuf = stages + kStages * kStageBytes;           // 2 x kQImageBytes
  uint32_t* hist = reinterpret_cast<uint32_t*>(qbuf + 2 * kQImageBytes);   // 2 x 4096
  ScoreSmem* sm = reinterpret_cast<ScoreSmem*>(hist + 2 * kHistBins);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = a.N;
  const int acc_cols = FP8 ? 4 * N : N;

  // work range of this block
  long long total = 0;
  for (int b = 0; b < a.B; ++b) total += (visible(a, b) + kTileRows - 1) / kTileRows;
  const long long per = (total + gridDim.x - 1) / gridDim.x;
  const long long start = min(total, per * blockIdx.x);
  const long long end = min(total, start + per);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) { mbar_init(&sm->full[s], 1); mbar_init(&sm->empty[s], 1); }
    for (int g = 0; g < 2; ++g) {
      mbar_init(&sm->accfull[g], 1);
      mbar_init(&sm->accempty[g], 128);
      mbar_init(&sm->qfull[g], 1);
      mbar_init(&sm->qempty[g], 1);
    }
    mbar_init(&sm->drain, 1);
    sm->abort = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < 2 * kHistBins; i += blockDim.x) hist[i] = 0;
  uint32_t ncols = 32;
  while (ncols < 2u * acc_cols) ncols <<= 1;
  if (warp == 1) tmem_alloc(&sm->tmem_base, ncols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && start < end) {
      prefetch_tmap(&tmap);
      TileWalker tw;
      tw.init(a, start, end);
      long long issued = 0;
      int nreq = 0;
      bool need_q = true;
      while (tw.valid()) {
        if (need_q) {
          // query image of the new request into buffer nreq % 2
          const int p = nreq & 1;
          if (nreq >= 2 && !role_wait(sm, &sm->qempty[p], ((nreq >> 1) - 1) & 1, a.spin)) break;
          mbar_expect_tx(&sm->qfull[p], kQImageBytes);
          bulk_g2s(qbuf + p * kQImageBytes, a.ws + a.L.qimg + size_t(tw.b) * kQImageBytes,
                   kQImageBytes, &sm->qfull[p]);
          ++nreq;
          need_q = false;
        }
        const int s = static_cast<int>(issued % kStages);
        const long long round = issued / kStages;
        if (round > 0 && !role_wait(sm, &sm->empty[s], (round - 1) & 1, a.spin)) break;
        uint8_t* dst = stages + s * kStageBytes;
        uint32_t bytes = 0;
        int pages[2] = {-1, -1};
        for (int pg = 0; pg < 2; ++pg) {
          const long long lp = static_cast<long long>(tw.t) * 2 + pg;
          if (lp * kPageRows >= tw.n_b) continue;
          if (lp >= a.keys.max_pages) { set_err(CSKV_ERR_BOUNDS); continue; }
          const int pid = a.keys.block_table[static_cast<long long>(tw.b) * a.keys.max_pages + lp];
          if (pid < 0 || pid >= a.keys.num_pages) { set_err(CSKV_ERR_BOUNDS); continue; }
          pages[pg] = pid;
          bytes += FP8 ? 64 * 128 : 64 * 256;
        }
        mbar_expect_tx(&sm->full[s], bytes);
        for (int pg = 0; pg < 2; ++pg) {
          if (pages[pg] < 0) continue;
          tma_load_3d(dst + pg * 8192, &tmap, 0, 0, pages[pg], &sm->full[s]);
          if (!FP8) tma_load_3d(dst + 16384 + pg * 8192, &tmap, 64, 0, pages[pg], &sm->full[s]);
        }
        ++issued;
        if (tw.next(a)) need_q = true;
      }
      // drain: every issued copy must land before the block exits
      for (int s = 0; s < kStages && s < issued; ++s) {
        const long long uses = (issued - s + kStages - 1) / kStages;
        mbar_wait(&sm->full[s], (uses - 1) & 1, kDefaultSpinLimit);
      }
      const int last_q = nreq;   // query copies land on qfull
      for (int p = 0; p < 2 && p < last_q; ++p) {
        const int uses = (last_q - p + 1) / 2;
        mbar_wait(&sm->qfull[p], (uses - 1) & 1, kDefaultSpinLimit);
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
      int nreq = 0, p = 0;
      bool need_q = true;
      while (tw.valid()) {
        if (need_q) {
          p = nreq & 1;
          if (!role_wait(sm, &sm->qfull[p], (nreq >> 1) & 1, a.spin)) break;
          ++nreq;
          need_q = false;
        }
        const int s = static_cast<int>(it % kStages);
        const int g = static_cast<int>(it & 1);
        const long long use = it >> 1;
        if (!role_wait(sm, &sm->full[s], (it / kStages) & 1, a.spin)) break;
        if (use > 0 && !role_wait(sm, &sm->accempty[g], (use - 1) & 1, a.spin)) break;
        tc_fence_after();
        const uint32_t a_addr = smem_u32(stages + s * kStageBytes);
        const uint32_t b_addr = smem_u32(qbuf + p * kQImageBytes);
        const uint32_t d = tmem + g * acc_cols;
        if (FP8) {
#pragma unroll
          for (int kb = 0; kb < 4; ++kb) {
            mma_f8(d + kb * N, smem_desc_sw128(a_addr + kb * 32, 16, 1024),
                   smem_desc_sw128(b_addr + kb * 32, 16, 1024), id, 0);
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const int c = kk >> 2, o = (kk & 3) * 32;
            mma_f16(d, smem_desc_sw128(a_addr + c * 16384 + o, 16, 1024),
                    smem_desc_sw128(b_addr + c * (N * 128) + o, 16, 1024), id, kk > 0);
          }
        }
        mma_commit(&sm->empty[s]);
        mma_commit(&sm->accfull[g]);
        ++it;
        if (tw.next(a)) {
          mma_commit(&sm->qempty[p]);
          need_q = true;
        }
      }
      // drain: all issued MMAs complete before TMEM is released
      mma_commit(&sm->drain);
      mbar_wait(&sm->drain, 0, kDefaultSpinLimit);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int g = (warp - 2) >> 2;                 // warpgroup 0 or 1
    const int sub = warp & 3;                      // TMEM sub-partition of this warp
    const int row = sub * 32 + lane;               // entry within the tile
    const int tid_g = threadIdx.x - 64 - g * 128;  // 0..127 inside the warpgroup
    uint32_t* h = hist + g * kHistBins;
    float* scores_all = reinterpret_cast<float*>(a.ws + a.L.scores);
    uint32_t* ghist = reinterpret_cast<uint32_t*>(a.ws + a.L.hist);
    const float* wq_all = reinterpret_cast<const float*>(a.ws + a.L.wq);
    if (start < end) {
      TileWalker tw;
      tw.init(a, start, end);
      long long it = 0;
      int cur_b = -1;
      float wq[64];
      auto flush = [&](int b) {
        asm volatile("bar.sync %0, 128;" ::"r"(1 + g));
        for (int i = tid_g; i < kHistBins; i += 128) {
          const uint32_t c = h[i];
          if (c) { atomicAdd(ghist + size_t(b) * kHistBins + i, c); h[i] = 0; }
        }
        asm volatile("bar.sync %0, 128;" ::"r"(1 + g));
      };
      while (tw.valid()) {
        if ((it & 1) == g) {
          if (tw.b != cur_b) {
            if (cur_b >= 0) flush(cur_b);
            cur_b = tw.b;
#pragma unroll
            for (int i = 0; i < 64; ++i) wq[i] = (i < N) ? wq_all[cur_b * 64 + i] : 0.f;
          }
          const long long j = static_cast<long long>(tw.t) * kTileRows + row;
          bool valid = j < tw.n_b;
          float ks[4] = {1.f, 1.f, 1.f, 1.f};
          if (valid) {
            const long long lp = j / kPageRows;
            const int pid = (lp < a.keys.max_pages)
                                ? a.keys.block_table[static_cast<long long>(tw.b) * a.keys.max_pages + lp]
                                : -1;
            if (pid < 0 || pid >= a.keys.num_pages) {
              valid = false;
            } else if (FP8) {
              const uint8_t* pg = static_cast<const uint8_t*>(a.keys.pool) + size_t(pid) * a.keys.page_bytes;
              const uint32_t sc = *reinterpret_cast<const uint32_t*>(pg + kPageRows * 128 + (j % kPageRows) * 4);
#pragma unroll
              for (int kb = 0; kb < 4; ++kb) ks[kb] = exp2i(static_cast<int>((sc >> (8 * kb)) & 0xFF) - 127);
            }
          }
          const long long use = it >> 1;
          if (!role_wait(sm, &sm->accfull[g], use & 1, a.spin)) break;
          tc_fence_after();
          const uint32_t tbase = tmem + (static_cast<uint32_t>(sub * 32) << 16) + g * acc_cols;
          float I = 0.f;
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            if (cc * 16 >= N) break;
            const int c0 = cc * 16;
            if (FP8) {
              float P0[16], P1[16], P2[16], P3[16];
              tmem_ld16(tbase + 0 * N + c0, P0);
              tmem_ld16(tbase + 1 * N + c0, P1);
              tmem_ld16(tbase + 2 * N + c0, P2);
              tmem_ld16(tbase + 3 * N + c0, P3);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                float x = P0[i] * ks[0];
                x = fmaf(P1[i], ks[1], x);
                x = fmaf(P2[i], ks[2], x);
                x = fmaf(P3[i], ks[3], x);
                I = fmaf(wq[c0 + i], fmaxf(x, 0.f), I);
              }
            } else {
              float P0[16];
              tmem_ld16(tbase + c0, P0);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i) I = fmaf(wq[c0 + i], fmaxf(P0[i], 0.f), I);
            }
          }
          tc_fence_before();
          mbar_arrive(&sm->accempty[g]);
          if (valid) {
            scores_all[size_t(tw.b) * a.L.n_pad + j] = I;
            atomicAdd(&h[order_key(I) >> (32 - kHistBits)], 1u);
          }
        }
        ++it;
        tw.next(a);
      }
      if (cur_b >= 0) flush(cur_b);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
}

// ---------------------------------------------------------------------------
// 3. select, first pass: threshold bin, entries above it, candidates in it
// ---------------------------------------------------------------------------
constexpr int kSelChunk = 4096;

__device__ __forceinline__ void threshold_bin(const uint32_t* ghist, int k, int& T, uint32_t& above) {
  // T = the largest bin with (count of bins >= T) >= k; above = count of bins > T
  __shared__ uint32_t part[256];
  __shared__ int sT;
  __shared__ uint32_t sAbove;
  const int t = threadIdx.x;   // 256 threads, 16 bins each
  uint32_t local = 0;
  for (int i = 0; i < 16; ++i) local += ghist[t * 16 + i];
  part[t] = local;
  __syncthreads();
  if (t == 0) {
    uint32_t acc = 0;
    int T0 = -1;
    for (int u = 255; u >= 0 && T0 < 0; --u) {
      if (acc + part[u] >= static_cast<uint32_t>(k)) {
        uint32_t a2 = acc;
        for (int i = 15; i >= 0; --i) {
          const uint32_t c = ghist[u * 16 + i];
          if (a2 + c >= static_cast<uint32_t>(k)) { T0 = u * 16 + i; break; }
          a2 += c;
        }
        acc = a2;
      } else {
        acc += part[u];
      }
    }
    sT = T0;
    sAbove = acc;
  }
  __syncthreads();
  T = sT;
  above = sAbove;
}

__global__ void __launch_bounds__(256) index_select1_kernel(const IndexArgs a) {
  const int b = blockIdx.y;
  const int n = visible(a, b);
  const long long j0 = static_cast<long long>(blockIdx.x) * kSelChunk;
  const float* scores = reinterpret_cast<const float*>(a.ws + a.L.scores) + size_t(b) * a.L.n_pad;
  if (n <= a.k) {
    // every visible entry is selected, in order; the rest is -1
    for (long long j = j0 + threadIdx.x; j < j0 + kSelChunk && j < a.k; j += blockDim.x) {
      const bool in = j < n;
      a.topk_idx[size_t(b) * a.k + j] = in ? static_cast<int32_t>(j) : -1;
      if (a.topk_score) a.topk_score[size_t(b) * a.k + j] = in ? scores[j] : -INFINITY;
    }
    return;
  }
  if (j0 >= n) return;
  const uint32_t* ghist = reinterpret_cast<const uint32_t*>(a.ws + a.L.hist) + size_t(b) * kHistBins;
  uint32_t* ctr = reinterpret_cast<uint32_t*>(a.ws + a.L.ctr) + b * 4;
  int32_t* sel = reinterpret_cast<int32_t*>(a.ws + a.L.sel) + size_t(b) * a.k;
  unsigned long long* cand = reinterpret_cast<unsigned long long*>(a.ws + a.L.cand) + size_t(b) * a.L.n_pad;
  int T;
  uint32_t above;
  threshold_bin(ghist, a.k, T, above);
  if (T < 0) return;   // inconsistent histogram (an aborted score pass): nothing to emit
  const int lane = threadIdx.x & 31;
  for (long long base = j0; base < j0 + kSelChunk && base < n; base += blockDim.x) {
    const long long j = base + threadIdx.x;
    uint32_t key = 0;
    int bin = -1;
    if (j < n && j < j0 + kSelChunk) {
      key = order_key(scores[j]);
      bin = static_cast<int>(key >> (32 - kHistBits));
    }
    const unsigned up = __ballot_sync(0xFFFFFFFFu, bin > T);
    const unsigned eq = __ballot_sync(0xFFFFFFFFu, bin == T);
    uint32_t bu = 0, be = 0;
    if (lane == 0) {
      if (up) bu = atomicAdd(&ctr[0], __popc(up));
      if (eq) be = atomicAdd(&ctr[1], __popc(eq));
    }
    bu = __shfl_sync(0xFFFFFFFFu, bu, 0);
    be = __shfl_sync(0xFFFFFFFFu, be, 0);
    const unsigned below = (1u << lane) - 1;
    if (bin > T) {
      const uint32_t pos = bu + __popc(up & below);
      if (pos < static_cast<uint32_t>(a.k)) sel[pos] = static_cast<int32_t>(j);
    } else if (bin == T) {
      const uint32_t pos = be + __popc(eq & below);
      if (pos < static_cast<uint32_t>(a.L.n_pad))
        cand[pos] = (static_cast<unsigned long long>(key) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(j));
    }
  }
}

// ---------------------------------------------------------------------------
// 4. select, second pass: radix select among the candidates, sort, write
// ---------------------------------------------------------------------------
constexpr int kSel2Threads = 1024;

__global__ void __launch_bounds__(kSel2Threads) index_select2_kernel(const IndexArgs a) {
  const int b = blockIdx.x;
  const int n = visible(a, b);
  if (n <= a.k) return;
  const float* scores = reinterpret_cast<const float*>(a.ws + a.L.scores) + size_t(b) * a.L.n_pad;
  uint32_t* ctr = reinterpret_cast<uint32_t*>(a.ws + a.L.ctr) + b * 4;
  int32_t* sel = reinterpret_cast<int32_t*>(a.ws + a.L.sel) + size_t(b) * a.k;
  const unsigned long long* cand =
      reinterpret_cast<const unsigned long long*>(a.ws + a.L.cand) + size_t(b) * a.L.n_pad;

  __shared__ uint32_t dh[256];
  __shared__ unsigned long long s_prefix, s_mask;
  __shared__ uint32_t s_need, s_done, s_out;
  __shared__ int32_t s_sorted[2048];

  const uint32_t above = min(ctr[0], static_cast<uint32_t>(a.k));
  const uint32_t c = min(ctr[1], static_cast<uint32_t>(a.L.n_pad));
  if (threadIdx.x == 0) {
    s_need = min(static_cast<uint32_t>(a.k) - above, c);
    s_done = 0;
    s_out = 0;
    // the first 12 key bits are the threshold bin, shared by every candidate
    s_mask = 0;
    s_prefix = 0;
    if (c > 0) {
      s_mask = ~0ull << 52;
      s_prefix = cand[0] & s_mask;
    }
  }
  __syncthreads();
  // radix passes over the remaining 52 bits: 8-bit digits, then a last 4-bit one
  for (int shift = 44; shift >= 0 && !s_done && s_need > 0; shift = (shift >= 8 ? shift - 8 : (shift > 0 ? 0 : -1))) {
    const int width = shift >= 4 ? 8 : 4;
    const unsigned long long dmask = ((1ull << width) - 1) << shift;
    for (int i = threadIdx.x; i < 256; i += blockDim.x) dh[i] = 0;
    __syncthreads();
    const unsigned long long pm = s_mask, pp = s_prefix;
    for (uint32_t i = threadIdx.x; i < c; i += blockDim.x) {
      const unsigned long long key = cand[i];
      if ((key & pm) == pp) atomicAdd(&dh[(key & dmask) >> shift], 1u);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t acc = 0;
      int d = (1 << width) - 1;
      for (; d >= 0; --d) {
        if (acc + dh[d] >= s_need) break;
        acc += dh[d];
      }
      if (d < 0) d = 0;
      // candidates with a larger digit are all selected; continue inside digit d
      s_need -= acc;
      s_prefix = pp | (static_cast<unsigned long long>(d) << shift);
      s_mask = pm | dmask;
      if (dh[d] == s_need) s_done = 1;   // all of digit d are selected
    }
    __syncthreads();
    if (shift == 0) break;
  }
  // emit: masked key >= prefix
  {
    const unsigned long long pm = s_mask, pp = s_prefix;
    const uint32_t room = static_cast<uint32_t>(a.k) - above;
    for (uint32_t i = threadIdx.x; i < c; i += blockDim.x) {
      const unsigned long long key = cand[i];
      if ((key & pm) >= pp) {
        const uint32_t pos = atomicAdd(&s_out, 1u);
        if (pos < room) sel[above + pos] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(key));
      }
    }
  }
  __syncthreads();
  // sort the k selected indices ascending (bitonic, power-of-two padded with INT_MAX)
  int P = 1;
  while (P < a.k) P <<= 1;
  const uint32_t filled = min(static_cast<uint32_t>(a.k), above + s_out);
  for (int i = threadIdx.x; i < P; i += blockDim.x)
    s_sorted[i] = (i < static_cast<int>(filled)) ? sel[i] : 0x7FFFFFFF;
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
    const bool ok = v != 0x7FFFFFFF && v >= 0 && v < n;
    a.topk_idx[size_t(b) * a.k + i] = ok ? v : -1;
    if (a.topk_score) a.topk_score[size_t(b) * a.k + i] = ok ? scores[v] : -INFINITY;
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
  return 1024 + kStages * kStageBytes + 2 * kQImageBytes + 2 * kHistBins * 4 + sizeof(ScoreSmem);
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
  a.fp8 = keys.fmt == CSKV_FMT_FP8_E4M3_E8M0_B32_PAGESPLIT;
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

  const int grid = sm_count();
  cudaEvent_t ev_begin, ev_end;
  timing_events(&ev_begin, &ev_end);
  record_timing_event(ev_begin, stream);
  if (a.fp8) {
    const size_t smem = score_smem_bytes<1>();
    cudaFuncSetAttribute(index_score_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    index_score_kernel<1><<<grid, kScoreThreads, smem, stream>>>(tmap, a);
  } else {
    const size_t smem = score_smem_bytes<0>();
    cudaFuncSetAttribute(index_score_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    index_score_kernel<0><<<grid, kScoreThreads, smem, stream>>>(tmap, a);
  }
  e = cudaGetLastError();
  record_timing_event(ev_end, stream);
  if (e != cudaSuccess) return e;

  dim3 g1((a.L.n_pad + kSelChunk - 1) / kSelChunk, B);
  if (g1.x < static_cast<unsigned>((k + kSelChunk - 1) / kSelChunk)) g1.x = (k + kSelChunk - 1) / kSelChunk;
  index_select1_kernel<<<g1, 256, 0, stream>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  index_select2_kernel<<<B, kSel2Threads, 0, stream>>>(a);
  return cudaGetLastError();
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
