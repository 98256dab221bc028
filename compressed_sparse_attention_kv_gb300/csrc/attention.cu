// Shared-KV sparse decode attention (cskv_sparse_decode_attn).
//
// "DeepSeek-V4 deep dive": section 3.1 (one 512-d entry is key and value of
// every head), section 3.3 (query rotated by its position, output rotated back),
// section 3.4 Eq. 27 (one softmax over window + compressed keys with a per-head
// sink in the denominator), section 5.3 (index list = window slots, then the
// selected entries; -1 skipped; duplicates kept) and section 6.1 (HCA reads
// every visible entry).
//
// GB300 design.  A request's key list is cut into 128-key tiles: tile 0 is the
// 128-slot window ring (in prefill, the query's request's raw rows at positions
// t-127 .. t, fewer at the start: causal), tiles 1.. are 128 consecutive list
// entries.  Prefill runs every query as its own list ("DeepSeek-V4 deep dive",
// section 5.3: the buffer [all raw rows of the prompt ; its compressed entries],
// the window indices t-127 .. t masked below 0); req_of maps a query to its
// request.  One block handles one (request, tile, head group: 64 heads, or 32 when
// the grid would otherwise leave most SMs idle):
//   * the query is copied into shared memory and its last 64 dims rotated (fp32) in
//     place, and a list tile's block-table row staged beside it, before the tile
//     waits for its selection; then the tile's rows (528 B FP8, 288 B FP4 or 1 KiB
//     bf16) come in by 16-byte asynchronous copies, all in flight together, and are
//     dequantised exactly into bf16, giving a 128 x 512 K-major tile with 128-byte
//     swizzle;
//   * one thread issues tcgen05 MMAs S^T = K Q^T (M = 128 keys, N = heads,
//     K = 512) into TMEM - keys are the MMA rows, so 16..64 heads need no padding;
//   * softmax statistics per head (max, sum of exp2) over the tile, straight from
//     TMEM by a transposing butterfly per warp, P^T stored as the bf16 MN-major B
//     operand;
//   * O^T = V^T P^T (M = 128 dims x 4 blocks, N = heads, K = 128 keys): the same
//     smem tile is read a second time as the MN-major A operand (K = V);
//   * the partial goes to the workspace: the head's (m, l) in fp32 and O / l in bf16
//     (a convex combination of the tile's values, so it has their range; half the
//     bytes of fp32 to write here and to read back in the merge).
// attn_combine_kernel merges the partials of a request in a fixed order with
// the sink, applies the inverse rotation and writes bf16.
#include <type_traits>

#include "codec.cuh"
#include "internal.h"

namespace cskv {

namespace {

constexpr int kD = 512;
constexpr int kKeys = 128;
constexpr int kAttnThreads = 512;   // 16 warps: four per TMEM lane quarter
constexpr int kMaxHeadsPerBlock = 64;
constexpr int kBtStage = kKeys * 128;  // block-table entries staged in the K tile's lower half (64 KiB)

__host__ __device__ inline size_t a256(size_t x) { return (x + 255) & ~size_t(255); }

struct AttnLayout {
  size_t opart, ml, total;
  int max_tiles;
};

__host__ __device__ inline AttnLayout attn_layout(int B, int H, int max_ctx, int ratio, int k) {
  AttnLayout L;
  const int comp = k > 0 ? k : (ratio > 0 ? max_ctx / ratio : 0);
  L.max_tiles = 1 + (comp + kKeys - 1) / kKeys;
  size_t o = 0;
  L.opart = o; o = a256(o + size_t(B) * L.max_tiles * H * kD * 2);
  L.ml = o;    o = a256(o + size_t(B) * L.max_tiles * H * 2 * 4);
  L.total = o;
  return L;
}

struct AttnArgs {
  const uint8_t* q;
  cskv_paged kv;
  int kv_row_bytes;
  const uint8_t* swa;          // decode: the 128-slot window ring [B, 128, row]
  int swa_fmt, swa_row_bytes;
  cskv_paged win;              // prefill (win.pool != nullptr): raw rows by position, per request
  const int32_t* req_of;       // request of each query (block tables, window); nullptr = the query's index
  const int32_t* ctx_len;
  const int32_t* topk;
  int k, ratio, max_ctx;
  const float* sink;
  float scale_log2;       // softmax_scale * log2(e)
  const float* q_rope;
  int B, H;
  uint8_t* out;
  __nv_bfloat16* opart;   // per (request, tile, head): O / l, bf16
  float* ml;              // per (request, tile, head): m (base 2) and l, fp32
  int max_tiles;
  uint8_t* out_host;           // optional second copy of out (a host buffer's device alias), or nullptr
  // Fused decode step: ready[b] turns 1 once the indexer has written request b's
  // selection; list tiles wait for it (bounded by spin cycles) instead of for the
  // whole indexer grid.  nullptr: list tiles wait for the kernel before to complete.
  const uint32_t* ready;
  int heads_per_block;         // 32 or 64 (the launch's choice, below)
  unsigned long long spin;
};

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ int query_len(const AttnArgs& a, int b) {
  int c = a.ctx_len[b];
  if (c < 1 || c > a.max_ctx) {
    set_err(CSKV_ERR_BOUNDS);
    c = max(1, min(c, a.max_ctx));
  }
  return c;
}

// number of compressed keys in the list of request b
__device__ __forceinline__ int comp_keys(const AttnArgs& a, int ctx) {
  return a.topk ? a.k : ctx / a.ratio;
}

// 16 dequantised values -> 32 bytes of bf16 at dst (two 16-byte chunks)
__device__ __forceinline__ void put16(uint8_t* tile, int row, int l, const float (&v)[16]) {
  // dims 16l .. 16l+15 -> chunk l/4 of the K tile, 16-byte chunks 2(l%4), 2(l%4)+1
  uint8_t* base = tile + (l >> 2) * (kKeys * 128);
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  const int c0 = (l & 3) * 2;
  *reinterpret_cast<uint4*>(base + sw128_offset(row, c0)) = make_uint4(w[0], w[1], w[2], w[3]);
  *reinterpret_cast<uint4*>(base + sw128_offset(row, c0 + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
}

// Raw bytes of 16 values of one row: codes (16 B FP8 / 8 B FP4 / 32 B bf16) and
// their scale byte.
struct RowBytes {
  uint4 lo, hi;
  uint32_t scb;
};

// Exact dequantisation of lane l's 16 values (dims 16l .. 16l+15) from its raw bytes.
__device__ __forceinline__ void convert16(int fmt, const RowBytes& r, float (&v)[16]) {
  if (fmt == CSKV_FMT_FP8_E4M3_E8M0_B32) {
    const float s = exp2i(static_cast<int>(r.scb) - 127);
    const uint32_t cw[4] = {r.lo.x, r.lo.y, r.lo.z, r.lo.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t h0, h1;
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h0) : "h"(static_cast<uint16_t>(cw[i] & 0xFFFF)));
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h1) : "h"(static_cast<uint16_t>(cw[i] >> 16)));
      v[4 * i + 0] = __fmul_rn(__half2float(__ushort_as_half(h0 & 0xFFFF)), s);
      v[4 * i + 1] = __fmul_rn(__half2float(__ushort_as_half(h0 >> 16)), s);
      v[4 * i + 2] = __fmul_rn(__half2float(__ushort_as_half(h1 & 0xFFFF)), s);
      v[4 * i + 3] = __fmul_rn(__half2float(__ushort_as_half(h1 >> 16)), s);
    }
  } else if (fmt == CSKV_FMT_FP4_E2M1_E4M3_B16) {
    const float s = e4m3_to_f32(r.scb);
    const uint32_t cw[2] = {r.lo.x, r.lo.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t h;
        asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
            : "=r"(h)
            : "r"((cw[i] >> (8 * j)) & 0xFF));
        v[8 * i + 2 * j + 0] = __fmul_rn(__half2float(__ushort_as_half(h & 0xFFFF)), s);
        v[8 * i + 2 * j + 1] = __fmul_rn(__half2float(__ushort_as_half(h >> 16)), s);
      }
    }
  } else {
    const uint32_t cw[8] = {r.lo.x, r.lo.y, r.lo.z, r.lo.w, r.hi.x, r.hi.y, r.hi.z, r.hi.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[2 * i] = bf16lo(cw[i]);
      v[2 * i + 1] = bf16hi(cw[i]);
    }
  }
}

struct AttnSmem {
  uint64_t bar_s, bar_o;
  uint32_t tmem_base;
  __align__(16) float mpart[4][kMaxHeadsPerBlock];   // per lane quarter: the largest logit of each head
  float lpart[4][kMaxHeadsPerBlock];                 // per lane quarter: the sum of exp2 of each head
  __align__(16) float linv[kMaxHeadsPerBlock];       // 1 / l of each head over the tile (0: no key)
  const uint8_t* rowp[kKeys];   // address of each key row of the tile, null = no key
  __align__(16) uint8_t scl[kKeys][32];   // staged scale bytes of each row (FP8: 16, FP4: 32)
};

// In-place dequantisation of the staged FP8 / FP4 rows into the bf16 K tile.  Item
// (r, l) = dims 16l .. 16l+15 of row r, converted exactly by the hardware conversions
// (e4m3 / e2m1 pairs to f16, times the block scale in fp32, rounded to bf16, which
// holds every such product).  The first half (dims 0-255: outputs in the lower half,
// codes in the upper half) is spread over all threads; each thread then reads the codes
// of its second-half items before any thread overwrites the upper half.  mid() - thread
// 0 issuing the first half's products - runs once the first half is in place and fenced
// for the tensor core; warp 0 takes no second-half item, so that the issue overlaps the
// other warps' conversions instead of following its own.
template <int FMT, class Mid>
__device__ __forceinline__ void dequant_tile(uint8_t* ktile, const uint8_t* stage, const AttnSmem* sm,
                                             Mid&& mid) {
  constexpr bool kFp8 = FMT == CSKV_FMT_FP8_E4M3_E8M0_B32;
  auto raw_of = [&](int r, int l) -> RowBytes {
    RowBytes rb;
    rb.hi = make_uint4(0u, 0u, 0u, 0u);
    if (kFp8) {
      rb.lo = *reinterpret_cast<const uint4*>(stage + r * kD + 16 * l);
      rb.scb = sm->scl[r][l >> 1];
    } else {
      const uint2 c = *reinterpret_cast<const uint2*>(stage + r * (kD / 2) + 8 * l);
      rb.lo = make_uint4(c.x, c.y, 0u, 0u);
      rb.scb = sm->scl[r][l];
    }
    return rb;
  };
  auto emit = [&](int r, int l, const RowBytes& rb) {
    float v[16];
    if (sm->rowp[r] != nullptr) {
      convert16(FMT, rb, v);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = 0.f;
    }
    put16(ktile, r, l, v);
  };
  constexpr int kItems = kKeys * 16;                    // items per half
  constexpr int kPer = kItems / kAttnThreads;           // 4
#pragma unroll 4
  for (int u = 0; u < kPer; ++u) {
    const int x = threadIdx.x + u * kAttnThreads;
    emit(x >> 4, x & 15, raw_of(x >> 4, x & 15));
  }
  constexpr int kThreads2 = kAttnThreads - 32;          // the second half: warps 1..
  constexpr int kPer2 = (kItems + kThreads2 - 1) / kThreads2;   // 5
  const int t2 = static_cast<int>(threadIdx.x) - 32;
  RowBytes rb[kPer2];
  if (t2 >= 0) {
#pragma unroll
    for (int u = 0; u < kPer2; ++u) {
      const int x = t2 + u * kThreads2;
      if (x < kItems) rb[u] = raw_of(x >> 4, 16 + (x & 15));
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  mid();
  if (t2 >= 0) {
#pragma unroll
    for (int u = 0; u < kPer2; ++u) {
      const int x = t2 + u * kThreads2;
      if (x < kItems) emit(x >> 4, 16 + (x & 15), rb[u]);
    }
  }
}

__global__ void __launch_bounds__(kAttnThreads, 1) attn_tile_kernel(const AttnArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned by pointer arithmetic on the shared array (an integer round trip
  // would lose the address space and turn every access into a generic one)
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* ktile = base;                                   // 8 chunks x 128 rows x 128 B = 128 KiB
  uint8_t* qtile = ktile + 8 * kKeys * 128;                // 8 chunks x Nq rows x 128 B <= 64 KiB
  uint8_t* ptile = qtile;                                  // reused after S: 128 keys x 128 B (1024-aligned)
  AttnSmem* sm = reinterpret_cast<AttnSmem*>(qtile + 8 * kMaxHeadsPerBlock * 128);

  const int b = blockIdx.y;
  const int tile = blockIdx.x;
  const int h0 = blockIdx.z * a.heads_per_block;
  const int Hb = min(a.heads_per_block, a.H - h0);
  const int Nq = (Hb + 15) / 16 * 16;
  const int ctx = query_len(a, b);
  const int t = ctx - 1;
  const int ncomp = comp_keys(a, ctx);
  const int ntiles = 1 + (ncomp + kKeys - 1) / kKeys;
  if (tile >= ntiles) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&sm->bar_s, 1);
    mbar_init(&sm->bar_o, 4);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&sm->tmem_base, 512);

  // Every global read of this block is a cp.async straight into shared memory, so
  // the loads are all in flight together and need no registers:
  //  - the query rows (bf16) into their places in the swizzled Q tile, the last 64
  //    dims rotated afterwards in shared memory;
  //  - bf16 key rows into their places in the swizzled K tile;
  //  - FP8 / FP4 key rows: the codes into the upper half of the K tile region, the
  //    scale bytes into sm->scl, then dequantised in place in two halves
  //    (dims 0-255 first; the codes of dims 256-511 are read into registers before
  //    the half they share is overwritten).
  // The code runs once per block from a cold instruction cache; loops stay rolled.
  const int row_fmt = tile == 0 ? a.swa_fmt : a.kv.fmt;
  uint8_t* stage = ktile + 4 * kKeys * 128;   // upper half of the K tile: dims 256-511
  // ---- query: 64 chunks of 16 bytes per head row, zero rows for padded heads
  {
    const uint8_t* qb = a.q + (size_t(b) * a.H + h0) * kD * 2;
#pragma unroll 1
    for (int x = threadIdx.x; x < Nq * 64; x += blockDim.x) {
      const int h = x >> 6, c = x & 63;   // dims 8c .. 8c+7
      uint8_t* dst = qtile + (c >> 3) * (Nq * 128) + sw128_offset(h, c & 7);
      if (h < Hb) cp_async16(dst, qb + (size_t(h) * kD + c * 8) * 2);
      else *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  // ---- list tiles: the request's block-table row into the lower half of the K tile
  // (untouched until the rows are resolved), so that the lookups after the selection
  // read shared memory
  const int rq = a.req_of ? a.req_of[b] : b;
  const int32_t* bt_s = reinterpret_cast<const int32_t*>(ktile);
  const int np = tile > 0 && a.kv.block_table != nullptr
                     ? min(a.kv.max_pages, (ctx / a.ratio + kPageRows - 1) / kPageRows)
                     : 0;
  const bool bt_staged = np > 0 && np <= kBtStage;
  if (bt_staged) {
    const int32_t* bt = a.kv.block_table + static_cast<long long>(rq) * a.kv.max_pages;
#pragma unroll 1
    for (int x = threadIdx.x; x < np; x += blockDim.x) cp_async4(ktile + 4 * x, bt + x);
  }
  cp_async_wait_all();
  __syncthreads();
  // ---- rotate the query's last 64 dims (pairs (2i, 2i+1) by the query position)
  {
    const float* cs = a.q_rope + size_t(b) * 64;
#pragma unroll 1
    for (int x = threadIdx.x; x < Hb * 8; x += blockDim.x) {
      const int h = x >> 3, g = x & 7;   // dims 448 + 8g .. +7: chunk 7, 16-byte chunk g
      uint4* pq = reinterpret_cast<uint4*>(qtile + 7 * (Nq * 128) + sw128_offset(h, g));
      const uint4 raw = *pq;
      float v[8] = {bf16lo(raw.x), bf16hi(raw.x), bf16lo(raw.y), bf16hi(raw.y),
                    bf16lo(raw.z), bf16hi(raw.z), bf16lo(raw.w), bf16hi(raw.w)};
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const int kk = 4 * g + p;
        const float c = cs[2 * kk], sn = cs[2 * kk + 1];
        const float y0 = v[2 * p], y1 = v[2 * p + 1];
        v[2 * p] = y0 * c - y1 * sn;
        v[2 * p + 1] = y0 * sn + y1 * c;
      }
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 hh = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t*>(&hh);
      }
      *pq = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  grid_dep_launch();   // the combine kernel may be scheduled; it waits for this grid
  // The selected entries come from the indexer, which may still be finishing (this
  // kernel is a programmatic dependent of it): compressed tiles wait here, the
  // window tile does not need it.  In a fused step each request's flag says when its
  // own selection is written.
  if (tile > 0) {
    if (a.ready == nullptr) {
      grid_dep_wait();
    } else {
      // a block-table row too long to stage: into L2 while the selection is being
      // written, so that the row lookups after it do not wait on HBM
      if (a.kv.block_table != nullptr && !bt_staged) {
        const int32_t* bt = a.kv.block_table + static_cast<long long>(rq) * a.kv.max_pages;
        for (int x = threadIdx.x * 32; x < np; x += blockDim.x * 32)
          asm volatile("prefetch.global.L2 [%0];" ::"l"(bt + x));
      }
      if (threadIdx.x == 0 && ld_acquire_gpu(a.ready + b) == 0) {
        const unsigned long long t0 = clock64();
        while (ld_acquire_gpu(a.ready + b) == 0) {
          if (clock64() - t0 > a.spin) {
            set_err(CSKV_ERR_TIMEOUT);
            break;
          }
          __nanosleep(100);
        }
      }
      __syncthreads();
    }
  }
  // ---- rows of this tile: thread r < 128 resolves row r's address (the list entry,
  // then the block table), all rows in parallel
  const bool bf16_rows = row_fmt == CSKV_FMT_BF16;
  const int code_bytes = row_fmt == CSKV_FMT_FP8_E4M3_E8M0_B32 ? kD : kD / 2;
  static_assert(kKeys <= kAttnThreads, "a thread per row");
  if (threadIdx.x < kKeys) {
    const int r = threadIdx.x;
    const uint8_t* p = nullptr;
    if (tile == 0) {
      if (a.win.pool == nullptr) {
        if ((t >= kKeys - 1) || (r <= t)) p = a.swa + (size_t(b) * kWindow + r) * a.swa_row_bytes;
      } else {
        const int pos = t - (kKeys - 1) + r;   // positions t-127 .. t; none below 0
        if (pos >= 0) p = paged_row(a.win, rq, pos, a.swa_row_bytes).data;
      }
    } else {
      const int li = (tile - 1) * kKeys + r;
      if (li < ncomp) {
        const int e = a.topk ? a.topk[size_t(b) * a.k + li] : li;
        if (e >= 0) {
          if (e >= ctx / a.ratio) {
            set_err(CSKV_ERR_BOUNDS);
          } else if (bt_staged) {   // the same checks as paged_row
            const int lp = e / kPageRows, pp = lp < np ? bt_s[lp] : -1;
            if (pp >= 0 && pp < a.kv.num_pages) p = page_row(a.kv, pp, e % kPageRows, a.kv_row_bytes).data;
            else set_err(CSKV_ERR_BOUNDS);
          } else {
            p = paged_row(a.kv, rq, e, a.kv_row_bytes).data;
          }
        }
      }
    }
    sm->rowp[r] = p;
  }
  __syncthreads();
  // ---- key rows: consecutive threads take consecutive 16-byte chunks of a row, so that
  // each warp's copies cover whole rows (CPR chunks per row, a constant divisor)
  auto copy_rows = [&](auto cpr_const) {
    constexpr int CPR = decltype(cpr_const)::value;
#pragma unroll 1
    for (int x = threadIdx.x; x < kKeys * CPR; x += blockDim.x) {
      const int r = x / CPR, c = x - r * CPR;
      const uint8_t* p = sm->rowp[r];
      if (CPR == 64) {   // bf16: straight into the row's swizzled places
        uint8_t* dst = ktile + (c >> 3) * (kKeys * 128) + sw128_offset(r, c & 7);
        if (p) cp_async16(dst, p + c * 16);
        else *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
      } else if (p) {    // FP8 / FP4: the codes into the staging half, the scale bytes beside
        if (c * 16 < code_bytes) cp_async16(stage + r * code_bytes + c * 16, p + c * 16);
        else cp_async16(&sm->scl[r][c * 16 - code_bytes], p + c * 16);
      }
    }
  };
  if (bf16_rows) copy_rows(std::integral_constant<int, 64>{});
  else if (row_fmt == CSKV_FMT_FP8_E4M3_E8M0_B32) copy_rows(std::integral_constant<int, (kD + kD / 32) / 16>{});
  else copy_rows(std::integral_constant<int, (kD / 2 + kD / 16) / 16>{});
  cp_async_wait_all();
  __syncthreads();
  // ---- S^T = K Q^T : M = 128 keys, N = Nq, K = 512, issued by one thread in two
  // halves of K: dims 0-255 as soon as the dequantisation has written them (the tensor
  // core works while the second half is dequantised), then dims 256-511
  auto issue_s = [&](int kk0, int kk1, bool last) {
    if (threadIdx.x == 0) {
      tc_fence_after();
      const uint32_t id = make_idesc(1, 1, 0, 0, 128, 0) | (static_cast<uint32_t>(Nq >> 3) << 17);
      // the descriptors' start-address field counts 16-byte units (no carry: shared
      // memory < 256 KiB): a 32-byte K step adds 2, a 128-row chunk kKeys * 8 / Nq * 8
      const uint64_t da = smem_desc_sw128(smem_u32(ktile), 16, 1024);
      const uint64_t dq = smem_desc_sw128(smem_u32(qtile), 16, 1024);
#pragma unroll 4
      for (int kk = kk0; kk < kk1; ++kk) {
        const int c = kk >> 2, o = (kk & 3) * 2;
        mma_f16(sm->tmem_base, da + c * (kKeys * 8) + o, dq + c * (Nq * 8) + o, id, kk > 0);
      }
      if (last) mma_commit(&sm->bar_s);
    }
  };
  // ---- dequantise FP8 / FP4 rows in place
  int kk_done = 0;
  if (row_fmt == CSKV_FMT_FP8_E4M3_E8M0_B32) {
    dequant_tile<CSKV_FMT_FP8_E4M3_E8M0_B32>(ktile, stage, sm, [&]() { issue_s(0, 16, false); });
    kk_done = 16;
  } else if (row_fmt == CSKV_FMT_FP4_E2M1_E4M3_B16) {
    dequant_tile<CSKV_FMT_FP4_E2M1_E4M3_B16>(ktile, stage, sm, [&]() { issue_s(0, 16, false); });
    kk_done = 16;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  issue_s(kk_done, 32, true);
  mbar_wait(&sm->bar_s, 0, kDefaultSpinLimit);
  tc_fence_after();

  // ---- softmax over the tile's keys, straight from TMEM.  Thread (lane quarter
  // warp & 3, lane) holds key r's logits for the warp's heads [cbase, cbase + quarter);
  // warps w, w+4, w+8, w+12 share lane quarter w and split the head columns.  Per head,
  // the largest logit and the sum of exp2 over the warp's 32 keys come from a
  // transposing butterfly (16 shuffles for all of a thread's heads), the four lane
  // quarters' partials meet in shared memory; P^T is stored as the MN-major B operand
  // [key][head], four heads per 8-byte store.
  {
    const int r = (warp & 3) * 32 + lane;
    const int qid = warp & 3;
    const bool ok = sm->rowp[r] != nullptr;
    const int quarter = Nq >> 2;   // 4, 8, 12 or 16
    const int cbase = (warp >> 2) * quarter;
    float z[16];
#pragma unroll
    for (int c0 = 0; c0 < 16; c0 += 4)
      if (c0 < quarter)
        tmem_ld4(tmem + (static_cast<uint32_t>(qid * 32) << 16) + cbase + c0, *reinterpret_cast<float(*)[4]>(z + c0));
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 16; ++i) z[i] = (i < quarter && ok) ? z[i] * a.scale_log2 : -INFINITY;
    // the reduction of slot j over the warp's 32 lanes ends in lanes 2j and 2j + 1
    const int hs = (lane >> 1) & 15;
    auto butterfly = [&](float (&t)[16], auto op) {
#pragma unroll
      for (int w = 8; w >= 1; w >>= 1) {   // offsets 16, 8, 4, 2: keep half the slots
        const int off = 2 * w;
        const bool hi = (lane & off) != 0;
#pragma unroll
        for (int j = 0; j < w; ++j) {
          const float send = hi ? t[j] : t[j + w];
          const float keep = hi ? t[j + w] : t[j];
          t[j] = op(keep, __shfl_xor_sync(0xFFFFFFFFu, send, off));
        }
      }
      return op(t[0], __shfl_xor_sync(0xFFFFFFFFu, t[0], 1));
    };
    float t[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) t[i] = z[i];
    const float mw = butterfly(t, [](float x, float y) { return fmaxf(x, y); });
    if ((lane & 1) == 0 && hs < quarter) sm->mpart[qid][cbase + hs] = mw;
    __syncthreads();
    float mh[16];
#pragma unroll
    for (int g = 0; g < 16; g += 4) {
      if (g < quarter) {
        float4 mx = *reinterpret_cast<const float4*>(&sm->mpart[0][cbase + g]);
#pragma unroll
        for (int q = 1; q < 4; ++q) {
          const float4 v = *reinterpret_cast<const float4*>(&sm->mpart[q][cbase + g]);
          mx = make_float4(fmaxf(mx.x, v.x), fmaxf(mx.y, v.y), fmaxf(mx.z, v.z), fmaxf(mx.w, v.w));
        }
        mh[g] = mx.x;
        mh[g + 1] = mx.y;
        mh[g + 2] = mx.z;
        mh[g + 3] = mx.w;
      } else {
        mh[g] = mh[g + 1] = mh[g + 2] = mh[g + 3] = -INFINITY;
      }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int h = cbase + i;
      t[i] = (i >= quarter || mh[i] == -INFINITY || h >= Hb) ? 0.f : exp2f(z[i] - mh[i]);
    }
#pragma unroll
    for (int g = 0; g < 16; g += 4) {
      if (g < quarter) {
        const int h = cbase + g;   // a multiple of 4: the 8 bytes lie inside one 16-byte chunk
        __nv_bfloat162 lo = __floats2bfloat162_rn(t[g], t[g + 1]);
        __nv_bfloat162 hi = __floats2bfloat162_rn(t[g + 2], t[g + 3]);
        *reinterpret_cast<uint2*>(ptile + sw128_offset(r, h >> 3) + (h & 7) * 2) =
            make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
      }
    }
    const float lw = butterfly(t, [](float x, float y) { return x + y; });
    if ((lane & 1) == 0 && hs < quarter) sm->lpart[qid][cbase + hs] = lw;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // ---- O^T = V^T P^T : 4 blocks of 128 dims, N = Nq, K = 128 keys; both operands MN-major.
  // The blocks write disjoint accumulators, so lane 0 of warps 0-3 issues one each and
  // commits it (bar_o counts four): four issuers instead of one serial chain of 32.
  if (lane == 0 && warp < 4) {
    const int mb = warp;
    const uint32_t id = make_idesc(1, 1, 1, 1, 128, 0) | (static_cast<uint32_t>(Nq >> 3) << 17);
    const uint64_t dv = smem_desc_sw128(smem_u32(ktile), kKeys * 128, 1024) + mb * (kKeys * 16);
    const uint64_t dp = smem_desc_sw128(smem_u32(ptile), kKeys * 128, 1024);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) mma_f16(tmem + 128 + mb * Nq, dv + ks * 128, dp + ks * 128, id, ks > 0);
    mma_commit(&sm->bar_o);
  }
  // the heads' statistics over the tile (lane quarters in order) while the product runs
  const size_t slot = (size_t(b) * a.max_tiles + tile) * a.H + h0;
  if (threadIdx.x < Hb) {
    const int h = threadIdx.x;
    const float m = fmaxf(fmaxf(sm->mpart[0][h], sm->mpart[1][h]), fmaxf(sm->mpart[2][h], sm->mpart[3][h]));
    const float l = ((sm->lpart[0][h] + sm->lpart[1][h]) + sm->lpart[2][h]) + sm->lpart[3][h];
    a.ml[(slot + h) * 2 + 0] = m;
    a.ml[(slot + h) * 2 + 1] = l;
    sm->linv[h] = l > 0.f ? 1.0f / l : 0.f;
  }
  __syncthreads();
  mbar_wait(&sm->bar_o, 0, kDefaultSpinLimit);
  tc_fence_after();

  // ---- partial out: O^T lanes = dims; warps 4m .. 4m+3 block m of 128 dims
  {
    const int sub = warp & 3;
    {
      const int mb = warp >> 2;
      const int d = mb * 128 + sub * 32 + lane;
      // all of the block's head columns, one wait
      float o[64];
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 16)
        if (c0 < Nq)
          tmem_ld16(tmem + (static_cast<uint32_t>(sub * 32) << 16) + 128 + mb * Nq + c0,
                    *reinterpret_cast<float(*)[16]>(o + c0));
      tmem_wait_ld();
      // straight out: for each head the warp's 32 dims are one 64-byte run
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 4) {
        if (c0 < Hb) {
          const float4 r = *reinterpret_cast<const float4*>(&sm->linv[c0]);
          const float rv[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
          for (int i = c0; i < c0 + 4; ++i)
            if (i < Hb) a.opart[(slot + i) * kD + d] = __float2bfloat16_rn(o[i] * rv[i - c0]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  // fused step: this grid completes only after the indexer has (the next step's prep
  // clears the indexer's workspace once the kernels before it are complete)
  if (a.ready != nullptr && threadIdx.x == 0) grid_dep_wait();
}

// merge the tiles of (request, head) in tile order, sink, inverse RoPE, bf16.  DPT dims
// per thread (launched with 8: four heads per 256-thread block, 16-byte loads and stores)
template <int DPT>
__global__ void __launch_bounds__(256) attn_combine_kernel(const AttnArgs a) {
  grid_dep_wait();   // the tile kernel's partials
  constexpr int kThreadsPerHead = kD / DPT;
  constexpr int kHeadsPerBlock = 256 / kThreadsPerHead;
  const int b = blockIdx.x;
  const int h = blockIdx.y * kHeadsPerBlock + static_cast<int>(threadIdx.x) / kThreadsPerHead;
  if (h >= a.H) return;
  const int ctx = query_len(a, b);
  const int ncomp = comp_keys(a, ctx);
  const int ntiles = 1 + (ncomp + kKeys - 1) / kKeys;
  const size_t slot0 = size_t(b) * a.max_tiles * a.H + h;
  const int d = DPT * (static_cast<int>(threadIdx.x) % kThreadsPerHead);
  // running (max, sum, output) in base 2, started from the sink; tiles taken in
  // batches of 8 whose loads are all issued before any is used.  A tile's partial is
  // O / l: it enters with weight exp2(m - M) * l.
  float M = a.sink ? a.sink[h] * 1.4426950408889634f : -INFINITY;
  float L = a.sink ? 1.f : 0.f;
  float o[DPT];
#pragma unroll
  for (int i = 0; i < DPT; ++i) o[i] = 0.f;
  for (int s0 = 0; s0 < ntiles; s0 += 8) {
    float m[8], l[8];
    float v[8][DPT];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const size_t sl = slot0 + size_t(s0 + u) * a.H;
      const bool in = s0 + u < ntiles;
      m[u] = in ? a.ml[sl * 2] : -INFINITY;
      l[u] = in ? a.ml[sl * 2 + 1] : 0.f;
      if constexpr (DPT % 8 == 0) {
#pragma unroll
        for (int i = 0; i < DPT; i += 8) {
          const uint4 x = in ? *reinterpret_cast<const uint4*>(a.opart + sl * kD + d + i) : make_uint4(0, 0, 0, 0);
          const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            v[u][i + 2 * j] = bf16lo(w[j]);
            v[u][i + 2 * j + 1] = bf16hi(w[j]);
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < DPT; i += 2) {
          const uint32_t x = in ? *reinterpret_cast<const uint32_t*>(a.opart + sl * kD + d + i) : 0u;
          v[u][i] = bf16lo(x);
          v[u][i + 1] = bf16hi(x);
        }
      }
    }
    float Mb = M;
#pragma unroll
    for (int u = 0; u < 8; ++u) Mb = fmaxf(Mb, m[u]);
    if (Mb == -INFINITY) continue;
    const float f = M == -INFINITY ? 0.f : exp2f(M - Mb);
    L *= f;
#pragma unroll
    for (int i = 0; i < DPT; ++i) o[i] *= f;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (m[u] == -INFINITY) continue;
      const float g = exp2f(m[u] - Mb) * l[u];
      L += g;
#pragma unroll
      for (int i = 0; i < DPT; ++i) o[i] += g * v[u][i];
    }
    M = Mb;
  }
  const float inv = L > 0.f ? 1.0f / L : 0.f;
#pragma unroll
  for (int i = 0; i < DPT; ++i) o[i] *= inv;
  if (d >= kD - 64) {   // the rotated dims: pairs (2i, 2i+1) lie inside one thread's dims
#pragma unroll
    for (int i = 0; i < DPT; i += 2) {
      const int kk = (d + i - (kD - 64)) / 2;
      const float c = a.q_rope[size_t(b) * 64 + 2 * kk], s = a.q_rope[size_t(b) * 64 + 2 * kk + 1];
      const float y0 = o[i], y1 = o[i + 1];
      o[i] = y0 * c + y1 * s;
      o[i + 1] = -y0 * s + y1 * c;
    }
  }
  uint32_t r[DPT / 2];
#pragma unroll
  for (int i = 0; i < DPT; i += 2) {
    __nv_bfloat162 x = __floats2bfloat162_rn(o[i], o[i + 1]);
    r[i / 2] = *reinterpret_cast<uint32_t*>(&x);
  }
  const size_t off = ((size_t(b) * a.H + h) * kD + d) * 2;
  if constexpr (DPT == 2) {
    *reinterpret_cast<uint32_t*>(a.out + off) = r[0];
    if (a.out_host != nullptr) *reinterpret_cast<uint32_t*>(a.out_host + off) = r[0];
  } else {
    static_assert(DPT == 8, "2 or 8 dims per thread");
    const uint4 x = make_uint4(r[0], r[1], r[2], r[3]);
    *reinterpret_cast<uint4*>(a.out + off) = x;
    if (a.out_host != nullptr) *reinterpret_cast<uint4*>(a.out_host + off) = x;
  }
}

int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

// 16 KiB of slack keeps every descriptor-addressed read inside the allocation
size_t attn_smem_bytes() { return 1024 + 8 * kKeys * 128 + 8 * kMaxHeadsPerBlock * 128 + sizeof(AttnSmem) + 16384; }

}  // namespace

size_t attn_workspace_bytes(int B, int H, int max_ctx, int ratio, int k) {
  return attn_layout(B, H, max_ctx, ratio, k).total;
}

static cudaError_t launch_attn(const void* q, const cskv_paged& kv, const void* swa, const cskv_paged* win,
                               int swa_fmt, const int32_t* req_of, const int32_t* ctx_len, const int32_t* topk,
                               int k, int ratio, int max_ctx, const float* sink, float softmax_scale,
                               const float* q_rope, int B, int H, void* out, void* out_host, void* workspace,
                               cudaStream_t stream, const uint32_t* ready) {
  const AttnLayout L = attn_layout(B, H, max_ctx, ratio, topk ? k : 0);
  AttnArgs a;
  a.q = static_cast<const uint8_t*>(q);
  a.kv = kv;
  a.kv_row_bytes = static_cast<int>(cskv_row_bytes(kv.fmt, kv.dim));
  a.swa = static_cast<const uint8_t*>(swa);
  a.swa_fmt = swa_fmt;
  a.swa_row_bytes = static_cast<int>(cskv_row_bytes(swa_fmt, kD));
  a.win = win ? *win : cskv_paged{};
  a.req_of = req_of;
  a.ctx_len = ctx_len;
  a.topk = topk;
  a.k = k;
  a.ratio = ratio;
  a.max_ctx = max_ctx;
  a.sink = sink;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.q_rope = q_rope;
  a.B = B;
  a.H = H;
  a.out = static_cast<uint8_t*>(out);
  a.opart = reinterpret_cast<__nv_bfloat16*>(static_cast<uint8_t*>(workspace) + L.opart);
  a.ml = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + L.ml);
  a.max_tiles = L.max_tiles;
  a.out_host = static_cast<uint8_t*>(out_host);
  a.ready = ready;
  a.spin = spin_limit();
  const size_t smem = attn_smem_bytes();
  cudaFuncSetAttribute(attn_tile_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  // A tile's heads in one block, or in blocks of 32 when the grid would otherwise leave
  // most SMs idle (a decode batch of a few long requests): each block then repeats the
  // tile's gather and dequantisation, but its products, softmax and partial are half as
  // long, and the tile's latency is what the step waits for.
  a.heads_per_block = (H > 32 && static_cast<long long>(L.max_tiles) * B * ((H + 31) / 32) <= num_sms())
                          ? 32 : kMaxHeadsPerBlock;
  dim3 grid(L.max_tiles, B, (H + a.heads_per_block - 1) / a.heads_per_block);
  // both kernels are programmatic dependents of the work before them in the stream
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, attn_tile_kernel, a);
  if (e != cudaSuccess) return e;
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  // four heads per block: few enough blocks to be resident beside the tiles from the
  // start (a decode step's 128 for 8 requests), so that they begin the moment the tiles'
  // grid completes
  cfg.gridDim = dim3(B, (H + 3) / 4);
  return cudaLaunchKernelEx(&cfg, attn_combine_kernel<8>, a);
}

cudaError_t launch_sparse_decode_attn(const void* q, const cskv_paged& kv, const void* swa, int swa_fmt,
                                      const int32_t* ctx_len, const int32_t* topk, int k, int ratio,
                                      int max_ctx, const float* sink, float softmax_scale,
                                      const float* q_rope, int B, int H, void* out, void* workspace,
                                      cudaStream_t stream, void* out_host, const uint32_t* ready) {
  return launch_attn(q, kv, swa, nullptr, swa_fmt, nullptr, ctx_len, topk, k, ratio, max_ctx, sink,
                     softmax_scale, q_rope, B, H, out, out_host, workspace, stream, ready);
}

cudaError_t launch_sparse_prefill_attn(const void* q, const cskv_paged& kv, const cskv_paged& win,
                                       const int32_t* req_of, const int32_t* pos1, const int32_t* topk, int k,
                                       int ratio, int max_ctx, const float* sink, float softmax_scale,
                                       const float* q_rope, int T, int H, void* out, void* workspace,
                                       cudaStream_t stream) {
  return launch_attn(q, kv, nullptr, &win, win.fmt, req_of, pos1, topk, k, ratio, max_ctx, sink, softmax_scale,
                     q_rope, T, H, out, nullptr, workspace, stream, nullptr);
}

unsigned int take_err_attention() { return take_dev_err(); }

}  // namespace cskv
