// The KV compressor (cskv_compress) and the row coder (cskv_encode_rows).
//
// "DeepSeek-V4 deep dive", section 4.1: entry i pools, channel by channel, the
// softmax over its slots of (gate + slot bias) times the projected values;
// section 4.2: ratio 4 reads the previous block through channel half 0 and its
// own block through half 1 (8 slots, bias added before the transform, the first
// entry's missing half has value 0 and score -inf); ratio 128 pools its own 128
// tokens; then RMSNorm over the channels and RoPE on the last 64 dims at the
// position of the entry's first token.
//
// Design: threads own 4 consecutive channels (8-byte bf16 loads, coalesced across
// the group); an entry of D channels is a group of D/4 threads (one warp at
// D = 128, the whole 128-thread block at D = 512).  The slots' rows are staged in
// shared memory by cp.async, eight slots per batch, two batches in flight.  The
// arithmetic is the bit-exact fp32 contract: separately rounded __f*_rn
// operations (never contracted to FMA), exp_own below, a pairwise sum of squares
// that follows the channel order (in-thread pairs, then warp xor-shuffles, then
// the warps of the block), and the coding of codec.cuh.
#include "codec.cuh"
#include "internal.h"

namespace cskv {

// ---------------------------------------------------------------------------
// exp_own: e^x in a fixed fp32 operation order (Cody & Waite range reduction,
// degree-7 Taylor polynomial).  Constants derived from ln 2: LN2_HI is ln 2 to
// 16 significant bits (so n * LN2_HI is exact), LN2_LO the fp32 remainder,
// C_k = fp32(1/k!).  Returns 0 below 2^-126 and for -inf.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float exp_own(float x) {
  // every constant is the fp32 rounding of a double-precision expression
  constexpr double kLn2 = 0.69314718055994530942;
  const float kLog2e = static_cast<float>(1.0 / kLn2);
  const float kLn2Hi = 0.693145751953125f;                       // 45426 / 65536
  const float kLn2Lo = static_cast<float>(kLn2 - 0.693145751953125);
  const float t = __fmul_rn(x, kLog2e);
  if (!(t >= -126.0f)) return 0.0f;
  const float n = rintf(t);
  const float r = __fsub_rn(__fsub_rn(x, __fmul_rn(n, kLn2Hi)), __fmul_rn(n, kLn2Lo));
  float p = static_cast<float>(1.0 / 5040.0);
  p = __fadd_rn(__fmul_rn(p, r), static_cast<float>(1.0 / 720.0));
  p = __fadd_rn(__fmul_rn(p, r), static_cast<float>(1.0 / 120.0));
  p = __fadd_rn(__fmul_rn(p, r), static_cast<float>(1.0 / 24.0));
  p = __fadd_rn(__fmul_rn(p, r), static_cast<float>(1.0 / 6.0));
  p = __fadd_rn(__fmul_rn(p, r), 0.5f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);
  return __fmul_rn(p, exp2i(static_cast<int>(n)));
}

struct CompressArgs {
  const uint8_t* kv;
  const uint8_t* gate;
  const uint8_t* prev_kv;
  const uint8_t* prev_gate;
  const float* ape;
  const float* norm_w;
  const float* rope_cs;
  const int32_t* req;
  const int32_t* first_entry;
  float eps;
  int S, T, ratio, overlap, n;  // n = T / ratio entries per sequence
  cskv_paged out;
  int out_row_bytes;
  // Decode mode (pos != nullptr): sequence s is request s's state ring and only its
  // last entry (i = n - 1) is computed, when the token at position pos[s] completes
  // its block (always with ring > 0); it goes to row (pos + 1) / ratio - 1 of
  // request s, or to row pos % ring; rope_cs holds one (cos, sin) row per request.
  const int32_t* pos;
  int ring;
};

// bf16 row pointer of token `tok` (channel half `half`) of sequence s.
__device__ __forceinline__ const uint8_t* tok_ptr(const uint8_t* base, long long s, long long T,
                                                  long long tok, int coff, int half, int D) {
  return base + (((s * T + tok) * coff + half) * D) * 2;
}

template <int D>
__device__ __forceinline__ float block_sum_pairwise(float v, int lt) {
  // channel groups of 4 are already reduced in-thread; now threads in channel
  // order: xor 1, 2, 4, 8, 16 inside a warp ...
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  if constexpr (D == 512) {
    // ... then the four warps of the block: (w0 + w1) + (w2 + w3)
    __shared__ float part[4];
    if ((lt & 31) == 0) part[lt >> 5] = v;
    __syncthreads();
    v = __fadd_rn(__fadd_rn(part[0], part[1]), __fadd_rn(part[2], part[3]));
  }
  return v;
}

constexpr int kBatch = 8;   // slots staged per batch
constexpr size_t kCompressSmem = 2 * kBatch * 128 * (8 + 8 + 16);   // two batches of kv, gate, bias

// The entries of block `blk` of one compressor job (a whole 128-thread block).
template <int D>
__device__ __forceinline__ void compress_block(const CompressArgs& a, long long blk) {
  constexpr int TPE = D / 4;        // threads per entry
  constexpr int EPB = 128 / TPE;    // entries per block
  const int lt = threadIdx.x % TPE;
  const long long gentry = blk * EPB + threadIdx.x / TPE;
  const bool dec = a.pos != nullptr;
  const long long total = dec ? a.S : static_cast<long long>(a.S) * a.n;
  bool live = gentry < total;
  int p = 0;
  if (dec && live) {
    p = a.pos[gentry];
    live = p >= 0 && (a.ring > 0 || (p + 1) % a.ratio == 0);   // p < 0: no token this step
  }
  // D == 512: one entry per block, the whole block stays for the block-wide sum.
  if (!live && D != 512) return;
  const long long s = live ? (dec ? gentry : gentry / a.n) : 0;
  const int i = live ? (dec ? a.n - 1 : static_cast<int>(gentry % a.n)) : 0;
  const int c0 = 4 * lt;
  const int r = a.ratio;
  const int coff = a.overlap ? 2 : 1;
  const int slots = a.overlap ? 2 * r : r;

  // slot j -> (value row, score row, bias offset in ape); nullptr value = the empty half
  auto slot_src = [&](int j, const uint8_t*& vp, const uint8_t*& gp, long long& ao) {
    if (a.overlap && j < r) {
      ao = static_cast<long long>(j) * coff * D + c0;   // half 0 bias
      if (i > 0) {
        const long long tok = static_cast<long long>(i - 1) * r + j;
        vp = tok_ptr(a.kv, s, a.T, tok, coff, 0, D) + 2 * c0;
        gp = a.gate ? tok_ptr(a.gate, s, a.T, tok, coff, 0, D) + 2 * c0 : nullptr;
      } else if (a.prev_kv != nullptr) {
        vp = tok_ptr(a.prev_kv, s, r, j, 2, 0, D) + 2 * c0;
        gp = tok_ptr(a.prev_gate, s, r, j, 2, 0, D) + 2 * c0;
      } else {
        vp = nullptr;
        gp = nullptr;
      }
    } else {
      const int jj = a.overlap ? j - r : j;
      const int half = a.overlap ? 1 : 0;
      const long long tok = static_cast<long long>(i) * r + jj;
      ao = static_cast<long long>(jj) * coff * D + half * D + c0;
      vp = tok_ptr(a.kv, s, a.T, tok, coff, half, D) + 2 * c0;
      gp = a.gate ? tok_ptr(a.gate, s, a.T, tok, coff, half, D) + 2 * c0 : nullptr;   // no gate: scores 0
    }
  };
  // Loads that do not depend on the slots go first, so their latency (and the
  // req -> block table -> row chain) overlaps the slot loops.
  RowPtr dst{nullptr, nullptr};
  if (live) {
    const long long row = dec ? (a.ring > 0 ? p % a.ring : (p + 1) / a.ratio - 1)
                              : static_cast<long long>(a.first_entry[s]) + i;
    dst = paged_row(a.out, dec ? static_cast<int>(s) : a.req[s], row, a.out_row_bytes);
  }
  const float4 nw = a.norm_w != nullptr ? *reinterpret_cast<const float4*>(a.norm_w + c0)
                                        : make_float4(1.f, 1.f, 1.f, 1.f);
  const bool rotate = a.rope_cs != nullptr && live && c0 >= D - 64;
  const float4 cs = rotate ? *reinterpret_cast<const float4*>(
                                 a.rope_cs + ((dec ? s : s * a.n + i) * 32 + (c0 - (D - 64)) / 2) * 2)
                           : make_float4(1.f, 0.f, 1.f, 0.f);

  // Slots are staged through shared memory in batches of kBatch with cp.async (the
  // next batch's copies in flight while this one is computed), then taken one at a
  // time in slot order by a rolled loop: the kernel runs once per decode step from
  // a cold instruction cache, so its code stays small.  Each thread copies and reads
  // only its own channels, so no block barrier is needed around the stages.
  extern __shared__ __align__(16) uint8_t cmp_smem[];
  uint2* s_kv = reinterpret_cast<uint2*>(cmp_smem);                 // [2][kBatch][128]
  uint2* s_g = s_kv + 2 * kBatch * 128;                              // [2][kBatch][128]
  float4* s_ap = reinterpret_cast<float4*>(s_g + 2 * kBatch * 128);  // [2][kBatch][128]
  const int t = threadIdx.x;
  const int nbatch = (slots + kBatch - 1) / kBatch;
  auto issue = [&](int bt) {
    const int buf = bt & 1;
#pragma unroll 1
    for (int u = 0; u < kBatch; ++u) {
      const int j = bt * kBatch + u;
      if (live && j < slots) {
        const uint8_t *vp, *gp;
        long long ao;
        slot_src(j, vp, gp, ao);
        if (vp != nullptr) {
          cp_async8(&s_kv[(buf * kBatch + u) * 128 + t], vp);
          if (gp != nullptr) cp_async8(&s_g[(buf * kBatch + u) * 128 + t], gp);
        }
        if (a.ape != nullptr) cp_async16(&s_ap[(buf * kBatch + u) * 128 + t], a.ape + ao);
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  // which slots are the empty half, and which have gate scores (the same cases as
  // slot_src, without its addresses): slot_at reads the staged copies by these alone
  const bool first_half_empty = a.overlap && i == 0 && a.prev_kv == nullptr;
  const bool first_half_gated = i > 0 ? a.gate != nullptr : a.prev_kv != nullptr;
  // slot j's biased score (-inf for the empty half) and, if wanted, its value
  auto slot_at = [&](int j, float4& sc, float4* v) {
    const int buf = (j / kBatch) & 1, u = j % kBatch;
    const bool first = a.overlap && j < r;
    if (first && first_half_empty) {
      sc = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      if (v) *v = make_float4(0.f, 0.f, 0.f, 0.f);
      return;
    }
    const bool gated = first ? first_half_gated : a.gate != nullptr;
    const uint2 g = gated ? s_g[(buf * kBatch + u) * 128 + t] : make_uint2(0u, 0u);
    // no slot bias (ape == nullptr) adds +0: the same bits as a zero bias table
    const float4 b = a.ape != nullptr ? s_ap[(buf * kBatch + u) * 128 + t] : make_float4(0.f, 0.f, 0.f, 0.f);
    sc = make_float4(__fadd_rn(bf16lo(g.x), b.x), __fadd_rn(bf16hi(g.x), b.y), __fadd_rn(bf16lo(g.y), b.z),
                     __fadd_rn(bf16hi(g.y), b.w));
    if (v) {
      const uint2 x = s_kv[(buf * kBatch + u) * 128 + t];
      *v = make_float4(bf16lo(x.x), bf16hi(x.x), bf16lo(x.y), bf16hi(x.y));
    }
  };

  float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
  float4 den = make_float4(0.f, 0.f, 0.f, 0.f);
  float4 m = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  // pass 1: m = max over slots of the biased scores; pass 2: weights and slot-ordered
  // sums (the scores recomputed bit for bit).  One batch: the stage serves both passes.
#pragma unroll 1
  for (int pass = 1; pass <= 2; ++pass) {
    const bool reuse = pass == 2 && nbatch == 1;
    if (!reuse) issue(0);
#pragma unroll 1
    for (int bt = 0; bt < nbatch; ++bt) {
      if (!reuse) {
        if (bt + 1 < nbatch) issue(bt + 1);
        else asm volatile("cp.async.commit_group;" ::: "memory");
        asm volatile("cp.async.wait_group 1;" ::: "memory");
      }
      if (!live) continue;
#pragma unroll 1
      for (int j = bt * kBatch; j < min(slots, (bt + 1) * kBatch); ++j) {
        float4 sc, v;
        if (pass == 1) {
          slot_at(j, sc, nullptr);
          m.x = fmaxf(m.x, sc.x); m.y = fmaxf(m.y, sc.y); m.z = fmaxf(m.z, sc.z); m.w = fmaxf(m.w, sc.w);
        } else {
          slot_at(j, sc, &v);
          const float e0 = exp_own(__fsub_rn(sc.x, m.x)), e1 = exp_own(__fsub_rn(sc.y, m.y));
          const float e2 = exp_own(__fsub_rn(sc.z, m.z)), e3 = exp_own(__fsub_rn(sc.w, m.w));
          num.x = __fadd_rn(num.x, __fmul_rn(e0, v.x)); den.x = __fadd_rn(den.x, e0);
          num.y = __fadd_rn(num.y, __fmul_rn(e1, v.y)); den.y = __fadd_rn(den.y, e1);
          num.z = __fadd_rn(num.z, __fmul_rn(e2, v.z)); den.z = __fadd_rn(den.z, e2);
          num.w = __fadd_rn(num.w, __fmul_rn(e3, v.w)); den.w = __fadd_rn(den.w, e3);
        }
      }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
  }
  float4 y = live ? make_float4(__fdiv_rn(num.x, den.x), __fdiv_rn(num.y, den.y),
                                __fdiv_rn(num.z, den.z), __fdiv_rn(num.w, den.w))
                  : make_float4(0.f, 0.f, 0.f, 0.f);

  if (a.norm_w != nullptr) {
    const float local = __fadd_rn(__fadd_rn(__fmul_rn(y.x, y.x), __fmul_rn(y.y, y.y)),
                                  __fadd_rn(__fmul_rn(y.z, y.z), __fmul_rn(y.w, y.w)));
    const float ss = block_sum_pairwise<D>(local, threadIdx.x % 128);
    const float rr = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(D)), a.eps)));
    y.x = __fmul_rn(__fmul_rn(y.x, rr), nw.x);
    y.y = __fmul_rn(__fmul_rn(y.y, rr), nw.y);
    y.z = __fmul_rn(__fmul_rn(y.z, rr), nw.z);
    y.w = __fmul_rn(__fmul_rn(y.w, rr), nw.w);
  }
  if (rotate) {
    const float y0 = y.x, y1 = y.y, y2 = y.z, y3 = y.w;
    y.x = __fsub_rn(__fmul_rn(y0, cs.x), __fmul_rn(y1, cs.y));
    y.y = __fadd_rn(__fmul_rn(y0, cs.y), __fmul_rn(y1, cs.x));
    y.z = __fsub_rn(__fmul_rn(y2, cs.z), __fmul_rn(y3, cs.w));
    y.w = __fadd_rn(__fmul_rn(y2, cs.w), __fmul_rn(y3, cs.z));
  }
  store_row_values(y, lt, a.out.fmt, D, dst, live && dst.data != nullptr);
}

// Blocks of one entry (D = 512) or four entries (D = 128).
inline long long compress_blocks(int S, int n, int dim) {
  const long long total = static_cast<long long>(S) * n;
  return dim == 512 ? total : (total + 3) / 4;
}

template <int D>
__global__ void __launch_bounds__(128) compress_kernel(const CompressArgs a) {
  grid_dep_launch();   // a programmatic dependent (the indexer's query prep) may start
  compress_block<D>(a, blockIdx.x);
}

// Several jobs in one launch: block b belongs to the job j with first[j] <= b < first[j + 1].
constexpr int kMaxCompressJobs = 4;
struct CompressMany {
  CompressArgs job[kMaxCompressJobs];
  int dim[kMaxCompressJobs];
  long long first[kMaxCompressJobs + 1];
  int njobs;
};

__global__ void __launch_bounds__(128) compress_many_kernel(const __grid_constant__ CompressMany m) {
  grid_dep_launch();
  int j = 0;
  while (j + 1 < m.njobs && static_cast<long long>(blockIdx.x) >= m.first[j + 1]) ++j;
  const long long blk = blockIdx.x - m.first[j];
  if (m.dim[j] == 512) compress_block<512>(m.job[j], blk);
  else compress_block<128>(m.job[j], blk);
}

// ---------------------------------------------------------------------------
// The decode step's state update ("DeepSeek-V4 deep dive", section 4.3 and the
// implementation notes to section 4): each request's new token goes into slot
// (overlap ? r : 0) + p mod r of its compressor's state ring ([2 blocks or 1] x r
// tokens x coff x D, bf16); a token that completes its block (p + 1 = 0 mod r)
// has the block's entry pooled from the ring (the previous block through half 0,
// this one through half 1) and written as entry (p + 1) / r - 1, and with overlap
// the block then moves into the previous-block slots.  A ratio-1 job pools
// nothing: its entry is the token itself, normalised, rotated and coded, written
// to row p or, with a ring, to row p mod ring (the 128-slot window).
// ---------------------------------------------------------------------------
constexpr int kMaxDecodeJobs = 8;
struct DecodeJob {
  CompressArgs a;           // decode mode; kv / gate = the state ring (ratio > 1) or the token (ratio 1)
  const uint8_t* tok_kv;    // bf16 [S, coff, D]: the new tokens (ratio > 1)
  const uint8_t* tok_gate;
  int dim;
};
struct DecodeMany {
  DecodeJob job[kMaxDecodeJobs];
  long long first[kMaxDecodeJobs + 1];
  int njobs;
};

template <int D>
__device__ __forceinline__ void decode_block(const DecodeJob& q, long long blk) {
  const CompressArgs& a = q.a;
  constexpr int TPE = D / 4;
  constexpr int EPB = 128 / TPE;
  const int lt = threadIdx.x % TPE;
  const long long s = blk * EPB + threadIdx.x / TPE;
  const int r = a.ratio;
  const int coff = a.overlap ? 2 : 1;
  const int p = s < a.S ? a.pos[s] : -1;
  const bool ringed = r > 1;
  uint8_t* ring_kv = const_cast<uint8_t*>(a.kv);
  uint8_t* ring_gate = const_cast<uint8_t*>(a.gate);
  // byte offset of (request s, ring slot, half h, this thread's 4 channels)
  const long long base = (s * a.T * coff * D + 4 * lt) * 2;
#define CSKV_RING_AT(slot, h) (base + ((static_cast<long long>(slot) * coff + (h)) * D) * 2)
  if (ringed && p >= 0) {
    const int slot = (a.overlap ? r : 0) + p % r;
#pragma unroll 1
    for (int h = 0; h < coff; ++h) {
      const long long src = ((s * coff + h) * D + 4 * lt) * 2;
      *reinterpret_cast<uint2*>(ring_kv + CSKV_RING_AT(slot, h)) = *reinterpret_cast<const uint2*>(q.tok_kv + src);
      *reinterpret_cast<uint2*>(ring_gate + CSKV_RING_AT(slot, h)) = *reinterpret_cast<const uint2*>(q.tok_gate + src);
    }
    __threadfence();   // the pooling below reads this slot back with cp.async
  }
  __syncthreads();
  compress_block<D>(a, blk);
  // the overlap shift (each thread moves its own channels, which the pooling has
  // finished reading: compress_block waits for all of its copies)
  if (ringed && a.overlap && p >= 0 && (p + 1) % r == 0) {
#pragma unroll 1
    for (int j = 0; j < r; ++j) {
#pragma unroll 1
      for (int h = 0; h < coff; ++h) {
        *reinterpret_cast<uint2*>(ring_kv + CSKV_RING_AT(j, h)) = *reinterpret_cast<const uint2*>(ring_kv + CSKV_RING_AT(r + j, h));
        *reinterpret_cast<uint2*>(ring_gate + CSKV_RING_AT(j, h)) = *reinterpret_cast<const uint2*>(ring_gate + CSKV_RING_AT(r + j, h));
      }
    }
  }
}
#undef CSKV_RING_AT

__global__ void __launch_bounds__(128, 1) decode_append_kernel(const __grid_constant__ DecodeMany m) {
  grid_dep_launch();
  int j = 0;
  while (j + 1 < m.njobs && static_cast<long long>(blockIdx.x) >= m.first[j + 1]) ++j;
  const long long blk = blockIdx.x - m.first[j];
  if (m.job[j].dim == 512) decode_block<512>(m.job[j], blk);
  else decode_block<128>(m.job[j], blk);
}

struct EncodeArgs {
  const uint8_t* src;
  int src_bf16;
  int n;
  const int32_t* req;
  const int32_t* row;
  cskv_paged out;
  int out_row_bytes;
};

template <int D>
__global__ void __launch_bounds__(128) encode_rows_kernel(const EncodeArgs a) {
  constexpr int TPE = D / 4;
  constexpr int EPB = 128 / TPE;
  const int lt = threadIdx.x % TPE;
  const long long i = static_cast<long long>(blockIdx.x) * EPB + threadIdx.x / TPE;
  if (i >= a.n) return;   // whole groups leave together
  float4 y;
  if (a.src_bf16) {
    y = load_bf16x4(a.src + (i * D + 4 * lt) * 2);
  } else {
    y = *reinterpret_cast<const float4*>(a.src + (i * D + 4 * lt) * 4);
  }
  const int req = a.req ? a.req[i] : 0;
  const long long row = a.row ? a.row[i] : i;
  const RowPtr dst = paged_row(a.out, req, row, a.out_row_bytes);
  store_row_values(y, lt, a.out.fmt, D, dst, dst.data != nullptr);
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
static CompressArgs compress_args(const void* kv, const void* gate, const void* prev_kv,
                                  const void* prev_gate, const float* ape, const float* norm_w, float eps,
                                  const float* rope_cs, int S, int T, int ratio, int overlap,
                                  const int32_t* req, const int32_t* first_entry, const cskv_paged& out,
                                  int out_row_bytes) {
  CompressArgs a;
  a.kv = static_cast<const uint8_t*>(kv);
  a.gate = static_cast<const uint8_t*>(gate);
  a.prev_kv = static_cast<const uint8_t*>(prev_kv);
  a.prev_gate = static_cast<const uint8_t*>(prev_gate);
  a.ape = ape;
  a.norm_w = norm_w;
  a.rope_cs = rope_cs;
  a.req = req;
  a.first_entry = first_entry;
  a.eps = eps;
  a.S = S;
  a.T = T;
  a.ratio = ratio;
  a.overlap = overlap;
  a.n = T / ratio;
  a.out = out;
  a.out_row_bytes = out_row_bytes;
  a.pos = nullptr;
  a.ring = 0;
  return a;
}

cudaError_t launch_compress(const void* kv, const void* gate, const void* prev_kv,
                            const void* prev_gate, const float* ape, const float* norm_w, float eps,
                            const float* rope_cs, int S, int T, int ratio, int overlap, int dim,
                            const int32_t* req, const int32_t* first_entry, const cskv_paged& out,
                            int out_row_bytes, cudaStream_t stream) {
  const CompressArgs a = compress_args(kv, gate, prev_kv, prev_gate, ape, norm_w, eps, rope_cs, S, T, ratio,
                                       overlap, req, first_entry, out, out_row_bytes);
  const long long total = static_cast<long long>(S) * a.n;
  if (total == 0) return cudaSuccess;
  if (dim == 512) {
    cudaFuncSetAttribute(compress_kernel<512>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(kCompressSmem));
    compress_kernel<512><<<static_cast<unsigned>(total), 128, kCompressSmem, stream>>>(a);
  } else {
    cudaFuncSetAttribute(compress_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(kCompressSmem));
    compress_kernel<128><<<static_cast<unsigned>((total + 3) / 4), 128, kCompressSmem, stream>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_compress_many(const cskv_compress_job* jobs, int njobs, cudaStream_t stream) {
  if (njobs < 1 || njobs > kMaxCompressJobs) return cudaErrorInvalidValue;
  CompressMany m;
  m.njobs = njobs;
  m.first[0] = 0;
  for (int j = 0; j < njobs; ++j) {
    const cskv_compress_job& q = jobs[j];
    m.job[j] = compress_args(q.kv, q.gate, q.prev_kv, q.prev_gate, q.ape, q.norm_w, q.eps, q.rope_cs, q.S, q.T,
                             q.ratio, q.overlap, q.req, q.first_entry, q.out,
                             static_cast<int>(cskv_row_bytes(q.out.fmt, q.dim)));
    m.dim[j] = q.dim;
    m.first[j + 1] = m.first[j] + compress_blocks(q.S, q.T / q.ratio, q.dim);
  }
  if (m.first[njobs] == 0) return cudaSuccess;
  cudaFuncSetAttribute(compress_many_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       static_cast<int>(kCompressSmem));
  compress_many_kernel<<<static_cast<unsigned>(m.first[njobs]), 128, kCompressSmem, stream>>>(m);
  return cudaGetLastError();
}

cudaError_t launch_decode_append(const cskv_decode_job* jobs, int njobs, const int32_t* pos, int B,
                                 cudaStream_t stream) {
  if (njobs < 1 || njobs > kMaxDecodeJobs) return cudaErrorInvalidValue;
  DecodeMany m;
  m.njobs = njobs;
  m.first[0] = 0;
  for (int j = 0; j < njobs; ++j) {
    const cskv_decode_job& q = jobs[j];
    const bool ringed = q.ratio > 1;
    const int T = ringed ? (q.overlap ? 2 : 1) * q.ratio : 1;
    m.job[j].a = compress_args(ringed ? q.state_kv : q.kv, ringed ? q.state_gate : q.gate, nullptr, nullptr, q.ape,
                               q.norm_w, q.eps, q.rope_cs, B, T, q.ratio, q.overlap, nullptr, nullptr, q.out,
                               static_cast<int>(cskv_row_bytes(q.out.fmt, q.dim)));
    m.job[j].a.pos = pos;
    m.job[j].a.ring = q.ring_rows;
    m.job[j].tok_kv = static_cast<const uint8_t*>(q.kv);
    m.job[j].tok_gate = static_cast<const uint8_t*>(q.gate);
    m.job[j].dim = q.dim;
    m.first[j + 1] = m.first[j] + compress_blocks(B, 1, q.dim);
  }
  if (m.first[njobs] == 0) return cudaSuccess;
  cudaFuncSetAttribute(decode_append_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       static_cast<int>(kCompressSmem));
  decode_append_kernel<<<static_cast<unsigned>(m.first[njobs]), 128, kCompressSmem, stream>>>(m);
  return cudaGetLastError();
}

cudaError_t launch_encode_rows(const void* src, int src_bf16, int n, int dim, const int32_t* req,
                               const int32_t* row, const cskv_paged& out, int out_row_bytes,
                               cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  EncodeArgs a{static_cast<const uint8_t*>(src), src_bf16, n, req, row, out, out_row_bytes};
  if (dim == 512) {
    encode_rows_kernel<512><<<static_cast<unsigned>(n), 128, 0, stream>>>(a);
  } else {
    encode_rows_kernel<128><<<static_cast<unsigned>((n + 3) / 4), 128, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

unsigned int take_err_compress() { return take_dev_err(); }

}  // namespace cskv
