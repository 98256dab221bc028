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
// Design: threads own CPT consecutive channels (CPT = 2 for the compressor launches,
// 256-thread blocks; 4 for the decode state update, 128-thread blocks); an entry of
// D channels is a group of D/CPT threads (a whole block at D = 512; at D = 128 one
// warp with CPT = 4, two with CPT = 2).  The slots' rows are staged in
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

template <int D, int CPT>
__device__ __forceinline__ float block_sum_pairwise(float v) {
  // channel groups of CPT are already reduced in-thread (pairwise); now threads in
  // channel order: xor 1, 2, 4, 8, 16 inside a warp ...
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  // ... then the warps of the entry, pairwise in channel order (every level of the
  // tree sums two halves of equal size, as in the in-thread and shuffle levels)
  constexpr int kWarps = D / CPT / 32;
  if constexpr (kWarps > 1) {
    __shared__ float part[8];
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) part[w] = v;
    __syncthreads();
    const float* q = part + (w / kWarps) * kWarps;   // this entry's warps
    if constexpr (kWarps == 2) {
      v = __fadd_rn(q[0], q[1]);
    } else if constexpr (kWarps == 4) {
      v = __fadd_rn(__fadd_rn(q[0], q[1]), __fadd_rn(q[2], q[3]));
    } else {
      static_assert(kWarps == 8, "2, 4 or 8 warps per entry");
      v = __fadd_rn(__fadd_rn(__fadd_rn(q[0], q[1]), __fadd_rn(q[2], q[3])),
                    __fadd_rn(__fadd_rn(q[4], q[5]), __fadd_rn(q[6], q[7])));
    }
    __syncthreads();   // part is reused by the next sum
  }
  return v;
}

constexpr int kBatch = 8;   // slots staged per batch
// two batches of kv, gate, bias for 128 threads x 4 channels or 256 threads x 2
constexpr size_t kCompressSmem = 2 * kBatch * 128 * (8 + 8 + 16);

// This thread's CPT channels of a staged bf16 row (KvT) and of the fp32 bias (BiasT).
template <int CPT> struct Lanes;
template <> struct Lanes<4> {
  using KvT = uint2;
  using BiasT = float4;
  static __device__ __forceinline__ void kv(const KvT& x, float (&v)[4]) {
    v[0] = bf16lo(x.x); v[1] = bf16hi(x.x); v[2] = bf16lo(x.y); v[3] = bf16hi(x.y);
  }
  static __device__ __forceinline__ void bias(const BiasT& b, float (&v)[4]) {
    v[0] = b.x; v[1] = b.y; v[2] = b.z; v[3] = b.w;
  }
  static __device__ __forceinline__ void copy_kv(void* dst, const void* src) { cp_async8(dst, src); }
  static __device__ __forceinline__ void copy_bias(void* dst, const void* src) { cp_async16(dst, src); }
};
template <> struct Lanes<2> {
  using KvT = uint32_t;
  using BiasT = float2;
  static __device__ __forceinline__ void kv(const KvT& x, float (&v)[2]) { v[0] = bf16lo(x); v[1] = bf16hi(x); }
  static __device__ __forceinline__ void bias(const BiasT& b, float (&v)[2]) { v[0] = b.x; v[1] = b.y; }
  static __device__ __forceinline__ void copy_kv(void* dst, const void* src) { cp_async4(dst, src); }
  static __device__ __forceinline__ void copy_bias(void* dst, const void* src) { cp_async8(dst, src); }
};

// The entries of block `blk` of one compressor job (a whole block of 512 / CPT threads).
template <int D, int CPT>
__device__ __forceinline__ void compress_block(const CompressArgs& a, long long blk) {
  constexpr int kThreads = 512 / CPT;
  constexpr int TPE = D / CPT;            // threads per entry
  constexpr int EPB = kThreads / TPE;     // entries per block
  using L = Lanes<CPT>;
  using KvT = typename L::KvT;
  using BiasT = typename L::BiasT;
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
  // An entry of more than one warp stays for the block-wide sums.
  if (!live && TPE <= 32) return;
  const long long s = live ? (dec ? gentry : gentry / a.n) : 0;
  const int i = live ? (dec ? a.n - 1 : static_cast<int>(gentry % a.n)) : 0;
  const int c0 = CPT * lt;
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
  float nw[CPT], cs[CPT];   // norm weights; (cos, sin) of this thread's CPT / 2 pairs
  if (a.norm_w != nullptr) L::bias(*reinterpret_cast<const BiasT*>(a.norm_w + c0), nw);
  else {
#pragma unroll
    for (int c = 0; c < CPT; ++c) nw[c] = 1.f;
  }
  const bool rotate = a.rope_cs != nullptr && live && c0 >= D - 64;
  if (rotate) {
    L::bias(*reinterpret_cast<const BiasT*>(a.rope_cs + ((dec ? s : s * a.n + i) * 32 + (c0 - (D - 64)) / 2) * 2),
            cs);
  } else {
#pragma unroll
    for (int c = 0; c < CPT; c += 2) { cs[c] = 1.f; cs[c + 1] = 0.f; }
  }

  // Slots are staged through shared memory in batches of kBatch with cp.async (the
  // next batch's copies in flight while this one is computed), then taken one at a
  // time in slot order by a rolled loop: the kernel runs once per decode step from
  // a cold instruction cache, so its code stays small.  Each thread copies and reads
  // only its own channels, so no block barrier is needed around the stages.
  extern __shared__ __align__(16) uint8_t cmp_smem[];
  KvT* s_kv = reinterpret_cast<KvT*>(cmp_smem);                         // [2][kBatch][kThreads]
  KvT* s_g = s_kv + 2 * kBatch * kThreads;                              // [2][kBatch][kThreads]
  BiasT* s_ap = reinterpret_cast<BiasT*>(s_g + 2 * kBatch * kThreads);  // [2][kBatch][kThreads]
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
          L::copy_kv(&s_kv[(buf * kBatch + u) * kThreads + t], vp);
          if (gp != nullptr) L::copy_kv(&s_g[(buf * kBatch + u) * kThreads + t], gp);
        }
        if (a.ape != nullptr) L::copy_bias(&s_ap[(buf * kBatch + u) * kThreads + t], a.ape + ao);
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  // which slots are the empty half, and which have gate scores (the same cases as
  // slot_src, without its addresses): slot_at reads the staged copies by these alone
  const bool first_half_empty = a.overlap && i == 0 && a.prev_kv == nullptr;
  const bool first_half_gated = i > 0 ? a.gate != nullptr : a.prev_kv != nullptr;
  // slot j's biased scores (-inf for the empty half) and, if wanted, its values
  auto slot_at = [&](int j, float (&sc)[CPT], float* v) {
    const int buf = (j / kBatch) & 1, u = j % kBatch;
    const bool first = a.overlap && j < r;
    if (first && first_half_empty) {
#pragma unroll
      for (int c = 0; c < CPT; ++c) {
        sc[c] = -INFINITY;
        if (v) v[c] = 0.f;
      }
      return;
    }
    const bool gated = first ? first_half_gated : a.gate != nullptr;
    float g[CPT], bb[CPT];
    if (gated) L::kv(s_g[(buf * kBatch + u) * kThreads + t], g);
    else {
#pragma unroll
      for (int c = 0; c < CPT; ++c) g[c] = 0.f;
    }
    // no slot bias (ape == nullptr) adds +0: the same bits as a zero bias table
    if (a.ape != nullptr) L::bias(s_ap[(buf * kBatch + u) * kThreads + t], bb);
    else {
#pragma unroll
      for (int c = 0; c < CPT; ++c) bb[c] = 0.f;
    }
#pragma unroll
    for (int c = 0; c < CPT; ++c) sc[c] = __fadd_rn(g[c], bb[c]);
    if (v) {
      float x[CPT];
      L::kv(s_kv[(buf * kBatch + u) * kThreads + t], x);
#pragma unroll
      for (int c = 0; c < CPT; ++c) v[c] = x[c];
    }
  };

  float num[CPT], den[CPT], m[CPT];
#pragma unroll
  for (int c = 0; c < CPT; ++c) {
    num[c] = 0.f;
    den[c] = 0.f;
    m[c] = -INFINITY;
  }
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
        float sc[CPT], v[CPT];
        if (pass == 1) {
          slot_at(j, sc, nullptr);
#pragma unroll
          for (int c = 0; c < CPT; ++c) m[c] = fmaxf(m[c], sc[c]);
        } else {
          slot_at(j, sc, v);
#pragma unroll
          for (int c = 0; c < CPT; ++c) {
            const float e = exp_own(__fsub_rn(sc[c], m[c]));
            num[c] = __fadd_rn(num[c], __fmul_rn(e, v[c]));
            den[c] = __fadd_rn(den[c], e);
          }
        }
      }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
  }
  float y[CPT];
#pragma unroll
  for (int c = 0; c < CPT; ++c) y[c] = live ? __fdiv_rn(num[c], den[c]) : 0.f;

  if (a.norm_w != nullptr) {
    float local;
    if constexpr (CPT == 4) {
      local = __fadd_rn(__fadd_rn(__fmul_rn(y[0], y[0]), __fmul_rn(y[1], y[1])),
                        __fadd_rn(__fmul_rn(y[2], y[2]), __fmul_rn(y[3], y[3])));
    } else {
      local = __fadd_rn(__fmul_rn(y[0], y[0]), __fmul_rn(y[1], y[1]));
    }
    const float ss = block_sum_pairwise<D, CPT>(local);
    const float rr = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(D)), a.eps)));
#pragma unroll
    for (int c = 0; c < CPT; ++c) y[c] = __fmul_rn(__fmul_rn(y[c], rr), nw[c]);
  }
  if (rotate) {
#pragma unroll
    for (int c = 0; c < CPT; c += 2) {
      const float y0 = y[c], y1 = y[c + 1];
      y[c] = __fsub_rn(__fmul_rn(y0, cs[c]), __fmul_rn(y1, cs[c + 1]));
      y[c + 1] = __fadd_rn(__fmul_rn(y0, cs[c + 1]), __fmul_rn(y1, cs[c]));
    }
  }
  if constexpr (CPT == 4) {
    store_row_values(make_float4(y[0], y[1], y[2], y[3]), lt, a.out.fmt, D, dst, live && dst.data != nullptr);
  } else {
    store_row_values2<D>(y[0], y[1], lt, a.out.fmt, dst, live && dst.data != nullptr);
  }
}

// Blocks of one entry (D = 512) or four entries (D = 128).
inline long long compress_blocks(int S, int n, int dim) {
  const long long total = static_cast<long long>(S) * n;
  return dim == 512 ? total : (total + 3) / 4;
}

template <int D>
__global__ void __launch_bounds__(256) compress_kernel(const CompressArgs a) {
  grid_dep_launch();   // a programmatic dependent (the indexer's query prep) may start
  compress_block<D, 2>(a, blockIdx.x);
}

// Several jobs in one launch: block b belongs to the job j with first[j] <= b < first[j + 1].
constexpr int kMaxCompressJobs = 4;
struct CompressMany {
  CompressArgs job[kMaxCompressJobs];
  int dim[kMaxCompressJobs];
  long long first[kMaxCompressJobs + 1];
  int njobs;
};

__global__ void __launch_bounds__(256) compress_many_kernel(const __grid_constant__ CompressMany m) {
  // Launched as a programmatic dependent (a fused decode step, after the indexer's
  // query prep), the kernel lets its own dependent (the score kernel) start only once
  // the kernel before it has completed: the score kernel then reads the prep's output
  // freely and waits for this kernel only before the index keys it writes.  In a
  // plain launch the wait returns at once.
  grid_dep_wait();
  grid_dep_launch();
  int j = 0;
  while (j + 1 < m.njobs && static_cast<long long>(blockIdx.x) >= m.first[j + 1]) ++j;
  const long long blk = blockIdx.x - m.first[j];
  if (m.dim[j] == 512) compress_block<512, 2>(m.job[j], blk);
  else compress_block<128, 2>(m.job[j], blk);
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
  compress_block<D, 4>(a, blk);
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
    compress_kernel<512><<<static_cast<unsigned>(total), 256, kCompressSmem, stream>>>(a);
  } else {
    cudaFuncSetAttribute(compress_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(kCompressSmem));
    compress_kernel<128><<<static_cast<unsigned>((total + 3) / 4), 256, kCompressSmem, stream>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_compress_many(const cskv_compress_job* jobs, int njobs, cudaStream_t stream, bool dependent) {
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
  if (!dependent) {
    compress_many_kernel<<<static_cast<unsigned>(m.first[njobs]), 256, kCompressSmem, stream>>>(m);
    return cudaGetLastError();
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(m.first[njobs]));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = kCompressSmem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, compress_many_kernel, m);
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
