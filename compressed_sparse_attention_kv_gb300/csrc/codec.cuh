// Device codecs of the cache formats and the row writer shared by the
// compressor and cskv_encode_rows.
//
// FP8 rows ("DeepSeek-V4-Flash" model record, engine kernel constraint (2)):
// e4m3 codes over all dims, one e8m0 scale per 32 values.  FP4 rows
// ("DeepSeek-V4.1-Flash" diagram, "The four compression axes"): e2m1 codes, one
// e4m3 scale per 16 channels.  Block rules (fixed here, as the pages give none):
//  - e8m0: the smallest 2^e with amax <= 448 * 2^e, e in [-127, 127]; an
//    all-zero block stores 127; values are RNE(x * 2^-e) saturated to +-448;
//  - FP4: s = RNE_e4m3(amax / 6); s == 0 zeroes the block; nibbles are
//    RNE_e2m1(x / s) saturated to +-6; channel 2i in the low nibble.
// The sign of an input that rounds to zero is kept (IEEE conversion rule).
// Rotated FP4 index keys ("DeepSeek-V4 deep dive", section 5.2: a Hadamard rotation,
// then FP4 rounding with block size 32): the 128 channels are multiplied by
// H / sqrt(128) (H the Sylvester Hadamard matrix) in a fixed fp32 order - butterflies
// of stride 1, 2, ..., 64, each (a, b) -> (a + b, a - b) with a the lower channel,
// then one product by fp32(1 / sqrt(128)) - and coded as e2m1 with one e8m0 scale
// per 32: the smallest 2^e with amax <= 6 * 2^e, nibbles RNE(x * 2^-e).
#pragma once

#include "common.cuh"

namespace cskv {

// Smallest e with amax <= 448 * 2^e, from the bits of amax (amax >= 0, finite).
__device__ __forceinline__ int e8m0_exponent(float amax) {
  if (amax == 0.f) return 0;
  const uint32_t bits = __float_as_uint(amax);
  const int biased = static_cast<int>(bits >> 23);
  const uint32_t mant = bits & 0x7FFFFFu;
  // amax = 1.mant * 2^(biased-127) and 448 = 1.75 * 2^8; 1.75 is mantissa 0x600000
  int e = (mant <= 0x600000u) ? biased - 135 : biased - 134;
  if (biased == 0) e = -127;
  return max(-127, min(127, e));
}

// 2^e as fp32 for e in [-149, 127] (exact; subnormal below -126).
__device__ __forceinline__ float exp2i(int e) {
  return e >= -126 ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23)
                   : __uint_as_float(1u << (e + 149));
}

// Two fp32 -> two e4m3 codes, RNE with saturation; `lo` lands in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two fp32 -> two e2m1 nibbles, RNE with saturation; `lo` lands in the low nibble.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "cvt.u16.u8 %0, t;\n\t}"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// e4m3 code -> fp32 (exact, through the f16x2 conversion).
__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(code & 0xFF)));
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFF)));
}

// Smallest e with amax <= 6 * 2^e (6 = 1.5 * 2^2: mantissa 0x400000), from the bits.
__device__ __forceinline__ int e8m0_exponent_fp4(float amax) {
  if (amax == 0.f) return 0;
  const uint32_t bits = __float_as_uint(amax);
  const int biased = static_cast<int>(bits >> 23);
  const uint32_t mant = bits & 0x7FFFFFu;
  int e = (mant <= 0x400000u) ? biased - 129 : biased - 128;
  if (biased == 0) e = -127;
  return max(-127, min(127, e));
}

// fp32(1 / sqrt(128)), the scale of the rotation
constexpr float kHadamardScale128 = 0x1.6a09e6p-4f;

// The rotation of a 128-channel vector held 4 channels per lane (lane l: channels
// 4l .. 4l+3, the 32 lanes of one warp).
__device__ __forceinline__ void hadamard128_x4(float (&y)[4], int l) {
  float a0 = __fadd_rn(y[0], y[1]), a1 = __fsub_rn(y[0], y[1]);
  float a2 = __fadd_rn(y[2], y[3]), a3 = __fsub_rn(y[2], y[3]);
  y[0] = __fadd_rn(a0, a2);
  y[2] = __fsub_rn(a0, a2);
  y[1] = __fadd_rn(a1, a3);
  y[3] = __fsub_rn(a1, a3);
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {   // stride 4o: partner lane l ^ o
    const bool upper = (l & o) != 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float p = __shfl_xor_sync(0xFFFFFFFFu, y[j], o);
      y[j] = upper ? __fsub_rn(p, y[j]) : __fadd_rn(y[j], p);
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) y[j] = __fmul_rn(y[j], kHadamardScale128);
}

// e2m1 codes of 4 consecutive channels at scale 2^e (16 bits: channel 4l in the low nibble).
__device__ __forceinline__ uint32_t e2m1x4_scaled(const float (&y)[4], int e) {
  const float inv = exp2i(-e);
  return e2m1x2(__fmul_rn(y[0], inv), __fmul_rn(y[1], inv)) | (e2m1x2(__fmul_rn(y[2], inv), __fmul_rn(y[3], inv)) << 8);
}

// Writes one row whose values are spread over the threads of a group: thread
// `lt` holds channels 4*lt .. 4*lt+3 in y.  The groups of 8 (FP8) or 4 (FP4)
// threads that share a scale block must be consecutive lanes of one warp and
// every thread of the group must call this (it shuffles).  `valid` false
// skips the stores (the shuffles still run).
__device__ __forceinline__ void store_row_values(const float4& y, int lt, int fmt, int dim,
                                                 RowPtr dst, bool valid) {
  const unsigned full = 0xFFFFFFFFu;
  if (fmt == CSKV_FMT_BF16) {
    if (valid) {
      __nv_bfloat162 a = __floats2bfloat162_rn(y.x, y.y);
      __nv_bfloat162 b = __floats2bfloat162_rn(y.z, y.w);
      uint2 u;
      u.x = *reinterpret_cast<uint32_t*>(&a);
      u.y = *reinterpret_cast<uint32_t*>(&b);
      *reinterpret_cast<uint2*>(dst.data + 8 * lt) = u;
    }
    return;
  }
  if (fmt == CSKV_FMT_FP4_E2M1_E8M0_HADAMARD_PAGESPLIT) {
    // rotated index key (dim 128: the group is one warp), blocks of 32 channels = 8 lanes
    float v[4] = {y.x, y.y, y.z, y.w};
    hadamard128_x4(v, lt);
    float am = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
    am = fmaxf(am, __shfl_xor_sync(full, am, 1));
    am = fmaxf(am, __shfl_xor_sync(full, am, 2));
    am = fmaxf(am, __shfl_xor_sync(full, am, 4));
    const int e = e8m0_exponent_fp4(am);
    const uint32_t codes = e2m1x4_scaled(v, e);
    if (valid) {
      *reinterpret_cast<uint16_t*>(dst.data + 2 * lt) = static_cast<uint16_t>(codes);
      if ((lt & 7) == 0) dst.scale[lt >> 3] = static_cast<uint8_t>(e + 127);
    }
    return;
  }
  float amax = fmaxf(fmaxf(fabsf(y.x), fabsf(y.y)), fmaxf(fabsf(y.z), fabsf(y.w)));
  if (fmt == CSKV_FMT_FP4_E2M1_E4M3_B16) {
    amax = fmaxf(amax, __shfl_xor_sync(full, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(full, amax, 2));
    const uint32_t scode = e4m3x2(__fdiv_rn(amax, 6.0f), 0.f) & 0xFF;
    const float s = e4m3_to_f32(scode);
    uint32_t packed = 0;
    if (s > 0.f) {
      packed = e2m1x2(__fdiv_rn(y.x, s), __fdiv_rn(y.y, s)) |
               (e2m1x2(__fdiv_rn(y.z, s), __fdiv_rn(y.w, s)) << 8);
    }
    if (valid) {
      *reinterpret_cast<uint16_t*>(dst.data + 2 * lt) = static_cast<uint16_t>(packed);
      if ((lt & 3) == 0) dst.scale[lt >> 2] = static_cast<uint8_t>(scode);
    }
    return;
  }
  if (fmt == CSKV_FMT_FP8_E4M3_ROWSCALE_PAGESPLIT) {
    // index key: one power-of-two scale for the whole row (the group is one warp at dim 128)
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(full, amax, o));
    const int e = e8m0_exponent(amax);
    const float inv = exp2i(-e);
    const uint32_t codes = e4m3x2(__fmul_rn(y.x, inv), __fmul_rn(y.y, inv)) |
                           (e4m3x2(__fmul_rn(y.z, inv), __fmul_rn(y.w, inv)) << 16);
    if (valid) {
      *reinterpret_cast<uint32_t*>(dst.data + 4 * lt) = codes;
      if (lt == 0) *reinterpret_cast<float*>(dst.scale) = exp2i(e);
    }
    return;
  }
  // FP8 inline rows: blocks of 32 channels = 8 threads
  amax = fmaxf(amax, __shfl_xor_sync(full, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(full, amax, 2));
  amax = fmaxf(amax, __shfl_xor_sync(full, amax, 4));
  const int e = e8m0_exponent(amax);
  const float inv = exp2i(-e);
  const uint32_t codes = e4m3x2(__fmul_rn(y.x, inv), __fmul_rn(y.y, inv)) |
                         (e4m3x2(__fmul_rn(y.z, inv), __fmul_rn(y.w, inv)) << 16);
  if (valid) {
    *reinterpret_cast<uint32_t*>(dst.data + 4 * lt) = codes;
    if ((lt & 7) == 0) dst.scale[lt >> 3] = static_cast<uint8_t>(e + 127);
  }
  (void)dim;
}

// store_row_values for threads that own 2 consecutive channels (c0 = 2 lt) of a
// D-channel entry of D / 2 threads (whole warps): the same codes and scales.  The
// row-scaled index key (D = 128, two warps) takes its row maximum across the two
// warps through shared memory, so every thread of the block must call this.
template <int D>
__device__ __forceinline__ void store_row_values2(float y0, float y1, int lt, int fmt, RowPtr dst, bool valid) {
  const unsigned full = 0xFFFFFFFFu;
  if (fmt == CSKV_FMT_BF16) {
    if (valid) {
      __nv_bfloat162 a = __floats2bfloat162_rn(y0, y1);
      *reinterpret_cast<uint32_t*>(dst.data + 4 * lt) = *reinterpret_cast<uint32_t*>(&a);
    }
    return;
  }
  if (fmt == CSKV_FMT_FP4_E2M1_E8M0_HADAMARD_PAGESPLIT) {
    // rotated index key (D = 128: two warps, lane lt holds channels 2lt, 2lt+1); the
    // stride-64 butterfly crosses the warps through shared memory, so every thread of the
    // block calls this
    float a0 = __fadd_rn(y0, y1), a1 = __fsub_rn(y0, y1);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {   // stride 2o: partner lane lt ^ o
      const bool upper = (lt & o) != 0;
      const float p0 = __shfl_xor_sync(full, a0, o), p1 = __shfl_xor_sync(full, a1, o);
      a0 = upper ? __fsub_rn(p0, a0) : __fadd_rn(a0, p0);
      a1 = upper ? __fsub_rn(p1, a1) : __fadd_rn(a1, p1);
    }
    __shared__ float2 xch[256];
    xch[threadIdx.x & 255] = make_float2(a0, a1);
    __syncthreads();
    const float2 p = xch[(threadIdx.x ^ 32) & 255];
    __syncthreads();
    const bool upper = (lt & 32) != 0;
    a0 = upper ? __fsub_rn(p.x, a0) : __fadd_rn(a0, p.x);
    a1 = upper ? __fsub_rn(p.y, a1) : __fadd_rn(a1, p.y);
    a0 = __fmul_rn(a0, kHadamardScale128);
    a1 = __fmul_rn(a1, kHadamardScale128);
    // blocks of 32 channels = 16 lanes
    float am = fmaxf(fabsf(a0), fabsf(a1));
    am = fmaxf(am, __shfl_xor_sync(full, am, 1));
    am = fmaxf(am, __shfl_xor_sync(full, am, 2));
    am = fmaxf(am, __shfl_xor_sync(full, am, 4));
    am = fmaxf(am, __shfl_xor_sync(full, am, 8));
    const int e = e8m0_exponent_fp4(am);
    const float inv = exp2i(-e);
    const uint32_t codes = e2m1x2(__fmul_rn(a0, inv), __fmul_rn(a1, inv));
    if (valid) {
      dst.data[lt] = static_cast<uint8_t>(codes);
      if ((lt & 15) == 0) dst.scale[lt >> 4] = static_cast<uint8_t>(e + 127);
    }
    return;
  }
  float amax = fmaxf(fabsf(y0), fabsf(y1));
  if (fmt == CSKV_FMT_FP4_E2M1_E4M3_B16) {
    // blocks of 16 channels = 8 threads
    amax = fmaxf(amax, __shfl_xor_sync(full, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(full, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(full, amax, 4));
    const uint32_t scode = e4m3x2(__fdiv_rn(amax, 6.0f), 0.f) & 0xFF;
    const float s = e4m3_to_f32(scode);
    const uint32_t packed = s > 0.f ? e2m1x2(__fdiv_rn(y0, s), __fdiv_rn(y1, s)) : 0u;
    if (valid) {
      dst.data[lt] = static_cast<uint8_t>(packed);
      if ((lt & 7) == 0) dst.scale[lt >> 3] = static_cast<uint8_t>(scode);
    }
    return;
  }
  if (fmt == CSKV_FMT_FP8_E4M3_ROWSCALE_PAGESPLIT) {
    // index key: one power-of-two scale for the whole row (D / 2 threads)
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(full, amax, o));
    constexpr int kWarps = D / 2 / 32;
    if constexpr (kWarps > 1) {
      __shared__ float wmax[8];
      const int w = threadIdx.x >> 5;
      if ((threadIdx.x & 31) == 0) wmax[w] = amax;
      __syncthreads();
      const float* q = wmax + (w / kWarps) * kWarps;
#pragma unroll
      for (int u = 0; u < kWarps; ++u) amax = fmaxf(amax, q[u]);
      __syncthreads();
    }
    const int e = e8m0_exponent(amax);
    const float inv = exp2i(-e);
    const uint32_t codes = e4m3x2(__fmul_rn(y0, inv), __fmul_rn(y1, inv));
    if (valid) {
      *reinterpret_cast<uint16_t*>(dst.data + 2 * lt) = static_cast<uint16_t>(codes);
      if (lt == 0) *reinterpret_cast<float*>(dst.scale) = exp2i(e);
    }
    return;
  }
  // FP8 inline rows: blocks of 32 channels = 16 threads
  amax = fmaxf(amax, __shfl_xor_sync(full, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(full, amax, 2));
  amax = fmaxf(amax, __shfl_xor_sync(full, amax, 4));
  amax = fmaxf(amax, __shfl_xor_sync(full, amax, 8));
  const int e = e8m0_exponent(amax);
  const float inv = exp2i(-e);
  const uint32_t codes = e4m3x2(__fmul_rn(y0, inv), __fmul_rn(y1, inv));
  if (valid) {
    *reinterpret_cast<uint16_t*>(dst.data + 2 * lt) = static_cast<uint16_t>(codes);
    if ((lt & 15) == 0) dst.scale[lt >> 4] = static_cast<uint8_t>(e + 127);
  }
}

}  // namespace cskv
