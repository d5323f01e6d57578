// Shared device helpers of the fused MoE library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gbmoe.h"

namespace gbmoe {

constexpr int kQBlock = 128;       // FP8 block-scale granularity (both dims)
constexpr int kDecodeBlock = 8;    // align block size of the decode path (= MMA N)
constexpr int kPrefillBlock = 16;  // align block size of the prefill path (MMA N granularity)
constexpr int kPrefillTileTokens = 128;  // sorted slots per prefill token tile (max MMA N)
constexpr int kStatusBytes = 256;  // head of every workspace: device status words

// Device status words at the start of a workspace.
struct DeviceStatus {
  int32_t bad_ids;  // topk_ids entries outside [0, E)
  int32_t flags;    // bit 0: a bounded wait gave up
};

// ---------------------------------------------------------------- conversions

// Four E4M3 codes (one 32-bit word, byte 0 first) -> two fp16 pairs; exact.
// One hardware conversion per 16-bit half (bytes 0,1 -> lo; bytes 2,3 -> hi).
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\t"
      "mov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// Four int8 values (one word, byte 0 first) -> two fp16 pairs; exact.
// Each byte b is biased to b+128 in [0, 255], placed as the low mantissa bits
// of the fp16 number 1024 (0x6400), so the lane reads 1152 + b; subtracting
// 1152 leaves b exactly (fp16 spacing is 1 on [1024, 2048)).
__device__ __forceinline__ void s8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  uint32_t l, h;
  asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(l) : "r"(u), "r"(0x64646464u));
  asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(h) : "r"(u), "r"(0x64646464u));
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
  __half2 lh = __hsub2(*reinterpret_cast<__half2*>(&l), bias);
  __half2 hh = __hsub2(*reinterpret_cast<__half2*>(&h), bias);
  lo = *reinterpret_cast<uint32_t*>(&lh);
  hi = *reinterpret_cast<uint32_t*>(&hh);
}

// f(w, a, b) = a ? (w ^ b) : b, bit by bit (one LOP3): where a is set the bit of
// w passes, inverted where b is set; elsewhere the bit of b is the result.
__device__ __forceinline__ uint32_t lop3_sel_xor(uint32_t w, uint32_t a, uint32_t b) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(r) : "r"(w), "r"(a), "r"(b));
  return r;
}

// Eight two's-complement int4 values (one word, nibble i = value k_i) -> four
// fp16 pairs, exact: r[0] = (k0, k4), r[1] = (k1, k5), r[2] = (k2, k6),
// r[3] = (k3, k7).  Each nibble is biased to k+8 in [0, 15] (its top bit
// inverted) and becomes mantissa bits of the fp16 number 1024 (0x6400): at bit
// 0 the half reads 1024 + (k+8), at bit 4 it reads 1024 + 16 (k+8).  One LOP3
// per pair selects the nibbles, inverts their top bit and sets the exponent; one
// subtraction of 1032, or one fused multiply-add by 1/16 and -72, leaves k exactly.
__device__ __forceinline__ void s4x8_to_f16x8(uint32_t w, uint32_t r[4]) {
  const uint32_t v = w >> 8;
  const uint32_t l0 = lop3_sel_xor(w, 0x000f000fu, 0x64086408u), h0 = lop3_sel_xor(w, 0x00f000f0u, 0x64806480u);
  const uint32_t l1 = lop3_sel_xor(v, 0x000f000fu, 0x64086408u), h1 = lop3_sel_xor(v, 0x00f000f0u, 0x64806480u);
  const __half2 bias = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));   // 1032
  const __half2 sixteenth = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));  // 1/16
  const __half2 m72 = __halves2half2(__ushort_as_half(0xD480), __ushort_as_half(0xD480));    // -72
  __half2 q0 = __hsub2(*reinterpret_cast<const __half2*>(&l0), bias);
  __half2 q1 = __hfma2(*reinterpret_cast<const __half2*>(&h0), sixteenth, m72);
  __half2 q2 = __hsub2(*reinterpret_cast<const __half2*>(&l1), bias);
  __half2 q3 = __hfma2(*reinterpret_cast<const __half2*>(&h1), sixteenth, m72);
  r[0] = *reinterpret_cast<uint32_t*>(&q0);
  r[1] = *reinterpret_cast<uint32_t*>(&q1);
  r[2] = *reinterpret_cast<uint32_t*>(&q2);
  r[3] = *reinterpret_cast<uint32_t*>(&q3);
}

// INT4 layer: activations (x, and h between the GEMMs) are stored as fp16 with
// every group of 8 consecutive K values in the order k0 k4 k1 k5 k2 k6 k3 k7, the
// order in which s4x8_to_f16x8 yields the weights.  Stored position of K index n:
__device__ __forceinline__ int int4_kperm(int n) {
  const int i = n & 7;
  return (n & ~7) | (i < 4 ? 2 * i : 2 * (i - 4) + 1);
}

template <int WK>
__device__ __forceinline__ void w8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  if constexpr (WK == MOE_WEIGHT_FP8) e4m3x4_to_f16x4(w, lo, hi);
  else s8x4_to_f16x4(w, lo, hi);
}

// Block-wide exclusive scan of one int per thread (blockDim == 1024).
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_tot[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    warp_tot[lane] = wi - w;  // exclusive prefix of warp totals
    if (lane == 31) warp_tot[32] = wi;
  }
  __syncthreads();
  const int res = warp_tot[warp] + incl - v;
  total = warp_tot[32];
  __syncthreads();
  return res;
}

// fp32 -> E4M3 code: round to nearest, ties to even, saturating to +-448.
__device__ __forceinline__ uint32_t e4m3_code(float v) {
  return static_cast<uint32_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ---------------------------------------------------------------- power-of-two frames of fp16 operands
// The weight-only paths multiply fp16 operands on the tensor cores, while x arrives as bf16 (the range of
// fp32) and the intermediate h is an fp32 result.  Both are therefore stored as fp16 values v * 2^-e in a
// frame 2^e chosen from their magnitude; the fp32 accumulators take the factor 2^e back.  Scaling by a power
// of two is exact, so a value keeps the full fp16 precision whenever it lies within 2^-14 of the frame's
// top binade, and the sums are the same as with unscaled operands wherever those were in range.
//
// x: one frame per row, with the row's max |x| in [2^14, 2^15).
// h: one frame per (row, 32 columns) block, with the block's max |h| in [2^7, 2^15) and the exponent a
// multiple of 8, so the blocks of a row mostly share one frame.  The row frame is the largest block
// exponent; blocks stored lower are scaled down to it before they enter the down projection.
// Exponents are kept biased by kExpBias (1..255); 0 marks an all-zero block.
constexpr int kExpBias = 128;
constexpr int kHBlock = 32;  // columns of h per frame block

// floor(log2(a)) for finite a > 0, with fp32 subnormals counted as 2^-127.
__device__ __forceinline__ int ilog2f(float a) { return ((__float_as_int(a) >> 23) & 0xff) - 127; }

// Frame exponent of an x row with max |x| = amax: amax * 2^-e in [2^14, 2^15); 0 for a zero row.
__device__ __forceinline__ int x_frame_exp(float amax) {
  if (!(amax > 0.f)) return 0;
  const int e = ilog2f(amax) - 14;
  return e < -126 ? -126 : e;
}

// Biased frame exponent of an h block with max |h| = amax (0 for a zero block): the smallest multiple
// of 8 with amax * 2^-e < 2^15, so amax * 2^-e lies in [2^7, 2^15).  (A coarser grid would let more
// blocks share a frame but would also let the row frame -- the largest block exponent -- sit higher above
// the row's values: with multiples of 8 every element within 2^-21 of its row's largest stays a normal
// fp16 number.)
__device__ __forceinline__ int h_frame_exp_biased(float amax) {
  if (!(amax > 0.f)) return 0;
  int e = ilog2f(amax) - 14;
  e = e < -120 ? -120 : (e > 120 ? 120 : e);
  e = (e + 127) / 8 * 8 - 120;  // round up to a multiple of 8 (e + 127 >= 7 keeps the division exact)
  return e + kExpBias;
}

// 2^e as fp32 for -126 <= e <= 127 (0 below).
__device__ __forceinline__ float exp2i(int e) { return e < -126 ? 0.f : __int_as_float((e + 127) << 23); }

// fp16 pair (2^d, 2^d) for d <= 0; zero below 2^-24 (fp16 subnormals cover 2^-24 .. 2^-15).
__device__ __forceinline__ __half2 exp2i_h2(int d) {
  const uint16_t b = d >= -14 ? static_cast<uint16_t>((d + 15) << 10)
                              : (d >= -24 ? static_cast<uint16_t>(1u << (d + 24)) : static_cast<uint16_t>(0));
  const __half h = __ushort_as_half(b);
  return __halves2half2(h, h);
}

// Two-term E4M3 form of values carried on the FP8 tensor cores in place of bf16 or fp32 operands: in a
// power-of-two frame 2^e per group of 128 with the group's max |v| * 2^-e in [2^7, 2^8), a value is
// hi + lo with hi = E4M3(v * 2^-e) and lo = E4M3(v * 2^-e - hi) (round to nearest even; |v| * 2^-e < 256,
// so nothing saturates).  A bf16 value is exact in this form when v * 2^-e >= 2^-2 (its 8 significant bits
// split into two 4-bit halves that are both E4M3 normals or exact subnormals); smaller values keep an
// absolute error below 2^-10 in the frame, i.e. below 2^-17 of the group's max.
__device__ __forceinline__ int e4m3_split_exp(float amax) {
  const int e = ilog2f(amax) - 7;
  return e < -126 ? -126 : (e > 120 ? 120 : e);
}

// E4M3 code pair (the low two bytes of w16) -> float2, exact.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t w16) {
  uint32_t h;
  asm("{\n\t.reg .b16 l;\n\tcvt.u16.u32 l, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, l;\n\t}" : "=r"(h) : "r"(w16));
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// The two-term form of four values, mul = 2^-e: hi and lo codes, byte i from value i.
__device__ __forceinline__ void e4m3_split4(float4 v, float mul, uint32_t& hi, uint32_t& lo) {
  const float a0 = v.x * mul, a1 = v.y * mul, a2 = v.z * mul, a3 = v.w * mul;
  const uint32_t h01 = __nv_cvt_float2_to_fp8x2(make_float2(a0, a1), __NV_SATFINITE, __NV_E4M3);
  const uint32_t h23 = __nv_cvt_float2_to_fp8x2(make_float2(a2, a3), __NV_SATFINITE, __NV_E4M3);
  const float2 b01 = e4m3x2_to_float2(h01), b23 = e4m3x2_to_float2(h23);
  const uint32_t l01 = __nv_cvt_float2_to_fp8x2(make_float2(a0 - b01.x, a1 - b01.y), __NV_SATFINITE, __NV_E4M3);
  const uint32_t l23 = __nv_cvt_float2_to_fp8x2(make_float2(a2 - b23.x, a3 - b23.y), __NV_SATFINITE, __NV_E4M3);
  hi = (h01 & 0xffffu) | (h23 << 16);
  lo = (l01 & 0xffffu) | (l23 << 16);
}

// Multiplies the 8 fp16 values of v by the power of two f (exact unless they become subnormal).
__device__ __forceinline__ void scale_h8(uint4& v, __half2 f) {
  uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&w[i]), f);
    w[i] = *reinterpret_cast<const uint32_t*>(&r);
  }
}

// ---------------------------------------------------------------- memory

// Streaming 16-byte load that does not allocate in L1 (weights are read once).
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint4 ld_v4(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// ---------------------------------------------------------------- tensor core (warp MMA)

// D[16x8] += A[16x16] * B[16x8], fp16 operands, fp32 accumulate.
// Fragment ownership (lane = 4*g + t):
//   a[0]: A[g][2t..2t+1]   a[1]: A[g+8][2t..2t+1]
//   a[2]: A[g][2t+8..+9]   a[3]: A[g+8][2t+8..+9]
//   b[0]: B[2t..2t+1][g]   b[1]: B[2t+8..+9][g]
//   d[0..1]: D[g][2t..2t+1]  d[2..3]: D[g+8][2t..2t+1]
__device__ __forceinline__ void mma_f16_16816(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// SiLU with the fast exponential and division (a few ulp; the result is rounded to fp16 or
// quantised right after).  __fdividef returns 0 once 1 + exp(-g) exceeds 2^126, i.e. for
// g < -87, where SiLU(g) is below 1e-36 anyway.
__device__ __forceinline__ float silu_f32(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// ---------------------------------------------------------------- programmatic dependent launch
// A kernel launched with programmatic stream serialization may start while its
// predecessor in the stream is still running: everything it reads from the
// predecessor must come after pdl_wait() (which returns once the predecessor has
// completed and its writes are visible).  pdl_trigger() lets the successor start
// launching.  The first kernel of a call (routing prologue, router gating) triggers
// at once, and every kernel that follows it waits before it reads anything.  Every
// other kernel triggers only after its own pdl_wait(), so a kernel placed behind
// one of those may read data written two kernels back without waiting.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Round-half-even of x / s in fp32 (IEEE division), clamped to +-127.
__device__ __forceinline__ float quant_s8_rne(float x, float s) {
  float q = rintf(__fdiv_rn(x, s));
  return fminf(fmaxf(q, -127.0f), 127.0f);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace gbmoe
