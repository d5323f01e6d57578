// Decode path of the fused MoE layer: weight-streaming expert GEMV/skinny GEMMs.
//
// At decode batch sizes each active expert sees only a few tokens, so the
// layer is bound by reading the activated experts' weights from HBM once
// (the FP8 MoE decode of the OSDI'26 local-MoE paper summary, section "CPU
// decode backend", and the bandwidth argument of the SGLang CPU backend
// write-up, section "(3) FusedMoE").  The math follows the pages:
//
//  * GEMM1 uses the A x [B1, B2] = [C1, C2] form: one work item owns 16 gate
//    rows AND the matching 16 up rows of one expert, so h = SiLU(C1) * C2 is
//    finished inside the CTA and up_proj is never stored (Xeon 6 / SGLang blog,
//    section "MoE", SiLU-fusion bullet).
//  * FP8 weights are expanded to fp16 in registers and never stored wider; the
//    128x128 block scale multiplies each 128-deep partial sum once
//    (post-scaling, OSDI'26 summary, section "CPU decode backend").
//  * INT8 weights (DA8W8) multiply per-row-quantised activations; the integer
//    products are exact in fp32 and the per-row x per-channel scales are
//    applied once at the end.
//  * GEMM2 owns a slice of 16 output channels for ALL tokens and walks every
//    active expert, so the weighted top-k combine happens in shared memory in a
//    fixed order: no atomics, no y buffer, deterministic.
//
// GB300 mapping: 128-bit streaming loads (L1 no-allocate) of weight rows; the
// products run on warp-level tensor-core MMA (m16n8k16, weights as the 16-row
// A operand, up to 8 tokens as the N operand -- a swap-AB skinny GEMM).  The
// K order inside each 128-wide block is permuted identically for both
// operands so that every lane's 32 consecutive weight bytes feed its MMA
// fragments directly, with no shared-memory staging.
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace gbmoe {

constexpr int kDecWarps = 8;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kRows = 16;  // rows of W per MMA tile

__device__ __forceinline__ uint32_t word8(const uint4& a, const uint4& b, int s) {
  switch (s) {
    case 0: return a.x; case 1: return a.y; case 2: return a.z; case 3: return a.w;
    case 4: return b.x; case 5: return b.y; case 6: return b.z; default: return b.w;
  }
}

__device__ __forceinline__ uint32_t word16(const uint4 (&x)[4], int i) {
  const uint4& v = x[i >> 2];
  switch (i & 3) {
    case 0: return v.x; case 1: return v.y; case 2: return v.z; default: return v.w;
  }
}

// 16 rows x 128 K of weights against up to 8 token columns.
// Lane (g, t) holds 32 consecutive bytes of rows g and g+8 starting at column
// t*32 (ra0/ra1, rb0/rb1) and the 32 matching activations of token column g
// (xb, fp16).  MMA step s uses bytes [4s, 4s+4) of each chunk: the pairs
// (4s, 4s+1) stand at logical k = 2t, 2t+1 and (4s+2, 4s+3) at 2t+8, 2t+9,
// and the activations follow the same map, so the sum over K is unchanged.
template <int WK>
__device__ __forceinline__ void tile_mma_128(float acc[4], const uint4& ra0, const uint4& ra1,
                                             const uint4& rb0, const uint4& rb1, const uint4 (&xb)[4]) {
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    uint32_t a[4];
    w8x4_to_f16x4<WK>(word8(ra0, ra1, s), a[0], a[2]);
    w8x4_to_f16x4<WK>(word8(rb0, rb1, s), a[1], a[3]);
    mma_f16_16816(acc, a, word16(xb, 2 * s), word16(xb, 2 * s + 1));
  }
}

__device__ __forceinline__ void load_x32(uint4 (&xb)[4], const __half* row, size_t kofs, bool valid) {
  if (valid) {
    const __half* p = row + kofs;
#pragma unroll
    for (int i = 0; i < 4; ++i) xb[i] = ld_v4(p + 8 * i);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) xb[i] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// ------------------------------------------------------------------ GEMM1: gate/up + SiLU * mul
template <int WK>
__global__ void __launch_bounds__(kDecThreads) decode_gemm1_kernel(DecodeArgs d) {
  __shared__ float red[kDecWarps][2][4][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int tiles = d.I / kRows;
  const int KB = d.H / kQBlock;
  const int n_items = *d.num_active * tiles;
  const int sblk_cols = d.H / kQBlock;

  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int j = item / tiles;
    const int r0 = (item - j * tiles) * kRows;
    const int e = d.active[j];
    const int off = d.offsets[e], cnt = d.counts[e];
    const uint8_t* wg = d.w13 + (static_cast<size_t>(e) * 2 * d.I + r0) * d.H;
    const uint8_t* wu = wg + static_cast<size_t>(d.I) * d.H;
    const uint8_t* wg_g = wg + static_cast<size_t>(g) * d.H;
    const uint8_t* wg_g8 = wg + static_cast<size_t>(g + 8) * d.H;
    const uint8_t* wu_g = wu + static_cast<size_t>(g) * d.H;
    const uint8_t* wu_g8 = wu + static_cast<size_t>(g + 8) * d.H;
    // FP8 block-scale rows of this tile (16 | 128, so one scale row per tile)
    const float* sg = d.s13 + (static_cast<size_t>(e) * (2 * d.I / kQBlock) + r0 / kQBlock) * sblk_cols;
    const float* su = d.s13 + (static_cast<size_t>(e) * (2 * d.I / kQBlock) + (d.I + r0) / kQBlock) * sblk_cols;

    for (int g0 = 0; g0 < cnt; g0 += 8) {
      const int colg = g0 + g;
      const int tokg = colg < cnt ? d.sorted_ids[off + colg] / d.topk : -1;
      const __half* xrow = d.xq + static_cast<size_t>(tokg < 0 ? 0 : tokg) * d.H;
      float tg[4] = {0.f, 0.f, 0.f, 0.f}, tu[4] = {0.f, 0.f, 0.f, 0.f};
      for (int kb = warp; kb < KB; kb += kDecWarps) {
        const size_t kofs = static_cast<size_t>(kb) * kQBlock + t * 32;
        const uint4 g0a = ld_stream_v4(wg_g + kofs), g0b = ld_stream_v4(wg_g + kofs + 16);
        const uint4 g8a = ld_stream_v4(wg_g8 + kofs), g8b = ld_stream_v4(wg_g8 + kofs + 16);
        const uint4 u0a = ld_stream_v4(wu_g + kofs), u0b = ld_stream_v4(wu_g + kofs + 16);
        const uint4 u8a = ld_stream_v4(wu_g8 + kofs), u8b = ld_stream_v4(wu_g8 + kofs + 16);
        uint4 xb[4];
        load_x32(xb, xrow, kofs, tokg >= 0);
        if constexpr (WK == MOE_WEIGHT_FP8) {
          float ag[4] = {0.f, 0.f, 0.f, 0.f}, au[4] = {0.f, 0.f, 0.f, 0.f};
          tile_mma_128<WK>(ag, g0a, g0b, g8a, g8b, xb);
          tile_mma_128<WK>(au, u0a, u0b, u8a, u8b, xb);
          const float scg = __ldg(sg + kb), scu = __ldg(su + kb);
#pragma unroll
          for (int i = 0; i < 4; ++i) { tg[i] = fmaf(scg, ag[i], tg[i]); tu[i] = fmaf(scu, au[i], tu[i]); }
        } else {
          tile_mma_128<WK>(tg, g0a, g0b, g8a, g8b, xb);
          tile_mma_128<WK>(tu, u0a, u0b, u8a, u8b, xb);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) { red[warp][0][i][lane] = tg[i]; red[warp][1][i][lane] = tu[i]; }
      __syncthreads();
      if (warp == 0) {
        float G[4], U[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float a = 0.f, b = 0.f;
#pragma unroll
          for (int w = 0; w < kDecWarps; ++w) { a += red[w][0][i][lane]; b += red[w][1][i][lane]; }
          G[i] = a; U[i] = b;
        }
        float cmax[2] = {0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = g + ((i & 2) ? 8 : 0);
          const int col = g0 + 2 * t + (i & 1);
          const bool valid = col < cnt;
          const size_t hidx = static_cast<size_t>(off + col) * d.I + r0 + row;
          if constexpr (WK == MOE_WEIGHT_FP8) {
            const float h = valid ? silu_f32(G[i]) * U[i] : 0.f;
            reinterpret_cast<__half*>(d.h)[hidx] = __float2half_rn(h);
          } else {
            float h = 0.f;
            if (valid) {
              const int tok = d.sorted_ids[off + col] / d.topk;
              const float sx = d.sx[tok];
              const float gv = G[i] * sx * __ldg(d.s13 + static_cast<size_t>(e) * 2 * d.I + r0 + row);
              const float uv = U[i] * sx * __ldg(d.s13 + static_cast<size_t>(e) * 2 * d.I + d.I + r0 + row);
              h = silu_f32(gv) * uv;
            }
            reinterpret_cast<float*>(d.h)[hidx] = h;
            cmax[i & 1] = fmaxf(cmax[i & 1], fabsf(h));
          }
        }
        if constexpr (WK == MOE_WEIGHT_INT8) {
          // max over the 16 rows of each column: reduce across g (lane bits 2..4)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            float v = cmax[c];
            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
            const int col = g0 + 2 * t + c;
            if (g == 0 && col < cnt) atomicMax(d.hmax + off + col, __float_as_uint(v));
          }
        }
      }
      __syncthreads();
    }
  }
}

// ------------------------------------------------------------------ INT8: requantise h per row
// One warp per row: s = max|h| / 127, codes = RNE(h / s) clamped to +-127, stored as fp16.
__global__ void __launch_bounds__(256) requant_h_kernel(const float* __restrict__ h, const uint32_t* __restrict__ hmax,
                                                        const int32_t* __restrict__ num_post, int I,
                                                        __half* __restrict__ hq, float* __restrict__ sh) {
  const int lane = threadIdx.x & 31;
  const int rows = *num_post;
  const int warps_total = gridDim.x * (blockDim.x >> 5);
  for (int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps_total) {
    const float amax = __uint_as_float(hmax[r]);
    const float s = amax > 0.f ? __fdiv_rn(amax, 127.0f) : 1.0f;
    const float* hr = h + static_cast<size_t>(r) * I;
    __half* qr = hq + static_cast<size_t>(r) * I;
    for (int c = lane; c < I; c += 32) qr[c] = __float2half_rn(quant_s8_rne(hr[c], s));
    if (lane == 0) sh[r] = s;
  }
}

cudaError_t launch_requant_rows(const void* h, const uint32_t* hmax, const int32_t* num_post, int cap, int I,
                                __half* hq, float* sh, int num_sms, cudaStream_t s) {
  int grid = (cap + 7) / 8;
  if (grid > num_sms * 8) grid = num_sms * 8;
  if (grid < 1) grid = 1;
  requant_h_kernel<<<grid, 256, 0, s>>>(static_cast<const float*>(h), hmax, num_post, I, hq, sh);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ GEMM2: down proj + weighted combine
template <int WK>
__global__ void __launch_bounds__(kDecThreads) decode_gemm2_kernel(DecodeArgs d) {
  extern __shared__ float acc_s[];  // [kDecWarps][M][16]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int KB2 = d.I / kQBlock;
  const int n_items = *d.num_active * KB2;
  const int M = d.M;
  const __half* hsrc = (WK == MOE_WEIGHT_FP8) ? reinterpret_cast<const __half*>(d.h) : d.hq;

  for (int tile = blockIdx.x; tile < d.H / kRows; tile += gridDim.x) {
    const int n0 = tile * kRows;
    for (int i = threadIdx.x; i < kDecWarps * M * kRows; i += kDecThreads) acc_s[i] = 0.f;
    __syncthreads();
    float* my = acc_s + warp * M * kRows;
    for (int it = warp; it < n_items; it += kDecWarps) {
      const int j = it / KB2, kb = it - j * KB2;
      const int e = d.active[j];
      const int off = d.offsets[e], cnt = d.counts[e];
      const uint8_t* w = d.w2 + (static_cast<size_t>(e) * d.H + n0) * d.I;
      const size_t kofs = static_cast<size_t>(kb) * kQBlock + t * 32;
      const uint4 a0 = ld_stream_v4(w + static_cast<size_t>(g) * d.I + kofs);
      const uint4 a1 = ld_stream_v4(w + static_cast<size_t>(g) * d.I + kofs + 16);
      const uint4 b0 = ld_stream_v4(w + static_cast<size_t>(g + 8) * d.I + kofs);
      const uint4 b1 = ld_stream_v4(w + static_cast<size_t>(g + 8) * d.I + kofs + 16);
      float sc = 1.f;
      if constexpr (WK == MOE_WEIGHT_FP8)
        sc = __ldg(d.s2 + (static_cast<size_t>(e) * (d.H / kQBlock) + n0 / kQBlock) * KB2 + kb);
      for (int g0 = 0; g0 < cnt; g0 += 8) {
        uint4 xb[4];
        // h rows of padded slots are zero, so every row in [off, off + padded) is readable
        load_x32(xb, hsrc + static_cast<size_t>(off + g0 + g) * d.I, kofs, true);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        tile_mma_128<WK>(acc, a0, a1, b0, b1, xb);
        float v[4];
        int tok[2];
        bool ok[2];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int col = g0 + 2 * t + c;
          ok[c] = col < cnt;
          tok[c] = 0;
          float wgt = 0.f, srow = 1.f;
          if (ok[c]) {
            const int slot = d.sorted_ids[off + col];
            tok[c] = slot / d.topk;
            wgt = d.topk_w[slot];
            if constexpr (WK == MOE_WEIGHT_INT8) srow = d.sh[off + col];
          }
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int i = hh * 2 + c;
            float s = sc * srow * wgt;
            if constexpr (WK == MOE_WEIGHT_INT8)
              s *= __ldg(d.s2 + static_cast<size_t>(e) * d.H + n0 + g + 8 * hh);
            v[i] = acc[i] * s;
          }
        }
        // fixed-order accumulation: lanes with equal t touch distinct rows
#pragma unroll
        for (int tt = 0; tt < 4; ++tt) {
          if (t == tt) {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              if (ok[c]) {
                my[tok[c] * kRows + g] += v[c];
                my[tok[c] * kRows + g + 8] += v[2 + c];
              }
            }
          }
          __syncwarp();
        }
      }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < M * kRows; i += kDecThreads) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) s += acc_s[w * M * kRows + i];
      const int tok = i / kRows, row = i - tok * kRows;
      d.out[static_cast<size_t>(tok) * d.H + n0 + row] = __float2bfloat16_rn(s);
    }
    __syncthreads();
  }
}

size_t decode_gemm2_smem_bytes(int M) { return static_cast<size_t>(kDecWarps) * M * kRows * sizeof(float); }

template <int WK>
static cudaError_t launch_decode_t(const DecodeArgs& d, int num_sms, cudaStream_t s, const StageHook& hook) {
  const int max_active = d.E < d.M * d.topk ? d.E : d.M * d.topk;
  const int items1 = max_active * (d.I / kRows);
  int grid1 = num_sms * 4;
  if (items1 < grid1) grid1 = items1;
  if (grid1 <= 0) return cudaSuccess;
  decode_gemm1_kernel<WK><<<grid1, kDecThreads, 0, s>>>(d);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  hook("decode_gemm1", s);
  if constexpr (WK == MOE_WEIGHT_INT8) {
    err = launch_requant_rows(d.h, d.hmax, d.num_post, d.cap, d.I, d.hq, d.sh, num_sms, s);
    if (err != cudaSuccess) return err;
    hook("requant_h", s);
  }
  const size_t smem2 = decode_gemm2_smem_bytes(d.M);
  err = set_smem_limit_once(reinterpret_cast<const void*>(decode_gemm2_kernel<WK>),
                            static_cast<int>(decode_gemm2_smem_bytes(MOE_MAX_DECODE_TOKENS)), 1 + WK);
  if (err != cudaSuccess) return err;
  decode_gemm2_kernel<WK><<<d.H / kRows, kDecThreads, smem2, s>>>(d);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  hook("decode_gemm2_combine", s);
  return cudaSuccess;
}

cudaError_t launch_decode(const DecodeArgs& d, int weight_kind, int num_sms, cudaStream_t s,
                          const StageHook& hook) {
  return weight_kind == MOE_WEIGHT_FP8 ? launch_decode_t<MOE_WEIGHT_FP8>(d, num_sms, s, hook)
                                       : launch_decode_t<MOE_WEIGHT_INT8>(d, num_sms, s, hook);
}

}  // namespace gbmoe
