// Masked (fixed-capacity) layout: the first kernel of fused_moe_masked.
//
// Expert-parallel low-latency dispatch hands the MoE layer its tokens already
// grouped by expert, E blocks of `cap` rows, with a device-side count of the
// real rows per expert (the masked grouped GEMM of the DeepGEMM integration in
// the news rewrite of the LMSYS large-scale-EP blog, section "DeepGEMM集成").
// Nothing needs sorting: this kernel turns the counts into the GEMMs' work
// description and prepares the activation rows.
//
// Positions: expert e's real rows take positions off[e] .. off[e] + m_e - 1,
// with off[] the exclusive prefix sum of the counts rounded up to the block (8
// for the decode kernels, 16 for the tcgen05 ones), so a token tile never reads
// past the buffers and starts where the tcgen05 path's 16-row loads need it.
// Every CTA computes the prefix sum itself (E <= 1024 counts, one scan); CTA 0
// writes the tile list and sorted_ids[pos] = e * cap + i (the output row), the others clear
// the intermediate's frame words and copy the real rows of x into position order, converted
// to fp16 in a power-of-two frame per row -- or, for FP8 weights on the tcgen05 path (kind 5),
// to the two-term E4M3 form that the FP8-operand kernels read.
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace gbmoe {

constexpr int kMaskedThreads = 1024;

__global__ void __launch_bounds__(kMaskedThreads) masked_prologue_kernel(MaskedArgs m) {
  __shared__ int off[MOE_MAX_EXPERTS + 1];
  __shared__ int cnt[MOE_MAX_EXPERTS];
  __shared__ int scan_tmp[33];
  pdl_trigger();  // the next kernel may set itself up; it waits for this grid before reading
  pdl_wait();     // the counts and x may come from the previous kernel (the dispatch)
  const int tid = threadIdx.x;
  int c = 0;
  if (tid < m.E) {
    c = __ldg(m.masked_m + tid);
    c = c < 0 ? 0 : (c > m.cap ? m.cap : c);
    cnt[tid] = c;
  }
  int total;
  const int o = block_exclusive_scan((c + m.block - 1) / m.block * m.block, scan_tmp, total);
  if (tid < m.E) off[tid] = o;
  if (tid == 0) off[m.E] = total;
  if (blockIdx.x == 0) {
    int ntiles;
    const int t0 = block_exclusive_scan((c + m.tile - 1) / m.tile, scan_tmp, ntiles);
    if (tid < m.E) {
      for (int j = 0; j * m.tile < c; ++j)
        m.ttiles[t0 + j] = make_int4(tid, o + m.tile * j, min(m.tile, c - m.tile * j), 0);
    }
    if (tid == 0) {
      *m.num_ttiles = ntiles;
      *m.num_post = total;
      if (m.status) { m.status->bad_ids = 0; m.status->flags = 0; }
    }
    __syncthreads();
    // sorted_ids: one warp per expert
    for (int e = tid >> 5; e < m.E; e += kMaskedThreads / 32)
      for (int i = tid & 31; i < cnt[e]; i += 32) m.sorted_ids[off[e] + i] = e * m.cap + i;
    return;
  }
  __syncthreads();
  // the intermediate's frame words of every position start at zero
  for (int i = (blockIdx.x - 1) * kMaskedThreads + tid; i < m.n_zero; i += (gridDim.x - 1) * kMaskedThreads)
    m.zero_words[i] = 0u;
  // activation rows, one warp per row; H is a multiple of 128, so a lane moves whole 8-column groups.
  // Each row is stored as fp16 x * 2^-e with its max |x| * 2^-e in [2^14, 2^15); xs[pos] = 2^e.
  const int warp = tid >> 5, lane = tid & 31;
  const int nw = kMaskedThreads / 32;
  const long long rows = static_cast<long long>(m.E) * m.cap;
  for (long long r = (blockIdx.x - 1) * static_cast<long long>(nw) + warp; r < rows;
       r += static_cast<long long>(gridDim.x - 1) * nw) {
    const int e = static_cast<int>(r / m.cap), i = static_cast<int>(r - static_cast<long long>(e) * m.cap);
    if (i >= cnt[e]) continue;
    const int pos = off[e] + i;
    if (m.kind == 5) {
      // the two-term E4M3 form, a frame 2^e per 128 columns (group max |x| * 2^-e in [2^7, 2^8)):
      // hi codes in row pos of act8, lo codes in row pcap + pos, sa8[group * pcap + pos] = 2^e
      const uint2* src2 = reinterpret_cast<const uint2*>(m.x + r * m.H);
      constexpr int kBatch = 8;  // groups whose loads are in flight together (the byte stores could alias them)
      const int G = m.H / kQBlock;
      for (int g0 = 0; g0 < G; g0 += kBatch) {
        uint2 raw[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
          raw[u] = g0 + u < G ? __ldg(src2 + (g0 + u) * 32 + lane) : make_uint2(0u, 0u);  // columns 128 gi + 4 lane..
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int gi = g0 + u;
          if (gi >= G) break;
          const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw[u].x));
          const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw[u].y));
          const float mx = warp_max(fmaxf(fmaxf(fabsf(f0.x), fabsf(f0.y)), fmaxf(fabsf(f1.x), fabsf(f1.y))));
          const int ex = mx > 0.f ? e4m3_split_exp(mx) : 0;
          uint32_t hi, lo;
          e4m3_split4(make_float4(f0.x, f0.y, f1.x, f1.y), exp2i(-ex), hi, lo);
          const size_t col = static_cast<size_t>(gi) * kQBlock + lane * 4;
          *reinterpret_cast<uint32_t*>(m.act8 + static_cast<size_t>(pos) * m.H + col) = hi;
          *reinterpret_cast<uint32_t*>(m.act8 + (static_cast<size_t>(m.pcap) + pos) * m.H + col) = lo;
          if (lane == 0) m.sa8[static_cast<size_t>(gi) * m.pcap + pos] = exp2i(ex);
        }
      }
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(m.x + r * m.H);
    uint4* dst = reinterpret_cast<uint4*>(m.xq + static_cast<size_t>(pos) * m.H);
    float amax = 0.f;
    for (int g = lane; g < m.H / 8; g += 32) {
      const uint4 raw = __ldg(src + g);
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[j]));
        amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
      }
    }
    const int ex = x_frame_exp(warp_max(amax));
    const float mul = exp2i(-ex);
    if (lane == 0) m.xs[pos] = exp2i(ex);
    for (int g = lane; g < m.H / 8; g += 32) {
      const uint4 raw = __ldg(src + g);
      const float2 f01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
      const float2 f23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
      const float2 f45 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.z));
      const float2 f67 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.w));
      dst[g] = m.kind == 4 ? make_uint4(pack_half2(f01.x * mul, f45.x * mul), pack_half2(f01.y * mul, f45.y * mul),
                                        pack_half2(f23.x * mul, f67.x * mul), pack_half2(f23.y * mul, f67.y * mul))
                           : make_uint4(pack_half2(f01.x * mul, f01.y * mul), pack_half2(f23.x * mul, f23.y * mul),
                                        pack_half2(f45.x * mul, f45.y * mul), pack_half2(f67.x * mul, f67.y * mul));
    }
  }
}

cudaError_t launch_masked_prologue(const MaskedArgs& m, int num_sms, cudaStream_t s) {
  const long long rows = static_cast<long long>(m.E) * m.cap;
  const long long per_cta = kMaskedThreads / 32;
  long long prep = (rows + per_cta - 1) / per_cta;
  if (prep > 2LL * num_sms) prep = 2LL * num_sms;
  if (prep < 1) prep = 1;
  return launch_kernel(masked_prologue_kernel, dim3(static_cast<unsigned>(1 + prep)), dim3(kMaskedThreads), 0, s,
                       true, m);
}

}  // namespace gbmoe
