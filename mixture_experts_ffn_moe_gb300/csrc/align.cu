// Routing alignment and activation preparation (the first launch of a layer call).
//
// Routing alignment restates the moe_align_index step of the SGLang CPU
// backend write-up (section "(3) FusedMoE"; Xeon 6 / SGLang DeepSeek-R1 blog,
// section "MoE"): an argsort of the flat topk_ids by expert, each expert's
// group padded to a multiple of the block size, with the expert of every
// block recorded.  Only group membership matters to the GEMMs, but the order
// inside a group is fixed here (ascending slot index) so the result equals a
// stable argsort and is deterministic.
//
// GB300 design: one CTA of 1024 threads does the whole alignment in three
// passes over shared memory -- per-warp expert histograms, one block-wide
// scan that turns them into write cursors, and a warp-ordered scatter in which
// __match_any_sync ranks equal ids inside each 32-slot step.  The other CTAs of
// the same launch prepare the activation rows for the expert GEMMs.
#include <cuda_runtime.h>

#include "common.cuh"
#include "gate.cuh"
#include "internal.h"

namespace gbmoe {

constexpr int kAlignThreads = 1024;
constexpr int kAlignWarps = kAlignThreads / 32;

// One CTA: the full alignment.  Shared memory: kAlignWarps * E ints (per-warp
// histograms, later per-warp write cursors) + 64 ints.
__device__ void align_cta(const AlignArgs& a) {
  extern __shared__ int smem[];
  int* cur = smem;                              // [kAlignWarps][E]
  int* scan_tmp = smem + kAlignWarps * a.E;     // [33]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = a.M * a.topk;
  const int sentinel = n;
  const int B = a.block;

  for (int i = tid; i < kAlignWarps * a.E; i += kAlignThreads) cur[i] = 0;
  for (int i = tid; i < a.cap; i += kAlignThreads) a.sorted_ids[i] = sentinel;
  for (int i = tid; i < a.cap / B; i += kAlignThreads) a.expert_ids[i] = -1;
  __syncthreads();

  // pass 1: per-warp histogram over a contiguous segment of slots
  const int seg = (n + kAlignWarps - 1) / kAlignWarps;
  const int beg = min(n, warp * seg), end = min(n, beg + seg);
  int bad = 0;
  for (int i = beg + lane; i < end; i += 32) {
    const int e = a.topk_ids[i];
    if (e >= 0 && e < a.E) atomicAdd(&cur[warp * a.E + e], 1);
    else ++bad;
  }
  bad = warp_sum_i(bad);
  if (lane == 0 && bad && a.status) atomicAdd(&a.status->bad_ids, bad);
  __syncthreads();

  // pass 2: expert totals -> padded offsets (scan), per-warp cursors, active list
  for (int e0 = 0; e0 < a.E; e0 += kAlignThreads) {
    // E <= MOE_MAX_EXPERTS == kAlignThreads, so this loop runs once
    const int e = e0 + tid;
    int cnt = 0;
    if (e < a.E) {
#pragma unroll 4
      for (int w = 0; w < kAlignWarps; ++w) cnt += cur[w * a.E + e];
    }
    const int padded = (cnt + B - 1) / B * B;
    int total;
    const int off = block_exclusive_scan(padded, scan_tmp, total);
    int nact;
    const int act_idx = block_exclusive_scan(cnt > 0 ? 1 : 0, scan_tmp, nact);
    const int ntt = a.ttiles ? (cnt + a.tile_tokens - 1) / a.tile_tokens : 0;
    int n_tt;
    const int tt0 = block_exclusive_scan(ntt, scan_tmp, n_tt);
    if (e < a.E) {
      int c = off;
      for (int w = 0; w < kAlignWarps; ++w) {
        const int t = cur[w * a.E + e];
        cur[w * a.E + e] = c;
        c += t;
      }
      if (a.expert_offsets) a.expert_offsets[e] = off;
      if (a.counts) a.counts[e] = cnt;
      if (a.active && cnt > 0) a.active[act_idx] = e;
      for (int b = off / B; b < (off + padded) / B; ++b) a.expert_ids[b] = e;
      for (int i = 0; i < ntt; ++i) {
        const int start = i * a.tile_tokens;
        a.ttiles[tt0 + i] = make_int4(e, off + start, min(a.tile_tokens, cnt - start), 0);
      }
    }
    if (tid == 0) {
      if (a.expert_offsets) a.expert_offsets[a.E] = total;
      if (a.num_post) *a.num_post = total;
      if (a.num_active) *a.num_active = nact;
      if (a.num_ttiles) *a.num_ttiles = n_tt;
    }
  }
  __syncthreads();

  // pass 3: stable scatter; each warp walks its segment in slot order
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int base = beg; base < end; base += 32) {
    const int i = base + lane;
    const int e = (i < end) ? a.topk_ids[i] : -1;
    const bool ok = (i < end) && e >= 0 && e < a.E;
    const unsigned peers = __match_any_sync(0xffffffffu, ok ? e : -1);
    const int rank = __popc(peers & lt_mask);
    if (ok) {
      const int pos = cur[warp * a.E + e] + rank;
      a.sorted_ids[pos] = i;
      if (a.inv_pos) a.inv_pos[i] = pos;
    } else if (i < end && a.inv_pos) {
      a.inv_pos[i] = -1;
    }
    __syncwarp();
    if (ok && rank == 0) cur[warp * a.E + e] += __popc(peers);
    __syncwarp();
  }
}

// FP8 E4M3 codes of one row in groups of 128 columns: s = amax / 448 (fp32,
// 1 for an all-zero group), q = E4M3(x / s) rounded to nearest even with
// saturation, the division in IEEE fp32.  One warp per group, 4 columns a lane.
__device__ void prep_row_fp8_1x128(const __nv_bfloat16* xr, uint8_t* qr, float* sr, int H) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int g = warp; g < H / kQBlock; g += nw) {
    const uint2 raw = *reinterpret_cast<const uint2*>(xr + g * kQBlock + lane * 4);
    const __nv_bfloat162 b0 = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
    const __nv_bfloat162 b1 = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
    const float2 f0 = __bfloat1622float2(b0), f1 = __bfloat1622float2(b1);
    float m = fmaxf(fmaxf(fabsf(f0.x), fabsf(f0.y)), fmaxf(fabsf(f1.x), fabsf(f1.y)));
    m = warp_max(m);
    const float s = m > 0.f ? __fdiv_rn(m, 448.0f) : 1.0f;
    const uint32_t c0 = e4m3_code(__fdiv_rn(f0.x, s)), c1 = e4m3_code(__fdiv_rn(f0.y, s));
    const uint32_t c2 = e4m3_code(__fdiv_rn(f1.x, s)), c3 = e4m3_code(__fdiv_rn(f1.y, s));
    *reinterpret_cast<uint32_t*>(qr + g * kQBlock + lane * 4) = c0 | (c1 << 8) | (c2 << 16) | (c3 << 24);
    if (lane == 0) sr[g] = s;
  }
}

// Row preparation of the activations, one CTA per row at a time.
//   kind 1: x bf16 -> fp16 (RN)               (FP8 weight-only path)
//   kind 2: x bf16 -> int8 codes + fp32 scale (DA8W8 path); codes stored as
//           fp16 (exact) or int8
//   kind 3: x bf16 -> E4M3 codes + one fp32 scale per 128 columns (FP8 A8 path)
//   kind 4: x bf16 -> fp16 (RN), each group of 8 columns stored in the order
//           0 4 1 5 2 6 3 7 (INT4 path: the order its weights expand in)
template <typename QT>
__device__ void prep_rows(const PrepArgs& p, int row0, int rstride) {
  __shared__ float red[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  for (int r = row0; r < p.M; r += rstride) {
    const __nv_bfloat16* xr = p.x + static_cast<size_t>(r) * p.H;
    if (p.kind == 3) {
      prep_row_fp8_1x128(xr, static_cast<uint8_t*>(p.q) + static_cast<size_t>(r) * p.H,
                         p.scale + static_cast<size_t>(r) * (p.H / kQBlock), p.H);
      continue;
    }
    if (p.kind == 4) {
      uint4* qr4 = reinterpret_cast<uint4*>(static_cast<__half*>(p.q) + static_cast<size_t>(r) * p.H);
      for (int c = tid; c < p.H / 8; c += blockDim.x) {
        const uint4 raw = *reinterpret_cast<const uint4*>(xr + 8 * c);
        const float2 f01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
        const float2 f23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
        const float2 f45 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.z));
        const float2 f67 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.w));
        qr4[c] = make_uint4(pack_half2(f01.x, f45.x), pack_half2(f01.y, f45.y), pack_half2(f23.x, f67.x),
                            pack_half2(f23.y, f67.y));
      }
      continue;
    }
    QT* qr = reinterpret_cast<QT*>(p.q) + static_cast<size_t>(r) * p.H;
    if (p.kind == 1) {
      for (int c = tid; c < p.H; c += blockDim.x) qr[c] = static_cast<QT>(__bfloat162float(xr[c]));
      continue;
    }
    float m = 0.f;
    for (int c = tid; c < p.H; c += blockDim.x) m = fmaxf(m, fabsf(__bfloat162float(xr[c])));
    m = warp_max(m);
    if (lane == 0) red[warp] = m;
    __syncthreads();
    if (warp == 0) {
      float v = lane < nw ? red[lane] : 0.f;
      v = warp_max(v);
      if (lane == 0) red[0] = v;
    }
    __syncthreads();
    const float amax = red[0];
    const float s = amax > 0.f ? __fdiv_rn(amax, 127.0f) : 1.0f;
    if (tid == 0 && p.scale) p.scale[r] = s;
    for (int c = tid; c < p.H; c += blockDim.x)
      qr[c] = static_cast<QT>(quant_s8_rne(__bfloat162float(xr[c]), s));
    __syncthreads();
  }
}

// GV > 0: the alignment CTA first ranks every token's experts (router gating,
// GV experts per lane) and writes topk_ids / topk_weights, then aligns them.
template <int GV>
__global__ void __launch_bounds__(kAlignThreads) prologue_kernel(AlignArgs a, PrepArgs p, GateArgs g) {
  pdl_trigger();  // the next kernel may set itself up; it waits for this grid before reading
  pdl_wait();     // inputs (and this workspace's previous readers) belong to earlier kernels
  if (blockIdx.x == 0) {
    if (a.status && threadIdx.x == 0) { a.status->bad_ids = 0; a.status->flags = 0; }
    if constexpr (GV > 0) {
      for (int t = threadIdx.x >> 5; t < g.M; t += kAlignWarps) gate_token<GV>(g, t, threadIdx.x & 31);
    }
    __syncthreads();  // the ids written above are read by the whole CTA below
    align_cta(a);
    return;
  }
  // zero the per-row amax words of the INT8 intermediate
  if (p.zero_words) {
    const int stride = (gridDim.x - 1) * blockDim.x;
    for (int i = (blockIdx.x - 1) * blockDim.x + threadIdx.x; i < p.n_zero; i += stride) p.zero_words[i] = 0u;
  }
  if (p.kind != 0) prep_rows<__half>(p, blockIdx.x - 1, gridDim.x - 1);
}

__global__ void __launch_bounds__(256) quant_rows_kernel(PrepArgs p) {
  prep_rows<int8_t>(p, blockIdx.x, gridDim.x);
}

size_t align_smem_bytes(int E) { return static_cast<size_t>(kAlignWarps * E + 64) * sizeof(int); }

template <int GV>
static cudaError_t launch_prologue_t(const AlignArgs& a, const PrepArgs& p, const GateArgs& g, int prep_ctas,
                                     cudaStream_t s) {
  const size_t smem = align_smem_bytes(a.E);
  cudaError_t err = set_smem_limit_once(reinterpret_cast<const void*>(prologue_kernel<GV>),
                                        static_cast<int>(align_smem_bytes(MOE_MAX_EXPERTS)));
  if (err != cudaSuccess) return err;
  return launch_kernel(prologue_kernel<GV>, dim3(1 + prep_ctas), dim3(kAlignThreads), smem, s, true, a, p, g);
}

cudaError_t launch_prologue(const AlignArgs& a, const PrepArgs& p, int prep_ctas, cudaStream_t s,
                            const GateArgs* inline_gate) {
  if (!inline_gate) return launch_prologue_t<0>(a, p, GateArgs{}, prep_ctas, s);
  switch (gate_vpl(inline_gate->E)) {
    case 1: return launch_prologue_t<1>(a, p, *inline_gate, prep_ctas, s);
    case 2: return launch_prologue_t<2>(a, p, *inline_gate, prep_ctas, s);
    case 4: return launch_prologue_t<4>(a, p, *inline_gate, prep_ctas, s);
    case 8: return launch_prologue_t<8>(a, p, *inline_gate, prep_ctas, s);
  }
  return cudaErrorInvalidValue;  // the caller ranks more than 256 experts in its own launch
}

cudaError_t launch_quant_rows(const PrepArgs& p, cudaStream_t s) {
  const int grid = p.M < 2048 ? p.M : 2048;
  if (grid == 0) return cudaSuccess;
  quant_rows_kernel<<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace gbmoe
