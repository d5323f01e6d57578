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
// GB300 design: the alignment runs in three passes over shared memory --
// per-warp expert histograms, one block-wide scan that turns them into write
// cursors, and a warp-ordered scatter in which __match_any_sync ranks equal
// ids inside each 32-slot step.  Up to kAlignChunkSlots slots one CTA of 1024
// threads does all of it, and the other CTAs of the same launch prepare the
// activation rows for the expert GEMMs.  Longer id lists are cut into
// consecutive chunks, one CTA each: the prologue's first CTAs write every
// chunk's expert histogram to the workspace, and a second launch gives each
// chunk's CTA the sum over the chunks before it as its starting cursors, so
// the scatter is the same stable order as the single CTA's; that launch's
// other CTAs prepare the activations.
#include <cuda_runtime.h>

#include "common.cuh"
#include "gate.cuh"
#include "internal.h"

namespace gbmoe {

constexpr int kAlignThreads = 1024;
constexpr int kAlignWarps = kAlignThreads / 32;

// Per-warp histograms of slots [lo, hi): warp w takes a contiguous segment
// [beg, end).  Returns the ids outside [0, E) the warp saw.
__device__ __forceinline__ int align_histogram(const AlignArgs& a, int* cur, int lo, int hi, int& beg, int& end) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int seg = (hi - lo + kAlignWarps - 1) / kAlignWarps;
  beg = min(hi, lo + warp * seg);
  end = min(hi, beg + seg);
  int bad = 0;
  for (int i = beg + lane; i < end; i += 32) {
    const int e = a.topk_ids[i];
    if (e >= 0 && e < a.E) atomicAdd(&cur[warp * a.E + e], 1);
    else ++bad;
  }
  return warp_sum_i(bad);
}

// The alignment of slots [lo, hi) by one CTA.  Shared memory: kAlignWarps * E
// ints (per-warp histograms, later per-warp write cursors) + 64 ints.
//   !SPLIT: [lo, hi) is every slot; this CTA fills the padding, counts, plans
//     and scatters (chunk_counts unused).
//   SPLIT: chunk_counts[c * E + e] holds every chunk's histogram; this CTA
//     is chunk `chunk` and scatters its slots after those of chunks
//     0..chunk-1 (the first launch filled the padding); chunk 0 writes the plan.
template <bool SPLIT>
__device__ void align_core(const AlignArgs& a, int lo, int hi, const int* chunk_counts, int chunk, int nchunks) {
  extern __shared__ int smem[];
  int* cur = smem;                              // [kAlignWarps][E]
  int* scan_tmp = smem + kAlignWarps * a.E;     // [33]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = a.block;
  const bool plan = !SPLIT || chunk == 0;  // CTA-uniform

  for (int i = tid; i < kAlignWarps * a.E; i += kAlignThreads) cur[i] = 0;
  if constexpr (!SPLIT) {
    const int sentinel = a.M * a.topk;
    for (int i = tid; i < a.cap; i += kAlignThreads) a.sorted_ids[i] = sentinel;
    for (int i = tid; i < a.cap / B; i += kAlignThreads) a.expert_ids[i] = -1;
  }
  __syncthreads();

  // pass 1: per-warp histogram over a contiguous segment of slots
  int beg, end;
  const int bad = align_histogram(a, cur, lo, hi, beg, end);
  if (lane == 0 && bad && a.status) atomicAdd(&a.status->bad_ids, bad);
  __syncthreads();

  // pass 2: expert totals -> padded offsets (scan), per-warp cursors, active list
  for (int e0 = 0; e0 < a.E; e0 += kAlignThreads) {
    // E <= MOE_MAX_EXPERTS == kAlignThreads, so this loop runs once
    const int e = e0 + tid;
    int cnt = 0, before = 0;  // slots of expert e in every chunk / in the chunks before this one
    if (e < a.E) {
      if constexpr (SPLIT) {
        for (int c = 0; c < nchunks; ++c) {
          const int v = chunk_counts[c * a.E + e];
          cnt += v;
          if (c < chunk) before += v;
        }
      } else {
#pragma unroll 4
        for (int w = 0; w < kAlignWarps; ++w) cnt += cur[w * a.E + e];
      }
    }
    const int padded = (cnt + B - 1) / B * B;
    int total;
    const int off = block_exclusive_scan(padded, scan_tmp, total);
    const int ntt = a.ttiles ? (cnt + a.tile_tokens - 1) / a.tile_tokens : 0;
    int nact = 0, n_tt = 0, act_idx = 0, tt0 = 0;
    if (plan) {
      act_idx = block_exclusive_scan(cnt > 0 ? 1 : 0, scan_tmp, nact);
      tt0 = block_exclusive_scan(ntt, scan_tmp, n_tt);
    }
    if (e < a.E) {
      int c = off + before;
      for (int w = 0; w < kAlignWarps; ++w) {
        const int t = cur[w * a.E + e];
        cur[w * a.E + e] = c;
        c += t;
      }
      if (plan) {
        if (a.expert_offsets) a.expert_offsets[e] = off;
        if (a.counts) a.counts[e] = cnt;
        if (a.active && cnt > 0) a.active[act_idx] = e;
        for (int b = off / B; b < (off + padded) / B; ++b) a.expert_ids[b] = e;
        for (int i = 0; i < ntt; ++i) {
          const int start = i * a.tile_tokens;
          a.ttiles[tt0 + i] = make_int4(e, off + start, min(a.tile_tokens, cnt - start), 0);
        }
      }
    }
    if (plan && tid == 0) {
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

__device__ void align_cta(const AlignArgs& a) { align_core<false>(a, 0, a.M * a.topk, nullptr, 0, 1); }

// First launch of the split alignment, CTA `chunk` of `nchunks`: its share of
// the padding fill and the expert histogram of its chunk.
__device__ void align_count_chunk(const AlignArgs& a, int* chunk_counts, int chunk, int nchunks) {
  extern __shared__ int smem[];
  int* cur = smem;
  const int tid = threadIdx.x;
  const int n = a.M * a.topk, sentinel = n;
  const int stride = nchunks * kAlignThreads;
  for (int i = chunk * kAlignThreads + tid; i < a.cap; i += stride) a.sorted_ids[i] = sentinel;
  for (int i = chunk * kAlignThreads + tid; i < a.cap / a.block; i += stride) a.expert_ids[i] = -1;
  for (int i = tid; i < kAlignWarps * a.E; i += kAlignThreads) cur[i] = 0;
  __syncthreads();
  const int S = align_chunk_slots(n, nchunks);
  int beg, end;
  align_histogram(a, cur, chunk * S, min(n, (chunk + 1) * S), beg, end);  // bad ids: counted by the scatter
  __syncthreads();
  for (int e = tid; e < a.E; e += kAlignThreads) {
    int cnt = 0;
#pragma unroll 4
    for (int w = 0; w < kAlignWarps; ++w) cnt += cur[w * a.E + e];
    chunk_counts[chunk * a.E + e] = cnt;
  }
}

// Second launch of the split alignment: CTA c < nchunks plans (c == 0) and
// scatters chunk c; the CTAs after them prepare the activations.
__device__ void prep_part(const PrepArgs& p, int cta, int nctas);

__global__ void __launch_bounds__(kAlignThreads) align_scatter_kernel(AlignArgs a, PrepArgs p,
                                                                      const int* chunk_counts, int nchunks) {
  pdl_trigger();
  pdl_wait();  // histograms, padding fill and status reset come from the previous launch
  if (blockIdx.x >= nchunks) {
    prep_part(p, blockIdx.x - nchunks, gridDim.x - nchunks);
    return;
  }
  const int n = a.M * a.topk, S = align_chunk_slots(n, nchunks);
  align_core<true>(a, blockIdx.x * S, min(n, (blockIdx.x + 1) * S), chunk_counts, blockIdx.x, nchunks);
}

// Activation preparation.  The row-wise kinds take one row at a time (its max
// |x| decides the row's scale); the FP8 kind runs as one flat pass over the
// [M, H] matrix (H is a multiple of 128, so rows never split a vector or a
// group); every thread keeps kPrepBatch 16-byte loads in flight.
//   kind 1: x bf16 -> fp16 x * 2^-e with the row's max |x| * 2^-e in [2^14, 2^15),
//           scale[r] = 2^e (FP8 weight-only path)
//   kind 2: x bf16 -> int8 codes + fp32 scale per row (DA8W8 path); codes stored
//           as fp16 (exact) or int8
//   kind 3: x bf16 -> E4M3 codes + one fp32 scale per 128 columns (FP8 A8 path)
//   kind 4: as kind 1, each group of 8 columns stored in the order 0 4 1 5 2 6 3 7
//           (INT4 path: the order its weights expand in)
//   kind 5: x bf16 -> two E4M3 codes per value in a power-of-two frame per 128 columns
//           (FP8 weight-only path on the FP8 tensor cores): hi = E4M3(x * 2^-e), lo = E4M3 of
//           the remainder, with the group's max |x| * 2^-e in [2^7, 2^8); hi codes in rows
//           0..M-1 of q, lo codes in rows M..2M-1, scale[r, g] = 2^e
// Kinds 1, 2 and 4 take a CTA per row when there are few rows and a warp per row
// otherwise.
constexpr int kPrepBatch = 4;

__device__ __forceinline__ float2 bf2_lo_hi(uint32_t w) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
}

// kind 3: FP8 E4M3 codes in groups of 128 columns, s = amax / 448 (fp32, 1 for an
// all-zero group), q = E4M3(x / s) rounded to nearest even with saturation, the
// division in IEEE fp32.  One warp per group, 4 columns a lane; `first` / `stride`
// count warps, and a group index is warp-uniform.
__device__ void prep_fp8_flat(const PrepArgs& p, long long first, long long stride) {
  const int lane = threadIdx.x & 31;
  const long long ng = static_cast<long long>(p.M) * (p.H / kQBlock);
  uint8_t* q = static_cast<uint8_t*>(p.q);
  for (long long g0 = first; g0 < ng; g0 += kPrepBatch * stride) {
    uint2 raw[kPrepBatch];
#pragma unroll
    for (int u = 0; u < kPrepBatch; ++u) {
      const long long gi = g0 + u * stride;
      if (gi < ng) raw[u] = *reinterpret_cast<const uint2*>(p.x + gi * kQBlock + lane * 4);
    }
#pragma unroll
    for (int u = 0; u < kPrepBatch; ++u) {
      const long long gi = g0 + u * stride;
      if (gi >= ng) break;
      const float2 f0 = bf2_lo_hi(raw[u].x), f1 = bf2_lo_hi(raw[u].y);
      float m = fmaxf(fmaxf(fabsf(f0.x), fabsf(f0.y)), fmaxf(fabsf(f1.x), fabsf(f1.y)));
      m = warp_max(m);
      const float sc = m > 0.f ? __fdiv_rn(m, 448.0f) : 1.0f;
      const uint32_t c0 = e4m3_code(__fdiv_rn(f0.x, sc)), c1 = e4m3_code(__fdiv_rn(f0.y, sc));
      const uint32_t c2 = e4m3_code(__fdiv_rn(f1.x, sc)), c3 = e4m3_code(__fdiv_rn(f1.y, sc));
      *reinterpret_cast<uint32_t*>(q + gi * kQBlock + lane * 4) = c0 | (c1 << 8) | (c2 << 16) | (c3 << 24);
      if (lane == 0) p.scale[gi] = sc;
    }
  }
}

// kind 5: x = 2^e (hi + lo) per 1 x 128 group, hi and lo E4M3 codes (round to nearest even; no
// saturation is reached: |x| * 2^-e < 2^8 < 448).  One warp per group, 4 columns a lane; `first` /
// `stride` count warps.
__device__ void prep_split_flat(const PrepArgs& p, long long first, long long stride) {
  const int lane = threadIdx.x & 31;
  const long long ng = static_cast<long long>(p.M) * (p.H / kQBlock);
  uint8_t* q = static_cast<uint8_t*>(p.q);
  const size_t lo_off = static_cast<size_t>(p.M) * p.H;
  for (long long g0 = first; g0 < ng; g0 += kPrepBatch * stride) {
    uint2 raw[kPrepBatch];
#pragma unroll
    for (int u = 0; u < kPrepBatch; ++u) {
      const long long gi = g0 + u * stride;
      if (gi < ng) raw[u] = *reinterpret_cast<const uint2*>(p.x + gi * kQBlock + lane * 4);
    }
#pragma unroll
    for (int u = 0; u < kPrepBatch; ++u) {
      const long long gi = g0 + u * stride;
      if (gi >= ng) break;
      const float2 f0 = bf2_lo_hi(raw[u].x), f1 = bf2_lo_hi(raw[u].y);
      const float m = warp_max(fmaxf(fmaxf(fabsf(f0.x), fabsf(f0.y)), fmaxf(fabsf(f1.x), fabsf(f1.y))));
      const int e = m > 0.f ? e4m3_split_exp(m) : 0;
      uint32_t hi, lo;
      e4m3_split4(make_float4(f0.x, f0.y, f1.x, f1.y), exp2i(-e), hi, lo);
      *reinterpret_cast<uint32_t*>(q + gi * kQBlock + lane * 4) = hi;
      *reinterpret_cast<uint32_t*>(q + lo_off + gi * kQBlock + lane * 4) = lo;
      if (lane == 0) p.scale[gi] = exp2i(e);
    }
  }
}

__device__ __forceinline__ float absmax8(const uint4& v) {
  const float2 f01 = bf2_lo_hi(v.x), f23 = bf2_lo_hi(v.y), f45 = bf2_lo_hi(v.z), f67 = bf2_lo_hi(v.w);
  return fmaxf(fmaxf(fmaxf(fabsf(f01.x), fabsf(f01.y)), fmaxf(fabsf(f23.x), fabsf(f23.y))),
               fmaxf(fmaxf(fabsf(f45.x), fabsf(f45.y)), fmaxf(fabsf(f67.x), fabsf(f67.y))));
}

// Row-wise kinds: the factor a row's values are stored with, from its max |x|, and
// the scale recorded for the row (kind 2: s = amax / 127, codes RNE(x / s) clamped
// to +-127; kinds 1 and 4: the row's power-of-two frame).
template <int KIND>
struct RowQuant {
  float store;   // kind 2: the divisor s; kinds 1, 4: the multiplier 2^-e
  float record;  // scale[r]
  __device__ __forceinline__ explicit RowQuant(float amax) {
    if constexpr (KIND == 2) {
      store = record = amax > 0.f ? __fdiv_rn(amax, 127.0f) : 1.0f;
    } else {
      const int e = x_frame_exp(amax);
      store = exp2i(-e);
      record = exp2i(e);
    }
  }
};

// Stores the 8 values of one 16-byte chunk of a row.
template <int KIND, typename QT>
__device__ __forceinline__ void store_row8(QT* dst, const uint4& v, const RowQuant<KIND>& rq) {
  const float2 f01 = bf2_lo_hi(v.x), f23 = bf2_lo_hi(v.y), f45 = bf2_lo_hi(v.z), f67 = bf2_lo_hi(v.w);
  if constexpr (KIND == 2) {
    const float e[8] = {f01.x, f01.y, f23.x, f23.y, f45.x, f45.y, f67.x, f67.y};
    QT o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j] = static_cast<QT>(quant_s8_rne(e[j], rq.store));
    if constexpr (sizeof(QT) == 2) {
      *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(o);
    } else {
      *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<const uint2*>(o);
    }
  } else {
    const float m = rq.store;
    *reinterpret_cast<uint4*>(dst) =
        KIND == 4 ? make_uint4(pack_half2(f01.x * m, f45.x * m), pack_half2(f01.y * m, f45.y * m),
                               pack_half2(f23.x * m, f67.x * m), pack_half2(f23.y * m, f67.y * m))
                  : make_uint4(pack_half2(f01.x * m, f01.y * m), pack_half2(f23.x * m, f23.y * m),
                               pack_half2(f45.x * m, f45.y * m), pack_half2(f67.x * m, f67.y * m));
  }
}

// Few rows per CTA: the whole CTA takes one row at a time (block-wide amax).
// Many rows: one warp per row, each lane keeping kPrepBatch loads in flight.
template <int KIND, typename QT>
__device__ void prep_rows_amax(const PrepArgs& p, int cta, int nctas) {
  __shared__ float red[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  const int chunks = p.H / 8;
  if (p.M <= 4 * nctas) {
    for (int r = cta; r < p.M; r += nctas) {
      const uint4* xr = reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(r) * p.H);
      float m = 0.f;
      for (int c = tid; c < chunks; c += blockDim.x) m = fmaxf(m, absmax8(ld_v4(xr + c)));
      m = warp_max(m);
      if (lane == 0) red[warp] = m;
      __syncthreads();
      if (warp == 0) {
        float v = lane < nw ? red[lane] : 0.f;
        v = warp_max(v);
        if (lane == 0) red[0] = v;
      }
      __syncthreads();
      const RowQuant<KIND> rq(red[0]);
      if (tid == 0 && p.scale) p.scale[r] = rq.record;
      QT* qr = static_cast<QT*>(p.q) + static_cast<size_t>(r) * p.H;
      for (int c = tid; c < chunks; c += blockDim.x) store_row8<KIND, QT>(qr + 8 * c, ld_v4(xr + c), rq);
      __syncthreads();  // red is rewritten for the next row
    }
    return;
  }
  const long long wstride = static_cast<long long>(nctas) * nw;
  for (long long r = static_cast<long long>(cta) * nw + warp; r < p.M; r += wstride) {
    const uint4* xr = reinterpret_cast<const uint4*>(p.x + r * p.H);
    float m = 0.f;
    for (int c0 = lane; c0 < chunks; c0 += 32 * kPrepBatch) {
      uint4 v[kPrepBatch];
#pragma unroll
      for (int u = 0; u < kPrepBatch; ++u)
        if (c0 + 32 * u < chunks) v[u] = ld_v4(xr + c0 + 32 * u);
#pragma unroll
      for (int u = 0; u < kPrepBatch; ++u)
        if (c0 + 32 * u < chunks) m = fmaxf(m, absmax8(v[u]));
    }
    const RowQuant<KIND> rq(warp_max(m));
    if (lane == 0 && p.scale) p.scale[r] = rq.record;
    QT* qr = static_cast<QT*>(p.q) + r * p.H;
    for (int c0 = lane; c0 < chunks; c0 += 32 * kPrepBatch) {
      uint4 v[kPrepBatch];
#pragma unroll
      for (int u = 0; u < kPrepBatch; ++u)
        if (c0 + 32 * u < chunks) v[u] = ld_v4(xr + c0 + 32 * u);
#pragma unroll
      for (int u = 0; u < kPrepBatch; ++u)
        if (c0 + 32 * u < chunks) store_row8<KIND, QT>(qr + 8 * (c0 + 32 * u), v[u], rq);
    }
  }
}

// The preparation pass spread over `nctas` CTAs, this being CTA `cta` of them.
template <typename QT>
__device__ void prep_rows(const PrepArgs& p, int cta, int nctas) {
  const long long tfirst = static_cast<long long>(cta) * blockDim.x + threadIdx.x;
  const long long tstride = static_cast<long long>(nctas) * blockDim.x;
  switch (p.kind) {
    case 1: prep_rows_amax<1, __half>(p, cta, nctas); break;
    case 4: prep_rows_amax<4, __half>(p, cta, nctas); break;
    case 3: prep_fp8_flat(p, tfirst >> 5, tstride >> 5); break;
    case 5: prep_split_flat(p, tfirst >> 5, tstride >> 5); break;
    case 2: prep_rows_amax<2, QT>(p, cta, nctas); break;
    default: break;
  }
}

// The preparation pass and the clearing of the intermediate's amax / frame words,
// on `nctas` CTAs of which this is CTA `cta`.
__device__ void prep_part(const PrepArgs& p, int cta, int nctas) {
  if (p.zero_words) {
    const int stride = nctas * blockDim.x;
    for (int i = cta * blockDim.x + threadIdx.x; i < p.n_zero; i += stride) p.zero_words[i] = 0u;
  }
  if (p.kind != 0) prep_rows<__half>(p, cta, nctas);
}

// GV > 0: the alignment CTA first ranks every token's experts (router gating,
// GV experts per lane) and writes topk_ids / topk_weights, then aligns them.
// chunk_counts != nullptr: the first launch of the split alignment, whose CTAs
// each histogram one chunk (the activations are prepared by the second launch,
// align_scatter_kernel); otherwise CTA 0 aligns and the others prepare.
template <int GV>
__global__ void __launch_bounds__(kAlignThreads) prologue_kernel(AlignArgs a, PrepArgs p, GateArgs g,
                                                                 int* chunk_counts, int nchunks) {
  pdl_trigger();  // the next kernel may set itself up; it waits for this grid before reading
  pdl_wait();     // inputs (and this workspace's previous readers) belong to earlier kernels
  if (blockIdx.x == 0 && a.status && threadIdx.x == 0) { a.status->bad_ids = 0; a.status->flags = 0; }
  if (chunk_counts) {
    align_count_chunk(a, chunk_counts, blockIdx.x, nchunks);
    return;
  }
  if (blockIdx.x == 0) {
    if constexpr (GV > 0) {
      for (int t = threadIdx.x >> 5; t < g.M; t += kAlignWarps) gate_token<GV>(g, t, threadIdx.x & 31);
    }
    __syncthreads();  // the ids written above are read by the whole CTA below
    align_cta(a);
    return;
  }
  prep_part(p, blockIdx.x - 1, gridDim.x - 1);
}

__global__ void __launch_bounds__(256) quant_rows_kernel(PrepArgs p) {
  prep_rows<int8_t>(p, blockIdx.x, gridDim.x);
}

size_t align_smem_bytes(int E) { return static_cast<size_t>(kAlignWarps * E + 64) * sizeof(int); }

template <int GV>
static cudaError_t launch_prologue_t(const AlignArgs& a, const PrepArgs& p, const GateArgs& g, int prep_ctas,
                                     int* chunk_counts, int nchunks, cudaStream_t s) {
  const size_t smem = align_smem_bytes(a.E);
  const int max_smem = static_cast<int>(align_smem_bytes(MOE_MAX_EXPERTS));
  cudaError_t err = set_smem_limit_once(reinterpret_cast<const void*>(prologue_kernel<GV>), max_smem);
  if (err != cudaSuccess) return err;
  const bool prep = p.kind != 0 || p.zero_words;
  const int first_ctas = chunk_counts ? nchunks : 1 + (prep ? prep_ctas : 0);
  err = launch_kernel(prologue_kernel<GV>, dim3(first_ctas), dim3(kAlignThreads), smem, s, true, a, p, g,
                      chunk_counts, nchunks);
  if (err != cudaSuccess || !chunk_counts) return err;
  err = set_smem_limit_once(reinterpret_cast<const void*>(align_scatter_kernel), max_smem);
  if (err != cudaSuccess) return err;
  return launch_kernel(align_scatter_kernel, dim3(nchunks + (prep ? prep_ctas : 0)), dim3(kAlignThreads), smem, s,
                       true, a, p, static_cast<const int*>(chunk_counts), nchunks);
}

cudaError_t launch_prologue(const AlignArgs& a, const PrepArgs& p, int prep_ctas, cudaStream_t s,
                            const GateArgs* inline_gate, int* chunk_counts) {
  const int nchunks = align_num_chunks(static_cast<long long>(a.M) * a.topk);
  if (nchunks < 2 || inline_gate) chunk_counts = nullptr;  // one CTA aligns (and ranks) everything
  if (!inline_gate) return launch_prologue_t<0>(a, p, GateArgs{}, prep_ctas, chunk_counts, nchunks, s);
  switch (gate_vpl(inline_gate->E)) {
    case 1: return launch_prologue_t<1>(a, p, *inline_gate, prep_ctas, nullptr, 1, s);
    case 2: return launch_prologue_t<2>(a, p, *inline_gate, prep_ctas, nullptr, 1, s);
    case 4: return launch_prologue_t<4>(a, p, *inline_gate, prep_ctas, nullptr, 1, s);
    case 8: return launch_prologue_t<8>(a, p, *inline_gate, prep_ctas, nullptr, 1, s);
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
