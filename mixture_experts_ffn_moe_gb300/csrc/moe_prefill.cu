// Prefill path of the fused MoE layer: grouped expert GEMMs on tcgen05 tensor cores.
//
// At prefill token counts the layer is a real dense contraction per expert.
// The pages' blocked formulation (SGLang CPU backend write-up, section "(3)
// FusedMoE": sort the slots by expert, cut them into blocks, run all experts'
// blocks in parallel) becomes, on GB300, a persistent grouped GEMM over tiles
//   (token tile of one expert: <= 256 consecutive sorted slots) x (128 weight rows).
// The expert-contiguous row layout is the "contiguous" grouped-GEMM layout of
// the LMSYS large-scale-EP news rewrite (section "DeepGEMM integration").
//
// Swap-AB: weights are the MMA's M = 128 side, tokens its N side (16..256,
// a multiple of 16), so a tile with few tokens wastes little tensor work.
// GEMM1 keeps two TMEM accumulators -- 128 gate rows and the matching 128 up
// rows -- against the same activation tile: A x [B1, B2] = [C1, C2], and the
// epilogue computes SiLU(C1) * C2 (Xeon 6 / SGLang blog, section "MoE").
//
// Weights stay FP8 E4M3 (or INT8) in HBM.  TMA brings raw 128x64-byte weight
// tiles into shared memory; converter warps expand them to fp16 in registers
// and write the tcgen05 operand (K-major, 128-byte swizzle).  For FP8 the
// 128x128 block scale is folded into that conversion (one fp32 multiply per
// weight, rounded once to fp16), because a tensor-core accumulator cannot be
// rescaled per K block without a second TMEM pass.  INT8 weights convert
// exactly and the per-row x per-channel scales are applied in the epilogue.
//
// Warp roles (15 warps, 1 CTA per SM, persistent):
//   warp 0      TMA producer of raw weight tiles        (ring of 5 stages)
//   warp 1      TMEM allocator + tcgen05.mma issuer
//   warp 2      TMA producer of activation tiles        (ring of 2 stages)
//   warps 3-10  converters: raw FP8/INT8 -> fp16 swizzled operand
//   warps 11-14 epilogue: TMEM -> registers -> SiLU*mul / routing weight -> HBM
// Every wait is bounded; a time-out sets the status flag and all roles drain.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace gbmoe {
namespace pf {

using namespace sm100;

constexpr int BK = 64;                 // K elements per pipeline stage
constexpr int BM = 128;                // weight rows per accumulator (MMA M)
constexpr int RAW_STAGES = 5;
constexpr int STAGES = 2;
constexpr int RAW_TILE = BM * BK;      // 8 KB of fp8/int8 codes
constexpr int A_TILE = BM * BK * 2;    // 16 KB fp16 operand
constexpr int B_TILE = kPrefillTileTokens * BK * 2;  // 32 KB fp16 activations
constexpr int N_CONV_WARPS = 8;
constexpr int N_EPI_WARPS = 4;
constexpr int WARP_WTMA = 0, WARP_MMA = 1, WARP_ATMA = 2, WARP_CONV0 = 3;
constexpr int WARP_EPI0 = WARP_CONV0 + N_CONV_WARPS;
constexpr int NUM_WARPS = WARP_EPI0 + N_EPI_WARPS;
constexpr int NUM_THREADS = NUM_WARPS * 32;
constexpr int CONV_THREADS = N_CONV_WARPS * 32;
constexpr int EPI_THREADS = N_EPI_WARPS * 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t UP_COL = 256;       // TMEM column of the up accumulator

constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + STAGES * 2 * A_TILE;
constexpr int OFF_RAW = OFF_B + STAGES * B_TILE;
constexpr int OFF_BAR = OFF_RAW + RAW_STAGES * 2 * RAW_TILE;
constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;  // + slack to align the base to 1024
constexpr long long kWaitLimit = 4000000000LL;    // ~2 s of SM clocks per wait

struct Bars {
  uint64_t raw_full[RAW_STAGES];
  uint64_t raw_empty[RAW_STAGES];
  uint64_t act_full[STAGES];
  uint64_t conv_full[STAGES];
  uint64_t stage_empty[STAGES];
  uint64_t acc_full;
  uint64_t acc_empty;
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block too large");

struct Tile {
  int e, pos0, cnt, n0, nmma;
};

__device__ __forceinline__ Tile get_tile(const PrefillArgs& p, int t) {
  const int tt = t / p.n_tiles;
  const int4 d = p.ttiles[tt];
  Tile r;
  r.e = d.x;
  r.pos0 = d.y;
  r.cnt = d.z;
  r.n0 = (t - tt * p.n_tiles) * BM;
  r.nmma = (d.z + 15) & ~15;
  return r;
}

template <int WK, bool GATED>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    prefill_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_b,
                        PrefillArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem + OFF_A;
  uint8_t* sB = smem + OFF_B;
  uint8_t* sRaw = smem + OFF_RAW;
  Bars* bars = reinterpret_cast<Bars*>(smem + OFF_BAR);
  volatile int* abort = &bars->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int total_tiles = *p.num_ttiles * p.n_tiles;
  const int KC = p.K / BK;
  constexpr int NACC = GATED ? 2 : 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < RAW_STAGES; ++i) { mbar_init(&bars->raw_full[i], 1); mbar_init(&bars->raw_empty[i], CONV_THREADS); }
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&bars->act_full[i], 1);
      mbar_init(&bars->conv_full[i], CONV_THREADS);
      mbar_init(&bars->stage_empty[i], 1);
    }
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_empty, EPI_THREADS);
    mbar_init(&bars->mma_done, 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == WARP_MMA) {
    tmem_alloc(&bars->tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == WARP_WTMA && lane == 0) { prefetch_tmap(&tmap_w); prefetch_tmap(&tmap_b); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars->tmem_base;

  if (warp == WARP_WTMA) {
    // ---------------------------------------------------------------- raw weight producer
    if (lane == 0) {
      int rs = 0;
      uint32_t rph = 0;
      int last_par[RAW_STAGES];
      for (int i = 0; i < RAW_STAGES; ++i) last_par[i] = -1;
      bool ok = true;
      for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
        const Tile tl = get_tile(p, t);
        const int row_g = tl.e * p.rows_per_expert + tl.n0;
        for (int kc = 0; kc < KC; ++kc) {
          if (!(ok = mbar_wait(&bars->raw_empty[rs], rph ^ 1, abort, p.status, kWaitLimit))) break;
          mbar_arrive_expect_tx(&bars->raw_full[rs], NACC * RAW_TILE);
          uint8_t* dst = sRaw + rs * 2 * RAW_TILE;
          tma_load_2d(dst, &tmap_w, &bars->raw_full[rs], kc * BK, row_g);
          if (GATED) tma_load_2d(dst + RAW_TILE, &tmap_w, &bars->raw_full[rs], kc * BK, row_g + p.up_offset);
          last_par[rs] = static_cast<int>(rph);
          if (++rs == RAW_STAGES) { rs = 0; rph ^= 1; }
        }
      }
      // never leave with copies in flight into this CTA's shared memory
      for (int i = 0; i < RAW_STAGES; ++i)
        if (last_par[i] >= 0) {
          int dummy = 0;
          mbar_wait(&bars->raw_full[i], static_cast<uint32_t>(last_par[i]), &dummy, nullptr, kWaitLimit);
        }
    }
  } else if (warp == WARP_ATMA) {
    // ---------------------------------------------------------------- activation producer
    if (lane == 0) {
      int cs = 0;
      uint32_t cph = 0;
      int last_par[STAGES];
      for (int i = 0; i < STAGES; ++i) last_par[i] = -1;
      bool ok = true;
      for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
        const Tile tl = get_tile(p, t);
        for (int kc = 0; kc < KC; ++kc) {
          if (!(ok = mbar_wait(&bars->stage_empty[cs], cph ^ 1, abort, p.status, kWaitLimit))) break;
          mbar_arrive_expect_tx(&bars->act_full[cs], tl.nmma * BK * 2);
          uint8_t* dst = sB + cs * B_TILE;
          for (int r = 0; r < tl.nmma; r += 16)
            tma_load_2d(dst + r * (BK * 2), &tmap_b, &bars->act_full[cs], kc * BK, tl.pos0 + r);
          last_par[cs] = static_cast<int>(cph);
          if (++cs == STAGES) { cs = 0; cph ^= 1; }
        }
      }
      for (int i = 0; i < STAGES; ++i)
        if (last_par[i] >= 0) {
          int dummy = 0;
          mbar_wait(&bars->act_full[i], static_cast<uint32_t>(last_par[i]), &dummy, nullptr, kWaitLimit);
        }
    }
  } else if (warp == WARP_MMA) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int cs = 0;
      uint32_t cph = 0, aph = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
        const Tile tl = get_tile(p, t);
        const uint32_t idesc = idesc_f16_f32(BM, tl.nmma);
        if (!(ok = mbar_wait(&bars->acc_empty, aph ^ 1, abort, p.status, kWaitLimit))) break;
        tc_fence_after();
        for (int kc = 0; kc < KC; ++kc) {
          if (!(ok = mbar_wait(&bars->conv_full[cs], cph, abort, p.status, kWaitLimit))) break;
          if (!(ok = mbar_wait(&bars->act_full[cs], cph, abort, p.status, kWaitLimit))) break;
          tc_fence_after();
          const uint64_t ag = sw128_kmajor_desc(smem_addr(sA + cs * 2 * A_TILE));
          const uint64_t au = sw128_kmajor_desc(smem_addr(sA + cs * 2 * A_TILE + A_TILE));
          const uint64_t bd = sw128_kmajor_desc(smem_addr(sB + cs * B_TILE));
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint32_t acc = (kc | k) != 0;
            umma_f16(tbase, ag + 2 * k, bd + 2 * k, idesc, acc);  // +32 bytes along K per step
            if (GATED) umma_f16(tbase + UP_COL, au + 2 * k, bd + 2 * k, idesc, acc);
          }
          umma_commit(&bars->stage_empty[cs]);
          if (++cs == STAGES) { cs = 0; cph ^= 1; }
        }
        if (!ok) break;
        umma_commit(&bars->acc_full);
        aph ^= 1;
      }
      // every issued MMA must finish before TMEM is released
      umma_commit(&bars->mma_done);
      int dummy = 0;
      mbar_wait(&bars->mma_done, 0, &dummy, nullptr, kWaitLimit);
    }
  } else if (warp < WARP_EPI0) {
    // ---------------------------------------------------------------- converters
    const int ct = threadIdx.x - WARP_CONV0 * 32;
    int rs = 0, cs = 0;
    uint32_t rph = 0, cph = 0;
    bool ok = true;
    const int kblocks = p.K / kQBlock;
    const int rblocks = p.rows_per_expert / kQBlock;
    for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
      const Tile tl = get_tile(p, t);
      for (int kc = 0; kc < KC; ++kc) {
        if (!(ok = mbar_wait(&bars->raw_full[rs], rph, abort, p.status, kWaitLimit))) break;
        if (!(ok = mbar_wait(&bars->stage_empty[cs], cph ^ 1, abort, p.status, kWaitLimit))) break;
        float sc[2] = {1.f, 1.f};
        if constexpr (WK == MOE_WEIGHT_FP8) {
          const float* s = p.wscale + static_cast<size_t>(tl.e) * rblocks * kblocks + (kc * BK) / kQBlock;
          sc[0] = __ldg(s + static_cast<size_t>(tl.n0 / kQBlock) * kblocks);
          if (GATED) sc[1] = __ldg(s + static_cast<size_t>((p.up_offset + tl.n0) / kQBlock) * kblocks);
        }
        const uint8_t* raw = sRaw + rs * 2 * RAW_TILE;
        uint8_t* dstA = sA + cs * 2 * A_TILE;
#pragma unroll
        for (int s = 0; s < NACC * (BM * BK / 16) / CONV_THREADS; ++s) {
          const int j = ct + s * CONV_THREADS;      // 16-byte chunk of the raw stage
          const int acc = j / (BM * BK / 16);        // 0 gate, 1 up
          const int idx = j - acc * (BM * BK / 16);
          const int row = idx >> 2, c16 = idx & 3;
          const uint4 v = *reinterpret_cast<const uint4*>(raw + acc * RAW_TILE + row * BK + c16 * 16);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
          uint32_t o[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            w8x4_to_f16x4<WK>(w[i], o[2 * i], o[2 * i + 1]);
            if constexpr (WK == MOE_WEIGHT_FP8) {
              const float s2 = sc[acc];
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&o[2 * i + h]));
                o[2 * i + h] = pack_half2(f.x * s2, f.y * s2);
              }
            }
          }
          uint8_t* rowp = dstA + acc * A_TILE + row * 128;
          const int r8 = row & 7;
          *reinterpret_cast<uint4*>(rowp + (((2 * c16) ^ r8) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<uint4*>(rowp + (((2 * c16 + 1) ^ r8) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
        }
        fence_proxy_async_smem();
        mbar_arrive(&bars->conv_full[cs]);
        mbar_arrive(&bars->raw_empty[rs]);
        if (++rs == RAW_STAGES) { rs = 0; rph ^= 1; }
        if (++cs == STAGES) { cs = 0; cph ^= 1; }
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    uint32_t aph = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
      const Tile tl = get_tile(p, t);
      if (!(ok = mbar_wait(&bars->acc_full, aph, abort, p.status, kWaitLimit))) break;
      tc_fence_after();
      const int n = tl.n0 + row;
      float swg = 1.f, swu = 1.f;
      if constexpr (WK == MOE_WEIGHT_INT8) {
        swg = __ldg(p.wscale + static_cast<size_t>(tl.e) * p.rows_per_expert + n);
        if (GATED) swu = __ldg(p.wscale + static_cast<size_t>(tl.e) * p.rows_per_expert + p.up_offset + n);
      }
      const uint32_t lane_addr = tbase + (static_cast<uint32_t>(q * 32) << 16);
      for (int c0 = 0; c0 < tl.nmma; c0 += 32) {
        uint32_t g[32], u[32];
        __syncwarp();
        tmem_ld32(lane_addr + c0, g);
        if (GATED) tmem_ld32(lane_addr + UP_COL + c0, u);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int col = c0 + j;
          if (col >= tl.cnt) continue;  // warp-uniform
          const int pos = tl.pos0 + col;
          const float gv = __uint_as_float(g[j]);
          if constexpr (GATED) {
            const float uv = __uint_as_float(u[j]);
            if constexpr (WK == MOE_WEIGHT_FP8) {
              reinterpret_cast<__half*>(p.out)[static_cast<size_t>(pos) * p.out_ld + n] =
                  __float2half_rn(silu_f32(gv) * uv);
            } else {
              const float sx = __ldg(p.sx + __ldg(p.sorted_ids + pos) / p.topk);
              const float h = silu_f32(gv * sx * swg) * (uv * sx * swu);
              reinterpret_cast<float*>(p.out)[static_cast<size_t>(pos) * p.out_ld + n] = h;
              float m = fabsf(h);
              m = warp_max(m);
              if (lane == 0) atomicMax(p.hmax + pos, __float_as_uint(m));
            }
          } else {
            const int slot = __ldg(p.sorted_ids + pos);
            float s = __ldg(p.topk_w + slot);
            if constexpr (WK == MOE_WEIGHT_INT8) s *= __ldg(p.sh + pos) * swg;
            reinterpret_cast<float*>(p.out)[static_cast<size_t>(pos) * p.out_ld + n] = gv * s;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bars->acc_empty);
      aph ^= 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, TMEM_COLS);
  }
}

}  // namespace pf

// ------------------------------------------------------------------ gather and combine
// Activation rows in sorted (expert-contiguous) order; padding rows are zero.
__global__ void __launch_bounds__(256) gather_rows_kernel(const __half* __restrict__ xq,
                                                          const int32_t* __restrict__ sorted_ids,
                                                          const int32_t* __restrict__ num_post, int n_slots,
                                                          int topk, int H, __half* __restrict__ act) {
  const int rows = *num_post;
  const int chunks = H / 8;
  const long long total = static_cast<long long>(rows) * chunks;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int pos = static_cast<int>(i / chunks), c = static_cast<int>(i - static_cast<long long>(pos) * chunks);
    const int slot = __ldg(sorted_ids + pos);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (slot < n_slots) v = ld_v4(xq + static_cast<size_t>(slot / topk) * H + c * 8);
    *reinterpret_cast<uint4*>(act + static_cast<size_t>(pos) * H + c * 8) = v;
  }
}

// out[t, n] = sum over k (in slot order) of y[pos(t, k), n]; y already carries the routing weight.
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y, const int32_t* __restrict__ inv_pos,
                                                      int M, int topk, int H, __nv_bfloat16* __restrict__ out) {
  const int q = H / 4;
  const long long total = static_cast<long long>(M) * q;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / q), c = static_cast<int>(i - static_cast<long long>(t) * q);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < topk; ++k) {
      const int pos = __ldg(inv_pos + t * topk + k);
      if (pos < 0) continue;
      const float4 v = __ldg(reinterpret_cast<const float4*>(y + static_cast<size_t>(pos) * H) + c);
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 pk = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
    *reinterpret_cast<uint2*>(out + static_cast<size_t>(t) * H + 4 * c) = pk;
  }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// 2D row-major tensor [outer, inner] of `esize`-byte elements, box [box_outer, box_inner].
static bool make_map(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, uint64_t inner,
                     uint64_t outer, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * static_cast<uint64_t>(esize)};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int WK, bool GATED>
static cudaError_t launch_gemm(const PrefillArgs& a, const void* w, uint64_t w_rows, const void* b, uint64_t b_rows,
                               int num_sms, cudaStream_t s) {
  CUtensorMap mw, mb;
  if (!make_map(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, w, static_cast<uint64_t>(a.K), w_rows, pf::BK, pf::BM,
                CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  if (!make_map(&mb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, b, static_cast<uint64_t>(a.K), b_rows, pf::BK, 16,
                CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  auto kern = pf::prefill_gemm_kernel<WK, GATED>;
  cudaError_t err = set_smem_limit_once(reinterpret_cast<const void*>(kern), pf::SMEM_BYTES,
                                        4 + WK * 2 + (GATED ? 1 : 0));
  if (err != cudaSuccess) return err;
  kern<<<num_sms, pf::NUM_THREADS, pf::SMEM_BYTES, s>>>(mw, mb, a);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const PrefillPlan& P, int weight_kind, int num_sms, cudaStream_t s, const StageHook& hook) {
  cudaError_t err;
  {
    int grid = num_sms * 8;
    gather_rows_kernel<<<grid, 256, 0, s>>>(P.xq, P.sorted_ids, P.num_post, P.M * P.topk, P.topk, P.H, P.act);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    hook("prefill_gather", s);
  }
  PrefillArgs g1{};
  g1.K = P.H;
  g1.rows_per_expert = 2 * P.I;
  g1.up_offset = P.I;
  g1.n_tiles = P.I / pf::BM;
  g1.ttiles = P.ttiles;
  g1.num_ttiles = P.num_ttiles;
  g1.wscale = P.s13;
  g1.sorted_ids = P.sorted_ids;
  g1.topk = P.topk;
  g1.sx = P.sx;
  g1.out = P.h;
  g1.out_ld = P.I;
  g1.hmax = P.hmax;
  g1.status = P.status;
  err = weight_kind == MOE_WEIGHT_FP8
            ? launch_gemm<MOE_WEIGHT_FP8, true>(g1, P.w13, static_cast<uint64_t>(P.E) * 2 * P.I, P.act, P.cap,
                                                num_sms, s)
            : launch_gemm<MOE_WEIGHT_INT8, true>(g1, P.w13, static_cast<uint64_t>(P.E) * 2 * P.I, P.act, P.cap,
                                                 num_sms, s);
  if (err != cudaSuccess) return err;
  hook("prefill_gemm1", s);
  const __half* b2 = reinterpret_cast<const __half*>(P.h);
  if (weight_kind == MOE_WEIGHT_INT8) {
    err = launch_requant_rows(P.h, P.hmax, P.num_post, P.cap, P.I, P.hq, P.sh, num_sms, s);
    if (err != cudaSuccess) return err;
    hook("requant_h", s);
    b2 = P.hq;
  }
  PrefillArgs g2{};
  g2.K = P.I;
  g2.rows_per_expert = P.H;
  g2.up_offset = 0;
  g2.n_tiles = P.H / pf::BM;
  g2.ttiles = P.ttiles;
  g2.num_ttiles = P.num_ttiles;
  g2.wscale = P.s2;
  g2.sorted_ids = P.sorted_ids;
  g2.topk = P.topk;
  g2.sh = P.sh;
  g2.topk_w = P.topk_w;
  g2.out = P.y;
  g2.out_ld = P.H;
  g2.status = P.status;
  err = weight_kind == MOE_WEIGHT_FP8
            ? launch_gemm<MOE_WEIGHT_FP8, false>(g2, P.w2, static_cast<uint64_t>(P.E) * P.H, b2, P.cap, num_sms, s)
            : launch_gemm<MOE_WEIGHT_INT8, false>(g2, P.w2, static_cast<uint64_t>(P.E) * P.H, b2, P.cap, num_sms,
                                                  s);
  if (err != cudaSuccess) return err;
  hook("prefill_gemm2", s);
  {
    const long long work = static_cast<long long>(P.M) * (P.H / 4);
    long long grid = (work + 255) / 256;
    if (grid > num_sms * 16) grid = num_sms * 16;
    if (grid < 1) grid = 1;
    combine_kernel<<<static_cast<int>(grid), 256, 0, s>>>(P.y, P.inv_pos, P.M, P.topk, P.H, P.out);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    hook("prefill_combine", s);
  }
  return cudaSuccess;
}

size_t prefill_smem_bytes() { return pf::SMEM_BYTES; }

}  // namespace gbmoe
