// Prefill path of the fused MoE layer: grouped expert GEMMs on tcgen05 tensor cores.
//
// At prefill token counts the layer is a real dense contraction per expert.
// The pages' blocked formulation (SGLang CPU backend write-up, section "(3)
// FusedMoE": sort the slots by expert, cut them into blocks, run all experts'
// blocks in parallel) becomes, on GB300, a persistent grouped GEMM over tiles
//   (token tile of one expert: <= 128 consecutive sorted slots) x (2 x 128 weight rows).
// The expert-contiguous row layout is the "contiguous" grouped-GEMM layout of
// the LMSYS large-scale-EP news rewrite (section "DeepGEMM integration").
//
// Each tile pairs two 128-row weight blocks with one activation tile:
//  * GEMM1: 128 gate rows and the matching 128 up rows, A x [B1, B2] =
//    [C1, C2], and the epilogue computes SiLU(C1) * C2 (Xeon 6 / SGLang blog,
//    section "MoE");
//  * GEMM2: two consecutive 128-row blocks of W2, so every activation byte
//    fetched feeds 256 output rows; it writes each slot's row times its
//    routing weight in bf16, and a separate pass sums every token's rows in
//    slot order.
// Orientation (measured).  Both GEMMs put the tokens on the MMA's M = 128 side
// and both converted weight blocks, adjacent in shared memory, on its N = 256
// side: one MMA per K step instead of two, and an epilogue in which each thread
// finishes one token.  TMEM holds two accumulators of 256 columns, so the
// epilogue of one tile overlaps the MMAs of the next.
//
// This kernel runs INT8 and INT4 weights (FP8 weights run on the FP8 tensor
// cores, moe_prefill_a8.cu).  Weights stay INT8 / INT4 in HBM.  TMA brings raw
// weight tiles into shared memory; converter warps expand them to fp16 in
// registers and write the tcgen05 operand (K-major, 128-byte swizzle).  INT8
// weights convert exactly and the per-row x per-channel scales are applied in
// the epilogue; INT4 activations arrive as fp16 in power-of-two frames (x per
// row; h per row and 32 columns, brought to one frame per row by h_frame_kernel
// between the GEMMs), and the epilogues take the frames back in fp32.
// INT4 weights (two per byte, one scale per row and 128 columns) arrive as
// 32-byte rows per stage, expand to fp16 in the INT4 K order (pairs k0,k4 /
// k1,k5 / ...; the activations and h are stored in that order too) and take
// their row's group scale in the same fp16 multiply.
//
// Warp roles (15 warps, 1 CTA per SM, persistent; rings sized so that about a
// microsecond of loads is in flight):
//   warp 0      TMA producer of raw weight tiles        (ring of 4 stages)
//   warp 1      TMEM allocator + tcgen05.mma issuer
//   warp 2      TMA producer of activation tiles        (ring of 4 stages)
//   warps 3-10  converters: raw INT8 / INT4 -> fp16 swizzled operand (3 stages)
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
constexpr int MAXN = kPrefillTileTokens;  // tokens per tile (MMA N <= 128)
constexpr int RAW_STAGES = 4;          // raw weight codes (HBM -> smem by TMA)
constexpr int ACT_STAGES = 4;          // activation tiles (TMA)
constexpr int CONV_STAGES = 3;         // converted fp16 weight operands
constexpr int RAW_TILE = BM * BK;      // 8 KB of int8 codes per accumulator
constexpr int A_TILE = BM * BK * 2;    // 16 KB fp16 operand per accumulator
constexpr int B_TILE = MAXN * BK * 2;  // 16 KB fp16 activations
constexpr int N_CONV_WARPS = 8;
constexpr int N_EPI_WARPS = 4;
constexpr int WARP_WTMA = 0, WARP_MMA = 1, WARP_ATMA = 2, WARP_CONV0 = 3;
constexpr int WARP_EPI0 = WARP_CONV0 + N_CONV_WARPS;
constexpr int NUM_WARPS = WARP_EPI0 + N_EPI_WARPS;
constexpr int NUM_THREADS = NUM_WARPS * 32;
constexpr int CONV_THREADS = N_CONV_WARPS * 32;
constexpr uint32_t TMEM_COLS = 512;    // 2 buffers x 2 accumulators x 128 columns
constexpr int CHUNKS_PER_ACC = BM * BK / 16;  // 16-byte raw chunks per accumulator and stage
constexpr int RAW_TILE_I4 = BM * BK / 2;      // INT4: 4 KB of codes per accumulator and stage
constexpr int CHUNKS_PER_ACC_I4 = RAW_TILE_I4 / 16;

constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + CONV_STAGES * 2 * A_TILE;
constexpr int OFF_RAW = OFF_B + ACT_STAGES * B_TILE;
constexpr int OFF_BAR = OFF_RAW + RAW_STAGES * 2 * RAW_TILE;
constexpr int SMEM_BYTES = OFF_BAR + 512 + 1024;  // + slack to align the base to 1024
constexpr long long kWaitLimit = 4000000000LL;    // ~2 s of SM clocks per wait

struct Bars {
  uint64_t raw_full[RAW_STAGES];
  uint64_t raw_empty[RAW_STAGES];
  uint64_t act_full[ACT_STAGES];
  uint64_t act_empty[ACT_STAGES];
  uint64_t conv_full[CONV_STAGES];
  uint64_t conv_empty[CONV_STAGES];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 512, "barrier block too large");

struct Tile {
  int e, pos0, cnt, n0;
  bool two;  // second accumulator in use
};

// Tile t -> (token tile, output block).  GEMM1 (gated): block = 128 gate rows
// n0.. plus the up rows up_offset + n0..; GEMM2: block = rows n0.. and n0+128..
template <bool GATED>
__device__ __forceinline__ Tile get_tile(const PrefillArgs& p, int t) {
  const int tt = t / p.n_tiles;
  const int4 d = p.ttiles[tt];
  Tile r;
  r.e = d.x;
  r.pos0 = d.y;
  r.cnt = d.z;
  const int nt = t - tt * p.n_tiles;
  r.n0 = nt * (GATED ? BM : 2 * BM);
  r.two = GATED || (r.n0 + BM < p.rows_per_expert);
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
  static_assert(WK == MOE_WEIGHT_INT8 || WK == MOE_WEIGHT_INT4, "FP8 weights run on the FP8-operand kernels");
  constexpr bool I4 = WK == MOE_WEIGHT_INT4;
  constexpr int RAWB = I4 ? RAW_TILE_I4 : RAW_TILE;  // raw bytes per accumulator and stage
  const int KC = p.K / BK;
  const int second_rows = GATED ? p.up_offset : BM;  // row offset of the second accumulator's block

  if (threadIdx.x == 0) {
    for (int i = 0; i < RAW_STAGES; ++i) {
      mbar_init(&bars->raw_full[i], 1);
      mbar_init(&bars->raw_empty[i], N_CONV_WARPS);
    }
    for (int i = 0; i < ACT_STAGES; ++i) {
      mbar_init(&bars->act_full[i], 1);
      mbar_init(&bars->act_empty[i], 1);
    }
    for (int i = 0; i < CONV_STAGES; ++i) {
      mbar_init(&bars->conv_full[i], N_CONV_WARPS);
      mbar_init(&bars->conv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->acc_full[i], 1);
      mbar_init(&bars->acc_empty[i], N_EPI_WARPS);
    }
    mbar_init(&bars->mma_done, 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == WARP_MMA) {
    tmem_alloc(&bars->tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == WARP_WTMA && lane == 0) {
    prefetch_tmap(&tmap_w);
    prefetch_tmap(&tmap_b);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars->tmem_base;
  // GEMM2's weight stream (raw producer, converters, MMA) needs only the tile list, written
  // two kernels back; its activation producer and epilogue read GEMM1's output (h, h scales)
  // and wait for it.  GEMM1 waits in every role: with the masked layout it directly follows
  // the kernel that writes the tile list (and its trigger then comes after that wait).
  if (GATED || warp == WARP_ATMA || warp >= WARP_EPI0) pdl_wait();
  pdl_trigger();

  if (warp == WARP_WTMA) {
    // ---------------------------------------------------------------- raw weight producer
    // The whole warp walks the tiles; lane 0 waits for ring slots and issues the copies.
    int rs = 0;
    uint32_t rph = 0;
    int last_par[RAW_STAGES];
#pragma unroll
    for (int i = 0; i < RAW_STAGES; ++i) last_par[i] = -1;
    bool ok = true;
    for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
      const Tile tl = get_tile<GATED>(p, t);
      const int row0 = tl.e * p.rows_per_expert + tl.n0;
      for (int kc = 0; kc < KC; ++kc) {
        if (lane == 0) {
          ok = mbar_wait(&bars->raw_empty[rs], rph ^ 1, abort, p.status, kWaitLimit);
          if (ok) {
            mbar_arrive_expect_tx(&bars->raw_full[rs], (tl.two ? 2 : 1) * RAWB);
            uint8_t* dst = sRaw + rs * 2 * RAW_TILE;
            const int kx = I4 ? kc * (BK / 2) : kc * BK;  // K offset in bytes of the stored rows
            tma_load_2d(dst, &tmap_w, &bars->raw_full[rs], kx, row0);
            if (tl.two) tma_load_2d(dst + RAW_TILE, &tmap_w, &bars->raw_full[rs], kx, row0 + second_rows);
#pragma unroll
            for (int i = 0; i < RAW_STAGES; ++i)
              if (i == rs) last_par[i] = static_cast<int>(rph);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (++rs == RAW_STAGES) { rs = 0; rph ^= 1; }
      }
    }
    // never leave with copies in flight into this CTA's shared memory
    if (lane == 0) {
#pragma unroll
      for (int i = 0; i < RAW_STAGES; ++i)
        if (last_par[i] >= 0) {
          int dummy = 0;
          mbar_wait(&bars->raw_full[i], static_cast<uint32_t>(last_par[i]), &dummy, nullptr, kWaitLimit);
        }
    }
  } else if (warp == WARP_ATMA) {
    // ---------------------------------------------------------------- activation producer
    if (lane == 0) {
      int as = 0;
      uint32_t aph = 0;
      int last_par[ACT_STAGES];
#pragma unroll
      for (int i = 0; i < ACT_STAGES; ++i) last_par[i] = -1;
      bool ok = true;
      for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
        const Tile tl = get_tile<GATED>(p, t);
        for (int kc = 0; kc < KC; ++kc) {
          if (!(ok = mbar_wait(&bars->act_empty[as], aph ^ 1, abort, p.status, kWaitLimit))) break;
          // one 128-row box: rows past the tile's count (the next positions, or zero fill past the
          // tensor) only feed accumulator lanes or columns that no epilogue reads
          mbar_arrive_expect_tx(&bars->act_full[as], B_TILE);
          tma_load_2d(sB + as * B_TILE, &tmap_b, &bars->act_full[as], kc * BK, tl.pos0);
#pragma unroll
          for (int i = 0; i < ACT_STAGES; ++i)
            if (i == as) last_par[i] = static_cast<int>(aph);
          if (++as == ACT_STAGES) { as = 0; aph ^= 1; }
        }
      }
#pragma unroll
      for (int i = 0; i < ACT_STAGES; ++i)
        if (last_par[i] >= 0) {
          int dummy = 0;
          mbar_wait(&bars->act_full[i], static_cast<uint32_t>(last_par[i]), &dummy, nullptr, kWaitLimit);
        }
    }
  } else if (warp == WARP_MMA) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int as = 0, cs = 0;
      uint32_t aph = 0, cph = 0;
      uint32_t eph[2] = {0, 0};
      int buf = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
        const Tile tl = get_tile<GATED>(p, t);
        // M = 128 tokens, N = both weight blocks at once (256 rows; 128 when the second is absent)
        const uint32_t idesc = idesc_f16_f32(MAXN, tl.two ? 2 * BM : BM);
        const uint32_t d0 = tbase + static_cast<uint32_t>(buf * 2 * BM);
        if (!(ok = mbar_wait(&bars->acc_empty[buf], eph[buf] ^ 1, abort, p.status, kWaitLimit))) break;
        tc_fence_after();
        for (int kc = 0; kc < KC; ++kc) {
          if (!(ok = mbar_wait(&bars->conv_full[cs], cph, abort, p.status, kWaitLimit))) break;
          if (!(ok = mbar_wait(&bars->act_full[as], aph, abort, p.status, kWaitLimit))) break;
          tc_fence_after();
          const uint64_t xd = sw128_kmajor_desc(smem_addr(sB + as * B_TILE));       // tokens
          const uint64_t wd = sw128_kmajor_desc(smem_addr(sA + cs * 2 * A_TILE));  // converted weight blocks
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)  // +32 bytes along K per step; tokens (A, M side) x the two weight
            umma_f16(d0, xd + 2 * k, wd + 2 * k, idesc, (kc | k) != 0);  // blocks, adjacent (B, N side)
          umma_commit(&bars->conv_empty[cs]);
          umma_commit(&bars->act_empty[as]);
          if (++cs == CONV_STAGES) { cs = 0; cph ^= 1; }
          if (++as == ACT_STAGES) { as = 0; aph ^= 1; }
        }
        if (!ok) break;
        umma_commit(&bars->acc_full[buf]);
        eph[buf] ^= 1;
        buf ^= 1;
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
    for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
      const Tile tl = get_tile<GATED>(p, t);
      const int nchunks = (tl.two ? 2 : 1) * (I4 ? CHUNKS_PER_ACC_I4 : CHUNKS_PER_ACC);
      // INT4: this thread expands row ct/2 of each weight block in every stage; its group scales
      // (one per 128 K, i.e. per two stages) are loaded one group ahead
      const int i4row = ct >> 1;
      const float* i4s0 = p.wscale + (static_cast<size_t>(tl.e) * p.rows_per_expert + tl.n0 + i4row) * kblocks;
      const float* i4s1 = i4s0 + static_cast<size_t>(second_rows) * kblocks;
      float i4cur[2] = {0.f, 0.f}, i4nxt[2] = {0.f, 0.f};
      if constexpr (I4) {
        i4nxt[0] = __ldg(i4s0);
        i4nxt[1] = tl.two ? __ldg(i4s1) : 0.f;
      }
      for (int kc = 0; kc < KC; ++kc) {
        if constexpr (I4) {
          if ((kc & 1) == 0) {  // a new 128-wide group: take the prefetched scales, fetch the next ones
            i4cur[0] = i4nxt[0];
            i4cur[1] = i4nxt[1];
            const int g = kc / 2 + 1;
            if (g < kblocks) {
              i4nxt[0] = __ldg(i4s0 + g);
              i4nxt[1] = tl.two ? __ldg(i4s1 + g) : 0.f;
            }
          }
        }
        if (!(ok = mbar_wait(&bars->raw_full[rs], rph, abort, p.status, kWaitLimit))) break;
        if (!(ok = mbar_wait(&bars->conv_empty[cs], cph ^ 1, abort, p.status, kWaitLimit))) break;
        const uint8_t* raw = sRaw + rs * 2 * RAW_TILE;
        uint8_t* dstA = sA + cs * 2 * A_TILE;
        if constexpr (I4) {
          // a 16-byte chunk holds 32 K values of one row and expands to four 16-byte fp16 chunks
#pragma unroll
          for (int s = 0; s < 2 * CHUNKS_PER_ACC_I4 / CONV_THREADS; ++s) {
            const int j = ct + s * CONV_THREADS;
            if (j < nchunks) {
              const int acc = j / CHUNKS_PER_ACC_I4;
              const int idx = j - acc * CHUNKS_PER_ACC_I4;
              const int row = idx >> 1, c16 = idx & 1;  // row == i4row
              const uint4 v = *reinterpret_cast<const uint4*>(raw + acc * RAW_TILE + row * (BK / 2) + c16 * 16);
              uint32_t o[16];
              s4x8_to_f16x8(v.x, o);
              s4x8_to_f16x8(v.y, o + 4);
              s4x8_to_f16x8(v.z, o + 8);
              s4x8_to_f16x8(v.w, o + 12);
              const float s2 = i4cur[acc];
              const float m = fabsf(s2);
              if (m >= 6.103515625e-05f && m * 8.f <= 65504.f) {
                const __half2 sh2 = __half2half2(__float2half_rn(s2));
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  __half2 v2 = __hmul2(*reinterpret_cast<const __half2*>(&o[i]), sh2);
                  o[i] = *reinterpret_cast<uint32_t*>(&v2);
                }
              } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&o[i]));
                  o[i] = pack_half2(f.x * s2, f.y * s2);
                }
              }
              uint8_t* rowp = dstA + acc * A_TILE + row * 128;
              const int r8 = row & 7;
#pragma unroll
              for (int i = 0; i < 4; ++i)
                *reinterpret_cast<uint4*>(rowp + (((4 * c16 + i) ^ r8) << 4)) =
                    make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
            }
          }
        } else {
#pragma unroll
        for (int s = 0; s < 2 * CHUNKS_PER_ACC / CONV_THREADS; ++s) {
          const int j = ct + s * CONV_THREADS;  // 16-byte chunk of the raw stage
          if (j < nchunks) {
            const int acc = j / CHUNKS_PER_ACC;
            const int idx = j - acc * CHUNKS_PER_ACC;
            const int row = idx >> 2, c16 = idx & 3;
            const uint4 v = *reinterpret_cast<const uint4*>(raw + acc * RAW_TILE + row * BK + c16 * 16);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t o[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) w8x4_to_f16x4<WK>(w[i], o[2 * i], o[2 * i + 1]);  // INT8: exact
            // 128-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ (r % 8)
            uint8_t* rowp = dstA + acc * A_TILE + row * 128;
            const int r8 = row & 7;
            *reinterpret_cast<uint4*>(rowp + (((2 * c16) ^ r8) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(rowp + (((2 * c16 + 1) ^ r8) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
          }
        }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bars->conv_full[cs]);
          mbar_arrive(&bars->raw_empty[rs]);
        }
        if (++rs == RAW_STAGES) { rs = 0; rph ^= 1; }
        if (++cs == CONV_STAGES) { cs = 0; cph ^= 1; }
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    // TMEM lane = token: every thread finishes one token's outputs of the tile
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int tok = q * 32 + lane;
    uint32_t fph[2] = {0, 0};
    int buf = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
      const Tile tl = get_tile<GATED>(p, t);
      const bool live = tok < tl.cnt;
      const int pos = tl.pos0 + tok;
      if (!(ok = mbar_wait(&bars->acc_full[buf], fph[buf], abort, p.status, kWaitLimit))) break;
      tc_fence_after();
      const uint32_t lane_addr = tbase + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * 2 * BM);
      const float* chs = p.wscale + static_cast<size_t>(tl.e) * p.rows_per_expert;  // INT8 channel scales
      if constexpr (GATED && WK == MOE_WEIGHT_INT8) {
        float hmax = 0.f;
        const float sx = live ? __ldg(p.sx + __ldg(p.sorted_ids + pos) / p.topk) : 0.f;
        for (int c0 = 0; c0 < BM; c0 += 32) {  // gate columns c0.., up columns BM + c0..
          uint32_t g[32], u[32];
          tmem_ld32(lane_addr + c0, g);
          tmem_ld32(lane_addr + BM + c0, u);
          tmem_ld_wait();
          const int n = tl.n0 + c0;
          float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + static_cast<size_t>(pos) * p.out_ld + n);
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const float4 sg = __ldg(reinterpret_cast<const float4*>(chs + n) + v);
            const float4 su = __ldg(reinterpret_cast<const float4*>(chs + p.up_offset + n) + v);
            float h[4];
            const float sgv[4] = {sg.x, sg.y, sg.z, sg.w}, suv[4] = {su.x, su.y, su.z, su.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int j = 4 * v + i;
              h[i] = silu_f32(__uint_as_float(g[j]) * sx * sgv[i]) * (__uint_as_float(u[j]) * sx * suv[i]);
              hmax = fmaxf(hmax, fabsf(h[i]));
            }
            if (live) dst[v] = make_float4(h[0], h[1], h[2], h[3]);
          }
        }
        if (live) atomicMax(p.hmax + pos, __float_as_uint(hmax));
      } else if constexpr (GATED) {
        // INT4: h = SiLU(g) * u in fp32, with the token's x frame taken back; each 32 columns (one frame
        // block) stored in fp16 in their own frame.
        float gm = 0.f, um = 0.f;
        if (live) gm = um = __ldg(p.sx + (p.x_by_pos ? pos : __ldg(p.sorted_ids + pos) / p.topk));
        uint32_t emax = 0;
        for (int c0 = 0; c0 < BM; c0 += kHBlock) {  // gate columns c0.., up columns BM + c0..
          uint32_t g[32], u[32];
          tmem_ld32(lane_addr + c0, g);
          tmem_ld32(lane_addr + BM + c0, u);
          tmem_ld_wait();
          float m = 0.f;
#pragma unroll
          for (int j = 0; j < 32; ++j) {  // h in place of the gate values
            const float h = silu_f32(__uint_as_float(g[j]) * gm) * (__uint_as_float(u[j]) * um);
            g[j] = __float_as_uint(h);
            m = fmaxf(m, fabsf(h));
          }
          const uint32_t eb = static_cast<uint32_t>(h_frame_exp_biased(m));
          const float mb = eb ? exp2i(kExpBias - static_cast<int>(eb)) : 1.f;
          emax = eb > emax ? eb : emax;
          const int n = tl.n0 + c0;
          uint32_t hw[16];
          if constexpr (I4) {  // h feeds GEMM2's activations: INT4 K order within each 8 columns
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int a = 8 * (j >> 2) + (j & 3), b = a + 4;
              hw[j] = pack_half2(__uint_as_float(g[a]) * mb, __uint_as_float(g[b]) * mb);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) hw[j] = pack_half2(__uint_as_float(g[2 * j]) * mb, __uint_as_float(g[2 * j + 1]) * mb);
          }
          if (live) {
            p.hblk[static_cast<size_t>(pos) * (p.out_ld / kHBlock) + n / kHBlock] = static_cast<uint8_t>(eb);
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__half*>(p.out) + static_cast<size_t>(pos) * p.out_ld + n);
#pragma unroll
            for (int v = 0; v < 4; ++v) dst[v] = make_uint4(hw[4 * v], hw[4 * v + 1], hw[4 * v + 2], hw[4 * v + 3]);
          }
        }
        if (live && emax) atomicMax(p.hexp + pos, emax);
      } else {
        int slot = 0;
        float wgt = 0.f;
        if (live) {
          slot = __ldg(p.sorted_ids + pos);
          wgt = p.out_bf16 ? 1.f : __ldg(p.topk_w + slot);  // masked layout: unweighted bf16 rows
          if constexpr (WK == MOE_WEIGHT_INT8) wgt *= __ldg(p.sh + pos);
          else wgt *= __ldg(p.hsc + pos);  // h's row frame
        }
#pragma unroll 1
        for (int c0 = 0; c0 < (tl.two ? 2 * BM : BM); c0 += 32) {  // output rows n0 + c0..
          uint32_t g[32];
          tmem_ld32(lane_addr + c0, g);
          tmem_ld_wait();
          const int n = tl.n0 + c0;
          __nv_bfloat16* yb = p.out_bf16 ? p.out_bf16 : static_cast<__nv_bfloat16*>(p.out);
          uint4* dstb = reinterpret_cast<uint4*>(yb + static_cast<size_t>(slot) * p.out_ld + n);
#pragma unroll
          for (int v = 0; v < 4; ++v) {  // 8 columns, one 16-byte store
            uint32_t w[4];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int q = 2 * v + h;
              float4 sc = make_float4(wgt, wgt, wgt, wgt);
              if constexpr (WK == MOE_WEIGHT_INT8) {
                const float4 cs = __ldg(reinterpret_cast<const float4*>(chs + n) + q);
                sc = make_float4(wgt * cs.x, wgt * cs.y, wgt * cs.z, wgt * cs.w);
              }
              const __nv_bfloat162 lo = __floats2bfloat162_rn(__uint_as_float(g[4 * q]) * sc.x,
                                                              __uint_as_float(g[4 * q + 1]) * sc.y);
              const __nv_bfloat162 hi = __floats2bfloat162_rn(__uint_as_float(g[4 * q + 2]) * sc.z,
                                                              __uint_as_float(g[4 * q + 3]) * sc.w);
              w[2 * h] = *reinterpret_cast<const uint32_t*>(&lo);
              w[2 * h + 1] = *reinterpret_cast<const uint32_t*>(&hi);
            }
            if (live) dstb[v] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->acc_empty[buf]);
      fph[buf] ^= 1;
      buf ^= 1;
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
  pdl_wait();
  pdl_trigger();
  // one warp per position, its lanes over the row's 16-byte chunks
  const int rows = *num_post;
  const int chunks = H / 8, lane = threadIdx.x & 31;
  const int nw = gridDim.x * (blockDim.x >> 5);
  for (int pos = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); pos < rows; pos += nw) {
    const int slot = __ldg(sorted_ids + pos);
    const bool valid = slot < n_slots;
    const uint4* src = reinterpret_cast<const uint4*>(xq + static_cast<size_t>(valid ? slot / topk : 0) * H);
    uint4* dst = reinterpret_cast<uint4*>(act + static_cast<size_t>(pos) * H);
#pragma unroll 4
    for (int c = lane; c < chunks; c += 32) dst[c] = valid ? ld_v4(src + c) : make_uint4(0u, 0u, 0u, 0u);
  }
}

// The intermediate's row frames (INT4 weights on this path): GEMM1 stored every 32-column
// block of h in its own power-of-two frame; the down projection needs one frame per row, the
// largest.  Blocks stored lower are scaled down to it in place (rare: a block's frame exponent is
// a multiple of 8, so the blocks of a row mostly share it), and hsc[pos] = 2^e of the row frame.
// One warp per position, lanes over its blocks.
__global__ void __launch_bounds__(256) h_frame_kernel(__half* __restrict__ h, const uint32_t* __restrict__ hexp,
                                                      const uint8_t* __restrict__ hblk,
                                                      const int32_t* __restrict__ num_post, int I,
                                                      float* __restrict__ hsc) {
  pdl_wait();
  pdl_trigger();
  const int rows = *num_post, nb = I / kHBlock, lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  for (int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += nwarps) {
    const uint32_t ef = hexp[r];  // 0: no nonzero block (a padding row or an all-zero h)
    if (lane == 0) hsc[r] = ef ? exp2i(static_cast<int>(ef) - kExpBias) : 1.f;
    if (!ef) continue;
    for (int b = lane; b < nb; b += 32) {
      const uint32_t eb = hblk[static_cast<size_t>(r) * nb + b];
      if (eb == 0u || eb == ef) continue;
      const __half2 f = exp2i_h2(static_cast<int>(eb) - static_cast<int>(ef));
      uint4* q = reinterpret_cast<uint4*>(h + static_cast<size_t>(r) * I + b * kHBlock);
#pragma unroll
      for (int i = 0; i < kHBlock / 8; ++i) {
        uint4 v = q[i];
        scale_h8(v, f);
        q[i] = v;
      }
    }
  }
}

cudaError_t launch_h_frame(__half* h, const uint32_t* hexp, const uint8_t* hblk, const int32_t* num_post, int cap,
                           int I, float* hsc, int num_sms, cudaStream_t s) {
  int grid = (cap + 7) / 8;
  if (grid > num_sms * 4) grid = num_sms * 4;
  if (grid < 1) grid = 1;
  return launch_kernel(h_frame_kernel, dim3(grid), dim3(256), 0, s, true, h, hexp, hblk, num_post, I, hsc);
}

// out[t, n] = sum over k (in slot order) of y[t*topk + k, n] for the slots that were routed
// (inv_pos >= 0); y already carries the routing weight.
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y, const int32_t* __restrict__ inv_pos,
                                                      int M, int topk, int H, __nv_bfloat16* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int q = H / 4;
  const long long total = static_cast<long long>(M) * q;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / q), c = static_cast<int>(i - static_cast<long long>(t) * q);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k0 = 0; k0 < topk; k0 += 8) {
      float4 v[8];  // all loads of a group in flight together, then summed in slot order
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int k = k0 + j, slot = t * topk + k;
        v[j] = (k < topk && __ldg(inv_pos + slot) >= 0)
                   ? __ldg(reinterpret_cast<const float4*>(y + static_cast<size_t>(slot) * H) + c)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        acc.x += v[j].x; acc.y += v[j].y; acc.z += v[j].z; acc.w += v[j].w;
      }
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 pk = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
    *reinterpret_cast<uint2*>(out + static_cast<size_t>(t) * H + 4 * c) = pk;
  }
}

// The same sum over bf16 y rows (the tcgen05 path), eight columns per lane: a warp per (token, 32 chunks),
// so that the token's routed slots are read once, as a ballot (topk <= 32), and no thread divides per chunk.
__global__ void __launch_bounds__(256) combine_bf16_kernel(const __nv_bfloat16* __restrict__ y,
                                                           const int32_t* __restrict__ inv_pos, int M, int topk, int H,
                                                           __nv_bfloat16* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int q = H / 8, lane = threadIdx.x & 31, nseg = (q + 31) / 32;
  const long long nw = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long it = blockIdx.x * static_cast<long long>(blockDim.x >> 5) + (threadIdx.x >> 5);
       it < static_cast<long long>(M) * nseg; it += nw) {
    const int t = static_cast<int>(it / nseg), c = static_cast<int>(it - static_cast<long long>(t) * nseg) * 32 + lane;
    const unsigned routed = __ballot_sync(0xffffffffu, lane < topk && __ldg(inv_pos + t * topk + lane) >= 0);
    const uint4* yt = reinterpret_cast<const uint4*>(y + static_cast<size_t>(t) * topk * H);
    if (c < q) {
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int k0 = 0; k0 < topk; k0 += 8) {
        uint4 v[8];  // all loads of a group in flight together, then summed in slot order
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int k = k0 + j;
          v[j] = (k < topk && ((routed >> k) & 1u)) ? __ldg(yt + static_cast<size_t>(k) * q + c)
                                                    : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[u]));
            acc[2 * u] += f.x;
            acc[2 * u + 1] += f.y;
          }
        }
      }
      uint32_t o[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * u], acc[2 * u + 1]);
        o[u] = *reinterpret_cast<const uint32_t*>(&b);
      }
      *reinterpret_cast<uint4*>(out + static_cast<size_t>(t) * H + 8 * c) = make_uint4(o[0], o[1], o[2], o[3]);
    }
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

bool encode_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, uint64_t inner,
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
  constexpr bool I4 = WK == MOE_WEIGHT_INT4;  // rows of K/2 bytes, 32 of them per stage
  if (!encode_tmap_2d(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, w, static_cast<uint64_t>(I4 ? a.K / 2 : a.K), w_rows,
                      I4 ? pf::BK / 2 : pf::BK, pf::BM, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  if (!encode_tmap_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, b, static_cast<uint64_t>(a.K), b_rows, pf::BK, pf::MAXN,
                CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  auto kern = pf::prefill_gemm_kernel<WK, GATED>;
  cudaError_t err = set_smem_limit_once(reinterpret_cast<const void*>(kern), pf::SMEM_BYTES);
  if (err != cudaSuccess) return err;
  return launch_kernel(kern, dim3(num_sms), dim3(pf::NUM_THREADS), pf::SMEM_BYTES, s, true, mw, mb, a);
}

cudaError_t launch_prefill(const LayerPlan& P, int weight_kind, int num_sms, cudaStream_t s, const StageHook& hook) {
  if (weight_kind != MOE_WEIGHT_INT8 && weight_kind != MOE_WEIGHT_INT4) return cudaErrorInvalidValue;  // (FP8: a8)
  cudaError_t err;
  if (!P.out_direct) {  // (the masked layout's prologue already wrote the rows in position order)
    int grid = num_sms * 8;
    err = launch_kernel(gather_rows_kernel, dim3(grid), dim3(256), 0, s, true, P.xq, P.sorted_ids, P.num_post,
                        P.M * P.topk, P.topk, P.H, P.act);
    if (err != cudaSuccess) return err;
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
  g1.x_by_pos = P.x_by_pos ? 1 : 0;
  g1.hexp = P.hexp;
  g1.hblk = P.hblk;
  const uint64_t rows1 = static_cast<uint64_t>(P.E) * 2 * P.I;
  err = weight_kind == MOE_WEIGHT_INT4 ? launch_gemm<MOE_WEIGHT_INT4, true>(g1, P.w13, rows1, P.act, P.cap, num_sms, s)
                                       : launch_gemm<MOE_WEIGHT_INT8, true>(g1, P.w13, rows1, P.act, P.cap, num_sms, s);
  if (err != cudaSuccess) return err;
  hook("prefill_gemm1", s);
  const __half* b2 = reinterpret_cast<const __half*>(P.h);
  if (weight_kind == MOE_WEIGHT_INT8) {
    // padded positions: the slots plus at most B - 1 padding rows for each of at most min(E, slots) experts
    const long long slots = static_cast<long long>(P.M) * P.topk;
    const long long rows = slots + (slots < P.E ? slots : P.E) * (kPrefillBlock - 1);
    err = launch_requant_rows(P.h, P.hmax, P.num_post, rows < P.cap ? static_cast<int>(rows) : P.cap, P.I, P.hq,
                              P.sh, num_sms, s);
    if (err != cudaSuccess) return err;
    hook("requant_h", s);
    b2 = P.hq;
  } else {
    err = launch_h_frame(static_cast<__half*>(P.h), P.hexp, P.hblk, P.num_post, P.cap, P.I, P.hsc, num_sms, s);
    if (err != cudaSuccess) return err;
    hook("h_frame", s);
  }
  PrefillArgs g2{};
  g2.K = P.I;
  g2.rows_per_expert = P.H;
  g2.up_offset = 0;
  g2.n_tiles = (P.H + 2 * pf::BM - 1) / (2 * pf::BM);
  g2.ttiles = P.ttiles;
  g2.num_ttiles = P.num_ttiles;
  g2.wscale = P.s2;
  g2.sorted_ids = P.sorted_ids;
  g2.topk = P.topk;
  g2.sh = P.sh;
  g2.hsc = P.hsc;
  g2.topk_w = P.topk_w;
  g2.out = P.y;
  g2.out_ld = P.H;
  g2.status = P.status;
  g2.out_bf16 = P.out_direct;
  const uint64_t rows2 = static_cast<uint64_t>(P.E) * P.H;
  err = weight_kind == MOE_WEIGHT_INT4 ? launch_gemm<MOE_WEIGHT_INT4, false>(g2, P.w2, rows2, b2, P.cap, num_sms, s)
                                       : launch_gemm<MOE_WEIGHT_INT8, false>(g2, P.w2, rows2, b2, P.cap, num_sms, s);
  if (err != cudaSuccess) return err;
  hook("prefill_gemm2", s);
  if (P.out_direct) return cudaSuccess;  // masked layout: GEMM2 wrote the output rows
  err = launch_combine(reinterpret_cast<const __nv_bfloat16*>(P.y), P.inv_pos, P.M, P.topk, P.H, P.out, num_sms, s);
  if (err != cudaSuccess) return err;
  hook("combine", s);
  return cudaSuccess;
}

cudaError_t launch_combine(const float* y, const int32_t* inv_pos, int M, int topk, int H, __nv_bfloat16* out,
                           int num_sms, cudaStream_t s) {
  const long long work = static_cast<long long>(M) * (H / 4);
  long long grid = (work + 255) / 256;
  if (grid > num_sms * 16) grid = num_sms * 16;
  if (grid < 1) grid = 1;
  return launch_kernel(combine_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, s, true, y, inv_pos, M, topk,
                       H, out);
}

cudaError_t launch_combine(const __nv_bfloat16* y, const int32_t* inv_pos, int M, int topk, int H,
                           __nv_bfloat16* out, int num_sms, cudaStream_t s) {
  const long long warps = static_cast<long long>(M) * ((H / 8 + 31) / 32);
  long long grid = (warps + 7) / 8;
  if (grid > num_sms * 16) grid = num_sms * 16;
  if (grid < 1) grid = 1;
  return launch_kernel(combine_bf16_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, s, true, y, inv_pos, M,
                       topk, H, out);
}

size_t prefill_smem_bytes() { return pf::SMEM_BYTES; }

}  // namespace gbmoe
