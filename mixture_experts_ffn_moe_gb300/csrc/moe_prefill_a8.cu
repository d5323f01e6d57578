// Prefill path with FP8 activations ("A8": E4M3 codes in 1 x 128 groups, one
// fp32 scale per token and 128 columns): FP8 x FP8 grouped GEMMs on tcgen05
// tensor cores (kind::f8f6f4).
//
// The pages run their FP8 weights against BF16 activations (Xeon 6 / SGLang
// blog, section "FP8 推理"); this mode is the FP8 x FP8 form of the grouped
// GEMMs that the news rewrite of the LMSYS large-scale-EP blog integrates
// (section "DeepGEMM集成"), offered next to the weight-only path because at
// large token counts the layer is bound by tensor-core throughput, and FP8 x FP8
// runs at twice the fp16 rate with half the operand bytes.
//
// A tile is a token tile of one expert (up to 128 sorted slots) against two
// 128-row weight blocks.  Tokens are the MMA's M side (TMEM lane = token) and
// the weight rows its N side, so every thread owns one token.  Both operands
// stay E4M3 in shared memory: TMA writes them in the 128-byte swizzled K-major
// layout the MMA reads, so nothing is converted.
//
// Block scales.  A K block of 128 is one scale block of the weights and one
// scale group of the activations.  Its partial sums P go to TMEM, and the
// accumulator warps fold them into fp32 registers:
//   acc[token, row] += P[token, row] * a_scale(token, K block) * w_scale(row block, K block)
// (the post-scaling of the OSDI'26 local-MoE summary, section "CPU 解码后端").
// Within a tile the factor is one scalar per (token, weight block), so a thread
// needs two factors per K block.  TMEM holds the partials of two K blocks
// (2 buffers x 2 accumulators x 128 columns), so the MMAs of one K block
// overlap the promotion of the previous one.  One commit per K block frees the
// operand stage and hands the partials over; the accumulator warps give the
// TMEM buffer back as soon as its last partials are in registers.
//
// The weight-only layer runs on the same kernels with NT = 2: its bf16 x and fp32
// h enter as two E4M3 terms (hi and lo codes in a power-of-two frame per 128
// columns), whose two products accumulate into the same partial sums.
//
// Warp roles (12 warps = 3 warpgroups, 1 CTA per SM, persistent):
//   warp 0      TMA producer of weight tiles (2 x 16 KB per K block, ring of 4 in GEMM1, 3 in GEMM2 and with NT = 2)
//   warp 1      TMEM allocator + tcgen05.mma issuer
//   warp 2      TMA producer of activation tiles (per term one box of 32, 64 or 128 rows of 128 bytes) and
//               activation scale vectors (ring of 8)
//   warp 3      scale warp: per K block, the factor vectors a_scale x w_scale of both accumulators
//   warps 4-11  accumulators (setmaxnreg: 224 registers, the first warpgroup gives up its share)
//               promotion, then the epilogue of the tile:
//                 GEMM1: h = SiLU(gate) * up, quantised to E4M3 per 1 x 128 group (the tile's
//                        128 rows are one group of I) -> h codes [cap, I] and scales [I/128, cap]
//                 GEMM2: y[slot] = acc * routing weight in bf16, staged through shared memory so
//                        that every store instruction writes whole 128-byte row segments
// Every wait is bounded; a time-out sets the status flag and every role drains.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace gbmoe {
namespace pfa8 {

using namespace sm100;

constexpr int BK = 128;                  // K per stage: one 128-deep scale block (bytes of E4M3)
constexpr int BM = 128;                  // weight rows per accumulator (MMA N)
constexpr int MAXN = kPrefillTileTokens; // tokens per tile (MMA M = 128)
constexpr int MAX_STAGES = 4;            // K-block stages of the weight and activation rings (they advance together)
constexpr int S_STAGES = 8;              // deeper than the stages + the 2 TMEM buffers the MMA may lead by
constexpr int W_TILE = BM * BK;          // 16 KB per accumulator
constexpr int A_TILE = MAXN * BK;        // 16 KB
constexpr int S_SLOT = 3 * MAXN * 4;     // activation scales, factors of accumulator 0, factors of accumulator 1
constexpr int N_ACC_WARPS = 8;
constexpr int WARP_WTMA = 0, WARP_MMA = 1, WARP_ATMA = 2, WARP_SCALE = 3, WARP_ACC0 = 4;
constexpr int NUM_WARPS = WARP_ACC0 + N_ACC_WARPS;
constexpr int NUM_THREADS = NUM_WARPS * 32;
constexpr int REGS_AT_LAUNCH = 65536 / NUM_THREADS / 8 * 8;  // what __launch_bounds__(NUM_THREADS, 1) allows
constexpr int REGS_SUPPORT = 56;         // warpgroup 0
constexpr int REGS_ACC = 224;            // warpgroups 1 and 2
static_assert(128 * REGS_SUPPORT + 256 * REGS_ACC <= NUM_THREADS * REGS_AT_LAUNCH, "register split exceeds the pool");
constexpr uint32_t TMEM_COLS = 512;      // 2 buffers x 2 accumulators x 128 columns

constexpr int RED_BYTES = 2 * 2 * MAXN * 4;  // [tile parity][column half][token] floats

// Shared-memory layout per GEMM (measured): GEMM1 keeps 4 K-block stages; GEMM2, whose short
// K loop (I = 2048) makes its y stores a large share of the tile, trades one stage for a
// 4 KB y staging buffer per accumulator warp (64 bf16 columns, 128-byte row segments).
// NT = 2 (two activation terms per value) doubles the activation tiles of a stage: both GEMMs then
// keep 3 stages, and GEMM2 stages 32 columns of y at a time (2 KB per accumulator warp).
template <bool GATED, int NT>
struct Lay {
  static constexpr int STAGES = NT == 1 ? (GATED ? 4 : 3) : 3;
  static constexpr int STG_COLS = NT == 1 ? 64 : 32;                // y columns staged per pass
  static constexpr int STG_BYTES = GATED ? 0 : 32 * STG_COLS * 2;    // per accumulator warp: 32 tokens
  static constexpr int OFF_W = 0;
  static constexpr int OFF_A = OFF_W + STAGES * 2 * W_TILE;
  static constexpr int OFF_S = OFF_A + STAGES * NT * A_TILE;
  static constexpr int OFF_RED = OFF_S + S_STAGES * S_SLOT;
  static constexpr int OFF_STG = OFF_RED + RED_BYTES;
  static constexpr int OFF_BAR = OFF_STG + N_ACC_WARPS * STG_BYTES;
  static constexpr int SMEM_BYTES = OFF_BAR + 512 + 1024;  // + slack to align the base to 1024
  static_assert(STAGES <= MAX_STAGES && SMEM_BYTES <= 232448, "shared memory per CTA");
  static_assert(STAGES >= 3, "the accumulator warps wait on the stage barriers: more stages than TMEM buffers");
};
constexpr long long kWaitLimit = 4000000000LL;    // ~2 s of SM clocks per wait

struct Bars {
  uint64_t op_full[MAX_STAGES];   // weight and activation stages of a K block landed (TMA, two producers)
  uint64_t st_empty[MAX_STAGES];  // the MMAs of a K block are done: its stages are free, its partials in TMEM
  uint64_t s_full[S_STAGES];   // activation scale vector landed (TMA)
  uint64_t f_full[S_STAGES];   // factor vectors written (scale warp)
  uint64_t s_empty[S_STAGES];  // factor vectors consumed (accumulator warps)
  uint64_t p_empty[2];         // the accumulator warps have read a TMEM buffer
  uint64_t red_full[2][4];     // [tile parity][lane quarter]: both column halves wrote their token maxima
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 512, "barrier block too large");

struct Args {
  int K;                 // H (GEMM1) or I (GEMM2)
  int rows_per_expert;   // 2I (GEMM1) or H (GEMM2)
  int second_rows;       // row offset of the second accumulator's block: I (GEMM1) or 128 (GEMM2)
  int n_tiles;           // output tiles per token tile
  int n_rows_out;        // GEMM1: I (leading dimension of h codes); GEMM2: H (of y)
  int cap;               // positions (leading dimension of the h scale rows)
  const int4* ttiles;
  const int32_t* num_ttiles;
  const float* wscale;   // [E, rows/128, K/128]
  const int32_t* sorted_ids;
  const float* topk_w;   // GEMM2
  uint8_t* hq;           // GEMM1 out: h codes [cap, I]
  float* hs;             // GEMM1 out: h scales [I/128, cap]
  __nv_bfloat16* y;      // GEMM2 out: [M*topk, H]
  DeviceStatus* status;
  int tiles_from_prev;   // the tile list comes from the kernel right before this one
};

struct Tile {
  int e, pos0, cnt, n0;
  bool two;
};

template <bool GATED>
__device__ __forceinline__ Tile get_tile(const Args& p, int t) {
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

__device__ __forceinline__ float elem(const float2* a, int j) { return (j & 1) ? a[j >> 1].y : a[j >> 1].x; }

// Waits (bounded) for the last min(seq, stages) fills of a ring to land: a
// producer must not exit with copies in flight into shared memory.  Fill i
// went to slot i % stages with phase parity (i / stages) & 1.
__device__ __forceinline__ void drain_ring(uint64_t* full, int stages, long long seq) {
  const long long n = seq < stages ? seq : stages;
  for (long long i = seq - n; i < seq; ++i) {
    int dummy = 0;
    mbar_wait(&full[i % stages], static_cast<uint32_t>((i / stages) & 1), &dummy, nullptr, kWaitLimit);
  }
}

// NT: activation terms per value -- 1: E4M3 activations (MOE_ACT_FP8_1X128); 2: the two-term E4M3 form
// of the weight-only layer's bf16 x and fp32 h (hi codes in rows 0..cap-1 of the activation tensor, lo
// codes in rows cap..2cap-1), whose two products accumulate into one partial sum.
template <bool GATED, int NT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    prefill_a8_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_b,
                      const __grid_constant__ CUtensorMap tmap_b32, const __grid_constant__ CUtensorMap tmap_b64,
                      const __grid_constant__ CUtensorMap tmap_s, Args p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  using L = Lay<GATED, NT>;
  constexpr int W_STAGES = L::STAGES, A_STAGES = L::STAGES;
  uint8_t* sW = smem + L::OFF_W;
  uint8_t* sA = smem + L::OFF_A;
  float* sS = reinterpret_cast<float*>(smem + L::OFF_S);
  float* red = reinterpret_cast<float*>(smem + L::OFF_RED);
  Bars* bars = reinterpret_cast<Bars*>(smem + L::OFF_BAR);
  volatile int* abort = &bars->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KC = p.K / BK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < W_STAGES; ++i) {
      mbar_init(&bars->op_full[i], 2);  // both producers arrive: weights and activations of a K block
      mbar_init(&bars->st_empty[i], 1);
    }
    for (int i = 0; i < S_STAGES; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->f_full[i], 1);
      mbar_init(&bars->s_empty[i], N_ACC_WARPS);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->p_empty[i], N_ACC_WARPS);
      for (int j = 0; j < 4; ++j) mbar_init(&bars->red_full[i][j], 64);
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
    prefetch_tmap(&tmap_b32);
    prefetch_tmap(&tmap_b64);
    prefetch_tmap(&tmap_s);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars->tmem_base;
  // The weight stream and the MMA issuer need only the tile list, written two
  // kernels back on the routed layer, so they start at once; the activation
  // producer, the scale warp and the accumulators read the predecessor's output
  // and wait for it.  When the predecessor itself wrote the tile list (GEMM1
  // of the masked layout, right after its prologue), every role waits.
  if (p.tiles_from_prev || warp == WARP_ATMA || warp >= WARP_SCALE) pdl_wait();
  pdl_trigger();
  const int total_tiles = *p.num_ttiles * p.n_tiles;
  if (warp < WARP_ACC0) {
    // ================================================================ support warpgroup
    regs_dec<REGS_SUPPORT>();
    if (warp == WARP_WTMA) {
      // ---------------------------------------------------------------- weight producer
      if (lane == 0) {
        int ws = 0;
        uint32_t wph = 0;
        long long seq = 0;  // stages issued
        bool ok = true;
        for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
          const Tile tl = get_tile<GATED>(p, t);
          const int row0 = tl.e * p.rows_per_expert + tl.n0;
          for (int kc = 0; kc < KC; ++kc) {
            if (!(ok = mbar_wait(&bars->st_empty[ws], wph ^ 1, abort, p.status, kWaitLimit))) break;
            mbar_arrive_expect_tx(&bars->op_full[ws], (tl.two ? 2 : 1) * W_TILE);
            uint8_t* dst = sW + ws * 2 * W_TILE;
            tma_load_2d(dst, &tmap_w, &bars->op_full[ws], kc * BK, row0);
            if (tl.two) tma_load_2d(dst + W_TILE, &tmap_w, &bars->op_full[ws], kc * BK, row0 + p.second_rows);
            ++seq;
            if (++ws == W_STAGES) { ws = 0; wph ^= 1; }
          }
        }
        drain_ring(bars->op_full, W_STAGES, seq);  // never leave with copies in flight into shared memory
      }
    } else if (warp == WARP_ATMA) {
      // ---------------------------------------------------------------- activation + scale producer
      if (lane == 0) {
        int as = 0, ss = 0;
        uint32_t aph = 0, sph = 0;
        long long aseq = 0, sseq = 0;  // stages issued
        bool ok = true;
        for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
          const Tile tl = get_tile<GATED>(p, t);
          for (int kc = 0; kc < KC; ++kc) {
            if (!(ok = mbar_wait(&bars->st_empty[as], aph ^ 1, abort, p.status, kWaitLimit))) break;
            // one box per term of the first 32, 64 or 128 rows, whichever holds the tile's tokens: the MMA
            // always reads 128 token rows, and the rows past the tile's count (the next positions, zero fill
            // past the tensor, or rows a smaller box left as they were) only feed TMEM lanes nobody reads
            const int arows = tl.cnt <= 32 ? 32 : tl.cnt <= 64 ? 64 : MAXN;
            const CUtensorMap* amap = arows == 32 ? &tmap_b32 : arows == 64 ? &tmap_b64 : &tmap_b;
            mbar_arrive_expect_tx(&bars->op_full[as], NT * arows * BK);
            uint8_t* dst = sA + as * NT * A_TILE;
#pragma unroll
            for (int term = 0; term < NT; ++term)  // the lo codes of a position sit cap rows below its hi codes
              tma_load_2d(dst + term * A_TILE, amap, &bars->op_full[as], kc * BK, term * p.cap + tl.pos0);
            ++aseq;
            if (++as == A_STAGES) { as = 0; aph ^= 1; }

            if (!(ok = mbar_wait(&bars->s_empty[ss], sph ^ 1, abort, p.status, kWaitLimit))) break;
            mbar_arrive_expect_tx(&bars->s_full[ss], MAXN * 4);
            tma_load_2d(sS + ss * (S_SLOT / 4), &tmap_s, &bars->s_full[ss], tl.pos0, kc);
            ++sseq;
            if (++ss == S_STAGES) { ss = 0; sph ^= 1; }
          }
        }
        drain_ring(bars->op_full, A_STAGES, aseq);
        drain_ring(bars->s_full, S_STAGES, sseq);
      }
    } else if (warp == WARP_MMA) {
      // ---------------------------------------------------------------- MMA issuer
      if (lane == 0) {
        int ws = 0, as = 0, buf = 0;
        uint32_t wph = 0;
        uint32_t eph[2] = {0, 0};
        bool ok = true;
        for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
          const Tile tl = get_tile<GATED>(p, t);
          const uint32_t idesc = idesc_e4m3_f32(MAXN, BM);  // M = 128 tokens, N = 128 weight rows
          for (int kc = 0; kc < KC; ++kc) {
            if (!(ok = mbar_wait(&bars->p_empty[buf], eph[buf] ^ 1, abort, p.status, kWaitLimit))) break;
            if (!(ok = mbar_wait(&bars->op_full[ws], wph, abort, p.status, kWaitLimit))) break;
            tc_fence_after();
            const uint32_t d0 = tbase + static_cast<uint32_t>(buf * 2 * BM);
            uint64_t ad[NT];  // tokens: one tile per activation term
#pragma unroll
            for (int term = 0; term < NT; ++term)
              ad[term] = sw128_kmajor_desc(smem_addr(sA + (as * NT + term) * A_TILE));
            const uint64_t b0 = sw128_kmajor_desc(smem_addr(sW + ws * 2 * W_TILE));        // weight block 0
            const uint64_t b1 = sw128_kmajor_desc(smem_addr(sW + ws * 2 * W_TILE + W_TILE));  // block 1
#pragma unroll
            for (int k = 0; k < BK / 32; ++k) {  // 32 bytes (K = 32) per instruction: +2 in the encoded address
#pragma unroll
              for (int term = 0; term < NT; ++term) {  // every term of the tokens into the same partial sum
                umma_e4m3(d0, ad[term] + 2 * k, b0 + 2 * k, idesc, (k | term) != 0);
                if (tl.two) umma_e4m3(d0 + BM, ad[term] + 2 * k, b1 + 2 * k, idesc, (k | term) != 0);
              }
            }
            // one commit per K block (== as: both rings advance one stage per K block): it frees the stage and
            // tells the accumulator warps that the partial sums are in TMEM buffer `buf`
            umma_commit(&bars->st_empty[ws]);
            eph[buf] ^= 1;
            buf ^= 1;
            if (++ws == W_STAGES) { ws = 0; wph ^= 1; }
            if (++as == A_STAGES) as = 0;
          }
        }
        // every issued MMA must finish before TMEM is released
        umma_commit(&bars->mma_done);
        int dummy = 0;
        mbar_wait(&bars->mma_done, 0, &dummy, nullptr, kWaitLimit);
      }
    } else if (warp == WARP_SCALE) {
      // ---------------------------------------------------------------- scale warp
      const int kblocks = p.K / kQBlock, rblocks = p.rows_per_expert / kQBlock;
      int ss = 0;
      uint32_t sph = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
        const Tile tl = get_tile<GATED>(p, t);
        const float* w0 = p.wscale + (static_cast<size_t>(tl.e) * rblocks + tl.n0 / kQBlock) * kblocks;
        const float* w1 = p.wscale + (static_cast<size_t>(tl.e) * rblocks + (tl.n0 + p.second_rows) / kQBlock) * kblocks;
        // weight block scales of 64 K blocks at a time, one load per lane (K block kc sits
        // in lane kc % 32 of register kc / 32 % 2): the latency is paid once per 64 K blocks
        float w0r[2] = {0.f, 0.f}, w1r[2] = {0.f, 0.f};
        for (int kc = 0; kc < KC; ++kc) {
          if ((kc & 63) == 0) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int k = kc + h * 32 + lane;
              w0r[h] = k < KC ? __ldg(w0 + k) : 0.f;
              w1r[h] = (k < KC && tl.two) ? __ldg(w1 + k) : 0.f;
            }
          }
          const int hsel = (kc >> 5) & 1;
          const float s0 = __shfl_sync(0xffffffffu, hsel ? w0r[1] : w0r[0], kc & 31);
          const float s1 = __shfl_sync(0xffffffffu, hsel ? w1r[1] : w1r[0], kc & 31);
          if (!(ok = mbar_wait(&bars->s_full[ss], sph, abort, p.status, kWaitLimit))) break;
          float* slot = sS + ss * (S_SLOT / 4);
          const float4 a = reinterpret_cast<const float4*>(slot)[lane];
          reinterpret_cast<float4*>(slot + MAXN)[lane] = make_float4(a.x * s0, a.y * s0, a.z * s0, a.w * s0);
          reinterpret_cast<float4*>(slot + 2 * MAXN)[lane] = make_float4(a.x * s1, a.y * s1, a.z * s1, a.w * s1);
          // the scale vector was read by generic loads; order them before its next TMA refill
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->f_full[ss]);
          if (++ss == S_STAGES) { ss = 0; sph ^= 1; }
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- accumulators
    regs_inc<REGS_ACC>();
    const int q = warp & 3;                     // TMEM lane quarter this warp may access
    const int ch = (warp - WARP_ACC0) >> 2;     // column half: outputs 64*ch .. 64*ch+63 of each block
    const int tok = q * 32 + lane;              // token (TMEM lane) inside the tile
    const uint32_t lane_addr = tbase + (static_cast<uint32_t>(q * 32) << 16);
    int ntile = 0;  // tiles this CTA has finished (selects the exchange buffer and its phase)
    // The partial sums of K block j are ready when its stage barrier st_empty[j % STAGES] completes phase
    // j / STAGES.  That barrier cannot run a phase ahead of these warps: its next phase needs the MMAs of
    // K block j + STAGES, which wait for the TMEM buffer these warps free after K block j + STAGES - 2 > j.
    int ss = 0, buf = 0, ks = 0;
    uint32_t fph = 0, kph = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
      const Tile tl = get_tile<GATED>(p, t);
      const bool quarter_live = q * 32 < tl.cnt;  // warp-uniform: this quarter holds real tokens
      const bool live = tok < tl.cnt;
      float2 acc0[32], acc1[32];  // outputs 2i, 2i+1 of this thread's 64 in block 0 / block 1
#pragma unroll
      for (int j = 0; j < 32; ++j) { acc0[j] = make_float2(0.f, 0.f); acc1[j] = make_float2(0.f, 0.f); }
      // GEMM2: the token's slot now, its routing weight after the first K block (off the critical path)
      int slot = 0;
      float wgt = 0.f;
      if constexpr (!GATED) {
        if (live) slot = __ldg(p.sorted_ids + tl.pos0 + tok);
      }
      for (int kc = 0; kc < KC; ++kc) {
        // a lane that gives up takes its whole warp with it (the warp meets at __syncwarp below)
        ok = mbar_wait(&bars->f_full[ss], fph, abort, p.status, kWaitLimit) &&
             mbar_wait(&bars->st_empty[ks], kph, abort, p.status, kWaitLimit);
        if (!(ok = __all_sync(0xffffffffu, ok))) break;
        tc_fence_after();
        // the TMEM buffer and the factor slot go back as soon as the last partials are in registers,
        // before their FMAs
        auto release = [&]() {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&bars->p_empty[buf]);
            mbar_arrive(&bars->s_empty[ss]);
          }
        };
        if (quarter_live) {
          const float* fs = sS + ss * (S_SLOT / 4);
          const float2 fa = make_float2(fs[MAXN + tok], fs[MAXN + tok]);          // a_scale x w_scale, block 0
          const float2 fb = make_float2(fs[2 * MAXN + tok], fs[2 * MAXN + tok]);  // block 1
          const uint32_t base = lane_addr + static_cast<uint32_t>(buf * 2 * BM + ch * 64);
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t r0[32], r1[32];
            tmem_ld32(base + c * 32, r0);
            if (tl.two) tmem_ld32(base + BM + c * 32, r1);
            tmem_ld_wait();
            if (c == 1) release();
#pragma unroll
            for (int j = 0; j < 32; j += 2)
              acc0[(c * 32 + j) / 2] =
                  __ffma2_rn(make_float2(__uint_as_float(r0[j]), __uint_as_float(r0[j + 1])), fa, acc0[(c * 32 + j) / 2]);
            if (tl.two) {
#pragma unroll
              for (int j = 0; j < 32; j += 2)
                acc1[(c * 32 + j) / 2] = __ffma2_rn(make_float2(__uint_as_float(r1[j]), __uint_as_float(r1[j + 1])),
                                                    fb, acc1[(c * 32 + j) / 2]);
            }
          }
        } else {
          release();
        }
        if constexpr (!GATED) {
          // the slot has arrived by now (no routing weights: the masked layout's unweighted rows)
          if (kc == 0 && live) wgt = p.topk_w ? __ldg(p.topk_w + slot) : 1.f;
        }
        buf ^= 1;
        if (++ks == W_STAGES) { ks = 0; kph ^= 1; }
        if (++ss == S_STAGES) { ss = 0; fph ^= 1; }
      }
      if (!ok) break;

      if constexpr (GATED) {
        // h = SiLU(gate) * up for this token's 64 outputs; its 1 x 128 group (the tile's 128
        // outputs) is split between this warp and the warp of the other column half, which
        // exchange their maxima through a buffer that alternates between tiles.
        float hv[64];
        float m = 0.f;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          const float g = elem(acc0, j);
          hv[j] = __fdividef(g, 1.0f + __expf(-g)) * elem(acc1, j);  // fast division: 0 once exp(-g) > 2^126
          m = fmaxf(m, fabsf(hv[j]));
        }
        const int rb = ntile & 1;
        red[(rb * 2 + ch) * MAXN + tok] = m;
        mbar_arrive(&bars->red_full[rb][q]);
        ok = mbar_wait(&bars->red_full[rb][q], static_cast<uint32_t>((ntile >> 1) & 1), abort, p.status, kWaitLimit);
        if (!(ok = __all_sync(0xffffffffu, ok))) break;
        const float amax = fmaxf(m, red[(rb * 2 + (ch ^ 1)) * MAXN + tok]);
        if (live && NT == 2) {
          // the two-term form of h in the frame of its 1 x 128 group: hi codes in row pos, lo codes in
          // row cap + pos, the group's scale 2^e
          const int e = amax > 0.f ? e4m3_split_exp(amax) : 0;
          const float mul = exp2i(-e);
          const int pos = tl.pos0 + tok;
          uint4* dhi = reinterpret_cast<uint4*>(p.hq + static_cast<size_t>(pos) * p.n_rows_out + tl.n0 + ch * 64);
          uint4* dlo = reinterpret_cast<uint4*>(p.hq + static_cast<size_t>(p.cap + pos) * p.n_rows_out + tl.n0 + ch * 64);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t whi[4], wlo[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int j = v * 16 + u * 4;
              e4m3_split4(make_float4(hv[j], hv[j + 1], hv[j + 2], hv[j + 3]), mul, whi[u], wlo[u]);
            }
            dhi[v] = make_uint4(whi[0], whi[1], whi[2], whi[3]);
            dlo[v] = make_uint4(wlo[0], wlo[1], wlo[2], wlo[3]);
          }
          if (ch == 0) p.hs[static_cast<size_t>(tl.n0 / kQBlock) * p.cap + pos] = exp2i(e);
        } else if (live) {
          // s = amax / 448 and codes of h / s, by reciprocals (h codes are covered by the layer tolerance)
          const float s = amax > 0.f ? amax * (1.0f / 448.0f) : 1.0f;
          const float inv = amax > 0.f ? 448.0f * __frcp_rn(amax) : 1.0f;
          const int pos = tl.pos0 + tok;
          uint4* dst = reinterpret_cast<uint4*>(p.hq + static_cast<size_t>(pos) * p.n_rows_out + tl.n0 + ch * 64);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t w[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int j = v * 16 + u * 4;
              const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(hv[j] * inv, hv[j + 1] * inv), __NV_SATFINITE,
                                                           __NV_E4M3);
              const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(hv[j + 2] * inv, hv[j + 3] * inv),
                                                           __NV_SATFINITE, __NV_E4M3);
              w[u] = lo | (hi << 16);
            }
            dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
          }
          if (ch == 0) p.hs[static_cast<size_t>(tl.n0 / kQBlock) * p.cap + pos] = s;
        }
      } else {
        // y[slot] = acc x routing weight in bf16.  A thread holds one token's row, so direct stores
        // would put 32 rows in every warp instruction; instead the warp stages STG_COLS columns of its
        // 32 rows in shared memory at a time and writes them back row by row (2 * STG_COLS contiguous
        // bytes per row).  The 16-byte chunk j of row r sits at chunk j ^ (r & 7) with 8 chunks a row,
        // j ^ ((r >> 1) & 3) with 4, which keeps both the row-wise writes and the column-wise reads
        // free of bank conflicts (8 lanes, one 128-byte phase, always touch 8 different chunk columns).
        constexpr int CH = L::STG_COLS / 8;  // 16-byte chunks per staged row
        constexpr int RPI = 32 / CH;         // rows per read-back instruction
        auto swz = [](int r, int j) { return CH == 8 ? (j ^ (r & 7)) : (j ^ ((r >> 1) & 3)); };
        uint4* stg = reinterpret_cast<uint4*>(smem + L::OFF_STG + (warp - WARP_ACC0) * L::STG_BYTES);
        const int rr = lane / CH, cj = lane % CH;  // read-back: rows rr + RPI i, chunk cj
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          if (!quarter_live || (b == 1 && !tl.two)) break;
          const float2* a = b ? acc1 : acc0;
#pragma unroll
          for (int part = 0; part < 64 / L::STG_COLS; ++part) {
#pragma unroll
            for (int j = 0; j < CH; ++j) {
              uint32_t w[4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const float2 v2 = a[4 * (part * CH + j) + u];
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(v2.x * wgt, v2.y * wgt);
                w[u] = *reinterpret_cast<const uint32_t*>(&h2);
              }
              stg[lane * CH + swz(lane, j)] = make_uint4(w[0], w[1], w[2], w[3]);
            }
            __syncwarp();
            const int col = tl.n0 + b * BM + ch * 64 + part * L::STG_COLS + cj * 8;
#pragma unroll
            for (int i = 0; i < CH; ++i) {
              const int r = rr + RPI * i;
              const int rslot = __shfl_sync(0xffffffffu, slot, r);
              const uint4 val = stg[r * CH + swz(r, cj)];
              if (q * 32 + r < tl.cnt)
                *reinterpret_cast<uint4*>(p.y + static_cast<size_t>(rslot) * p.n_rows_out + col) = val;
            }
            __syncwarp();
          }
        }
      }
      ++ntile;
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

}  // namespace pfa8

// ------------------------------------------------------------------ gather
// E4M3 activation rows and their 1 x 128 scales in sorted (expert-contiguous)
// order; padding rows get zero codes and zero scales.  Scales are stored
// transposed, [H/128, cap], so a token tile's scales of one K block are
// contiguous for the TMA.  With nt = 2 the codes come in two terms: rows
// M..2M-1 of xq (the lo codes) go to rows cap..2cap-1 of act.
// One warp per (term, position) row, its lanes over the row's 16-byte chunks; then one thread
// per position writes its scales, so that every group's row of sa is written coalesced.
__global__ void __launch_bounds__(256) gather_a8_kernel(const uint8_t* __restrict__ xq, const float* __restrict__ sx,
                                                        const int32_t* __restrict__ sorted_ids,
                                                        const int32_t* __restrict__ num_post, int n_slots, int topk,
                                                        int H, int cap, int M, int nt, uint8_t* __restrict__ act,
                                                        float* __restrict__ sa) {
  pdl_wait();
  pdl_trigger();
  const int rows = *num_post;
  const int chunks = H / 16, G = H / kQBlock, lane = threadIdx.x & 31;
  const int nw = gridDim.x * (blockDim.x >> 5);
  for (int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < nt * rows; r += nw) {
    const int term = r >= rows ? 1 : 0;  // nt <= 2
    const int pos = r - term * rows;
    const int slot = __ldg(sorted_ids + pos);
    const bool valid = slot < n_slots;
    const uint4* src = reinterpret_cast<const uint4*>(xq + (static_cast<size_t>(term) * M + (valid ? slot / topk : 0)) * H);
    uint4* dst = reinterpret_cast<uint4*>(act + (static_cast<size_t>(term) * cap + pos) * H);
#pragma unroll 4
    for (int c = lane; c < chunks; c += 32) dst[c] = valid ? ld_v4(src + c) : make_uint4(0u, 0u, 0u, 0u);
  }
  const int nthr = gridDim.x * blockDim.x;
  for (int pos = blockIdx.x * blockDim.x + threadIdx.x; pos < rows; pos += nthr) {
    const int slot = __ldg(sorted_ids + pos);
    const bool valid = slot < n_slots;
    const float* s = sx + static_cast<size_t>(valid ? slot / topk : 0) * G;
    for (int g = 0; g < G; ++g) sa[static_cast<size_t>(g) * cap + pos] = valid ? __ldg(s + g) : 0.f;
  }
}

// ------------------------------------------------------------------ host side
template <bool GATED, int NT>
static cudaError_t launch_a8_gemm(const pfa8::Args& a, const void* w, uint64_t w_rows, const void* b,
                                  const float* bs, int num_sms, cudaStream_t s) {
  using namespace pfa8;
  auto kern = prefill_a8_kernel<GATED, NT>;
  // The register split (setmaxnreg) is only safe when the kernel was built with
  // the launch-bounds register count it was designed for.
  cudaFuncAttributes fa;
  cudaError_t err = cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(kern));
  if (err != cudaSuccess) return err;
  if (fa.numRegs != REGS_AT_LAUNCH) return cudaErrorInvalidConfiguration;
  CUtensorMap mw, mb, ms;
  if (!encode_tmap_2d(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, w, static_cast<uint64_t>(a.K), w_rows, BK, BM,
                      CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  CUtensorMap mb32, mb64;  // the same activations in boxes of 128, 32 and 64 rows
  if (!encode_tmap_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, b, static_cast<uint64_t>(a.K),
                      static_cast<uint64_t>(NT) * a.cap, BK, MAXN, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_2d(&mb32, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, b, static_cast<uint64_t>(a.K),
                      static_cast<uint64_t>(NT) * a.cap, BK, 32, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_2d(&mb64, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, b, static_cast<uint64_t>(a.K),
                      static_cast<uint64_t>(NT) * a.cap, BK, 64, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (!encode_tmap_2d(&ms, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, bs, static_cast<uint64_t>(a.cap),
                      static_cast<uint64_t>(a.K / kQBlock), MAXN, 1, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  constexpr int SMEM_BYTES = Lay<GATED, NT>::SMEM_BYTES;
  err = set_smem_limit_once(reinterpret_cast<const void*>(kern), SMEM_BYTES);
  if (err != cudaSuccess) return err;
  return launch_kernel(kern, dim3(num_sms), dim3(NUM_THREADS), SMEM_BYTES, s, true, mw, mb, mb32, mb64, ms, a);
}

template <int NT>
static cudaError_t launch_prefill_e4m3(const LayerPlan& P, int num_sms, cudaStream_t s, const StageHook& hook) {
  cudaError_t err;
  if (!P.out_direct) {  // (the masked layout's prologue already wrote the codes in position order)
    const int grid = num_sms * 8;
    err = launch_kernel(gather_a8_kernel, dim3(grid), dim3(256), 0, s, true, P.xq8, P.sx8, P.sorted_ids,
                        P.num_post, P.M * P.topk, P.topk, P.H, P.cap, P.M, NT, P.act8, P.sa8);
    if (err != cudaSuccess) return err;
    hook("prefill_gather", s);
  }
  pfa8::Args g1{};
  g1.K = P.H;
  g1.rows_per_expert = 2 * P.I;
  g1.second_rows = P.I;
  g1.n_tiles = P.I / pfa8::BM;
  g1.n_rows_out = P.I;
  g1.cap = P.cap;
  g1.ttiles = P.ttiles;
  g1.num_ttiles = P.num_ttiles;
  g1.wscale = P.s13;
  g1.sorted_ids = P.sorted_ids;
  g1.hq = P.h8;
  g1.hs = P.sh8;
  g1.tiles_from_prev = P.out_direct ? 1 : 0;  // the masked layout: its prologue wrote the tile list
  g1.status = P.status;
  err = launch_a8_gemm<true, NT>(g1, P.w13, static_cast<uint64_t>(P.E) * 2 * P.I, P.act8, P.sa8, num_sms, s);
  if (err != cudaSuccess) return err;
  hook("prefill_gemm1", s);
  pfa8::Args g2{};
  g2.K = P.I;
  g2.rows_per_expert = P.H;
  g2.second_rows = pfa8::BM;
  g2.n_tiles = (P.H + 2 * pfa8::BM - 1) / (2 * pfa8::BM);
  g2.n_rows_out = P.H;
  g2.cap = P.cap;
  g2.ttiles = P.ttiles;
  g2.num_ttiles = P.num_ttiles;
  g2.wscale = P.s2;
  g2.sorted_ids = P.sorted_ids;
  g2.topk_w = P.topk_w;
  // bf16 rows by slot in the fp32 buffer's space; the masked layout's output rows, unweighted
  g2.y = P.out_direct ? P.out_direct : reinterpret_cast<__nv_bfloat16*>(P.y);
  g2.status = P.status;
  err = launch_a8_gemm<false, NT>(g2, P.w2, static_cast<uint64_t>(P.E) * P.H, P.h8, P.sh8, num_sms, s);
  if (err != cudaSuccess) return err;
  hook("prefill_gemm2", s);
  if (P.out_direct) return cudaSuccess;  // the masked layout has no combine
  err = launch_combine(reinterpret_cast<const __nv_bfloat16*>(P.y), P.inv_pos, P.M, P.topk, P.H, P.out, num_sms, s);
  if (err != cudaSuccess) return err;
  hook("combine", s);
  return cudaSuccess;
}

cudaError_t launch_prefill_a8(const LayerPlan& P, int num_sms, cudaStream_t s, const StageHook& hook) {
  return P.e4m3_terms == 2 ? launch_prefill_e4m3<2>(P, num_sms, s, hook) : launch_prefill_e4m3<1>(P, num_sms, s, hook);
}

}  // namespace gbmoe
