// Decode path of the fused MoE layer: weight-streaming skinny grouped GEMMs.
//
// At decode batch sizes each active expert sees only a few tokens, so the
// layer is bound by reading the activated experts' weights from HBM once
// (the FP8 MoE decode of the OSDI'26 local-MoE paper summary, section "CPU
// decode backend", and the bandwidth argument of the SGLang CPU backend
// write-up, section "(3) FusedMoE").  The math follows the pages:
//
//  * GEMM1 uses the A x [B1, B2] = [C1, C2] form: one work item owns 64 gate
//    rows AND the matching 64 up rows of one expert, so h = SiLU(C1) * C2 is
//    finished inside the CTA and up_proj is never stored (Xeon 6 / SGLang blog,
//    section "MoE", SiLU-fusion bullet).
//  * FP8 weights are expanded to fp16 in registers and never stored wider; the
//    128x128 block scale multiplies each 128-deep partial sum once
//    (post-scaling, OSDI'26 summary, section "CPU decode backend").
//  * INT8 weights (DA8W8) multiply per-row-quantised activations; the integer
//    products are exact in fp32 and the per-row x per-channel scales are
//    applied once at the end.
//  * INT4 weights (two per byte, one scale per row and 128 columns) expand to
//    fp16 in registers like FP8; each 128-deep partial sum is scaled by its
//    row's group scale.  A stage holds the same 128 bytes of every row, which
//    are 256 K values (two scale groups).
//  * GEMM2 (down projection) writes each (token, slot) row already times its
//    routing weight, indexed by slot; a separate pass sums the top-k rows of
//    every token in slot order (deterministic, no atomics).
//  * FP8 and INT4: x rows arrive as fp16 in a power-of-two frame per row, and
//    GEMM1 stores h as fp16 in a frame per (row, 32 columns); GEMM1 takes x's
//    frames back in its epilogue, GEMM2 scales the rare blocks below their
//    row's frame down to it and takes the row frame back in its epilogue, so
//    no operand leaves fp16's range whatever the magnitudes.
//
// GB300 mapping.  A work item is (token tile of <= 8 slots of one expert) x
// (a block of weight rows).  One producer warp streams the item's weight rows
// through a deep shared-memory ring with TMA (128-byte-swizzled boxes, one
// 128-wide K block of 128 weight rows per 16 KB stage, ~176 KB in flight per
// SM).  Eight consumer warps take every stage in order; warp w owns 16-row
// m-tile w, reads its MMA fragments from shared memory without bank conflicts,
// expands E4M3 / INT8 to fp16 in registers and runs warp MMA m16n8k16 with the
// weights as the 16-row A operand and up to 8 tokens as N (swap-AB).  Inside
// each 128-wide K block the K order is permuted the same way for both
// operands, so every lane's 32 consecutive weight bytes feed its fragments
// directly.
#include <cuda.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace gbmoe {
namespace dec {

using namespace sm100;

constexpr int NCW = 8;                        // consumer warps
constexpr int NUM_THREADS = (NCW + 1) * 32;   // + one producer warp
constexpr int KBLK = 128;                     // K per stage (one FP8 scale block)

constexpr long long kWaitLimit = 4000000000LL;  // ~2 s of SM clocks per wait

// OCC resident CTAs per SM (measured): 2 CTAs with an 80 KB ring each when
// there are few work items, 3 CTAs with 48 KB rings otherwise -- more warps
// hide more latency.  B fragments are loaded one K block ahead (two ahead at
// 2 CTAs per SM measured no faster, three slower).
// INT4 (always 2 CTAs per SM) is bound by its nibble expansion, not by bytes in
// flight, and runs fastest with 48 KB rings (measured against 64 and 80 KB).
template <bool GATED, int OCC, bool I4 = false> struct Cfg {
  // One stage = 128 bytes of 128 weight rows (GATED: 64 gate rows and the matching
  // 64 up rows): one 128-wide K block of 8-bit codes or 256 K values of INT4.
  // Consumer warp w owns 16-row m-tile w of every stage.
  static constexpr int RING_BYTES = OCC == 2 && !I4 ? 80 * 1024 : 48 * 1024;
  static constexpr int BPF = 1;                            // stages of B fragments loaded ahead
  static constexpr int STAGE = NCW * 16 * KBLK;            // 16 KB of weight codes
  static constexpr int NS = RING_BYTES / STAGE;            // ring stages
  static constexpr int OFF_RED = RING_BYTES;
  static constexpr int RED_BYTES = 4 * 4 * 32 * 4 + 256;   // up accumulators handed to the gate warps, then the
                                                           // h block maxima (4 x 8) and frame exponents (8)
  static constexpr int OFF_BAR = OFF_RED + RED_BYTES;
  static constexpr int SMEM = OFF_BAR + 2 * NS * 8 + 64 + 1024;
  static constexpr int ROWS = GATED ? 64 : 128;            // output rows per item
};

__device__ __forceinline__ uint32_t word8(const uint4& a, const uint4& b, int s) {
  switch (s) {
    case 0: return a.x; case 1: return a.y; case 2: return a.z; case 3: return a.w;
    case 4: return b.x; case 5: return b.y; case 6: return b.z; default: return b.w;
  }
}

__device__ __forceinline__ uint32_t word16(const uint4* x, int i) {
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
// Even and odd MMA steps accumulate into two independent chains (acc0, acc1) so
// that consecutive tensor-core instructions do not wait on each other.
template <int WK>
__device__ __forceinline__ void tile_mma_128(float acc0[4], float acc1[4], const uint4& ra0, const uint4& ra1,
                                             const uint4& rb0, const uint4& rb1, const uint4* xb) {
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    uint32_t a[4];
    w8x4_to_f16x4<WK>(word8(ra0, ra1, s), a[0], a[2]);
    w8x4_to_f16x4<WK>(word8(rb0, rb1, s), a[1], a[3]);
    mma_f16_16816((s & 1) ? acc1 : acc0, a, word16(xb, 2 * s), word16(xb, 2 * s + 1));
  }
}

// INT4: 16 rows x 128 K.  Lane (g, t) holds 16 consecutive bytes (32 values) of
// rows g and g+8 from column 32t (ra, rb) and the 32 matching activations of
// token column g, stored in the INT4 K order (xb).  Word w of ra expands to the
// pairs (k0,k4) (k1,k5) (k2,k6) (k3,k7) of K values 32t+8w..32t+8w+7: the first
// two pairs feed one MMA step, the last two the next, and xb[w] holds the
// activations of the same K values in the same order.
__device__ __forceinline__ void tile_mma_int4(float acc0[4], float acc1[4], const uint4& ra, const uint4& rb,
                                              const uint4* xb) {
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const uint32_t wa = w == 0 ? ra.x : w == 1 ? ra.y : w == 2 ? ra.z : ra.w;
    const uint32_t wb = w == 0 ? rb.x : w == 1 ? rb.y : w == 2 ? rb.z : rb.w;
    uint32_t fa[4], fb[4];
    s4x8_to_f16x8(wa, fa);
    s4x8_to_f16x8(wb, fb);
    const uint32_t a0[4] = {fa[0], fb[0], fa[1], fb[1]};
    mma_f16_16816(acc0, a0, xb[w].x, xb[w].y);
    const uint32_t a1[4] = {fa[2], fb[2], fa[3], fb[3]};
    mma_f16_16816(acc1, a1, xb[w].z, xb[w].w);
  }
}

// Shared-memory fragment load that the compiler may not repeat or defer: the ring
// slot is released right after these loads.
__device__ __forceinline__ uint4 lds_v4_once(const void* p) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p)))
               : "memory");
  return r;
}

__device__ __forceinline__ void load_b32(uint4* xb, const __half* row, bool valid) {
#pragma unroll
  for (int i = 0; i < 4; ++i) xb[i] = valid ? ld_v4(row + 8 * i) : make_uint4(0u, 0u, 0u, 0u);
}

// Consumer-warps-only barrier (named barrier 1).
__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, %0;" ::"n"(NCW * 32) : "memory"); }
// Gate-warps-only barrier of GEMM1's epilogue (named barrier 2, warps 0-3).
__device__ __forceinline__ void gate_warps_sync() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

struct Item {
  int e, pos0, cnt, rt;
};

__device__ __forceinline__ Item get_item(const SkinnyArgs& a, int it) {
  const int tt = it / a.n_rt;
  const int4 d = a.ttiles[tt];
  return Item{d.x, d.y, d.z, it - tt * a.n_rt};
}

// RQ: INT8 GEMM2 that quantises h itself: its B fragments are read from GEMM1's fp32 h and coded per
// position (s = max|h| / 127) in registers, so no requant launch sits between the GEMMs.
// EQ: only as many CTAs take items as give every one of them the same count (a separate build: the
// item bounds it keeps in registers slowed the kernel where it does not help).
template <int WK, bool GATED, int OCC, bool RQ = false, bool EQ = false>
__global__ void __launch_bounds__(NUM_THREADS, OCC)
    skinny_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w, SkinnyArgs a) {
  static_assert(!RQ || (WK == MOE_WEIGHT_INT8 && !GATED), "h is quantised in the INT8 down projection only");
  using C = Cfg<GATED, OCC, WK == MOE_WEIGHT_INT4>;
  constexpr bool I4 = WK == MOE_WEIGHT_INT4;
  constexpr int KST = I4 ? 2 * KBLK : KBLK;  // K values per stage
  constexpr int XB = I4 ? 8 : 4;             // 16-byte B fragments per stage and lane
  constexpr int BPF = I4 ? 1 : C::BPF;       // an INT4 stage already carries twice the B fragments
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* red = reinterpret_cast<float*>(smem + C::OFF_RED);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + C::NS;
  int* abort_flag = reinterpret_cast<int*>(empty + C::NS);
  volatile int* abort = abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KB = (a.K + KST - 1) / KST;  // stages per item (INT4: the last may hold one group)

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], NCW);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  // GEMM1 needs the predecessor's tile list and prepared activations before anything;
  // GEMM2's weight stream only needs the tile list (written two kernels back), so its
  // producer starts at once and its consumers wait before reading h.
  if (GATED || warp < NCW) pdl_wait();
  const int n_items = *a.num_ttiles * a.n_rt;
  // GEMM2's grid may launch early (its CTAs set up and prefetch weights).  A long
  // GEMM1 (more than two items per CTA) does not trigger it: GEMM2 CTAs placed one
  // by one into the slots of finished GEMM1 CTAs made the layer slower (measured).
  if (!GATED || n_items <= 2 * static_cast<int>(gridDim.x)) pdl_trigger();

  // Item order (measured): GEMM1 items go round-robin over the CTAs; GEMM2 items
  // go in contiguous runs per CTA, so a CTA streams adjacent weight rows.  EQ: k =
  // ceil(items / grid) items for each of ceil(items / k) CTAs, the others leave at
  // once -- a last round that leaves part of the CTAs idle streams too few bytes at
  // once to keep HBM busy.
  int ctas = static_cast<int>(gridDim.x);
  if constexpr (EQ) {
    const int k = (n_items + ctas - 1) / ctas;
    if (k > 1) ctas = (n_items + k - 1) / k;
  }
  const bool has_items = !EQ || static_cast<int>(blockIdx.x) < ctas;
  const int it_begin =
      !has_items ? 0
      : GATED    ? static_cast<int>(blockIdx.x)
                 : static_cast<int>(static_cast<long long>(n_items) * blockIdx.x / ctas);
  const int it_end = !has_items ? 0
                     : GATED    ? n_items
                                : static_cast<int>(static_cast<long long>(n_items) * (blockIdx.x + 1) / ctas);
  const int it_step = GATED ? ctas : 1;

  if (warp == NCW) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      prefetch_tmap(&tmap_w);
      long long seq = 0;
      int slot = 0;
      uint32_t par = 0;
      bool ok = true;
      for (int it = it_begin; it < it_end && ok; it += it_step) {
        const Item im = get_item(a, it);
        const int row0 = im.e * a.rows_per_expert + im.rt * C::ROWS;
        for (int kb = 0; kb < KB; ++kb, ++seq) {
          if (!(ok = mbar_wait(&empty[slot], par ^ 1, abort, a.status, kWaitLimit))) break;
          mbar_arrive_expect_tx(&full[slot], C::STAGE);
          uint8_t* dst = smem + slot * C::STAGE;
          // (INT4 with K % 256 == 128: the last box reaches past the row end and is zero-filled)
          if (GATED) {
            tma_load_2d(dst, &tmap_w, &full[slot], kb * KBLK, row0);
            tma_load_2d(dst + C::STAGE / 2, &tmap_w, &full[slot], kb * KBLK, row0 + a.up_offset);
          } else {
            tma_load_2d(dst, &tmap_w, &full[slot], kb * KBLK, row0);
          }
          if (++slot == C::NS) { slot = 0; par ^= 1; }
        }
      }
      // never leave with copies in flight into this CTA's shared memory
      const long long n_last = seq < C::NS ? seq : C::NS;
      for (long long i = 1; i <= n_last; ++i) {
        const long long s = seq - i;
        int dummy = 0;
        mbar_wait(&full[s % C::NS], static_cast<uint32_t>((s / C::NS) & 1), &dummy, nullptr, kWaitLimit);
      }
    }
    return;  // the producer takes no part in the consumers' named barriers
  }

  // ------------------------------------------------------------------ consumers
  // Every consumer warp takes part in every stage, in order (so the ring's phase
  // parity always refers to the stage it expects); warp w owns m-tile w.
  const int g = lane >> 2, t = lane & 3;
  int slot = 0;          // ring slot of the next stage
  uint32_t phase = 0;    // its phase parity
  bool ok = true;
  const int kblocks = a.K / kQBlock, rblocks = a.rows_per_expert / kQBlock;
  // B operand row of this lane's token column g (GEMM1: x by token; GEMM2: h by position)
  auto b_row = [&](const Item& x, bool& valid) -> const __half* {
    valid = g < x.cnt;
    if constexpr (GATED) {
      if (a.b_by_pos) return a.b + static_cast<size_t>(x.pos0 + (valid ? g : 0)) * a.K;  // masked layout
      const int tok = valid ? __ldg(a.sorted_ids + x.pos0 + g) / a.topk : 0;
      return a.b + static_cast<size_t>(tok) * a.K;
    } else {
      return a.b + static_cast<size_t>(x.pos0 + g) * a.K;  // rows of padded slots are readable
    }
  };
  // B fragments of the next BPF stages are loaded ahead (a ring in registers).  INT4:
  // the two groups of a stage, the second absent past K.
  uint4 xr[BPF][XB];
  // RQ: the lane's 32 fp32 values of h of the next BPF stages, and 127 / max|h| of its B column
  uint4 hr[RQ ? BPF : 1][RQ ? 8 : 1];
  float rq_r = 1.f;
  auto load_stage_rq = [&](uint4* raw, const float* hrow, int kb, bool valid) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      raw[i] = valid ? ld_v4(hrow + static_cast<size_t>(kb) * KBLK + t * 32 + 4 * i) : make_uint4(0u, 0u, 0u, 0u);
  };
  auto quant_stage = [&](uint4* xb, const uint4* raw) {  // codes RNE(h * 127 / max|h|), as fp16
    auto q = [&](uint32_t v) { return fminf(fmaxf(rintf(__uint_as_float(v) * rq_r), -127.0f), 127.0f); };
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 a0 = raw[2 * i], a1 = raw[2 * i + 1];
      xb[i] = make_uint4(pack_half2(q(a0.x), q(a0.y)), pack_half2(q(a0.z), q(a0.w)), pack_half2(q(a1.x), q(a1.y)),
                         pack_half2(q(a1.z), q(a1.w)));
    }
  };
  auto load_stage = [&](uint4* xb, const __half* brow, int kb, bool valid) {
    load_b32(xb, brow + static_cast<size_t>(kb) * KST + t * 32, valid);
    if constexpr (I4) load_b32(xb + 4, brow + static_cast<size_t>(kb) * KST + KBLK + t * 32,
                               valid && kb * KST + KBLK < a.K);
  };
  // GEMM2 on h (FP8, INT4): the lane's B values of a stage are one 32-column block of h per 128 K
  // (FP8: block 4kb + t; INT4: blocks 8kb + t and 8kb + 4 + t), stored in that block's frame.
  // The epilogue applies the row frame (the largest block exponent).  A row whose blocks do not all
  // share it ("mixed": its smallest block exponent is lower) has those blocks scaled down here, after
  // the stage's fragments have arrived; items whose rows each have one frame, the usual case, run a
  // K loop without this step.
  constexpr bool HF = !GATED && WK != MOE_WEIGHT_INT8;
  const int hld = a.K / kHBlock;
  // bits 0-7: biased row frame of this lane's B column (0: none, nothing to scale); bit 8: the row has
  // blocks below its frame; bit 9: some lane of the warp has such a row
  uint32_t fst = 0;
  auto frame_fix = [&](uint4* xb, const Item& x, int kb) {
    if constexpr (HF) {
      const uint32_t eg = fst & 0xffu;
      const int b0 = (I4 ? 8 * kb : 4 * kb) + t;
      const uint8_t* hp = a.hblk + static_cast<size_t>(x.pos0 + g) * hld + b0;
#pragma unroll
      for (int grp = 0; grp < (I4 ? 2 : 1); ++grp) {  // INT4: the stage's two 128-wide groups in turn
        const uint32_t b = (fst & 0x100u) && b0 + 4 * grp < hld ? __ldg(hp + 4 * grp) : 0u;
        if (b != 0u && b != eg) {
          const __half2 f = exp2i_h2(static_cast<int>(b) - static_cast<int>(eg));
#pragma unroll
          for (int i = 0; i < 4; ++i) scale_h8(xb[4 * grp + i], f);
        }
      }
    }
  };
  for (int it = it_begin; it < it_end; it += it_step) {
    const Item im = get_item(a, it);
    const int r0 = im.rt * C::ROWS;  // first output row of the item inside the expert
    // weight row (inside the expert) of this warp's m-tile
    const int mrow = GATED ? (warp < 4 ? r0 + warp * 16 : a.up_offset + r0 + (warp - 4) * 16) : r0 + warp * 16;
    const float* scale_row = a.wscale + (static_cast<size_t>(im.e) * rblocks + mrow / kQBlock) * kblocks;
    // INT4: group scales of this lane's rows g and g+8, [E, rows, K/128]
    const float* sg_row = a.wscale + (static_cast<size_t>(im.e) * a.rows_per_expert + mrow + g) * kblocks;
    bool bvalid;
    const __half* brow = b_row(im, bvalid);
    const float* hrow = nullptr;  // RQ: the fp32 h row of the lane's B column
    if constexpr (RQ) {
      hrow = a.bh + static_cast<size_t>(im.pos0 + (bvalid ? g : 0)) * a.K;
      const float amax = bvalid ? __uint_as_float(__ldg(a.hmax + im.pos0 + g)) : 0.f;
      rq_r = amax > 0.f ? 127.0f / amax : 1.0f;
    }
    // GEMM2 on h: the B column's row frame and lowest block frame (consumed after the fragment prefetch
    // below is in flight, so the two loads' latencies overlap)
    uint32_t eg_ld = 0u, lo_ld = 0u;
    if constexpr (HF) {
      if (bvalid) {
        eg_ld = __ldg(a.hexp + im.pos0 + g);
        lo_ld = __ldg(a.hexp_lo + im.pos0 + g);
      }
    }
    // GEMM1 (FP8, INT4): the x frames of this thread's two epilogue columns 2t, 2t+1 -- loaded here
    // for FP8, in the epilogue for INT4 (whose registers are all taken by the K loop)
    float sxc[2] = {0.f, 0.f};
    auto load_sxc = [&]() {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int col = 2 * t + c, pos = im.pos0 + col;
        if (col < im.cnt) sxc[c] = __ldg(a.sx + (a.b_by_pos ? pos : __ldg(a.sorted_ids + pos) / a.topk));
      }
    };
    if constexpr (GATED && WK == MOE_WEIGHT_FP8) {
      if (warp < 4) load_sxc();
    }
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
    float scr[BPF];     // FP8 block scales of the prefetched stages
    float sgs[BPF][4];  // INT4: group scales of rows g, g+8 (group 0) and g, g+8 (group 1)
    auto load_scales = [&](int d, int kb) {
      if constexpr (WK == MOE_WEIGHT_FP8) scr[d] = __ldg(scale_row + kb);
      if constexpr (I4) {
        const bool two = 2 * kb + 1 < kblocks;
        sgs[d][0] = __ldg(sg_row + 2 * kb);
        sgs[d][1] = __ldg(sg_row + 8 * kblocks + 2 * kb);
        sgs[d][2] = two ? __ldg(sg_row + 2 * kb + 1) : 0.f;
        sgs[d][3] = two ? __ldg(sg_row + 8 * kblocks + 2 * kb + 1) : 0.f;
      }
    };
#pragma unroll
    for (int d = 0; d < BPF; ++d) {
      if (d < KB) {
        if constexpr (RQ) load_stage_rq(hr[d], hrow, d, bvalid);
        else load_stage(xr[d], brow, d, bvalid);
        load_scales(d, d);
      }
    }
    if constexpr (HF) {
      fst = eg_ld | (lo_ld != 0u && 256u - lo_ld != eg_ld ? 0x100u : 0u);
      if (__any_sync(0xffffffffu, fst & 0x100u)) fst |= 0x200u;
    }
    // The K loop, compiled twice: with the frame fix for items where some lane's row of h has blocks
    // below its frame, and without it (the usual case, which then pays nothing per stage).
    auto k_loop = [&](auto fix_tag) {
      constexpr bool FIX = decltype(fix_tag)::value;
      for (int kb0 = 0; kb0 < KB; kb0 += BPF) {
#pragma unroll
      for (int d = 0; d < BPF; ++d) {
        const int kb = kb0 + d;
        if (kb >= KB) break;
        uint4* xb = xr[d];
        if (ok) ok = mbar_wait(&full[slot], phase, abort, a.status, kWaitLimit);
        if constexpr (FIX) frame_fix(xb, im, kb);
        if (!ok) {
        } else if constexpr (I4) {
          // rows warp*16 + g and + 8 of the stage; 16-byte chunk c of row r sits at c ^ (r % 8);
          // chunks 0-3 are group 0, chunks 4-7 group 1, and lane t takes chunk t of each
          const uint8_t* rg = smem + slot * C::STAGE + (warp * 16 + g) * KBLK;
          const uint8_t* rh = rg + 8 * KBLK;
          const uint4 ra0 = lds_v4_once(rg + ((t ^ g) << 4));
          const uint4 ra1 = lds_v4_once(rg + (((t + 4) ^ g) << 4));
          const uint4 rb0 = lds_v4_once(rh + ((t ^ g) << 4));
          const uint4 rb1 = lds_v4_once(rh + (((t + 4) ^ g) << 4));
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[slot]);
          float p0[4] = {0.f, 0.f, 0.f, 0.f}, p1[4] = {0.f, 0.f, 0.f, 0.f};
          float q0[4] = {0.f, 0.f, 0.f, 0.f}, q1[4] = {0.f, 0.f, 0.f, 0.f};
          tile_mma_int4(p0, p1, ra0, rb0, xb);
          tile_mma_int4(q0, q1, ra1, rb1, xb + 4);  // zero codes and activations past K
          const float* sc = sgs[d];
          acc[0] = fmaf(sc[0], p0[0] + p1[0], fmaf(sc[2], q0[0] + q1[0], acc[0]));
          acc[1] = fmaf(sc[0], p0[1] + p1[1], fmaf(sc[2], q0[1] + q1[1], acc[1]));
          acc[2] = fmaf(sc[1], p0[2] + p1[2], fmaf(sc[3], q0[2] + q1[2], acc[2]));
          acc[3] = fmaf(sc[1], p0[3] + p1[3], fmaf(sc[3], q0[3] + q1[3], acc[3]));
        } else {
          // rows warp*16 + g and + 8 of the stage; 16-byte chunk c of row r sits at c ^ (r % 8)
          const uint8_t* rg = smem + slot * C::STAGE + (warp * 16 + g) * KBLK;
          const uint8_t* rh = rg + 8 * KBLK;
          const uint4 ra0 = lds_v4_once(rg + (((2 * t) ^ g) << 4));
          const uint4 ra1 = lds_v4_once(rg + (((2 * t + 1) ^ g) << 4));
          const uint4 rb0 = lds_v4_once(rh + (((2 * t) ^ g) << 4));
          const uint4 rb1 = lds_v4_once(rh + (((2 * t + 1) ^ g) << 4));
          // the fragments are in registers; order these generic-proxy reads before the
          // TMA (async proxy) that will overwrite the slot once every warp has released it
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[slot]);
          if constexpr (RQ) quant_stage(xb, hr[d]);  // after the release (its loads were issued a stage ago)
          if constexpr (WK == MOE_WEIGHT_FP8) {
            float p0[4] = {0.f, 0.f, 0.f, 0.f}, p1[4] = {0.f, 0.f, 0.f, 0.f};
            tile_mma_128<WK>(p0, p1, ra0, ra1, rb0, rb1, xb);
            const float sc = scr[d];
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i] = fmaf(sc, p0[i] + p1[i], acc[i]);
          } else {
            tile_mma_128<WK>(acc, acc1, ra0, ra1, rb0, rb1, xb);
          }
        }
        if (kb + BPF < KB) {
          if constexpr (RQ) load_stage_rq(hr[d], hrow, kb + BPF, bvalid);
          else load_stage(xr[d], brow, kb + BPF, bvalid);
          load_scales(d, kb + BPF);
        }
        if (++slot == C::NS) { slot = 0; phase ^= 1; }
      }
      }
    };
    if constexpr (HF) {
      if (fst & 0x200u) k_loop(std::true_type{});
      else k_loop(std::false_type{});
    } else {
      k_loop(std::false_type{});
    }

    if constexpr (WK == MOE_WEIGHT_INT8) {
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i] += acc1[i];
    }
    // ---- epilogue (fragment: rows g, g+8 x token columns 2t, 2t+1)
    if constexpr (GATED) {
      if (warp >= 4) {
#pragma unroll
        for (int i = 0; i < 4; ++i) red[((warp - 4) * 4 + i) * 32 + lane] = acc[i];
      }
      consumers_sync();
      if (warp < 4) {
        if constexpr (WK == MOE_WEIGHT_INT8) {
          float cmax[2] = {0.f, 0.f};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float G = acc[i], U = red[(warp * 4 + i) * 32 + lane];
            const int row = g + ((i & 2) ? 8 : 0);
            const int col = 2 * t + (i & 1);
            const int pos = im.pos0 + col;
            const int n = r0 + warp * 16 + row;
            float h = 0.f;
            if (col < im.cnt) {
              const float sx = __ldg(a.sx + __ldg(a.sorted_ids + pos) / a.topk);
              const float gv = G * sx * __ldg(a.wscale + static_cast<size_t>(im.e) * a.rows_per_expert + n);
              const float uv =
                  U * sx * __ldg(a.wscale + static_cast<size_t>(im.e) * a.rows_per_expert + a.up_offset + n);
              h = silu_f32(gv) * uv;
              reinterpret_cast<float*>(a.out)[static_cast<size_t>(pos) * a.out_ld + n] = h;
            }
            cmax[i & 1] = fmaxf(cmax[i & 1], fabsf(h));
          }
#pragma unroll
          for (int c = 0; c < 2; ++c) {  // max over the 16 rows of each column (lanes with equal t)
            float v = cmax[c];
            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
            const int col = 2 * t + c;
            if (g == 0 && col < im.cnt) atomicMax(a.hmax + im.pos0 + col, __float_as_uint(v));
          }
        } else {
          // FP8 / INT4: h = SiLU(g) * u in fp32 from the x frames of the thread's two token columns, then
          // stored in fp16 in the frame of its (position, 32-column block): gate warps 0-1 hold the item's
          // first block, warps 2-3 its second, and the max over a pair's 32 rows decides the frame
          float* hred = red + 4 * 4 * 32;                               // [4 warps][8 columns]
          uint32_t* hexp_s = reinterpret_cast<uint32_t*>(hred + 32);    // [2 blocks][8 columns]
          float hv[4], cmax[2] = {0.f, 0.f};
          if constexpr (WK == MOE_WEIGHT_INT4) load_sxc();
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float G = acc[i] * sxc[i & 1], U = red[(warp * 4 + i) * 32 + lane] * sxc[i & 1];
            hv[i] = silu_f32(G) * U;
            cmax[i & 1] = fmaxf(cmax[i & 1], fabsf(hv[i]));
          }
#pragma unroll
          for (int c = 0; c < 2; ++c) {  // max over the warp's 16 rows of each column (lanes with equal t)
            float v = cmax[c];
            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
            if (g == 0) hred[warp * 8 + 2 * t + c] = v;
          }
          gate_warps_sync();
          if (warp == 0 && lane < 16) {  // one lane per (token column, block) decides the block's frame
            const int col = lane & 7, blk = lane >> 3;
            uint32_t eb = 0;
            if (col < im.cnt) {
              eb = static_cast<uint32_t>(h_frame_exp_biased(fmaxf(hred[16 * blk + col], hred[16 * blk + 8 + col])));
              const int pos = im.pos0 + col;
              a.hblk[static_cast<size_t>(pos) * (a.out_ld / kHBlock) + 2 * im.rt + blk] = static_cast<uint8_t>(eb);
              if (eb) {
                atomicMax(a.hexp + pos, eb);
                atomicMax(a.hexp_lo + pos, 256u - eb);  // 256 - the smallest nonzero block exponent
              }
            }
            hexp_s[lane] = eb;
          }
          gate_warps_sync();
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int row = g + ((i & 2) ? 8 : 0);
            const int col = 2 * t + (i & 1);
            if (col >= im.cnt) continue;
            const uint32_t eb = hexp_s[8 * (warp >> 1) + col];
            const float mul = eb ? exp2i(kExpBias - static_cast<int>(eb)) : 1.f;
            const int pos = im.pos0 + col;
            const int n = r0 + warp * 16 + row;
            // (INT4: h feeds GEMM2's activations, stored in the INT4 K order)
            reinterpret_cast<__half*>(a.out)[static_cast<size_t>(pos) * a.out_ld +
                                             (WK == MOE_WEIGHT_INT4 ? int4_kperm(n) : n)] = __float2half_rn(hv[i] * mul);
          }
        }
      }
      consumers_sync();  // red is reused by the next item
    } else {
      // h's row frames of the thread's columns 2t, 2t+1, from the lanes that hold them as B columns
      float hf[2] = {1.f, 1.f};
      if constexpr (HF) {
#pragma unroll
        for (int c = 0; c < 2; ++c)
          hf[c] = exp2i(static_cast<int>(__shfl_sync(0xffffffffu, fst & 0xffu, 4 * (2 * t + c))) - kExpBias);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int row = g + ((i & 2) ? 8 : 0);
        const int col = 2 * t + (i & 1);
        if (col < im.cnt) {
          const int pos = im.pos0 + col;
          const int n = r0 + warp * 16 + row;
          const int slot = __ldg(a.sorted_ids + pos);
          const float v = acc[i] * hf[i & 1];
          if (a.out_bf16) {  // masked layout: the output row itself, unweighted
            a.out_bf16[static_cast<size_t>(slot) * a.out_ld + n] = __float2bfloat16_rn(v);
            continue;
          }
          float wgt = __ldg(a.topk_w + slot);
          if constexpr (RQ) {  // the scale of the codes this kernel made
            const float amax = __uint_as_float(__ldg(a.hmax + pos));
            wgt *= (amax > 0.f ? amax * (1.0f / 127.0f) : 1.0f) *
                   __ldg(a.wscale + static_cast<size_t>(im.e) * a.rows_per_expert + n);
          } else if constexpr (WK == MOE_WEIGHT_INT8) {
            wgt *= __ldg(a.sh + pos) * __ldg(a.wscale + static_cast<size_t>(im.e) * a.rows_per_expert + n);
          }
          reinterpret_cast<float*>(a.out)[static_cast<size_t>(slot) * a.out_ld + n] = v * wgt;
        }
      }
    }
  }
}

}  // namespace dec

// ------------------------------------------------------------------ INT8: requantise h per row
// One CTA per row: s = max|h| / 127, codes = RNE(h / s) clamped to +-127, stored as fp16.
// I is a multiple of 128, so every thread moves whole 4-element vectors.
__global__ void __launch_bounds__(128) requant_h_kernel(const float* __restrict__ h, const uint32_t* __restrict__ hmax,
                                                        const int32_t* __restrict__ num_post, int I,
                                                        __half* __restrict__ hq, float* __restrict__ sh) {
  pdl_wait();
  pdl_trigger();
  const int rows = *num_post;
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    const float amax = __uint_as_float(hmax[r]);
    const float s = amax > 0.f ? __fdiv_rn(amax, 127.0f) : 1.0f;
    const float4* hr = reinterpret_cast<const float4*>(h + static_cast<size_t>(r) * I);
    uint2* qr = reinterpret_cast<uint2*>(hq + static_cast<size_t>(r) * I);
    for (int c = threadIdx.x; c < I / 4; c += blockDim.x) {
      const float4 v = __ldg(hr + c);
      qr[c] = make_uint2(pack_half2(quant_s8_rne(v.x, s), quant_s8_rne(v.y, s)),
                         pack_half2(quant_s8_rne(v.z, s), quant_s8_rne(v.w, s)));
    }
    if (threadIdx.x == 0) sh[r] = s;
  }
}

cudaError_t launch_requant_rows(const void* h, const uint32_t* hmax, const int32_t* num_post, int cap, int I,
                                __half* hq, float* sh, int num_sms, cudaStream_t s) {
  // cap: an upper bound of the padded positions (a CTA per row up to 8 per SM); the device count decides
  int grid = cap < num_sms * 8 ? cap : num_sms * 8;
  if (grid < 1) grid = 1;
  return launch_kernel(requant_h_kernel, dim3(grid), dim3(128), 0, s, true, static_cast<const float*>(h), hmax,
                       num_post, I, hq, sh);
}

template <int WK, bool GATED, int OCC, bool RQ = false, bool EQ = false>
static cudaError_t launch_skinny_occ(const SkinnyArgs& a, const void* w, uint64_t w_rows, int num_sms,
                                     cudaStream_t s) {
  using C = dec::Cfg<GATED, OCC, WK == MOE_WEIGHT_INT4>;
  CUtensorMap mw;
  // a row holds K bytes of 8-bit codes or K/2 bytes of INT4; a stage takes 128 of them
  const uint64_t row_bytes = WK == MOE_WEIGHT_INT4 ? a.K / 2 : a.K;
  if (!encode_tmap_2d(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, w, row_bytes, w_rows, dec::KBLK, C::ROWS,
                      CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  auto kern = dec::skinny_gemm_kernel<WK, GATED, OCC, RQ, EQ>;
  cudaError_t err = set_smem_limit_once(reinterpret_cast<const void*>(kern), C::SMEM);
  if (err != cudaSuccess) return err;
  return launch_kernel(kern, dim3(OCC * num_sms), dim3(dec::NUM_THREADS), C::SMEM, s, true, mw, a);
}

// The EQ build where the host's bound puts 2.5 to 10 items on a CTA (measured: DeepSeek-R1 at 4 and 8
// tokens 2-3% faster; at 1, 2 and 64 tokens and with INT4 weights it gained nothing).
template <int WK, bool GATED, int OCC>
static cudaError_t launch_skinny_eq(const SkinnyArgs& a, const void* w, uint64_t w_rows, long long max_items,
                                    int num_sms, cudaStream_t s) {
  const long long grid = static_cast<long long>(OCC) * num_sms;
  return 2 * max_items >= 5 * grid && max_items <= 10 * grid
             ? launch_skinny_occ<WK, GATED, OCC, false, true>(a, w, w_rows, num_sms, s)
             : launch_skinny_occ<WK, GATED, OCC>(a, w, w_rows, num_sms, s);
}

// max_items: an upper bound of the work items the launch can see.
template <int WK, bool GATED>
static cudaError_t launch_skinny(const SkinnyArgs& a, const void* w, uint64_t w_rows, long long max_items,
                                 int num_sms, cudaStream_t s) {
  if constexpr (WK == MOE_WEIGHT_INT8 && !GATED) {
    if (a.bh) return launch_skinny_occ<WK, GATED, 2, true>(a, w, w_rows, num_sms, s);  // (two CTAs per SM only)
  }
  // INT4 keeps two CTAs per SM: at three, its B fragments of two groups do not fit the registers
  if constexpr (WK == MOE_WEIGHT_INT4) {
    (void)max_items;
    return launch_skinny_occ<WK, GATED, 2>(a, w, w_rows, num_sms, s);
  } else {
    // Two CTAs per SM (the deeper rings) below 9 (GEMM1) or 6 (GEMM2) items per SM, measured: at
    // DeepSeek-R1 shapes GEMM1 of two tokens 0.102 -> 0.092 ms and of four 0.172 -> 0.166 ms, GEMM2
    // of one token 0.037 -> 0.031 ms (its 504 items no longer leave 48 of 456 CTAs a second
    // item); GEMM2 of two tokens is faster at three CTAs per SM.
    const long long occ3_min = GATED ? 9LL * num_sms : 6LL * num_sms;
    return max_items >= occ3_min ? launch_skinny_eq<WK, GATED, 3>(a, w, w_rows, max_items, num_sms, s)
                                 : launch_skinny_eq<WK, GATED, 2>(a, w, w_rows, max_items, num_sms, s);
  }
}

cudaError_t launch_decode(const LayerPlan& P, int weight_kind, int num_sms, cudaStream_t s, const StageHook& hook) {
  // token tiles: at most one per (expert, 8 slots) -- bounded by min(E, slots) + slots / 8
  const long long slots = static_cast<long long>(P.M) * P.topk;
  const long long max_tiles = (slots < P.E ? slots : P.E) + slots / kDecodeBlock;
  SkinnyArgs g1{};
  g1.K = P.H;
  g1.rows_per_expert = 2 * P.I;
  g1.up_offset = P.I;
  g1.n_rt = P.I / dec::Cfg<true, 2>::ROWS;
  g1.ttiles = P.ttiles;
  g1.num_ttiles = P.num_ttiles;
  g1.wscale = P.s13;
  g1.sorted_ids = P.sorted_ids;
  g1.topk = P.topk;
  g1.b = P.xq;
  g1.sx = P.sx;
  g1.out = P.h;
  g1.out_ld = P.I;
  g1.hmax = P.hmax;
  g1.status = P.status;
  g1.b_by_pos = P.out_direct ? 1 : 0;
  g1.hexp = P.hexp;
  g1.hexp_lo = P.hexp + P.cap;
  g1.hblk = P.hblk;
  const uint64_t rows1 = static_cast<uint64_t>(P.E) * 2 * P.I;
  cudaError_t err =
      weight_kind == MOE_WEIGHT_FP8
          ? launch_skinny<MOE_WEIGHT_FP8, true>(g1, P.w13, rows1, max_tiles * g1.n_rt, num_sms, s)
      : weight_kind == MOE_WEIGHT_INT4
          ? launch_skinny<MOE_WEIGHT_INT4, true>(g1, P.w13, rows1, max_tiles * g1.n_rt, num_sms, s)
          : launch_skinny<MOE_WEIGHT_INT8, true>(g1, P.w13, rows1, max_tiles * g1.n_rt, num_sms, s);
  if (err != cudaSuccess) return err;
  hook("decode_gemm1", s);
  const __half* b2 = static_cast<const __half*>(P.h);
  const int n_rt2 = (P.H + dec::Cfg<false, 2>::ROWS - 1) / dec::Cfg<false, 2>::ROWS;
  // INT8 with a GEMM2 of two CTAs per SM (few items, under 6 per SM): GEMM2 quantises h itself from GEMM1's
  // fp32 h and row maxima, and the requant launch goes (measured at one Qwen3 token: 6 us of a 60 us layer)
  const bool rq = weight_kind == MOE_WEIGHT_INT8 && !P.out_direct && max_tiles * n_rt2 < 6LL * num_sms;
  if (weight_kind == MOE_WEIGHT_INT8 && !rq) {
    // padded positions: the slots plus at most B - 1 padding rows for each of at most min(E, slots) experts
    const long long rows = slots + (slots < P.E ? slots : P.E) * (kDecodeBlock - 1);
    err = launch_requant_rows(P.h, P.hmax, P.num_post, rows < P.cap ? static_cast<int>(rows) : P.cap, P.I, P.hq,
                              P.sh, num_sms, s);
    if (err != cudaSuccess) return err;
    hook("requant_h", s);
    b2 = P.hq;
  }
  SkinnyArgs g2{};
  g2.K = P.I;
  g2.rows_per_expert = P.H;
  g2.up_offset = 0;
  g2.n_rt = n_rt2;
  g2.ttiles = P.ttiles;
  g2.num_ttiles = P.num_ttiles;
  g2.wscale = P.s2;
  g2.sorted_ids = P.sorted_ids;
  g2.topk = P.topk;
  g2.b = b2;
  g2.sh = P.sh;
  g2.topk_w = P.topk_w;
  g2.out = P.y;
  g2.out_ld = P.H;
  g2.status = P.status;
  g2.out_bf16 = P.out_direct;
  g2.hexp = P.hexp;
  g2.hexp_lo = P.hexp + P.cap;
  g2.hblk = P.hblk;
  if (rq) {
    g2.bh = static_cast<const float*>(P.h);
    g2.hmax = P.hmax;
  }
  const uint64_t rows2 = static_cast<uint64_t>(P.E) * P.H;
  err = weight_kind == MOE_WEIGHT_FP8
            ? launch_skinny<MOE_WEIGHT_FP8, false>(g2, P.w2, rows2, max_tiles * g2.n_rt, num_sms, s)
        : weight_kind == MOE_WEIGHT_INT4
            ? launch_skinny<MOE_WEIGHT_INT4, false>(g2, P.w2, rows2, max_tiles * g2.n_rt, num_sms, s)
            : launch_skinny<MOE_WEIGHT_INT8, false>(g2, P.w2, rows2, max_tiles * g2.n_rt, num_sms, s);
  if (err != cudaSuccess) return err;
  hook("decode_gemm2", s);
  if (P.out_direct) return cudaSuccess;  // masked layout: GEMM2 wrote the output rows
  err = launch_combine(P.y, P.inv_pos, P.M, P.topk, P.H, P.out, num_sms, s);
  if (err != cudaSuccess) return err;
  hook("combine", s);
  return cudaSuccess;
}

}  // namespace gbmoe
