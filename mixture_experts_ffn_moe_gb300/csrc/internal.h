// Internal interfaces between the C-ABI front end and the kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <string>
#include <utility>

#include "gbmoe.h"

namespace gbmoe {

struct DeviceStatus;
struct GateArgs;

struct AlignArgs {
  const int32_t* topk_ids;
  int M, topk, E, block, cap;
  int32_t* sorted_ids;      // [cap]
  int32_t* expert_ids;      // [cap / block]
  int32_t* num_post;        // [1]
  int32_t* expert_offsets;  // [E + 1]  (may be null)
  int32_t* counts;          // [E]      (may be null)
  int32_t* active;          // [E]      (may be null) ascending ids of experts with slots
  int32_t* num_active;      // [1]      (may be null)
  int32_t* inv_pos;         // [M*topk] (may be null) slot -> position in sorted_ids, -1 if dropped
  int4* ttiles;             // (may be null) token tiles {expert, first position, count, 0}
  int32_t* num_ttiles;      // [1]
  int tile_tokens;          // slots per token tile
  DeviceStatus* status;     // may be null
};

struct PrepArgs {
  const __nv_bfloat16* x;  // [M, H]
  int M, H;
  int kind;                // 0 none, 1 bf16 -> fp16, 2 per-row int8, 3 FP8 E4M3 per 1x128 group,
                           // 4 bf16 -> fp16 in the INT4 K order, 5 two-term E4M3 per 1x128 group
  void* q;                 // [M, H] fp16 (kinds 1, 2 in the prologue), int8 (quant entry) or E4M3 codes (kind 3)
  float* scale;            // [M] (kind 2) or [M, H/128] (kind 3)
  uint32_t* zero_words;    // words to clear (may be null)
  int n_zero;
};

// Called after each kernel of a fused call (per-kernel timing); may be empty.
struct StageHook {
  void (*fn)(void* ctx, const char* stage, cudaStream_t s) = nullptr;
  void* ctx = nullptr;
  void operator()(const char* stage, cudaStream_t s) const {
    if (fn) fn(ctx, stage, s);
  }
};

// One tcgen05 grouped GEMM of the prefill path (device view).
struct PrefillArgs {
  int K;                 // reduction length: H (GEMM1) or I (GEMM2)
  int rows_per_expert;   // weight rows of one expert: 2I (GEMM1) or H (GEMM2)
  int up_offset;         // row offset of the up half inside an expert (GEMM1), else 0
  int n_tiles;           // 128-row output tiles per expert
  const int4* ttiles;    // token tiles {expert, first position, count, 0}
  const int32_t* num_ttiles;
  const float* wscale;   // FP8: [E, rows/128, K/128] block scales; INT8: [E, rows] channel scales
  const int32_t* sorted_ids;
  int topk;
  const float* sx;       // INT8 GEMM1: per-token activation scale
  const float* sh;       // INT8 GEMM2: per-position scale of the requantised h
  const float* topk_w;   // GEMM2: routing weights per slot
  void* out;             // GEMM1: h by position (fp16 FP8 / fp32 INT8); GEMM2: y bf16 by slot (weighted)
  int out_ld;
  uint32_t* hmax;        // INT8 GEMM1: per-position max |h| (bits)
  DeviceStatus* status;
  __nv_bfloat16* out_bf16;  // GEMM2: if set, bf16 output rows out_bf16[slot] (unweighted), not y
  // power-of-two frames of the fp16 operands (FP8 and INT4 weights)
  int x_by_pos;          // GEMM1: sx is indexed by position (masked layout), else by token
  uint32_t* hexp;        // GEMM1: per position, the largest biased frame exponent of its h blocks (atomicMax)
  uint8_t* hblk;         // GEMM1: [cap, I/32] biased frame exponent each 32-column block of h was stored with
  const float* hsc;      // GEMM2: per position, 2^e of the row frame h was brought to
};

// Everything the path launchers need (host view of one call).
struct LayerPlan {
  int M, H, I, E, topk, cap;
  const __half* xq;
  const float* sx;
  const uint8_t* w13;
  const float* s13;
  const uint8_t* w2;
  const float* s2;
  const float* topk_w;
  const int32_t* sorted_ids;
  const int32_t* num_post;
  const int32_t* inv_pos;
  const int4* ttiles;
  const int32_t* num_ttiles;
  __half* act;           // [cap, H] gathered activations (prefill path)
  void* h;               // [cap, I]
  uint32_t* hmax;        // INT8
  __half* hq;            // INT8
  float* sh;             // INT8
  float* y;              // [M*topk, H] weighted expert outputs by slot
  __nv_bfloat16* out;
  DeviceStatus* status;
  // FP8-operand prefill (MOE_ACT_FP8_1X128, and the FP8 weight-only layer's two-term form)
  int e4m3_terms;        // 1: E4M3 activations; 2: x and h as two E4M3 terms (hi rows, then lo rows)
  const uint8_t* xq8;    // [terms * M, H] E4M3 codes of x
  const float* sx8;      // [M, H/128] their scales
  uint8_t* act8;         // [terms * cap, H] gathered codes by position
  float* sa8;            // [H/128, cap] gathered scales, transposed
  uint8_t* h8;           // [terms * cap, I] E4M3 codes of h by position
  float* sh8;            // [I/128, cap] their scales, transposed
  // masked layout: GEMM1 reads its activations by position (xq holds them in position
  // order) and GEMM2 writes bf16 rows straight to out_direct[sorted_ids[pos]], unweighted;
  // there is no combine
  __nv_bfloat16* out_direct;
  // power-of-two frames of the fp16 operands (FP8 and INT4 weights): sx holds 2^e of every x row
  // (by token, or by position on the masked layout); GEMM1 stores h blocks in their own frames
  uint32_t* hexp;        // [2 cap] largest biased block exponent of each position, then 256 - the smallest
                         // nonzero one (decode path); zeroed by the prologue
  uint8_t* hblk;         // [cap, I/32] biased exponent of each 32-column block of h
  float* hsc;            // [cap] tcgen05 path: 2^e of the row frame after the frame pass
  bool x_by_pos;         // masked layout: sx by position
};

// One skinny grouped GEMM of the decode path (device view).
struct SkinnyArgs {
  int K;                 // reduction length: H (GEMM1) or I (GEMM2)
  int rows_per_expert;   // weight rows of one expert: 2I (GEMM1) or H (GEMM2)
  int up_offset;         // row offset of the up half inside an expert (GEMM1), else 0
  int n_rt;              // 64-row tiles per expert (64 gate + 64 up rows for GEMM1)
  const int4* ttiles;    // token tiles {expert, first position, count <= 8, 0}
  const int32_t* num_ttiles;
  const float* wscale;   // FP8: [E, rows/128, K/128]; INT8: [E, rows]
  const int32_t* sorted_ids;
  int topk;
  const __half* b;       // B operand rows: GEMM1 prepared x [M, H] (by token); GEMM2 h [cap, I] (by position)
  const float* sx;       // INT8 GEMM1: per-token activation scale
  const float* sh;       // INT8 GEMM2: per-position scale of the requantised h
  const float* topk_w;   // GEMM2: routing weights per slot
  void* out;             // GEMM1: h by position (fp16 FP8 / fp32 INT8); GEMM2: y fp32 by slot (weighted)
  int out_ld;
  uint32_t* hmax;        // INT8 GEMM1: per-position max |h| (bits); INT8 GEMM2 with bh: read, to quantise h
  const float* bh;       // INT8 GEMM2 quantising h itself: GEMM1's fp32 h [cap, I] by position (else null)
  DeviceStatus* status;
  int b_by_pos;          // GEMM1: activation rows by position (masked layout), not by token
  __nv_bfloat16* out_bf16;  // GEMM2: if set, bf16 output rows out_bf16[slot] (unweighted), not y
  // power-of-two frames of the fp16 operands (FP8 and INT4 weights): GEMM1 takes x's row frames from sx
  // and writes h's block frames; GEMM2 reads them
  uint32_t* hexp;        // per position, the largest biased frame exponent of its h blocks
  uint32_t* hexp_lo;     // per position, 256 - the smallest nonzero one (0: none)
  uint8_t* hblk;         // [cap, I/32] biased frame exponent of each 32-column block of h
};

size_t align_smem_bytes(int E);

// Alignment of more than kAlignChunkSlots slots runs split over consecutive
// chunks of slots, one CTA each (at most kAlignMaxChunks), which needs a
// workspace of kAlignMaxChunks * E ints for the chunks' histograms.
constexpr int kAlignChunkSlots = 4096;
constexpr int kAlignMaxChunks = 64;
__host__ __device__ inline int align_num_chunks(long long n) {
  if (n <= kAlignChunkSlots) return 1;
  const long long c = (n + kAlignChunkSlots - 1) / kAlignChunkSlots;
  return c < kAlignMaxChunks ? static_cast<int>(c) : kAlignMaxChunks;
}
__host__ __device__ inline int align_chunk_slots(int n, int nchunks) { return (n + nchunks - 1) / nchunks; }

// inline_gate (may be null; at most 256 experts): rank the tokens' experts in
// the alignment CTA before aligning; a.topk_ids must then be inline_gate->ids.
// chunk_counts (may be null: one CTA aligns): kAlignMaxChunks * E ints of
// scratch, used when the slots need more than one chunk.  A split alignment is
// two launches (the second one a single-purpose scatter kernel).
cudaError_t launch_prologue(const AlignArgs& a, const PrepArgs& p, int prep_ctas, cudaStream_t s,
                            const GateArgs* inline_gate = nullptr, int* chunk_counts = nullptr);
cudaError_t launch_gate(const GateArgs& g, int num_sms, cudaStream_t s);

// Masked layout: from masked_m [E] (clamped to [0, cap]) builds the token tiles of
// every expert's rows (positions: each expert's rows padded to a multiple of
// `block`; tiles of up to `tile` rows), sorted_ids[pos] = e * cap + i, and the
// prepared activations xq [positions, H] (kind 1: fp16; kind 4: fp16 in the INT4
// K order).  Decode path: block = tile = 8; tcgen05 path: block 16, tile 128.
struct MaskedArgs {
  const __nv_bfloat16* x;   // [E * cap, H]
  const int32_t* masked_m;  // [E]
  int E, cap, H, kind, block, tile;
  __half* xq;               // [E * round16(cap), H]  x * 2^-e per row (frame of the row's max |x|)
  float* xs;                // [E * round16(cap)]     2^e of each position's row
  uint32_t* zero_words;     // words to clear (the intermediate's frame words)
  int n_zero;
  int32_t* sorted_ids;      // [E * round16(cap)]
  int4* ttiles;             // [E * ceil(cap / tile)]
  int32_t* num_ttiles;
  int32_t* num_post;
  DeviceStatus* status;
  // kind 5 (FP8 weights on the tcgen05 path): x in its two-term E4M3 form by position instead of xq/xs
  uint8_t* act8;            // [2 * pcap, H] hi codes in row pos, lo codes in row pcap + pos
  float* sa8;               // [H / 128, pcap] 2^e of each (position, 128-column group)
  int pcap;                 // positions: E * round16(cap)
};
cudaError_t launch_masked_prologue(const MaskedArgs& m, int num_sms, cudaStream_t s);
cudaError_t launch_wait_timeout(DeviceStatus* status, long long limit, int32_t* gave_up, cudaStream_t s);
cudaError_t launch_quant_rows(const PrepArgs& p, cudaStream_t s);
cudaError_t launch_decode(const LayerPlan& P, int weight_kind, int num_sms, cudaStream_t s, const StageHook& hook);
cudaError_t launch_prefill(const LayerPlan& P, int weight_kind, int num_sms, cudaStream_t s, const StageHook& hook);
cudaError_t launch_prefill_a8(const LayerPlan& P, int num_sms, cudaStream_t s, const StageHook& hook);
cudaError_t launch_combine(const float* y, const int32_t* inv_pos, int M, int topk, int H, __nv_bfloat16* out,
                           int num_sms, cudaStream_t s);
// y in bf16 (the FP8-activation path)
cudaError_t launch_combine(const __nv_bfloat16* y, const int32_t* inv_pos, int M, int topk, int H,
                           __nv_bfloat16* out, int num_sms, cudaStream_t s);
// 2D row-major tensor [outer, inner] of `esize`-byte elements, TMA box [box_outer, box_inner].
bool encode_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, uint64_t inner,
                    uint64_t outer, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw);
cudaError_t launch_requant_rows(const void* h, const uint32_t* hmax, const int32_t* num_post, int cap, int I,
                                __half* hq, float* sh, int num_sms, cudaStream_t s);
// tcgen05 path, FP8 and INT4 weights: brings every position's h blocks to the row frame (the largest
// block exponent) in place and writes hsc[pos] = 2^e of that frame.
cudaError_t launch_h_frame(__half* h, const uint32_t* hexp, const uint8_t* hblk, const int32_t* num_post, int cap,
                           int I, float* hsc, int num_sms, cudaStream_t s);
size_t prefill_smem_bytes();

// The host-side argument checks of fused_moe_fp8 (sizes, flags, NULL pointers), without the workspace:
// MOE_OK or the status fused_moe_fp8 would return, with its message.
moe_status_t check_fp8_layer_args(const void* x, const int32_t* ids, const float* tw, const void* w13,
                                  const float* s13, const void* w2, const float* s2, int M, int H, int I, int E,
                                  int topk, unsigned flags, const void* out);

// Records `msg` as the calling thread's last error (moe_last_error) and returns `st`.
moe_status_t report_error(moe_status_t st, const std::string& msg);

// Launches `kern` on `s`; with pdl the launch may overlap the previous kernel in
// the stream (the kernel then calls pdl_wait() before reading its outputs).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                          Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Sets a kernel's dynamic shared memory limit once per device (and size).
cudaError_t set_smem_limit_once(const void* func, int bytes);

}  // namespace gbmoe
