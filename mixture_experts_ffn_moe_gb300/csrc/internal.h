// Internal interfaces between the C-ABI front end and the kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <string>

#include "gbmoe.h"

namespace gbmoe {

struct DeviceStatus;

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
  int kind;                // 0 none, 1 bf16 -> fp16, 2 per-row int8 quantisation
  void* q;                 // [M, H] fp16 (kinds 1, 2 in the prologue) or int8 (quant entry)
  float* scale;            // [M] (kind 2)
  uint32_t* zero_words;    // words to clear (may be null)
  int n_zero;
};

// Decode (weight-streaming) path.
struct DecodeArgs {
  int M, H, I, E, topk;
  const __half* xq;             // [M, H] fp16 activations (or int8 codes as fp16)
  const float* sx;              // [M] per-row activation scale (INT8 path)
  const uint8_t* w13;           // [E, 2I, H] codes
  const float* s13;             // FP8 [E, 2I/128, H/128]; INT8 [E, 2I]
  const uint8_t* w2;            // [E, H, I] codes
  const float* s2;              // FP8 [E, H/128, I/128]; INT8 [E, H]
  const float* topk_w;          // [M, topk]
  const int32_t* sorted_ids;    // [cap]
  const int32_t* offsets;       // [E + 1]
  const int32_t* counts;        // [E]
  const int32_t* active;        // [E]
  const int32_t* num_active;    // [1]
  const int32_t* num_post;      // [1]
  int cap;
  void* h;                      // FP8: fp16 [cap, I]; INT8: fp32 [cap, I]
  uint32_t* hmax;               // INT8: [cap] bits of max |h| per row
  __half* hq;                   // INT8: [cap, I] requantised codes as fp16
  float* sh;                    // INT8: [cap] per-row scale of hq
  __nv_bfloat16* out;           // [M, H]
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
  void* out;             // GEMM1: h (fp16 FP8 path / fp32 INT8 path); GEMM2: y fp32 (weighted)
  int out_ld;
  uint32_t* hmax;        // INT8 GEMM1: per-position max |h| (bits)
  DeviceStatus* status;
};

// Everything the prefill launcher needs (host view of one call).
struct PrefillPlan {
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
  __half* act;           // [cap, H] gathered activations
  void* h;               // [cap, I]
  uint32_t* hmax;        // INT8
  __half* hq;            // INT8
  float* sh;             // INT8
  float* y;              // [cap, H]
  __nv_bfloat16* out;
  DeviceStatus* status;
};

size_t align_smem_bytes(int E);
cudaError_t launch_prologue(const AlignArgs& a, const PrepArgs& p, int prep_ctas, cudaStream_t s);
cudaError_t launch_quant_rows_s8(const PrepArgs& p, cudaStream_t s);
cudaError_t launch_decode(const DecodeArgs& d, int weight_kind, int num_sms, cudaStream_t s, const StageHook& hook);
size_t decode_gemm2_smem_bytes(int M);
cudaError_t launch_prefill(const PrefillPlan& P, int weight_kind, int num_sms, cudaStream_t s, const StageHook& hook);
cudaError_t launch_requant_rows(const void* h, const uint32_t* hmax, const int32_t* num_post, int cap, int I,
                                __half* hq, float* sh, int num_sms, cudaStream_t s);
size_t prefill_smem_bytes();

// Records `msg` as the calling thread's last error (moe_last_error) and returns `st`.
moe_status_t report_error(moe_status_t st, const std::string& msg);

// Sets a kernel's dynamic shared memory limit once per device.
cudaError_t set_smem_limit_once(const void* func, int bytes, int slot);

}  // namespace gbmoe
