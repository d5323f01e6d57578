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

size_t align_smem_bytes(int E);
cudaError_t launch_prologue(const AlignArgs& a, const PrepArgs& p, int prep_ctas, cudaStream_t s);
cudaError_t launch_quant_rows_s8(const PrepArgs& p, cudaStream_t s);
cudaError_t launch_decode(const DecodeArgs& d, int weight_kind, int num_sms, cudaStream_t s, const StageHook& hook);
size_t decode_gemm2_smem_bytes(int M);

// Records `msg` as the calling thread's last error (moe_last_error) and returns `st`.
moe_status_t report_error(moe_status_t st, const std::string& msg);

// Sets a kernel's dynamic shared memory limit once per device.
cudaError_t set_smem_limit_once(const void* func, int bytes, int slot);

}  // namespace gbmoe
