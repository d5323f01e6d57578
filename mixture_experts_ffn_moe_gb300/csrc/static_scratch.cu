// fused_moe_fp8_static_scratch: the FP8 layer for callers that cannot allocate
// device memory.
//
// Some callers hold only raw input and output pointers and have no device
// allocator they are allowed to use: a plugin whose host framework owns every
// device buffer, a C caller that links this library but not an allocator, or
// a latency-critical loop that must not pay for cudaMalloc / cudaFree and the
// device-wide synchronisation they can cause.  For them this entry point runs
// exactly the kernels of fused_moe_fp8, with its scratch taken from a fixed
// buffer that lives in this file instead of a caller-supplied workspace.
//
// The buffer is a file-scope __device__ array of MOE_STATIC_SCRATCH_BYTES.
// Every device on which this entry point runs holds it from the first such
// call until the process exits.  Host code cannot use the array's name as a
// device address (on the host it names a stand-in object), so the first call
// on each device, with that device current, looks the address up with
// cudaGetSymbolAddress; make that first call before any stream capture.  The
// address is kept with the id of the CUDA context it was taken in: after a
// device reset the next call on that device finds a new context and looks
// the address up again (so that call, too, must come before any capture).
//
// All calls share the one buffer and it keeps the previous call's contents.
// The kernels clear everything that must start at zero (the status words and
// the intermediate's frame words) and overwrite everything else they read
// before reading it.  Calls that overlap on the GPU (different streams, or
// several host threads) race on the buffer and must be serialised by the
// caller.  moe_read_static_scratch_status reads the buffer's status words.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "gbmoe.h"
#include "internal.h"

namespace gbmoe {

static __device__ __align__(256) unsigned char g_static_scratch[MOE_STATIC_SCRATCH_BYTES];

constexpr int kMaxScratchDevices = 64;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current CUDA context (0 if it cannot be read).
static unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx && get_id(ctx, &id) == CUDA_SUCCESS)
    return id;
  return 0;
}

// Device address of g_static_scratch on the current device, looked up once per device and context.
static cudaError_t static_scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[kMaxScratchDevices] = {};
  static unsigned long long ctx_of[kMaxScratchDevices] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxScratchDevices) return cudaErrorInvalidDevice;
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr || (ctx != 0 && ctx != ctx_of[dev])) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_static_scratch);
    if (err != cudaSuccess) return err;
    addr[dev] = p;
    ctx_of[dev] = ctx;
  }
  *out = addr[dev];
  return cudaSuccess;
}

}  // namespace gbmoe

extern "C" moe_status_t fused_moe_fp8_static_scratch(const void* x_bf16, const int32_t* topk_ids,
                                                     const float* topk_weights, const void* w13_e4m3,
                                                     const float* w13_scale, const void* w2_e4m3,
                                                     const float* w2_scale, int M, int H, int I, int E, int topk,
                                                     unsigned flags, void* out_bf16, moe_stream_t stream) {
  // the layer's own argument checks first, so a bad call gets their message rather than the size limit's
  moe_status_t st = gbmoe::check_fp8_layer_args(x_bf16, topk_ids, topk_weights, w13_e4m3, w13_scale, w2_e4m3,
                                                w2_scale, M, H, I, E, topk, flags, out_bf16);
  if (st != MOE_OK || M == 0) return st;
  const size_t need = moe_workspace_size(M, H, I, E, topk, MOE_WEIGHT_FP8, flags);
  if (need > MOE_STATIC_SCRATCH_BYTES) {
    return gbmoe::report_error(MOE_ERR_UNSUPPORTED,
                               "fused_moe_fp8_static_scratch: these sizes need " + std::to_string(need) +
                                   " bytes of scratch, more than the " + std::to_string(MOE_STATIC_SCRATCH_BYTES) +
                                   "-byte static buffer (MOE_STATIC_SCRATCH_BYTES); use fused_moe_fp8 with a "
                                   "caller workspace");
  }
  void* scratch = nullptr;
  const cudaError_t err = gbmoe::static_scratch_address(&scratch);
  if (err != cudaSuccess) {
    return gbmoe::report_error(MOE_ERR_CUDA, std::string("fused_moe_fp8_static_scratch: cudaGetSymbolAddress: ") +
                                                 cudaGetErrorString(err));
  }
  return fused_moe_fp8(x_bf16, topk_ids, topk_weights, w13_e4m3, w13_scale, w2_e4m3, w2_scale, M, H, I, E, topk,
                       flags, out_bf16, scratch, MOE_STATIC_SCRATCH_BYTES, stream);
}

extern "C" moe_status_t moe_read_static_scratch_status(int32_t status_out[2], moe_stream_t stream) {
  if (!status_out) return gbmoe::report_error(MOE_ERR_INVALID_ARG, "moe_read_static_scratch_status: NULL pointer");
  void* scratch = nullptr;
  const cudaError_t err = gbmoe::static_scratch_address(&scratch);
  if (err != cudaSuccess) {
    return gbmoe::report_error(MOE_ERR_CUDA, std::string("moe_read_static_scratch_status: cudaGetSymbolAddress: ") +
                                                 cudaGetErrorString(err));
  }
  return moe_read_status(scratch, status_out, stream);
}
