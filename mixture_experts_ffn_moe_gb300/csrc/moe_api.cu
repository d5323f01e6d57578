// C-ABI front end: argument checks, workspace carving, path choice, status.
#include <cuda_runtime.h>

#include <mutex>
#include <set>
#include <string>
#include <tuple>
#include <vector>

#include "common.cuh"
#include "gate.cuh"
#include "internal.h"

namespace gbmoe {

static thread_local std::string g_last_error;

static moe_status_t fail(moe_status_t st, const std::string& msg) {
  g_last_error = msg;
  return st;
}

static moe_status_t cuda_fail(cudaError_t err, const char* where) {
  return fail(MOE_ERR_CUDA, std::string(where) + ": " + cudaGetErrorString(err));
}

moe_status_t report_error(moe_status_t st, const std::string& msg) { return fail(st, msg); }

constexpr int kMaxDevices = 64;

cudaError_t set_smem_limit_once(const void* func, int bytes) {
  static std::mutex mu;
  static std::set<std::tuple<int, const void*, int>> done;  // (device, kernel, bytes) already set
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_tuple(dev, func, bytes);
  if (done.count(key)) return cudaSuccess;
  err = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (err == cudaSuccess) done.insert(key);
  return err;
}

static int num_sms_current() {
  static std::mutex mu;
  static int cache[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

// ------------------------------------------------------------------ per-kernel timing
struct Profiler {
  std::vector<cudaEvent_t> events;
  std::vector<const char*> names;  // stage name of each recorded event (nullptr = call start)
  int max_calls = 0, calls = 0;
  size_t used = 0;
  bool recording_call = false;
};
static thread_local Profiler g_prof;

static void prof_record(void*, const char* stage, cudaStream_t s) {
  Profiler& P = g_prof;
  if (!P.recording_call || P.used >= P.events.size()) { P.recording_call = false; return; }
  cudaEventRecord(P.events[P.used], s);
  P.names[P.used] = stage;
  ++P.used;
}

static StageHook prof_begin_call(cudaStream_t s) {
  Profiler& P = g_prof;
  StageHook h;
  if (P.max_calls <= 0 || P.calls >= P.max_calls) return h;
  P.recording_call = true;
  prof_record(nullptr, nullptr, s);
  ++P.calls;
  h.fn = prof_record;
  return h;
}

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

static size_t max_padded(int M, int topk, int E, int B) {
  const size_t n = static_cast<size_t>(M) * topk + static_cast<size_t>(E) * (B - 1);
  return align_up(n, static_cast<size_t>(B));
}

// Offsets (bytes) of every buffer inside a fused-call workspace.
struct Layout {
  int path = 0, B = 0;
  size_t cap = 0;
  size_t status = 0, sorted = 0, expert_ids = 0, offsets = 0, counts = 0, active = 0, scalars = 0,
         inv_pos = 0, xq = 0, sx = 0, h = 0, hmax = 0, hq = 0, sh = 0, ttiles = 0, act = 0, sa = 0, y = 0,
         chunk_counts = 0, hexp = 0, hblk = 0, hsc = 0, total = 0;
  int align_chunks = 1;  // CTAs of the alignment (more than one: split over chunks of slots)
  bool a8 = false;
  int terms = 0;  // FP8-operand tcgen05 kernels: 1 (E4M3 activations), 2 (two-term form of bf16 x / fp32 h)
  size_t max_ttiles = 0;
  int tile_tokens = 0;
};

static int choose_path(int M, int kind, unsigned flags) {
  const unsigned p = flags & MOE_PATH_MASK;
  if (p == MOE_PATH_DECODE || p == MOE_PATH_PREFILL) return static_cast<int>(p);
  if (flags & MOE_ACT_FP8_1X128) return MOE_PATH_PREFILL;  // the FP8 x FP8 products run on tcgen05 only
  // measured crossover (A/B on GB300): the weight-streaming kernels win at 96 tokens (DeepSeek-R1 FP8 3%, Qwen3
  // INT8 14%), the tcgen05 kernels at 128 (3% and 7%); INT4 keeps the weight-streaming kernels up to 128
  if (kind == MOE_WEIGHT_INT4) return M <= MOE_MAX_DECODE_TOKENS ? MOE_PATH_DECODE : MOE_PATH_PREFILL;
  return M < MOE_AUTO_PREFILL_TOKENS ? MOE_PATH_DECODE : MOE_PATH_PREFILL;
}

static Layout plan(int M, int H, int I, int E, int topk, int kind, unsigned flags) {
  Layout L;
  L.path = choose_path(M, kind, flags);
  L.B = L.path == MOE_PATH_PREFILL ? kPrefillBlock : kDecodeBlock;
  L.cap = max_padded(M, topk, E, L.B);
  size_t o = 0;
  auto take = [&](size_t bytes) { const size_t at = o; o = align_up(o + bytes, 256); return at; };
  L.status = take(kStatusBytes);
  L.sorted = take(L.cap * 4);
  L.expert_ids = take(L.cap / L.B * 4);
  L.offsets = take((static_cast<size_t>(E) + 1) * 4);
  L.counts = take(static_cast<size_t>(E) * 4);
  L.active = take(static_cast<size_t>(E) * 4);
  L.scalars = take(16);
  L.inv_pos = take(static_cast<size_t>(M) * topk * 4);
  L.align_chunks = align_num_chunks(static_cast<long long>(M) * topk);
  if (L.align_chunks > 1) L.chunk_counts = take(static_cast<size_t>(kAlignMaxChunks) * E * 4);
  L.a8 = kind == MOE_WEIGHT_FP8 && (flags & MOE_ACT_FP8_1X128);
  // FP8 weights on the tcgen05 path run on the FP8 tensor cores: E4M3 activations (A8), or for the
  // weight-only layer x and h in their two-term E4M3 form
  L.terms = L.a8 ? 1 : (kind == MOE_WEIGHT_FP8 && L.path == MOE_PATH_PREFILL) ? 2 : 0;
  L.tile_tokens = L.path == MOE_PATH_PREFILL ? kPrefillTileTokens : kDecodeBlock;
  L.max_ttiles = static_cast<size_t>(E) + static_cast<size_t>(M) * topk / L.tile_tokens + 1;
  if (L.terms) {
    // E4M3 codes (per term) with 1 x 128 scales; scales of gathered rows are stored transposed [K/128, cap]
    L.xq = take(static_cast<size_t>(L.terms) * M * H);
    L.sx = take(static_cast<size_t>(M) * (H / kQBlock) * 4);
    L.h = take(L.terms * L.cap * I);
    L.sh = take(L.cap * (I / kQBlock) * 4);
    L.ttiles = take(L.max_ttiles * 16);
    L.act = take(L.terms * L.cap * H);
    L.sa = take(L.cap * (H / kQBlock) * 4);
    L.y = take(static_cast<size_t>(M) * topk * H * 2);  // bf16 y
    L.total = o;
    return L;
  }
  L.xq = take(static_cast<size_t>(M) * H * 2);
  L.sx = take(static_cast<size_t>(M) * 4);
  if (kind != MOE_WEIGHT_INT8) {
    L.h = take(L.cap * I * 2);  // fp16 h (FP8, INT4), each 32-column block in its power-of-two frame
    L.hexp = take(L.cap * 8);   // largest and smallest block exponent per position (cleared by the prologue)
    L.hblk = take(L.cap * (I / kHBlock));
    if (L.path == MOE_PATH_PREFILL) L.hsc = take(L.cap * 4);
  } else {
    L.h = take(L.cap * I * 4);
    L.hmax = take(L.cap * 4);
    L.hq = take(L.cap * I * 2);
    L.sh = take(L.cap * 4);
  }
  L.ttiles = take(L.max_ttiles * 16);
  if (L.path == MOE_PATH_PREFILL) L.act = take(L.cap * H * 2);
  L.y = take(static_cast<size_t>(M) * topk * H * (L.path == MOE_PATH_PREFILL ? 2 : 4));  // bf16 / fp32 y
  L.total = o;
  return L;
}

static bool known_kind(int kind) {
  return kind == MOE_WEIGHT_FP8 || kind == MOE_WEIGHT_INT8 || kind == MOE_WEIGHT_INT4;
}

static bool known_flags(int kind, unsigned flags) {
  const unsigned allowed = MOE_PATH_MASK | (kind == MOE_WEIGHT_FP8 ? MOE_ACT_FP8_1X128 : 0u);
  return (flags & ~allowed) == 0;
}

static moe_status_t check_layer_args(int kind, const void* x, const void* ids, const void* tw, const void* w13,
                                     const void* s13, const void* w2, const void* s2, int M, int H, int I,
                                     int E, int topk, unsigned flags, const void* out) {
  if (M < 0 || H <= 0 || I <= 0 || E <= 0 || topk <= 0)
    return fail(MOE_ERR_INVALID_ARG, "sizes must be positive (M >= 0)");
  if (topk > 32) return fail(MOE_ERR_UNSUPPORTED, "topk > 32");
  if (E > MOE_MAX_EXPERTS) return fail(MOE_ERR_UNSUPPORTED, "more than MOE_MAX_EXPERTS experts");
  if (H % kQBlock || I % kQBlock) return fail(MOE_ERR_UNSUPPORTED, "H and I must be multiples of 128");
  if (!known_flags(kind, flags)) return fail(MOE_ERR_INVALID_ARG, "unknown flag bits for this weight kind");
  if ((flags & MOE_PATH_MASK) == MOE_PATH_MASK) return fail(MOE_ERR_INVALID_ARG, "both path flags set");
  if ((flags & MOE_ACT_FP8_1X128) && (flags & MOE_PATH_MASK) == MOE_PATH_DECODE)
    return fail(MOE_ERR_UNSUPPORTED, "MOE_ACT_FP8_1X128 runs on the tcgen05 (prefill) path only");
  if (static_cast<long long>(M) * topk > (1LL << 30) || static_cast<long long>(M) * H > (1LL << 40))
    return fail(MOE_ERR_UNSUPPORTED, "problem too large");
  if (M == 0) return MOE_OK;
  if (!x || !ids || !tw || !w13 || !s13 || !w2 || !s2 || !out) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  const int path = choose_path(M, kind, flags);
  if (path == MOE_PATH_DECODE && M > MOE_MAX_DECODE_TOKENS && kind != MOE_WEIGHT_INT4)
    return fail(MOE_ERR_UNSUPPORTED, "decode path takes at most MOE_MAX_DECODE_TOKENS tokens");
  return MOE_OK;
}

moe_status_t check_fp8_layer_args(const void* x, const int32_t* ids, const float* tw, const void* w13,
                                  const float* s13, const void* w2, const float* s2, int M, int H, int I, int E,
                                  int topk, unsigned flags, const void* out) {
  g_last_error.clear();
  return check_layer_args(MOE_WEIGHT_FP8, x, ids, tw, w13, s13, w2, s2, M, H, I, E, topk, flags, out);
}

template <typename T>
static T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}

// Checks a gating request over E routed experts and fills the kernel arguments
// (all but ids / w).
static moe_status_t check_gate(const float* logits, int M, int E, int topk, const moe_gate_config_t* gate,
                               GateArgs& g) {
  if (!gate) return fail(MOE_ERR_INVALID_ARG, "gate config is NULL");
  if (M < 0 || E <= 0 || topk <= 0) return fail(MOE_ERR_INVALID_ARG, "sizes must be positive (M >= 0)");
  if (E > MOE_MAX_EXPERTS) return fail(MOE_ERR_UNSUPPORTED, "more than MOE_MAX_EXPERTS experts");
  if (gate->shared_expert != 0 && gate->shared_expert != 1)
    return fail(MOE_ERR_INVALID_ARG, "shared_expert must be 0 or 1");
  if (topk > E) return fail(MOE_ERR_INVALID_ARG, "topk > E");
  if (topk + gate->shared_expert > 32) return fail(MOE_ERR_UNSUPPORTED, "topk + shared_expert > 32");
  if (gate->scoring == MOE_GATE_SOFTMAX) {
    if (gate->n_group != 1 || gate->topk_group != 1 || gate->routed_scaling != 1.0f || gate->bias)
      return fail(MOE_ERR_INVALID_ARG, "softmax gating takes n_group = topk_group = 1, scaling 1, no bias");
  } else if (gate->scoring == MOE_GATE_SIGMOID_GROUPED) {
    if (gate->n_group < 1 || gate->n_group > 32 || E % gate->n_group)
      return fail(MOE_ERR_INVALID_ARG, "n_group must lie in 1..32 and divide E");
    if (gate->topk_group < 1 || gate->topk_group > gate->n_group)
      return fail(MOE_ERR_INVALID_ARG, "topk_group must lie in 1..n_group");
    if (topk > gate->topk_group * (E / gate->n_group))
      return fail(MOE_ERR_INVALID_ARG, "topk exceeds the experts of the kept groups");
    if (!(gate->routed_scaling > 0.0f) || gate->routed_scaling > 3.0e38f)
      return fail(MOE_ERR_INVALID_ARG, "routed_scaling must be positive and finite");
  } else {
    return fail(MOE_ERR_INVALID_ARG, "unknown gate scoring");
  }
  if (M > 0 && !logits) return fail(MOE_ERR_INVALID_ARG, "NULL logits");
  g = GateArgs{};
  g.logits = logits;
  g.bias = gate->bias;
  g.M = M; g.E = E; g.topk = topk; g.ld = topk + gate->shared_expert;
  g.scoring = gate->scoring;
  g.n_group = gate->n_group; g.topk_group = gate->topk_group;
  g.scale = gate->routed_scaling;
  g.shared = gate->shared_expert;
  g.vec_ok = (E % 4 == 0 && reinterpret_cast<uintptr_t>(logits) % 16 == 0) ? 1 : 0;
  return MOE_OK;
}

// gate (may be null): the ids / weights are first written by the router gating
// (gate->ids == ids, gate->w == tw), inside the prologue for small calls.
static moe_status_t fused_impl(int kind, const void* x, const int32_t* ids, const float* tw, const void* w13,
                               const float* s13, const void* w2, const float* s2, int M, int H, int I, int E,
                               int topk, unsigned flags, void* out, void* ws, size_t ws_bytes,
                               cudaStream_t stream, const GateArgs* gate = nullptr) {
  if (!gate) g_last_error.clear();
  moe_status_t st = check_layer_args(kind, x, ids, tw, w13, s13, w2, s2, M, H, I, E, topk, flags, out);
  if (st != MOE_OK || M == 0) return st;
  const Layout L = plan(M, H, I, E, topk, kind, flags);
  if (!ws) return fail(MOE_ERR_WORKSPACE, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(ws) % 256) return fail(MOE_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (ws_bytes < L.total) return fail(MOE_ERR_WORKSPACE, "workspace smaller than moe_workspace_size()");
  if (reinterpret_cast<uintptr_t>(x) % 16 || reinterpret_cast<uintptr_t>(w13) % 16 ||
      reinterpret_cast<uintptr_t>(w2) % 16 || reinterpret_cast<uintptr_t>(out) % 4)
    return fail(MOE_ERR_INVALID_ARG, "x, w13 and w2 must be 16-byte aligned, out 4-byte aligned");
  const int sms = num_sms_current();
  if (sms <= 0) return fail(MOE_ERR_CUDA, "cannot query the current device");

  AlignArgs a{};
  a.topk_ids = ids;
  a.M = M; a.topk = topk; a.E = E; a.block = L.B; a.cap = static_cast<int>(L.cap);
  a.sorted_ids = at<int32_t>(ws, L.sorted);
  a.expert_ids = at<int32_t>(ws, L.expert_ids);
  a.num_post = at<int32_t>(ws, L.scalars);
  a.num_active = at<int32_t>(ws, L.scalars) + 1;
  a.expert_offsets = at<int32_t>(ws, L.offsets);
  a.counts = at<int32_t>(ws, L.counts);
  a.active = at<int32_t>(ws, L.active);
  a.inv_pos = at<int32_t>(ws, L.inv_pos);
  a.status = at<DeviceStatus>(ws, L.status);
  a.ttiles = at<int4>(ws, L.ttiles);
  a.num_ttiles = at<int32_t>(ws, L.scalars) + 2;
  a.tile_tokens = L.tile_tokens;

  PrepArgs p{};
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.M = M; p.H = H;
  p.kind = L.terms == 1 ? 3 : L.terms == 2 ? 5 : kind == MOE_WEIGHT_FP8 ? 1 : kind == MOE_WEIGHT_INT4 ? 4 : 2;
  p.q = at<void>(ws, L.xq);
  p.scale = at<float>(ws, L.sx);
  if (!L.terms) {  // the intermediate's amax (INT8) or frame exponent (FP8, INT4) per position starts at zero
    p.zero_words = at<uint32_t>(ws, kind == MOE_WEIGHT_INT8 ? L.hmax : L.hexp);
    p.n_zero = static_cast<int>(kind == MOE_WEIGHT_INT8 ? L.cap : 2 * L.cap);
  }
  const bool gate_inline = gate && M <= MOE_GATE_INLINE_TOKENS && gate->E <= 256;
  // one 1024-thread prologue CTA per SM (its register count allows no second one): the
  // alignment CTA(s) -- one when it also ranks the experts -- and the flat activation pass
  const int align_ctas = gate_inline ? 1 : L.align_chunks;
  const int free_sms = sms - align_ctas > 1 ? sms - align_ctas : 1;
  const int prep_ctas = M < free_sms ? (M > 0 ? M : 1) : free_sms;
  const StageHook hook = prof_begin_call(stream);
  cudaError_t err;
  if (gate && !gate_inline) {
    err = launch_gate(*gate, sms, stream);
    if (err != cudaSuccess) return cuda_fail(err, "gate launch");
    hook("gate", stream);
  }
  err = launch_prologue(a, p, prep_ctas, stream, gate_inline ? gate : nullptr,
                        L.align_chunks > 1 ? at<int>(ws, L.chunk_counts) : nullptr);
  if (err != cudaSuccess) return cuda_fail(err, "prologue launch");
  hook(gate_inline ? "prologue_gate_align_prep" : "prologue_align_prep", stream);

  LayerPlan P{};
  P.M = M; P.H = H; P.I = I; P.E = E; P.topk = topk; P.cap = static_cast<int>(L.cap);
  P.xq = at<__half>(ws, L.xq);
  P.sx = at<float>(ws, L.sx);
  P.w13 = static_cast<const uint8_t*>(w13);
  P.s13 = s13;
  P.w2 = static_cast<const uint8_t*>(w2);
  P.s2 = s2;
  P.topk_w = tw;
  P.sorted_ids = a.sorted_ids;
  P.num_post = a.num_post;
  P.inv_pos = a.inv_pos;
  P.ttiles = a.ttiles;
  P.num_ttiles = a.num_ttiles;
  if (L.path == MOE_PATH_PREFILL) P.act = at<__half>(ws, L.act);
  P.h = at<void>(ws, L.h);
  if (kind == MOE_WEIGHT_INT8) {
    P.hmax = at<uint32_t>(ws, L.hmax);
    P.hq = at<__half>(ws, L.hq);
    P.sh = at<float>(ws, L.sh);
  } else if (!L.terms) {
    P.hexp = at<uint32_t>(ws, L.hexp);
    P.hblk = at<uint8_t>(ws, L.hblk);
    if (L.path == MOE_PATH_PREFILL) P.hsc = at<float>(ws, L.hsc);
  }
  P.y = at<float>(ws, L.y);
  P.out = static_cast<__nv_bfloat16*>(out);
  P.status = a.status;
  if (L.terms) {
    P.e4m3_terms = L.terms;
    P.xq8 = at<uint8_t>(ws, L.xq);
    P.sx8 = at<float>(ws, L.sx);
    P.act8 = at<uint8_t>(ws, L.act);
    P.sa8 = at<float>(ws, L.sa);
    P.h8 = at<uint8_t>(ws, L.h);
    P.sh8 = at<float>(ws, L.sh);
    err = launch_prefill_a8(P, sms, stream, hook);
    if (err == cudaErrorInvalidConfiguration)
      return fail(MOE_ERR_CUDA, "FP8 x FP8 kernel was not built with its designed register count");
    if (err != cudaSuccess) return cuda_fail(err, "prefill (FP8 tensor cores) launch");
    return MOE_OK;
  }
  if (L.path == MOE_PATH_PREFILL) {
    err = launch_prefill(P, kind, sms, stream, hook);
    if (err != cudaSuccess) return cuda_fail(err, "prefill launch");
  } else {
    err = launch_decode(P, kind, sms, stream, hook);
    if (err != cudaSuccess) return cuda_fail(err, "decode launch");
  }
  return MOE_OK;
}

// ------------------------------------------------------------------ masked layout
// FP8 weights on the tcgen05 path use the FP8-operand kernels: x's two-term codes (2 x positions x H bytes) take
// xq's space, h's codes (2 x positions x I) h's, h's group frames (positions x I/128 floats) hblk's, and x's
// group frames have sa8.
struct MaskedLayout {
  size_t status = 0, sorted = 0, ttiles = 0, scalars = 0, xq = 0, xs = 0, h = 0, hexp = 0, hblk = 0, hsc = 0,
         sa8 = 0, total = 0;
  size_t positions = 0;
};

static MaskedLayout plan_masked(int E, int cap, int H, int I) {
  MaskedLayout L;
  // positions for either path: rows padded to 16 per expert (8 suffice for the decode kernels)
  const size_t positions = static_cast<size_t>(E) * ((static_cast<size_t>(cap) + 15) / 16 * 16);
  size_t o = 0;
  auto take = [&](size_t bytes) { const size_t at = o; o = align_up(o + bytes, 256); return at; };
  L.status = take(kStatusBytes);
  L.sorted = take(positions * 4);
  L.ttiles = take(static_cast<size_t>(E) * ((cap + 7) / 8) * 16);  // decode tiles (8 rows) outnumber tcgen05 ones
  L.scalars = take(16);
  L.xq = take(positions * H * 2);
  L.xs = take(positions * 4);
  L.h = take(positions * I * 2);
  L.hexp = take(positions * 8);
  L.hblk = take(positions * (I / kHBlock));
  L.hsc = take(positions * 4);
  L.sa8 = take(positions * (H / kQBlock) * 4);
  L.positions = positions;
  L.total = o;
  return L;
}

static moe_status_t masked_impl(int kind, const void* x, const int32_t* masked_m, const void* w13,
                                const float* s13, const void* w2, const float* s2, int E, int cap, int H, int I,
                                unsigned flags, void* out, void* ws, size_t ws_bytes, cudaStream_t stream) {
  g_last_error.clear();
  if (!known_kind(kind)) return fail(MOE_ERR_INVALID_ARG, "unknown weight kind");
  if (kind == MOE_WEIGHT_INT8)
    return fail(MOE_ERR_UNSUPPORTED, "the masked layout takes FP8 or INT4 weights (INT8 needs per-token scales)");
  if (E <= 0 || cap <= 0 || H <= 0 || I <= 0) return fail(MOE_ERR_INVALID_ARG, "sizes must be positive");
  if (E > MOE_MAX_EXPERTS) return fail(MOE_ERR_UNSUPPORTED, "more than MOE_MAX_EXPERTS experts");
  if (H % kQBlock || I % kQBlock) return fail(MOE_ERR_UNSUPPORTED, "H and I must be multiples of 128");
  if (flags & ~MOE_PATH_MASK) return fail(MOE_ERR_INVALID_ARG, "unknown flag bits for the masked layout");
  if ((flags & MOE_PATH_MASK) == MOE_PATH_MASK) return fail(MOE_ERR_INVALID_ARG, "both path flags set");
  // The counts are on the device, so the path is the caller's choice: the weight-streaming kernels
  // (default) suit a few rows per expert, the tcgen05 kernels (MOE_PATH_PREFILL) many.
  const bool tc = (flags & MOE_PATH_MASK) == MOE_PATH_PREFILL;
  if (static_cast<long long>(E) * cap > (1LL << 28)) return fail(MOE_ERR_UNSUPPORTED, "problem too large");
  if (!x || !masked_m || !w13 || !s13 || !w2 || !s2 || !out) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (reinterpret_cast<uintptr_t>(x) % 16 || reinterpret_cast<uintptr_t>(w13) % 16 ||
      reinterpret_cast<uintptr_t>(w2) % 16 || reinterpret_cast<uintptr_t>(out) % 2)
    return fail(MOE_ERR_INVALID_ARG, "x, w13 and w2 must be 16-byte aligned, out 2-byte aligned");
  if (tc && reinterpret_cast<uintptr_t>(out) % 16)  // the tcgen05 epilogue writes 16-byte row pieces
    return fail(MOE_ERR_INVALID_ARG, "out must be 16-byte aligned with MOE_PATH_PREFILL");
  const MaskedLayout L = plan_masked(E, cap, H, I);
  if (!ws) return fail(MOE_ERR_WORKSPACE, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(ws) % 256) return fail(MOE_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (ws_bytes < L.total) return fail(MOE_ERR_WORKSPACE, "workspace smaller than moe_workspace_size_masked()");
  const int sms = num_sms_current();
  if (sms <= 0) return fail(MOE_ERR_CUDA, "cannot query the current device");

  MaskedArgs m{};
  m.x = static_cast<const __nv_bfloat16*>(x);
  m.masked_m = masked_m;
  m.E = E; m.cap = cap; m.H = H;
  // FP8 weights on the tcgen05 path: the FP8-operand kernels with x and h in their two-term E4M3 form
  const bool e4m3 = tc && kind == MOE_WEIGHT_FP8;
  m.kind = e4m3 ? 5 : kind == MOE_WEIGHT_INT4 ? 4 : 1;
  m.block = tc ? kPrefillBlock : kDecodeBlock;
  m.tile = tc ? kPrefillTileTokens : kDecodeBlock;
  m.xq = at<__half>(ws, L.xq);
  m.xs = at<float>(ws, L.xs);
  m.zero_words = at<uint32_t>(ws, L.hexp);
  m.n_zero = e4m3 ? 0 : static_cast<int>(2 * L.positions);  // (the two-term form keeps no frame words)
  m.act8 = at<uint8_t>(ws, L.xq);
  m.sa8 = at<float>(ws, L.sa8);
  m.pcap = static_cast<int>(L.positions);
  m.sorted_ids = at<int32_t>(ws, L.sorted);
  m.ttiles = at<int4>(ws, L.ttiles);
  m.num_ttiles = at<int32_t>(ws, L.scalars);
  m.num_post = at<int32_t>(ws, L.scalars) + 1;
  m.status = at<DeviceStatus>(ws, L.status);
  const StageHook hook = prof_begin_call(stream);
  cudaError_t err = launch_masked_prologue(m, sms, stream);
  if (err != cudaSuccess) return cuda_fail(err, "masked prologue launch");
  hook("masked_prologue", stream);

  LayerPlan P{};
  P.M = E * cap; P.H = H; P.I = I; P.E = E; P.topk = 1;
  P.cap = static_cast<int>(static_cast<size_t>(E) * ((cap + 15) / 16 * 16));
  P.xq = m.xq;
  P.sx = m.xs;
  P.x_by_pos = true;
  P.act = m.xq;  // tcgen05 path: the activation rows, already in position order
  P.w13 = static_cast<const uint8_t*>(w13);
  P.s13 = s13;
  P.w2 = static_cast<const uint8_t*>(w2);
  P.s2 = s2;
  P.sorted_ids = m.sorted_ids;
  P.num_post = m.num_post;
  P.ttiles = m.ttiles;
  P.num_ttiles = m.num_ttiles;
  P.h = at<void>(ws, L.h);
  P.hexp = at<uint32_t>(ws, L.hexp);
  P.hblk = at<uint8_t>(ws, L.hblk);
  P.hsc = at<float>(ws, L.hsc);
  P.status = m.status;
  P.out_direct = static_cast<__nv_bfloat16*>(out);
  if (e4m3) {
    P.e4m3_terms = 2;
    P.act8 = m.act8;
    P.sa8 = m.sa8;
    P.h8 = at<uint8_t>(ws, L.h);
    P.sh8 = at<float>(ws, L.hblk);
    err = launch_prefill_a8(P, sms, stream, hook);
  } else {
    err = tc ? launch_prefill(P, kind, sms, stream, hook) : launch_decode(P, kind, sms, stream, hook);
  }
  if (err != cudaSuccess) return cuda_fail(err, "masked layout launch");
  return MOE_OK;
}

}  // namespace gbmoe

using namespace gbmoe;

extern "C" {

size_t moe_align_max_padded(int M, int topk, int num_experts, int block_size) {
  if (M < 0 || topk <= 0 || num_experts <= 0 || block_size <= 0) return 0;
  return gbmoe::max_padded(M, topk, num_experts, block_size);
}

moe_status_t moe_align_block_size(const int32_t* topk_ids, int M, int topk, int num_experts, int block_size,
                                  int32_t* sorted_ids, int32_t* expert_ids, int32_t* num_tokens_post_padded,
                                  int32_t* expert_offsets, moe_stream_t stream) {
  g_last_error.clear();
  if (M < 0 || topk <= 0 || num_experts <= 0 || block_size <= 0)
    return fail(MOE_ERR_INVALID_ARG, "sizes must be positive (M >= 0)");
  if (num_experts > MOE_MAX_EXPERTS) return fail(MOE_ERR_UNSUPPORTED, "more than MOE_MAX_EXPERTS experts");
  if (block_size > 256) return fail(MOE_ERR_UNSUPPORTED, "block_size > 256");
  if (static_cast<long long>(M) * topk > (1LL << 30)) return fail(MOE_ERR_UNSUPPORTED, "too many slots");
  if ((M > 0 && !topk_ids) || !sorted_ids || !expert_ids || !num_tokens_post_padded)
    return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  AlignArgs a{};
  a.topk_ids = topk_ids;
  a.M = M; a.topk = topk; a.E = num_experts; a.block = block_size;
  a.cap = static_cast<int>(gbmoe::max_padded(M, topk, num_experts, block_size));
  a.sorted_ids = sorted_ids;
  a.expert_ids = expert_ids;
  a.num_post = num_tokens_post_padded;
  a.expert_offsets = expert_offsets;
  PrepArgs p{};
  cudaError_t err = launch_prologue(a, p, 0, reinterpret_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "moe_align_block_size launch");
  return MOE_OK;
}

moe_status_t moe_gate_topk(const float* logits, int M, int E, int topk, const moe_gate_config_t* gate,
                           int32_t* topk_ids, float* topk_weights, moe_stream_t stream) {
  g_last_error.clear();
  GateArgs g;
  moe_status_t st = check_gate(logits, M, E, topk, gate, g);
  if (st != MOE_OK || M == 0) return st;
  if (!topk_ids || !topk_weights) return fail(MOE_ERR_INVALID_ARG, "NULL output pointer");
  g.ids = topk_ids;
  g.w = topk_weights;
  const int sms = num_sms_current();
  if (sms <= 0) return fail(MOE_ERR_CUDA, "cannot query the current device");
  cudaError_t err = launch_gate(g, sms, reinterpret_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "moe_gate_topk launch");
  return MOE_OK;
}

moe_status_t fused_moe_gated(int weight_kind, const void* x_bf16, const float* router_logits,
                             const moe_gate_config_t* gate, const void* w13, const float* w13_scale,
                             const void* w2, const float* w2_scale, int M, int H, int I, int E, int topk,
                             unsigned flags, int32_t* topk_ids, float* topk_weights, void* out_bf16,
                             void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  g_last_error.clear();
  if (!known_kind(weight_kind)) return fail(MOE_ERR_INVALID_ARG, "unknown weight kind");
  GateArgs g;
  moe_status_t st = check_gate(router_logits, M, E, topk, gate, g);
  if (st != MOE_OK) return st;
  g.ids = topk_ids;
  g.w = topk_weights;
  const int sh = gate->shared_expert;
  if (M > 0 && E + sh > MOE_MAX_EXPERTS) return fail(MOE_ERR_UNSUPPORTED, "more than MOE_MAX_EXPERTS experts");
  return fused_impl(weight_kind, x_bf16, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale, M, H, I, E + sh,
                    topk + sh, flags, out_bf16, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream),
                    &g);
}

moe_status_t moe_quant_act_int8(const void* x_bf16, int M, int H, int8_t* q, float* scale, moe_stream_t stream) {
  g_last_error.clear();
  if (M < 0 || H <= 0) return fail(MOE_ERR_INVALID_ARG, "M >= 0 and H > 0 required");
  if (M == 0) return MOE_OK;
  if (!x_bf16 || !q || !scale) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  PrepArgs p{};
  p.x = static_cast<const __nv_bfloat16*>(x_bf16);
  p.M = M; p.H = H; p.kind = 2; p.q = q; p.scale = scale;
  cudaError_t err = launch_quant_rows(p, reinterpret_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "moe_quant_act_int8 launch");
  return MOE_OK;
}

moe_status_t moe_quant_act_fp8(const void* x_bf16, int M, int H, uint8_t* q, float* scale, moe_stream_t stream) {
  g_last_error.clear();
  if (M < 0 || H <= 0) return fail(MOE_ERR_INVALID_ARG, "M >= 0 and H > 0 required");
  if (H % kQBlock) return fail(MOE_ERR_UNSUPPORTED, "H must be a multiple of 128");
  if (M == 0) return MOE_OK;
  if (!x_bf16 || !q || !scale) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (reinterpret_cast<uintptr_t>(x_bf16) % 16 || reinterpret_cast<uintptr_t>(q) % 4)
    return fail(MOE_ERR_INVALID_ARG, "x must be 16-byte aligned and q 4-byte aligned");
  PrepArgs p{};
  p.x = static_cast<const __nv_bfloat16*>(x_bf16);
  p.M = M; p.H = H; p.kind = 3; p.q = q; p.scale = scale;
  cudaError_t err = launch_quant_rows(p, reinterpret_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "moe_quant_act_fp8 launch");
  return MOE_OK;
}

size_t moe_workspace_size(int M, int H, int I, int E, int topk, int weight_kind, unsigned flags) {
  if (M < 0 || H <= 0 || I <= 0 || E <= 0 || topk <= 0 || E > MOE_MAX_EXPERTS) return 0;
  if (!known_kind(weight_kind)) return 0;
  if (!known_flags(weight_kind, flags)) return 0;
  return plan(M, H, I, E, topk, weight_kind, flags).total;
}

moe_status_t fused_moe_fp8(const void* x_bf16, const int32_t* topk_ids, const float* topk_weights,
                           const void* w13_e4m3, const float* w13_scale, const void* w2_e4m3,
                           const float* w2_scale, int M, int H, int I, int E, int topk, unsigned flags,
                           void* out_bf16, void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  return fused_impl(MOE_WEIGHT_FP8, x_bf16, topk_ids, topk_weights, w13_e4m3, w13_scale, w2_e4m3, w2_scale,
                    M, H, I, E, topk, flags, out_bf16, workspace, workspace_bytes,
                    reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t fused_moe_int8(const void* x_bf16, const int32_t* topk_ids, const float* topk_weights,
                            const int8_t* w13, const float* w13_scale, const int8_t* w2, const float* w2_scale,
                            int M, int H, int I, int E, int topk, unsigned flags, void* out_bf16,
                            void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  return fused_impl(MOE_WEIGHT_INT8, x_bf16, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale, M, H, I, E,
                    topk, flags, out_bf16, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t fused_moe_int4(const void* x_bf16, const int32_t* topk_ids, const float* topk_weights,
                            const uint8_t* w13, const float* w13_scale, const uint8_t* w2, const float* w2_scale,
                            int M, int H, int I, int E, int topk, unsigned flags, void* out_bf16,
                            void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  return fused_impl(MOE_WEIGHT_INT4, x_bf16, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale, M, H, I, E,
                    topk, flags, out_bf16, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

size_t moe_workspace_size_masked(int E, int cap, int H, int I, int weight_kind) {
  if (E <= 0 || cap <= 0 || H <= 0 || I <= 0 || E > MOE_MAX_EXPERTS) return 0;
  if (weight_kind != MOE_WEIGHT_FP8 && weight_kind != MOE_WEIGHT_INT4) return 0;
  if (static_cast<long long>(E) * cap > (1LL << 28)) return 0;
  return plan_masked(E, cap, H, I).total;
}

moe_status_t fused_moe_masked(int weight_kind, const void* x_bf16, const int32_t* masked_m, const void* w13,
                              const float* w13_scale, const void* w2, const float* w2_scale, int E, int cap,
                              int H, int I, unsigned flags, void* out_bf16, void* workspace,
                              size_t workspace_bytes, moe_stream_t stream) {
  return masked_impl(weight_kind, x_bf16, masked_m, w13, w13_scale, w2, w2_scale, E, cap, H, I, flags, out_bf16,
                     workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_selftest_wait_timeout(void* workspace, long long limit_cycles, int32_t* gave_up,
                                       moe_stream_t stream) {
  g_last_error.clear();
  if (!workspace || !gave_up) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (reinterpret_cast<uintptr_t>(workspace) % 256) return fail(MOE_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (limit_cycles < 1000 || limit_cycles > (1LL << 31))
    return fail(MOE_ERR_INVALID_ARG, "limit_cycles must lie in [1000, 2^31]");
  cudaError_t err = launch_wait_timeout(static_cast<DeviceStatus*>(workspace), limit_cycles, gave_up,
                                        reinterpret_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "moe_selftest_wait_timeout launch");
  return MOE_OK;
}

moe_status_t moe_read_status(const void* workspace, int32_t status_out[2], moe_stream_t stream) {
  g_last_error.clear();
  if (!workspace || !status_out) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  DeviceStatus host{};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t err = cudaMemcpyAsync(&host, workspace, sizeof(host), cudaMemcpyDeviceToHost, s);
  if (err == cudaSuccess) err = cudaStreamSynchronize(s);
  if (err != cudaSuccess) return cuda_fail(err, "moe_read_status");
  status_out[0] = host.bad_ids;
  status_out[1] = host.flags;
  if (host.flags & 1) return fail(MOE_ERR_TIMEOUT, "a bounded device wait gave up");
  if (host.bad_ids) return fail(MOE_ERR_BAD_IDS, "topk_ids outside [0, E)");
  return MOE_OK;
}

moe_status_t moe_read_routing(const void* workspace, int M, int H, int I, int E, int topk, int weight_kind,
                              unsigned flags, int* block_size, int32_t* sorted_ids, int32_t* expert_ids,
                              int32_t* num_tokens_post_padded, int32_t* expert_offsets, moe_stream_t stream) {
  g_last_error.clear();
  if (M <= 0 || H <= 0 || I <= 0 || E <= 0 || topk <= 0 || E > MOE_MAX_EXPERTS || topk > 32 ||
      !known_kind(weight_kind) || !known_flags(weight_kind, flags) ||
      static_cast<long long>(M) * topk > (1LL << 30) || static_cast<long long>(M) * H > (1LL << 40))
    return fail(MOE_ERR_INVALID_ARG, "sizes, weight kind or flags do not describe a routed layer call");
  const Layout L = plan(M, H, I, E, topk, weight_kind, flags);
  if (block_size) *block_size = L.B;
  if (!sorted_ids && !expert_ids && !num_tokens_post_padded && !expert_offsets) return MOE_OK;
  if (!workspace) return fail(MOE_ERR_INVALID_ARG, "NULL workspace");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const char* ws = static_cast<const char*>(workspace);
  struct { void* dst; size_t off, bytes; } copies[] = {
      {sorted_ids, L.sorted, L.cap * 4},
      {expert_ids, L.expert_ids, L.cap / L.B * 4},
      {num_tokens_post_padded, L.scalars, 4},
      {expert_offsets, L.offsets, (static_cast<size_t>(E) + 1) * 4},
  };
  for (const auto& c : copies) {
    if (!c.dst) continue;
    cudaError_t err = cudaMemcpyAsync(c.dst, ws + c.off, c.bytes, cudaMemcpyDeviceToDevice, s);
    if (err != cudaSuccess) return cuda_fail(err, "moe_read_routing");
  }
  return MOE_OK;
}

moe_status_t moe_profile_enable(int max_calls) {
  g_last_error.clear();
  Profiler& P = g_prof;
  for (cudaEvent_t e : P.events) cudaEventDestroy(e);
  P = Profiler{};
  if (max_calls < 0 || max_calls > 100000) return fail(MOE_ERR_INVALID_ARG, "max_calls out of range");
  if (max_calls == 0) return MOE_OK;
  const size_t n = static_cast<size_t>(max_calls) * 8;  // a call records at most 8 events
  P.events.resize(n);
  P.names.assign(n, nullptr);
  for (size_t i = 0; i < n; ++i) {
    cudaError_t err = cudaEventCreate(&P.events[i]);
    if (err != cudaSuccess) {
      P.events.resize(i);
      return cuda_fail(err, "moe_profile_enable");
    }
  }
  P.max_calls = max_calls;
  return MOE_OK;
}

moe_status_t moe_profile_read(float* stage_ms, const char** stage_names, int max_stages, int* n_stages,
                              int* n_calls) {
  g_last_error.clear();
  Profiler& P = g_prof;
  if (!stage_ms || !n_stages || !n_calls || max_stages <= 0) return fail(MOE_ERR_INVALID_ARG, "bad arguments");
  *n_stages = 0;
  *n_calls = 0;
  if (P.used == 0) return MOE_OK;
  cudaError_t err = cudaEventSynchronize(P.events[P.used - 1]);
  if (err != cudaSuccess) return cuda_fail(err, "moe_profile_read");
  std::vector<float> sums;
  std::vector<const char*> names;
  int calls = 0;
  size_t stage = 0;
  for (size_t i = 0; i < P.used; ++i) {
    if (P.names[i] == nullptr) { ++calls; stage = 0; continue; }
    float ms = 0.f;
    err = cudaEventElapsedTime(&ms, P.events[i - 1], P.events[i]);
    if (err != cudaSuccess) return cuda_fail(err, "moe_profile_read");
    if (stage >= sums.size()) { sums.push_back(0.f); names.push_back(P.names[i]); }
    if (names[stage] != P.names[i]) return fail(MOE_ERR_INVALID_ARG, "recorded calls took different paths");
    sums[stage] += ms;
    ++stage;
  }
  const int n = static_cast<int>(sums.size()) < max_stages ? static_cast<int>(sums.size()) : max_stages;
  for (int i = 0; i < n; ++i) {
    stage_ms[i] = sums[i];
    if (stage_names) stage_names[i] = names[i];
  }
  *n_stages = n;
  *n_calls = calls;
  P.used = 0;
  P.calls = 0;
  return MOE_OK;
}

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported size or option";
    case MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "bounded device wait gave up";
    case MOE_ERR_BAD_IDS: return "expert ids outside [0, E)";
  }
  return "unknown status";
}

const char* moe_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
