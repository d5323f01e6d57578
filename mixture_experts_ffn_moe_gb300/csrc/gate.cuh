// Router gating on the GPU: one warp ranks one token's experts.
//
// The gating functions are those of the served model configurations (the
// pages take the router's output as given): softmax top-k with the chosen
// probabilities renormalised, and the sigmoid router with a selection bias
// and group-limited top-k.  Equal scores go to the lower expert index.
//
// Layout: lane l holds the V consecutive experts [l*V, l*V + V) in
// registers, so a lower lane always holds lower expert indices.  Every
// ranking step is then a warp-wide max of a 32-bit order key (redux.sync)
// followed by a ballot whose lowest set lane is the winner: ties resolve to
// the lower index with no index comparison at all.
#pragma once

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "gbmoe.h"

namespace gbmoe {

struct GateArgs {
  const float* logits;  // [M, E]
  const float* bias;    // [E] or null (sigmoid router only)
  int M, E, topk, ld;   // ld = topk + shared
  int scoring;          // MOE_GATE_SOFTMAX / MOE_GATE_SIGMOID_GROUPED
  int n_group, topk_group;
  float scale;          // routed scaling (sigmoid router)
  int shared;           // 1: column topk = (E, 1.0)
  int vec_ok;           // logits rows may be read as float4 (E % 4 == 0, 16-byte aligned base)
  int32_t* ids;         // [M, ld]
  float* w;             // [M, ld]
};

// Monotone map of a float onto uint32 (a < b  <=>  key(a) < key(b) for
// non-NaN a, b), clamped to >= 2 so that 0 means "taken or absent" and 1
// "outside the kept groups".
__device__ __forceinline__ uint32_t gate_key(float v) {
  const uint32_t b = __float_as_uint(v);
  const uint32_t k = b ^ ((b >> 31) ? 0xffffffffu : 0x80000000u);
  return k < 2u ? 2u : k;
}

__device__ __forceinline__ float gate_sigmoid(float x) { return __fdiv_rn(1.0f, 1.0f + expf(-x)); }

// Merge of two (largest, second largest) pairs.
__device__ __forceinline__ void top2_merge(float& a1, float& a2, float b1, float b2) {
  const float hi = fmaxf(a1, b1), lo = fminf(a1, b1);
  a2 = fmaxf(lo, fmaxf(a2, b2));
  a1 = hi;
}

template <int V>
__device__ __forceinline__ void gate_token(const GateArgs& g, int t, int lane) {
  const float* row = g.logits + static_cast<size_t>(t) * g.E;
  const int e0 = lane * V;
  float sc[V];  // ranking score: the logit (softmax) or s + bias (sigmoid)
  float wv[V];  // value the weight is formed from: the logit or s
  uint32_t key[V];
  if (V % 4 == 0 && g.vec_ok && e0 + V <= g.E) {
#pragma unroll
    for (int j = 0; j < V; j += 4) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(row + e0 + j));
      sc[j] = v.x; sc[j + 1] = v.y; sc[j + 2] = v.z; sc[j + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < V; ++j) sc[j] = e0 + j < g.E ? __ldg(row + e0 + j) : 0.f;
  }
  const bool sigm = g.scoring == MOE_GATE_SIGMOID_GROUPED;
#pragma unroll
  for (int j = 0; j < V; ++j) {
    const bool valid = e0 + j < g.E;
    if (sigm) {
      const float s = gate_sigmoid(sc[j]);
      wv[j] = s;
      sc[j] = (g.bias && valid) ? s + __ldg(g.bias + e0 + j) : s;
    } else {
      wv[j] = sc[j];
    }
    key[j] = valid ? gate_key(sc[j]) : 0u;
  }

  // ---- group-limited selection: keep the topk_group best groups
  if (sigm && g.topk_group < g.n_group) {
    const int gs = g.E / g.n_group;
    uint32_t gkey = 0u;  // order key of a group score, held by one lane per group
    int span;            // lanes per group (fast layout) or 0 (group g scored on lane g)
    if (g.E == 32 * V && (32 % g.n_group) == 0) {
      // every lane lies inside one group and a group is an aligned run of 32/n_group lanes
      span = 32 / g.n_group;
      float t1 = sc[0], t2 = -INFINITY;
#pragma unroll
      for (int j = 1; j < V; ++j) top2_merge(t1, t2, sc[j], -INFINITY);
      for (int o = 1; o < span; o <<= 1)
        top2_merge(t1, t2, __shfl_xor_sync(0xffffffffu, t1, o), __shfl_xor_sync(0xffffffffu, t2, o));
      if ((lane & (span - 1)) == 0) gkey = gate_key(gs >= 2 ? t1 + t2 : t1);
    } else {
      span = 0;
      for (int gi = 0; gi < g.n_group; ++gi) {
        float t1 = -INFINITY, t2 = -INFINITY;
#pragma unroll
        for (int j = 0; j < V; ++j) {
          const int e = e0 + j;
          if (e < g.E && e / gs == gi) top2_merge(t1, t2, sc[j], -INFINITY);
        }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1)
          top2_merge(t1, t2, __shfl_xor_sync(0xffffffffu, t1, o), __shfl_xor_sync(0xffffffffu, t2, o));
        if (lane == gi) gkey = gate_key(gs >= 2 ? t1 + t2 : t1);
      }
    }
    uint32_t kept = 0u;  // bit = the lane holding a kept group's key
    for (int r = 0; r < g.topk_group; ++r) {
      const uint32_t m = __reduce_max_sync(0xffffffffu, gkey);
      const int src = __ffs(__ballot_sync(0xffffffffu, gkey == m && m != 0u)) - 1;
      if (src < 0) break;
      kept |= 1u << src;
      if (lane == src) gkey = 0u;
    }
#pragma unroll
    for (int j = 0; j < V; ++j) {
      const int e = e0 + j;
      const int holder = span ? (lane & ~(span - 1)) : (e < g.E ? e / gs : 0);
      if (!((kept >> holder) & 1u) && key[j] != 0u) key[j] = 1u;
    }
  }

  // ---- top-k: topk rounds of warp argmax; round r's expert lands on lane r
  uint32_t bk = 0u;
  int bj = 0;
  float bw = 0.f;
#pragma unroll
  for (int j = 0; j < V; ++j)
    if (key[j] > bk) { bk = key[j]; bj = j; bw = wv[j]; }
  int my_id = 0;
  float my_v = 0.f;
  for (int r = 0; r < g.topk; ++r) {
    const uint32_t m = __reduce_max_sync(0xffffffffu, bk);
    int src = __ffs(__ballot_sync(0xffffffffu, bk == m)) - 1;
    const int jj = __shfl_sync(0xffffffffu, bj, src);
    const float v = __shfl_sync(0xffffffffu, bw, src);
    if (lane == r) { my_id = src * V + jj; my_v = v; }
    if (lane == src) {
#pragma unroll
      for (int j = 0; j < V; ++j)
        if (j == jj) key[j] = 0u;
      bk = 0u; bj = 0; bw = 0.f;
#pragma unroll
      for (int j = 0; j < V; ++j)
        if (key[j] > bk) { bk = key[j]; bj = j; bw = wv[j]; }
    }
  }
  // ids stay in [0, E) whatever the scores: keys of existing experts are >= 1
  // and topk <= E, so every selection step's maximum lies on an existing expert.
  if (my_id >= g.E) my_id = g.E - 1;

  // ---- weights
  float ex;
  if (sigm) {
    ex = lane < g.topk ? my_v : 0.f;
  } else {
    const float vmax = __shfl_sync(0xffffffffu, my_v, 0);  // the first selection took the largest logit
    ex = lane < g.topk ? expf(my_v - vmax) : 0.f;
  }
  float sum = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const size_t base = static_cast<size_t>(t) * g.ld;
  if (lane < g.topk) {
    float w = __fdiv_rn(ex, sum);
    if (sigm) w *= g.scale;
    g.ids[base + lane] = my_id;
    g.w[base + lane] = w;
  } else if (g.shared && lane == g.topk) {
    g.ids[base + lane] = g.E;
    g.w[base + lane] = 1.0f;
  }
}

// Experts per lane for E experts (0 when E exceeds 32 * 32).
inline int gate_vpl(int E) {
  const int v = (E + 31) / 32;
  return v <= 1 ? 1 : v <= 2 ? 2 : v <= 4 ? 4 : v <= 8 ? 8 : v <= 16 ? 16 : v <= 32 ? 32 : 0;
}

}  // namespace gbmoe
