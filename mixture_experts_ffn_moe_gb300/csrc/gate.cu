// Standalone router gating kernel (moe_gate_topk and the gated layer's first
// launch when the ranking does not run inside the alignment kernel).
#include <cuda_runtime.h>

#include "common.cuh"
#include "gate.cuh"
#include "internal.h"

namespace gbmoe {

constexpr int kGateThreads = 256;

template <int V>
__global__ void __launch_bounds__(kGateThreads) gate_kernel(GateArgs g) {
  pdl_trigger();  // the layer's first kernel may be scheduled now; it waits for this grid
  pdl_wait();     // the logits come from the stream's previous kernel
  const int lane = threadIdx.x & 31, wpb = kGateThreads / 32;
  for (int t = blockIdx.x * wpb + (threadIdx.x >> 5); t < g.M; t += gridDim.x * wpb) gate_token<V>(g, t, lane);
}

cudaError_t launch_gate(const GateArgs& g, int num_sms, cudaStream_t s) {
  if (g.M == 0) return cudaSuccess;
  const int wpb = kGateThreads / 32;
  int grid = (g.M + wpb - 1) / wpb;
  const int cap = 8 * (num_sms > 0 ? num_sms : 1);  // 8 resident CTAs of 256 threads per SM
  if (grid > cap) grid = cap;
  const dim3 gd(grid), bd(kGateThreads);
  switch (gate_vpl(g.E)) {
    case 1: return launch_kernel(gate_kernel<1>, gd, bd, 0, s, true, g);
    case 2: return launch_kernel(gate_kernel<2>, gd, bd, 0, s, true, g);
    case 4: return launch_kernel(gate_kernel<4>, gd, bd, 0, s, true, g);
    case 8: return launch_kernel(gate_kernel<8>, gd, bd, 0, s, true, g);
    case 16: return launch_kernel(gate_kernel<16>, gd, bd, 0, s, true, g);
    case 32: return launch_kernel(gate_kernel<32>, gd, bd, 0, s, true, g);
  }
  return cudaErrorInvalidValue;
}

}  // namespace gbmoe
