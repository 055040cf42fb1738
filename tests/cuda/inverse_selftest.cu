// Test harness for the two forms of T = (I + A)^{-1} in gated_deltanet_cpr_gb300/csrc/common.cuh:
// the generic blocked_unit_lower_inverse and the unrolled unit_lower_inverse64 (C = 64) must
// give the same bits.  Built and driven by tests/test_gpu_tc_primitives.py only.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../gated_deltanet_cpr_gb300/csrc/common.cuh"

using namespace gdn;

// A: 64 x 64 row-major (strictly lower part used); Tg, Tf: the two inverses, lower triangle
// (upper entries zero)
__global__ void __launch_bounds__(256) k_inverse_selftest(const float* A, float* Tg, float* Tf) {
  constexpr int C = 64, CP = C + 1;
  __shared__ float As[C * CP];
  __shared__ float Ts[C * CP];
  __shared__ float Xs[3 * 256];
  const int t = threadIdx.x;
  for (int e = t; e < C * C; e += 256) As[(e / C) * CP + e % C] = A[e];
  for (int e = t; e < C * CP; e += 256) Ts[e] = 0.f;
  __syncthreads();
  blocked_unit_lower_inverse<256>(As, CP, Ts, CP, Xs, C);
  for (int e = t; e < C * C; e += 256) Tg[e] = (e % C <= e / C) ? Ts[(e / C) * CP + e % C] : 0.f;
  for (int e = t; e < C * CP; e += 256) Ts[e] = 0.f;
  __syncthreads();
  unit_lower_inverse64(As, CP, Ts, CP, Xs);
  for (int e = t; e < C * C; e += 256) Tf[e] = (e % C <= e / C) ? Ts[(e / C) * CP + e % C] : 0.f;
}

extern "C" int inverse_selftest(const float* A, float* Tg, float* Tf, cudaStream_t st) {
  k_inverse_selftest<<<1, 256, 0, st>>>(A, Tg, Tf);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}
