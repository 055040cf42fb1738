// Test harness for the tcgen05 building blocks in gated_deltanet_cpr_gb300/csrc/tc.cuh:
// D (128 x N, fp32) = [Cinit +] A (128 x K, bf16) * B^T (B: N x K, bf16), with A and B laid
// out K-major without swizzle in shared memory, the accumulator in tensor memory, and
// every wait bounded.  Built and driven by tests/test_gpu_tc_primitives.py only.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../gated_deltanet_cpr_gb300/csrc/tc.cuh"

using namespace gdn::tc;

__global__ void __launch_bounds__(128) k_tc_selftest(const __nv_bfloat16* A, const __nv_bfloat16* B,
                                                     const float* Cinit, float* D, int N, int K,
                                                     uint32_t ncols, int* status) {
  extern __shared__ __align__(128) unsigned char sm[];
  unsigned char* As = sm;
  unsigned char* Bs = sm + 128 * K * 2;
  uint64_t* bar = reinterpret_cast<uint64_t*>(Bs + N * K * 2);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 1);
  const int t = threadIdx.x, warp = t / 32;
  for (int e = t; e < 128 * K; e += 128)
    *reinterpret_cast<__nv_bfloat16*>(As + kmajor_off(e / K, e % K, K)) = A[e];
  for (int e = t; e < N * K; e += 128)
    *reinterpret_cast<__nv_bfloat16*>(Bs + kmajor_off(e / K, e % K, K)) = B[e];
  if (t == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tslot, ncols);
  fence_proxy_async();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tbase = *tslot;
  if (Cinit) {
    for (int c0 = 0; c0 < N; c0 += 16) {
      float v[16];
      for (int i = 0; i < 16; ++i) v[i] = Cinit[t * N + c0 + i];
      tmem_st16(tmem_lane_addr(tbase, warp, c0), v);
    }
    tmem_st_wait();
  }
  fence_before_sync();
  __syncthreads();
  if (t == 0) {
    fence_after_sync();
    const uint32_t idesc = idesc_bf16(128, N);
    for (int k0 = 0; k0 < K; k0 += 16) {
      const uint64_t ad = make_desc(smem_u32(As) + (k0 / 8) * 128, 128, (K / 8) * 128);
      const uint64_t bd = make_desc(smem_u32(Bs) + (k0 / 8) * 128, 128, (K / 8) * 128);
      mma_bf16(tbase, ad, bd, idesc, (Cinit != nullptr || k0 > 0) ? 1u : 0u);
    }
    mma_commit(bar);
  }
  const int ok = __syncthreads_and(mbar_wait(bar, 0) ? 1 : 0);
  fence_after_sync();
  if (ok) {
    for (int c0 = 0; c0 < N; c0 += 16) {
      float v[16];
      tmem_ld16(tmem_lane_addr(tbase, warp, c0), v);
      for (int i = 0; i < 16; ++i) D[t * N + c0 + i] = v[i];
    }
  } else if (t == 0) {
    atomicExch(status, 1);
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, ncols);
}

extern "C" int tc_selftest(const void* A, const void* B, const float* Cinit, float* D, int N, int K,
                           int* status, cudaStream_t st) {
  if (N % 16 || N < 16 || N > 256 || K % 16 || K < 16 || K > 256) return 1;
  uint32_t ncols = 32;
  while (ncols < (uint32_t)N) ncols <<= 1;
  const size_t smem = (size_t)(128 + N) * K * 2 + 16;
  if (cudaFuncSetAttribute(k_tc_selftest, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return 2;
  k_tc_selftest<<<1, 128, smem, st>>>(static_cast<const __nv_bfloat16*>(A),
                                       static_cast<const __nv_bfloat16*>(B), Cinit, D, N, K, ncols,
                                       status);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

// transpose_image: a Ks x R bf16 matrix X (row-major in global memory) into its K-major
// shared-memory image, transposed there by all 256 threads, read back as the R x Ks image of X^T
__global__ void __launch_bounds__(256) k_transpose_selftest(const uint16_t* X, uint16_t* Y, int R, int Ks) {
  extern __shared__ __align__(128) unsigned char sm[];
  unsigned char* src = sm;
  unsigned char* dst = sm + R * Ks * 2;
  for (int e = threadIdx.x; e < Ks * R; e += 256)
    *reinterpret_cast<uint16_t*>(src + kmajor_off(e / R, e % R, R)) = X[e];
  __syncthreads();
  transpose_image(dst, src, R, Ks);
  __syncthreads();
  for (int e = threadIdx.x; e < R * Ks; e += 256) Y[e] = *reinterpret_cast<const uint16_t*>(dst + kmajor_off(e / Ks, e % Ks, Ks));
}

extern "C" int transpose_selftest(const void* X, void* Y, int R, int Ks, cudaStream_t st) {
  if (R % 16 || Ks % 16 || R < 16 || Ks < 16 || R * Ks > 128 * 128) return 1;
  const size_t smem = (size_t)2 * R * Ks * 2;
  if (cudaFuncSetAttribute(k_transpose_selftest, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return 2;
  k_transpose_selftest<<<1, 256, smem, st>>>(static_cast<const uint16_t*>(X), static_cast<uint16_t*>(Y), R, Ks);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

// MN-major operands (Opnd, mma_part): D (128 x N) = A B^T with A (128 x K) and / or B (N x K)
// given to the tensor core as the image of its transpose (A^T: K rows x 128, B^T: K rows x N,
// each K-major over its own columns) read MN-major; amode / bmode 0 = the K-major image of the
// operand itself.  One term, no initial accumulator.
__global__ void __launch_bounds__(128) k_mn_selftest(const __nv_bfloat16* A, const __nv_bfloat16* B, float* D,
                                                     int N, int K, int amode, int bmode, uint32_t ncols,
                                                     int* status) {
  extern __shared__ __align__(128) unsigned char sm[];
  unsigned char* As = sm;
  unsigned char* Bs = sm + 128 * K * 2;
  uint64_t* bar = reinterpret_cast<uint64_t*>(Bs + N * K * 2);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 1);
  const int t = threadIdx.x, warp = t / 32;
  for (int e = t; e < 128 * K; e += 128) {
    const int r = e / K, k = e % K;
    *reinterpret_cast<__nv_bfloat16*>(As + (amode ? kmajor_off(k, r, 128) : kmajor_off(r, k, K))) = A[e];
  }
  for (int e = t; e < N * K; e += 128) {
    const int r = e / K, k = e % K;
    *reinterpret_cast<__nv_bfloat16*>(Bs + (bmode ? kmajor_off(k, r, N) : kmajor_off(r, k, K))) = B[e];
  }
  if (t == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tslot, ncols);
  fence_proxy_async();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tbase = *tslot;
  if (t == 0) {
    const Opnd a = amode ? opnd_mn(smem_u32(As), 0u, 128) : opnd_k(smem_u32(As), 0u, K);
    const Opnd b = bmode ? opnd_mn(smem_u32(Bs), 0u, N) : opnd_k(smem_u32(Bs), 0u, K);
    const uint32_t idesc = idesc_bf16(128, N) | (amode ? IDESC_A_MN : 0u) | (bmode ? IDESC_B_MN : 0u);
    mma_part(tbase, a, false, b, false, K, idesc, false);
    mma_commit(bar);
  }
  const int ok = __syncthreads_and(mbar_wait(bar, 0) ? 1 : 0);
  fence_after_sync();
  if (ok) {
    for (int c0 = 0; c0 < N; c0 += 16) {
      float v[16];
      tmem_ld16(tmem_lane_addr(tbase, warp, c0), v);
      for (int i = 0; i < 16; ++i) D[t * N + c0 + i] = v[i];
    }
  } else if (t == 0) {
    atomicExch(status, 1);
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, ncols);
}

extern "C" int mn_selftest(const void* A, const void* B, float* D, int N, int K, int amode, int bmode, int* status,
                           cudaStream_t st) {
  if ((N != 64 && N != 128) || (K != 64 && K != 128)) return 1;
  const uint32_t ncols = (uint32_t)N;
  const size_t smem = (size_t)(128 + N) * K * 2 + 16;
  if (cudaFuncSetAttribute(k_mn_selftest, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return 2;
  k_mn_selftest<<<1, 128, smem, st>>>(static_cast<const __nv_bfloat16*>(A), static_cast<const __nv_bfloat16*>(B), D,
                                       N, K, amode, bmode, ncols, status);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}
