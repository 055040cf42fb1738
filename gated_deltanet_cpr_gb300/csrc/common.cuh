// common.cuh -- device definitions shared by every CPR kernel.
//
// Bit-exactness across prefill, trainer forward and decode rests on two routines that
// every mode calls with the same operands in the same order:
//   * token_step  -- one step of the gated delta rule on a state row (the recurrence that
//                    CPR keeps as its main computation; IsoExec page, section
//                    "Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet");
//   * the boundary routines (prep_* and chain_*) -- the chunk (WY/UT) form that advances
//                    a boundary state over one full chunk, used by the prefill boundary
//                    pass and by the decode resynchronisation every C tokens.
// All floating-point arithmetic in them is written with explicit round-to-nearest
// intrinsics (__fmaf_rn, __fmul_rn, __fadd_rn, __fsub_rn), which the compiler never fuses
// or reorders, and every reduction has one fixed order that depends only on (C, D).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

constexpr int kMaxChunk = 64;
constexpr int kRowsPerChain = 16;   // state rows per boundary-chain CTA
constexpr int kPrepThreads = 256;   // boundary pre-pass CTA size
constexpr int kChainThreads = 256;  // boundary chain CTA size

// ---------------------------------------------------------------- workspace ----
struct WsHeader {
  int32_t err;    // gdn_device_error, first error wins
  int32_t valid;  // 1 once the work list is built and consistent with the host's copy
  int32_t pad[62];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

struct ChunkRec {  // one chunk of one sequence
  int32_t seq, tok0, len, jloc;
};
struct SeqRec {  // one sequence
  int32_t tok0, len, chunk0, nchunks;
};

__device__ __forceinline__ void set_error(WsHeader* h, int code) { atomicCAS(&h->err, 0, code); }

// ---------------------------------------------------------------- conversions ----
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// 8 consecutive elements -> fp32 (16-byte aligned source)
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float* o) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    o[2 * i] = __uint_as_float(w[i] << 16);
    o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ void load8(const float* p, float* o) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 b = reinterpret_cast<const float4*>(p)[1];
  o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
  o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}

// 4 consecutive elements -> fp32 (8-byte aligned bf16 source / 16-byte aligned fp32 source)
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}
__device__ __forceinline__ float4 load4(const float* p) { return *reinterpret_cast<const float4*>(p); }

__device__ __forceinline__ void store_out(float* p, float x) { *p = x; }
__device__ __forceinline__ void store_out(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// ---------------------------------------------------------------- fixed dot ----
// Canonical dot product of length D (multiple of 4) over fp32 arrays in shared memory:
// four partial sums, partial e takes elements 4m+e in ascending m, combined as
// (p0 + p1) + (p2 + p3).  Every boundary-pass dot uses exactly this order.
template <int D>
__device__ __forceinline__ float dot_canon(const float* __restrict__ a, const float* __restrict__ b) {
  float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll
  for (int m = 0; m < D / 4; ++m) {
    const float4 x = reinterpret_cast<const float4*>(a)[m];
    const float4 y = reinterpret_cast<const float4*>(b)[m];
    p0 = __fmaf_rn(x.x, y.x, p0);
    p1 = __fmaf_rn(x.y, y.y, p1);
    p2 = __fmaf_rn(x.z, y.z, p2);
    p3 = __fmaf_rn(x.w, y.w, p3);
  }
  return __fadd_rn(__fadd_rn(p0, p1), __fadd_rn(p2, p3));
}

// ---------------------------------------------------------------- token step ----
// Packed fp32 pairs (Blackwell f32x2 instructions): each lane of the pair is rounded exactly
// like the scalar __fmaf_rn / __fmul_rn, so these are the same arithmetic in half the
// instructions.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(*reinterpret_cast<const uint64_t*>(&a)), "l"(*reinterpret_cast<const uint64_t*>(&b)),
        "l"(*reinterpret_cast<const uint64_t*>(&c)));
  return *reinterpret_cast<const float2*>(&d);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;"
      : "=l"(d)
      : "l"(*reinterpret_cast<const uint64_t*>(&a)), "l"(*reinterpret_cast<const uint64_t*>(&b)));
  return *reinterpret_cast<const float2*>(&d);
}

// shared-memory vector load that the compiler may not merge with an earlier load of the
// same address (keeps the first pass's k out of registers during the update pass)
__device__ __forceinline__ float4 lds4_fresh(const float* p) {
  float4 v;
  asm volatile("ld.volatile.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"((uint32_t)__cvta_generic_to_shared(p)));
  return v;
}

// One gated delta-rule step on row i of the state, held by a pair of adjacent lanes
// (half = lane & 1).  The pair splits the D columns into float4 groups: register group m
// holds columns [8m + 4*half, 8m + 4*half + 4).  Order of operations (the recurrence's
// own order):
//     S <- a S;   p = S k;   u = beta (v_i - p);   S <- S + u k^T;   o_i = S q
// Each dot is four partial sums over the lane's columns in ascending m (partial e takes
// component e of every group), combined as (p0 + p1) + (p2 + p3), then added to the
// partner lane's partial with one xor-shuffle; fp32 addition is commutative, so both lanes
// hold identical bits.  k and q are fp32 copies in shared memory (exact widenings of the
// inputs).  The update S <- S + u k^T and the output dot are two passes over the state
// (the same operations on every element, in the same order), so that k and q are never
// both held in registers.  All 32 lanes of the warp must call this together.
template <int D>
__device__ __forceinline__ float token_step(float4 (&S)[D / 8], const float* __restrict__ k_sh,
                                            const float* __restrict__ q_sh, float a, float beta,
                                            float v_i, int half) {
  const float2 a2 = make_float2(a, a);
  float2 p01 = make_float2(0.f, 0.f), p23 = make_float2(0.f, 0.f);
#pragma unroll
  for (int m = 0; m < D / 8; ++m) {
    const float4 kk = *reinterpret_cast<const float4*>(k_sh + 8 * m + 4 * half);
    float2 s01 = mul2(a2, make_float2(S[m].x, S[m].y));
    float2 s23 = mul2(a2, make_float2(S[m].z, S[m].w));
    p01 = fma2(s01, make_float2(kk.x, kk.y), p01);
    p23 = fma2(s23, make_float2(kk.z, kk.w), p23);
    S[m] = make_float4(s01.x, s01.y, s23.x, s23.y);
  }
  float part = __fadd_rn(__fadd_rn(p01.x, p01.y), __fadd_rn(p23.x, p23.y));
  const float p = __fadd_rn(part, __shfl_xor_sync(0xffffffffu, part, 1));
  const float u = __fmul_rn(beta, __fsub_rn(v_i, p));
  const float2 u2 = make_float2(u, u);
#pragma unroll
  for (int m = 0; m < D / 8; ++m) {
    const float4 kk = lds4_fresh(k_sh + 8 * m + 4 * half);
    const float2 s01 = fma2(u2, make_float2(kk.x, kk.y), make_float2(S[m].x, S[m].y));
    const float2 s23 = fma2(u2, make_float2(kk.z, kk.w), make_float2(S[m].z, S[m].w));
    S[m] = make_float4(s01.x, s01.y, s23.x, s23.y);
  }
  p01 = make_float2(0.f, 0.f);
  p23 = make_float2(0.f, 0.f);
#pragma unroll
  for (int m = 0; m < D / 8; ++m) {
    const float4 qq = *reinterpret_cast<const float4*>(q_sh + 8 * m + 4 * half);
    p01 = fma2(make_float2(S[m].x, S[m].y), make_float2(qq.x, qq.y), p01);
    p23 = fma2(make_float2(S[m].z, S[m].w), make_float2(qq.z, qq.w), p23);
  }
  part = __fadd_rn(__fadd_rn(p01.x, p01.y), __fadd_rn(p23.x, p23.y));
  return __fadd_rn(part, __shfl_xor_sync(0xffffffffu, part, 1));
}

// T = (I + A)^{-1} for a strictly lower C x C matrix A in shared memory (row stride CPA; T
// written with row stride CPT),
// blocked by 16.  Diagonal blocks by forward substitution, one column per thread:
//     T[r][r] = 1,  T[i][r] = -sum_{m=r}^{i-1} A[i][m] T[m][r];
// then off-diagonal blocks (I > J) by increasing I - J:
//     X[i][r] = sum_{m=r}^{16I-1} A[i][m] T[m][r],   T[i][r] = -sum_{m=16I}^{i} T[i][m] X[m][r]
// (every sum in ascending m with one accumulator).  Only the lower triangle of T is
// written.  Xs: 3 * 16 * 16 floats of scratch.  All NT threads of the block must call it.
template <int NT>
__device__ __forceinline__ void blocked_unit_lower_inverse(const float* A, int CPA, float* Tm, int CPT, float* Xs,
                                                           int C) {
  constexpr int TB = 16;
  const int t = threadIdx.x;
  const int nb = C / TB;
  if (t < C) {  // column r of its diagonal block, kept in registers (col[k] = T[rb + k][r])
    const int r = t, rb = (r / TB) * TB, rr = r - rb;
    float col[TB];
#pragma unroll
    for (int k = 0; k < TB; ++k) col[k] = (k == rr) ? 1.f : 0.f;
#pragma unroll
    for (int ii = 1; ii < TB; ++ii) {
      float acc = 0.f;
#pragma unroll
      for (int m = 0; m < ii; ++m)
        if (m >= rr) acc = __fmaf_rn(A[(rb + ii) * CPA + rb + m], col[m], acc);
      if (ii > rr) col[ii] = -acc;
    }
#pragma unroll
    for (int k = 0; k < TB; ++k)
      if (k >= rr) Tm[(rb + k) * CPT + r] = col[k];
  }
  __syncthreads();
  for (int off = 1; off < nb; ++off) {
    const int nel = (nb - off) * TB * TB;
    for (int e = t; e < nel; e += NT) {
      const int I = off + e / (TB * TB), ii = (e / TB) % TB, rr = e % TB;
      const int i = I * TB + ii, r = (I - off) * TB + rr;
      float acc = 0.f;
#pragma unroll 4
      for (int m = r; m < I * TB; ++m) acc = __fmaf_rn(A[i * CPA + m], Tm[m * CPT + r], acc);
      Xs[e] = acc;
    }
    __syncthreads();
    for (int e = t; e < nel; e += NT) {
      const int I = off + e / (TB * TB), ii = (e / TB) % TB, rr = e % TB;
      const int i = I * TB + ii, r = (I - off) * TB + rr;
      const float* X = Xs + (e / (TB * TB)) * TB * TB;
      float acc = 0.f;
#pragma unroll 4
      for (int m = I * TB; m <= i; ++m) acc = __fmaf_rn(Tm[i * CPT + m], X[(m - I * TB) * TB + rr], acc);
      Tm[i * CPT + r] = -acc;
    }
    __syncthreads();
  }
}

// The same with one row stride for A and T.
template <int NT>
__device__ __forceinline__ void blocked_unit_lower_inverse(const float* A, float* Tm, float* Xs, int C, int CP) {
  blocked_unit_lower_inverse<NT>(A, CP, Tm, CP, Xs, C);
}

// State row i, half h: global float offset of register group m.
template <int D>
__device__ __forceinline__ int state_col(int m, int half) {
  return 8 * m + 4 * half;
}

}  // namespace gdn
