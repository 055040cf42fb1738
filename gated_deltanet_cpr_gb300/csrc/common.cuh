// common.cuh -- device definitions shared by every CPR kernel.
//
// Bit-exactness across prefill, trainer forward and decode rests on two routines that
// every mode calls with the same operands in the same order:
//   * token_step  -- one step of the gated delta rule on the register-held state (the recurrence that
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

// Bounds-checked builds (compiled with -DGDN_CHECKED=1): every kernel checks the index range
// of each work item it derives from device data (chunk and sequence records, slots, positions)
// against the buffers it was given, and an item outside them records GDN_DEVERR_BOUNDS and is
// skipped instead of touching memory.  In ordinary builds the check compiles to nothing.
#ifndef GDN_CHECKED
#define GDN_CHECKED 0
#endif
__device__ __forceinline__ bool in_bounds(WsHeader* h, bool ok) {
#if GDN_CHECKED
  if (!ok) set_error(h, GDN_DEVERR_BOUNDS);
  return ok;
#else
  (void)h;
  (void)ok;
  return true;
#endif
}

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

// Register layout of the state for the token step.  A warp holds 16 state rows; lane l is in
// row group g = l >> 3 (rows 16 w + 4 g + r, r = 0..3, of warp w) at column block b = l & 7,
// and holds the float4 column groups 8 j + b (columns 32 j + 4 b .. + 3, j = 0 .. d/32 - 1)
// of its 4 rows: S[r][j].  A d x d state takes 2 d threads (d / 16 warps), d / 2 floats each.
template <int D>
struct StateLayout {
  static constexpr int J = D / 32;
  int row0;  // first of the lane's 4 rows
  int b;     // column block
  __device__ __forceinline__ explicit StateLayout(int t) : row0(16 * (t >> 5) + 4 * ((t & 31) >> 3)), b(t & 7) {}
  __device__ __forceinline__ int col(int j) const { return 32 * j + 4 * b; }
  // the row whose output this lane's reduction ends with, and whether the lane writes it
  __device__ __forceinline__ int out_row() const { return row0 + ((b >> 1) & 3); }
  __device__ __forceinline__ bool writes_out() const { return (b & 1) == 0; }
  // state rows start at src (row stride D floats)
  __device__ __forceinline__ void load(float4 (&S)[4][J], const float* src) const {
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int j = 0; j < J; ++j) S[r][j] = *reinterpret_cast<const float4*>(src + (int64_t)(row0 + r) * D + col(j));
  }
  __device__ __forceinline__ void store(const float4 (&S)[4][J], float* dst) const {
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int j = 0; j < J; ++j) *reinterpret_cast<float4*>(dst + (int64_t)(row0 + r) * D + col(j)) = S[r][j];
  }
  // the explicit state c S (one round-to-nearest product per element)
  __device__ __forceinline__ void store_scaled(const float4 (&S)[4][J], float c, float* dst) const {
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int j = 0; j < J; ++j)
        *reinterpret_cast<float4*>(dst + (int64_t)(row0 + r) * D + col(j)) =
            make_float4(__fmul_rn(c, S[r][j].x), __fmul_rn(c, S[r][j].y), __fmul_rn(c, S[r][j].z),
                        __fmul_rn(c, S[r][j].w));
  }
};

// Sum over the 8 lanes of a row group of x[r] (r = 0..3, one value per row of the group):
// a fixed xor-4, xor-2, xor-1 tree.  The xor-4 step leaves rows 0, 1 on lanes with bit 2
// clear and rows 2, 3 on the others, the xor-2 step one row per lane, the xor-1 step adds
// the partner holding the same row; lane b ends with the total of row (b >> 1) & 3.  Every
// total is one fixed expression of the 8 lane values (fp32 addition is commutative, so the
// two lanes holding a total hold the same bits).
__device__ __forceinline__ float group_reduce4(const float (&x)[4], int b) {
  const bool h2 = (b & 4) != 0, h1 = (b & 2) != 0;
  const float y0 = __fadd_rn(h2 ? x[2] : x[0], __shfl_xor_sync(0xffffffffu, h2 ? x[0] : x[2], 4));
  const float y1 = __fadd_rn(h2 ? x[3] : x[1], __shfl_xor_sync(0xffffffffu, h2 ? x[1] : x[3], 4));
  const float z = __fadd_rn(h1 ? y1 : y0, __shfl_xor_sync(0xffffffffu, h1 ? y0 : y1, 2));
  return __fadd_rn(z, __shfl_xor_sync(0xffffffffu, z, 1));
}
// The same four totals on every lane of the group, by an xor-4, xor-2, xor-1 butterfly over
// all four values: the same tree as group_reduce4 (each level adds the two halves of the
// level below, in either order), so the same bits, in three exchange levels instead of five.
__device__ __forceinline__ void group_allreduce4(const float (&x)[4], float (&tot)[4]) {
  float y[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) y[r] = __fadd_rn(x[r], __shfl_xor_sync(0xffffffffu, x[r], 4));
#pragma unroll
  for (int r = 0; r < 4; ++r) y[r] = __fadd_rn(y[r], __shfl_xor_sync(0xffffffffu, y[r], 2));
#pragma unroll
  for (int r = 0; r < 4; ++r) tot[r] = __fadd_rn(y[r], __shfl_xor_sync(0xffffffffu, y[r], 1));
}

// One gated delta-rule step on the lane's 4 state rows (StateLayout).  The recurrence
//     S <- a S;   p = S k;   u = beta (v - p);   S <- S + u k^T;   o = S q
// runs on a scaled copy: the state is S = c S~ (c the product of the decays since S~ was
// last made equal to S), so the decay is one scalar product instead of a pass over the state:
//     c <- c a;   p = c (S~ k);   u = beta (v - p);   S~ <- S~ + (u / c) k^T;   o = c (S~ q)
// with u / c = beta (v / c - S~ k) formed as fma(beta rcp(c), v, -(beta (S~ k))), rcp the
// hardware reciprocal approximation.  Whenever c leaves [2^-64, 2^64] the state is
// made explicit first (S~ <- c S~, c <- 1), so S~ stays within 2^64 of S and no scale under-
// or overflows; c is the same in every lane, so the choice is warp-uniform.  Each row's dot:
// per lane one float2 partial over the lane's columns in the order (j, pair): .x takes
// columns 32j + 4b, then 32j + 4b + 2, .y columns 32j + 4b + 1, then 32j + 4b + 3, ascending j;
// then x + y, then the 8 lanes' fixed tree (group_reduce4; for p every lane needs all four
// rows, group_allreduce4, the same tree).  k (kept in registers from the dot to the update)
// and q are fp32 copies in shared memory (exact widenings of the inputs); v4 is v of the
// lane's 4 rows.  The step is split in two sweeps so that a token loop can overlap the output
// reduction of one token with the first sweep of the next:
//   ts_dot_k       k into registers, the lane's partials of S~ k
//   ts_update_dot  S~ <- S~ + us_r k^T (us_r = u_r / c per row), the lane's partials of S~ q
// token_step is the whole step.  All 32 lanes of the warp call these together.
constexpr float kScaleLo = 0x1p-64f, kScaleHi = 0x1p64f;

// c <- c a; if c leaves [2^-64, 2^64] the state becomes explicit (S~ <- c S~, c <- 1)
template <int D>
__device__ __forceinline__ void ts_decay(float4 (&S)[4][D / 32], float& c, float a) {
  constexpr int J = D / 32;
  c = __fmul_rn(c, a);
  if (!(c >= kScaleLo && c <= kScaleHi)) {
    const float2 c2 = make_float2(c, c);
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const float2 s01 = mul2(c2, make_float2(S[r][j].x, S[r][j].y));
        const float2 s23 = mul2(c2, make_float2(S[r][j].z, S[r][j].w));
        S[r][j] = make_float4(s01.x, s01.y, s23.x, s23.y);
      }
    c = 1.f;
  }
}
template <int D>
__device__ __forceinline__ void ts_dot_k(const float4 (&S)[4][D / 32], const float* __restrict__ k_sh, int b,
                                         float4 (&kk)[D / 32], float (&part)[4]) {
  constexpr int J = D / 32;
#pragma unroll
  for (int j = 0; j < J; ++j) kk[j] = *reinterpret_cast<const float4*>(k_sh + 32 * j + 4 * b);
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    float2 pr = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < J; ++j) {
      pr = fma2(make_float2(S[r][j].x, S[r][j].y), make_float2(kk[j].x, kk[j].y), pr);
      pr = fma2(make_float2(S[r][j].z, S[r][j].w), make_float2(kk[j].z, kk[j].w), pr);
    }
    part[r] = __fadd_rn(pr.x, pr.y);
  }
}
// hardware reciprocal approximation (one MUFU instruction; deterministic, c is normal here)
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
// us_r = u_r / c for the lane's rows from the reduced S~ k (p4, all four rows), as
// us = beta (v / c - p) = fma(beta rcp(c), v, -(beta p))
__device__ __forceinline__ void ts_scaled_u(const float (&p4)[4], float4 v4, float beta, float c,
                                            float (&us)[4]) {
  const float bic = __fmul_rn(beta, rcp_approx(c));
  const float v[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
  for (int r = 0; r < 4; ++r) us[r] = __fmaf_rn(bic, v[r], -__fmul_rn(beta, p4[r]));
}
template <int D>
__device__ __forceinline__ void ts_update_dot(float4 (&S)[4][D / 32], const float4 (&kk)[D / 32],
                                              const float* __restrict__ q_sh, const float (&us)[4], int b,
                                              float (&opart)[4]) {
  constexpr int J = D / 32;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const float2 u2 = make_float2(us[r], us[r]);
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const float2 s01 = fma2(u2, make_float2(kk[j].x, kk[j].y), make_float2(S[r][j].x, S[r][j].y));
      const float2 s23 = fma2(u2, make_float2(kk[j].z, kk[j].w), make_float2(S[r][j].z, S[r][j].w));
      S[r][j] = make_float4(s01.x, s01.y, s23.x, s23.y);
    }
  }
  float4 qq[J];
#pragma unroll
  for (int j = 0; j < J; ++j) qq[j] = *reinterpret_cast<const float4*>(q_sh + 32 * j + 4 * b);
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    float2 pr = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < J; ++j) {
      pr = fma2(make_float2(S[r][j].x, S[r][j].y), make_float2(qq[j].x, qq[j].y), pr);
      pr = fma2(make_float2(S[r][j].z, S[r][j].w), make_float2(qq[j].z, qq[j].w), pr);
    }
    opart[r] = __fadd_rn(pr.x, pr.y);
  }
}
// The whole step on S~ with scale c (updated); returns o of row out_row().
template <int D>
__device__ __forceinline__ float token_step(float4 (&S)[4][D / 32], float& c, const float* __restrict__ k_sh,
                                            const float* __restrict__ q_sh, float a, float beta, float4 v4,
                                            int b) {
  float4 kk[D / 32];
  float part[4], p[4], us[4], opart[4];
  ts_decay<D>(S, c, a);
  ts_dot_k<D>(S, k_sh, b, kk, part);
  group_allreduce4(part, p);
  ts_scaled_u(p, v4, beta, c, us);
  ts_update_dot<D>(S, kk, q_sh, us, b, opart);
  return __fmul_rn(c, group_reduce4(opart, b));
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

// The same inverse for C = 64 on 256 threads, with the same operations in the same order.
// The off-diagonal rounds are bound by shared-memory loads (two per fma when every thread
// owns one element), so a thread owns a 2 x 2 tile of one block instead (rows ii, ii + 8,
// columns rr, rr + 8; round `off` has 4 - off blocks, 64 threads each) and every value it
// loads feeds two fma.  Each element's sum is still the generic loop's sequence of fma: it
// is unrolled over its longest length with a per-element select in place of the loop
// bounds (a skipped term leaves the accumulator unchanged).  Operands outside a sum's range
// are read (inside the matrices) and discarded.
__device__ __forceinline__ void unit_lower_inverse64(const float* A, int CPA, float* Tm, int CPT, float* Xs) {
  constexpr int TB = 16, C = 64, NB = C / TB;
  const int t = threadIdx.x;
  if (t < C) {  // diagonal blocks as in blocked_unit_lower_inverse
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
  const int q = t >> 6, ii = (t >> 3) & 7, rr = t & 7;  // block q of the round, tile corner
#pragma unroll
  for (int off = 1; off < NB; ++off) {
    const bool live = q < NB - off;
    const int I = off + q, J = I - off;  // block row I, block column J
    if (live) {
      // X[e] = sum_{m = r}^{16 I - 1} A[i][m] T[m][r],  m = 16 J + k,  k = rr .. 16 off - 1
      const float* a0 = A + (I * TB + ii) * CPA + J * TB;
      const float* a1 = a0 + 8 * CPA;
      const float* t0 = Tm + (J * TB) * CPT + J * TB + rr;
      float x00 = 0.f, x01 = 0.f, x10 = 0.f, x11 = 0.f;
#pragma unroll
      for (int k = 0; k < off * TB; ++k) {
        const float p0 = a0[k], p1 = a1[k], y0 = t0[k * CPT], y1 = t0[k * CPT + 8];
        x00 = (k >= rr) ? __fmaf_rn(p0, y0, x00) : x00;
        x01 = (k >= rr + 8) ? __fmaf_rn(p0, y1, x01) : x01;
        x10 = (k >= rr) ? __fmaf_rn(p1, y0, x10) : x10;
        x11 = (k >= rr + 8) ? __fmaf_rn(p1, y1, x11) : x11;
        if ((k & 7) == 7) asm volatile("" ::: "memory");
      }
      float* xs = Xs + q * 256;
      xs[ii * TB + rr] = x00;
      xs[ii * TB + rr + 8] = x01;
      xs[(ii + 8) * TB + rr] = x10;
      xs[(ii + 8) * TB + rr + 8] = x11;
    }
    __syncthreads();
    if (live) {
      // T[i][r] = -sum_{m = 16 I}^{i} T[i][m] X[m - 16 I][rr],  m = 16 I + k,  k = 0 .. ii
      const float* p0r = Tm + (I * TB + ii) * CPT + I * TB;
      const float* p1r = p0r + 8 * CPT;
      const float* xq = Xs + q * 256 + rr;
      float y00 = 0.f, y01 = 0.f, y10 = 0.f, y11 = 0.f;
#pragma unroll
      for (int k = 0; k < TB; ++k) {
        const float p0 = p0r[k], p1 = p1r[k], x0 = xq[k * TB], x1 = xq[k * TB + 8];
        y00 = (k <= ii) ? __fmaf_rn(p0, x0, y00) : y00;
        y01 = (k <= ii) ? __fmaf_rn(p0, x1, y01) : y01;
        y10 = (k <= ii + 8) ? __fmaf_rn(p1, x0, y10) : y10;
        y11 = (k <= ii + 8) ? __fmaf_rn(p1, x1, y11) : y11;
        if ((k & 7) == 7) asm volatile("" ::: "memory");
      }
      float* o0 = Tm + (I * TB + ii) * CPT + J * TB + rr;
      o0[0] = -y00;
      o0[8] = -y01;
      o0[8 * CPT] = -y10;
      o0[8 * CPT + 8] = -y11;
    }
    __syncthreads();
  }
}

// The same with one row stride for A and T.
template <int NT>
__device__ __forceinline__ void blocked_unit_lower_inverse(const float* A, float* Tm, float* Xs, int C, int CP) {
  blocked_unit_lower_inverse<NT>(A, CP, Tm, CP, Xs, C);
}

}  // namespace gdn
