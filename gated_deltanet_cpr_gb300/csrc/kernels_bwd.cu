// kernels_bwd.cu -- reverse mode of CPR Gated DeltaNet for sm_103a (trainer backward; the
// IsoExec page's CPR timing table, row "Trainer Fwd+Bwd").
//
// The backward follows the forward's schedule in reverse.  Chunk j (local tokens
// i = 0..n-1, zero-padded to C) with start state S0 = S^(j) computes, in exact arithmetic,
//     G = cumsum g,  Gam_is = e^{G_i - G_s},  A_is = beta_i Gam_is k_i.k_s (i > s),
//     T = (I + A)^{-1},  W = T diag(beta e^G) K,  Ut = T diag(beta) V,  U = Ut - W S0^T,
//     P_is = Gam_is q_i.k_s (i >= s),  O = diag(e^G) Q S0^T + P U,
//     S_end = e^{G_last} S0 + U^T diag(dec) K,   dec_s = e^{G_last - G_s},
// which is the token recurrence rewritten.  Its reverse mode:
//   KB1 k_bwd_prep   per chunk: G, T, W, Ut, P and the chunk's own adjoint of S0,
//                    L = dO^T (diag(e^G) Q - P W)
//   KB2 k_bwd_chain  per (sequence, head, 16-row block), chunks in reverse order:
//                    dS^(j) = L_j + e^{G_last} dS^(j+1) - (dS^(j+1) K^T) diag(dec) W,
//                    starting from dstate_out; dstate_in = dS^(0)
//   KB3 k_bwd_big    per chunk: the products with the d x d matrices S0 and dS_end:
//                    U, dU = P^T dO + diag(dec) K dS_end^T, dO S0, U dS_end, dW = -dU S0,
//                    <dS_end, S0>
//   KB4 k_bwd_grad   per chunk: X = T^T dU, Y = T^T dW, dA = -(X Ut^T + Y W^T) (strictly lower)
//                    and the gradients of q, k, v, g, beta (per value head)
//   KB5 k_bwd_gqa    dq, dk summed over the value heads of each group, ascending
// Every sum has one fixed order, there are no atomics, and nothing depends on the batch
// composition, so the backward is deterministic.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <set>
#include <utility>

#include "../../include/gdn_cpr.h"
#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace gdn {
namespace {

constexpr int NT = 256;
constexpr int CP = kMaxChunk + 4;  // padded row of a C x C matrix in shared memory (16-byte rows)

template <typename F>
void ensure_smem_bwd(F* fn, size_t bytes) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  if (done.insert({reinterpret_cast<const void*>(fn), dev}).second)
    cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

// rows [0, n) of a row-major source (row r at src + r * stride), widened to fp32, into
// dst[r * ld + c]; rows [n, C) are zero.
template <int D, typename T>
__device__ __forceinline__ void load_rows(float* dst, int ld, const T* src, int64_t stride, int n,
                                          int C) {
  for (int idx = threadIdx.x; idx < C * (D / 4); idx += NT) {
    const int r = idx / (D / 4), c4 = idx % (D / 4);
    const float4 x = (r < n) ? load4(src + r * stride + 4 * c4) : make_float4(0.f, 0.f, 0.f, 0.f);
    *reinterpret_cast<float4*>(dst + r * ld + 4 * c4) = x;
  }
}

template <int D>
__device__ __forceinline__ void load_rows_any(float* dst, int ld, const void* src, bool bf16,
                                              int64_t stride, int n, int C) {
  if (bf16)
    load_rows<D>(dst, ld, static_cast<const __nv_bfloat16*>(src), stride, n, C);
  else
    load_rows<D>(dst, ld, static_cast<const float*>(src), stride, n, C);
}

// D(m, n) = sum_k A(m, k) B(k, n) over shared-memory operands, k ascending with one
// accumulator per output, every output handed to epi(m, n, value).  Layouts:
//   AT = false: A(m, k) = A[m * lda + k]      AT = true: A(m, k) = A[k * lda + m]
//   BT = false: B(k, n) = B[k * ldb + n]      BT = true: B(k, n) = B[n * ldb + k]
// NN and TN: a thread owns a contiguous TM x TN tile; B (and A when AT) are read as float4
// rows along n (m).  NT: a thread owns rows m = mt + r M/TM and columns n = nt + c N/TN, and
// both operands are read as float4 along k, so neighbouring threads read neighbouring rows
// (row strides of 4 mod 32 words keep those reads free of bank conflicts).
// Requires: TM, TN, K multiples of 4; lda, ldb multiples of 4; 16-byte aligned operands.
template <int TM, int TN, bool AT, bool BT, typename Epi>
__device__ __forceinline__ void gemm(int M, int N, int K, const float* __restrict__ A, int lda,
                                     const float* __restrict__ B, int ldb, Epi epi) {
  const int ntn = N / TN;
  const int tiles = (M / TM) * ntn;
  for (int tile = threadIdx.x; tile < tiles; tile += NT) {
    float acc[TM][TN];
#pragma unroll
    for (int r = 0; r < TM; ++r)
#pragma unroll
      for (int c = 0; c < TN; ++c) acc[r][c] = 0.f;
    if constexpr (BT) {
      static_assert(!AT, "TT products are not used");
      const int mt = tile / ntn, nt = tile % ntn;
      const int ms = M / TM, ns = N / TN;
      for (int k = 0; k < K; k += 4) {
        float4 av[TM], bv[TN];
#pragma unroll
        for (int r = 0; r < TM; ++r) av[r] = *reinterpret_cast<const float4*>(A + (mt + r * ms) * lda + k);
#pragma unroll
        for (int c = 0; c < TN; ++c) bv[c] = *reinterpret_cast<const float4*>(B + (nt + c * ns) * ldb + k);
#pragma unroll
        for (int r = 0; r < TM; ++r)
#pragma unroll
          for (int c = 0; c < TN; ++c) {
            acc[r][c] = __fmaf_rn(av[r].x, bv[c].x, acc[r][c]);
            acc[r][c] = __fmaf_rn(av[r].y, bv[c].y, acc[r][c]);
            acc[r][c] = __fmaf_rn(av[r].z, bv[c].z, acc[r][c]);
            acc[r][c] = __fmaf_rn(av[r].w, bv[c].w, acc[r][c]);
          }
      }
#pragma unroll
      for (int r = 0; r < TM; ++r)
#pragma unroll
        for (int c = 0; c < TN; ++c) epi(mt + r * ms, nt + c * ns, acc[r][c]);
    } else {
      // this thread's TN columns: TN/4 groups of 4, group g starting at g * (N / (TN/4)) + 4 * nt
      const int m0 = (tile / ntn) * TM, nt = tile % ntn;
      constexpr int NG = TN / 4;
      const int gstride = N / NG;
      auto col = [&](int c) { return (c / 4) * gstride + 4 * nt + (c % 4); };
      for (int k = 0; k < K; ++k) {
        float av[TM], bv[TN];
        if constexpr (AT) {
#pragma unroll
          for (int r = 0; r < TM; r += 4) {
            const float4 x = *reinterpret_cast<const float4*>(A + k * lda + m0 + r);
            av[r] = x.x; av[r + 1] = x.y; av[r + 2] = x.z; av[r + 3] = x.w;
          }
        } else {
#pragma unroll
          for (int r = 0; r < TM; ++r) av[r] = A[(m0 + r) * lda + k];
        }
#pragma unroll
        for (int c = 0; c < TN; c += 4) {
          const float4 x = *reinterpret_cast<const float4*>(B + k * ldb + col(c));
          bv[c] = x.x; bv[c + 1] = x.y; bv[c + 2] = x.z; bv[c + 3] = x.w;
        }
#pragma unroll
        for (int r = 0; r < TM; ++r)
#pragma unroll
          for (int c = 0; c < TN; ++c) acc[r][c] = __fmaf_rn(av[r], bv[c], acc[r][c]);
      }
#pragma unroll
      for (int r = 0; r < TM; ++r)
#pragma unroll
        for (int c = 0; c < TN; ++c) epi(m0 + r, col(c), acc[r][c]);
    }
  }
}

// src (D x D, row-major, global) -> dst[r * DP + c] = src[c * D + r] (transposed) in shared memory
template <int D>
__device__ __forceinline__ void load_transposed(float* dst, const float* __restrict__ src) {
  constexpr int DP = D + 4;
  for (int e = threadIdx.x; e < D * D; e += NT) dst[(e % D) * DP + e / D] = src[e];
}

// T = (I + A)^{-1} for strictly lower A (C x C in shared memory, row stride CP), blocked
// by 16: diagonal blocks by forward substitution (one column per thread), then the
// off-diagonal blocks by increasing distance from the diagonal.  Xs: 3*16*16 floats.
__device__ __forceinline__ void unit_lower_inverse(const float* A, float* Tm, float* Xs, int C) {
  constexpr int TB = 16;
  const int t = threadIdx.x;
  const int nb = C / TB;
  for (int idx = t; idx < C * C; idx += NT) Tm[(idx / C) * CP + idx % C] = 0.f;
  __syncthreads();
  if (t < C) {
    const int r = t, rend = (r / TB) * TB + TB;
    Tm[r * CP + r] = 1.f;
    for (int i = r + 1; i < rend; ++i) {
      float acc = 0.f;
      for (int m = r; m < i; ++m) acc = __fmaf_rn(A[i * CP + m], Tm[m * CP + r], acc);
      Tm[i * CP + r] = -acc;
    }
  }
  __syncthreads();
  for (int off = 1; off < nb; ++off) {
    const int nel = (nb - off) * TB * TB;
    for (int e = t; e < nel; e += NT) {
      const int I = off + e / (TB * TB), ii = (e / TB) % TB, rr = e % TB;
      const int i = I * TB + ii, r = (I - off) * TB + rr;
      float acc = 0.f;
      for (int m = r; m < I * TB; ++m) acc = __fmaf_rn(A[i * CP + m], Tm[m * CP + r], acc);
      Xs[e] = acc;
    }
    __syncthreads();
    for (int e = t; e < nel; e += NT) {
      const int I = off + e / (TB * TB), ii = (e / TB) % TB, rr = e % TB;
      const int i = I * TB + ii, r = (I - off) * TB + rr;
      const float* X = Xs + (e / (TB * TB)) * TB * TB;
      float acc = 0.f;
      for (int m = I * TB; m <= i; ++m) acc = __fmaf_rn(Tm[i * CP + m], X[(m - I * TB) * TB + rr], acc);
      Tm[i * CP + r] = -acc;
    }
    __syncthreads();
  }
}

// Per chunk-head workspace (floats), chunk length padded to C.
struct BwdBufs {
  float *W, *Ut, *T, *P, *G, *L, *dSE, *U, *dU, *dOS0, *UdSe, *dW, *sdot;
  float* img;  // tensor-core shapes: per chunk-head the K rows bf16 image, then scratch
  float *dq_part, *dk_part;  // [T, Hv, D]
};

struct BwdArgs {
  Dims dm;
  TokenArrays in;
  const void* dO;
  const ChunkRec* chunks;
  const SeqRec* seqs;
  const float* saved_bnd;
  const float* dstate_out;
  float* dstate_in;
  BwdBufs b;
  float *dq, *dk, *dv, *dg, *dbeta;
  int64_t T;
  int64_t n_chunks;  // chunk records (rows of saved_bnd and of the per-chunk workspace)
  int N;             // sequences
  WsHeader* hdr;
};

// ===================================================================  KB1  ====
template <int D>
constexpr size_t bprep_smem() {
  return sizeof(float) * (4 * kMaxChunk * (D + 4) + 2 * kMaxChunk * CP + 6 * kMaxChunk + 3 * 256);
}

template <int D, typename Tin>
__global__ void __launch_bounds__(NT) k_bwd_prep(BwdArgs a) {
  constexpr int DP = D + 4;
  extern __shared__ __align__(16) float sm[];
  float* B0 = sm;                 // K, then dO
  float* B1 = B0 + kMaxChunk * DP;  // V, then Ut
  float* B2 = B1 + kMaxChunk * DP;  // W
  float* B3 = B2 + kMaxChunk * DP;  // Q, then Qt = diag(e^G) Q - P W
  float* M0 = B3 + kMaxChunk * DP;  // A, then P
  float* M1 = M0 + kMaxChunk * CP;  // T
  float* gs = M1 + kMaxChunk * CP;
  float* Gs = gs + kMaxChunk;
  float* bs = Gs + kMaxChunk;
  float* eG = bs + kMaxChunk;
  float* bk = eG + kMaxChunk;
  float* Xs = bk + 2 * kMaxChunk;
  if (!a.hdr->valid) return;
  const Dims dm = a.dm;
  const int t = threadIdx.x, C = dm.C;
  const int64_t c = blockIdx.x;
  const int h = blockIdx.y, hq = h / (dm.hv / dm.hqk);
  const ChunkRec rec = a.chunks[c];
  if (!in_bounds(a.hdr, rec.tok0 >= 0 && rec.len >= 0 && rec.len <= a.dm.C && (int64_t)rec.tok0 + rec.len <= a.T))
    return;
  const int n = rec.len;
  const int64_t tok0 = rec.tok0;
  const int64_t ch = c * dm.hv + h;
  const Tin* kin = static_cast<const Tin*>(a.in.k);
  const Tin* vin = static_cast<const Tin*>(a.in.v);
  const Tin* qin = static_cast<const Tin*>(a.in.q);

  load_rows<D>(B0, DP, kin + (tok0 * dm.hqk + hq) * D, (int64_t)dm.hqk * D, n, C);
  load_rows<D>(B1, DP, vin + (tok0 * dm.hv + h) * D, (int64_t)dm.hv * D, n, C);
  if (t < C) {
    gs[t] = t < n ? a.in.g[(tok0 + t) * dm.hv + h] : 0.f;
    bs[t] = t < n ? a.in.beta[(tok0 + t) * dm.hv + h] : 0.f;
  }
  __syncthreads();
  if (t == 0) {
    float run = gs[0];
    Gs[0] = run;
#pragma unroll 8
    for (int i = 1; i < C; ++i) {
      run = __fadd_rn(run, gs[i]);
      Gs[i] = run;
    }
  }
  __syncthreads();
  if (t < C) {
    eG[t] = expf(Gs[t]);
    bk[t] = __fmul_rn(bs[t], eG[t]);
  }
  for (int o = t; o < C * C; o += NT) {
    const int i = o / C, s = o % C;
    M0[i * CP + s] = (i > s) ? __fmul_rn(__fmul_rn(bs[i], expf(__fsub_rn(Gs[i], Gs[s]))),
                                         dot_canon<D>(B0 + i * DP, B0 + s * DP))
                             : 0.f;
  }
  __syncthreads();
  unit_lower_inverse(M0, M1, Xs, C);
  // W = T diag(beta e^G) K, Ut = T diag(beta) V (r ascending)
  constexpr int RG = NT / D;
  constexpr int RPT = kMaxChunk / RG;
  {
    const int cc = t % D, i0 = t / D;
    float aw[RPT], au[RPT];
#pragma unroll
    for (int j = 0; j < RPT; ++j) aw[j] = au[j] = 0.f;
    for (int r = 0; r < C; ++r) {
      const float kv = B0[r * DP + cc], vv = B1[r * DP + cc];
#pragma unroll
      for (int j = 0; j < RPT; ++j) {
        const int i = i0 + RG * j;
        if (i >= r && i < C) {
          const float tr = M1[i * CP + r];
          aw[j] = __fmaf_rn(__fmul_rn(tr, bk[r]), kv, aw[j]);
          au[j] = __fmaf_rn(__fmul_rn(tr, bs[r]), vv, au[j]);
        }
      }
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
      const int i = i0 + RG * j;
      if (i < C) {
        B2[i * DP + cc] = aw[j];
        B1[i * DP + cc] = au[j];
        a.b.W[ch * C * D + i * D + cc] = aw[j];
        a.b.Ut[ch * C * D + i * D + cc] = au[j];
      }
    }
  }
  for (int o = t; o < C * C; o += NT) a.b.T[ch * C * C + o] = M1[(o / C) * CP + o % C];
  if (t < C) a.b.G[ch * C + t] = Gs[t];
  load_rows<D>(B3, DP, qin + (tok0 * dm.hqk + hq) * D, (int64_t)dm.hqk * D, n, C);
  __syncthreads();
  if constexpr (D == 128) {
    if (boundary_on_tensor_cores(dm)) {  // operand images for the tensor-core reverse chain
      unsigned char* img = reinterpret_cast<unsigned char*>(a.b.img + ch * (int64_t)prep_w_floats(C, D));
      for (int q = t; q < C * (D / 8); q += NT) {  // K rows (exact in bf16)
        int r, c0;
        tc::kmajor_piece(q, D, r, c0);
        uint32_t w4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          w4[e] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(B0[r * DP + c0 + 2 * e])) |
                  ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(B0[r * DP + c0 + 2 * e + 1])) << 16);
        *reinterpret_cast<uint4*>(img + tc::kmajor_off(r, c0, D)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
      for (int q = t; q < D * (C / 8); q += NT) {  // W^T split: row c, 8 chunk positions
        const int cc = q % D, i0 = (q / D) * 8;
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          __nv_bfloat16 h0, l0, h1, l1;
          tc::split_bf16(B2[(i0 + 2 * e) * DP + cc], h0, l0);
          tc::split_bf16(B2[(i0 + 2 * e + 1) * DP + cc], h1, l1);
          hw[e] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
          lw[e] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
        }
        const uint32_t off = tc::kmajor_off(cc, i0, C);
        *reinterpret_cast<uint4*>(img + C * D * 2 + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4*>(img + 2 * C * D * 2 + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
    }
  }
  // P = Gam * (Q K^T), lower triangle with diagonal
  gemm<4, 4, false, true>(C, C, D, B3, DP, B0, DP, [&](int i, int s, float v) {
    const float p = (i >= s) ? __fmul_rn(expf(__fsub_rn(Gs[i], Gs[s])), v) : 0.f;
    M0[i * CP + s] = p;
    a.b.P[ch * C * C + i * C + s] = p;
  });
  __syncthreads();
  // Qt = diag(e^G) Q - P W (in place)
  gemm<4, 8, false, false>(C, D, C, M0, CP, B2, DP, [&](int i, int k, float v) {
    B3[i * DP + k] = __fsub_rn(__fmul_rn(eG[i], B3[i * DP + k]), v);
  });
  __syncthreads();
  if (a.dm.out_bf16)
    load_rows<D>(B0, DP, static_cast<const __nv_bfloat16*>(a.dO) + (tok0 * dm.hv + h) * D,
                 (int64_t)dm.hv * D, n, C);
  else
    load_rows<D>(B0, DP, static_cast<const float*>(a.dO) + (tok0 * dm.hv + h) * D,
                 (int64_t)dm.hv * D, n, C);
  __syncthreads();
  // L = dO^T Qt  (D x D)
  gemm<8, 8, true, false>(D, D, C, B0, DP, B3, DP,
                          [&](int p, int q, float v) { a.b.L[ch * D * D + p * D + q] = v; });
}

// ===================================================================  KB2  ====
template <int D>
constexpr size_t bchain_smem() {
  return sizeof(float) * (2 * kMaxChunk * (D + 4) + 2 * kRowsPerChain * (D + 4) +
                          kMaxChunk * kRowsPerChain + 2 * kMaxChunk);
}

template <int D, typename Tin>
__global__ void __launch_bounds__(NT) k_bwd_chain(BwdArgs a) {
  constexpr int DP = D + 4;
  constexpr int R = kRowsPerChain;
  extern __shared__ __align__(16) float sm[];
  float* Ks = sm;
  float* Ws = Ks + kMaxChunk * DP;
  float* dS = Ws + kMaxChunk * DP;
  float* Ls = dS + R * DP;
  float* Xd = Ls + R * DP;
  float* dec = Xd + kMaxChunk * R;
  float* gm = dec + kMaxChunk;
  if (!a.hdr->valid) return;
  const Dims dm = a.dm;
  const int t = threadIdx.x, C = dm.C;
  const int n = blockIdx.x, h = blockIdx.y, r0 = blockIdx.z * R;
  const int hq = h / (dm.hv / dm.hqk);
  const SeqRec rec = a.seqs[n];
  if (!in_bounds(a.hdr, rec.chunk0 >= 0 && (int64_t)rec.chunk0 + rec.nchunks <= a.n_chunks && rec.tok0 >= 0 &&
                            (int64_t)rec.tok0 + rec.len <= a.T))
    return;
  const int64_t SZ = (int64_t)D * D;
  const Tin* kin = static_cast<const Tin*>(a.in.k);
  for (int idx = t; idx < R * D; idx += NT) {
    const int i = idx / D, cc = idx % D;
    dS[i * DP + cc] = a.dstate_out ? a.dstate_out[((int64_t)n * dm.hv + h) * SZ + (int64_t)(r0 + i) * D + cc] : 0.f;
  }
  __syncthreads();
  for (int j = rec.nchunks - 1; j >= 0; --j) {
    const int64_t c = (int64_t)rec.chunk0 + j;
    const ChunkRec cr = a.chunks[c];
    const int64_t ch = c * dm.hv + h;
    for (int idx = t; idx < R * D; idx += NT) {
      const int i = idx / D, cc = idx % D;
      a.b.dSE[ch * SZ + (int64_t)(r0 + i) * D + cc] = dS[i * DP + cc];
      Ls[i * DP + cc] = a.b.L[ch * SZ + (int64_t)(r0 + i) * D + cc];
    }
    load_rows<D>(Ks, DP, kin + ((int64_t)cr.tok0 * dm.hqk + hq) * D, (int64_t)dm.hqk * D, cr.len, C);
    load_rows<D>(Ws, DP, a.b.W + ch * C * D, D, C, C);
    if (t < C) dec[t] = expf(__fsub_rn(a.b.G[ch * C + C - 1], a.b.G[ch * C + t]));
    if (t == 0) gm[0] = expf(a.b.G[ch * C + C - 1]);
    __syncthreads();
    {  // Xd[s][i] = -dec_s (k_s . dS_i)
      const int i = t / 16, s0 = t % 16;
      for (int s = s0; s < C; s += 16)
        Xd[s * R + i] = __fmul_rn(-dec[s], dot_canon<D>(Ks + s * DP, dS + i * DP));
    }
    __syncthreads();
    {  // dS <- L + gamma dS + sum_s Xd[s][i] W[s]
      constexpr int RG = NT / D;
      constexpr int RJ = R / RG;
      const int cc = t % D, i0 = t / D;
      const float g = gm[0];
      float acc[RJ];
#pragma unroll
      for (int jj = 0; jj < RJ; ++jj) {
        const int i = i0 + RG * jj;
        acc[jj] = __fadd_rn(Ls[i * DP + cc], __fmul_rn(g, dS[i * DP + cc]));
      }
      for (int s = 0; s < C; ++s) {
        const float wv = Ws[s * DP + cc];
#pragma unroll
        for (int jj = 0; jj < RJ; ++jj) acc[jj] = __fmaf_rn(Xd[s * R + i0 + RG * jj], wv, acc[jj]);
      }
      __syncthreads();
#pragma unroll
      for (int jj = 0; jj < RJ; ++jj) dS[(i0 + RG * jj) * DP + cc] = acc[jj];
    }
    __syncthreads();
  }
  if (a.dstate_in) {
    for (int idx = t; idx < R * D; idx += NT) {
      const int i = idx / D, cc = idx % D;
      a.dstate_in[((int64_t)n * dm.hv + h) * SZ + (int64_t)(r0 + i) * D + cc] = dS[i * DP + cc];
    }
  }
}

// ===================================================================  KB3  ====
template <int D>
constexpr size_t bbig_smem() {
  return sizeof(float) * (4 * kMaxChunk * (D + 4) + kMaxChunk * CP + D * (D + 4) + kMaxChunk + NT);
}

template <int D, typename Tin>
__global__ void __launch_bounds__(NT) k_bwd_big(BwdArgs a) {
  constexpr int DP = D + 4;
  extern __shared__ __align__(16) float sm[];
  float* B0 = sm;                   // W, then dU
  float* B1 = B0 + kMaxChunk * DP;  // Ut, then U
  float* B2 = B1 + kMaxChunk * DP;  // dO
  float* B3 = B2 + kMaxChunk * DP;  // K
  float* M0 = B3 + kMaxChunk * DP;  // P
  float* SM = M0 + kMaxChunk * CP;  // S0, dS_end, S0
  float* dec = SM + D * DP;
  float* red = dec + kMaxChunk;
  if (!a.hdr->valid) return;
  const Dims dm = a.dm;
  const int t = threadIdx.x, C = dm.C;
  const int64_t c = blockIdx.x;
  const int h = blockIdx.y, hq = h / (dm.hv / dm.hqk);
  const ChunkRec rec = a.chunks[c];
  if (!in_bounds(a.hdr, rec.tok0 >= 0 && rec.len >= 0 && rec.len <= a.dm.C && (int64_t)rec.tok0 + rec.len <= a.T))
    return;
  const int n = rec.len;
  const int64_t tok0 = rec.tok0;
  const int64_t ch = c * dm.hv + h;
  const int64_t SZ = (int64_t)D * D;
  const Tin* kin = static_cast<const Tin*>(a.in.k);
  load_rows<D>(B0, DP, a.b.W + ch * C * D, D, C, C);
  load_rows<D>(B1, DP, a.b.Ut + ch * C * D, D, C, C);
  load_rows_any<D>(B2, DP, a.dm.out_bf16
                               ? static_cast<const void*>(static_cast<const __nv_bfloat16*>(a.dO) + (tok0 * dm.hv + h) * D)
                               : static_cast<const void*>(static_cast<const float*>(a.dO) + (tok0 * dm.hv + h) * D),
                   a.dm.out_bf16, (int64_t)dm.hv * D, n, C);
  load_rows<D>(B3, DP, kin + (tok0 * dm.hqk + hq) * D, (int64_t)dm.hqk * D, n, C);
  for (int o = t; o < C * C; o += NT) M0[(o / C) * CP + o % C] = a.b.P[ch * C * C + o];
  if (t < C) dec[t] = expf(__fsub_rn(a.b.G[ch * C + C - 1], a.b.G[ch * C + t]));
  load_transposed<D>(SM, a.saved_bnd + ch * SZ);
  __syncthreads();
  // U = Ut - W S0^T (in place; SM holds S0^T)
  gemm<4, 8, false, false>(C, D, D, B0, DP, SM, DP, [&](int s, int q, float v) {
    const float u = __fsub_rn(B1[s * DP + q], v);
    B1[s * DP + q] = u;
    a.b.U[ch * C * D + s * D + q] = u;
  });
  {  // <dS_end, S0> straight from global memory
    float part = 0.f;
    for (int e = t; e < D * D; e += NT) part = __fmaf_rn(a.b.dSE[ch * SZ + e], a.saved_bnd[ch * SZ + e], part);
    red[t] = part;
  }
  __syncthreads();
  for (int w = NT / 2; w > 0; w >>= 1) {
    if (t < w) red[t] = __fadd_rn(red[t], red[t + w]);
    __syncthreads();
  }
  if (t == 0) a.b.sdot[ch] = red[0];
  load_rows<D>(SM, DP, a.saved_bnd + ch * SZ, D, D, D);
  __syncthreads();
  // dO S0
  gemm<4, 8, false, false>(C, D, D, B2, DP, SM, DP,
                           [&](int i, int q, float v) { a.b.dOS0[ch * C * D + i * D + q] = v; });
  // dU = P^T dO (+ below)
  gemm<4, 8, true, false>(C, D, C, M0, CP, B2, DP, [&](int s, int q, float v) { B0[s * DP + q] = v; });
  __syncthreads();
  load_transposed<D>(SM, a.b.dSE + ch * SZ);
  __syncthreads();
  // dU += diag(dec) K dS_end^T (SM holds dS_end^T)
  gemm<4, 8, false, false>(C, D, D, B3, DP, SM, DP, [&](int s, int q, float v) {
    const float du = __fmaf_rn(dec[s], v, B0[s * DP + q]);
    B0[s * DP + q] = du;
    a.b.dU[ch * C * D + s * D + q] = du;
  });
  __syncthreads();
  load_rows<D>(SM, DP, a.b.dSE + ch * SZ, D, D, D);
  __syncthreads();
  // U dS_end
  gemm<4, 8, false, false>(C, D, D, B1, DP, SM, DP,
                           [&](int s, int q, float v) { a.b.UdSe[ch * C * D + s * D + q] = v; });
  __syncthreads();
  load_rows<D>(SM, DP, a.saved_bnd + ch * SZ, D, D, D);
  __syncthreads();
  // dW = -dU S0
  gemm<4, 8, false, false>(C, D, D, B0, DP, SM, DP,
                           [&](int s, int q, float v) { a.b.dW[ch * C * D + s * D + q] = -v; });
}

// ===================================================================  KB4  ====
template <int D>
constexpr size_t bgrad_smem() {
  return sizeof(float) * (5 * kMaxChunk * (D + 4) + 2 * kMaxChunk * CP + 16 * kMaxChunk);
}

template <int D, typename Tin>
__global__ void __launch_bounds__(NT) k_bwd_grad(BwdArgs a) {
  constexpr int DP = D + 4;
  extern __shared__ __align__(16) float sm[];
  float* B0 = sm;                   // dO -> dU -> Y
  float* B1 = B0 + kMaxChunk * DP;  // U -> dW -> W -> Ut -> U dS_end
  float* B2 = B1 + kMaxChunk * DP;  // Q
  float* B3 = B2 + kMaxChunk * DP;  // K
  float* B4 = B3 + kMaxChunk * DP;  // dO S0 -> X
  float* M0 = B4 + kMaxChunk * DP;  // Pm -> A' = Gam k.k
  float* M1 = M0 + kMaxChunk * CP;  // QK -> T -> dA -> dAm
  float* Gs = M1 + kMaxChunk * CP;
  float* eG = Gs + kMaxChunk;
  float* dec = eG + kMaxChunk;
  float* bs = dec + kMaxChunk;
  float* dGa = bs + kMaxChunk;
  float* dGb = dGa + kMaxChunk;
  float* dGe = dGb + kMaxChunk;
  float* kY = dGe + kMaxChunk;
  float* dba = kY + kMaxChunk;
  float* dbc = dba + kMaxChunk;
  float* cs = dbc + kMaxChunk;
  float* dgv = cs + kMaxChunk;
  if (!a.hdr->valid) return;
  const Dims dm = a.dm;
  const int t = threadIdx.x, C = dm.C;
  const int64_t c = blockIdx.x;
  const int h = blockIdx.y, hq = h / (dm.hv / dm.hqk);
  const ChunkRec rec = a.chunks[c];
  if (!in_bounds(a.hdr, rec.tok0 >= 0 && rec.len >= 0 && rec.len <= a.dm.C && (int64_t)rec.tok0 + rec.len <= a.T))
    return;
  const int n = rec.len;
  const int64_t tok0 = rec.tok0;
  const int64_t ch = c * dm.hv + h;
  const Tin* kin = static_cast<const Tin*>(a.in.k);
  const Tin* qin = static_cast<const Tin*>(a.in.q);
  const Tin* vin = static_cast<const Tin*>(a.in.v);
  const float* Gc = a.b.G + ch * C;

  // ---- pass A: Pm = Gam * (dO U^T) (lower with diagonal), QK strictly lower, dG from P
  load_rows_any<D>(B0, DP, a.dm.out_bf16
                               ? static_cast<const void*>(static_cast<const __nv_bfloat16*>(a.dO) + (tok0 * dm.hv + h) * D)
                               : static_cast<const void*>(static_cast<const float*>(a.dO) + (tok0 * dm.hv + h) * D),
                   a.dm.out_bf16, (int64_t)dm.hv * D, n, C);
  load_rows<D>(B1, DP, a.b.U + ch * C * D, D, C, C);
  load_rows<D>(B2, DP, qin + (tok0 * dm.hqk + hq) * D, (int64_t)dm.hqk * D, n, C);
  load_rows<D>(B3, DP, kin + (tok0 * dm.hqk + hq) * D, (int64_t)dm.hqk * D, n, C);
  if (t < C) {
    Gs[t] = Gc[t];
    bs[t] = t < n ? a.in.beta[(tok0 + t) * dm.hv + h] : 0.f;
  }
  __syncthreads();
  if (t < C) {
    eG[t] = expf(Gs[t]);
    dec[t] = expf(__fsub_rn(Gs[C - 1], Gs[t]));
  }
  gemm<4, 4, false, true>(C, C, D, B0, DP, B1, DP, [&](int i, int s, float v) {
    M0[i * CP + s] = (i >= s) ? __fmul_rn(expf(__fsub_rn(Gs[i], Gs[s])), v) : 0.f;
  });
  gemm<4, 4, false, true>(C, C, D, B2, DP, B3, DP,
                          [&](int i, int s, float v) { M1[i * CP + s] = (i > s) ? v : 0.f; });
  __syncthreads();
  if (t < C) {
    float row = 0.f, col = 0.f;
    for (int s = 0; s < t; ++s) row = __fmaf_rn(M0[t * CP + s], M1[t * CP + s], row);
    for (int i = t + 1; i < C; ++i) col = __fmaf_rn(M0[i * CP + t], M1[i * CP + t], col);
    dGb[t] = __fsub_rn(row, col);
  }
  // ---- pass B: dQ = diag(e^G) dO S0 + Pm K;  dK <- Pm^T Q
  load_rows<D>(B4, DP, a.b.dOS0 + ch * C * D, D, C, C);
  __syncthreads();
  gemm<4, 8, false, false>(C, D, C, M0, CP, B3, DP, [&](int i, int k, float v) {
    if (i < n) a.b.dq_part[((tok0 + i) * dm.hv + h) * D + k] = __fmaf_rn(eG[i], B4[i * DP + k], v);
  });
  if (t < C) dGa[t] = __fmul_rn(eG[t], dot_canon<D>(B4 + t * DP, B2 + t * DP));
  constexpr int KTN = 8;
  const int ntn = D / KTN;
  const bool owns = t < (C / 4) * ntn;
  const int km0 = (t / ntn) * 4, kn0 = (t % ntn) * KTN;
  float dk[4][KTN];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int q = 0; q < KTN; ++q) dk[r][q] = 0.f;
  if (owns) {
    for (int i = 0; i < C; ++i) {
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float pm = M0[i * CP + km0 + r];
#pragma unroll
        for (int q = 0; q < KTN; ++q) dk[r][q] = __fmaf_rn(pm, B2[i * DP + kn0 + q], dk[r][q]);
      }
    }
  }
  __syncthreads();
  // ---- pass C: X = T^T dU -> B4, Y = T^T dW -> B0, dV, kY, dbeta(v)
  load_rows<D>(B0, DP, a.b.dU + ch * C * D, D, C, C);
  load_rows<D>(B1, DP, a.b.dW + ch * C * D, D, C, C);
  for (int o = t; o < C * C; o += NT) M1[(o / C) * CP + o % C] = a.b.T[ch * C * C + o];
  __syncthreads();
  gemm<4, 8, true, false>(C, D, C, M1, CP, B0, DP, [&](int s, int k, float v) { B4[s * DP + k] = v; });
  __syncthreads();
  gemm<4, 8, true, false>(C, D, C, M1, CP, B1, DP, [&](int s, int k, float v) { B0[s * DP + k] = v; });
  __syncthreads();
  for (int idx = t; idx < C * D; idx += NT) {
    const int i = idx / D, k = idx % D;
    if (i < n) a.dv[((tok0 + i) * dm.hv + h) * D + k] = __fmul_rn(bs[i], B4[i * DP + k]);
  }
  if (t < C) {
    kY[t] = dot_canon<D>(B3 + t * DP, B0 + t * DP);
    float acc = 0.f;
    if (t < n) {
      const Tin* vr = vin + ((tok0 + t) * dm.hv + h) * D;
      for (int k = 0; k < D; ++k) acc = __fmaf_rn(to_f32(vr[k]), B4[t * DP + k], acc);
    }
    dba[t] = acc;
  }
  // ---- pass D: dA = -(Y W^T + X Ut^T) strictly lower; A' = Gam k.k; dG, dbeta from A
  load_rows<D>(B1, DP, a.b.W + ch * C * D, D, C, C);
  __syncthreads();
  gemm<4, 4, false, true>(C, C, D, B0, DP, B1, DP,
                          [&](int i, int s, float v) { M1[i * CP + s] = (i > s) ? -v : 0.f; });
  __syncthreads();
  load_rows<D>(B1, DP, a.b.Ut + ch * C * D, D, C, C);
  __syncthreads();
  gemm<4, 4, false, true>(C, C, D, B4, DP, B1, DP, [&](int i, int s, float v) {
    if (i > s) M1[i * CP + s] = __fsub_rn(M1[i * CP + s], v);
  });
  gemm<4, 4, false, true>(C, C, D, B3, DP, B3, DP, [&](int i, int s, float v) {
    M0[i * CP + s] = (i > s) ? __fmul_rn(expf(__fsub_rn(Gs[i], Gs[s])), v) : 0.f;
  });
  __syncthreads();
  if (t < C) {
    float b = 0.f, row = 0.f, col = 0.f;
    for (int s = 0; s < t; ++s) {
      b = __fmaf_rn(M1[t * CP + s], M0[t * CP + s], b);
      row = __fmaf_rn(__fmul_rn(M1[t * CP + s], bs[t]), M0[t * CP + s], row);
    }
    for (int i = t + 1; i < C; ++i) col = __fmaf_rn(__fmul_rn(M1[i * CP + t], bs[i]), M0[i * CP + t], col);
    dbc[t] = b;
    dGe[t] = __fsub_rn(row, col);
  }
  __syncthreads();
  for (int o = t; o < C * C; o += NT) {  // dAm = dA * beta_i * Gam_is
    const int i = o / C, s = o % C;
    if (i > s)
      M1[i * CP + s] = __fmul_rn(__fmul_rn(M1[i * CP + s], bs[i]), expf(__fsub_rn(Gs[i], Gs[s])));
  }
  load_rows<D>(B1, DP, a.b.UdSe + ch * C * D, D, C, C);
  __syncthreads();
  // ---- pass E: dK += dAm K + dAm^T K + diag(dec) U dS_end + diag(beta e^G) Y
  if (owns) {
    for (int r = 0; r < C; ++r) {
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const float am = M1[(km0 + rr) * CP + r];
#pragma unroll
        for (int q = 0; q < KTN; ++q) dk[rr][q] = __fmaf_rn(am, B3[r * DP + kn0 + q], dk[rr][q]);
      }
    }
    for (int r = 0; r < C; ++r) {
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const float am = M1[r * CP + km0 + rr];
#pragma unroll
        for (int q = 0; q < KTN; ++q) dk[rr][q] = __fmaf_rn(am, B3[r * DP + kn0 + q], dk[rr][q]);
      }
    }
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int s = km0 + rr;
      const float bkv = __fmul_rn(bs[s], eG[s]);
#pragma unroll
      for (int q = 0; q < KTN; ++q) {
        float v = __fmaf_rn(dec[s], B1[s * DP + kn0 + q], dk[rr][q]);
        v = __fmaf_rn(bkv, B0[s * DP + kn0 + q], v);
        if (s < n) a.b.dk_part[((tok0 + s) * dm.hv + h) * D + kn0 + q] = v;
      }
    }
  }
  if (t < C) cs[t] = __fmul_rn(dec[t], dot_canon<D>(B1 + t * DP, B3 + t * DP));
  __syncthreads();
  // ---- pass F: dG, reverse cumulative sum -> dg; dbeta
  if (t == 0) {
    float tot = 0.f;
    for (int s = 0; s < C; ++s) tot = __fadd_rn(tot, cs[s]);
    float run = 0.f;
    for (int i = C - 1; i >= 0; --i) {
      float v = __fadd_rn(dGa[i], dGb[i]);
      v = __fsub_rn(v, cs[i]);
      v = __fmaf_rn(__fmul_rn(bs[i], eG[i]), kY[i], v);
      v = __fadd_rn(v, dGe[i]);
      if (i == C - 1) v = __fadd_rn(v, __fmaf_rn(expf(Gs[C - 1]), a.b.sdot[ch], tot));
      run = __fadd_rn(run, v);
      dgv[i] = run;
    }
  }
  __syncthreads();
  if (t < n) {
    a.dg[(tok0 + t) * dm.hv + h] = dgv[t];
    a.dbeta[(tok0 + t) * dm.hv + h] = __fadd_rn(__fmaf_rn(eG[t], kY[t], dba[t]), dbc[t]);
  }
}

// ===================================================================  KB5  ====
__global__ void k_bwd_gqa(const float* __restrict__ dq_part, const float* __restrict__ dk_part,
                          float* __restrict__ dq, float* __restrict__ dk, int64_t T, int hqk,
                          int hv, int D, const WsHeader* __restrict__ hdr) {
  if (!hdr->valid) return;
  // one thread per float4 of one (token, query/key head) row; a block covers 256 / (D / 4)
  // rows; the value heads of the group are summed in ascending order
  const int grp = hv / hqk, d4 = D / 4;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x / d4) + threadIdx.x / d4;
  if (row >= T * hqk) return;
  const int c = 4 * (threadIdx.x % d4);
  const int64_t tok = row / hqk;
  const int hq = (int)(row - tok * hqk);
  const int64_t base = (tok * hv + (int64_t)hq * grp) * D + c;
  float4 sq = *reinterpret_cast<const float4*>(dq_part + base);
  float4 sk = *reinterpret_cast<const float4*>(dk_part + base);
  for (int j = 1; j < grp; ++j) {
    const float4 xq = *reinterpret_cast<const float4*>(dq_part + base + (int64_t)j * D);
    const float4 xk = *reinterpret_cast<const float4*>(dk_part + base + (int64_t)j * D);
    sq = make_float4(__fadd_rn(sq.x, xq.x), __fadd_rn(sq.y, xq.y), __fadd_rn(sq.z, xq.z), __fadd_rn(sq.w, xq.w));
    sk = make_float4(__fadd_rn(sk.x, xk.x), __fadd_rn(sk.y, xk.y), __fadd_rn(sk.z, xk.z), __fadd_rn(sk.w, xk.w));
  }
  *reinterpret_cast<float4*>(dq + row * D + c) = sq;
  *reinterpret_cast<float4*>(dk + row * D + c) = sk;
}

// ============================================================  KB2 (tcgen05)  ===
// Reverse boundary chain on tensor cores (bf16 inputs, d = 128, C = 64): one CTA of 256
// threads per (sequence, head); adjoint row i is TMEM lane i, read by the two warps of its
// lane quadrant, one half of the columns each.  Per chunk j, from the end adjoint
// dS = dS^(j+1):
//     D1 (128 x 64)  = dS K^T                     2 MMAs: dS_hi K + dS_lo K (K exact)
//     D2 (128 x 128) = gamma_j dS + dO_j^T Qt_j    D2 preloaded; 2 MMAs (Qt = Qt_hi + Qt_lo,
//                                                  bf16 dO exact; fp32 dO: 3)
//     Xd[i][s]       = -dec_s D1[i][s]            (split to bf16 hi/lo)
//     D2            += Xd W                       3 MMAs with W = W_hi + W_lo
// giving dS^(j).  The K rows and W rows (hi | lo) images come by bulk copy a chunk ahead;
// the dO and Qt rows images (the prep kernel's, in L's slot) by another, issued as soon as
// the previous step's Xd W has consumed the region.  W^T, dO^T and Qt^T are the MN-major
// readings of the row images.
namespace tcb {
constexpr int D = 128, C = 64;
constexpr uint32_t A1_BYTES = 128 * D * 2, A2_BYTES = 128 * C * 2, STAGE_BYTES = 3 * C * D * 2;
// the L = dO^T Qt operands of a step, as the prep kernel left them in L's slot (row images):
// dO hi | Qt hi | Qt lo | dO lo (the last only for fp32 dO); Xd is built over them
constexpr uint32_t IMG = C * D * 2, LA_BYTES = 4 * IMG;
constexpr size_t SMEM = 2 * (size_t)A1_BYTES + 2 * (size_t)STAGE_BYTES + LA_BYTES + 64 * 4 + 64;
constexpr uint32_t TMEM_COLS = 256, D1_COL = 0, D2_COL = 64;
static_assert(2 * A2_BYTES <= LA_BYTES, "Xd hi | lo over the L operands");
}  // namespace tcb

__device__ __forceinline__ void split_store16(unsigned char* hi, unsigned char* lo, int row, int k0, int K,
                                              const float* v) {
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      __nv_bfloat16 h0, l0, h1, l1;
      tc::split_bf16(v[8 * g + 2 * e], h0, l0);
      tc::split_bf16(v[8 * g + 2 * e + 1], h1, l1);
      hw[e] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
      lw[e] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
    }
    const uint32_t off = tc::kmajor_off(row, k0 + 8 * g, K);
    *reinterpret_cast<uint4*>(hi + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint4*>(lo + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
  }
}

__global__ void __launch_bounds__(256, 1) k_bwd_chain_tc(BwdArgs a) {
  using namespace tcb;
  using namespace tc;
  extern __shared__ __align__(128) unsigned char smb[];
  unsigned char* A1h = smb;
  unsigned char* A1l = A1h + A1_BYTES;
  unsigned char* stage0 = A1l + A1_BYTES;
  unsigned char* LA = stage0 + 2 * STAGE_BYTES;  // this step's dO, Qt rows images; then Xd
  unsigned char* A2h = LA;
  unsigned char* A2l = LA + A2_BYTES;
  float* decs = reinterpret_cast<float*>(LA + LA_BYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(decs + 64);  // stage 0, stage 1, MMA, L operands
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 4);
  if (!a.hdr->valid) return;
  const Dims dm = a.dm;
  // warp w reads TMEM lanes 32 (w % 4) .. + 31 (state rows) and column half w / 4
  const int t = threadIdx.x, warp = t >> 5, row = (warp & 3) * 32 + (t & 31), half = warp >> 2;
  const int cs0 = half * (D / 2), us0 = half * (C / 2);
  // CTA b = blockIdx.y * gridDim.x + blockIdx.x (launch order) takes the b-th (sequence, head)
  // with the sequences longest first (ranked by chunk count, ties by index; up to 64
  // sequences, beyond that in sequence order), so that the longest chains do not start last
  constexpr int kRankSeqs = 64;
  __shared__ int s_nch[kRankSeqs], s_order[kRankSeqs];
  const bool by_length = a.N <= kRankSeqs;
  if (by_length && t < a.N) s_nch[t] = a.seqs[t].nchunks;
  __syncthreads();
  if (by_length && t < a.N) {
    const int mine = s_nch[t];
    int r = 0;
    for (int s2 = 0; s2 < a.N; ++s2) r += (s_nch[s2] > mine || (s_nch[s2] == mine && s2 < t)) ? 1 : 0;
    s_order[r] = t;
  }
  __syncthreads();
  const int lin = (int)(blockIdx.y * gridDim.x + blockIdx.x);
  const int n = by_length ? s_order[lin / dm.hv] : (int)blockIdx.x;
  const int h = by_length ? lin % dm.hv : (int)blockIdx.y;
  const SeqRec rec = a.seqs[n];
  if (!in_bounds(a.hdr, rec.chunk0 >= 0 && (int64_t)rec.chunk0 + rec.nchunks <= a.n_chunks && rec.tok0 >= 0 &&
                            (int64_t)rec.tok0 + rec.len <= a.T))
    return;
  const int64_t SZ = (int64_t)D * D;
  const int64_t IW = (int64_t)prep_w_floats(C, D);
  const int64_t srow = ((int64_t)n * dm.hv + h) * SZ + (int64_t)row * D;
  const int nch = rec.nchunks;
  if (nch == 0) {  // no tokens: dstate_in = dstate_out
    if (a.dstate_in)
      for (int c0 = cs0; c0 < cs0 + D / 2; ++c0) a.dstate_in[srow + c0] = a.dstate_out ? a.dstate_out[srow + c0] : 0.f;
    return;
  }
  if (t == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    mbar_init(&bars[2], 1);
    mbar_init(&bars[3], 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tslot, TMEM_COLS);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tbase = *tslot;
  const uint32_t tlane = tmem_lane_addr(tbase, warp, 0);
  auto chead = [&](int j) { return ((int64_t)rec.chunk0 + j) * dm.hv + h; };
  auto gamma_of = [&](int j) { return expf(a.b.G[chead(j) * C + C - 1]); };
  const bool dexact = dm.out_bf16;  // bf16 dO: no dO^T lo image
  const uint32_t la_bytes = dexact ? 3 * IMG : 4 * IMG;
  auto load_la = [&](int j) {  // thread 0: chunk j's dO and Qt rows images
    mbar_expect_tx(&bars[3], la_bytes);
    bulk_g2s(LA, a.b.L + chead(j) * SZ, la_bytes, &bars[3]);
  };
  auto load_stage = [&](int j, int b) {  // thread 0: chunk j's K rows and W rows (hi | lo) images
    unsigned char* dst = stage0 + b * STAGE_BYTES;
    mbar_expect_tx(&bars[b], STAGE_BYTES);
    bulk_g2s(dst, a.b.img + chead(j) * IW, IMG, &bars[b]);
    bulk_g2s(dst + IMG, a.b.W + chead(j) * C * D, 2 * IMG, &bars[b]);
  };
  // prologue: dS^(nch) = dstate_out is the end adjoint of the last chunk
  {
    const int j = nch - 1;
    if (t == 0) {
      load_stage(j, 0);
      load_la(j);
    }
    const float g = gamma_of(j);
    for (int c0 = cs0; c0 < cs0 + D / 2; c0 += 16) {
      float v[16], w[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) v[e] = a.dstate_out ? a.dstate_out[srow + c0 + e] : 0.f;
#pragma unroll
      for (int e = 0; e < 16; e += 4)
        *reinterpret_cast<float4*>(a.b.dSE + chead(j) * SZ + (int64_t)row * D + c0 + e) =
            make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
      split_store16(A1h, A1l, row, c0, D, v);
#pragma unroll
      for (int e = 0; e < 16; ++e) w[e] = __fmul_rn(g, v[e]);
      tmem_st16(tlane + D2_COL + c0, w);
    }
    tmem_st_wait();
  }
  fence_proxy_async();
  fence_before_sync();
  __syncthreads();
  uint32_t uses[2] = {0u, 0u}, la_uses = 0, mma_phase = 0;
  int pending = 0;
  bool mma_pending = false, la_pending = true, ok = true;
  int q = 0;
  for (; q < nch; ++q) {
    const int j = nch - 1 - q;
    const int buf = q & 1;
    unsigned char* stg = stage0 + buf * STAGE_BYTES;
    if (j > 0 && t == 0) load_stage(j - 1, buf ^ 1);
    if (t < C) decs[t] = -expf(__fsub_rn(a.b.G[chead(j) * C + C - 1], a.b.G[chead(j) * C + t]));
    const float gpre = j > 0 ? gamma_of(j - 1) : 0.f;
    ok = __syncthreads_and(mbar_wait(&bars[buf], uses[buf] & 1u) && mbar_wait(&bars[3], la_uses & 1u)) != 0;
    if (!ok) break;
    ++uses[buf];
    ++la_uses;
    la_pending = false;
    pending = j > 0 ? (buf ^ 1) : -1;
    if (t == 0) {  // D1 = dS K^T; D2 += dO^T Qt
      fence_after_sync();
      const uint32_t kimg = smem_u32(stg), sbo = (D / 8) * 128;
#pragma unroll 1
      for (int term = 0; term < 2; ++term) {
        const uint32_t aa = smem_u32(term == 0 ? A1h : A1l);
        for (int kk = 0; kk < D / 16; ++kk)
          mma_bf16(tbase + D1_COL, make_desc(aa + kk * 256, 128, sbo), make_desc(kimg + kk * 256, 128, sbo),
                   idesc_bf16(128, C), (term > 0 || kk > 0) ? 1u : 0u);
      }
      // dO_hi Qt_hi + dO_hi Qt_lo (+ dO_lo Qt_hi), dO^T and Qt^T the MN-major readings of the
      // row images
      const uint32_t dh = smem_u32(LA);
      const Opnd dOt = opnd_mn(dh, dh + 3 * IMG, D), Qtt = opnd_mn(dh + IMG, dh + 2 * IMG, D);
      const uint32_t il = idesc_bf16(128, D) | IDESC_A_MN | IDESC_B_MN;
      mma_part(tbase + D2_COL, dOt, false, Qtt, false, C, il, true);
      mma_part(tbase + D2_COL, dOt, false, Qtt, true, C, il, true);
      if (!dexact) mma_part(tbase + D2_COL, dOt, true, Qtt, false, C, il, true);
      mma_commit(&bars[2]);
    }
    mma_pending = true;
    ok = __syncthreads_and(mbar_wait(&bars[2], mma_phase)) != 0;
    if (!ok) break;
    mma_phase ^= 1u;
    mma_pending = false;
    fence_after_sync();
#pragma unroll
    for (int s0 = us0; s0 < us0 + C / 2; s0 += 16) {  // Xd = -dec_s (dS K^T), split into A2
      float v[16];
      tmem_ld16(tlane + D1_COL + s0, v);
#pragma unroll
      for (int e = 0; e < 16; ++e) v[e] = __fmul_rn(decs[s0 + e], v[e]);
      split_store16(A2h, A2l, row, s0, C, v);
    }
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    if (t == 0) {  // D2 += Xd W (three split terms; W^T the MN-major reading of the W rows)
      fence_after_sync();
      const uint32_t wh = smem_u32(stg) + C * D * 2;
      const Opnd xd = opnd_k(smem_u32(A2h), smem_u32(A2l), C), wt = opnd_mn(wh, wh + C * D * 2, D);
      const uint32_t iw = idesc_bf16(128, D) | IDESC_B_MN;
      mma_part(tbase + D2_COL, xd, false, wt, false, C, iw, true);
      mma_part(tbase + D2_COL, xd, false, wt, true, C, iw, true);
      mma_part(tbase + D2_COL, xd, true, wt, false, C, iw, true);
      mma_commit(&bars[2]);
    }
    mma_pending = true;
    ok = __syncthreads_and(mbar_wait(&bars[2], mma_phase)) != 0;
    if (!ok) break;
    mma_phase ^= 1u;
    mma_pending = false;
    fence_after_sync();
    if (j > 0 && t == 0) {  // the next step's dO, Qt rows images over the consumed Xd
      load_la(j - 1);
      la_pending = true;
    }
    {  // dS^(j): end adjoint of chunk j-1 (or dstate_in), next A operand, next D2 preload
      const bool more = j > 0;
      const float g = gpre;
      // dS^(j) leaves through a per-warp staging tile in this step's (now consumed) operand
      // stage, so that each store instruction writes 8 rows x 64 contiguous bytes
      float* tile = reinterpret_cast<float*>(stg) + warp * (32 * 20);
      const int lane = t & 31, rq = (warp & 3) * 32;
#pragma unroll
      for (int c0 = cs0; c0 < cs0 + D / 2; c0 += 16) {
        float v[16];
        tmem_ld16(tlane + D2_COL + c0, v);
        if (more) {
#pragma unroll
          for (int x = 0; x < 4; ++x)
            *reinterpret_cast<float4*>(tile + lane * 20 + 4 * x) = make_float4(v[4 * x], v[4 * x + 1], v[4 * x + 2], v[4 * x + 3]);
          __syncwarp();
#pragma unroll
          for (int k2 = 0; k2 < 4; ++k2) {
            const int rl = 8 * k2 + (lane >> 2), f = lane & 3;
            *reinterpret_cast<float4*>(a.b.dSE + chead(j - 1) * SZ + (int64_t)(rq + rl) * D + c0 + 4 * f) =
                *reinterpret_cast<const float4*>(tile + rl * 20 + 4 * f);
          }
          __syncwarp();
          split_store16(A1h, A1l, row, c0, D, v);
          float w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) w[e] = __fmul_rn(g, v[e]);
          tmem_st16(tlane + D2_COL + c0, w);
        } else if (a.dstate_in) {
#pragma unroll
          for (int e = 0; e < 16; e += 4)
            *reinterpret_cast<float4*>(a.dstate_in + srow + c0 + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
        }
      }
      tmem_st_wait();
    }
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
  }
  if (!ok && t == 0) {
    set_error(a.hdr, GDN_DEVERR_TIMEOUT);
    if (pending >= 0) mbar_wait(&bars[pending], uses[pending] & 1u);
    if (la_pending) mbar_wait(&bars[3], la_uses & 1u);
    if (mma_pending) mbar_wait(&bars[2], mma_phase);
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, TMEM_COLS);
}

// ============================================================  KB3 (tcgen05)  ===
// The backward's products with the d x d matrices S0 = S^(j) and E = dS_end, on tensor
// cores (bf16 inputs, d = 128, C = 64), one CTA of 256 threads per chunk-head.  Every
// product is taken transposed so that a 128 x 128 state matrix is the A operand (M = 128):
//   phase 1  A = S0     : U^T   = Ut^T - S0 W^T
//   phase 2  A = E      : (E K^T) and, with A = dO^T, dO^T P  ->  dU^T = dO^T P + (E K^T) diag(dec)
//   phase 3  A = E^T    : (U E)^T  = E^T U^T
//   phase 4  A = S0^T   : (dO S0)^T = S0^T dO^T,   dW^T = -S0^T dU^T
// fp32 operands are split into bf16 hi + lo (three MMAs per product, lo x lo dropped);
// bf16 inputs are exact.  A transposed operand is the MN-major reading of an image already
// in shared memory (E^T and S0^T of the E and S0 images, dO^T of the dO rows image, U and dU
// rows of the U^T and dU^T images built from the TMEM readouts), so nothing is transposed.
// The S0 image built in phase 1 leaves by bulk copy for two workspace slots that are free
// here (the SIMT path's dU rows and the second half of the adjoint L slot) and comes back the
// same way for phase 4.  Sized for two CTAs per SM (the A image pair, a 64 x 128 B image
// pair and one more 64 x 128 image, 256 TMEM columns, 128 registers), so that one CTA's
// loads and waits overlap the other's work.
namespace tcg {
constexpr int D = 128, C = 64;
constexpr uint32_t RA = 2 * 128 * D * 2;       // A operand hi | lo (64 KB)
constexpr uint32_t RB = 2 * C * D * 2;         // B operand hi | lo (32 KB)
constexpr uint32_t RX = C * D * 2;             // one more 64 x 128 image (16 KB)
constexpr size_t SMEM = (size_t)RA + RB + RX + C * 4 + 128 * 4 + 64;
static_assert(SMEM <= 115712, "two CTAs per SM");
constexpr uint32_t TMEM_COLS = 256;
constexpr uint32_t COL_0 = 0, COL_1 = 64, COL_2 = 128;  // 128 x 64 results
}  // namespace tcg

// 8 fp32 values -> hi / lo bf16 16-byte pieces at byte offset `off` of the two images
__device__ __forceinline__ void split8(unsigned char* hi, unsigned char* lo, uint32_t off, const float* v) {
  uint32_t hw[4], lw[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    __nv_bfloat16 h0, l0, h1, l1;
    tc::split_bf16(v[2 * e], h0, l0);
    tc::split_bf16(v[2 * e + 1], h1, l1);
    hw[e] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
    lw[e] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
  }
  *reinterpret_cast<uint4*>(hi + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
  *reinterpret_cast<uint4*>(lo + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
}

// R x K image pair (hi at `hi`, lo at `lo`) of a row-major fp32 matrix src[r * ld + k]
// (rows >= nvalid are zero); TRANS takes src[k * ld + r] instead (columns >= nvalid zero).
// SplitTile::load fetches the pieces of thread `tid` (of NTH) into registers and store
// writes them, so that the loads of several builds can be in flight before the first store.
template <bool TRANS, int R, int K, int NTH = 256>
struct SplitTile {
  static constexpr int ITER = R * (K / 8) / NTH;
  static_assert(ITER * NTH == R * (K / 8), "tile must split evenly over the threads");
  float v[ITER][8];
  __device__ __forceinline__ static void piece(int q, int& r, int& k0) {
    if (TRANS) {
      r = q % R;
      k0 = (q / R) * 8;
    } else {
      tc::kmajor_piece(q, K, r, k0);
    }
  }
  // A row-major source whose row stride is a multiple of 4 floats (16-byte aligned rows) is
  // read as two float4 per piece; otherwise (and for TRANS, whose warps read consecutive
  // rows of one column) element by element.
  __device__ __forceinline__ void load(const float* __restrict__ src, int ld, int nvalid, int tid) {
    const bool vec = !TRANS && (ld & 3) == 0;
#pragma unroll
    for (int it = 0; it < ITER; ++it) {
      int r, k0;
      piece(tid + it * NTH, r, k0);
      if (vec) {
        float4 x0 = make_float4(0.f, 0.f, 0.f, 0.f), x1 = x0;
        if (r < nvalid) {
          x0 = *reinterpret_cast<const float4*>(src + (int64_t)r * ld + k0);
          x1 = *reinterpret_cast<const float4*>(src + (int64_t)r * ld + k0 + 4);
        }
        v[it][0] = x0.x; v[it][1] = x0.y; v[it][2] = x0.z; v[it][3] = x0.w;
        v[it][4] = x1.x; v[it][5] = x1.y; v[it][6] = x1.z; v[it][7] = x1.w;
        continue;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (TRANS)
          v[it][e] = (k0 + e < nvalid) ? src[(int64_t)(k0 + e) * ld + r] : 0.f;
        else
          v[it][e] = (r < nvalid) ? src[(int64_t)r * ld + k0 + e] : 0.f;
      }
    }
  }
  __device__ __forceinline__ void store(unsigned char* hi, unsigned char* lo, int tid) const {
#pragma unroll
    for (int it = 0; it < ITER; ++it) {
      int r, k0;
      piece(tid + it * NTH, r, k0);
      split8(hi, lo, tc::kmajor_off(r, k0, K), v[it]);
    }
  }
  __device__ __forceinline__ void load(const float* __restrict__ src, int ld, int nvalid) {
    load(src, ld, nvalid, (int)threadIdx.x);
  }
  __device__ __forceinline__ void store(unsigned char* hi, unsigned char* lo) const {
    store(hi, lo, (int)threadIdx.x);
  }
};

template <bool TRANS, int R, int K>
__device__ __forceinline__ void build_split(unsigned char* hi, unsigned char* lo, const float* __restrict__ src,
                                            int ld, int nvalid) {
  SplitTile<TRANS, R, K> tile;
  tile.load(src, ld, nvalid);
  tile.store(hi, lo);
}

__device__ __forceinline__ void unpack8(const uint4 u, float* o) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    o[2 * i] = __uint_as_float(w[i] << 16);
    o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}


// dO pieces of 256 threads for d = 128, C = 64 (4 per thread), tokens >= n zero.  The
// dtype branch is outside the loops, so that all of a thread's loads are in flight together.
// load_dO_rows: piece q = t + 256 it is 8 consecutive dims of one token, in kmajor_piece order
// (a K-major image of dO), read as one 16-byte (bf16) or two (fp32) loads.
template <typename T>
__device__ __forceinline__ void load_dO_rows_t(float (&v)[4][8], const T* p, int64_t tstride, int n) {
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    int r, k0;
    tc::kmajor_piece(threadIdx.x + it * 256, 128, r, k0);
    if (r < n) {
      load8(p + (int64_t)r * tstride + k0, v[it]);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) v[it][e] = 0.f;
    }
  }
}
__device__ __forceinline__ void load_dO_rows(float (&v)[4][8], const void* dO, bool bf16, int64_t base,
                                             int64_t tstride, int n) {
  if (bf16)
    load_dO_rows_t(v, static_cast<const __nv_bfloat16*>(dO) + base, tstride, n);
  else
    load_dO_rows_t(v, static_cast<const float*>(dO) + base, tstride, n);
}

// 128 x 128 image pair of a row-major fp32 d x d matrix, built in four 32-row quarters with
// two in flight (a thread holds 32 values at a time: one quarter's loads overlap the previous
// quarter's wait)
__device__ __forceinline__ void build_dd4(unsigned char* hi, unsigned char* lo, const float* src) {
  SplitTile<false, 32, 128> a, b;
  a.load(src, 128, 32);
  b.load(src + 32 * 128, 128, 32);
  a.store(hi, lo);
  a.load(src + 64 * 128, 128, 32);
  b.store(hi + 8192, lo + 8192);
  b.load(src + 96 * 128, 128, 32);
  a.store(hi + 16384, lo + 16384);
  b.store(hi + 24576, lo + 24576);
}

// D = A B^T over K with split operands: terms = 3 gives A_hi B_hi + A_hi B_lo + A_lo B_hi;
// terms = 2 (B exact, blo ignored) gives A_hi B + A_lo B; `accumulate` adds onto D.
__device__ __forceinline__ void mma_terms(uint32_t d, uint32_t ahi, uint32_t alo, uint32_t bhi, uint32_t blo,
                                          int K, uint32_t idesc, int terms, bool accumulate = false) {
  const uint32_t sbo = (uint32_t)(K / 8) * 128;
  for (int term = 0; term < terms; ++term) {
    const uint32_t aa = (terms == 3 ? term == 2 : term == 1) ? alo : ahi;
    const uint32_t bb = (terms == 3 && term == 1) ? blo : bhi;
    for (int kk = 0; kk < K / 16; ++kk)
      tc::mma_bf16(d, tc::make_desc(aa + kk * 256, 128, sbo), tc::make_desc(bb + kk * 256, 128, sbo), idesc,
                   (accumulate || term > 0 || kk > 0) ? 1u : 0u);
  }
}

// 8 values exact in bf16 (widened bf16 inputs) as one 16-byte piece of a bf16 image
__device__ __forceinline__ void store_bf16x8(unsigned char* img, uint32_t off, const float* v) {
  uint32_t w[4];
#pragma unroll
  for (int e = 0; e < 4; ++e)
    w[e] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[2 * e])) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[2 * e + 1])) << 16);
  *reinterpret_cast<uint4*>(img + off) = make_uint4(w[0], w[1], w[2], w[3]);
}

__global__ void __launch_bounds__(256, 2) k_bwd_big_tc(BwdArgs a) {
  using namespace tcg;
  using namespace tc;
  extern __shared__ __align__(128) unsigned char smg[];
  unsigned char* Ah = smg;            // A: the S0 or E image pair (128 x 128)
  unsigned char* Al = Ah + RA / 2;
  unsigned char* Bh = smg + RA;       // B: 64 x 128 or 128 x 64 image pairs, P rows
  unsigned char* Bl = Bh + RB / 2;
  unsigned char* Xh = Bh + RB;        // a third 64 x 128 image
  float* dec = reinterpret_cast<float*>(Xh + RX);
  float* red = dec + C;                                    // 128 partial sums
  uint64_t* bar = reinterpret_cast<uint64_t*>(red + 128);  // [0] MMA, [1] bulk copies, [2] S0 image back
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 3);
  if (!a.hdr->valid) return;
  const Dims dm = a.dm;
  const int t = threadIdx.x, warp = t >> 5;
  const int64_t c = blockIdx.x;
  const int h = blockIdx.y;
  const ChunkRec rec = a.chunks[c];
  if (!in_bounds(a.hdr, rec.tok0 >= 0 && rec.len >= 0 && rec.len <= a.dm.C && (int64_t)rec.tok0 + rec.len <= a.T))
    return;
  const int n = rec.len;
  const int64_t tok0 = rec.tok0;
  const int64_t ch = c * dm.hv + h;
  const int64_t SZ = (int64_t)D * D, CD = (int64_t)C * D;
  const float* S0 = a.saved_bnd + ch * SZ;
  const float* E = a.b.dSE + ch * SZ;
  float* s0_hi = a.b.dU + ch * CD;           // where the S0 image waits for phase 4 (32 KB each)
  float* s0_lo = a.b.L + ch * SZ + SZ / 2;
  const int lane_row = (warp & 3) * 32 + (t & 31);  // TMEM lane = row of the transposed result
  const int cbase = (warp >> 2) * 32;               // this warp's 32 result columns
  constexpr uint32_t IMGB = C * D * 2;  // one 64 x 128 (or 128 x 64) bf16 image
  const bool exact = dm.out_bf16;       // bf16 dO: no lo image, no dO_lo term
  if (t < C) dec[t] = expf(__fsub_rn(a.b.G[ch * C + C - 1], a.b.G[ch * C + t]));
  if (t == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    mbar_init(&bar[2], 1);
    fence_mbar_init();
    mbar_expect_tx(&bar[1], RB);  // the prep kernel's W rows image (hi | lo) for phase 1
    bulk_g2s(Bh, a.b.W + ch * CD, RB, &bar[1]);
  }
  if (warp == 0) tmem_alloc(tslot, TMEM_COLS);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tb = *tslot;
  const uint32_t tl = tmem_lane_addr(tb, warp, 0);
  uint32_t phase = 0, cphase = 0;
  bool ok = true, pending = false, cpending = true, spending = false;
  auto run = [&]() {  // all threads: wait for the committed MMAs
    const bool done = mbar_wait(&bar[0], phase);
    if (done) {
      phase ^= 1u;
      pending = false;
    }
    ok = __syncthreads_and(done) != 0;
    fence_after_sync();
  };
  auto issue = [&](auto&& mmas) {  // operands written -> one thread issues and commits
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    if (t == 0) {
      fence_after_sync();
      mmas();
      mma_commit(&bar[0]);
    }
    pending = true;
  };
  // the same after thread 0 has waited for the bulk copies in flight on barrier `cb` (phase
  // `cp`); every thread learns whether they arrived
  auto issue_after = [&](uint64_t* cb, uint32_t& cp, bool& cpend, auto&& mmas) {
    fence_proxy_async();
    fence_before_sync();
    bool got = true;
    if (t == 0) {
      got = mbar_wait(cb, cp);
      if (got) {
        cp ^= 1u;
        cpend = false;
      }
    }
    ok = __syncthreads_and(got) != 0;
    if (ok && t == 0) {
      fence_after_sync();
      mmas();
      mma_commit(&bar[0]);
    }
    pending = ok;
  };
  const uint32_t sa_h = smem_u32(Ah), sa_l = smem_u32(Al), sb_h = smem_u32(Bh), sb_l = smem_u32(Bl),
                 sx = smem_u32(Xh);
  const uint32_t I_KK = idesc_bf16(128, C);

  // ---- phase 1: U^T = Ut^T - S0 W^T; the S0 image also leaves for phase 4
  build_dd4(Ah, Al, S0);
  SplitTile<false, 64, D> e_first;  // E rows 0..63 for phase 2a
  issue_after(&bar[1], cphase, cpending, [&] {
    mma_split(tb + COL_0, opnd_k(sa_h, sa_l, D), opnd_k(sb_h, sb_l, D), D, I_KK, 3);
    bulk_s2g(s0_hi, Ah, RA / 2);
    bulk_s2g(s0_lo, Al, RA / 2);
    bulk_store_commit();
  });
  {
    float ut[32];  // Ut for the readout, loaded while the product runs
#pragma unroll
    for (int x = 0; x < 32; ++x) ut[x] = a.b.Ut[ch * CD + (int64_t)(cbase + x) * D + lane_row];
    e_first.load(E, D, 64);  // phase 2a's first E half, also in flight meanwhile
    run();
    if (ok) {  // U = Ut - (U^T)^T as the U^T image (rows d, K = s): hi in X, lo in B's second
      // half (phase 2a's K image takes the first)
#pragma unroll
      for (int s1 = 0; s1 < 2; ++s1) {
        float v[16];
        tmem_ld16(tl + COL_0 + cbase + 16 * s1, v);
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = __fsub_rn(ut[16 * s1 + e], v[e]);
        split8(Xh, Bl, kmajor_off(lane_row, cbase + 16 * s1, C), v);
        split8(Xh, Bl, kmajor_off(lane_row, cbase + 16 * s1 + 8, C), v + 8);
      }
    }
  }
  fence_before_sync();
  __syncthreads();

  // ---- phase 2a: E K^T (K rows: the prep kernel's image, one bulk copy); <E, S0> from the
  // E build; the U^T image leaves for the first gradients kernel
  float part = 0.f;
  if (ok) {
    if (t == 0) {
      mbar_expect_tx(&bar[1], IMGB);
      bulk_g2s(Bh, a.b.img + ch * (int64_t)prep_w_floats(C, D), IMGB, &bar[1]);
      cpending = true;
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {  // E image by halves, with S0 at the same positions (the
      // first E half loaded during phase 1)
      SplitTile<false, 64, D> et, st;
      if (hh == 1) et.load(E + 64 * D, D, 64);
      st.load(S0 + hh * 64 * D, D, 64);
      const SplitTile<false, 64, D>& eh = hh == 0 ? e_first : et;
#pragma unroll
      for (int it = 0; it < SplitTile<false, 64, D>::ITER; ++it)
#pragma unroll
        for (int e = 0; e < 8; ++e) part = __fmaf_rn(eh.v[it][e], st.v[it][e], part);
      if (hh == 0) {
        if (t == 0) bulk_wait_read();  // the S0 image store has read A
        __syncthreads();
      }
      eh.store(Ah + hh * 16384, Al + hh * 16384);
    }
    issue_after(&bar[1], cphase, cpending, [&] {
      mma_split(tb + COL_0, opnd_k(sa_h, sa_l, D), opnd_k(sb_h, sb_h, D), D, I_KK, 2);
      bulk_s2g(a.b.U + ch * CD, Xh, IMGB);  // U^T image: hi, then lo
      bulk_s2g(a.b.U + ch * CD + IMGB / 4, Bl, IMGB);
      bulk_store_commit();
    });
  }
  // ---- phase 3: (U E)^T = E^T U^T, both operands MN-major readings of the E and U^T images;
  // P rows (the prep kernel's image) come into B's first half meanwhile
  if (ok) {
    run();
    if (ok) {
      if (t == 0) {
        mbar_expect_tx(&bar[1], C * C * 4);
        bulk_g2s(Bh, a.b.P + ch * C * C, C * C * 4, &bar[1]);
        cpending = true;
      }
      issue([&] {
        mma_split(tb + COL_2, opnd_mn(sa_h, sa_l, D), opnd_mn(sx, sb_l, C), D, I_KK | IDESC_A_MN | IDESC_B_MN, 3);
      });
    }
  }
  // <E, S0>: the 256 partial sums added pairwise at strides 128, 64, ..., 1
  if (t >= 128) red[t - 128] = part;
  __syncthreads();
  if (t < 128) part = __fadd_rn(part, red[t]);
  __syncthreads();
  if (t >= 64 && t < 128) red[t - 64] = part;
  __syncthreads();
  if (t < 64) part = __fadd_rn(part, red[t]);
  __syncthreads();
  if (t >= 32 && t < 64) red[t - 32] = part;
  __syncthreads();
  if (t < 32) {
    part = __fadd_rn(part, red[t]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part = __fadd_rn(part, __shfl_down_sync(0xffffffffu, part, o));
    if (t == 0) a.b.sdot[ch] = part;
  }
  // ---- phase 2b: dO^T P: dO^T the MN-major reading of the dO rows image (in X; fp32 dO: lo in
  // B's second half), P^T that of the P rows (B's first half); the S0 image comes back into A
  // meanwhile
  if (ok) {
    float v[4][8];  // dO rows, loaded while E^T U^T runs
    load_dO_rows(v, a.dO, dm.out_bf16, (tok0 * dm.hv + h) * D, (int64_t)dm.hv * D, n);
    run();
    if (ok) {
      if (t == 0) {
        bulk_wait_all();  // the S0 image is in the workspace; the U^T image store has read X, B
        mbar_expect_tx(&bar[2], RA);
        bulk_g2s(Ah, s0_hi, RA / 2, &bar[2]);
        bulk_g2s(Al, s0_lo, RA / 2, &bar[2]);
        spending = true;
      }
      __syncthreads();
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        int r, k0;
        kmajor_piece(t + it * 256, D, r, k0);
        if (exact)
          store_bf16x8(Xh, kmajor_off(r, k0, D), v[it]);
        else
          split8(Xh, Bl, kmajor_off(r, k0, D), v[it]);
      }
      issue_after(&bar[1], cphase, cpending, [&] {
        mma_split(tb + COL_1, opnd_mn(sx, sb_l, D), opnd_mn(sb_h, sb_h + C * C * 2, C), C,
                  I_KK | IDESC_A_MN | IDESC_B_MN, exact ? -2 : 3);
      });
    }
  }
  if (ok) {  // U dS_end while dO^T P runs
#pragma unroll
    for (int s1 = 0; s1 < 2; ++s1) {
      float w[16];
      tmem_ld16(tl + COL_2 + cbase + 16 * s1, w);
#pragma unroll
      for (int e = 0; e < 16; ++e) a.b.UdSe[ch * CD + (int64_t)(cbase + 16 * s1 + e) * D + lane_row] = w[e];
    }
    run();
  }
  if (ok) {  // dU^T = dO^T P + (E K^T) diag(dec) as the dU^T image (rows d, K = s; hi | lo) in
    // B: one bulk copy into the second half of this chunk-head's adjoint L slot for the
    // gradients kernel (the first half still holds the prep's dO rows image, which the
    // gradients kernel reads too), and read MN-major as the dU rows operand of dW^T
#pragma unroll
    for (int s1 = 0; s1 < 2; ++s1) {
      float e1[16], p1[16];
      tmem_ld16(tl + COL_0 + cbase + 16 * s1, e1);
      tmem_ld16(tl + COL_1 + cbase + 16 * s1, p1);
#pragma unroll
      for (int e = 0; e < 16; ++e) p1[e] = __fmaf_rn(dec[cbase + 16 * s1 + e], e1[e], p1[e]);
      split8(Bh, Bl, kmajor_off(lane_row, cbase + 16 * s1, C), p1);
      split8(Bh, Bl, kmajor_off(lane_row, cbase + 16 * s1 + 8, C), p1 + 8);
    }
  }
  // ---- phase 4: dW^T = -S0^T dU^T and (dO S0)^T = S0^T dO^T, S0^T the MN-major reading of the
  // S0 image; bf16 dO rows (exact) are still in X and both products go together, fp32 dO
  // (hi | lo) is split again into B once dW^T is done
  if (ok) {
    float v[4][8];
    if (!exact) load_dO_rows(v, a.dO, false, (tok0 * dm.hv + h) * D, (int64_t)dm.hv * D, n);
    uint32_t sph = 0;
    issue_after(&bar[2], sph, spending, [&] {
      const Opnd s0t = opnd_mn(sa_h, sa_l, D);
      mma_split(tb + COL_1, s0t, opnd_mn(sb_h, sb_l, C), D, I_KK | IDESC_A_MN | IDESC_B_MN, 3);
      if (exact) mma_split(tb + COL_0, s0t, opnd_k(sx, sx, D), D, I_KK | IDESC_A_MN, 2);
      bulk_s2g(a.b.L + ch * SZ + SZ / 2, Bh, RB);  // over the S0 lo image, back in A by now
      bulk_store_commit();
    });
    run();
    if (ok && !exact) {
      if (t == 0) bulk_wait_read();  // the dU^T image store has read B
      __syncthreads();
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        int r, k0;
        kmajor_piece(t + it * 256, D, r, k0);
        split8(Bh, Bl, kmajor_off(r, k0, D), v[it]);
      }
      issue([&] {
        mma_split(tb + COL_0, opnd_mn(sa_h, sa_l, D), opnd_k(sb_h, sb_l, D), D, I_KK | IDESC_A_MN, 3);
      });
      run();
    }
  }
  if (ok) {  // dO S0 rows (fp32) and the dW^T operand image (rows d, K = s; hi | lo)
    unsigned char* wimg = reinterpret_cast<unsigned char*>(a.b.dW + ch * CD);
#pragma unroll
    for (int s1 = 0; s1 < 2; ++s1) {
      float v[16], w[16];
      tmem_ld16(tl + COL_0 + cbase + 16 * s1, v);
      tmem_ld16(tl + COL_1 + cbase + 16 * s1, w);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        a.b.dOS0[ch * CD + (int64_t)(cbase + 16 * s1 + e) * D + lane_row] = v[e];
        w[e] = -w[e];
      }
      split8(wimg, wimg + C * D * 2, kmajor_off(lane_row, cbase + 16 * s1, C), w);
      split8(wimg, wimg + C * D * 2, kmajor_off(lane_row, cbase + 16 * s1 + 8, C), w + 8);
    }
  } else if (t == 0) {
    set_error(a.hdr, GDN_DEVERR_TIMEOUT);
    if (pending) mbar_wait(&bar[0], phase);  // let this CTA's products and copies finish
    if (cpending) mbar_wait(&bar[1], cphase);
    if (spending) mbar_wait(&bar[2], 0);
  }
  if (t == 0) bulk_wait_all();  // the image stores are complete
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, TMEM_COLS);
}

// e^{G_i - G_s} for s <= i, packed by rows at i (i + 1) / 2 + s; all 256 threads, C = 64
__device__ __forceinline__ void decay_table_lower(float* tab, const float* Gs) {
  const int i = threadIdx.x & 63;
  for (int s = threadIdx.x >> 6; s <= i; s += 4) tab[i * (i + 1) / 2 + s] = expf(__fsub_rn(Gs[i], Gs[s]));
}

// ============================================================  KB1 (tcgen05)  ===
// Backward prep on tensor cores (bf16 inputs, d = 128, C = 64), one CTA of 256 threads per
// chunk-head, every chunk zero-padded to C:
//   Gram = K K^T, T = (I + A)^{-1} (SIMT), W = TK K, U^T = V^T TV^T    (as the forward pre-pass)
//   P    = Gam (.) (Q K^T), lower with diagonal                       (exact bf16 inputs)
//   Qt   = diag(e^G) Q - P W                                          (P, W split hi/lo)
//   dO, Qt rows                                                       (the operands of L = dO^T Qt)
// Outputs: the W rows image (W's slot), Ut, G, the K rows image (the reverse chain's, with
// the W rows), the operands of L (L's slot; the reverse chain forms L = dO^T Qt on its tensor
// cores, reading the row images MN-major), and two more operand images: P rows for the
// big-products kernel (in P's slot) and T^T for the gradients kernel (in T's slot).  W, P
// and Qt also leave their readouts as split images in shared memory, where the later
// products read them (W^T as the MN-major reading of the W rows).
namespace tcq {
constexpr int D = 128, C = 64, QCP = C + 1, TCP = C;  // row strides of A (padded) and T
constexpr uint32_t TILE = C * D * 2;  // 16 KB
constexpr uint32_t OFF_K = 0, OFF_KT = TILE, OFF_VT = 2 * TILE, OFF_TK = 3 * TILE, OFF_TV = 4 * TILE,
                   OFF_A = 5 * TILE, OFF_T = OFF_A + C * QCP * 4, OFF_VEC = OFF_T + C * TCP * 4;
constexpr size_t SMEM = OFF_VEC + 2 * C * 4 + 64;  // fits two CTAs per SM
constexpr uint32_t TMEM_COLS = 256;  // the products run one after another: W and U^T (192) at most
constexpr uint32_t COL_G = 0, COL_W = 0, COL_UT = 128, COL_P = 0, COL_QT = 0;
}  // namespace tcq

__global__ void __launch_bounds__(256, 2) k_bwd_prep_tc(BwdArgs a) {
  using namespace tcq;
  using namespace tc;
  extern __shared__ __align__(128) unsigned char smq[];
  unsigned char* Ki = smq + OFF_K;
  unsigned char* KT = smq + OFF_KT;
  unsigned char* VT = smq + OFF_VT;
  unsigned char* TKh = smq + OFF_TK;
  unsigned char* TKl = TKh + C * C * 2;
  unsigned char* TVh = smq + OFF_TV;
  unsigned char* TVl = TVh + C * C * 2;
  float* A = reinterpret_cast<float*>(smq + OFF_A);
  float* Tm = reinterpret_cast<float*>(smq + OFF_T);
  float* Gs = reinterpret_cast<float*>(smq + OFF_VEC);  // g, then its cumulative sum G
  float* bs = Gs + C;
  uint64_t* bar = reinterpret_cast<uint64_t*>(bs + C);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 1);
  float* Xs = reinterpret_cast<float*>(TKh);
  if (!a.hdr->valid) return;
  const Dims dm = a.dm;
  const int t = threadIdx.x, warp = t >> 5;
  const int64_t c = blockIdx.x;
  const int h = blockIdx.y, hq = h / (dm.hv / dm.hqk);
  const ChunkRec rec = a.chunks[c];
  if (!in_bounds(a.hdr, rec.tok0 >= 0 && rec.len >= 0 && rec.len <= a.dm.C && (int64_t)rec.tok0 + rec.len <= a.T))
    return;
  const int n = rec.len;
  const int64_t tok0 = rec.tok0;
  const int64_t ch = c * dm.hv + h;
  const int64_t CD = (int64_t)C * D;
  const int64_t kstride = (int64_t)dm.hqk * D, vstride = (int64_t)dm.hv * D;
  const __nv_bfloat16* kb = static_cast<const __nv_bfloat16*>(a.in.k) + tok0 * kstride + (int64_t)hq * D;
  const __nv_bfloat16* vb = static_cast<const __nv_bfloat16*>(a.in.v) + tok0 * vstride + (int64_t)h * D;
  const __nv_bfloat16* qb = static_cast<const __nv_bfloat16*>(a.in.q) + tok0 * kstride + (int64_t)hq * D;
  unsigned char* img = reinterpret_cast<unsigned char*>(a.b.img + ch * (int64_t)prep_w_floats(C, D));
  const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);

  // ---- 1. images of K rows and V rows (V in the V^T region: step 3 reads K^T and V^T as the
  // MN-major readings of the row images), g, beta (zero beyond the chunk's tokens); every
  // load issued before the first store
  unsigned char* Vi = VT;
  {
    float g0 = 0.f, b0 = 0.f;
    if (t < n) {
      g0 = a.in.g[(tok0 + t) * dm.hv + h];
      b0 = a.in.beta[(tok0 + t) * dm.hv + h];
    }
    uint4 kr[4], vr[4];
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      int r, c0;
      kmajor_piece(t + it * 256, D, r, c0);
      kr[it] = r < n ? *reinterpret_cast<const uint4*>(kb + r * kstride + c0) : z4;
      vr[it] = r < n ? *reinterpret_cast<const uint4*>(vb + r * vstride + c0) : z4;
    }
    if (t < C) {
      Gs[t] = g0;
      bs[t] = b0;
    }
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      int r, c0;
      kmajor_piece(t + it * 256, D, r, c0);
      *reinterpret_cast<uint4*>(Ki + kmajor_off(r, c0, D)) = kr[it];
      *reinterpret_cast<uint4*>(Vi + kmajor_off(r, c0, D)) = vr[it];
    }
  }
  if (t == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tslot, TMEM_COLS);
  fence_proxy_async();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tb = *tslot;
  uint32_t phase = 0;
  bool ok = true;
  auto wait_mma = [&]() {
    const bool done = mbar_wait(bar, phase);
    if (done) phase ^= 1u;
    ok = __syncthreads_and(done) != 0;
    fence_after_sync();
  };
  auto sync_for_mma = [&]() {
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
  };
  const int lrow = (warp & 3) * 32 + (t & 31);  // TMEM lane of this thread
  const int chalf = warp >> 2;                  // which half of the columns this warp reads

  // ---- 2. Gram, G
  if (t == 0) {
    const uint32_t ka = smem_u32(Ki);
    for (int kk = 0; kk < D / 16; ++kk)
      mma_bf16(tb + COL_G, make_desc(ka + kk * 256, 128, (D / 8) * 128), make_desc(ka + kk * 256, 128, (D / 8) * 128),
               idesc_bf16(128, C), kk > 0 ? 1u : 0u);
    mma_commit(bar);
    float run = Gs[0];  // in place: G_i = G_{i-1} + g_i
#pragma unroll
    for (int i = 1; i < C; ++i) {
      run = __fadd_rn(run, Gs[i]);
      Gs[i] = run;
    }
  }
  __syncthreads();
  if (t < C) a.b.G[ch * C + t] = Gs[t];
  // beta_i e^{G_i - G_s} (i > s) into A while the Gram product runs (V^T is built), by all
  // threads; the readout multiplies in place
  tc::decay_matrix64(A, QCP, bs, Gs);
  wait_mma();
  if (ok && (warp & 3) < 2) {
    const int i = lrow;
    for (int s0 = chalf * 32; s0 < chalf * 32 + 32; s0 += 16) {
      float v[16];
      tmem_ld16(tmem_lane_addr(tb, warp, COL_G + s0), v);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int s = s0 + e;
        A[i * QCP + s] = (i > s) ? __fmul_rn(A[i * QCP + s], v[e]) : 0.f;
      }
    }
  }
  fence_before_sync();
  __syncthreads();
  // ---- 3. T, TK, TV; W = TK K and U^T = V^T TV^T
  unit_lower_inverse64(A, QCP, Tm, TCP, Xs);
  {  // T^T as the gradients kernel's operand image (rows r, K = i; hi | lo), T lower
    unsigned char* timg = reinterpret_cast<unsigned char*>(a.b.T + ch * C * C);
#pragma unroll
    for (int it = 0; it < 2; ++it) {
      const int q = t + it * 256, r = q % C, i0 = (q / C) * 8;
      float v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = (r <= i0 + e) ? Tm[(i0 + e) * TCP + r] : 0.f;
      split8(timg, timg + C * C * 2, kmajor_off(r, i0, C), v);
    }
  }
  for (int q = t; q < C * (C / 8); q += 256) {
    int i, r0;
    kmajor_piece(q, C, i, r0);
    float tk[8], tv[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int r = r0 + e;
      const float x = (r <= i) ? Tm[i * TCP + r] : 0.f;
      tk[e] = __fmul_rn(x, __fmul_rn(bs[r], expf(Gs[r])));  // beta e^G
      tv[e] = __fmul_rn(x, bs[r]);
    }
    const uint32_t off = kmajor_off(i, r0, C);
    split8(TKh, TKl, off, tk);
    split8(TVh, TVl, off, tv);
  }
  sync_for_mma();
  if (ok && t == 0) {
    fence_after_sync();
    const Opnd tk = opnd_k(smem_u32(TKh), smem_u32(TKl), C), tv = opnd_k(smem_u32(TVh), smem_u32(TVl), C);
    const Opnd kt = opnd_mn(smem_u32(Ki), 0u, D), vt = opnd_mn(smem_u32(Vi), 0u, D);
    const uint32_t iw = idesc_bf16(128, D) | IDESC_B_MN, iu = idesc_bf16(128, C) | IDESC_A_MN;
    mma_part(tb + COL_W, tk, false, kt, false, C, iw, false);  // W = TK_hi K + TK_lo K
    mma_part(tb + COL_UT, vt, false, tv, false, C, iu, false);  // U^T = V^T TV_hi^T + V^T TV_lo^T
    mma_part(tb + COL_W, tk, true, kt, false, C, iw, true);
    mma_part(tb + COL_UT, vt, false, tv, true, C, iu, true);
    mma_commit(bar);
  }
  unsigned char* Qi = smq + OFF_A;  // Q rows image over the dead A region, while the products run
  {
    uint4 qr[4];
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      int r, c0;
      kmajor_piece(t + it * 256, D, r, c0);
      qr[it] = r < n ? *reinterpret_cast<const uint4*>(qb + r * kstride + c0) : z4;
    }
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      int r, c0;
      kmajor_piece(t + it * 256, D, r, c0);
      *reinterpret_cast<uint4*>(Qi + kmajor_off(r, c0, D)) = qr[it];
    }
  }
  if (ok) wait_mma();
  // W, P and Qt also leave their readouts as split images in shared memory (the transposed
  // operands are built there), so that nothing this CTA wrote is read back from global memory
  unsigned char* Wr = smq + OFF_TK;  // W rows hi | lo (32 KB over the dead TK and TV)
  if (ok) {
    if ((warp & 3) < 2) {  // W rows (not decayed)
      const int i = lrow;
      for (int c0 = chalf * 64; c0 < chalf * 64 + 64; c0 += 16) {
        float v[16];
        tmem_ld16(tmem_lane_addr(tb, warp, COL_W + c0), v);
        split8(Wr, Wr + TILE, kmajor_off(i, c0, D), v);
        split8(Wr, Wr + TILE, kmajor_off(i, c0 + 8, D), v + 8);
      }
    }
    {  // Ut[i][e] = U^T[e][i]
      const int e = lrow;
      for (int i0 = chalf * 32; i0 < chalf * 32 + 32; i0 += 16) {
        float v[16];
        tmem_ld16(tmem_lane_addr(tb, warp, COL_UT + i0), v);
#pragma unroll
        for (int x = 0; x < 16; ++x) a.b.Ut[ch * CD + (int64_t)(i0 + x) * D + e] = v[x];
      }
    }
  }
  // ---- 4. P = Gam (.) (Q K^T); the W rows image stays for step 5 (its B operand is W^T, the
  // MN-major reading of the W rows)
  sync_for_mma();
  if (ok && t == 0) {
    fence_after_sync();
    const uint32_t qa = smem_u32(Qi), ka = smem_u32(Ki), sbo = (D / 8) * 128;
    for (int kk = 0; kk < D / 16; ++kk)
      mma_bf16(tb + COL_P, make_desc(qa + kk * 256, 128, sbo), make_desc(ka + kk * 256, 128, sbo),
               idesc_bf16(128, C), kk > 0 ? 1u : 0u);
    mma_commit(bar);
  }
  if (t == 0) {  // asynchronous bulk stores: the K and Q rows images into the image slot (the
                 // reverse chain's and the later kernels' operands), and the W rows image
                 // (hi | lo) into W's slot for the reverse chain, the d x d products and
                 // gradients kernels
    bulk_s2g(img, Ki, TILE);
    bulk_s2g(img + TILE, Qi, TILE);
    bulk_s2g(a.b.W + ch * CD, Wr, 2 * TILE);
    bulk_store_commit();
  }
  float* gam = Tm;  // e^{G_i - G_s} (s <= i) over the dead T, by all threads
  decay_table_lower(gam, Gs);
  unsigned char* Ph = KT;  // P rows image, hi | lo (8 KB each), in the K^T region
  if (ok) wait_mma();
  if (ok && (warp & 3) < 2) {
    const int i = lrow;
    for (int s0 = chalf * 32; s0 < chalf * 32 + 32; s0 += 16) {
      float v[16];
      tmem_ld16(tmem_lane_addr(tb, warp, COL_P + s0), v);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int s = s0 + e;
        v[e] = (i >= s) ? __fmul_rn(gam[i * (i + 1) / 2 + s], v[e]) : 0.f;
      }
      split8(Ph, Ph + C * C * 2, kmajor_off(i, s0, C), v);
      split8(Ph, Ph + C * C * 2, kmajor_off(i, s0 + 8, C), v + 8);
    }
  }
  // ---- 5. Qt = diag(e^G) Q - P W: A = P (rows i), B = W^T; dO rows for step 6, loaded while
  // the product runs (bf16 dO held bit for bit in dov[it][0..3], fp32 dO as values)
  float dov[4][8];
  if (ok) {
    sync_for_mma();
    if (t == 0) {
      fence_after_sync();
      mma_split(tb + COL_QT, opnd_k(smem_u32(Ph), smem_u32(Ph) + C * C * 2, C),
                opnd_mn(smem_u32(Wr), smem_u32(Wr) + TILE, D), C, idesc_bf16(128, D) | IDESC_B_MN, 3);
      mma_commit(bar);
      bulk_s2g(a.b.P + ch * C * C, Ph, C * C * 4);  // the P rows image for the d x d products kernel
      bulk_store_commit();
    }
    if (dm.out_bf16) {
      const __nv_bfloat16* ob = static_cast<const __nv_bfloat16*>(a.dO) + (tok0 * dm.hv + h) * D;
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        int r, c0;
        kmajor_piece(t + it * 256, D, r, c0);
        const uint4 x = r < n ? *reinterpret_cast<const uint4*>(ob + (int64_t)r * dm.hv * D + c0) : z4;
        dov[it][0] = __uint_as_float(x.x);
        dov[it][1] = __uint_as_float(x.y);
        dov[it][2] = __uint_as_float(x.z);
        dov[it][3] = __uint_as_float(x.w);
      }
    } else {
      load_dO_rows(dov, a.dO, false, (tok0 * dm.hv + h) * D, (int64_t)dm.hv * D, n);
    }
    if (t == 0) bulk_wait_read();  // the Qt readout writes over P, step 6 over the K and W rows
    wait_mma();
  }
  // Qt rows hi | lo over the dead P and V rows
  unsigned char* Qrh = KT;
  unsigned char* Qrl = VT;
  if (ok && (warp & 3) < 2) {
    const int i = lrow;
    const float egi = expf(Gs[i]);
    for (int c0 = chalf * 64; c0 < chalf * 64 + 64; c0 += 16) {
      float v[16], qf[16];
      tmem_ld16(tmem_lane_addr(tb, warp, COL_QT + c0), v);
      unpack8(*reinterpret_cast<const uint4*>(Qi + kmajor_off(i, c0, D)), qf);
      unpack8(*reinterpret_cast<const uint4*>(Qi + kmajor_off(i, c0 + 8, D)), qf + 8);
#pragma unroll
      for (int e = 0; e < 16; ++e) v[e] = __fsub_rn(__fmul_rn(egi, qf[e]), v[e]);
      split8(Qrh, Qrl, kmajor_off(i, c0, D), v);
      split8(Qrh, Qrl, kmajor_off(i, c0 + 8, D), v + 8);
    }
  }
  // ---- 6. the operands of L = dO^T Qt, which the reverse chain forms on its tensor cores
  // reading dO^T and Qt^T MN-major from the row images: dO rows over the dead K rows (its lo
  // image, fp32 dO only, over the dead W rows hi), after the Qt rows; the four regions are
  // contiguous and leave as one bulk store into L's slot: [dO hi | Qt hi | Qt lo (| dO lo)]
  static_assert(OFF_KT == OFF_K + TILE && OFF_VT == OFF_KT + TILE && OFF_TK == OFF_VT + TILE,
                "dO, Qt hi, Qt lo, dO lo contiguous");
  if (ok) {
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      int r, c0;
      kmajor_piece(t + it * 256, D, r, c0);
      const uint32_t off = kmajor_off(r, c0, D);
      if (dm.out_bf16)
        *reinterpret_cast<uint4*>(Ki + off) = make_uint4(__float_as_uint(dov[it][0]), __float_as_uint(dov[it][1]),
                                                         __float_as_uint(dov[it][2]), __float_as_uint(dov[it][3]));
      else
        split8(Ki, TKh, off, dov[it]);
    }
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    if (t == 0) {
      bulk_s2g(a.b.L + ch * (int64_t)D * D, smq + OFF_K, dm.out_bf16 ? 3 * TILE : 4 * TILE);
      bulk_store_commit();
    }
  } else if (t == 0) {
    set_error(a.hdr, GDN_DEVERR_TIMEOUT);
    mbar_wait(bar, phase);
  }
  if (t == 0) bulk_wait_all();  // the image stores are complete
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, TMEM_COLS);
}

// ============================================================  KB4 (tcgen05)  ===
// Backward gradients on tensor cores (bf16 inputs, d = 128, C = 64) as two kernels, each
// sized for two CTAs per SM (96 KB operand arena, at most 256 TMEM columns, 128 registers)
// so that one CTA's loads and waits overlap the other's work; the arithmetic of k_bwd_grad
// with its products as MMAs:
//   G1  Pm = Gam (.) (dO U^T) (lower with diagonal), QK = Q K^T      -> dG_b sums, Pm image
//       dQ = diag(e^G) dO S0 + Pm K,  dK1 = Pm^T Q                   -> dq, dG_a
//       X = T^T dU,  Y = T^T dW                                       -> dv, dbeta_a, kY;
//       dk <- dK1 + diag(beta e^G) Y; X and Y as operand images for G2
//   G2  dA = -(Y W^T + X Ut^T) (strictly lower), A' = Gam (.) (K K^T)  -> dbeta_c, dG_e sums
//       dAm = dA beta_i Gam,  dK2 = dAm K + dAm^T K                   -> dk += dK2 + diag(dec) U dS_end
//       dG, reverse cumulative sum -> dg, dbeta
// The row and column sums of the dG terms come straight from the TMEM readouts (per-thread
// row sums, warp-shuffle column sums in a fixed tree).  G1's operands T^T, U^T, dU^T and dW^T
// arrive as ready-made images by bulk copy (the prep and big-products kernels write them),
// as do the Q, K and (bf16) dO rows; X and Y travel through the workspace (the adjoint L,
// dead after the reverse chain) as images that G2 brings in the same way; the per-token
// partial sums go through the image workspace.  Transposed operands are MN-major readings
// of the row images.  A 64-row result is read out by the four warps that own TMEM lanes
// 0..63; the other four meanwhile stage the next readout's global operands (dO S0 and the V
// rows in G1, U dS_end and G1's dk rows in G2) in shared memory.
// 64-row operands use 128-row MMAs whose extra rows read neighbouring arena bytes and are
// never read back.
namespace tcd {
constexpr int D = 128, C = 64;
constexpr uint32_t KB = 1024, ARENA = 96 * KB;
constexpr uint32_t IMG = 16 * KB;  // a 64 x 128 or 128 x 64 bf16 image (hi or lo)
constexpr int TRI = C * (C + 1) / 2;  // packed lower triangle with the diagonal
constexpr size_t SMEM1 = ARENA + (13 * C + TRI) * 4 + 64;
constexpr size_t SMEM2 = ARENA + (18 * C + TRI) * 4 + 64;
constexpr uint32_t TMEM1 = 256, TMEM2 = 128;
}  // namespace tcd

// fixed-order warp sum (xor tree); every lane gets the total
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, off));
  return x;
}

__global__ void __launch_bounds__(256, 2) k_bwd_grad1_tc(BwdArgs a) {
  using namespace tcd;
  using namespace tc;
  extern __shared__ __align__(128) unsigned char smd[];
  unsigned char* ar = smd;
  float* Gs = reinterpret_cast<float*>(smd + ARENA);
  float* eG = Gs + C;
  float* bs = eG + C;
  float* rowp = bs + C;      // [2][C] dG_b row sums, one per column half
  float* colp = rowp + 2 * C;  // [2][C] dG_b column sums, one per row half
  float* dGa = colp + 2 * C;   // [2][C]
  float* dba = dGa + 2 * C;    // [2][C]
  float* kY = dba + 2 * C;     // [2][C]
  float* gam = kY + 2 * C;     // e^{G_i - G_s}, s <= i (decay_table_lower)
  uint64_t* bar = reinterpret_cast<uint64_t*>(gam + TRI);  // [0] MMA, [1] bulk copies
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 2);
  if (!a.hdr->valid) return;
  const Dims dm = a.dm;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int64_t c = blockIdx.x;
  const int h = blockIdx.y;
  const ChunkRec rec = a.chunks[c];
  if (!in_bounds(a.hdr, rec.tok0 >= 0 && rec.len >= 0 && rec.len <= a.dm.C && (int64_t)rec.tok0 + rec.len <= a.T))
    return;
  const int n = rec.len;
  const int64_t tok0 = rec.tok0;
  const int64_t ch = c * dm.hv + h;
  const int64_t CD = (int64_t)C * D;
  const int64_t vstride = (int64_t)dm.hv * D;
  const int64_t orow0 = tok0 * vstride + (int64_t)h * D;  // token 0 of this head in [T, Hv, D]
  const __nv_bfloat16* vb = static_cast<const __nv_bfloat16*>(a.in.v) + orow0;
  unsigned char* gX = reinterpret_cast<unsigned char*>(a.b.L + ch * (int64_t)D * D);  // X hi | lo images
  unsigned char* gY = gX + 2 * IMG;                                                   // Y hi | lo images
  const bool rowlane = (warp & 3) < 2;  // TMEM lanes 0..63 = the chunk's rows
  const int row = (warp & 3) * 32 + lane;
  const int half = warp >> 2;
  const int helper = half * 64 + ((warp & 3) - 2) * 32 + lane;  // 0..127 on warps 2, 3, 6, 7
  const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
  if (t == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
    // the operands of products 1 by bulk copy: the d x d products kernel's U^T image (hi | lo),
    // the prep's Q and K rows images (the image slot) and, for bf16 dO, its dO rows image (the
    // start of L's slot); all of them zero beyond the chunk's tokens
    const unsigned char* qk = reinterpret_cast<const unsigned char*>(a.b.img + ch * (int64_t)prep_w_floats(C, D));
    mbar_expect_tx(&bar[1], (dm.out_bf16 ? 5 : 4) * IMG);
    bulk_g2s(ar + 64 * KB, a.b.U + ch * CD, 2 * IMG, &bar[1]);
    bulk_g2s(ar, qk + IMG, IMG, &bar[1]);
    bulk_g2s(ar + 16 * KB, qk, IMG, &bar[1]);
    if (dm.out_bf16) bulk_g2s(ar + 32 * KB, a.b.L + ch * (int64_t)D * D, IMG, &bar[1]);
  }
  // arena: products 1 Q rows @0, K rows @16, dO hi/lo @32/@48, U^T hi/lo @64/@80; then Pm hi/lo
  // @32/@40 (with Q, K rows), dO S0 rows @48 and V rows @80 (staged); then T^T @0/@8, dU^T
  // @16/@32; then K rows @16, dW^T @48/@64
  {
    float g0 = 0.f, b0 = 0.f;
    if (t < C) {
      g0 = a.b.G[ch * C + t];
      b0 = t < n ? a.in.beta[(tok0 + t) * dm.hv + h] : 0.f;
    }
    if (!dm.out_bf16) {  // fp32 dO rows, split into hi | lo
      float vo[4][8];
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        int r, k0;
        kmajor_piece(t + it * 256, D, r, k0);
        if (r < n) {
          load8(static_cast<const float*>(a.dO) + orow0 + (int64_t)r * vstride + k0, vo[it]);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) vo[it][e] = 0.f;
        }
      }
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        int r, k0;
        kmajor_piece(t + it * 256, D, r, k0);
        split8(ar + 32 * KB, ar + 48 * KB, kmajor_off(r, k0, D), vo[it]);
      }
    }
    if (t < C) {
      Gs[t] = g0;
      bs[t] = b0;
    }
  }
  if (warp == 0) tmem_alloc(tslot, TMEM1);
  fence_proxy_async();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tb = *tslot;
  const uint32_t tl = tmem_lane_addr(tb, warp, 0);
  const uint32_t sa = smem_u32(ar);
  uint32_t phase = 0;
  uint32_t cphase = 0;
  bool ok = true, pending = false, cpending = true;
  auto wait_mma = [&]() {
    const bool done = mbar_wait(&bar[0], phase);
    if (done) {
      phase ^= 1u;
      pending = false;
    }
    ok = __syncthreads_and(done) != 0;
    fence_after_sync();
  };
  // all threads: generic-proxy writes -> tensor core; with copies, thread 0 first waits for
  // the bulk copies in flight and every thread learns whether they arrived
  auto issue = [&](bool copies, auto&& mmas) {
    fence_proxy_async();
    fence_before_sync();
    bool got = true;
    if (t == 0 && copies) {
      got = mbar_wait(&bar[1], cphase);
      if (got) {
        cphase ^= 1u;
        cpending = false;
      }
    }
    ok = __syncthreads_and(got) != 0;
    if (ok && t == 0) {
      fence_after_sync();
      mmas();
      mma_commit(&bar[0]);
      pending = true;
    }
  };
  // ---- products 1: Pm (raw) = dO U^T -> TMEM 0 (U rows: the MN-major reading of the U^T
  // image), QK = Q K^T -> TMEM 64 (after the U^T image)
  issue(true, [&] {
    mma_split(tb + 0, opnd_k(sa + 32 * KB, sa + 48 * KB, D), opnd_mn(sa + 64 * KB, sa + 80 * KB, C), D,
              idesc_bf16(128, C) | IDESC_B_MN, dm.out_bf16 ? -2 : 3);
    mma_terms(tb + 64, sa, sa, sa + 16 * KB, sa + 16 * KB, D, idesc_bf16(128, C), 1);
  });
  if (t < C) eG[t] = expf(Gs[t]);
  decay_table_lower(gam, Gs);  // while the products run
  wait_mma();
  if (ok && rowlane) {  // Pm, dG_b row / column sums, Pm image
    const int i = row;
    float rp = 0.f;
#pragma unroll
    for (int s1 = 0; s1 < 2; ++s1) {
      const int s0 = half * 32 + 16 * s1;
      float pm[16], qk[16];
      tmem_ld16(tl + 0 + s0, pm);
      tmem_ld16(tl + 64 + s0, qk);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int s = s0 + e;
        const float pv = (i >= s) ? __fmul_rn(gam[i * (i + 1) / 2 + s], pm[e]) : 0.f;
        const float pr = (i > s) ? __fmul_rn(pv, qk[e]) : 0.f;
        pm[e] = pv;
        qk[e] = pr;
        rp = __fadd_rn(rp, pr);
      }
      split8(ar + 32 * KB, ar + 40 * KB, kmajor_off(i, s0, C), pm);
      split8(ar + 32 * KB, ar + 40 * KB, kmajor_off(i, s0 + 8, C), pm + 8);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float cs = warp_sum(qk[e]);
        if (lane == 0) colp[(warp & 3) * C + s0 + e] = cs;
      }
    }
    rowp[half * C + i] = rp;
  } else if (ok) {
    // meanwhile the other warps stage, in the operands of products 1 that are dead now, the
    // d x d products kernel's dO S0 rows for the dQ readout (@48..@80; row r's 16-byte piece j
    // at r * 512 + ((j ^ (r & 7)) * 16), so that the readout's lanes, consecutive rows, hit
    // distinct banks) and the V rows image for the dv readout (@80)
    const float* dos_g = a.b.dOS0 + ch * CD;
#pragma unroll
    for (int bt = 0; bt < 2; ++bt) {
      float4 u[8];
      uint4 vr[4];
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        const int q = helper + 128 * (8 * bt + x), r = q >> 5, j = q & 31;
        u[x] = *reinterpret_cast<const float4*>(dos_g + r * D + 4 * j);
      }
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        int r, k0;
        kmajor_piece(helper + (4 * bt + it) * 128, D, r, k0);
        vr[it] = r < n ? *reinterpret_cast<const uint4*>(vb + r * vstride + k0) : zero4;
      }
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        const int q = helper + 128 * (8 * bt + x), r = q >> 5, j = q & 31;
        *reinterpret_cast<float4*>(ar + 48 * KB + r * 512 + ((j ^ (r & 7)) << 4)) = u[x];
      }
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        int r, k0;
        kmajor_piece(helper + (4 * bt + it) * 128, D, r, k0);
        *reinterpret_cast<uint4*>(ar + 80 * KB + kmajor_off(r, k0, D)) = vr[it];
      }
    }
  }
  fence_before_sync();
  __syncthreads();
  // ---- products 2: dQ = Pm K -> TMEM 0, dK1 = Pm^T Q -> TMEM 128; K^T, Q^T and Pm^T are the
  // MN-major readings of the K rows, Q rows and Pm images.  Meanwhile the row warps take their
  // q pieces for the dQ readout from the Q rows image (products 3's T^T comes in over it)
  uint4 qall[8];
  if (ok) {
    issue(false, [&] {
      const Opnd pm_k = opnd_k(sa + 32 * KB, sa + 40 * KB, C), pm_t = opnd_mn(sa + 32 * KB, sa + 40 * KB, C);
      mma_split(tb + 0, pm_k, opnd_mn(sa + 16 * KB, sa + 16 * KB, D), C, idesc_bf16(128, D) | IDESC_B_MN, 2);
      mma_split(tb + 128, pm_t, opnd_mn(sa, sa, D), C, idesc_bf16(128, D) | IDESC_A_MN | IDESC_B_MN, 2);
    });
    if (rowlane) {
#pragma unroll
      for (int x = 0; x < 8; ++x) qall[x] = *reinterpret_cast<const uint4*>(ar + kmajor_off(row, half * 64 + 8 * x, D));
    }
    if (ok) wait_mma();
  }
  // products 3's operands T^T and dU^T: ready-made images (the prep and big-products kernels
  // wrote them), one bulk copy each into the dead operands of products 1 and 2
  if (ok && t == 0) {
    mbar_expect_tx(&bar[1], 2 * C * C * 2 + 2 * IMG);
    bulk_g2s(ar, a.b.T + ch * C * C, 2 * C * C * 2, &bar[1]);
    bulk_g2s(ar + 16 * KB, a.b.L + ch * (int64_t)D * D + D * D / 2, 2 * IMG, &bar[1]);
    cpending = true;
  }
  // dQ readout (row warps): dO S0 from the staged rows, q from registers
  if (ok && rowlane) {
    {
      const int i = row;
      const bool live = i < n;
      const float egi = eG[i];
      const unsigned char* dos_s = ar + 48 * KB + i * 512;
      float pga = 0.f;
#pragma unroll
      for (int c0 = half * 64; c0 < half * 64 + 64; c0 += 16) {
        float4 ds4[4];
#pragma unroll
        for (int x = 0; x < 4; ++x)
          ds4[x] = *reinterpret_cast<const float4*>(dos_s + ((((c0 >> 2) + x) ^ (i & 7)) << 4));
        float dq[16], qf[16], ds[16];
        tmem_ld16(tl + 0 + c0, dq);
        unpack8(qall[(c0 - half * 64) / 8], qf);
        unpack8(qall[(c0 - half * 64) / 8 + 1], qf + 8);
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          ds[4 * x] = ds4[x].x;
          ds[4 * x + 1] = ds4[x].y;
          ds[4 * x + 2] = ds4[x].z;
          ds[4 * x + 3] = ds4[x].w;
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          pga = __fmaf_rn(ds[e], qf[e], pga);
          dq[e] = __fmaf_rn(egi, ds[e], dq[e]);
        }
        if (live) {
          float4* dqp = reinterpret_cast<float4*>(a.b.dq_part + orow0 + (int64_t)i * vstride + c0);
#pragma unroll
          for (int x = 0; x < 4; ++x) dqp[x] = make_float4(dq[4 * x], dq[4 * x + 1], dq[4 * x + 2], dq[4 * x + 3]);
        }
      }
      dGa[half * C + i] = pga;
    }
  }
  // ---- products 3: X = T^T dU -> TMEM 0
  if (ok) {
    issue(true, [&] { mma_terms(tb + 0, sa, sa + 8 * KB, sa + 16 * KB, sa + 32 * KB, C, idesc_bf16(128, D), 3); });
    if (ok) wait_mma();
  }
  // K rows image (the prep kernel's) for the dk readout over the dead dU^T, and products 4's
  // dW^T image (the d x d products kernel's) over the consumed dO S0 rows
  if (ok && t == 0) {
    mbar_expect_tx(&bar[1], 3 * IMG);
    bulk_g2s(ar + 16 * KB, a.b.img + ch * (int64_t)prep_w_floats(C, D), IMG, &bar[1]);
    bulk_g2s(ar + 48 * KB, a.b.dW + ch * CD, 2 * IMG, &bar[1]);
    cpending = true;
  }
  if (ok && rowlane) {  // dv, dbeta_a; X image -> workspace
    const int i = row;
    const bool live = i < n;
    const float bi = bs[i];
    float pba = 0.f;
    for (int cb = half * 64; cb < half * 64 + 64; cb += 32) {
      uint4 vv[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) vv[x] = *reinterpret_cast<const uint4*>(ar + 80 * KB + kmajor_off(i, cb + 8 * x, D));
#pragma unroll
      for (int sub = 0; sub < 2; ++sub) {
        const int c0 = cb + 16 * sub;
        float xr[16], vf[16], dv[16];
        tmem_ld16(tl + 0 + c0, xr);
        unpack8(vv[2 * sub], vf);
        unpack8(vv[2 * sub + 1], vf + 8);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          dv[e] = __fmul_rn(bi, xr[e]);
          pba = __fmaf_rn(vf[e], xr[e], pba);
        }
        if (live) {
          float4* dvp = reinterpret_cast<float4*>(a.dv + orow0 + (int64_t)i * vstride + c0);
#pragma unroll
          for (int x = 0; x < 4; ++x) dvp[x] = make_float4(dv[4 * x], dv[4 * x + 1], dv[4 * x + 2], dv[4 * x + 3]);
        }
        split8(gX, gX + IMG, kmajor_off(i, c0, D), xr);
        split8(gX, gX + IMG, kmajor_off(i, c0 + 8, D), xr + 8);
      }
    }
    dba[half * C + i] = pba;
  }
  // ---- products 4: Y = T^T dW -> TMEM 0 (operands already in place; the K rows copy lands first)
  if (ok) {
    issue(true, [&] { mma_terms(tb + 0, sa, sa + 8 * KB, sa + 48 * KB, sa + 64 * KB, C, idesc_bf16(128, D), 3); });
    if (ok) wait_mma();
  }
  if (ok && rowlane) {  // kY; dk <- dK1 + beta e^G Y; Y image -> workspace
    const int s2 = row;
    const bool live = s2 < n;
    const float bkv = __fmul_rn(bs[s2], eG[s2]);
    float pky = 0.f;
    for (int cb = half * 64; cb < half * 64 + 64; cb += 32) {
      uint4 kv[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) kv[x] = *reinterpret_cast<const uint4*>(ar + 16 * KB + kmajor_off(s2, cb + 8 * x, D));
#pragma unroll
      for (int sub = 0; sub < 2; ++sub) {
        const int c0 = cb + 16 * sub;
        float yr[16], d1[16], kf[16];
        tmem_ld16(tl + 0 + c0, yr);
        tmem_ld16(tl + 128 + c0, d1);
        unpack8(kv[2 * sub], kf);
        unpack8(kv[2 * sub + 1], kf + 8);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          pky = __fmaf_rn(kf[e], yr[e], pky);
          d1[e] = __fmaf_rn(bkv, yr[e], d1[e]);
        }
        if (live) {
          float4* dkp = reinterpret_cast<float4*>(a.b.dk_part + orow0 + (int64_t)s2 * vstride + c0);
#pragma unroll
          for (int x = 0; x < 4; ++x) dkp[x] = make_float4(d1[4 * x], d1[4 * x + 1], d1[4 * x + 2], d1[4 * x + 3]);
        }
        split8(gY, gY + IMG, kmajor_off(s2, c0, D), yr);
        split8(gY, gY + IMG, kmajor_off(s2, c0 + 8, D), yr + 8);
      }
    }
    kY[half * C + s2] = pky;
  }
  fence_before_sync();
  __syncthreads();
  if (ok && t < C) {  // per-token partial sums for G2
    float* gp = a.b.img + ch * (int64_t)prep_w_floats(C, D) + C * D;  // after the K and Q rows images
    gp[t] = __fmul_rn(eG[t], __fadd_rn(dGa[t], dGa[C + t]));                                // e^G dO S0 . q
    gp[C + t] = __fsub_rn(__fadd_rn(rowp[t], rowp[C + t]), __fadd_rn(colp[t], colp[C + t]));  // dG_b
    gp[2 * C + t] = __fadd_rn(dba[t], dba[C + t]);                                          // v . X
    gp[3 * C + t] = __fadd_rn(kY[t], kY[C + t]);                                            // k . Y
  }
  if (!ok && t == 0) {
    set_error(a.hdr, GDN_DEVERR_TIMEOUT);
    if (pending) mbar_wait(&bar[0], phase);
    if (cpending) mbar_wait(&bar[1], cphase);
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, TMEM1);
}

__global__ void __launch_bounds__(256, 2) k_bwd_grad2_tc(BwdArgs a) {
  using namespace tcd;
  using namespace tc;
  extern __shared__ __align__(128) unsigned char smd[];
  unsigned char* ar = smd;
  float* Gs = reinterpret_cast<float*>(smd + ARENA);
  float* eG = Gs + C;
  float* dec = eG + C;
  float* bs = dec + C;
  float* gp = bs + C;          // [4][C] G1's per-token sums
  float* rowb = gp + 4 * C;    // [2][C] dbeta_c row sums, one per column half
  float* rowg = rowb + 2 * C;  // [2][C] dG_e row sums
  float* colg = rowg + 2 * C;  // [2][C] dG_e column sums, one per row half
  float* cs = colg + 2 * C;    // [2][C] U dS_end . k
  float* dgv = cs + 2 * C;
  float* csv = dgv + C;
  float* gtab = csv + C;  // e^{G_i - G_s}, s <= i (decay_table_lower)
  uint64_t* bar = reinterpret_cast<uint64_t*>(gtab + TRI);  // [0] MMA, [1] bulk copies
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 2);
  if (!a.hdr->valid) return;
  const Dims dm = a.dm;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int64_t c = blockIdx.x;
  const int h = blockIdx.y;
  const ChunkRec rec = a.chunks[c];
  if (!in_bounds(a.hdr, rec.tok0 >= 0 && rec.len >= 0 && rec.len <= a.dm.C && (int64_t)rec.tok0 + rec.len <= a.T))
    return;
  const int n = rec.len;
  const int64_t tok0 = rec.tok0;
  const int64_t ch = c * dm.hv + h;
  const int64_t CD = (int64_t)C * D;
  const int64_t vstride = (int64_t)dm.hv * D;
  const int64_t orow0 = tok0 * vstride + (int64_t)h * D;
  const unsigned char* gX = reinterpret_cast<const unsigned char*>(a.b.L + ch * (int64_t)D * D);
  const unsigned char* gY = gX + 2 * IMG;
  const float* img = a.b.img + ch * (int64_t)prep_w_floats(C, D);  // K rows image, then G1's sums
  const bool rowlane = (warp & 3) < 2;
  const int row = (warp & 3) * 32 + lane;
  const int half = warp >> 2;
  // arena: products A W hi/lo @0/@16, Y hi|lo @32, K rows @64; products B Ut hi/lo @0/@16,
  // X hi|lo @32; products C dAm hi/lo @0/@8 (with the K rows), U dS_end rows @16, the first
  // gradients kernel's dk rows @48 and @80 (staged for the dk readout)
  if (t == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
    mbar_expect_tx(&bar[1], 5 * IMG);
    bulk_g2s(ar, a.b.W + ch * CD, 2 * IMG, &bar[1]);  // the prep kernel's W rows image (hi | lo)
    bulk_g2s(ar + 32 * KB, gY, 2 * IMG, &bar[1]);
    bulk_g2s(ar + 64 * KB, img, IMG, &bar[1]);
  }
  {
    float g0 = 0.f, b0 = 0.f, p0 = 0.f;
    if (t < C) {
      g0 = a.b.G[ch * C + t];
      b0 = t < n ? a.in.beta[(tok0 + t) * dm.hv + h] : 0.f;
    }
    p0 = img[C * D + t];  // t < 4 C
    if (t < C) {
      Gs[t] = g0;
      bs[t] = b0;
    }
    gp[t] = p0;
  }
  if (warp == 0) tmem_alloc(tslot, TMEM2);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tb = *tslot;
  const uint32_t tl = tmem_lane_addr(tb, warp, 0);
  const uint32_t sa = smem_u32(ar);
  uint32_t phase = 0, cphase = 0;
  bool ok = true, pending = false, cpending = true;
  auto wait_mma = [&]() {
    const bool done = mbar_wait(&bar[0], phase);
    if (done) {
      phase ^= 1u;
      pending = false;
    }
    ok = __syncthreads_and(done) != 0;
    fence_after_sync();
  };
  // all threads: generic-proxy writes -> tensor core; thread 0 waits for the bulk copies
  // (copies = true), then issues; every thread learns whether the copies arrived
  auto issue = [&](bool copies, auto&& mmas) {
    fence_proxy_async();
    fence_before_sync();
    bool got = true;
    if (t == 0 && copies) {
      got = mbar_wait(&bar[1], cphase);
      if (got) {
        cphase ^= 1u;
        cpending = false;
      }
    }
    ok = __syncthreads_and(got) != 0;
    if (ok && t == 0) {
      fence_after_sync();
      mmas();
      mma_commit(&bar[0]);
      pending = true;
    }
  };
  // ---- products A: dA = Y W^T -> TMEM 0, K K^T -> TMEM 64
  issue(true, [&] {
    mma_terms(tb + 0, sa + 32 * KB, sa + 48 * KB, sa, sa + 16 * KB, D, idesc_bf16(128, C), 3);
    mma_terms(tb + 64, sa + 64 * KB, sa + 64 * KB, sa + 64 * KB, sa + 64 * KB, D, idesc_bf16(128, C), 1);
  });
  SplitTile<false, C, D> ut;
  ut.load(a.b.Ut + ch * CD, D, C);
  if (t < C) {
    eG[t] = expf(Gs[t]);
    dec[t] = expf(__fsub_rn(Gs[C - 1], Gs[t]));
  }
  decay_table_lower(gtab, Gs);  // while the products run
  if (ok) wait_mma();
  // ---- products B: dA += X Ut^T
  if (ok) {
    if (t == 0) {
      mbar_expect_tx(&bar[1], 2 * IMG);
      bulk_g2s(ar + 32 * KB, gX, 2 * IMG, &bar[1]);
      cpending = true;
    }
    ut.store(ar, ar + 16 * KB);
    issue(true, [&] {
      mma_terms(tb + 0, sa + 32 * KB, sa + 48 * KB, sa, sa + 16 * KB, D, idesc_bf16(128, C), 3, true);
    });
    if (ok) wait_mma();
  }
  if (ok && rowlane) {  // dA (strictly lower), A' = Gam (.) K K^T; dbeta_c, dG_e sums; dAm image
    const int i = row;
    const float bi = bs[i];
    float rb = 0.f, rg = 0.f;
#pragma unroll
    for (int s1 = 0; s1 < 2; ++s1) {
      const int s0 = half * 32 + 16 * s1;
      float v[16], kk[16];
      tmem_ld16(tl + 0 + s0, v);
      tmem_ld16(tl + 64 + s0, kk);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int s = s0 + e;
        const bool low = i > s;
        const float gam = low ? gtab[i * (i + 1) / 2 + s] : 0.f;
        const float da = low ? -v[e] : 0.f;
        const float ap = low ? __fmul_rn(gam, kk[e]) : 0.f;
        const float dab = __fmul_rn(da, bi);
        rb = __fmaf_rn(da, ap, rb);
        const float tg = __fmul_rn(dab, ap);
        rg = __fadd_rn(rg, tg);
        v[e] = low ? __fmul_rn(dab, gam) : 0.f;
        kk[e] = tg;
      }
      split8(ar, ar + 8 * KB, kmajor_off(i, s0, C), v);
      split8(ar, ar + 8 * KB, kmajor_off(i, s0 + 8, C), v + 8);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float cg = warp_sum(kk[e]);
        if (lane == 0) colg[(warp & 3) * C + s0 + e] = cg;
      }
    }
    rowb[half * C + i] = rb;
    rowg[half * C + i] = rg;
  } else if (ok) {
    // meanwhile the other warps stage U dS_end and the first gradients kernel's dk rows for
    // the dk readout in the free arena (@16..@64 after products B, @80..@96): row r's 16-byte
    // piece j at r * 512 + ((j ^ (r & 7)) * 16), so that the readout's lanes (consecutive
    // rows, one piece each) hit distinct banks; two batches of 8 + 8 pieces per thread
    const int hl = (warp >> 2) * 64 + ((warp & 3) - 2) * 32 + lane;  // 0..127 on warps 2, 3, 6, 7
    const float* ue_g = a.b.UdSe + ch * CD;
    const float* pk_g = a.b.dk_part + orow0;
#pragma unroll
    for (int bt = 0; bt < 2; ++bt) {
      float4 u[8], pk[8];
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        const int q = hl + 128 * (8 * bt + x), r = q >> 5, j = q & 31;
        u[x] = *reinterpret_cast<const float4*>(ue_g + r * D + 4 * j);
        pk[x] = r < n ? *reinterpret_cast<const float4*>(pk_g + (int64_t)r * vstride + 4 * j)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        const int q = hl + 128 * (8 * bt + x), r = q >> 5, j = q & 31;
        const uint32_t sw = (uint32_t)((j ^ (r & 7)) << 4);
        *reinterpret_cast<float4*>(ar + 16 * KB + r * 512 + sw) = u[x];
        *reinterpret_cast<float4*>((r < 32 ? ar + 48 * KB + r * 512 : ar + 80 * KB + (r - 32) * 512) + sw) = pk[x];
      }
    }
  }
  fence_before_sync();
  __syncthreads();
  // ---- products C: dK2 = dAm K + dAm^T K -> TMEM 0; dAm^T and K^T are the MN-major readings
  // of the dAm and K rows images
  if (ok) {
    issue(false, [&] {
      const Opnd kt = opnd_mn(sa + 64 * KB, sa + 64 * KB, D);
      mma_split(tb + 0, opnd_k(sa, sa + 8 * KB, C), kt, C, idesc_bf16(128, D) | IDESC_B_MN, 2);
      const Opnd dat = opnd_mn(sa, sa + 8 * KB, C);
      mma_part(tb + 0, dat, false, kt, false, C, idesc_bf16(128, D) | IDESC_A_MN | IDESC_B_MN, true);
      mma_part(tb + 0, dat, true, kt, false, C, idesc_bf16(128, D) | IDESC_A_MN | IDESC_B_MN, true);
    });
    if (ok) wait_mma();
  }
  if (ok && rowlane) {  // dk = G1's part + dK2 + dec U dS_end; U dS_end . k
    const int s2 = row;
    const bool live = s2 < n;
    const unsigned char* ue_s = ar + 16 * KB + s2 * 512;  // the staged rows (swizzled pieces)
    const unsigned char* pk_s = (s2 < 32 ? ar + 48 * KB : ar + 80 * KB - 32 * 512) + s2 * 512;
    float* dk_row = a.b.dk_part + orow0 + (int64_t)s2 * vstride;
    const float ds = dec[s2];
    float pcs = 0.f;
    for (int cb = half * 64; cb < half * 64 + 64; cb += 16) {
      float4 ue4[4], pk4[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const uint32_t sw = (uint32_t)((((cb >> 2) + x) ^ (s2 & 7)) << 4);
        ue4[x] = *reinterpret_cast<const float4*>(ue_s + sw);
        pk4[x] = live ? *reinterpret_cast<const float4*>(pk_s + sw) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      const uint4 k0 = *reinterpret_cast<const uint4*>(ar + 64 * KB + kmajor_off(s2, cb, D));
      const uint4 k1 = *reinterpret_cast<const uint4*>(ar + 64 * KB + kmajor_off(s2, cb + 8, D));
      float v[16], kf[16], ue[16], pk[16];
      tmem_ld16(tl + 0 + cb, v);
      unpack8(k0, kf);
      unpack8(k1, kf + 8);
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        ue[4 * x] = ue4[x].x;
        ue[4 * x + 1] = ue4[x].y;
        ue[4 * x + 2] = ue4[x].z;
        ue[4 * x + 3] = ue4[x].w;
        pk[4 * x] = pk4[x].x;
        pk[4 * x + 1] = pk4[x].y;
        pk[4 * x + 2] = pk4[x].z;
        pk[4 * x + 3] = pk4[x].w;
      }
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        v[e] = __fmaf_rn(ds, ue[e], __fadd_rn(pk[e], v[e]));
        pcs = __fmaf_rn(ue[e], kf[e], pcs);
      }
      if (live) {
        float4* o4 = reinterpret_cast<float4*>(dk_row + cb);
#pragma unroll
        for (int x = 0; x < 4; ++x) o4[x] = make_float4(v[4 * x], v[4 * x + 1], v[4 * x + 2], v[4 * x + 3]);
      }
    }
    cs[half * C + s2] = pcs;
  }
  fence_before_sync();
  __syncthreads();
  if (!ok) {
    if (t == 0) {
      set_error(a.hdr, GDN_DEVERR_TIMEOUT);
      if (pending) mbar_wait(&bar[0], phase);
      if (cpending) mbar_wait(&bar[1], cphase);
    }
  }
  // dG per token (independent terms, one thread each), then thread 0 takes the two
  // sequential sums: the total of the U dS_end terms and the reverse cumulative sum -> dg
  if (ok && t < C) {
    const int i = t;
    const float csi = __fmul_rn(dec[i], __fadd_rn(cs[i], cs[C + i]));
    const float dGe = __fsub_rn(__fadd_rn(rowg[i], rowg[C + i]), __fadd_rn(colg[i], colg[C + i]));
    float v = __fadd_rn(gp[i], gp[C + i]);
    v = __fsub_rn(v, csi);
    v = __fmaf_rn(__fmul_rn(bs[i], eG[i]), gp[3 * C + i], v);
    v = __fadd_rn(v, dGe);
    dgv[i] = v;
    csv[i] = csi;
  }
  __syncthreads();
  if (ok && t == 0) {
    float tot = 0.f;
#pragma unroll
    for (int s2 = 0; s2 < C; ++s2) tot = __fadd_rn(tot, csv[s2]);
    float run = 0.f;
#pragma unroll
    for (int i = C - 1; i >= 0; --i) {
      float v = dgv[i];
      if (i == C - 1) v = __fadd_rn(v, __fmaf_rn(expf(Gs[C - 1]), a.b.sdot[ch], tot));
      run = __fadd_rn(run, v);
      dgv[i] = run;
    }
  }
  __syncthreads();
  if (ok && t < n) {
    const float dbc = __fadd_rn(rowb[t], rowb[C + t]);
    a.dg[(tok0 + t) * dm.hv + h] = dgv[t];
    a.dbeta[(tok0 + t) * dm.hv + h] = __fadd_rn(__fmaf_rn(eG[t], gp[3 * C + t], gp[2 * C + t]), dbc);
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, TMEM2);
}
template <int D, typename Tin>
void launch_bwd_t(const BwdArgs& a, int64_t n_chunks, int N, BwdStageFn mark, void* mark_ctx,
                  cudaStream_t st) {
  const dim3 gc((unsigned)n_chunks, a.dm.hv);
  if (n_chunks > 0) {
    if (boundary_on_tensor_cores(a.dm)) {
      ensure_smem_bwd(k_bwd_prep_tc, tcq::SMEM);
      k_bwd_prep_tc<<<gc, 256, tcq::SMEM, st>>>(a);
    } else {
      ensure_smem_bwd(k_bwd_prep<D, Tin>, bprep_smem<D>());
      k_bwd_prep<D, Tin><<<gc, NT, bprep_smem<D>(), st>>>(a);
    }
  }
  mark(mark_ctx, n_chunks > 0 ? 1 : 0);
  if (boundary_on_tensor_cores(a.dm)) {
    ensure_smem_bwd(k_bwd_chain_tc, tcb::SMEM);
    k_bwd_chain_tc<<<dim3((unsigned)N, a.dm.hv), 256, tcb::SMEM, st>>>(a);
  } else {
    ensure_smem_bwd(k_bwd_chain<D, Tin>, bchain_smem<D>());
    k_bwd_chain<D, Tin><<<dim3((unsigned)N, a.dm.hv, D / kRowsPerChain), NT, bchain_smem<D>(), st>>>(a);
  }
  mark(mark_ctx, 1);
  if (n_chunks > 0) {
    if (boundary_on_tensor_cores(a.dm)) {
      ensure_smem_bwd(k_bwd_big_tc, tcg::SMEM);
      k_bwd_big_tc<<<gc, 256, tcg::SMEM, st>>>(a);
    } else {
      ensure_smem_bwd(k_bwd_big<D, Tin>, bbig_smem<D>());
      k_bwd_big<D, Tin><<<gc, NT, bbig_smem<D>(), st>>>(a);
    }
  }
  mark(mark_ctx, n_chunks > 0 ? 1 : 0);
  if (n_chunks > 0) {
    if (boundary_on_tensor_cores(a.dm)) {
      ensure_smem_bwd(k_bwd_grad1_tc, tcd::SMEM1);
      k_bwd_grad1_tc<<<gc, 256, tcd::SMEM1, st>>>(a);
      ensure_smem_bwd(k_bwd_grad2_tc, tcd::SMEM2);
      k_bwd_grad2_tc<<<gc, 256, tcd::SMEM2, st>>>(a);
    } else {
      ensure_smem_bwd(k_bwd_grad<D, Tin>, bgrad_smem<D>());
      k_bwd_grad<D, Tin><<<gc, NT, bgrad_smem<D>(), st>>>(a);
    }
  }
  mark(mark_ctx, n_chunks > 0 ? (boundary_on_tensor_cores(a.dm) ? 2 : 1) : 0);
  if (a.T > 0) {
    const int64_t rows = a.T * a.dm.hqk, per_block = 256 / (D / 4);
    k_bwd_gqa<<<(unsigned)((rows + per_block - 1) / per_block), 256, 0, st>>>(a.b.dq_part, a.b.dk_part, a.dq, a.dk,
                                                                              a.T, a.dm.hqk, a.dm.hv, D, a.hdr);
  }
  mark(mark_ctx, a.T > 0 ? 1 : 0);
}

}  // namespace

size_t bwd_workspace_floats_per_chunk_head(int C, int D) {
  return (size_t)7 * C * D + 2 * (size_t)C * C + C + 2 * (size_t)D * D + 1 + prep_w_floats(C, D) + 3;
}

void launch_bwd(const Dims& d, const TokenArrays& in, const void* dO, const ChunkRec* chunks,
                const SeqRec* seqs, int N, int64_t n_chunks, int64_t T, const float* saved_bnd,
                const float* dstate_out, float* dstate_in, float* per_chunk, float* dq_part,
                float* dk_part, float* dq, float* dk, float* dv, float* dg, float* dbeta,
                WsHeader* hdr, BwdStageFn mark, void* mark_ctx, cudaStream_t st) {
  BwdArgs a{};
  a.dm = d;
  a.in = in;
  a.dO = dO;
  a.chunks = chunks;
  a.seqs = seqs;
  a.saved_bnd = saved_bnd;
  a.dstate_out = dstate_out;
  a.dstate_in = dstate_in;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.dg = dg;
  a.dbeta = dbeta;
  a.T = T;
  a.n_chunks = n_chunks;
  a.N = N;
  a.hdr = hdr;
  const size_t C = d.C, D = d.D, nch = (size_t)n_chunks * d.hv;
  float* p = per_chunk;
  a.b.W = p;    p += nch * C * D;
  a.b.Ut = p;   p += nch * C * D;
  a.b.U = p;    p += nch * C * D;
  a.b.dU = p;   p += nch * C * D;
  a.b.dOS0 = p; p += nch * C * D;
  a.b.UdSe = p; p += nch * C * D;
  a.b.dW = p;   p += nch * C * D;
  a.b.T = p;    p += nch * C * C;
  a.b.P = p;    p += nch * C * C;
  a.b.L = p;    p += nch * D * D;
  a.b.dSE = p;  p += nch * D * D;
  a.b.G = p;    p += nch * C;
  a.b.sdot = p; p += nch;
  p += (4 - ((p - per_chunk) & 3)) & 3;  // 16-byte alignment for the bulk-copied images
  a.b.img = p;  p += nch * prep_w_floats((int)C, (int)D);
  a.b.dq_part = dq_part;
  a.b.dk_part = dk_part;
  if (d.in_bf16) {
    switch (d.D) {
      case 32: launch_bwd_t<32, __nv_bfloat16>(a, n_chunks, N, mark, mark_ctx, st); break;
      case 64: launch_bwd_t<64, __nv_bfloat16>(a, n_chunks, N, mark, mark_ctx, st); break;
      default: launch_bwd_t<128, __nv_bfloat16>(a, n_chunks, N, mark, mark_ctx, st); break;
    }
  } else {
    switch (d.D) {
      case 32: launch_bwd_t<32, float>(a, n_chunks, N, mark, mark_ctx, st); break;
      case 64: launch_bwd_t<64, float>(a, n_chunks, N, mark, mark_ctx, st); break;
      default: launch_bwd_t<128, float>(a, n_chunks, N, mark, mark_ctx, st); break;
    }
  }
}

}  // namespace gdn
