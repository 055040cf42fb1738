// kernels_fwd.cu -- forward-path kernels of CPR Gated DeltaNet for sm_103a.
//
// CPR (IsoExec page, section "Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet") keeps
// the gated delta-rule recurrence as the main computation and evaluates it in parallel
// across chunks; decode resynchronises its state every C tokens.  Here:
//   K0 k_worklist  chunk/sequence records from cu_seqlens (device-checked)
//   K1a k_prep     chunk pre-pass, parallel over (chunk, head):
//                    G = cumsum g, A_is = beta_i e^{G_i-G_s} k_i.k_s (i>s), T = (I+A)^-1,
//                    Wd = diag(e^{G_C-G}) T diag(beta e^G) K,  Ud = diag(e^{G_C-G}) T diag(beta) V
//   K1b k_chain    boundary chain, sequential over chunks per (sequence, head, row block):
//                    Vd = Ud - Wd S^T,   S <- e^{G_C} S + Vd^T K
//   K2 k_intra     token recurrence inside every chunk from its boundary state
//   K3 k_decode    one token step per decode slot, appended to the slot's chunk tail
// Prefill and decode resync run the very same k_prep/k_chain code on the same values, and
// K2 and K3 call the same token_step, which is what makes every mode bit-identical.
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

// Opt a kernel into more than 48 KB of dynamic shared memory, once per (kernel, device):
// later calls (including ones made while a CUDA graph is being captured) skip the runtime
// call entirely.
template <typename F>
static void ensure_smem(F* fn, size_t bytes) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  if (done.insert({reinterpret_cast<const void*>(fn), dev}).second)
    cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

constexpr int kRankSeqs = 64;  // batches the boundary chains order longest first (ranked per CTA)

// Streaming multiprocessors of the current device (looked up once per device).
static int sm_count() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

// =====================================================================  K0  ====
__global__ void __launch_bounds__(1024) k_worklist(const int32_t* __restrict__ cu, int N, int T,
                                                   int C, int64_t n_chunks, uint32_t cu_hash,
                                                   ChunkRec* __restrict__ chunks,
                                                   SeqRec* __restrict__ seqs,
                                                   WsHeader* __restrict__ hdr) {
  __shared__ int64_t scan[1024];
  __shared__ int bad;
  __shared__ uint32_t hsum;
  const int t = threadIdx.x;
  if (t == 0) {
    bad = 0;
    hsum = 0;
  }
  __syncthreads();
  int64_t carry = 0;
  for (int base = 0; base <= N; base += 1024) {
    const int s = base + t;
    int64_t nc = 0;
    int32_t tok0 = 0, L = 0;
    if (s <= N) {
      const int32_t c = cu[s];
      atomicAdd(&hsum, (uint32_t)c * (uint32_t)(2 * s + 1));
      if (s == 0 && c != 0) bad = 1;
      if (s == N && c != T) bad = 1;
    }
    if (s < N) {
      tok0 = cu[s];
      L = cu[s + 1] - tok0;
      if (L < 0 || tok0 < 0) bad = 1;
      nc = (L > 0) ? (L + C - 1) / C : 0;
    }
    scan[t] = nc;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {
      const int64_t x = (t >= off) ? scan[t - off] : 0;
      __syncthreads();
      scan[t] += x;
      __syncthreads();
    }
    const int64_t first = carry + scan[t] - nc;
    if (s < N && L >= 0) {
      seqs[s] = SeqRec{tok0, L, (int32_t)first, (int32_t)nc};
      for (int64_t j = 0; j < nc; ++j) {
        const int64_t c = first + j;
        if (c < n_chunks) {
          const int32_t rem = L - (int32_t)(j * C);
          chunks[c] = ChunkRec{s, tok0 + (int32_t)(j * C), rem < C ? rem : C, (int32_t)j};
        }
      }
    }
    carry += scan[1023];
    __syncthreads();
  }
  if (t == 0) {
    if (bad || carry != n_chunks || hsum != cu_hash) {
      set_error(hdr, GDN_DEVERR_CU_SEQLENS);
      hdr->valid = 0;
    } else {
      hdr->valid = 1;
    }
  }
}

void launch_worklist(const int32_t* cu, int N, int T, int C, int64_t n_chunks, uint32_t cu_hash,
                     ChunkRec* chunks, SeqRec* seqs, WsHeader* hdr, cudaStream_t st) {
  k_worklist<<<1, 1024, 0, st>>>(cu, N, T, C, n_chunks, cu_hash, chunks, seqs, hdr);
}

// =====================================================================  K1a  ===
// Shared-memory plan (floats): Ks[64][D+4] Vs[64][D+4] A[64][65] T[64][65] + 5 vectors.
template <int D>
constexpr size_t prep_smem_bytes() {
  return sizeof(float) * (2 * kMaxChunk * (D + 4) + 2 * kMaxChunk * (kMaxChunk + 1) + 5 * kMaxChunk +
                          3 * 16 * 16 + 4);
}

template <int D, typename Tin, bool TC>
__global__ void __launch_bounds__(kPrepThreads) k_prep(Dims dm, TokenArrays in, PrepWork w,
                                                       float* __restrict__ Wout,
                                                       float* __restrict__ Uout,
                                                       float* __restrict__ gamma_out,
                                                       WsHeader* __restrict__ hdr) {
  constexpr int DP = D + 4;
  constexpr int CP = kMaxChunk + 1;
  extern __shared__ __align__(16) float sm[];
  float* Ks = sm;
  float* Vs = Ks + kMaxChunk * DP;
  float* A = Vs + kMaxChunk * DP;
  float* Tm = A + kMaxChunk * CP;
  float* gs = Tm + kMaxChunk * CP;
  float* Gs = gs + kMaxChunk;
  float* bs = Gs + kMaxChunk;
  float* bk = bs + kMaxChunk;
  float* dec = bk + kMaxChunk;
  float* Xs = dec + kMaxChunk;  // off-diagonal block scratch of the triangular solve

  const int t = threadIdx.x;
  const int C = dm.C;
  const int h = blockIdx.y;
  const int hq = h / (dm.hv / dm.hqk);
  const int64_t item = blockIdx.x;
  int64_t tok0;
  if (w.chunks) {  // prefill: chunk record
    if (!hdr->valid) return;
    const ChunkRec rec = w.chunks[item];
    if (rec.len != C) return;  // only full chunks advance a boundary state
    tok0 = rec.tok0;
    if (!in_bounds(hdr, tok0 >= 0 && tok0 + C <= in.n_tokens)) return;
  } else {  // decode: the slot's tail, when this token completes it
    const int sl = w.slot[item];
    if (sl < 0 || sl >= w.slots) {
      if (t == 0 && h == 0) set_error(hdr, GDN_DEVERR_SLOT);
      return;
    }
    const int p = w.pos[sl];
    if (p < 0) {
      if (t == 0 && h == 0) set_error(hdr, GDN_DEVERR_POS);
      return;
    }
    if ((p + 1) % C != 0) return;
    tok0 = (int64_t)sl * C;
    if (!in_bounds(hdr, tok0 + C <= in.n_tokens)) return;
  }
  const Tin* kin = static_cast<const Tin*>(in.k);
  const Tin* vin = static_cast<const Tin*>(in.v);

  // 1. chunk inputs -> fp32 shared memory
  for (int idx = t; idx < C * (D / 4); idx += kPrepThreads) {
    const int r = idx / (D / 4), c4 = idx % (D / 4);
    *reinterpret_cast<float4*>(Ks + r * DP + 4 * c4) = load4(kin + ((tok0 + r) * dm.hqk + hq) * D + 4 * c4);
    *reinterpret_cast<float4*>(Vs + r * DP + 4 * c4) = load4(vin + ((tok0 + r) * dm.hv + h) * D + 4 * c4);
  }
  if (t < C) {
    gs[t] = in.g[(tok0 + t) * dm.hv + h];
    bs[t] = in.beta[(tok0 + t) * dm.hv + h];
  }
  __syncthreads();
  // 2. G_i = g_0 + ... + g_i, left to right
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
  // 3. decay factors and A (strictly lower)
  if (t < C) {
    bk[t] = __fmul_rn(bs[t], expf(Gs[t]));
    dec[t] = expf(__fsub_rn(Gs[C - 1], Gs[t]));
  }
  for (int o = t; o < C * C; o += kPrepThreads) {
    const int i = o / C, s = o % C;
    if (i > s) {
      const float e = expf(__fsub_rn(Gs[i], Gs[s]));
      A[i * CP + s] = __fmul_rn(__fmul_rn(bs[i], e), dot_canon<D>(Ks + i * DP, Ks + s * DP));
    }
  }
  __syncthreads();
  // 4. T = (I + A)^{-1} (blocked forward substitution, fixed order)
  blocked_unit_lower_inverse<kPrepThreads>(A, Tm, Xs, C, CP);
  // 5. TK = T diag(beta e^G) (into A), TV = T diag(beta) (in place)
  for (int o = t; o < C * C; o += kPrepThreads) {
    const int i = o / C, r = o % C;
    if (r <= i) {
      const float x = Tm[i * CP + r];
      A[i * CP + r] = __fmul_rn(x, bk[r]);
      Tm[i * CP + r] = __fmul_rn(x, bs[r]);
    }
  }
  __syncthreads();
  // 6. Wd[i][c] = dec_i * sum_{r<=i} TK[i][r] K[r][c];  Ud[i][c] = dec_i * sum_{r<=i} TV[i][r] V[r][c]
  //    (r ascending).  Each thread owns one column c and every RG-th row.
  constexpr int RG = kPrepThreads / D;  // row groups
  constexpr int RPT = kMaxChunk / RG;   // rows per thread at the largest chunk
  const int c = t % D, i0 = t / D;
  float* Wo = Wout + (item * dm.hv + h) * (int64_t)prep_w_floats(C, D);
  float* Uo = Uout + ((item * dm.hv + h) * C) * (int64_t)D;
  float aw[RPT], au[RPT];
#pragma unroll
  for (int j = 0; j < RPT; ++j) aw[j] = au[j] = 0.f;
  for (int r = 0; r < C; ++r) {
    const float kv = Ks[r * DP + c], vv = Vs[r * DP + c];
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
      const int i = i0 + RG * j;
      if (i >= r && i < C) {
        aw[j] = __fmaf_rn(A[i * CP + r], kv, aw[j]);
        au[j] = __fmaf_rn(Tm[i * CP + r], vv, au[j]);
      }
    }
  }
  if constexpr (!TC) {
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
      const int i = i0 + RG * j;
      if (i < C) {
        Wo[i * D + c] = __fmul_rn(dec[i], aw[j]);
        Uo[i * D + c] = __fmul_rn(dec[i], au[j]);
      }
    }
  } else {
    // Tensor-core chain operands, as ready-made K-major shared-memory images:
    //   [Wd hi (C x D) | Wd lo (C x D) | K^T (D x C)] in bf16; Ud stays fp32.
    unsigned char* img = reinterpret_cast<unsigned char*>(Wo);
    unsigned char* imgK = img + 2 * C * D * 2;
    for (int q = t; q < D * (C / 8); q += kPrepThreads) {  // K^T: row c, 8 keys at a time
      const int cc = q / (C / 8), s0 = (q % (C / 8)) * 8;
      uint32_t w4[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t lo16 = __bfloat16_as_ushort(__float2bfloat16_rn(Ks[(s0 + 2 * e) * DP + cc]));
        const uint32_t hi16 = __bfloat16_as_ushort(__float2bfloat16_rn(Ks[(s0 + 2 * e + 1) * DP + cc]));
        w4[e] = lo16 | (hi16 << 16);
      }
      *reinterpret_cast<uint4*>(imgK + tc::kmajor_off(cc, s0, C)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
      const int i = i0 + RG * j;
      if (i < C) {
        Ks[i * DP + c] = __fmul_rn(dec[i], aw[j]);
        Uo[i * D + c] = __fmul_rn(dec[i], au[j]);
      }
    }
    __syncthreads();
    for (int q = t; q < C * (D / 8); q += kPrepThreads) {  // Wd split: row s, 8 columns at a time
      int s, b0;
      tc::kmajor_piece(q, D, s, b0);
      uint32_t hw[4], lw[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        __nv_bfloat16 h0, l0, h1, l1;
        tc::split_bf16(Ks[s * DP + b0 + 2 * e], h0, l0);
        tc::split_bf16(Ks[s * DP + b0 + 2 * e + 1], h1, l1);
        hw[e] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
        lw[e] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
      }
      const uint32_t off = tc::kmajor_off(s, b0, D);
      *reinterpret_cast<uint4*>(img + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      *reinterpret_cast<uint4*>(img + C * D * 2 + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
  }
  if (t == 0) gamma_out[item * dm.hv + h] = expf(Gs[C - 1]);
}

template <int D, typename Tin, bool TC = false>
static void launch_prep_t(const Dims& d, const TokenArrays& in, const PrepWork& w, float* W,
                          float* U, float* gamma, WsHeader* hdr, cudaStream_t st) {
  constexpr size_t smem = prep_smem_bytes<D>();
  ensure_smem(k_prep<D, Tin, TC>, smem);
  dim3 grid((unsigned)w.n_items, d.hv);
  k_prep<D, Tin, TC><<<grid, kPrepThreads, smem, st>>>(d, in, w, W, U, gamma, hdr);
}

// =====================================================================  K1b  ===
// Shared-memory plan (floats): Ws[64][D+4] Ks[64][D+4] Ss[16][D+4] Us[64][16] Vd[64][16].
template <int D>
constexpr size_t chain_smem_bytes() {
  return sizeof(float) * (2 * kMaxChunk * (D + 4) + kRowsPerChain * (D + 4) + 2 * kMaxChunk * kRowsPerChain);
}

// One boundary step on rows [r0, r0+16) of S (in Ss):  Vd = Ud - Wd S^T,  S <- gamma S + Vd^T K.
// Vd[s][i] = Ud[s][i] - dot_canon(Wd[s], S[i]);  S[i][c] = gamma S[i][c] + sum_s Vd[s][i] K[s][c]
// with s ascending after the gamma term.
template <int D, typename Tin>
__device__ __forceinline__ void chain_step(float* Ss, float* Ws, float* Ks, float* Us, float* Vd,
                                           const float* __restrict__ Wg, const float* __restrict__ Ug,
                                           float gamma, const Tin* __restrict__ keys, int64_t tok0,
                                           int hqk, int hq, int C, int r0) {
  constexpr int DP = D + 4;
  constexpr int R = kRowsPerChain;
  const int t = threadIdx.x;
  for (int idx = t; idx < C * (D / 4); idx += kChainThreads) {
    const int s = idx / (D / 4), c4 = idx % (D / 4);
    *reinterpret_cast<float4*>(Ws + s * DP + 4 * c4) = reinterpret_cast<const float4*>(Wg + s * D)[c4];
  }
  for (int idx = t; idx < C * (D / 8); idx += kChainThreads) {
    const int s = idx / (D / 8), c8 = idx % (D / 8);
    float tmp[8];
    load8(keys + ((tok0 + s) * hqk + hq) * D + 8 * c8, tmp);
#pragma unroll
    for (int e = 0; e < 8; ++e) Ks[s * DP + 8 * c8 + e] = tmp[e];
  }
  for (int idx = t; idx < C * (R / 4); idx += kChainThreads) {
    const int s = idx / (R / 4), i4 = idx % (R / 4);
    *reinterpret_cast<float4*>(Us + s * R + 4 * i4) = *reinterpret_cast<const float4*>(Ug + s * D + r0 + 4 * i4);
  }
  __syncthreads();
  {  // Vd: thread owns row i = t / 16 and chunk rows s = t % 16 + 16 j
    const int i = t / 16, s0 = t % 16;
    constexpr int SJ = kMaxChunk / 16;
    float p[SJ][4];
#pragma unroll
    for (int j = 0; j < SJ; ++j) p[j][0] = p[j][1] = p[j][2] = p[j][3] = 0.f;
#pragma unroll 4
    for (int m = 0; m < D / 4; ++m) {
      const float4 sv = *reinterpret_cast<const float4*>(Ss + i * DP + 4 * m);
#pragma unroll
      for (int j = 0; j < SJ; ++j) {
        if (s0 + 16 * j < C) {
          const float4 wv = *reinterpret_cast<const float4*>(Ws + (s0 + 16 * j) * DP + 4 * m);
          p[j][0] = __fmaf_rn(wv.x, sv.x, p[j][0]);
          p[j][1] = __fmaf_rn(wv.y, sv.y, p[j][1]);
          p[j][2] = __fmaf_rn(wv.z, sv.z, p[j][2]);
          p[j][3] = __fmaf_rn(wv.w, sv.w, p[j][3]);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < SJ; ++j) {
      const int s = s0 + 16 * j;
      if (s < C) {
        const float dot = __fadd_rn(__fadd_rn(p[j][0], p[j][1]), __fadd_rn(p[j][2], p[j][3]));
        Vd[s * R + i] = __fsub_rn(Us[s * R + i], dot);
      }
    }
  }
  __syncthreads();
  {  // S <- gamma S + Vd^T K: thread owns column c and rows i0 + RG j
    constexpr int RG = kChainThreads / D;
    constexpr int RJ = R / RG;
    const int c = t % D, i0 = t / D;
    float acc[RJ];
#pragma unroll
    for (int j = 0; j < RJ; ++j) acc[j] = __fmul_rn(gamma, Ss[(i0 + RG * j) * DP + c]);
    for (int s = 0; s < C; ++s) {
      const float kv = Ks[s * DP + c];
#pragma unroll
      for (int j = 0; j < RJ; ++j) acc[j] = __fmaf_rn(Vd[s * R + i0 + RG * j], kv, acc[j]);
    }
#pragma unroll
    for (int j = 0; j < RJ; ++j) Ss[(i0 + RG * j) * DP + c] = acc[j];
  }
  __syncthreads();
}

template <int D>
__device__ __forceinline__ void rows_to_global(const float* Ss, float* dst /* row r0 of a state */) {
  constexpr int DP = D + 4;
  for (int idx = threadIdx.x; idx < kRowsPerChain * (D / 4); idx += kChainThreads) {
    const int i = idx / (D / 4), c4 = idx % (D / 4);
    reinterpret_cast<float4*>(dst + i * D)[c4] = *reinterpret_cast<const float4*>(Ss + i * DP + 4 * c4);
  }
}

template <int D, typename Tin>
__global__ void __launch_bounds__(kChainThreads) k_chain(Dims dm, const void* keys_v,
                                                         const float* __restrict__ W,
                                                         const float* __restrict__ U,
                                                         const float* __restrict__ gamma,
                                                         ChainWork w, WsHeader* __restrict__ hdr) {
  constexpr int DP = D + 4;
  constexpr int R = kRowsPerChain;
  extern __shared__ __align__(16) float sm[];
  float* Ws = sm;
  float* Ks = Ws + kMaxChunk * DP;
  float* Ss = Ks + kMaxChunk * DP;
  float* Us = Ss + R * DP;
  float* Vd = Us + kMaxChunk * R;
  const int t = threadIdx.x;
  const int C = dm.C;
  const int n = blockIdx.x, h = blockIdx.y, r0 = blockIdx.z * R;
  const int hq = h / (dm.hv / dm.hqk);
  const Tin* keys = static_cast<const Tin*>(keys_v);
  const int64_t SZ = (int64_t)D * D;

  if (w.seqs) {  // ------------------------------------------------ prefill chain
    if (!hdr->valid) return;
    const SeqRec rec = w.seqs[n];
    const int nfull = rec.len / C;
    if (!in_bounds(hdr, rec.chunk0 >= 0 && (int64_t)rec.chunk0 + rec.nchunks <= w.n_chunks && rec.tok0 >= 0 &&
                            (int64_t)rec.tok0 + rec.len <= w.n_tokens))
      return;
    // S <- state_in rows (or 0)
    for (int idx = t; idx < R * (D / 4); idx += kChainThreads) {
      const int i = idx / (D / 4), c4 = idx % (D / 4);
      float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
      if (w.state_in)
        x = reinterpret_cast<const float4*>(w.state_in + ((int64_t)(w.state_in_slot ? w.state_in_slot[n] : n) * dm.hv + h) * SZ +
                                            (int64_t)(r0 + i) * D)[c4];
      *reinterpret_cast<float4*>(Ss + i * DP + 4 * c4) = x;
    }
    __syncthreads();
    for (int j = 0; j < nfull; ++j) {
      const int64_t c = (int64_t)rec.chunk0 + j;
      rows_to_global<D>(Ss, w.bnd + (c * dm.hv + h) * SZ + (int64_t)r0 * D);
      const int64_t wo = (c * dm.hv + h) * (int64_t)C * D;
      chain_step<D, Tin>(Ss, Ws, Ks, Us, Vd, W + (c * dm.hv + h) * (int64_t)prep_w_floats(C, D), U + wo, gamma[c * dm.hv + h], keys,
                         (int64_t)rec.tok0 + (int64_t)j * C, dm.hqk, hq, C, r0);
    }
    if (rec.len % C != 0) {
      const int64_t c = (int64_t)rec.chunk0 + nfull;  // start state of the partial chunk
      rows_to_global<D>(Ss, w.bnd + (c * dm.hv + h) * SZ + (int64_t)r0 * D);
    } else if (w.state_out) {
      rows_to_global<D>(Ss, w.state_out + ((int64_t)n * dm.hv + h) * SZ + (int64_t)r0 * D);
    }
    if (w.cache_bnd) {
      const int sl = w.slot_of_seq ? w.slot_of_seq[n] : n;
      if (sl < 0 || sl >= w.cache_slots) {
        if (t == 0) set_error(hdr, GDN_DEVERR_SLOT);
        return;
      }
      rows_to_global<D>(Ss, w.cache_bnd + ((int64_t)sl * dm.hv + h) * SZ + (int64_t)r0 * D);
      if (rec.len % C == 0) {  // an explicit running state: scale 1
        rows_to_global<D>(Ss, w.cache_run + ((int64_t)sl * dm.hv + h) * SZ + (int64_t)r0 * D);
        if (t == 0 && blockIdx.z == 0) w.cache_c_run[(int64_t)sl * dm.hv + h] = 1.f;
      }
    }
  } else {  // ---------------------------------------------------- decode resync
    const int sl = w.slot[n];
    if (sl < 0 || sl >= w.slots) return;  // reported by k_decode
    const int p = w.pos[sl];
    if (p < 0 || (p + 1) % C != 0) return;
    if (!in_bounds(hdr, ((int64_t)sl + 1) * C <= w.n_tokens && n < w.n_chunks)) return;
    const int64_t so = ((int64_t)sl * dm.hv + h) * SZ + (int64_t)r0 * D;
    for (int idx = t; idx < R * (D / 4); idx += kChainThreads) {
      const int i = idx / (D / 4), c4 = idx % (D / 4);
      *reinterpret_cast<float4*>(Ss + i * DP + 4 * c4) = reinterpret_cast<const float4*>(w.s_bnd + so + (int64_t)i * D)[c4];
    }
    __syncthreads();
    const int64_t wo = ((int64_t)n * dm.hv + h) * (int64_t)C * D;
    chain_step<D, Tin>(Ss, Ws, Ks, Us, Vd, W + ((int64_t)n * dm.hv + h) * (int64_t)prep_w_floats(C, D),
                       U + wo, gamma[(int64_t)n * dm.hv + h], keys,
                       (int64_t)sl * C, dm.hqk, hq, C, r0);
    rows_to_global<D>(Ss, w.s_bnd + so);
    rows_to_global<D>(Ss, w.s_run + so);
    if (t == 0 && blockIdx.z == 0) w.c_run[(int64_t)sl * dm.hv + h] = 1.f;  // explicit: scale 1
  }
}

template <int D, typename Tin>
static void launch_chain_t(const Dims& d, const void* keys, const float* W, const float* U,
                           const float* gamma, const ChainWork& w, WsHeader* hdr, cudaStream_t st) {
  constexpr size_t smem = chain_smem_bytes<D>();
  ensure_smem(k_chain<D, Tin>, smem);
  dim3 grid((unsigned)w.N, d.hv, D / kRowsPerChain);
  k_chain<D, Tin><<<grid, kChainThreads, smem, st>>>(d, keys, W, U, gamma, w, hdr);
}

// ============================================================  K1b (tcgen05)  ===
// Boundary chain on tensor cores for d = 128, C = 64, bf16 inputs.  One CTA of 256 threads
// per (sequence, head): state row i is TMEM lane i, read by the two warps of its lane
// quadrant, one half of the columns each.  The state
// S^(j) lives in TMEM (fp32) between steps; each step is
//     D1 (128 x 64)  = S Wd^T                        3 MMAs: S_hi Wd_hi + S_hi Wd_lo + S_lo Wd_hi
//     Vd^T[i][s]     = Ud[s][i] - D1[i][s]           (registers; then split to bf16 hi/lo)
//     D2 (128 x 128) = gamma S + Vd^T K               D2 preloaded with gamma S, 2 MMAs: Vd_hi K + Vd_lo K
// with fp32 operands split as x = hi + lo (bf16 each) and bf16 inputs exact.  The pre-pass
// wrote Wd hi/lo and the K rows as ready-made shared-memory images (K^T is the MN-major
// reading of the K rows), so a step's operands arrive by one bulk copy, issued a step ahead
// into the other of two stage buffers.
namespace tcc {
constexpr int D = 128, C = 64;
constexpr uint32_t A1_BYTES = 128 * D * 2;  // state operand, per hi / lo
constexpr uint32_t A2_BYTES = 128 * C * 2;  // Vd^T operand, per hi / lo
constexpr uint32_t STAGE_BYTES = 3 * C * D * 2;  // Wd hi | Wd lo | K rows
constexpr size_t SMEM = 2 * (size_t)A1_BYTES + 2 * (size_t)A2_BYTES + 2 * (size_t)STAGE_BYTES + 64;
constexpr uint32_t TMEM_COLS = 256, D1_COL = 0, D2_COL = 64;
constexpr uint32_t IDESC1 = tc::idesc_bf16(128, C);
constexpr uint32_t IDESC2 = tc::idesc_bf16(128, D);
}  // namespace tcc

// split 16 fp32 values of row `row` (columns k0..k0+15) into the hi/lo K-major images
__device__ __forceinline__ void store_split16(unsigned char* hi, unsigned char* lo, int row, int k0, int K,
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

__device__ __forceinline__ void store_row16(float* dst, const float* v) {
#pragma unroll
  for (int e = 0; e < 16; e += 4) *reinterpret_cast<float4*>(dst + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
}

__global__ void __launch_bounds__(256, 1) k_chain_tc(Dims dm, const float* __restrict__ Wimg,
                                                     const float* __restrict__ U,
                                                     const float* __restrict__ gamma, ChainWork w,
                                                     WsHeader* __restrict__ hdr) {
  using namespace tcc;
  using namespace tc;
  extern __shared__ __align__(128) unsigned char smc[];
  unsigned char* A1h = smc;
  unsigned char* A1l = A1h + A1_BYTES;
  unsigned char* A2h = A1l + A1_BYTES;
  unsigned char* A2l = A2h + A2_BYTES;
  unsigned char* stage0 = A2l + A2_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(stage0 + 2 * STAGE_BYTES);  // load0, load1, mma
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 3);
  // warp w reads TMEM lanes 32 (w % 4) .. + 31 (state rows) and column half w / 4
  const int t = threadIdx.x, warp = t >> 5, row = (warp & 3) * 32 + (t & 31), half = warp >> 2;
  const int cs0 = half * (D / 2), us0 = half * (C / 2);  // first state column / first Ud column
  const int64_t SZ = (int64_t)D * D;
  const int64_t WS = (int64_t)prep_w_floats(C, D);
  if (w.seqs && !hdr->valid) return;
  const int64_t total = (int64_t)w.N * dm.hv;
  // This CTA's items (wi = blockIdx.x + j * gridDim.x) that have work, tested one per
  // thread; a CTA with none exits before touching tensor memory.
  __shared__ int64_t s_list[128];
  __shared__ int s_cnt;
  // Prefill: the CTAs (launched in order) take the (sequence, head) chains longest first, so
  // that the longest chains do not start last; sequences ranked by chunk count, ties by index
  // (up to kRankSeqs sequences, each CTA ranking them; beyond that, in sequence order).
  __shared__ int s_nch[kRankSeqs], s_order[kRankSeqs];
  const bool by_length = w.seqs && w.N <= kRankSeqs;
  if (by_length && t < w.N) s_nch[t] = w.seqs[t].nchunks;
  if (t == 0) s_cnt = 0;
  __syncthreads();
  if (by_length && t < w.N) {
    const int mine = s_nch[t];
    int r = 0;
    for (int s2 = 0; s2 < w.N; ++s2) r += (s_nch[s2] > mine || (s_nch[s2] == mine && s2 < t)) ? 1 : 0;
    s_order[r] = t;
  }
  __syncthreads();
  if (t < 128) {
    const int64_t wc = blockIdx.x + (int64_t)t * gridDim.x;
    const int64_t wi = (by_length && wc < total) ? (int64_t)s_order[wc / dm.hv] * dm.hv + wc % dm.hv : wc;
    if (wc < total) {
      bool work = true;
      if (!w.seqs) {
        const int sl = w.slot[wi / dm.hv];
        work = sl >= 0 && sl < w.slots && w.pos[sl] >= 0 && (w.pos[sl] + 1) % C == 0;
      } else if (w.bnd_in_place && w.bnd_skip) {  // continued prefill: see the item loop
        const int n2 = (int)(wi / dm.hv);
        const int len2 = w.seqs[n2].len;
        work = !(len2 < C && w.bnd_skip[n2] > 0);
      }
      if (work) s_list[atomicAdd(&s_cnt, 1)] = wi;
    }
  }
  __syncthreads();
  const int count = s_cnt;
  if (count == 0) return;

  // tensor memory and barriers, once per CTA
  if (t == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    mbar_init(&bars[2], 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tslot, TMEM_COLS);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tbase = *tslot;
  const uint32_t tlane = tmem_lane_addr(tbase, warp, 0);
  uint32_t uses[2] = {0u, 0u};  // completed waits per stage barrier
  uint32_t mma_phase = 0;
  uint32_t gstep = 0;           // steps run by this CTA (selects the stage buffer)
  int pending = -1;             // stage buffer with a copy in flight
  bool mma_pending = false;
  bool ok = true;
  if (w.fault_wait && blockIdx.x == 0)  // test hook: phase 0 of bars[0] never completes here
    ok = __syncthreads_and(t == 0 ? mbar_wait(&bars[0], 0u, 1024u) : true) != 0;

  for (int li = 0; li < count && ok; ++li) {
    const int64_t wi = s_list[li];
    const int n = (int)(wi / dm.hv), h = (int)(wi % dm.hv);
    // ---- the work of this item (uniform)
    int nfull, nchunks = 0, len = 0, sl = -1;
    int64_t item0;
    const float* src;  // S^(0) rows, or NULL for zero
    if (w.seqs) {
      const SeqRec rec = w.seqs[n];
      nfull = rec.len / C;
      nchunks = rec.nchunks;
      len = rec.len;
      item0 = rec.chunk0;
      if (!in_bounds(hdr, rec.chunk0 >= 0 && (int64_t)rec.chunk0 + rec.nchunks <= w.n_chunks)) continue;
      src = w.state_in ? w.state_in + ((int64_t)(w.state_in_slot ? w.state_in_slot[n] : n) * dm.hv + h) * SZ
                       : nullptr;
      if (w.cache_bnd) {
        sl = w.slot_of_seq ? w.slot_of_seq[n] : n;
        if (sl < 0 || sl >= w.cache_slots) {
          if (t == 0) set_error(hdr, GDN_DEVERR_SLOT);
          sl = -1;
        }
      }
    } else {
      sl = w.slot[n];
      if (sl < 0 || sl >= w.slots) continue;  // reported by the decode step kernel
      const int p = w.pos[sl];
      if (p < 0 || (p + 1) % C != 0) continue;
      if (!in_bounds(hdr, n < w.n_chunks)) continue;
      nfull = 1;
      item0 = n;
      src = w.s_bnd + ((int64_t)sl * dm.hv + h) * SZ;
    }
    // continued prefill: S^(0) already in place in the cache, and not needed in bnd when
    // the first chunk starts from the running state
    const bool skip0 = w.seqs && w.bnd_skip && w.bnd_skip[n] > 0;
    if (w.seqs && nfull == 0 && skip0 && w.bnd_in_place && len % C != 0) continue;  // nothing to write
    // a running state written below is explicit: its scale is 1
    if (t == 0) {
      if (!w.seqs)
        w.c_run[(int64_t)sl * dm.hv + h] = 1.f;
      else if (sl >= 0 && len % C == 0)
        w.cache_c_run[(int64_t)sl * dm.hv + h] = 1.f;
    }
    // outputs for the state after full chunk j (j = 0 .. nfull): rows of S^(j)
    auto write_state = [&](int j, const float* v, int c0) {
      if (w.seqs) {
        if (j < nchunks && !(j == 0 && skip0))
          store_row16(w.bnd + ((item0 + j) * dm.hv + h) * SZ + (int64_t)row * D + c0, v);
        if (j == nfull) {
          if (len % C == 0 && w.state_out)
            store_row16(w.state_out + ((int64_t)n * dm.hv + h) * SZ + (int64_t)row * D + c0, v);
          if (sl >= 0) {
            if (!(j == 0 && w.bnd_in_place))
              store_row16(w.cache_bnd + ((int64_t)sl * dm.hv + h) * SZ + (int64_t)row * D + c0, v);
            if (len % C == 0)
              store_row16(w.cache_run + ((int64_t)sl * dm.hv + h) * SZ + (int64_t)row * D + c0, v);
          }
        }
      } else if (j > 0) {
        store_row16(w.s_bnd + ((int64_t)sl * dm.hv + h) * SZ + (int64_t)row * D + c0, v);
        store_row16(w.s_run + ((int64_t)sl * dm.hv + h) * SZ + (int64_t)row * D + c0, v);
      }
    };
    // the same outputs for one float4 of state row r2, columns c2 .. c2 + 3
    auto write_state4 = [&](int j, int r2, int c2, float4 x) {
      const int64_t o = (int64_t)r2 * D + c2;
      auto put = [&](float* base) { *reinterpret_cast<float4*>(base + o) = x; };
      if (w.seqs) {
        if (j < nchunks && !(j == 0 && skip0)) put(w.bnd + ((item0 + j) * dm.hv + h) * SZ);
        if (j == nfull) {
          if (len % C == 0 && w.state_out) put(w.state_out + ((int64_t)n * dm.hv + h) * SZ);
          if (sl >= 0) {
            if (!(j == 0 && w.bnd_in_place)) put(w.cache_bnd + ((int64_t)sl * dm.hv + h) * SZ);
            if (len % C == 0) put(w.cache_run + ((int64_t)sl * dm.hv + h) * SZ);
          }
        }
      } else if (j > 0) {
        put(w.s_bnd + ((int64_t)sl * dm.hv + h) * SZ);
        put(w.s_run + ((int64_t)sl * dm.hv + h) * SZ);
      }
    };
    // this thread's half row of S^(0), all loads in flight at once
    float4 s0v[D / 8];
#pragma unroll
    for (int x = 0; x < D / 8; ++x)
      s0v[x] = src ? *reinterpret_cast<const float4*>(src + (int64_t)row * D + cs0 + 4 * x)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
    auto s0_cols = [&](int g, float* v) {  // columns cs0 + 16 g .. + 15
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        v[4 * x] = s0v[4 * g + x].x;
        v[4 * x + 1] = s0v[4 * g + x].y;
        v[4 * x + 2] = s0v[4 * g + x].z;
        v[4 * x + 3] = s0v[4 * g + x].w;
      }
    };
    if (nfull == 0) {  // no full chunk: S^(0) passes straight to the outputs
#pragma unroll
      for (int g = 0; g < D / 32; ++g) {
        float v[16];
        s0_cols(g, v);
        write_state(0, v, cs0 + 16 * g);
      }
      continue;
    }
    if (t == 0) {
      const int b = (int)(gstep & 1u);
      mbar_expect_tx(&bars[b], STAGE_BYTES);
      bulk_g2s(stage0 + b * STAGE_BYTES, Wimg + (item0 * dm.hv + h) * WS, STAGE_BYTES, &bars[b]);
    }
    pending = (int)(gstep & 1u);
    {  // S^(0): outputs, A operand (split) and gamma_0 S^(0) into D2
      const float g0 = gamma[item0 * dm.hv + h];
#pragma unroll
      for (int g = 0; g < D / 32; ++g) {
        const int c0 = cs0 + 16 * g;
        float v[16];
        s0_cols(g, v);
        write_state(0, v, c0);
        store_split16(A1h, A1l, row, c0, D, v);
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = __fmul_rn(g0, v[e]);
        tmem_st16(tlane + D2_COL + c0, v);
      }
      tmem_st_wait();
    }
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();

    for (int j = 0; j < nfull; ++j, ++gstep) {
      const int64_t item = item0 + j;
      const int buf = (int)(gstep & 1u);
      unsigned char* stg = stage0 + buf * STAGE_BYTES;
      if (j + 1 < nfull) {
        if (t == 0) {
          mbar_expect_tx(&bars[buf ^ 1], STAGE_BYTES);
          bulk_g2s(stage0 + (buf ^ 1) * STAGE_BYTES, Wimg + ((item + 1) * dm.hv + h) * WS, STAGE_BYTES,
                   &bars[buf ^ 1]);
        }
      }
      float ud[C / 2];
      {
        const float* Ug = U + (item * dm.hv + h) * (int64_t)C * D + (int64_t)us0 * D + row;
#pragma unroll
        for (int s = 0; s < C / 2; ++s) ud[s] = Ug[(int64_t)s * D];
      }
      ok = __syncthreads_and(mbar_wait(&bars[buf], uses[buf] & 1u)) != 0;
      if (!ok) break;
      ++uses[buf];
      pending = (j + 1 < nfull) ? (buf ^ 1) : -1;
      if (t == 0) {  // D1 = S Wd^T (three split terms)
        fence_after_sync();
        const uint32_t a_hi = smem_u32(A1h), a_lo = smem_u32(A1l);
        const uint32_t w_hi = smem_u32(stg), w_lo = w_hi + C * D * 2;
        const uint32_t sbo = (D / 8) * 128;
#pragma unroll 1
        for (int term = 0; term < 3; ++term) {
          const uint32_t a = term == 2 ? a_lo : a_hi;
          const uint32_t b = term == 1 ? w_lo : w_hi;
          for (int kk = 0; kk < D / 16; ++kk)
            mma_bf16(tbase + D1_COL, make_desc(a + kk * 256, 128, sbo), make_desc(b + kk * 256, 128, sbo), IDESC1,
                     (term > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&bars[2]);
      }
      mma_pending = true;
      ok = __syncthreads_and(mbar_wait(&bars[2], mma_phase)) != 0;
      if (!ok) break;
      mma_phase ^= 1u;
      mma_pending = false;
      fence_after_sync();
      float d1[C / 2];  // this thread's half of its D1 row, one load
      tmem_ld32(tlane + D1_COL + us0, d1);
#pragma unroll
      for (int s1 = 0; s1 < C / 2; s1 += 16) {  // Vd^T row = Ud column - D1 row, split into A2
        float* v = d1 + s1;
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = __fsub_rn(ud[s1 + e], v[e]);
        store_split16(A2h, A2l, row, us0 + s1, C, v);
      }
      fence_proxy_async();
      fence_before_sync();
      __syncthreads();
      if (t == 0) {  // D2 += Vd^T K (two split terms; K^T the MN-major reading of the K rows image)
        fence_after_sync();
        const uint32_t k_img = smem_u32(stg) + 2 * C * D * 2;
        const Opnd vd = opnd_k(smem_u32(A2h), smem_u32(A2l), C), kr = opnd_mn(k_img, 0u, D);
        mma_part(tbase + D2_COL, vd, false, kr, false, C, IDESC2 | IDESC_B_MN, true);
        mma_part(tbase + D2_COL, vd, true, kr, false, C, IDESC2 | IDESC_B_MN, true);
        mma_commit(&bars[2]);
      }
      mma_pending = true;
      ok = __syncthreads_and(mbar_wait(&bars[2], mma_phase)) != 0;
      if (!ok) break;
      mma_phase ^= 1u;
      mma_pending = false;
      fence_after_sync();
      {  // S^(j+1): outputs, next step's A operand and gamma_{j+1} S^(j+1)
        const bool more = j + 1 < nfull;
        const float gn = more ? gamma[(item + 1) * dm.hv + h] : 0.f;
        // S^(j+1) leaves through a per-warp staging tile in the (now free) Vd^T operand
        // region, so that each store instruction writes 8 rows x 64 contiguous bytes
        float* tile = reinterpret_cast<float*>(A2h) + warp * (32 * 20);
        const int lane = t & 31, rq = (warp & 3) * 32;
        float s1v[D / 2];  // this thread's half of its state row, one load
        tmem_ld64(tlane + D2_COL + cs0, s1v);
#pragma unroll
        for (int c0 = cs0; c0 < cs0 + D / 2; c0 += 16) {
          float* v = s1v + (c0 - cs0);
#pragma unroll
          for (int x = 0; x < 4; ++x)
            *reinterpret_cast<float4*>(tile + lane * 20 + 4 * x) = make_float4(v[4 * x], v[4 * x + 1], v[4 * x + 2], v[4 * x + 3]);
          __syncwarp();
#pragma unroll
          for (int k2 = 0; k2 < 4; ++k2) {
            const int rl = 8 * k2 + (lane >> 2), f = lane & 3;
            write_state4(j + 1, rq + rl, c0 + 4 * f, *reinterpret_cast<const float4*>(tile + rl * 20 + 4 * f));
          }
          __syncwarp();
          if (more) {
            store_split16(A1h, A1l, row, c0, D, v);
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = __fmul_rn(gn, v[e]);
            tmem_st16(tlane + D2_COL + c0, v);
          }
        }
        tmem_st_wait();
      }
      fence_proxy_async();
      fence_before_sync();
      __syncthreads();
    }
  }
  if (!ok && t == 0) {
    set_error(hdr, GDN_DEVERR_TIMEOUT);
    // let the operations this CTA may still have in flight finish before releasing TMEM
    if (pending >= 0) mbar_wait(&bars[pending], uses[pending] & 1u);
    if (mma_pending) mbar_wait(&bars[2], mma_phase);
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, TMEM_COLS);
}

// ============================================================  K1a (tcgen05)  ===
// Boundary pre-pass on tensor cores for d = 128, C = 64, bf16 inputs, one CTA of 256
// threads per (chunk, head) as k_prep:
//   Gram = K K^T                        1 MMA chain (bf16 inputs exact, fp32 accumulation)
//   A, T = (I + A)^{-1}                 fp32 SIMT (blocked forward substitution)
//   W    = (T diag(beta e^G)) K         A = TK split hi/lo, B = K^T (MN-major reading of the K rows)
//   U^T  = V^T (T diag(beta))^T         A = V^T (MN-major reading of the V rows), B = TV split hi/lo
// Outputs as k_prep's tensor-core variant: the chain's images [Wd hi | Wd lo | K rows]
// (Wd = diag(dec) W; the K rows image leaves by bulk copy as soon as it lands) and
// Ud = diag(dec) U in fp32, plus gamma.  Gram and W use 128-row MMAs
// of which rows 0..63 are the chunk (the other rows read neighbouring shared memory and
// are never read back).
namespace tcp {
constexpr int D = 128, C = 64, CP = C + 1;
constexpr uint32_t TILE = C * D * 2;                   // 16 KB: a C x D or D x C bf16 image
constexpr uint32_t MAT = C * CP * 4;                   // fp32 C x C with padded rows
constexpr size_t SMEM = 3 * (size_t)TILE + 2 * (size_t)MAT + 5 * C * 4 + 64;
constexpr uint32_t TMEM_COLS = 256, W_COL = 0, UT_COL = 128, GRAM_COL = 0;
}  // namespace tcp

constexpr int kPrepMaxItems = 1024;  // items one k_prep_tc CTA can hold (the launch sizes the grid)

__global__ void __launch_bounds__(256, 2) k_prep_tc(Dims dm, TokenArrays in, PrepWork w,
                                                    float* __restrict__ Wout, float* __restrict__ Uout,
                                                    float* __restrict__ gamma_out, WsHeader* __restrict__ hdr) {
  using namespace tcp;
  extern __shared__ __align__(128) unsigned char smp[];
  unsigned char* R0 = smp;             // K rows image (C x D); W's B operand K^T is its MN-major reading
  unsigned char* KT = R0 + TILE;       // Xs, then TK hi | TK lo (C x C each)
  unsigned char* VT = KT + TILE;       // V rows image (C x D); U^T's A operand V^T is its MN-major reading
  float* A = reinterpret_cast<float*>(VT + TILE);  // then TV hi | TV lo images
  float* Tm = A + C * CP;
  float* gs = Tm + C * CP;
  float* Gs = gs + C;
  float* bs = Gs + C;
  float* bk = bs + C;
  float* dec = bk + C;
  uint64_t* bar = reinterpret_cast<uint64_t*>(dec + C);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 1);
  float* Xs = reinterpret_cast<float*>(KT);
  unsigned char* TKh = KT;
  unsigned char* TKl = KT + C * C * 2;
  unsigned char* TVh = reinterpret_cast<unsigned char*>(A);
  unsigned char* TVl = TVh + C * C * 2;
  const int t = threadIdx.x, warp = t >> 5;
  if (w.chunks && !hdr->valid) return;
  const int64_t total = w.n_items * dm.hv;
  // Which of this CTA's items (wi = blockIdx.x + j * gridDim.x) need the pre-pass: all
  // tested at once, one per thread; a CTA with none exits before touching tensor memory.
  __shared__ int64_t s_list[kPrepMaxItems];
  __shared__ int64_t s_tok0[kPrepMaxItems];
  __shared__ int s_cnt;
  if (t == 0) s_cnt = 0;
  __syncthreads();
  for (int cand = t; cand < kPrepMaxItems; cand += 256) {
    const int64_t wi = blockIdx.x + (int64_t)cand * gridDim.x;
    if (wi < total) {
      const int64_t item = wi / dm.hv;
      const int h = (int)(wi % dm.hv);
      int64_t tok0 = -1;
      if (w.chunks) {
        const ChunkRec rec = w.chunks[item];
        if (rec.len == C) tok0 = rec.tok0;
      } else {
        const int sl = w.slot[item];
        if (sl < 0 || sl >= w.slots) {
          if (h == 0) set_error(hdr, GDN_DEVERR_SLOT);
        } else {
          const int p = w.pos[sl];
          if (p < 0) {
            if (h == 0) set_error(hdr, GDN_DEVERR_POS);
          } else if ((p + 1) % C == 0) {
            tok0 = (int64_t)sl * C;
          }
        }
      }
      if (tok0 >= 0 && !in_bounds(hdr, tok0 + C <= in.n_tokens)) tok0 = -1;
      if (tok0 >= 0) {
        const int k = atomicAdd(&s_cnt, 1);
        s_list[k] = wi;
        s_tok0[k] = tok0;
      }
    }
  }
  __syncthreads();
  const int count = s_cnt;
  if (count == 0) return;

  // tensor memory and the MMA barrier, once per CTA
  if (t == 0) {
    tc::mbar_init(bar, 1);
    tc::fence_mbar_init();
  }
  if (warp == 0) tc::tmem_alloc(tslot, TMEM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = *tslot;
  uint32_t phase = 0;
  bool ok = true;
  const __nv_bfloat16* kin = static_cast<const __nv_bfloat16*>(in.k);
  const __nv_bfloat16* vin = static_cast<const __nv_bfloat16*>(in.v);
  const int64_t kstride = (int64_t)dm.hqk * D, vstride = (int64_t)dm.hv * D;

  // Item lj's K rows (as the image in R0), V rows (staged in the A region), g and beta by
  // asynchronous copies, 16 bytes a piece; item 0's before the loop, every later one's as
  // soon as the previous item's W and U^T products have consumed those regions, so that
  // they land while that item writes its outputs.
  auto load_item = [&](int lj) {
    const int64_t wj = s_list[lj];
    const int hj = (int)(wj % dm.hv), hqj = hj / (dm.hv / dm.hqk);
    const int64_t tj = s_tok0[lj];
    const __nv_bfloat16* kbj = kin + tj * kstride + (int64_t)hqj * D;
    const __nv_bfloat16* vbj = vin + tj * vstride + (int64_t)hj * D;
#pragma unroll
    for (int it = 0; it < 4; ++it) {  // C * D / 8 = 1024 pieces of 16 bytes
      int r, c0;
      tc::kmajor_piece(t + it * 256, D, r, c0);
      tc::cp_async16(R0 + tc::kmajor_off(r, c0, D), kbj + r * kstride + c0);
      tc::cp_async16(VT + tc::kmajor_off(r, c0, D), vbj + r * vstride + c0);
    }
    if (t < C) {
      tc::cp_async4(gs + t, in.g + (tj + t) * dm.hv + hj);
      tc::cp_async4(bs + t, in.beta + (tj + t) * dm.hv + hj);
    }
    tc::cp_async_commit();
  };
  load_item(0);

  for (int li = 0; li < count && ok; ++li) {
    const int64_t wi = s_list[li];
    const int64_t item = wi / dm.hv;
    const int h = (int)(wi % dm.hv);

    // 1. this item's K, V, g and beta in shared memory; the K rows image leaves at once for
    // the chain (its K^T operand is the MN-major reading of this image)
    float* Wo = Wout + (item * dm.hv + h) * (int64_t)prep_w_floats(C, D);
    unsigned char* img = reinterpret_cast<unsigned char*>(Wo);
    tc::cp_async_wait_all();
    tc::fence_proxy_async();
    tc::fence_before_sync();
    __syncthreads();
    if (t == 0) {
      tc::bulk_s2g(img + 2 * TILE, R0, TILE);
      tc::bulk_store_commit();
    }
    // 2. Gram on the tensor cores while one thread forms G
    if (t == 0) {
      tc::fence_after_sync();
      const uint32_t a = tc::smem_u32(R0);
      for (int kk = 0; kk < D / 16; ++kk)
        tc::mma_bf16(tbase + GRAM_COL, tc::make_desc(a + kk * 256, 128, (D / 8) * 128),
                     tc::make_desc(a + kk * 256, 128, (D / 8) * 128), tc::idesc_bf16(128, C), kk > 0 ? 1u : 0u);
      tc::mma_commit(bar);
      float run = gs[0];
      Gs[0] = run;
#pragma unroll
      for (int i = 1; i < C; ++i) {
        run = __fadd_rn(run, gs[i]);
        Gs[i] = run;
      }
    }
    __syncthreads();
    if (t < C) {
      bk[t] = __fmul_rn(bs[t], expf(Gs[t]));
      dec[t] = expf(__fsub_rn(Gs[C - 1], Gs[t]));
    }
    // beta_i e^{G_i - G_s} (i > s) into A while the Gram product runs, by all threads; the
    // readout multiplies in place
    tc::decay_matrix64(A, CP, bs, Gs);
    {
      const bool done = tc::mbar_wait(bar, phase);
      ok = __syncthreads_and(done) != 0;
      if (!ok) break;
      phase ^= 1u;
    }
    tc::fence_after_sync();
    if ((warp & 3) < 2) {  // rows 0..63: A_is = beta_i e^{G_i - G_s} Gram_is (i > s)
      const int i = (warp & 3) * 32 + (t & 31);
      const int cbase = (warp >> 2) * 32;
      for (int s0 = cbase; s0 < cbase + 32; s0 += 16) {
        float v[16];
        tc::tmem_ld16(tc::tmem_lane_addr(tbase, warp, GRAM_COL + s0), v);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int s = s0 + e;
          A[i * CP + s] = (i > s) ? __fmul_rn(A[i * CP + s], v[e]) : 0.f;
        }
      }
    }
    tc::fence_before_sync();
    __syncthreads();
    // 3. T = (I + A)^{-1}
    unit_lower_inverse64(A, CP, Tm, CP, Xs);
    // 4. TK = T diag(beta e^G), TV = T diag(beta), split into bf16 images (lower triangle)
    for (int q = t; q < C * (C / 8); q += 256) {
      int i, r0;
      tc::kmajor_piece(q, C, i, r0);
      float tk[8], tv[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int r = r0 + e;
        const float x = (r <= i) ? Tm[i * CP + r] : 0.f;
        tk[e] = __fmul_rn(x, bk[r]);
        tv[e] = __fmul_rn(x, bs[r]);
      }
      uint32_t a[4], b[4], c2[4], d2[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        __nv_bfloat16 h0, l0, h1, l1;
        tc::split_bf16(tk[2 * e], h0, l0);
        tc::split_bf16(tk[2 * e + 1], h1, l1);
        a[e] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
        b[e] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
        tc::split_bf16(tv[2 * e], h0, l0);
        tc::split_bf16(tv[2 * e + 1], h1, l1);
        c2[e] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
        d2[e] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
      }
      const uint32_t off = tc::kmajor_off(i, r0, C);
      *reinterpret_cast<uint4*>(TKh + off) = make_uint4(a[0], a[1], a[2], a[3]);
      *reinterpret_cast<uint4*>(TKl + off) = make_uint4(b[0], b[1], b[2], b[3]);
      *reinterpret_cast<uint4*>(TVh + off) = make_uint4(c2[0], c2[1], c2[2], c2[3]);
      *reinterpret_cast<uint4*>(TVl + off) = make_uint4(d2[0], d2[1], d2[2], d2[3]);
    }
    tc::fence_proxy_async();
    tc::fence_before_sync();
    __syncthreads();
    // 5. W = TK K (rows 0..63 of a 128-row MMA) and U^T = V^T TV^T
    if (t == 0) {
      tc::fence_after_sync();
      const tc::Opnd tk = tc::opnd_k(tc::smem_u32(TKh), tc::smem_u32(TKl), C);
      const tc::Opnd tv = tc::opnd_k(tc::smem_u32(TVh), tc::smem_u32(TVl), C);
      const tc::Opnd kt = tc::opnd_mn(tc::smem_u32(R0), 0u, D), vt = tc::opnd_mn(tc::smem_u32(VT), 0u, D);
      const uint32_t iw = tc::idesc_bf16(128, D) | tc::IDESC_B_MN, iu = tc::idesc_bf16(128, C) | tc::IDESC_A_MN;
      tc::mma_part(tbase + W_COL, tk, false, kt, false, C, iw, false);  // W = TK_hi K + TK_lo K
      tc::mma_part(tbase + UT_COL, vt, false, tv, false, C, iu, false);  // U^T = V^T (TV_hi + TV_lo)^T
      tc::mma_part(tbase + W_COL, tk, true, kt, false, C, iw, true);
      tc::mma_part(tbase + UT_COL, vt, false, tv, true, C, iu, true);
      tc::mma_commit(bar);
    }
    if (t == 0) tc::bulk_wait_read();  // the K rows image store has read R0 (the next item's lands there)
    {
      const bool done = tc::mbar_wait(bar, phase);
      ok = __syncthreads_and(done) != 0;
      if (!ok) break;
      phase ^= 1u;
    }
    tc::fence_after_sync();
    if (li + 1 < count) load_item(li + 1);  // R0, V rows, g and beta are free now
    float* Uo = Uout + ((item * dm.hv + h) * C) * (int64_t)D;
    if ((warp & 3) < 2) {  // Wd rows 0..63 -> split image
      const int i = (warp & 3) * 32 + (t & 31);
      const int cbase = (warp >> 2) * 64;
      for (int c0 = cbase; c0 < cbase + 64; c0 += 16) {
        float v[16];
        tc::tmem_ld16(tc::tmem_lane_addr(tbase, warp, W_COL + c0), v);
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = __fmul_rn(dec[i], v[e]);
#pragma unroll
        for (int g2 = 0; g2 < 2; ++g2) {
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            __nv_bfloat16 h0, l0, h1, l1;
            tc::split_bf16(v[8 * g2 + 2 * e], h0, l0);
            tc::split_bf16(v[8 * g2 + 2 * e + 1], h1, l1);
            hw[e] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
            lw[e] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
          }
          const uint32_t off = tc::kmajor_off(i, c0 + 8 * g2, D);
          *reinterpret_cast<uint4*>(img + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(img + TILE + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
      }
    }
    {  // Ud[i][e] = dec_i U^T[e][i]: lane e, columns i
      const int e = (warp & 3) * 32 + (t & 31);
      const int ibase = (warp >> 2) * 32;
      for (int i0 = ibase; i0 < ibase + 32; i0 += 16) {
        float v[16];
        tc::tmem_ld16(tc::tmem_lane_addr(tbase, warp, UT_COL + i0), v);
#pragma unroll
        for (int x = 0; x < 16; ++x) Uo[(int64_t)(i0 + x) * D + e] = __fmul_rn(dec[i0 + x], v[x]);
      }
    }
    if (t == 0) gamma_out[item * dm.hv + h] = expf(Gs[C - 1]);
    tc::fence_before_sync();
    __syncthreads();  // shared memory and tensor memory are reused by the next item
  }
  tc::cp_async_wait_all();  // no copy of this thread still in flight
  if (!ok && t == 0) {
    set_error(hdr, GDN_DEVERR_TIMEOUT);
    tc::mbar_wait(bar, phase);  // let the MMA in flight finish before releasing its memory
  }
  if (t == 0) tc::bulk_wait_all();  // the K rows image stores are complete
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tbase, TMEM_COLS);
}

// ====================================================  K1c decode resync, fused (tcgen05)  ===
// The decode resynchronisation in one kernel (d = 128, C = 64, bf16): for every (step token
// n, head) whose slot completes a chunk with this token, k_prep_tc's pre-pass on the slot's
// chunk tail followed by one step of k_chain_tc,
//     s_bnd <- gamma s_bnd + (Ud - Wd s_bnd^T)^T K,   s_run <- s_bnd,   c_run <- 1,
// with the pre-pass outputs kept on chip: the Wd hi / lo and K^T images stay in shared
// memory where the step reads them, Ud goes from the U^T readout straight into the
// registers of the thread that owns the state row, gamma is recomputed.  Every value is
// formed by the same operations in the same order as in those two kernels, which the
// prefill's boundary pass runs, so a resynchronised boundary state has the bits the prefill
// of the same tokens gives.  The CTAs are persistent, two per SM (shared memory: the state
// operand hi | lo, 64 KB, and the stage [Wd hi | Wd lo | K^T], 48 KB; the pre-pass's K / V
// images, A, T and vectors live in the state operand and the Wd images while those are
// still unwritten), and each prefetches its next item's operands into L2.
namespace tcf {
constexpr int D = 128, C = 64, CP = C + 1;
constexpr uint32_t TILE = C * D * 2;        // a C x D or D x C bf16 image
constexpr uint32_t MAT = C * CP * 4;        // fp32 C x C with padded rows
constexpr uint32_t A1_BYTES = 128 * D * 2;  // state operand, per hi / lo
constexpr uint32_t OFF_A1H = 0, OFF_A1L = A1_BYTES, OFF_STG = 2 * A1_BYTES, OFF_KT = OFF_STG + 2 * TILE;
constexpr uint32_t OFF_R0 = 0, OFF_VT = TILE, OFF_A = A1_BYTES, OFF_VEC = OFF_A + MAT, OFF_T = OFF_STG;
constexpr size_t SMEM = OFF_STG + 3 * (size_t)TILE + 64;
constexpr int MAX_ITEMS = 64;  // items per CTA (the launch sizes the grid for it)
constexpr uint32_t TMEM_COLS = 256, GRAM_COL = 0, W_COL = 0, UT_COL = 128, D1_COL = 0, D2_COL = 64;
static_assert(OFF_VEC + 5 * C * 4 <= OFF_A1L + A1_BYTES, "pre-pass vectors inside the lo state image");
static_assert(OFF_T + MAT <= OFF_KT, "T inside the Wd images");
}  // namespace tcf

__global__ void __launch_bounds__(256, 2) k_resync_fused_tc(Dims dm, TokenArrays in, PrepWork pw, ChainWork w,
                                                            WsHeader* __restrict__ hdr) {
  using namespace tcf;
  using namespace tc;
  extern __shared__ __align__(128) unsigned char smf[];
  unsigned char* A1h = smf + OFF_A1H;
  unsigned char* A1l = smf + OFF_A1L;
  unsigned char* stg = smf + OFF_STG;  // Wd hi | Wd lo | K^T
  unsigned char* KT = smf + OFF_KT;
  unsigned char* A2h = stg;         // Vd^T hi over Wd hi, after the first product
  unsigned char* A2l = stg + TILE;  // Vd^T lo over Wd lo
  unsigned char* R0 = smf + OFF_R0;  // K image, then Xs, then TK hi | lo
  unsigned char* VT = smf + OFF_VT;
  float* A = reinterpret_cast<float*>(smf + OFF_A);  // V rows, then A, then TV hi | lo
  float* Tm = reinterpret_cast<float*>(smf + OFF_T);
  float* gs = reinterpret_cast<float*>(smf + OFF_VEC);
  float* Gs = gs + C;
  float* bs = Gs + C;
  float* bk = bs + C;
  float* dec = bk + C;
  float* Xs = reinterpret_cast<float*>(R0);
  unsigned char* TKh = R0;
  unsigned char* TKl = R0 + C * C * 2;
  unsigned char* TVh = reinterpret_cast<unsigned char*>(A);
  unsigned char* TVl = TVh + C * C * 2;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smf + OFF_STG + 3 * TILE);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 1);
  // warp w reads TMEM lanes 32 (w % 4) .. + 31 (state rows) and column half w / 4
  const int t = threadIdx.x, warp = t >> 5, row = (warp & 3) * 32 + (t & 31), half = warp >> 2;
  const int cs0 = half * (D / 2), us0 = half * (C / 2);
  const int64_t SZ = (int64_t)D * D;
  const int64_t total = pw.n_items * dm.hv;
  // this CTA's items (wi = blockIdx.x + j * gridDim.x) whose slot resynchronises
  __shared__ int64_t s_list[MAX_ITEMS];
  __shared__ int s_cnt;
  if (t == 0) s_cnt = 0;
  __syncthreads();
  if (t < MAX_ITEMS) {
    const int64_t wi = blockIdx.x + (int64_t)t * gridDim.x;
    if (wi < total) {
      const int64_t n = wi / dm.hv;
      const int h = (int)(wi % dm.hv);
      const int sl = pw.slot[n];
      if (sl < 0 || sl >= pw.slots) {
        if (h == 0) set_error(hdr, GDN_DEVERR_SLOT);
      } else {
        const int p = pw.pos[sl];
        if (p < 0) {
          if (h == 0) set_error(hdr, GDN_DEVERR_POS);
        } else if ((p + 1) % C == 0 &&
                   in_bounds(hdr, (int64_t)sl * C + C <= in.n_tokens && n < w.n_chunks && sl < w.slots)) {
          s_list[atomicAdd(&s_cnt, 1)] = wi;
        }
      }
    }
  }
  __syncthreads();
  const int count = s_cnt;
  if (count == 0) return;

  // tensor memory and the MMA barrier, once per CTA
  if (t == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tslot, TMEM_COLS);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tbase = *tslot;
  const uint32_t tlane = tmem_lane_addr(tbase, warp, 0);
  uint32_t phase = 0;
  bool ok = true, pending = false;
  auto wait_mma = [&]() {
    const bool done = mbar_wait(bar, phase);
    ok = __syncthreads_and(done) != 0;
    if (ok) {
      phase ^= 1u;
      pending = false;
    }
  };
  const __nv_bfloat16* kin = static_cast<const __nv_bfloat16*>(in.k);
  const __nv_bfloat16* vin = static_cast<const __nv_bfloat16*>(in.v);
  const int64_t kstride = (int64_t)dm.hqk * D, vstride = (int64_t)dm.hv * D;

  // Item lj's K rows (as the image in R0), V rows (staged in the A region), g and beta of the
  // slot's chunk tail by asynchronous copies, 16 bytes a piece: item 0's before the loop,
  // every later one's as soon as the previous item's first boundary product has consumed
  // the state operand those regions lie in.  Its boundary state goes to L2 meanwhile.
  auto load_item = [&](int lj) {
    const int64_t wj = s_list[lj];
    const int64_t nj = wj / dm.hv;
    const int hj = (int)(wj % dm.hv), hqj = hj / (dm.hv / dm.hqk);
    const int64_t tj = (int64_t)pw.slot[nj] * C;
    const __nv_bfloat16* kbj = kin + tj * kstride + (int64_t)hqj * D;
    const __nv_bfloat16* vbj = vin + tj * vstride + (int64_t)hj * D;
#pragma unroll
    for (int it = 0; it < 4; ++it) {  // C * D / 8 = 1024 pieces of 16 bytes
      int r, c0;
      kmajor_piece(t + it * 256, D, r, c0);
      cp_async16(R0 + kmajor_off(r, c0, D), kbj + r * kstride + c0);
      cp_async16(reinterpret_cast<unsigned char*>(A) + kmajor_off(r, c0, D), vbj + r * vstride + c0);
    }
    if (t < C) {
      cp_async4(gs + t, in.g + (tj + t) * dm.hv + hj);
      cp_async4(bs + t, in.beta + (tj + t) * dm.hv + hj);
    }
    cp_async_commit();
    const float* sp = w.s_bnd + ((int64_t)pw.slot[nj] * dm.hv + hj) * SZ;
    for (int q = t; q < D * D / 32; q += 256) prefetch_l2(sp + 32 * q);
  };
  load_item(0);

  for (int li = 0; li < count && ok; ++li) {
    const int64_t wi = s_list[li];
    const int64_t n = wi / dm.hv;
    const int h = (int)(wi % dm.hv);
    const int sl = pw.slot[n];

    // ---- the pre-pass, k_prep_tc's steps
    // 1. this item's K, V, g and beta in shared memory
    cp_async_wait_all();
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    // 2. Gram on the tensor cores while one thread forms G
    if (t == 0) {
      fence_after_sync();
      const uint32_t a = smem_u32(R0);
      for (int kk = 0; kk < D / 16; ++kk)
        mma_bf16(tbase + GRAM_COL, make_desc(a + kk * 256, 128, (D / 8) * 128), make_desc(a + kk * 256, 128, (D / 8) * 128),
                 idesc_bf16(128, C), kk > 0 ? 1u : 0u);
      mma_commit(bar);
      float run = gs[0];
      Gs[0] = run;
#pragma unroll
      for (int i = 1; i < C; ++i) {
        run = __fadd_rn(run, gs[i]);
        Gs[i] = run;
      }
    }
    pending = true;
    // K^T and V^T images from the row images while the Gram product runs (it reads only R0)
    transpose_image(KT, R0, D, C);
    transpose_image(VT, reinterpret_cast<const unsigned char*>(A), D, C);
    __syncthreads();
    if (t < C) {
      bk[t] = __fmul_rn(bs[t], expf(Gs[t]));
      dec[t] = expf(__fsub_rn(Gs[C - 1], Gs[t]));
    }
    // beta_i e^{G_i - G_s} (i > s) into A while the Gram product runs; the readout multiplies
    tc::decay_matrix64(A, CP, bs, Gs);
    wait_mma();
    if (!ok) break;
    fence_after_sync();
    if ((warp & 3) < 2) {  // rows 0..63: A_is = beta_i e^{G_i - G_s} Gram_is (i > s)
      const int i = row;
      const int cbase = half * 32;
      for (int s0 = cbase; s0 < cbase + 32; s0 += 16) {
        float v[16];
        tmem_ld16(tlane + GRAM_COL + s0, v);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int s = s0 + e;
          A[i * CP + s] = (i > s) ? __fmul_rn(A[i * CP + s], v[e]) : 0.f;
        }
      }
    }
    fence_before_sync();
    __syncthreads();
    // 3. T = (I + A)^{-1}
    unit_lower_inverse64(A, CP, Tm, CP, Xs);
    // 4. TK = T diag(beta e^G), TV = T diag(beta), split into bf16 images (lower triangle)
    for (int q = t; q < C * (C / 8); q += 256) {
      int i, r0;
      kmajor_piece(q, C, i, r0);
      float tk[8], tv[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int r = r0 + e;
        const float x = (r <= i) ? Tm[i * CP + r] : 0.f;
        tk[e] = __fmul_rn(x, bk[r]);
        tv[e] = __fmul_rn(x, bs[r]);
      }
      uint32_t a[4], b[4], c2[4], d2[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        __nv_bfloat16 h0, l0, h1, l1;
        split_bf16(tk[2 * e], h0, l0);
        split_bf16(tk[2 * e + 1], h1, l1);
        a[e] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
        b[e] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
        split_bf16(tv[2 * e], h0, l0);
        split_bf16(tv[2 * e + 1], h1, l1);
        c2[e] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
        d2[e] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
      }
      const uint32_t off = kmajor_off(i, r0, C);
      *reinterpret_cast<uint4*>(TKh + off) = make_uint4(a[0], a[1], a[2], a[3]);
      *reinterpret_cast<uint4*>(TKl + off) = make_uint4(b[0], b[1], b[2], b[3]);
      *reinterpret_cast<uint4*>(TVh + off) = make_uint4(c2[0], c2[1], c2[2], c2[3]);
      *reinterpret_cast<uint4*>(TVl + off) = make_uint4(d2[0], d2[1], d2[2], d2[3]);
    }
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    // 5. W = TK K (rows 0..63 of a 128-row MMA) and U^T = V^T TV^T
    if (t == 0) {
      fence_after_sync();
      const uint32_t sbo = (C / 8) * 128;
      const uint32_t kt = smem_u32(KT), vt = smem_u32(VT);
      for (int term = 0; term < 2; ++term) {
        const uint32_t a = smem_u32(term == 0 ? TKh : TKl);
        const uint32_t b = smem_u32(term == 0 ? TVh : TVl);
        for (int kk = 0; kk < C / 16; ++kk) {
          mma_bf16(tbase + W_COL, make_desc(a + kk * 256, 128, sbo), make_desc(kt + kk * 256, 128, sbo),
                   idesc_bf16(128, D), (term > 0 || kk > 0) ? 1u : 0u);
          mma_bf16(tbase + UT_COL, make_desc(vt + kk * 256, 128, sbo), make_desc(b + kk * 256, 128, sbo),
                   idesc_bf16(128, C), (term > 0 || kk > 0) ? 1u : 0u);
        }
      }
      mma_commit(bar);
    }
    pending = true;
    wait_mma();
    if (!ok) break;
    fence_after_sync();
    // 6. Wd = diag(dec) W rows 0..63 -> the stage's split image; Ud column of this thread's
    // state row (Ud[s][row] = dec_s U^T[row][s]) -> registers; gamma
    if ((warp & 3) < 2) {
      const int i = row;
      const int cbase = half * 64;
      for (int c0 = cbase; c0 < cbase + 64; c0 += 16) {
        float v[16];
        tmem_ld16(tlane + W_COL + c0, v);
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = __fmul_rn(dec[i], v[e]);
        store_split16(stg, stg + TILE, i, c0, D, v);
      }
    }
    float ud[C / 2];
#pragma unroll
    for (int s1 = 0; s1 < C / 2; s1 += 16) {
      float v[16];
      tmem_ld16(tlane + UT_COL + us0 + s1, v);
#pragma unroll
      for (int x = 0; x < 16; ++x) ud[s1 + x] = __fmul_rn(dec[us0 + s1 + x], v[x]);
    }
    const float g0 = expf(Gs[C - 1]);
    fence_before_sync();
    __syncthreads();  // W, U^T and the vectors are read before the state overwrites them

    // ---- the boundary step (k_chain_tc's step on one chunk)
    const int64_t so = ((int64_t)sl * dm.hv + h) * SZ;
    if (t == 0) w.c_run[(int64_t)sl * dm.hv + h] = 1.f;  // the running state written below is explicit
    {  // S^(0): A operand (split) and gamma_0 S^(0) into D2, one 16-column slice at a time
      const float* src = w.s_bnd + so + (int64_t)row * D;
#pragma unroll 1
      for (int g = 0; g < D / 32; ++g) {
        const int c0 = cs0 + 16 * g;
        float v[16];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const float4 f = *reinterpret_cast<const float4*>(src + c0 + 4 * x);
          v[4 * x] = f.x; v[4 * x + 1] = f.y; v[4 * x + 2] = f.z; v[4 * x + 3] = f.w;
        }
        store_split16(A1h, A1l, row, c0, D, v);
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = __fmul_rn(g0, v[e]);
        tmem_st16(tlane + D2_COL + c0, v);
      }
      tmem_st_wait();
    }
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    if (t == 0) {  // D1 = S Wd^T (three split terms)
      fence_after_sync();
      const uint32_t a_hi = smem_u32(A1h), a_lo = smem_u32(A1l);
      const uint32_t w_hi = smem_u32(stg), w_lo = w_hi + TILE;
      const uint32_t sbo = (D / 8) * 128;
#pragma unroll 1
      for (int term = 0; term < 3; ++term) {
        const uint32_t a = term == 2 ? a_lo : a_hi;
        const uint32_t b = term == 1 ? w_lo : w_hi;
        for (int kk = 0; kk < D / 16; ++kk)
          mma_bf16(tbase + D1_COL, make_desc(a + kk * 256, 128, sbo), make_desc(b + kk * 256, 128, sbo),
                   idesc_bf16(128, C), (term > 0 || kk > 0) ? 1u : 0u);
      }
      mma_commit(bar);
    }
    pending = true;
    wait_mma();
    if (!ok) break;
    fence_after_sync();
    if (li + 1 < count) load_item(li + 1);  // the state operand is consumed
#pragma unroll
    for (int s1 = 0; s1 < C / 2; s1 += 16) {  // Vd^T row = Ud column - D1 row, split into A2
      float v[16];
      tmem_ld16(tlane + D1_COL + us0 + s1, v);
#pragma unroll
      for (int e = 0; e < 16; ++e) v[e] = __fsub_rn(ud[s1 + e], v[e]);
      store_split16(A2h, A2l, row, us0 + s1, C, v);
    }
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    if (t == 0) {  // D2 += Vd^T K (two split terms)
      fence_after_sync();
      const uint32_t k_img = smem_u32(KT);
      const uint32_t sbo = (C / 8) * 128;
#pragma unroll 1
      for (int term = 0; term < 2; ++term) {
        const uint32_t a = smem_u32(term == 0 ? A2h : A2l);
        for (int kk = 0; kk < C / 16; ++kk)
          mma_bf16(tbase + D2_COL, make_desc(a + kk * 256, 128, sbo), make_desc(k_img + kk * 256, 128, sbo),
                   idesc_bf16(128, D), 1u);
      }
      mma_commit(bar);
    }
    pending = true;
    wait_mma();
    if (!ok) break;
    fence_after_sync();
    {  // S^(1) -> s_bnd and s_run through a per-warp staging tile over the dead Vd^T operand,
       // so that each store instruction writes 8 rows x 64 contiguous bytes
      float* tile = reinterpret_cast<float*>(A2h) + warp * (32 * 20);
      const int lane = t & 31, rq = (warp & 3) * 32;
      for (int c0 = cs0; c0 < cs0 + D / 2; c0 += 16) {
        float v[16];
        tmem_ld16(tlane + D2_COL + c0, v);
#pragma unroll
        for (int x = 0; x < 4; ++x)
          *reinterpret_cast<float4*>(tile + lane * 20 + 4 * x) = make_float4(v[4 * x], v[4 * x + 1], v[4 * x + 2], v[4 * x + 3]);
        __syncwarp();
#pragma unroll
        for (int k2 = 0; k2 < 4; ++k2) {
          const int rl = 8 * k2 + (lane >> 2), f = lane & 3;
          const int64_t o = so + (int64_t)(rq + rl) * D + c0 + 4 * f;
          const float4 x4 = *reinterpret_cast<const float4*>(tile + rl * 20 + 4 * f);
          *reinterpret_cast<float4*>(w.s_bnd + o) = x4;
          *reinterpret_cast<float4*>(w.s_run + o) = x4;
        }
        __syncwarp();
      }
    }
    fence_before_sync();
    __syncthreads();  // shared and tensor memory are reused by the next item
  }
  cp_async_wait_all();  // no copy of this thread still in flight
  if (!ok && t == 0) {
    set_error(hdr, GDN_DEVERR_TIMEOUT);
    if (pending) mbar_wait(bar, phase);  // let the MMA in flight finish before releasing its memory
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, TMEM_COLS);
}

// =====================================================================  K2  ====
template <int D>
constexpr size_t intra_smem_bytes() {
  return sizeof(float) * (3 * kMaxChunk * D + 2 * kMaxChunk);
}

template <int D, typename Tin, typename Tout, bool kSkip>
__global__ void __launch_bounds__(2 * D, 2) k_intra(Dims dm, TokenArrays in, IntraWork w,
                                                 WsHeader* __restrict__ hdr) {
  extern __shared__ __align__(16) float sm[];
  float* ks = sm;
  float* qs = ks + kMaxChunk * D;
  float* vs = qs + kMaxChunk * D;  // v, then o (staged)
  float* as = vs + kMaxChunk * D;
  float* bs = as + kMaxChunk;
  if (!hdr->valid) return;
  const int t = threadIdx.x;
  const int64_t c = blockIdx.x;
  const int h = blockIdx.y;
  const int hq = h / (dm.hv / dm.hqk);
  const ChunkRec rec = w.chunks[c];
  if (!in_bounds(hdr, rec.tok0 >= 0 && rec.len >= 0 && rec.len <= dm.C && (int64_t)rec.tok0 + rec.len <= in.n_tokens &&
                          rec.seq >= 0 && rec.seq < w.n_seqs))
    return;
  if constexpr (kSkip) {  // this launch's part of the chunks
    const bool from_run = rec.jloc == 0 && w.skip[rec.seq] > 0;
    if (from_run != (w.part == 1)) return;
  }
  const int len = rec.len;
  const int64_t tok0 = rec.tok0;
  const int64_t SZ = (int64_t)D * D;
  const Tin* qin = static_cast<const Tin*>(in.q);
  const Tin* kin = static_cast<const Tin*>(in.k);
  const Tin* vin = static_cast<const Tin*>(in.v);

  // first token of the recurrence in this chunk: a continued prefill resumes its first chunk
  // from the cache's running state after the tail tokens it already holds
  int first = 0;
  if constexpr (kSkip) {
    if (rec.jloc == 0) first = w.skip[rec.seq];
  }
  for (int idx = first * (D / 4) + t; idx < len * (D / 4); idx += 2 * D) {
    const int r = idx / (D / 4), c4 = idx % (D / 4);
    *reinterpret_cast<float4*>(ks + r * D + 4 * c4) = load4(kin + ((tok0 + r) * dm.hqk + hq) * D + 4 * c4);
    *reinterpret_cast<float4*>(qs + r * D + 4 * c4) = load4(qin + ((tok0 + r) * dm.hqk + hq) * D + 4 * c4);
    *reinterpret_cast<float4*>(vs + r * D + 4 * c4) = load4(vin + ((tok0 + r) * dm.hv + h) * D + 4 * c4);
  }
  for (int r = first + t; r < len; r += 2 * D) {
    as[r] = expf(in.g[(tok0 + r) * dm.hv + h]);
    bs[r] = in.beta[(tok0 + r) * dm.hv + h];
  }
  const StateLayout<D> lay(t);
  float4 S[4][D / 32];
  const float* src = w.bnd + (c * dm.hv + h) * SZ;
  float cs = 1.f;  // the state is cs * S (token_step)
  if constexpr (kSkip) {
    if (first > 0) {
      const int64_t rs = (int64_t)w.run_slot[rec.seq] * dm.hv + h;
      src = w.run_state + rs * SZ;
      cs = w.run_c[rs];
    }
  }
  lay.load(S, src);
  __syncthreads();

  // The token steps (token_step, split in its two sweeps): the output reduction of token
  // tt - 1 runs in the same block as the first sweep of token tt, which does not depend on it.
  // o overwrites v in place: every lane of the row group read that v before contributing to o.
  const int orow = lay.out_row();
  const bool writer = lay.writes_out();
  float opart[4] = {0.f, 0.f, 0.f, 0.f};
  float cprev = 1.f;  // the scale of the previous token's output partials
  for (int tt = first; tt < len; ++tt) {
    float4 kk[D / 32];
    float part[4], p[4], us[4];
    const float4 v4 = *reinterpret_cast<const float4*>(vs + tt * D + lay.row0);
    ts_decay<D>(S, cs, as[tt]);
    ts_dot_k<D>(S, ks + tt * D, lay.b, kk, part);
    const float o_prev = __fmul_rn(cprev, group_reduce4(opart, lay.b));
    if (writer && tt > first) vs[(tt - 1) * D + orow] = o_prev;
    group_allreduce4(part, p);
    ts_scaled_u(p, v4, bs[tt], cs, us);
    ts_update_dot<D>(S, kk, qs + tt * D, us, lay.b, opart);
    cprev = cs;
  }
  if (first < len) {
    const float o_last = __fmul_rn(cprev, group_reduce4(opart, lay.b));
    if (writer) vs[(len - 1) * D + orow] = o_last;
  }
  __syncthreads();
  // the chunk record again (an L2 read instead of registers held through the token loop)
  ChunkRec rc;
  rc.seq = __ldcg(&w.chunks[c].seq);
  rc.tok0 = __ldcg(&w.chunks[c].tok0);
  rc.len = __ldcg(&w.chunks[c].len);
  rc.jloc = __ldcg(&w.chunks[c].jloc);
  Tout* out = static_cast<Tout*>(w.o);
  for (int idx = first * D + t; idx < rc.len * D; idx += 2 * D) {
    const int r = idx / D, e = idx % D;
    store_out(out + (((int64_t)rc.tok0 + r) * dm.hv + h) * D + e, vs[idx]);
  }
  // state decode continues from: the token recurrence through a final partial chunk
  const SeqRec sr = w.seqs[rc.seq];
  if (rc.jloc == sr.nchunks - 1 && (sr.len % dm.C) != 0) {
    if (w.state_out) lay.store_scaled(S, cs, w.state_out + ((int64_t)rc.seq * dm.hv + h) * SZ);
    if (w.cache_run) {  // the scaled state and its scale, for decode to continue from
      const int sl = w.slot_of_seq ? w.slot_of_seq[rc.seq] : rc.seq;
      if (sl >= 0 && sl < w.cache_slots) {
        lay.store(S, w.cache_run + ((int64_t)sl * dm.hv + h) * SZ);
        if (t == 0) w.cache_c_run[(int64_t)sl * dm.hv + h] = cs;
      }
    }
  }
}

template <int D, typename Tin, typename Tout>
static void launch_intra_t(const Dims& d, const TokenArrays& in, const IntraWork& w, WsHeader* hdr,
                           cudaStream_t st) {
  constexpr size_t smem = intra_smem_bytes<D>();
  dim3 grid((unsigned)w.n_chunks, d.hv);
  if (w.skip) {
    ensure_smem(k_intra<D, Tin, Tout, true>, smem);
    k_intra<D, Tin, Tout, true><<<grid, 2 * D, smem, st>>>(d, in, w, hdr);
  } else {
    ensure_smem(k_intra<D, Tin, Tout, false>, smem);
    k_intra<D, Tin, Tout, false><<<grid, 2 * D, smem, st>>>(d, in, w, hdr);
  }
}

// =====================================================================  K3  ====
template <int D, typename Tin, typename Tout>
__global__ void __launch_bounds__(2 * D, 2) k_decode(Dims dm, TokenArrays in, DecodeWork w,
                                                  WsHeader* __restrict__ hdr) {
  __shared__ __align__(16) float ks[D];
  __shared__ __align__(16) float qs[D];
  const int t = threadIdx.x;
  const int n = blockIdx.x, h = blockIdx.y;
  const int grp = dm.hv / dm.hqk;
  const int hq = h / grp;
  const int C = dm.C;
  if (w.no_resync) {  // the host's claim: no token of this step completes a chunk
    bool bad = false;
    for (int m = t; m < w.N; m += 2 * D) {
      const int s2 = w.slot[m];
      if (s2 >= 0 && s2 < w.slots && (w.pos[s2] + 1) % C == 0) bad = true;
    }
    if (__syncthreads_or(bad)) {
      if (t == 0 && n == 0 && h == 0) set_error(hdr, GDN_DEVERR_POS_HOST);
      return;
    }
  }
  const int sl = w.slot[n];
  if (sl < 0 || sl >= w.slots) {
    if (t == 0 && h == 0) set_error(hdr, GDN_DEVERR_SLOT);
    return;
  }
  const int p = w.pos[sl];
  if (p < 0) {
    if (t == 0 && h == 0) set_error(hdr, GDN_DEVERR_POS);
    return;
  }
  const Tin* qin = static_cast<const Tin*>(in.q);
  const Tin* kin = static_cast<const Tin*>(in.k);
  const Tin* vin = static_cast<const Tin*>(in.v);
  const int64_t SZ = (int64_t)D * D;
  if (t < D / 8) {
    float tmp[8];
    load8(kin + ((int64_t)n * dm.hqk + hq) * D + 8 * t, tmp);
#pragma unroll
    for (int e = 0; e < 8; ++e) ks[8 * t + e] = tmp[e];
    load8(qin + ((int64_t)n * dm.hqk + hq) * D + 8 * t, tmp);
#pragma unroll
    for (int e = 0; e < 8; ++e) qs[8 * t + e] = tmp[e];
  }
  const StateLayout<D> lay(t);
  float4 S[4][D / 32];
  float* st = w.s_run + ((int64_t)sl * dm.hv + h) * SZ;
  float* cst = w.c_run + (int64_t)sl * dm.hv + h;
  lay.load(S, st);
  float cs = *cst;  // the running state is cs * S (token_step)
  const float a = expf(in.g[(int64_t)n * dm.hv + h]);
  const float b = in.beta[(int64_t)n * dm.hv + h];
  const Tin* vrow = vin + ((int64_t)n * dm.hv + h) * D;
  const float4 v4 = make_float4(to_f32(vrow[lay.row0]), to_f32(vrow[lay.row0 + 1]), to_f32(vrow[lay.row0 + 2]),
                                to_f32(vrow[lay.row0 + 3]));
  __syncthreads();
  const float o = token_step<D>(S, cs, ks, qs, a, b, v4, lay.b);
  lay.store(S, st);
  if (t == 0) *cst = cs;
  const int ti = p % C;
  if (lay.writes_out()) store_out(static_cast<Tout*>(w.o) + ((int64_t)n * dm.hv + h) * D + lay.out_row(), o);
  if (t < D) static_cast<Tin*>(w.tail_v)[(((int64_t)sl * C + ti) * dm.hv + h) * D + t] = vrow[t];
  if (t == 0) {
    w.tail_g[((int64_t)sl * C + ti) * dm.hv + h] = in.g[(int64_t)n * dm.hv + h];
    w.tail_beta[((int64_t)sl * C + ti) * dm.hv + h] = b;
  }
  if (h % grp == 0 && t < D) {
    static_cast<Tin*>(w.tail_k)[(((int64_t)sl * C + ti) * dm.hqk + hq) * D + t] =
        kin[((int64_t)n * dm.hqk + hq) * D + t];
  }
}

template <int D, typename Tin, typename Tout>
static void launch_decode_t(const Dims& d, const TokenArrays& in, const DecodeWork& w,
                            WsHeader* hdr, cudaStream_t st) {
  dim3 grid((unsigned)w.N, d.hv);
  k_decode<D, Tin, Tout><<<grid, 2 * D, 0, st>>>(d, in, w, hdr);
}

// ============================================================ small helpers ====
__global__ void k_advance(int N, const int32_t* __restrict__ slot, int slots, int32_t* pos,
                          const WsHeader* __restrict__ hdr) {
  if (hdr->err == GDN_DEVERR_POS_HOST) return;  // the step was refused
  for (int n = blockIdx.x * blockDim.x + threadIdx.x; n < N; n += gridDim.x * blockDim.x) {
    const int sl = slot[n];
    if (sl >= 0 && sl < slots && pos[sl] >= 0) pos[sl] += 1;
  }
}

// The workspace header zeroed by one small kernel: a memset node costs several microseconds
// more per call in a replayed CUDA graph, which a decode step's few-microsecond kernels feel.
__global__ void k_reset_header(WsHeader* hdr) { reinterpret_cast<int32_t*>(hdr)[threadIdx.x] = 0; }

void launch_reset_header(WsHeader* hdr, cudaStream_t st) {
  k_reset_header<<<1, sizeof(WsHeader) / sizeof(int32_t), 0, st>>>(hdr);
}

void launch_advance(int N, const int32_t* slot, int slots, int32_t* pos, const WsHeader* hdr, cudaStream_t st) {
  k_advance<<<(N + 255) / 256, 256, 0, st>>>(N, slot, slots, pos, hdr);
}

// The explicit running state of selected cache slots: out[i] = c_run[s] * s_run[s] for
// s = sel[i] (sel NULL: s = i), one round-to-nearest product per element, exactly as the
// kernels form state_out from a scaled state (StateLayout::store_scaled).  A slot outside
// [0, slots) gives an all-NaN block, so a bad index cannot pass for a state.
__global__ void __launch_bounds__(256) k_running_state(int D, int hv, const float* __restrict__ s_run,
                                                       const float* __restrict__ c_run, int slots,
                                                       const int32_t* __restrict__ sel,
                                                       float* __restrict__ out) {
  const int i = blockIdx.x, h = blockIdx.y;
  const int s = sel ? sel[i] : i;
  const int64_t SZ = (int64_t)D * D;
  float4* dst = reinterpret_cast<float4*>(out + ((int64_t)i * hv + h) * SZ);
  if (s < 0 || s >= slots) {
    const float nan = __int_as_float(0x7fffffff);
    for (int64_t e = threadIdx.x; e < SZ / 4; e += blockDim.x) dst[e] = make_float4(nan, nan, nan, nan);
    return;
  }
  const float c = c_run[(int64_t)s * hv + h];
  const float4* src = reinterpret_cast<const float4*>(s_run + ((int64_t)s * hv + h) * SZ);
  for (int64_t e = threadIdx.x; e < SZ / 4; e += blockDim.x) {
    const float4 x = src[e];
    dst[e] = make_float4(__fmul_rn(c, x.x), __fmul_rn(c, x.y), __fmul_rn(c, x.z), __fmul_rn(c, x.w));
  }
}

void launch_running_state(int D, int hv, const float* s_run, const float* c_run, int slots,
                          const int32_t* sel, int n, float* out, cudaStream_t st) {
  if (n <= 0) return;
  k_running_state<<<dim3((unsigned)n, (unsigned)hv), 256, 0, st>>>(D, hv, s_run, c_run, slots, sel, out);
}

template <typename Tin>
__global__ void k_tail_fill(Dims dm, TokenArrays in, const SeqRec* __restrict__ seqs,
                            const int32_t* __restrict__ slot_of_seq, int slots, Tin* tail_k,
                            Tin* tail_v, float* tail_g, float* tail_beta, int32_t* pos,
                            const int32_t* __restrict__ pos_base, const int32_t* __restrict__ keep_rows,
                            WsHeader* __restrict__ hdr) {
  if (!hdr->valid) return;
  const int n = blockIdx.x;
  const SeqRec rec = seqs[n];
  const int sl = slot_of_seq ? slot_of_seq[n] : n;
  if (sl < 0 || sl >= slots) {
    if (threadIdx.x == 0) set_error(hdr, GDN_DEVERR_SLOT);
    return;
  }
  const int C = dm.C, D = dm.D;
  const int nt = rec.len % C;
  if (!in_bounds(hdr, rec.tok0 >= 0 && (int64_t)rec.tok0 + rec.len <= in.n_tokens)) return;
  // rows the slot's tail already holds (continued prefill whose chunk stays open)
  const int k0 = (keep_rows && rec.len < C) ? keep_rows[n] : 0;
  const int64_t base = (int64_t)rec.tok0 + rec.len - nt;
  const Tin* kin = static_cast<const Tin*>(in.k);
  const Tin* vin = static_cast<const Tin*>(in.v);
  // rows k0 .. nt-1 of the last chunk: one contiguous range in the inputs and in the tail
  // (a row of K or V is a multiple of 16 bytes), copied 16 bytes at a time by the
  // gridDim.y CTAs of this sequence
  const int64_t tid = (int64_t)blockIdx.y * blockDim.x + threadIdx.x, nth = (int64_t)gridDim.y * blockDim.x;
  const int64_t rk = (int64_t)dm.hqk * D, rv = (int64_t)dm.hv * D;
  {
    const uint4* src = reinterpret_cast<const uint4*>(kin + (base + k0) * rk);
    uint4* dst = reinterpret_cast<uint4*>(tail_k + ((int64_t)sl * C + k0) * rk);
    const int64_t n16 = (int64_t)(nt - k0) * rk * (int64_t)sizeof(Tin) / 16;
    for (int64_t q = tid; q < n16; q += nth) dst[q] = src[q];
  }
  {
    const uint4* src = reinterpret_cast<const uint4*>(vin + (base + k0) * rv);
    uint4* dst = reinterpret_cast<uint4*>(tail_v + ((int64_t)sl * C + k0) * rv);
    const int64_t n16 = (int64_t)(nt - k0) * rv * (int64_t)sizeof(Tin) / 16;
    for (int64_t q = tid; q < n16; q += nth) dst[q] = src[q];
  }
  const int64_t ng = (int64_t)nt * dm.hv;
  for (int64_t e = (int64_t)k0 * dm.hv + tid; e < ng; e += nth) {
    tail_g[(int64_t)sl * C * dm.hv + e] = in.g[base * dm.hv + e];
    tail_beta[(int64_t)sl * C * dm.hv + e] = in.beta[base * dm.hv + e];
  }
  if (blockIdx.y == 0 && threadIdx.x == 0) pos[sl] = (pos_base ? pos_base[n] : 0) + rec.len;
}

void launch_tail_fill(const Dims& d, const TokenArrays& in, const SeqRec* seqs, int N,
                      const int32_t* slot_of_seq, int slots, void* tail_k, void* tail_v,
                      float* tail_g, float* tail_beta, int32_t* pos, const int32_t* pos_base,
                      const int32_t* keep_rows, WsHeader* hdr, cudaStream_t st) {
  if (N <= 0) return;
  // CTAs per sequence sharing its copy: about two per SM in all, at most 16
  const int64_t per = (2 * (int64_t)sm_count() + N - 1) / N;
  const dim3 grid((unsigned)N, (unsigned)(per < 1 ? 1 : per > 16 ? 16 : per));
  if (d.in_bf16)
    k_tail_fill<__nv_bfloat16><<<grid, 256, 0, st>>>(d, in, seqs, slot_of_seq, slots,
                                                  static_cast<__nv_bfloat16*>(tail_k),
                                                  static_cast<__nv_bfloat16*>(tail_v), tail_g,
                                                  tail_beta, pos, pos_base, keep_rows, hdr);
  else
    k_tail_fill<float><<<grid, 256, 0, st>>>(d, in, seqs, slot_of_seq, slots,
                                          static_cast<float*>(tail_k), static_cast<float*>(tail_v),
                                          tail_g, tail_beta, pos, pos_base, keep_rows, hdr);
}

// ================================================================= dispatch ====
#define GDN_DISPATCH_D(D_, ...)         \
  switch (D_) {                         \
    case 32: { constexpr int DD = 32; __VA_ARGS__; } break; \
    case 64: { constexpr int DD = 64; __VA_ARGS__; } break; \
    default: { constexpr int DD = 128; __VA_ARGS__; } break; \
  }

void launch_prep(const Dims& d, const TokenArrays& in, const PrepWork& w, float* W, float* U,
                 float* gamma, WsHeader* hdr, cudaStream_t st) {
  if (w.n_items <= 0) return;
  if (boundary_on_tensor_cores(d)) {
    ensure_smem(k_prep_tc, tcp::SMEM);
    const int64_t total = w.n_items * d.hv;
    int64_t cap = 2 * (int64_t)sm_count();  // persistent: two CTAs per SM walk the items
    if ((total + cap - 1) / cap > kPrepMaxItems) cap = (total + kPrepMaxItems - 1) / kPrepMaxItems;
    k_prep_tc<<<(unsigned)(total < cap ? total : cap), 256, tcp::SMEM, st>>>(d, in, w, W, U, gamma, hdr);
  } else if (d.in_bf16) {
    GDN_DISPATCH_D(d.D, launch_prep_t<DD, __nv_bfloat16>(d, in, w, W, U, gamma, hdr, st))
  } else {
    GDN_DISPATCH_D(d.D, launch_prep_t<DD, float>(d, in, w, W, U, gamma, hdr, st))
  }
}

bool launch_resync_fused(const Dims& d, const TokenArrays& tail, const PrepWork& pw, const ChainWork& cw,
                         WsHeader* hdr, cudaStream_t st) {
  if (!boundary_on_tensor_cores(d)) return false;
  if (pw.n_items <= 0) return true;
  ensure_smem(k_resync_fused_tc, tcf::SMEM);
  const int64_t total = pw.n_items * d.hv;
  int64_t cap = 2 * (int64_t)sm_count();  // persistent: two CTAs per SM walk the items
  if ((total + cap - 1) / cap > tcf::MAX_ITEMS) cap = (total + tcf::MAX_ITEMS - 1) / tcf::MAX_ITEMS;
  k_resync_fused_tc<<<(unsigned)(total < cap ? total : cap), 256, tcf::SMEM, st>>>(d, tail, pw, cw, hdr);
  return true;
}

void launch_chain(const Dims& d, const void* keys, const float* W, const float* U,
                  const float* gamma, const ChainWork& w, WsHeader* hdr, cudaStream_t st) {
  if (w.N <= 0) return;
  if (boundary_on_tensor_cores(d)) {
    const int64_t total = (int64_t)w.N * d.hv;
    ensure_smem(k_chain_tc, tcc::SMEM);
    // one CTA per chain, scheduled by the hardware (longest first); for batches of short
    // chains (fewer than two chunk records per sequence: continued prefill in small pieces)
    // one wave of CTAs walking the items instead, since most CTAs would find nothing to do
    int64_t cap = total;
    if (w.n_chunks < 2 * (int64_t)w.N && total > (int64_t)sm_count()) cap = sm_count();
    if ((total + cap - 1) / cap > 128) cap = (total + 127) / 128;  // at most 128 items per CTA
    k_chain_tc<<<(unsigned)(total < cap ? total : cap), 256, tcc::SMEM, st>>>(d, W, U, gamma, w, hdr);
  } else if (d.in_bf16) {
    GDN_DISPATCH_D(d.D, launch_chain_t<DD, __nv_bfloat16>(d, keys, W, U, gamma, w, hdr, st))
  } else {
    GDN_DISPATCH_D(d.D, launch_chain_t<DD, float>(d, keys, W, U, gamma, w, hdr, st))
  }
}

void launch_intra(const Dims& d, const TokenArrays& in, const IntraWork& w, WsHeader* hdr,
                  cudaStream_t st) {
  if (w.n_chunks <= 0) return;
  if (d.in_bf16) {
    if (d.out_bf16) {
      GDN_DISPATCH_D(d.D, (launch_intra_t<DD, __nv_bfloat16, __nv_bfloat16>(d, in, w, hdr, st)))
    } else {
      GDN_DISPATCH_D(d.D, (launch_intra_t<DD, __nv_bfloat16, float>(d, in, w, hdr, st)))
    }
  } else {
    if (d.out_bf16) {
      GDN_DISPATCH_D(d.D, (launch_intra_t<DD, float, __nv_bfloat16>(d, in, w, hdr, st)))
    } else {
      GDN_DISPATCH_D(d.D, (launch_intra_t<DD, float, float>(d, in, w, hdr, st)))
    }
  }
}

void launch_decode(const Dims& d, const TokenArrays& in, const DecodeWork& w, WsHeader* hdr,
                   cudaStream_t st) {
  if (w.N <= 0) return;
  if (d.in_bf16) {
    if (d.out_bf16) {
      GDN_DISPATCH_D(d.D, (launch_decode_t<DD, __nv_bfloat16, __nv_bfloat16>(d, in, w, hdr, st)))
    } else {
      GDN_DISPATCH_D(d.D, (launch_decode_t<DD, __nv_bfloat16, float>(d, in, w, hdr, st)))
    }
  } else {
    if (d.out_bf16) {
      GDN_DISPATCH_D(d.D, (launch_decode_t<DD, float, __nv_bfloat16>(d, in, w, hdr, st)))
    } else {
      GDN_DISPATCH_D(d.D, (launch_decode_t<DD, float, float>(d, in, w, hdr, st)))
    }
  }
}


// =====================================================================  K5  ====
// Prefill continued from a decode cache (chunked prefill, multi-token decode): sequence s
// is replayed as a virtual sequence made of its cache tail (the r_s = pos % C tokens since
// its last chunk boundary; their outputs already exist, so q is zero) followed by its L_s
// new tokens, from that chunk boundary and the cache's boundary state.  Chunk boundaries of
// the virtual sequence are those of the whole sequence, so the prefill kernels that run on
// it give the bits one prefill of the whole sequence gives.

// One block: tail length and base position of every sequence from the device cache, and
// the virtual cu_seqlens (a fixed-order prefix sum).  A slot or position out of range sets
// the error word and poisons the virtual total, which the work-list check then rejects.
__global__ void __launch_bounds__(1024) k_continue_prep(const int32_t* __restrict__ cu,
                                                        const int32_t* __restrict__ slot,
                                                        const int32_t* __restrict__ pos, int slots, int N,
                                                        int C, int32_t* __restrict__ vcu,
                                                        int32_t* __restrict__ rlen, int32_t* __restrict__ base,
                                                        WsHeader* __restrict__ hdr) {
  __shared__ int32_t scan[1024];
  __shared__ int bad;
  const int t = threadIdx.x;
  if (t == 0) bad = 0;
  __syncthreads();
  int32_t carry = 0;
  for (int b0 = 0; b0 < N; b0 += 1024) {
    const int s = b0 + t;
    int32_t V = 0;
    if (s < N) {
      const int sl = slot[s];
      int32_t r = 0, p = 0;
      if (sl < 0 || sl >= slots) {
        bad = 1;
        set_error(hdr, GDN_DEVERR_SLOT);
      } else {
        p = pos[sl];
        if (p < 0) {
          bad = 1;
          set_error(hdr, GDN_DEVERR_POS);
          p = 0;
        } else {
          r = p % C;
        }
      }
      rlen[s] = r;
      base[s] = p - r;
      V = r + (cu[s + 1] - cu[s]);
    }
    scan[t] = V;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {
      const int32_t x = (t >= off) ? scan[t - off] : 0;
      __syncthreads();
      scan[t] += x;
      __syncthreads();
    }
    if (s < N) vcu[s + 1] = carry + scan[t];
    carry += scan[1023];
    __syncthreads();
  }
  if (t == 0) {
    vcu[0] = 0;
    if (bad) vcu[N] = -1;
  }
}

// index s with cu[s] <= x < cu[s + 1] (cu non-decreasing, cu[0] <= x < cu[n])
__device__ __forceinline__ int seq_of(const int32_t* __restrict__ cu, int n, int64_t x) {
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cu[mid] <= x) lo = mid; else hi = mid;
  }
  return lo;
}

// bytes (a multiple of 16) from src to dst, 16 at a time, by the block's threads; src NULL
// writes zeros
__device__ __forceinline__ void copy16(void* dst, const void* src, int64_t bytes) {
  uint4* d = static_cast<uint4*>(dst);
  const uint4* s = static_cast<const uint4*>(src);
  for (int64_t e = threadIdx.x; e < bytes / 16; e += blockDim.x) d[e] = s ? s[e] : make_uint4(0u, 0u, 0u, 0u);
}

// One block per virtual token: its q, k, v, g, beta rows, from the cache tail or the inputs.
__global__ void k_continue_gather(Dims dm, TokenArrays in, const int32_t* __restrict__ cu,
                                  const int32_t* __restrict__ vcu, const int32_t* __restrict__ rlen,
                                  const int32_t* __restrict__ slot, int N, int esz, const void* tail_k,
                                  const void* tail_v, const float* __restrict__ tail_g,
                                  const float* __restrict__ tail_beta, TokenArrays out,
                                  const WsHeader* __restrict__ hdr) {
  if (!hdr->valid) return;
  const int64_t vt = blockIdx.x;
  const int s = seq_of(vcu, N, vt);
  const int local = (int)(vt - vcu[s]);
  const int r = rlen[s];
  // a tail token is read only by the pre-pass of a completed first chunk (the recurrence
  // resumes after the tail, and the cache keeps its tail rows when the chunk stays open)
  if (local < r && vcu[s + 1] - vcu[s] < dm.C) return;
  const int64_t nq = (int64_t)dm.hqk * dm.D * esz, nv = (int64_t)dm.hv * dm.D * esz;
  const int64_t ng = (int64_t)dm.hv;
  char* qo = static_cast<char*>(const_cast<void*>(out.q)) + vt * nq;
  char* ko = static_cast<char*>(const_cast<void*>(out.k)) + vt * nq;
  char* vo = static_cast<char*>(const_cast<void*>(out.v)) + vt * nv;
  float* go = const_cast<float*>(out.g) + vt * ng;
  float* bo = const_cast<float*>(out.beta) + vt * ng;
  if (local < r) {
    const int64_t row = (int64_t)slot[s] * dm.C + local;  // tail row of the slot
    copy16(qo, nullptr, nq);
    copy16(ko, static_cast<const char*>(tail_k) + row * nq, nq);
    copy16(vo, static_cast<const char*>(tail_v) + row * nv, nv);
    for (int64_t e = threadIdx.x; e < ng; e += blockDim.x) {
      go[e] = tail_g[row * ng + e];
      bo[e] = tail_beta[row * ng + e];
    }
  } else {
    const int64_t src = (int64_t)cu[s] + (local - r);
    if (!in_bounds(const_cast<WsHeader*>(hdr), src >= 0 && src < in.n_tokens)) return;
    copy16(qo, static_cast<const char*>(in.q) + src * nq, nq);
    copy16(ko, static_cast<const char*>(in.k) + src * nq, nq);
    copy16(vo, static_cast<const char*>(in.v) + src * nv, nv);
    for (int64_t e = threadIdx.x; e < ng; e += blockDim.x) {
      go[e] = in.g[src * ng + e];
      bo[e] = in.beta[src * ng + e];
    }
  }
}

// One block per new token: its output row from the virtual sequence's output.
__global__ void k_continue_scatter(const int32_t* __restrict__ cu, const int32_t* __restrict__ vcu,
                                   const int32_t* __restrict__ rlen, int N, int64_t vT, int64_t row_bytes,
                                   const void* __restrict__ vo, void* __restrict__ o,
                                   const WsHeader* __restrict__ hdr) {
  if (!hdr->valid) return;
  const int64_t tk = blockIdx.x;
  const int s = seq_of(cu, N, tk);
  const int64_t vrow = (int64_t)vcu[s] + rlen[s] + (tk - cu[s]);
  if (!in_bounds(const_cast<WsHeader*>(hdr), vrow >= 0 && vrow < vT)) return;
  copy16(static_cast<char*>(o) + tk * row_bytes, static_cast<const char*>(vo) + vrow * row_bytes, row_bytes);
}

void launch_continue_prep(const int32_t* cu, const int32_t* slot, const int32_t* pos, int slots, int N, int C,
                          int32_t* vcu, int32_t* rlen, int32_t* base, WsHeader* hdr, cudaStream_t st) {
  if (N > 0) k_continue_prep<<<1, 1024, 0, st>>>(cu, slot, pos, slots, N, C, vcu, rlen, base, hdr);
}

void launch_continue_gather(const Dims& d, const TokenArrays& in, const int32_t* cu, const int32_t* vcu,
                            const int32_t* rlen, const int32_t* slot, int N, int64_t vT,
                            const gdn_cpr_cache& cache, const TokenArrays& out, WsHeader* hdr, cudaStream_t st) {
  if (vT > 0)
    k_continue_gather<<<(unsigned)vT, 256, 0, st>>>(d, in, cu, vcu, rlen, slot, N, d.in_bf16 ? 2 : 4,
                                                    cache.tail_k, cache.tail_v, cache.tail_g, cache.tail_beta,
                                                    out, hdr);
}

void launch_continue_scatter(const Dims& d, const int32_t* cu, const int32_t* vcu, const int32_t* rlen, int N,
                             int64_t T, int64_t vT, const void* vo, void* o, WsHeader* hdr, cudaStream_t st) {
  if (T > 0)
    k_continue_scatter<<<(unsigned)T, 128, 0, st>>>(cu, vcu, rlen, N, vT, (int64_t)d.hv * d.D * (d.out_bf16 ? 2 : 4),
                                                    vo, o, hdr);
}

}  // namespace gdn
