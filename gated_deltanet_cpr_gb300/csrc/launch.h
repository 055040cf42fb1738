// launch.h -- internal interface between the C-ABI host code and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gdn_cpr.h"
#include "common.cuh"

namespace gdn {

// Pointers to a run of tokens laid out as the packed inputs ([tok, H, D] / [tok, H]);
// the decode tail of slot s is such a run starting at token s * C.
struct TokenArrays {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  int64_t n_tokens;  // rows the arrays hold (bounds-checked builds check every range against it)
};

struct Dims {
  int hqk, hv, D, C;
  bool in_bf16, out_bf16;
};

// Floats reserved per (chunk, head) for the pre-pass's W output: fp32 Wd (C x D) on the
// SIMT path, or three bf16 C x D shared-memory images (Wd hi, Wd lo, K^T) on the
// tensor-core path.
__host__ __device__ inline size_t prep_w_floats(int C, int D) { return (size_t)3 * C * D / 2; }

// The boundary pass runs on tcgen05 tensor cores for bf16 inputs with d = 128, C = 64, and
// on fp32 SIMT otherwise (fp32 inputs keep an fp32 boundary pass).  Prefill and decode
// resynchronisation always take the same path for a given shape.
__host__ __device__ inline bool boundary_on_tensor_cores(const Dims& d) { return d.in_bf16 && d.D == 128 && d.C == 64; }

// K0: chunk and sequence records from the device cu_seqlens, checked against the host's
// chunk count and a hash of the host copy.
void launch_worklist(const int32_t* cu, int N, int T, int C, int64_t n_chunks, uint32_t cu_hash,
                     ChunkRec* chunks, SeqRec* seqs, WsHeader* hdr, cudaStream_t st);

// K1a: boundary pre-pass over full chunks.  Prefill: one CTA per (chunk record, head),
// partial chunks skip.  Decode: one CTA per (step token n, head) whose slot completes a
// chunk with this token; the chunk is read from the slot's tail.
struct PrepWork {
  // prefill
  const ChunkRec* chunks;  // NULL in decode mode
  int64_t n_items;
  // decode
  const int32_t* slot;
  const int32_t* pos;
  int slots;
};
void launch_prep(const Dims& d, const TokenArrays& in, const PrepWork& w, float* W, float* U,
                 float* gamma, WsHeader* hdr, cudaStream_t st);

// K1b: boundary chain.  Prefill: one CTA per (sequence, head, 16-row block), sequential
// over the sequence's full chunks; writes the start state of every chunk to bnd and the
// final boundary state to state_out (if L % C == 0) and to the cache.  Decode: one step per
// resynchronising (token n, head, row block): s_bnd <- F(s_bnd, tail), s_run <- s_bnd.
struct ChainWork {
  // prefill
  const SeqRec* seqs;  // NULL in decode mode
  int N;
  const float* state_in;
  const int32_t* state_in_slot;  // state_in row of sequence n is state_in_slot[n] (NULL: n)
  float* bnd;
  float* state_out;
  float* cache_bnd;  // cache s_bnd (prefill with cache) or NULL
  float* cache_run;  // cache s_run (prefill with cache, written when L % C == 0) or NULL
  float* cache_c_run;  // its scale c_run, set to 1 with it
  const int32_t* slot_of_seq;
  int cache_slots;
  // continued prefill: state_in is cache_bnd under the same slot map (S^(0) need not be
  // written back), and a sequence with bnd_skip[n] > 0 starts its first chunk from the
  // cache's running state (S^(0) is not needed in bnd)
  bool bnd_in_place;
  const int32_t* bnd_skip;
  int64_t n_chunks;  // chunk records (rows of the pre-pass outputs and of bnd)
  int64_t n_tokens;  // token rows behind `keys`
  // decode
  const int32_t* slot;
  const int32_t* pos;
  float* s_bnd;
  float* s_run;
  float* c_run;  // set to 1 with s_run
  int slots;
  // test hook (tensor-core chain only): nonzero makes CTA 0 wait, before any copy or MMA, on
  // a barrier phase that nothing completes, with a short poll limit, so that the bounded
  // wait runs out and the CTA records GDN_DEVERR_TIMEOUT, frees its tensor memory and exits
  int fault_wait;
};
// K1c: the decode resync's pre-pass and boundary step as one kernel on the tensor cores
// (the same values as launch_prep followed by launch_chain).  Returns false, launching
// nothing, for shapes without the tensor-core boundary path.
bool launch_resync_fused(const Dims& d, const TokenArrays& tail, const PrepWork& pw, const ChainWork& cw,
                         WsHeader* hdr, cudaStream_t st);
void launch_chain(const Dims& d, const void* keys, const float* W, const float* U,
                  const float* gamma, const ChainWork& w, WsHeader* hdr, cudaStream_t st);

// K2: token recurrence inside every chunk from its boundary state, all chunks at once.
struct IntraWork {
  const ChunkRec* chunks;
  const SeqRec* seqs;
  int n_seqs;
  int64_t n_chunks;
  const float* bnd;
  void* o;
  float* state_out;
  float* cache_run;    // the running state after a final partial chunk, scaled: s_run and
  float* cache_c_run;  // its scale c_run (the state is c_run * s_run)
  const int32_t* slot_of_seq;
  int cache_slots;
  // continued prefill: the first skip[seq] tokens of a sequence's first chunk are already in
  // run_state[run_slot[seq]] (the cache's running state), so that chunk's recurrence starts
  // there, from token skip[seq]; NULL otherwise
  const int32_t* skip;
  const float* run_state;
  const float* run_c;  // the scale of run_state
  const int32_t* run_slot;
  // with skip: 1 = only the chunks that start from run_state, 2 = all other chunks.  The
  // continued prefill launches part 1 before the boundary chain and part 2 after it, so
  // that every read of the cache's running state precedes every write to it.
  int part;
};
void launch_intra(const Dims& d, const TokenArrays& in, const IntraWork& w, WsHeader* hdr,
                  cudaStream_t st);

// K3: one decode token per slot: token step on s_run, output, append to the tail.
struct DecodeWork {
  int N;
  const int32_t* slot;
  int slots;
  float* s_run;
  float* c_run;
  void* tail_k;
  void* tail_v;
  float* tail_g;
  float* tail_beta;
  const int32_t* pos;
  void* o;
  // the host said no token of this step completes a chunk: every CTA first checks that on
  // the device and, if it is false for any slot, the step does nothing (GDN_DEVERR_POS_HOST)
  int no_resync;
};
void launch_decode(const Dims& d, const TokenArrays& in, const DecodeWork& w, WsHeader* hdr,
                   cudaStream_t st);

// Zero the workspace header (first kernel of every call).
void launch_reset_header(WsHeader* hdr, cudaStream_t st);

// pos[slot[n]] += 1 for every valid n (last kernel of a decode step), unless the step was
// refused (GDN_DEVERR_POS_HOST in the error word).
void launch_advance(int N, const int32_t* slot, int slots, int32_t* pos, const WsHeader* hdr, cudaStream_t st);

// out[i] = c_run[s] * s_run[s] (s = sel[i], or i if sel is NULL) for i < n, all heads:
// the explicit running state of cache slots.
void launch_running_state(int D, int hv, const float* s_run, const float* c_run, int slots,
                          const int32_t* sel, int n, float* out, cudaStream_t st);

// Prefill with a cache: copy the last L % C tokens of every sequence to its slot's tail and
// set pos = L, plus pos_base[n] when given (a continued prefill's chunk-aligned start); with
// keep_rows, a sequence shorter than C leaves its first keep_rows[n] tail rows as they are.
void launch_tail_fill(const Dims& d, const TokenArrays& in, const SeqRec* seqs, int N,
                      const int32_t* slot_of_seq, int slots, void* tail_k, void* tail_v,
                      float* tail_g, float* tail_beta, int32_t* pos, const int32_t* pos_base,
                      const int32_t* keep_rows, WsHeader* hdr, cudaStream_t st);

// K5: prefill continued from a decode cache.  prep: per sequence the cache tail length and
// base position, and the virtual cu_seqlens (tail + new tokens); gather: the virtual
// sequences' q, k, v, g, beta; scatter: the new tokens' outputs.
void launch_continue_prep(const int32_t* cu, const int32_t* slot, const int32_t* pos, int slots, int N, int C,
                          int32_t* vcu, int32_t* rlen, int32_t* base, WsHeader* hdr, cudaStream_t st);
void launch_continue_gather(const Dims& d, const TokenArrays& in, const int32_t* cu, const int32_t* vcu,
                            const int32_t* rlen, const int32_t* slot, int N, int64_t vT,
                            const gdn_cpr_cache& cache, const TokenArrays& out, WsHeader* hdr, cudaStream_t st);
void launch_continue_scatter(const Dims& d, const int32_t* cu, const int32_t* vcu, const int32_t* rlen, int N,
                             int64_t T, int64_t vT, const void* vo, void* o, WsHeader* hdr, cudaStream_t st);

// Backward (kernels_bwd.cu).  `mark(ctx, kernels)` is called after each stage (prep,
// chain, big products, gradients, grouped-head sum) with the kernels it launched.
typedef void (*BwdStageFn)(void* ctx, int kernels);
size_t bwd_workspace_floats_per_chunk_head(int C, int D);
void launch_bwd(const Dims& d, const TokenArrays& in, const void* dO, const ChunkRec* chunks,
                const SeqRec* seqs, int N, int64_t n_chunks, int64_t T, const float* saved_bnd,
                const float* dstate_out, float* dstate_in, float* per_chunk, float* dq_part,
                float* dk_part, float* dq, float* dk, float* dv, float* dg, float* dbeta,
                WsHeader* hdr, BwdStageFn mark, void* mark_ctx, cudaStream_t st);

}  // namespace gdn
