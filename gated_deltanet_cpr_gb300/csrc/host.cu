// host.cu -- the C ABI of include/gdn_cpr.h: argument checks, workspace layout and the
// launch sequence of every mode.  The host never touches tensor data; it only reads the
// caller's host copy of cu_seqlens to size grids and the workspace.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>
#include <string.h>

#include <vector>

#include "../../include/gdn_cpr.h"
#include "launch.h"

#define GDN_VERSION_NUM 200  // 0.2.0

namespace {
using namespace gdn;

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline bool ok_ptr(const void* p, size_t a) { return p != nullptr && aligned(p, a); }

gdn_status check_shape(const gdn_cpr_shape* s) {
  if (!s) return GDN_ERR_INVALID_ARG;
  if (s->num_seqs < 0 || s->total_tokens < 0 || s->h_qk <= 0 || s->h_v <= 0 || s->d_k <= 0 ||
      s->d_v <= 0 || s->chunk <= 0)
    return GDN_ERR_INVALID_ARG;
  if (s->h_v % s->h_qk != 0) return GDN_ERR_UNSUPPORTED;
  if (s->d_k != s->d_v) return GDN_ERR_UNSUPPORTED;
  if (s->d_k != 32 && s->d_k != 64 && s->d_k != 128) return GDN_ERR_UNSUPPORTED;
  if (s->chunk != 16 && s->chunk != 32 && s->chunk != 64) return GDN_ERR_UNSUPPORTED;
  if ((s->in_dtype != GDN_F32 && s->in_dtype != GDN_BF16) ||
      (s->out_dtype != GDN_F32 && s->out_dtype != GDN_BF16))
    return GDN_ERR_UNSUPPORTED;
  return GDN_OK;
}

// Host copy of cu_seqlens: checks it and returns the chunk count and the hash the
// work-list kernel compares the device copy against.
gdn_status scan_cu(const gdn_cpr_shape* s, const int32_t* cu, int64_t* n_chunks, uint32_t* hash) {
  const int N = s->num_seqs;
  if (!cu) return GDN_ERR_INVALID_ARG;
  if (cu[0] != 0 || cu[N] != s->total_tokens) return GDN_ERR_INVALID_ARG;
  int64_t nc = 0;
  uint32_t h = 0;
  for (int i = 0; i <= N; ++i) {
    if (i < N && cu[i + 1] < cu[i]) return GDN_ERR_INVALID_ARG;
    h += (uint32_t)cu[i] * (uint32_t)(2 * i + 1);
    if (i < N) nc += (cu[i + 1] - cu[i] + s->chunk - 1) / s->chunk;
  }
  *n_chunks = nc;
  *hash = h;
  return GDN_OK;
}

Dims dims_of(const gdn_cpr_shape* s) {
  Dims d;
  d.hqk = s->h_qk;
  d.hv = s->h_v;
  d.D = s->d_k;
  d.C = s->chunk;
  d.in_bf16 = s->in_dtype == GDN_BF16;
  d.out_bf16 = s->out_dtype == GDN_BF16;
  return d;
}

// ------------------------------------------------------------- layouts ----
struct FwdLayout {
  size_t chunks, seqs, W, U, gamma, bnd, total;
};

FwdLayout fwd_layout(const gdn_cpr_shape* s, int64_t n_chunks, bool own_bnd) {
  const size_t D = s->d_k, C = s->chunk, hv = s->h_v;
  FwdLayout L;
  size_t off = align_up(sizeof(WsHeader));
  L.chunks = off; off = align_up(off + sizeof(ChunkRec) * (size_t)n_chunks);
  L.seqs = off;   off = align_up(off + sizeof(SeqRec) * (size_t)s->num_seqs);
  L.W = off;      off = align_up(off + sizeof(float) * (size_t)n_chunks * hv * prep_w_floats((int)C, (int)D));
  L.U = off;      off = align_up(off + sizeof(float) * (size_t)n_chunks * hv * C * D);
  L.gamma = off;  off = align_up(off + sizeof(float) * (size_t)n_chunks * hv);
  L.bnd = off;
  if (own_bnd) off = align_up(off + sizeof(float) * (size_t)n_chunks * hv * D * D);
  L.total = off;
  return L;
}

struct DecLayout {
  size_t W, U, gamma, total;
};

DecLayout dec_layout(const gdn_cpr_shape* s) {
  const size_t D = s->d_k, C = s->chunk, hv = s->h_v, N = s->num_seqs;
  DecLayout L;
  size_t off = align_up(sizeof(WsHeader));
  L.W = off;     off = align_up(off + sizeof(float) * N * hv * prep_w_floats((int)C, (int)D));
  L.U = off;     off = align_up(off + sizeof(float) * N * hv * C * D);
  L.gamma = off; off = align_up(off + sizeof(float) * N * hv);
  L.total = off;
  return L;
}

struct BwdLayout {
  size_t chunks, seqs, per_chunk, dq_part, dk_part, total;
};

BwdLayout bwd_layout(const gdn_cpr_shape* s, int64_t n_chunks) {
  const size_t D = s->d_k, C = s->chunk, hv = s->h_v, T = s->total_tokens;
  BwdLayout L;
  size_t off = align_up(sizeof(WsHeader));
  L.chunks = off;    off = align_up(off + sizeof(ChunkRec) * (size_t)n_chunks);
  L.seqs = off;      off = align_up(off + sizeof(SeqRec) * (size_t)s->num_seqs);
  L.per_chunk = off; off = align_up(off + sizeof(float) * (size_t)n_chunks * hv *
                                              bwd_workspace_floats_per_chunk_head((int)C, (int)D));
  L.dq_part = off;   off = align_up(off + sizeof(float) * T * hv * D);
  L.dk_part = off;   off = align_up(off + sizeof(float) * T * hv * D);
  L.total = off;
  return L;
}

inline char* at(void* ws, size_t off) { return static_cast<char*>(ws) + off; }

gdn_status check_cache(const gdn_cpr_cache* c) {
  if (!c) return GDN_ERR_INVALID_ARG;
  if (c->slots <= 0) return GDN_ERR_INVALID_ARG;
  if (!ok_ptr(c->s_run, 16) || !ok_ptr(c->c_run, 4) || !ok_ptr(c->s_bnd, 16) || !ok_ptr(c->tail_k, 16) ||
      !ok_ptr(c->tail_v, 16) || !ok_ptr(c->tail_g, 4) || !ok_ptr(c->tail_beta, 4) ||
      !ok_ptr(c->pos, 4))
    return GDN_ERR_INVALID_ARG;
  return GDN_OK;
}

thread_local gdn_cpr_profile* t_profile = nullptr;
// gdn_cpr_test_wait_timeout: calls left that make the tensor-core chain's first CTA give up
// a wait that nothing completes
thread_local int32_t t_wait_fault = 0;

// Stage marker of the profiling hook: event `stage` after the stage's kernels, and the
// count of kernels those stages launched.
// Continued prefill: the virtual prefill's regions, then the virtual cu_seqlens, tail
// lengths, base positions, the gathered q, k, v, g, beta and the virtual output.
struct ContLayout {
  FwdLayout f;
  size_t vcu, rlen, base, q, k, v, g, beta, o, total;
};

ContLayout cont_layout(const gdn_cpr_shape* sv, int64_t vchunks) {
  ContLayout L;
  L.f = fwd_layout(sv, vchunks, true);
  const size_t N = sv->num_seqs, vT = sv->total_tokens, D = sv->d_k, hqk = sv->h_qk, hv = sv->h_v;
  const size_t esz = sv->in_dtype == GDN_BF16 ? 2 : 4, osz = sv->out_dtype == GDN_BF16 ? 2 : 4;
  size_t off = L.f.total;
  L.vcu = off;  off = align_up(off + sizeof(int32_t) * (N + 1));
  L.rlen = off; off = align_up(off + sizeof(int32_t) * N);
  L.base = off; off = align_up(off + sizeof(int32_t) * N);
  L.q = off;    off = align_up(off + vT * hqk * D * esz);
  L.k = off;    off = align_up(off + vT * hqk * D * esz);
  L.v = off;    off = align_up(off + vT * hv * D * esz);
  L.g = off;    off = align_up(off + vT * hv * sizeof(float));
  L.beta = off; off = align_up(off + vT * hv * sizeof(float));
  L.o = off;    off = align_up(off + vT * hv * D * osz);
  L.total = off;
  return L;
}

// Virtual cu_seqlens of a continued prefill: sequence i is r_i = pos_i % C tail tokens plus
// its new tokens (pos NULL: the largest tail, C - 1, for the workspace bound).
gdn_status virtual_cu(const gdn_cpr_shape* s, const int32_t* cu, const int32_t* pos, std::vector<int32_t>& vcu) {
  const int N = s->num_seqs;
  vcu.assign((size_t)N + 1, 0);
  int64_t acc = 0;
  for (int i = 0; i < N; ++i) {
    int32_t r = s->chunk - 1;
    if (pos) {
      if (pos[i] < 0) return GDN_ERR_INVALID_ARG;
      r = pos[i] % s->chunk;
    }
    acc += r + (int64_t)(cu[i + 1] - cu[i]);
    if (acc > INT32_MAX) return GDN_ERR_INVALID_ARG;
    vcu[(size_t)i + 1] = (int32_t)acc;
  }
  return GDN_OK;
}

// NVTX range over one entry point (host-side markers for profilers such as Nsight; no
// effect without a tool attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// Stage boundaries of one call: the profiling hook's events and kernel counts, and a nested
// NVTX range per stage (names[i] is stage i + 1; NULL-terminated).
struct Stages {
  cudaStream_t st;
  const char* const* names;
  int next = 0;
  bool open = false;
  Stages(cudaStream_t s, const char* const* stage_names) : st(s), names(stage_names) {
    if (t_profile) t_profile->stages = 0;
    mark(0);
  }
  ~Stages() {
    if (open) nvtxRangePop();
  }
  Stages(const Stages&) = delete;
  Stages& operator=(const Stages&) = delete;
  // a kernel launched at the start of the first stage (counted, no event of its own)
  void count(int kernels) {
    if (t_profile) t_profile->kernels += kernels;
  }
  void mark(int kernels) {
    if (open) nvtxRangePop();
    open = names && names[next] != nullptr;
    if (open) nvtxRangePushA(names[next]);
    if (!t_profile) {
      ++next;
      return;
    }
    t_profile->kernels += kernels;
    if (next < t_profile->n_events && next < 16 && t_profile->events[next]) {
      cudaEventRecord(static_cast<cudaEvent_t>(t_profile->events[next]), st);
      t_profile->stages = next + 1;
    }
    ++next;
  }
};

const char* const kFwdStages[] = {"work list", "boundary pre-pass", "boundary chain", "intra-chunk recurrence",
                                  "cache tail", nullptr};
const char* const kDecodeStages[] = {"decode token step", "resync", "position advance", nullptr};
const char* const kBwdStages[] = {"work list", "backward prep", "reverse boundary chain", "backward products",
                                  "backward gradients", "grouped-head sum", nullptr};
const char* const kContStages[] = {"continue: positions, work list, gather", "boundary pre-pass",
                                   "intra-chunk (cached part) + boundary chain", "intra-chunk recurrence",
                                   "cache tail + scatter", nullptr};

void stage_mark(void* ctx, int kernels) { static_cast<Stages*>(ctx)->mark(kernels); }

gdn_status finish(cudaStream_t st) {
  (void)st;
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

// Forward path shared by prefill and the trainer forward (same kernels, same order).
gdn_status run_forward(const gdn_cpr_shape* shape, const void* q, const void* k, const void* v,
                       const float* g, const float* beta, const float* state_in,
                       const int32_t* cu_dev, const int32_t* cu_host, void* o, float* state_out,
                       const gdn_cpr_cache* cache, const int32_t* slot_of_seq, float* saved_bnd,
                       void* ws, size_t ws_bytes, cudaStream_t st) {
  gdn_status rc = check_shape(shape);
  if (rc != GDN_OK) return rc;
  int64_t n_chunks = 0;
  uint32_t hash = 0;
  rc = scan_cu(shape, cu_host, &n_chunks, &hash);
  if (rc != GDN_OK) return rc;
  const int N = shape->num_seqs;
  const int64_t T = shape->total_tokens;
  if (T > 0 && (!ok_ptr(q, 16) || !ok_ptr(k, 16) || !ok_ptr(v, 16) || !ok_ptr(g, 4) ||
                !ok_ptr(beta, 4) || !ok_ptr(o, 16)))
    return GDN_ERR_INVALID_ARG;
  if (N > 0 && !ok_ptr(cu_dev, 4)) return GDN_ERR_INVALID_ARG;
  if (state_in && !aligned(state_in, 16)) return GDN_ERR_INVALID_ARG;
  if (state_out && !aligned(state_out, 16)) return GDN_ERR_INVALID_ARG;
  if (saved_bnd && !aligned(saved_bnd, 16)) return GDN_ERR_INVALID_ARG;
  if (cache) {
    rc = check_cache(cache);
    if (rc != GDN_OK) return rc;
    if (slot_of_seq && !aligned(slot_of_seq, 4)) return GDN_ERR_INVALID_ARG;
    if (!slot_of_seq && N > cache->slots) return GDN_ERR_INVALID_ARG;
  }
  const FwdLayout L = fwd_layout(shape, n_chunks, saved_bnd == nullptr);
  if (!ws || !aligned(ws, kAlign) || ws_bytes < L.total) return GDN_ERR_WORKSPACE;
  if (N == 0) return GDN_OK;

  const Dims d = dims_of(shape);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  ChunkRec* chunks = reinterpret_cast<ChunkRec*>(at(ws, L.chunks));
  SeqRec* seqs = reinterpret_cast<SeqRec*>(at(ws, L.seqs));
  float* W = reinterpret_cast<float*>(at(ws, L.W));
  float* U = reinterpret_cast<float*>(at(ws, L.U));
  float* gamma = reinterpret_cast<float*>(at(ws, L.gamma));
  float* bnd = saved_bnd ? saved_bnd : reinterpret_cast<float*>(at(ws, L.bnd));
  TokenArrays in{q, k, v, g, beta, T};

  Stages stg(st, kFwdStages);
  launch_reset_header(hdr, st);  // error word and work-list flag of this call
  stg.count(1);
  launch_worklist(cu_dev, N, (int)T, d.C, n_chunks, hash, chunks, seqs, hdr, st);
  stg.mark(1);

  PrepWork pw{};
  pw.chunks = chunks;
  pw.n_items = n_chunks;
  launch_prep(d, in, pw, W, U, gamma, hdr, st);
  stg.mark(n_chunks > 0 ? 1 : 0);

  ChainWork cw{};
  cw.seqs = seqs;
  cw.N = N;
  cw.n_chunks = n_chunks;
  cw.n_tokens = T;
  cw.state_in = state_in;
  cw.bnd = bnd;
  cw.state_out = state_out;
  if (cache) {
    cw.cache_bnd = cache->s_bnd;
    cw.cache_run = cache->s_run;
    cw.cache_c_run = cache->c_run;
    cw.cache_slots = cache->slots;
    cw.slot_of_seq = slot_of_seq;
  }
  if (t_wait_fault > 0 && boundary_on_tensor_cores(d)) {
    cw.fault_wait = 1;
    --t_wait_fault;
  }
  launch_chain(d, k, W, U, gamma, cw, hdr, st);
  stg.mark(1);

  IntraWork iw{};
  iw.chunks = chunks;
  iw.seqs = seqs;
  iw.n_seqs = N;
  iw.n_chunks = n_chunks;
  iw.bnd = bnd;
  iw.o = o;
  iw.state_out = state_out;
  if (cache) {
    iw.cache_run = cache->s_run;
    iw.cache_c_run = cache->c_run;
    iw.cache_slots = cache->slots;
    iw.slot_of_seq = slot_of_seq;
  }
  launch_intra(d, in, iw, hdr, st);
  stg.mark(n_chunks > 0 ? 1 : 0);

  if (cache) {
    launch_tail_fill(d, in, seqs, N, slot_of_seq, cache->slots, cache->tail_k, cache->tail_v,
                     cache->tail_g, cache->tail_beta, cache->pos, nullptr, nullptr, hdr, st);
    stg.mark(1);
  }
  return finish(st);
}

// One decode step (gdn_cpr_decode_step; with pos_host, gdn_cpr_decode_step_pos): the token
// step, then the resynchronisation (the same boundary pre-pass and chain step as prefill, on
// the cached chunk) for the tokens that complete a chunk, then the position advance.  With a
// host copy of the positions that shows no token completing a chunk, the resync kernels are
// not launched and the token step checks that claim on the device.
gdn_status run_decode(const gdn_cpr_shape* shape, const void* q, const void* k, const void* v, const float* g,
                      const float* beta, const int32_t* slot, const int32_t* pos_host, const gdn_cpr_cache* cache,
                      void* o, void* ws, size_t ws_bytes, gdn_stream_t stream) {
  gdn_status rc = check_shape(shape);
  if (rc != GDN_OK) return rc;
  const int N = shape->num_seqs;
  if (shape->total_tokens != N) return GDN_ERR_INVALID_ARG;
  rc = check_cache(cache);
  if (rc != GDN_OK) return rc;
  if (N > 0 && (!ok_ptr(q, 16) || !ok_ptr(k, 16) || !ok_ptr(v, 16) || !ok_ptr(g, 4) ||
                !ok_ptr(beta, 4) || !ok_ptr(o, 16) || !ok_ptr(slot, 4)))
    return GDN_ERR_INVALID_ARG;
  bool resync = true;  // whether any token of this step may complete a chunk
  if (pos_host) {
    resync = false;
    for (int n = 0; n < N; ++n) {
      if (pos_host[n] < 0) return GDN_ERR_INVALID_ARG;
      if ((pos_host[n] + 1) % shape->chunk == 0) resync = true;
    }
  }
  const DecLayout L = dec_layout(shape);
  if (!ws || !aligned(ws, kAlign) || ws_bytes < L.total) return GDN_ERR_WORKSPACE;
  if (N == 0) return GDN_OK;
  const Dims d = dims_of(shape);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  float* W = reinterpret_cast<float*>(at(ws, L.W));
  float* U = reinterpret_cast<float*>(at(ws, L.U));
  float* gamma = reinterpret_cast<float*>(at(ws, L.gamma));
  TokenArrays in{q, k, v, g, beta, N};
  Stages stg(stream, kDecodeStages);
  launch_reset_header(hdr, stream);  // error word and work-list flag of this call
  stg.count(1);

  DecodeWork dw{};
  dw.N = N;
  dw.slot = slot;
  dw.slots = cache->slots;
  dw.s_run = cache->s_run;
  dw.c_run = cache->c_run;
  dw.tail_k = cache->tail_k;
  dw.tail_v = cache->tail_v;
  dw.tail_g = cache->tail_g;
  dw.tail_beta = cache->tail_beta;
  dw.pos = cache->pos;
  dw.o = o;
  dw.no_resync = resync ? 0 : 1;
  launch_decode(d, in, dw, hdr, stream);
  stg.mark(1);

  if (resync) {
    const int64_t tail_rows = (int64_t)cache->slots * d.C;
    TokenArrays tail{nullptr, cache->tail_k, cache->tail_v, cache->tail_g, cache->tail_beta, tail_rows};
    PrepWork pw{};
    pw.chunks = nullptr;
    pw.n_items = N;
    pw.slot = slot;
    pw.pos = cache->pos;
    pw.slots = cache->slots;
    ChainWork cw{};
    cw.seqs = nullptr;
    cw.N = N;
    cw.slot = slot;
    cw.pos = cache->pos;
    cw.s_bnd = cache->s_bnd;
    cw.s_run = cache->s_run;
    cw.c_run = cache->c_run;
    cw.slots = cache->slots;
    cw.n_chunks = N;
    cw.n_tokens = tail_rows;
    if (launch_resync_fused(d, tail, pw, cw, hdr, stream)) {
      stg.mark(1);
    } else {
      launch_prep(d, tail, pw, W, U, gamma, hdr, stream);
      launch_chain(d, cache->tail_k, W, U, gamma, cw, hdr, stream);
      stg.mark(2);
    }
  } else {
    stg.mark(0);
  }

  launch_advance(N, slot, cache->slots, cache->pos, hdr, stream);
  stg.mark(1);
  return finish(stream);
}

}  // namespace

extern "C" {

int gdn_cpr_version(void) { return GDN_VERSION_NUM; }

const char* gdn_cpr_status_string(gdn_status s) {
  switch (s) {
    case GDN_OK: return "ok";
    case GDN_ERR_INVALID_ARG: return "invalid argument";
    case GDN_ERR_UNSUPPORTED: return "unsupported configuration";
    case GDN_ERR_CUDA: return "CUDA error";
    case GDN_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case GDN_ERR_DEVICE: return "device-side error recorded";
  }
  return "unknown status";
}

gdn_status gdn_cpr_workspace_size(const gdn_cpr_shape* shape, gdn_mode mode,
                                  const int32_t* cu_seqlens_host, size_t* bytes) {
  if (!bytes) return GDN_ERR_INVALID_ARG;
  gdn_status rc = check_shape(shape);
  if (rc != GDN_OK) return rc;
  if (mode == GDN_MODE_DECODE) {
    *bytes = dec_layout(shape).total;
    return GDN_OK;
  }
  int64_t n_chunks = 0;
  uint32_t hash = 0;
  rc = scan_cu(shape, cu_seqlens_host, &n_chunks, &hash);
  if (rc != GDN_OK) return rc;
  switch (mode) {
    case GDN_MODE_PREFILL: *bytes = fwd_layout(shape, n_chunks, true).total; return GDN_OK;
    case GDN_MODE_FWD: *bytes = fwd_layout(shape, n_chunks, false).total; return GDN_OK;
    case GDN_MODE_BWD: *bytes = bwd_layout(shape, n_chunks).total; return GDN_OK;
    case GDN_MODE_CONTINUE: {
      std::vector<int32_t> vcu;
      rc = virtual_cu(shape, cu_seqlens_host, nullptr, vcu);
      if (rc != GDN_OK) return rc;
      gdn_cpr_shape sv = *shape;
      sv.total_tokens = vcu[(size_t)shape->num_seqs];
      int64_t vchunks = 0;
      uint32_t vhash = 0;
      rc = scan_cu(&sv, vcu.data(), &vchunks, &vhash);
      if (rc != GDN_OK) return rc;
      *bytes = cont_layout(&sv, vchunks).total;
      return GDN_OK;
    }
    default: return GDN_ERR_INVALID_ARG;
  }
}

gdn_status gdn_cpr_prefill(const gdn_cpr_shape* shape, const void* q, const void* k,
                           const void* v, const float* g, const float* beta,
                           const float* state_in, const int32_t* cu_seqlens_dev,
                           const int32_t* cu_seqlens_host, void* o, float* state_out,
                           const gdn_cpr_cache* cache_out, const int32_t* slot_of_seq, void* ws,
                           size_t ws_bytes, gdn_stream_t stream) {
  NvtxRange nvtx("gdn_cpr_prefill");
  return run_forward(shape, q, k, v, g, beta, state_in, cu_seqlens_dev, cu_seqlens_host, o,
                     state_out, cache_out, slot_of_seq, nullptr, ws, ws_bytes, stream);
}

gdn_status gdn_cpr_fwd(const gdn_cpr_shape* shape, const void* q, const void* k, const void* v,
                       const float* g, const float* beta, const float* state_in,
                       const int32_t* cu_seqlens_dev, const int32_t* cu_seqlens_host, void* o,
                       float* state_out, float* saved_bnd, void* ws, size_t ws_bytes,
                       gdn_stream_t stream) {
  NvtxRange nvtx("gdn_cpr_fwd");
  if (!saved_bnd) return GDN_ERR_INVALID_ARG;
  return run_forward(shape, q, k, v, g, beta, state_in, cu_seqlens_dev, cu_seqlens_host, o,
                     state_out, nullptr, nullptr, saved_bnd, ws, ws_bytes, stream);
}

gdn_status gdn_cpr_decode_step(const gdn_cpr_shape* shape, const void* q, const void* k,
                               const void* v, const float* g, const float* beta,
                               const int32_t* slot, const gdn_cpr_cache* cache, void* o,
                               void* ws, size_t ws_bytes, gdn_stream_t stream) {
  NvtxRange nvtx("gdn_cpr_decode_step");
  return run_decode(shape, q, k, v, g, beta, slot, nullptr, cache, o, ws, ws_bytes, stream);
}

gdn_status gdn_cpr_decode_step_pos(const gdn_cpr_shape* shape, const void* q, const void* k,
                                   const void* v, const float* g, const float* beta,
                                   const int32_t* slot, const int32_t* pos_host,
                                   const gdn_cpr_cache* cache, void* o, void* ws, size_t ws_bytes,
                                   gdn_stream_t stream) {
  NvtxRange nvtx("gdn_cpr_decode_step_pos");
  if (!pos_host && shape && shape->num_seqs > 0) return GDN_ERR_INVALID_ARG;
  return run_decode(shape, q, k, v, g, beta, slot, pos_host, cache, o, ws, ws_bytes, stream);
}

gdn_status gdn_cpr_bwd(const gdn_cpr_shape* shape, const void* q, const void* k, const void* v,
                       const float* g, const float* beta, const float* state_in,
                       const int32_t* cu_seqlens_dev, const int32_t* cu_seqlens_host,
                       const float* saved_bnd, const void* dO, const float* dstate_out,
                       float* dq, float* dk, float* dv, float* dg, float* dbeta,
                       float* dstate_in, void* ws, size_t ws_bytes, gdn_stream_t stream) {
  NvtxRange nvtx("gdn_cpr_bwd");
  (void)state_in;  // its contribution reaches the backward through saved_bnd (chunk 0)
  gdn_status rc = check_shape(shape);
  if (rc != GDN_OK) return rc;
  int64_t n_chunks = 0;
  uint32_t hash = 0;
  rc = scan_cu(shape, cu_seqlens_host, &n_chunks, &hash);
  if (rc != GDN_OK) return rc;
  const int N = shape->num_seqs;
  const int64_t T = shape->total_tokens;
  if (T > 0 && (!ok_ptr(q, 16) || !ok_ptr(k, 16) || !ok_ptr(v, 16) || !ok_ptr(g, 4) ||
                !ok_ptr(beta, 4) || !ok_ptr(dO, 16) || !ok_ptr(dq, 16) || !ok_ptr(dk, 16) ||
                !ok_ptr(dv, 16) || !ok_ptr(dg, 4) || !ok_ptr(dbeta, 4)))
    return GDN_ERR_INVALID_ARG;
  if (n_chunks > 0 && !ok_ptr(saved_bnd, 16)) return GDN_ERR_INVALID_ARG;
  if (N > 0 && !ok_ptr(cu_seqlens_dev, 4)) return GDN_ERR_INVALID_ARG;
  if ((dstate_out && !aligned(dstate_out, 16)) || (dstate_in && !aligned(dstate_in, 16)))
    return GDN_ERR_INVALID_ARG;
  const BwdLayout L = bwd_layout(shape, n_chunks);
  if (!ws || !aligned(ws, kAlign) || ws_bytes < L.total) return GDN_ERR_WORKSPACE;
  if (N == 0) return GDN_OK;
  const Dims d = dims_of(shape);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  ChunkRec* chunks = reinterpret_cast<ChunkRec*>(at(ws, L.chunks));
  SeqRec* seqs = reinterpret_cast<SeqRec*>(at(ws, L.seqs));
  TokenArrays in{q, k, v, g, beta, T};
  Stages stg(stream, kBwdStages);
  launch_reset_header(hdr, stream);  // error word and work-list flag of this call
  stg.count(1);
  launch_worklist(cu_seqlens_dev, N, (int)T, d.C, n_chunks, hash, chunks, seqs, hdr, stream);
  stg.mark(1);
  launch_bwd(d, in, dO, chunks, seqs, N, n_chunks, T, saved_bnd, dstate_out, dstate_in,
             reinterpret_cast<float*>(at(ws, L.per_chunk)), reinterpret_cast<float*>(at(ws, L.dq_part)),
             reinterpret_cast<float*>(at(ws, L.dk_part)), dq, dk, dv, dg, dbeta, hdr, stage_mark,
             &stg, stream);
  return finish(stream);
}

void gdn_cpr_set_profile(gdn_cpr_profile* profile) { t_profile = profile; }

gdn_status gdn_cpr_prefill_continue(const gdn_cpr_shape* shape, const void* q, const void* k,
                                    const void* v, const float* g, const float* beta,
                                    const int32_t* cu_seqlens_dev, const int32_t* cu_seqlens_host,
                                    const int32_t* slot_dev, const int32_t* pos_host,
                                    const gdn_cpr_cache* cache, void* o, float* state_out, void* ws,
                                    size_t ws_bytes, gdn_stream_t stream) {
  NvtxRange nvtx("gdn_cpr_prefill_continue");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  gdn_status rc = check_shape(shape);
  if (rc != GDN_OK) return rc;
  int64_t n_chunks = 0;
  uint32_t hash = 0;
  rc = scan_cu(shape, cu_seqlens_host, &n_chunks, &hash);
  if (rc != GDN_OK) return rc;
  const int N = shape->num_seqs;
  const int64_t T = shape->total_tokens;
  if (!cache) return GDN_ERR_INVALID_ARG;
  rc = check_cache(cache);
  if (rc != GDN_OK) return rc;
  if (T > 0 && (!ok_ptr(q, 16) || !ok_ptr(k, 16) || !ok_ptr(v, 16) || !ok_ptr(g, 4) ||
                !ok_ptr(beta, 4) || !ok_ptr(o, 16)))
    return GDN_ERR_INVALID_ARG;
  if (N > 0 && (!ok_ptr(cu_seqlens_dev, 4) || !ok_ptr(slot_dev, 4) || !pos_host)) return GDN_ERR_INVALID_ARG;
  if (state_out && !aligned(state_out, 16)) return GDN_ERR_INVALID_ARG;
  std::vector<int32_t> vcu_h;
  rc = virtual_cu(shape, cu_seqlens_host, pos_host, vcu_h);
  if (rc != GDN_OK) return rc;
  gdn_cpr_shape sv = *shape;
  sv.total_tokens = vcu_h[(size_t)N];
  int64_t vchunks = 0;
  uint32_t vhash = 0;
  rc = scan_cu(&sv, vcu_h.data(), &vchunks, &vhash);
  if (rc != GDN_OK) return rc;
  const ContLayout L = cont_layout(&sv, vchunks);
  if (!ws || !aligned(ws, kAlign) || ws_bytes < L.total) return GDN_ERR_WORKSPACE;
  if (N == 0) return GDN_OK;

  const Dims d = dims_of(shape);
  const int64_t vT = sv.total_tokens;
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  ChunkRec* chunks = reinterpret_cast<ChunkRec*>(at(ws, L.f.chunks));
  SeqRec* seqs = reinterpret_cast<SeqRec*>(at(ws, L.f.seqs));
  float* W = reinterpret_cast<float*>(at(ws, L.f.W));
  float* U = reinterpret_cast<float*>(at(ws, L.f.U));
  float* gamma = reinterpret_cast<float*>(at(ws, L.f.gamma));
  float* bnd = reinterpret_cast<float*>(at(ws, L.f.bnd));
  int32_t* vcu = reinterpret_cast<int32_t*>(at(ws, L.vcu));
  int32_t* rlen = reinterpret_cast<int32_t*>(at(ws, L.rlen));
  int32_t* base = reinterpret_cast<int32_t*>(at(ws, L.base));
  void* vo = at(ws, L.o);
  TokenArrays in{q, k, v, g, beta, T};
  TokenArrays vin{at(ws, L.q), at(ws, L.k), at(ws, L.v), reinterpret_cast<const float*>(at(ws, L.g)),
                  reinterpret_cast<const float*>(at(ws, L.beta)), vT};

  Stages stg(st, kContStages);
  launch_reset_header(hdr, st);  // error word and work-list flag of this call
  stg.count(1);
  launch_continue_prep(cu_seqlens_dev, slot_dev, cache->pos, cache->slots, N, d.C, vcu, rlen, base, hdr, st);
  launch_worklist(vcu, N, (int)vT, d.C, vchunks, vhash, chunks, seqs, hdr, st);
  launch_continue_gather(d, in, cu_seqlens_dev, vcu, rlen, slot_dev, N, vT, *cache, vin, hdr, st);
  stg.mark(3);

  PrepWork pw{};
  pw.chunks = chunks;
  pw.n_items = vchunks;
  launch_prep(d, vin, pw, W, U, gamma, hdr, st);
  stg.mark(vchunks > 0 ? 1 : 0);

  IntraWork iw{};
  iw.chunks = chunks;
  iw.seqs = seqs;
  iw.n_seqs = N;
  iw.n_chunks = vchunks;
  iw.bnd = bnd;
  iw.o = vo;
  iw.state_out = state_out;
  iw.cache_run = cache->s_run;
  iw.cache_c_run = cache->c_run;
  iw.cache_slots = cache->slots;
  iw.slot_of_seq = slot_dev;
  iw.skip = rlen;  // the tail is already in the cache's running state
  iw.run_state = cache->s_run;
  iw.run_c = cache->c_run;
  iw.run_slot = slot_dev;
  iw.part = 1;  // chunks that start from the cache's running state, before anything writes it
  launch_intra(d, vin, iw, hdr, st);
  ChainWork cw{};
  cw.seqs = seqs;
  cw.N = N;
  cw.n_chunks = vchunks;
  cw.n_tokens = vT;
  cw.state_in = cache->s_bnd;
  cw.state_in_slot = slot_dev;
  cw.bnd = bnd;
  cw.state_out = state_out;
  cw.cache_bnd = cache->s_bnd;
  cw.cache_run = cache->s_run;
  cw.cache_c_run = cache->c_run;
  cw.cache_slots = cache->slots;
  cw.slot_of_seq = slot_dev;
  cw.bnd_in_place = true;
  cw.bnd_skip = rlen;
  launch_chain(d, vin.k, W, U, gamma, cw, hdr, st);
  stg.mark(vchunks > 0 ? 2 : 1);  // intra part 1 and the chain

  iw.part = 2;
  launch_intra(d, vin, iw, hdr, st);
  stg.mark(vchunks > 0 ? 1 : 0);

  launch_tail_fill(d, vin, seqs, N, slot_dev, cache->slots, cache->tail_k, cache->tail_v, cache->tail_g,
                   cache->tail_beta, cache->pos, base, rlen, hdr, st);
  launch_continue_scatter(d, cu_seqlens_dev, vcu, rlen, N, T, vT, vo, o, hdr, st);
  stg.mark(2);
  return finish(st);
}

gdn_status gdn_cpr_running_state(const gdn_cpr_shape* shape, const gdn_cpr_cache* cache,
                                 const int32_t* slots_dev, int32_t n, float* out, gdn_stream_t stream) {
  NvtxRange nvtx("gdn_cpr_running_state");
  gdn_status rc = check_shape(shape);
  if (rc != GDN_OK) return rc;
  rc = check_cache(cache);
  if (rc != GDN_OK) return rc;
  if (n < 0 || (!slots_dev && n > cache->slots)) return GDN_ERR_INVALID_ARG;
  if (n == 0) return GDN_OK;
  if (!ok_ptr(out, 16) || (slots_dev && !aligned(slots_dev, 4))) return GDN_ERR_INVALID_ARG;
  launch_running_state(shape->d_k, shape->h_v, cache->s_run, cache->c_run, cache->slots, slots_dev, n, out,
                       static_cast<cudaStream_t>(stream));
  return finish(static_cast<cudaStream_t>(stream));
}

void gdn_cpr_test_wait_timeout(int32_t calls) { t_wait_fault = calls > 0 ? calls : 0; }

gdn_status gdn_cpr_get_device_error(const void* ws, gdn_stream_t stream, int32_t* code) {
  if (!ws || !code) return GDN_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return GDN_ERR_CUDA;
  int32_t c = 0;
  if (cudaMemcpy(&c, ws, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return GDN_ERR_CUDA;
  *code = c;
  return c == 0 ? GDN_OK : GDN_ERR_DEVICE;
}

}  // extern "C"
