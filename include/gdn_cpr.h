/*
 * gdn_cpr.h -- C ABI of the CPR Gated DeltaNet library (sm_103a, one GPU).
 *
 * The operator (Gated DeltaNet; IsoExec page "IsoExec: SkyRLにおけるトレーナーと推論の
 * ミスマッチを解消する", section "Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet"), per
 * (sequence, value head) with an fp32 state S of d_v x d_k:
 *
 *     S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,      o_t = S_t q_t.
 *
 * CPR, as that section describes it, keeps this recurrence as the main computation but
 * evaluates it in parallel across chunks of C tokens, and resynchronises the decode
 * state every C tokens.  Concretely, in this library:
 *   - a boundary pass computes the state S^(j) before every chunk j (chunks aligned to
 *     each sequence's own first token) with the chunk (WY/UT) form, sequentially in j;
 *   - every chunk then runs the token recurrence from its own S^(j), all chunks at once;
 *   - decode runs the same token step on a running state and, whenever a chunk's C-th
 *     token has been appended, replaces that running state by the next boundary state,
 *     computed by the same boundary code on the cached chunk.
 * Every mode uses one token-step routine and one boundary routine with fixed reduction
 * orders, so prefill, trainer forward and decode give bit-identical o and states, for any
 * batch size, packing or slot assignment.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Layouts (row-major, densely packed; T = total tokens, N = sequences or decode slots):
 *     q, k        [T, H_qk, d_k]   in_dtype
 *     v           [T, H_v,  d_v]   in_dtype
 *     g, beta     [T, H_v]         fp32 (g is the log decay: the step multiplies S by exp(g))
 *     o           [T, H_v,  d_v]   out_dtype
 *     states      [N, H_v, d_v, d_k] fp32 (row i of S is value dim i; o = S q)
 *     cu_seqlens  [N + 1] int32, cu_seqlens[0] = 0, non-decreasing, cu_seqlens[N] = T
 * Grouped heads: value head h reads query/key head h / (H_v / H_qk).  No scale is applied
 * to q.  Sequences of length 0 are allowed (state_out = state_in, bit for bit).
 *
 * Supported configurations ("claims"; anything else returns GDN_ERR_UNSUPPORTED before any
 * work is queued, in the spirit of the IsoExec contract's topology claims on the
 * hegai.media page, section "Что именно объединяет IsoExec"):
 *     d_k == d_v in {32, 64, 128};  chunk C in {16, 32, 64};  H_v % H_qk == 0;
 *     in_dtype in {GDN_F32, GDN_BF16};  out_dtype in {GDN_F32, GDN_BF16};
 *     every tensor pointer 16-byte aligned (g, beta: 4-byte).
 *
 * Ownership: the caller allocates and owns every buffer, including the workspace.  The
 * library allocates no device memory and keeps no mutable global state apart from the
 * optional per-thread hooks (gdn_cpr_set_profile, gdn_cpr_test_wait_timeout) and the
 * built-in scratch array of gdn_cpr_decode_step_noalloc.
 *
 * Execution: every call only queues work on `stream` and returns; nothing synchronises
 * except gdn_cpr_get_device_error.  Inputs must stay valid until the stream reaches the
 * queued work.  cu_seqlens_host must describe the same values as cu_seqlens_dev; it is
 * read on the host during the call (grid and workspace sizing) and not kept.
 *
 * Errors: argument errors are returned synchronously and nothing is queued.  Errors that
 * only the device can see (device cu_seqlens disagreeing with the host copy, a decode
 * slot out of range, a bounded wait that gave up) are recorded in an error word inside the
 * workspace; the affected kernels then skip their work (they never read or write out of
 * bounds), and gdn_cpr_get_device_error reports the code.  Each call clears the word
 * when it starts.  No kernel traps or asserts.
 */
#ifndef GDN_CPR_H
#define GDN_CPR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *gdn_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad sizes, bad cu_seqlens_host */
    GDN_ERR_UNSUPPORTED = 2, /* outside the supported configurations listed above */
    GDN_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
    GDN_ERR_WORKSPACE = 4,   /* workspace NULL, misaligned or smaller than required */
    GDN_ERR_DEVICE = 5       /* returned by gdn_cpr_get_device_error when the word is set */
} gdn_status;

/* Codes stored in the device error word (read back by gdn_cpr_get_device_error). */
typedef enum {
    GDN_DEVERR_NONE = 0,
    GDN_DEVERR_CU_SEQLENS = 1, /* device cu_seqlens disagree with cu_seqlens_host */
    GDN_DEVERR_SLOT = 2,       /* decode slot index outside [0, cache.slots) */
    GDN_DEVERR_POS = 3,        /* negative cache position */
    GDN_DEVERR_TIMEOUT = 4,    /* a bounded on-device wait gave up */
    GDN_DEVERR_BOUNDS = 5,     /* bounds-checked builds only (GDN_CHECKED): a work item's index
                                  range fell outside its buffer; the item was skipped */
    GDN_DEVERR_POS_HOST = 6    /* gdn_cpr_decode_step_pos: the host positions said no token
                                  completes a chunk, the cache says one does; step skipped */
} gdn_device_error;

typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

typedef enum {
    GDN_MODE_PREFILL = 0, /* gdn_cpr_prefill */
    GDN_MODE_DECODE = 1,  /* gdn_cpr_decode_step */
    GDN_MODE_FWD = 2,     /* gdn_cpr_fwd */
    GDN_MODE_BWD = 3,     /* gdn_cpr_bwd */
    GDN_MODE_CONTINUE = 4 /* gdn_cpr_prefill_continue (upper bound over cache positions) */
} gdn_mode;

typedef struct {
    int32_t num_seqs;     /* N: sequences (prefill/fwd/bwd) or tokens this step (decode) */
    int32_t total_tokens; /* T: cu_seqlens[N] (prefill/fwd/bwd); N for decode */
    int32_t h_qk;         /* query/key heads */
    int32_t h_v;          /* value heads (state heads) */
    int32_t d_k;          /* key dim */
    int32_t d_v;          /* value dim */
    int32_t chunk;        /* C */
    gdn_dtype in_dtype;   /* q, k, v */
    gdn_dtype out_dtype;  /* o */
} gdn_cpr_shape;

/* Decode cache: everything needed to continue a sequence bit-exactly (also the full
 * checkpoint of a decoding sequence: copy it out and back to resume).  All arrays are
 * caller-owned device memory, indexed by slot.
 *   s_run     [slots, H_v, d_v, d_k] fp32   running state (recurrent since the last boundary),
 *                                             held scaled: the state is c_run * s_run
 *   c_run     [slots, H_v] fp32           its scale (1 right after a boundary; see token_step)
 *   s_bnd     [slots, H_v, d_v, d_k] fp32   boundary state before the current chunk
 *   tail_k    [slots, C, H_qk, d_k]  in_dtype  keys of the current, unfinished chunk
 *   tail_v    [slots, C, H_v,  d_v]  in_dtype  values of the current chunk
 *   tail_g    [slots, C, H_v]        fp32
 *   tail_beta [slots, C, H_v]        fp32
 *   pos       [slots] int32          tokens consumed so far by the slot's sequence          */
typedef struct {
    float *s_run;
    float *c_run;
    float *s_bnd;
    void *tail_k;
    void *tail_v;
    float *tail_g;
    float *tail_beta;
    int32_t *pos;
    int32_t slots;
} gdn_cpr_cache;

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int gdn_cpr_version(void);

/* Static, human-readable name of a status code. */
const char *gdn_cpr_status_string(gdn_status s);

/* Bytes of workspace the given mode needs for this shape.  cu_seqlens_host [N+1] is
 * required for PREFILL, FWD and BWD (the size depends on the number of chunks,
 * sum over sequences of ceil(L/C)) and ignored for DECODE.  The workspace must be
 * 256-byte aligned.  Returns GDN_ERR_INVALID_ARG / GDN_ERR_UNSUPPORTED like the calls. */
gdn_status gdn_cpr_workspace_size(const gdn_cpr_shape *shape, gdn_mode mode,
                                  const int32_t *cu_seqlens_host, size_t *bytes);

/* Prefill (rollout prefill; IsoExec page section "Chunkwise-Parallel Recurrent (CPR)
 * Gated DeltaNet": the recurrence evaluated in parallel across chunks).
 *   q, k, v, g, beta    inputs, layouts above (device)
 *   state_in            [N, H_v, d_v, d_k] fp32 or NULL for zero (device)
 *   cu_seqlens_dev/host the same N+1 offsets, on the device and on the host
 *   o                   output [T, H_v, d_v] in out_dtype (device)
 *   state_out           NULL or [N, H_v, d_v, d_k]: the state decode continues from --
 *                       the boundary state S^(L/C) if L % C == 0, else the token
 *                       recurrence from S^(floor(L/C)) through the last L % C tokens
 *   cache_out           NULL or a decode cache to initialise for these sequences:
 *                       s_run = state_out, s_bnd = S^(floor(L/C)), tail = the last L % C
 *                       tokens, pos = L, at slot slot_of_seq[n] (NULL: slot n)
 *   slot_of_seq         NULL or [N] int32 device array of distinct slots
 *   ws, ws_bytes        workspace of gdn_cpr_workspace_size(GDN_MODE_PREFILL) bytes  */
gdn_status gdn_cpr_prefill(const gdn_cpr_shape *shape, const void *q, const void *k,
                           const void *v, const float *g, const float *beta,
                           const float *state_in, const int32_t *cu_seqlens_dev,
                           const int32_t *cu_seqlens_host, void *o, float *state_out,
                           const gdn_cpr_cache *cache_out, const int32_t *slot_of_seq, void *ws,
                           size_t ws_bytes, gdn_stream_t stream);

/* One decode token for each of N slots (rollout decode; IsoExec page section
 * "Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet": the hidden state is resynchronised
 * every C tokens).  shape->num_seqs = shape->total_tokens = N.
 *   q, k [N, H_qk, d_k], v [N, H_v, d_v], g, beta [N, H_v]: this step's token per slot
 *   slot [N] int32 device: distinct cache slots (out of range -> device error, skipped)
 *   cache               updated in place: s_run stepped, token appended to the tail, pos+1;
 *                       when pos+1 is a multiple of C the boundary state is advanced over
 *                       the completed chunk and s_run is replaced by it
 *   o [N, H_v, d_v]     output
 * The launch configuration depends only on N and the shape, and the resync decision is
 * taken on the device from pos, so a step can be captured in a CUDA graph once the
 * workspace and pointers are fixed.                                                     */
gdn_status gdn_cpr_decode_step(const gdn_cpr_shape *shape, const void *q, const void *k,
                               const void *v, const float *g, const float *beta,
                               const int32_t *slot, const gdn_cpr_cache *cache, void *o,
                               void *ws, size_t ws_bytes, gdn_stream_t stream);

/* gdn_cpr_decode_step for callers that know the slots' positions on the host (a serving
 * scheduler tracks every sequence's length): pos_host [N] is the host copy of
 * cache->pos[slot[n]] before this step, read during the call and not kept.  When no token of
 * the step completes a chunk ((pos_host[n] + 1) % C != 0 for every n), the resynchronisation
 * kernels are not launched at all -- two launches fewer per step; otherwise the call is
 * exactly gdn_cpr_decode_step.  Results and bits are those of gdn_cpr_decode_step.  The
 * claim is checked on the device: if a slot's cache position does complete a chunk after
 * all, the whole step is skipped (nothing in the cache changes, o is not written) and the
 * workspace's error word reads GDN_DEVERR_POS_HOST.  A negative pos_host entry returns
 * GDN_ERR_INVALID_ARG.  The launch sequence depends on pos_host, so a CUDA graph captured
 * with it is valid only for steps at those positions.                                     */
gdn_status gdn_cpr_decode_step_pos(const gdn_cpr_shape *shape, const void *q, const void *k,
                                   const void *v, const float *g, const float *beta,
                                   const int32_t *slot, const int32_t *pos_host,
                                   const gdn_cpr_cache *cache, void *o, void *ws, size_t ws_bytes,
                                   gdn_stream_t stream);

/* Trainer forward (case "trainer_fwd" next to "engine_prefill" on the IsoExec page,
 * section on contract structure).  Identical arithmetic to gdn_cpr_prefill -- o and
 * state_out are bit-identical -- and additionally saves the boundary states:
 *   saved_bnd [sum_s ceil(L_s/C), H_v, d_v, d_k] fp32: the state before every chunk, chunks
 *             numbered in sequence order (chunk 0 of a sequence holds its state_in).     */
gdn_status gdn_cpr_fwd(const gdn_cpr_shape *shape, const void *q, const void *k, const void *v,
                       const float *g, const float *beta, const float *state_in,
                       const int32_t *cu_seqlens_dev, const int32_t *cu_seqlens_host, void *o,
                       float *state_out, float *saved_bnd, void *ws, size_t ws_bytes,
                       gdn_stream_t stream);

/* Trainer backward (IsoExec page, CPR timing table row "Trainer Fwd+Bwd").  Gradient of
 * loss = <dO, o> + <dstate_out, state_out> with respect to every input, where o and
 * state_out are gdn_cpr_fwd's outputs.  Uses saved_bnd from gdn_cpr_fwd on the same
 * inputs.  Reverse chain over chunks for the boundary adjoints, then every chunk in
 * parallel; grouped-head dq/dk are summed over the value heads of a group in ascending
 * order; no atomics, so results are deterministic.
 *   dO [T, H_v, d_v] out_dtype; dstate_out NULL (= 0) or [N, H_v, d_v, d_k] fp32
 *   dq, dk [T, H_qk, d_k] fp32; dv [T, H_v, d_v] fp32; dg, dbeta [T, H_v] fp32
 *   dstate_in NULL or [N, H_v, d_v, d_k] fp32                                            */
gdn_status gdn_cpr_bwd(const gdn_cpr_shape *shape, const void *q, const void *k, const void *v,
                       const float *g, const float *beta, const float *state_in,
                       const int32_t *cu_seqlens_dev, const int32_t *cu_seqlens_host,
                       const float *saved_bnd, const void *dO, const float *dstate_out,
                       float *dq, float *dk, float *dv, float *dg, float *dbeta,
                       float *dstate_in, void *ws, size_t ws_bytes, gdn_stream_t stream);

/* Prefill continued from a decode cache at any position: chunked prefill, and decode of
 * several tokens per sequence at once (the IsoExec page's CPR section: decode continues the
 * same recurrence and resynchronises every C tokens; this extends a cached sequence by any
 * number of tokens with the bits of one prefill of the whole sequence).  Sequence i appends
 * L_i = cu_seqlens[i+1] - cu_seqlens[i] tokens to cache slot slot_dev[i], whose position
 * pos_host[i] (host copy of cache->pos[slot_dev[i]]; checked on the device, a mismatch sets
 * GDN_DEVERR_CU_SEQLENS and nothing runs) may lie inside a chunk.  The r_i = pos_host[i] % C
 * tokens of the slot's tail are replayed with the new ones from the slot's boundary state,
 * so that every output and the updated cache are bit-identical to a single gdn_cpr_prefill
 * of the whole sequence (and to gdn_cpr_decode_step token by token).
 *   q, k, v, g, beta, o  the new tokens only, laid out as for gdn_cpr_prefill
 *   slot_dev [N] int32 device, distinct slots; cache  updated in place: s_run, s_bnd, tail,
 *                        pos += L_i
 *   state_out            NULL or [N, H_v, d_v, d_k]: the state after the last token
 *   ws, ws_bytes         gdn_cpr_workspace_size(GDN_MODE_CONTINUE, cu_seqlens_host) bytes
 * Argument errors (NULL or misaligned pointers, negative positions) are returned; a slot
 * out of range on the device sets GDN_DEVERR_SLOT.                                        */
gdn_status gdn_cpr_prefill_continue(const gdn_cpr_shape *shape, const void *q, const void *k,
                                    const void *v, const float *g, const float *beta,
                                    const int32_t *cu_seqlens_dev, const int32_t *cu_seqlens_host,
                                    const int32_t *slot_dev, const int32_t *pos_host,
                                    const gdn_cpr_cache *cache, void *o, float *state_out, void *ws,
                                    size_t ws_bytes, gdn_stream_t stream);

/* The explicit running state of decode cache slots (the state decode continues from, as
 * gdn_cpr_prefill returns it in state_out): out[i] = c_run[s] * s_run[s] for s = slots_dev[i],
 * every value head, one round-to-nearest fp32 product per element -- the same product the
 * kernels use when a scaled running state leaves them as state_out, so a cache read back
 * here equals the state_out of the same sequence bit for bit.  (IsoExec page, section
 * "Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet": decode continues the recurrence on a
 * running state; the cache holds it as c_run * s_run, see gdn_cpr_cache.)
 *   shape      only h_v, d_k = d_v (and the configuration checks) are used
 *   cache      the decode cache to read (device)
 *   slots_dev  [n] int32 device slot indices, or NULL for slots 0 .. n-1 (n <= cache->slots)
 *   out        [n, H_v, d_v, d_k] fp32 device, 16-byte aligned
 * Queues one kernel on `stream`.  A slot index outside [0, cache->slots) on the device gives
 * an all-NaN block for that entry.  Argument errors are returned and nothing is queued. */
gdn_status gdn_cpr_running_state(const gdn_cpr_shape *shape, const gdn_cpr_cache *cache,
                                 const int32_t *slots_dev, int32_t n, float *out,
                                 gdn_stream_t stream);

/* Numerical-policy identity (IsoExec pages, section on the structure of the execution
 * contract, item "Identities": SHA-256 digests by which trainer and rollout engine check
 * that they run the same verified numerical policy).  Writes into digest[32] the SHA-256
 * (FIPS 180-4) of a canonical text listing every choice that decides the bits of this
 * library's results for the given shape: d_k, d_v, chunk length, input and output dtypes,
 * the boundary path (tensor cores with split-bf16 operands, or fp32 SIMT), the reduction
 * orders of the token step, the triangular solve and the cumulative sum, the exponential,
 * the rounding of the output and the library version.  The number of sequences, tokens
 * and heads do not enter it: shapes whose results are bit-identical share a digest.
 * When text is non-NULL it also receives that text, NUL-terminated and truncated to
 * text_len bytes.  Host only, no GPU work.  Returns GDN_ERR_INVALID_ARG for a NULL shape
 * or digest and GDN_ERR_UNSUPPORTED / GDN_ERR_INVALID_ARG for shapes the calls reject.
 * This library's own addition: the pages name the digests but define no content.     */
gdn_status gdn_cpr_policy_digest(const gdn_cpr_shape *shape, unsigned char digest[32], char *text,
                                 size_t text_len);

/* Optional profiling hook (per calling thread; NULL disables it, the default).  While set,
 * every entry point called from this thread records events[i] (cudaEvent_t handles created
 * by the caller) on its stream at its stage boundaries -- events[0] before its first
 * kernel, events[s] after stage s -- for as many stages as it has, up to n_events, and
 * adds the number of kernels it launched to *kernels.  Stages:
 *   prefill / fwd : 1 work list, 2 boundary pre-pass, 3 boundary chain, 4 intra-chunk
 *                   recurrence, 5 cache tail (prefill with a cache only)
 *   decode_step   : 1 token step, 2 resync (pre-pass and boundary step), 3 position advance
 *   bwd           : see gdn_cpr_bwd's stages in the implementation notes
 * The structure must stay valid while set.  Has no effect on results.                   */
typedef struct {
    void *events[16];   /* cudaEvent_t */
    int32_t n_events;   /* how many of events[] are valid */
    int32_t stages;     /* set by each call: how many stage events it recorded (incl. [0]) */
    int64_t kernels;    /* incremented by each call by the kernels it launched */
} gdn_cpr_profile;

void gdn_cpr_set_profile(gdn_cpr_profile *profile);

/* Size of the built-in device scratch used by gdn_cpr_decode_step_noalloc (64 MiB). */
#define GDN_CPR_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/* gdn_cpr_decode_step without a caller-provided workspace, for callers that cannot
 * allocate device memory (a serving loop whose memory is reserved up front by another
 * allocator, code that must not call cudaMalloc while other GPU work is captured or
 * replayed, or a plain C host with no device allocator).  The IsoExec pages have no
 * counterpart: this is a deployment convenience, not part of CPR.
 *   Arguments, results and bits are exactly those of gdn_cpr_decode_step; only the
 *   workspace differs.  It lives in one file-scope device array of
 *   GDN_CPR_NOALLOC_SCRATCH_BYTES that every GPU which loads this library's module holds
 *   until the process exits.  The call itself allocates nothing (no cudaMalloc/cudaFree).
 *   Limit: the decode workspace of the shape (gdn_cpr_workspace_size with
 *   GDN_MODE_DECODE) must fit the array -- about 1000 (token, value head) pairs per step at
 *   d = 128, C = 64 (e.g. 31 slots x 32 heads); larger requests return GDN_ERR_WORKSPACE
 *   and queue nothing.
 *   The first call on a device looks up the array's device address (with that device
 *   current); make that first call before capturing any stream into a CUDA graph.  The
 *   address is kept with the identity of the context it belongs to; after a device reset
 *   the next call looks it up again (and is again a first call in that sense).
 *   Device-side errors of these calls (a slot out of range, ...) are recorded in the
 *   array's own error word: read them with gdn_cpr_noalloc_device_error.
 *   Every call on a device shares the array and leaves its contents behind; the step
 *   clears what must start at zero.  Calls that overlap on the GPU (other streams, other
 *   threads, concurrent graph replays) race on the array: serialise them.               */
gdn_status gdn_cpr_decode_step_noalloc(const gdn_cpr_shape *shape, const void *q, const void *k,
                                       const void *v, const float *g, const float *beta,
                                       const int32_t *slot, const gdn_cpr_cache *cache, void *o,
                                       gdn_stream_t stream);

/* Synchronises `stream`, then reads the device error word of the built-in scratch array
 * of the current device, which gdn_cpr_decode_step_noalloc uses as its workspace: the
 * device-side error (slot out of range, negative position, a bounded wait that gave up) of
 * the last no-alloc call on this device, as gdn_cpr_get_device_error reports it for a
 * caller-provided workspace.  Returns GDN_OK when the word is clear, GDN_ERR_DEVICE with
 * *code set when it is not, GDN_ERR_CUDA if the sync or read fails.  Allocates nothing.  */
gdn_status gdn_cpr_noalloc_device_error(gdn_stream_t stream, int32_t *code);

/* Test hook of the failure path (per calling thread; off by default): the next `calls`
 * prefill or trainer-forward calls from this thread whose boundary pass runs on tensor
 * cores make one CTA of the boundary chain wait, before it issues any copy or MMA, on a
 * barrier phase that nothing completes.  Its bounded wait (a short poll limit here) gives
 * up, the CTA records GDN_DEVERR_TIMEOUT in the workspace's error word, frees its tensor
 * memory and exits, so gdn_cpr_get_device_error reports the timeout and the context stays
 * usable.  The outputs of such a call are not valid.  calls <= 0 switches it off.       */
void gdn_cpr_test_wait_timeout(int32_t calls);

/* Synchronises `stream`, then reads the device error word of `ws` (the workspace of the
 * last call queued with it) into *code (a gdn_device_error).  Returns GDN_OK when the
 * word is clear, GDN_ERR_DEVICE when it is set, GDN_ERR_CUDA if the sync or copy fails. */
gdn_status gdn_cpr_get_device_error(const void *ws, gdn_stream_t stream, int32_t *code);

#ifdef __cplusplus
}
#endif

#endif /* GDN_CPR_H */
