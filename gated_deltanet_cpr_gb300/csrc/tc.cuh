// tc.cuh -- 5th-generation tensor-core (tcgen05) building blocks for sm_103a, written as
// inline PTX: tensor-memory (TMEM) allocation, single-thread MMA issue with fp32
// accumulation in TMEM, commit to an mbarrier, TMEM <-> register moves, bulk async copies,
// and mbarrier waits with an iteration limit (a wait that gives up reports it instead of
// hanging).
//
// Image layout used throughout: bf16, no swizzle.  A tile of R rows x K columns is stored as
// 8x8 "core matrices" (8 rows x 16 bytes, 128 contiguous bytes); the K/8 core matrices of one
// 8-row group are contiguous, and 8-row groups follow each other:
//     byte(r, k) = (r / 8) * (K / 8) * 128 + (k / 8) * 128 + (r % 8) * 16 + (k % 8) * 2.
// Read K-major it is an operand with M (or N) = R (leading-dimension offset 128 B, stride-
// dimension offset K/8 * 128 B; a step over 16 of K advances the start address by 256 B);
// read MN-major (the instruction descriptor's transpose bit) it is the transposed operand,
// with M (or N) = K and K = R (see Opnd).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// byte offset of element (r, k) in an R x K bf16 K-major no-swizzle tile
__device__ __forceinline__ uint32_t kmajor_off(int r, int k, int K) {
  return (uint32_t)((r >> 3) * (K >> 3) * 128 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2);
}

// Work index q over an R x K tile split into 16-byte pieces (8 bf16), ordered so that 8
// consecutive q fill one 128-byte core matrix (consecutive rows of an 8-row group): stores
// by neighbouring threads then hit different shared-memory banks.
__device__ __forceinline__ void kmajor_piece(int q, int K, int& r, int& k0) {
  const int kp = K / 8;
  r = (q / (8 * kp)) * 8 + (q & 7);
  k0 = ((q >> 3) % kp) * 8;
}

// Shared-memory matrix descriptor (no swizzle): start address, leading-dimension byte
// offset (between core matrices adjacent along K), stride-dimension byte offset (between
// 8-row groups), descriptor version 1 at bits 46-47, layout type 0 (no swizzle).
__device__ __forceinline__ uint64_t make_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1u << 46;
  return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major, dense.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// The same with the A (bit 15) and / or B (bit 16) operand read MN-major
constexpr uint32_t IDESC_A_MN = 1u << 15, IDESC_B_MN = 1u << 16;

// An MMA operand in shared memory: a split image pair (hi, lo; lo unused where the operand is
// exact) and how the descriptor walks it.  K-major: the layout above, rows along M (or N),
// K = the image's columns.  MN-major: the same bytes read as their transpose, so that an
// image with R rows and W columns serves as an operand with M (or N) = W and K = R (core
// matrices adjacent along M or N are 128 B apart, along K W/8 * 128 B); its descriptors
// advance by two 8-row groups per 16 of K.
struct Opnd {
  uint32_t hi, lo, lbo, sbo, kstep;
};
__device__ __forceinline__ Opnd opnd_k(uint32_t hi, uint32_t lo, int K) {
  return Opnd{hi, lo, 128u, (uint32_t)K * 16u, 256u};
}
__device__ __forceinline__ Opnd opnd_mn(uint32_t hi, uint32_t lo, int W) {
  return Opnd{hi, lo, (uint32_t)W * 16u, 128u, (uint32_t)W * 32u};
}

// ---------------------------------------------------------------- mbarrier ----
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase with the given parity to complete, at most `limit` polls.  Returns
// false if it gave up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t limit = (1u << 22)) {
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// ------------------------------------------------------------- bulk copies ----
// global -> shared bulk copy (16-byte aligned addresses, size a multiple of 16), completing
// `bytes` transactions on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// A[i][s] = beta_i e^{G_i - G_s} for s < i, C = 64, all 256 threads of the block.  Rows i
// and 63 - i are paired (63 entries between them) and each pair gets 8 threads, so every
// thread forms 7 or 8 entries and no lane idles on the upper triangle.
__device__ __forceinline__ void decay_matrix64(float* A, int CPA, const float* bs, const float* Gs) {
  const int p = threadIdx.x >> 3, q = threadIdx.x & 7;  // row pair p = 0 .. 31
  for (int e = q; e < 63; e += 8) {
    const int i = e < p ? p : 63 - p;
    const int s = e < p ? e : e - p;
    A[i * CPA + s] = __fmul_rn(bs[i], expf(__fsub_rn(Gs[i], Gs[s])));
  }
}

// Asynchronous global -> shared copies (generic proxy) that a thread issues and later waits
// for: 16 bytes (both addresses 16-byte aligned) or 4 bytes.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// every copy this thread issued has landed (the CTA still needs a barrier to see the others')
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// shared -> global bulk copy (16-byte aligned addresses, size a multiple of 16) in the
// issuing thread's bulk group; the generic-proxy writes that made the source must be fenced
// (fence_proxy_async) and synchronised before it.  bulk_store_commit closes the group;
// bulk_wait_read waits until the thread's committed stores have read their sources (so the
// region can be written again), bulk_wait_all until they are complete.
__device__ __forceinline__ void bulk_s2g(void* gdst, const void* ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(smem_u32(ssrc)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_store_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Hint: bring the 128-byte line holding p into L2 (no register result, no wait).  A CTA that
// walks items issues these for its next item's operands, so that their loads hit L2.
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Generic-proxy shared-memory writes -> visible to the tensor core (async proxy).
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// -------------------------------------------------------------------- TMEM ----
// Whole warp: allocate `ncols` (power of two >= 32) TMEM columns, address written to *dst.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// One thread: D[tmem] (+)= A * B^T, M x N x 16, A and B from shared memory descriptors.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// One thread: D (+)= A_x B_y^T over K for one pair of split parts (x, y: hi or lo)
__device__ __forceinline__ void mma_part(uint32_t d, const Opnd& A, bool alo, const Opnd& B, bool blo, int K,
                                         uint32_t idesc, bool accumulate) {
  const uint32_t a = alo ? A.lo : A.hi, b = blo ? B.lo : B.hi;
  for (int kk = 0; kk < K / 16; ++kk)
    mma_bf16(d, make_desc(a + kk * A.kstep, A.lbo, A.sbo), make_desc(b + kk * B.kstep, B.lbo, B.sbo), idesc,
             (accumulate || kk > 0) ? 1u : 0u);
}
// D = A B^T from split parts, in this order: terms 3: A_hi B_hi + A_hi B_lo + A_lo B_hi;
// 2 (B exact): A_hi B + A_lo B; -2 (A exact): A B_hi + A B_lo; 1 (both exact): A B
__device__ __forceinline__ void mma_split(uint32_t d, const Opnd& A, const Opnd& B, int K, uint32_t idesc,
                                          int terms) {
  mma_part(d, A, false, B, false, K, idesc, false);
  if (terms == 3 || terms == -2) mma_part(d, A, false, B, true, K, idesc, true);
  if (terms == 3 || terms == 2) mma_part(d, A, true, B, false, K, idesc, true);
}
// One thread: arrive on `bar` once all previously issued MMAs of this thread complete.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// Warp: 16 consecutive fp32 columns of this thread's TMEM lane (32x32b shape).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// Warp: 32 consecutive fp32 columns of this thread's TMEM lane in one load instruction,
// waited for in the same statement (so no use of the values can be scheduled before the wait).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// Warp: 64 consecutive fp32 columns of this thread's TMEM lane in one load instruction,
// waited for in the same statement (so no use of the values can be scheduled before the wait).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float* v) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// TMEM address of column `col` in the lanes of this thread's warp (warp w of a 4-warp
// group owns lanes 32w .. 32w + 31).
__device__ __forceinline__ uint32_t tmem_lane_addr(uint32_t base, int warp, int col) {
  return base + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)col;
}

// fp32 -> (hi, lo) bf16 pair with hi + lo = x to about 16 bits: hi = rn(x), lo = rn(x - hi).
__device__ __forceinline__ void split_bf16(float x, __nv_bfloat16& hi, __nv_bfloat16& lo) {
  hi = __float2bfloat16_rn(x);
  lo = __float2bfloat16_rn(__fsub_rn(x, __bfloat162float(hi)));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void stsm_x4(uint32_t addr, const uint32_t (&r)[4]) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(r[0]), "r"(r[1]),
               "r"(r[2]), "r"(r[3])
               : "memory");
}

// dst = transpose of a shared-memory image: src is Ks rows x R columns (K-major, K = R),
// dst is R rows x Ks columns (K = Ks); 256 threads, R and Ks multiples of 16 (whole groups of
// four core matrices).  In the no-swizzle K-major layout an 8 x 8
// core matrix is 8 rows of 16 contiguous bytes, and core matrix (xb, yb) of dst is the
// transpose of core matrix (yb, xb) of src: each warp moves four at a time with ldmatrix
// .trans and stmatrix (eight 16-byte rows per matrix on each side, one wavefront each), in
// batches of 128 cores with a warp's loads before its stores.
__device__ __forceinline__ void transpose_image(unsigned char* dst, const unsigned char* src, int R, int Ks) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int xbs = R / 8, ncore = (Ks / 8) * xbs;
  const uint32_t sbo_s = (uint32_t)xbs * 128, sbo_d = (uint32_t)(Ks / 8) * 128;
  const uint32_t s0 = smem_u32(src) + (lane & 7) * 16, d0 = smem_u32(dst) + (lane & 7) * 16;
  for (int c0 = 0; c0 < ncore; c0 += 128) {  // batches of 128 cores
    uint32_t r[4][4], da[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {  // op k of this warp: cores c0 + 32 k + 4 warp .. + 3
      const int q = c0 + 32 * k + 4 * warp + (lane >> 3);  // this lane's row address is in matrix lane / 8
      if (c0 + 32 * k + 4 * warp < ncore) {
        const int yb = q / xbs, xb = q % xbs;
        ldsm_x4_trans(s0 + yb * sbo_s + xb * 128, r[k]);
        da[k] = d0 + xb * sbo_d + yb * 128;
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (c0 + 32 * k + 4 * warp < ncore) stsm_x4(da[k], r[k]);
  }
}

}  // namespace tc
}  // namespace gdn
