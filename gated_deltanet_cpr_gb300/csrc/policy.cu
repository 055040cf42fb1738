// policy.cu -- the numerical-policy identity of this library (IsoExec pages, section on
// the structure of the execution contract, item "Identities": SHA-256 digests with which
// trainer and rollout engine check that they run the same verified numerical policy).
//
// The digest is SHA-256 (FIPS 180-4) of a canonical text that lists every choice deciding
// the bits of this library's results for a shape: head dimension, chunk length, input and
// output dtypes, which boundary path runs (tensor cores with split-bf16 operands, or fp32
// SIMT), the reduction orders of the token step, the triangular solve and the cumulative
// sum, the exponential, and the rounding of the output.  Nothing that leaves the bits
// unchanged enters it (number of sequences, tokens or heads, the grouping of heads, the
// slot of a sequence), so every caller whose results are bit-identical gets the same
// digest.  Host code only.
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <string>

#include "../../include/gdn_cpr.h"
#include "launch.h"

namespace {

// ---- SHA-256, from the definition in FIPS 180-4 ----------------------------------------
// Round constants: the first 32 bits of the fractional parts of the cube roots of the first
// 64 primes; initial hash: the same of the square roots of the first 8 primes.  Both are
// derived here from that definition: a double estimate of the root, then an exact integer
// correction so that floor(frac(root) * 2^32) is exact.
struct Sha256Consts {
  uint32_t k[64], h0[8];
  Sha256Consts() {
    int primes[64], np = 0;
    for (int n = 2; np < 64; ++n) {
      bool p = true;
      for (int d = 2; d * d <= n; ++d)
        if (n % d == 0) {
          p = false;
          break;
        }
      if (p) primes[np++] = n;
    }
    for (int i = 0; i < 64; ++i) k[i] = frac_root(primes[i], 3);
    for (int i = 0; i < 8; ++i) h0[i] = frac_root(primes[i], 2);
  }
  // floor(frac(p^(1/e)) * 2^32) for e = 2 or 3: x = floor(p^(1/e) * 2^32) is the largest
  // integer with x^e <= p * 2^(32 e); the low 32 bits of x are the fractional bits.
  static uint32_t frac_root(int p, int e) {
    const double r = e == 2 ? sqrt((double)p) : cbrt((double)p);
    uint64_t x = (uint64_t)(r * 4294967296.0);
    // v^e <= p * 2^(32 e), exactly: v < 2^35 here, so v^3 < 2^105 fits in 128 bits
    auto pow_le = [&](uint64_t v) {
      const unsigned __int128 v2 = (unsigned __int128)v * v;
      if (e == 2) return v2 <= ((unsigned __int128)p << 64);
      return v2 * v <= ((unsigned __int128)p << 96);
    };
    while (!pow_le(x)) --x;
    while (pow_le(x + 1)) ++x;
    return (uint32_t)x;
  }
};

inline uint32_t rotr(uint32_t x, int n) { return (x >> n) | (x << (32 - n)); }

void sha256(const unsigned char* msg, size_t len, unsigned char out[32]) {
  static const Sha256Consts C;
  uint32_t h[8];
  for (int i = 0; i < 8; ++i) h[i] = C.h0[i];
  // message || 0x80 || zeros || 64-bit big-endian bit length, in 64-byte blocks
  const size_t total = ((len + 9 + 63) / 64) * 64;
  std::string m(reinterpret_cast<const char*>(msg), len);
  m.push_back((char)0x80);
  m.resize(total - 8, '\0');
  const uint64_t bits = (uint64_t)len * 8;
  for (int i = 7; i >= 0; --i) m.push_back((char)((bits >> (8 * i)) & 0xff));
  const unsigned char* p = reinterpret_cast<const unsigned char*>(m.data());
  for (size_t blk = 0; blk < total; blk += 64) {
    uint32_t w[64];
    for (int t = 0; t < 16; ++t)
      w[t] = ((uint32_t)p[blk + 4 * t] << 24) | ((uint32_t)p[blk + 4 * t + 1] << 16) |
             ((uint32_t)p[blk + 4 * t + 2] << 8) | (uint32_t)p[blk + 4 * t + 3];
    for (int t = 16; t < 64; ++t) {
      const uint32_t s0 = rotr(w[t - 15], 7) ^ rotr(w[t - 15], 18) ^ (w[t - 15] >> 3);
      const uint32_t s1 = rotr(w[t - 2], 17) ^ rotr(w[t - 2], 19) ^ (w[t - 2] >> 10);
      w[t] = w[t - 16] + s0 + w[t - 7] + s1;
    }
    uint32_t a = h[0], b = h[1], c = h[2], d = h[3], e = h[4], f = h[5], g = h[6], hh = h[7];
    for (int t = 0; t < 64; ++t) {
      const uint32_t S1 = rotr(e, 6) ^ rotr(e, 11) ^ rotr(e, 25);
      const uint32_t ch = (e & f) ^ (~e & g);
      const uint32_t t1 = hh + S1 + ch + C.k[t] + w[t];
      const uint32_t S0 = rotr(a, 2) ^ rotr(a, 13) ^ rotr(a, 22);
      const uint32_t maj = (a & b) ^ (a & c) ^ (b & c);
      const uint32_t t2 = S0 + maj;
      hh = g;
      g = f;
      f = e;
      e = d + t1;
      d = c;
      c = b;
      b = a;
      a = t1 + t2;
    }
    h[0] += a; h[1] += b; h[2] += c; h[3] += d;
    h[4] += e; h[5] += f; h[6] += g; h[7] += hh;
  }
  for (int i = 0; i < 8; ++i)
    for (int j = 0; j < 4; ++j) out[4 * i + j] = (unsigned char)((h[i] >> (24 - 8 * j)) & 0xff);
}

const char* dtype_name(gdn_dtype t) { return t == GDN_BF16 ? "bf16" : "fp32"; }

std::string policy_text(const gdn_cpr_shape* s) {
  gdn::Dims d{};
  d.D = s->d_k;
  d.C = s->chunk;
  d.in_bf16 = s->in_dtype == GDN_BF16;
  d.out_bf16 = s->out_dtype == GDN_BF16;
  const bool tc = gdn::boundary_on_tensor_cores(d);
  char buf[2048];
  snprintf(buf, sizeof(buf),
           "gdn-cpr numerical policy 1\n"
           "library=%d\n"
           "d_k=%d\nd_v=%d\nchunk=%d\n"
           "in_dtype=%s\nout_dtype=%s\n"
           "state=fp32, d_v x d_k, row = value dimension\n"
           "chunks=aligned to each sequence's first token; state_out = token recurrence through a partial last chunk\n"
           "contraction=none (explicit round-to-nearest fma/mul/add)\n"
           "exp=expf\n"
           "token_step=4 state rows x d/8 columns per lane (columns 32j+4b..+3), 8 lanes per row group; "
           "state held as c*S~: c*=a; if c outside [2^-64,2^64] then S~*=c, c=1; "
           "S~+=fma(beta*rcp.approx(c), v, -(beta*(S~.k))) k^T; o=c*(S~.q); running state out = c*S~ elementwise; "
           "each dot: per lane and row one float2 partial (x: columns 4b, 4b+2; y: 4b+1, 4b+3; ascending j), x+y, "
           "then across the 8 lanes the tree ((l0+l4)+(l2+l6))+((l1+l5)+(l3+l7))\n"
           "cumsum_g=sequential fp32, ascending token\n"
           "triangular_solve=(I+A)^-1 blocked by 16: diagonal blocks by forward substitution, "
           "off-diagonal blocks by increasing distance, every sum ascending with one accumulator\n"
           "boundary=%s\n"
           "resync=eager, when a chunk completes, with the prefill boundary kernels on the chunk's tail\n"
           "output=%s\n",
           gdn_cpr_version(), s->d_k, s->d_v, s->chunk, dtype_name(s->in_dtype), dtype_name(s->out_dtype),
           tc ? "tcgen05 kind::f16, fp32 accumulate in tensor memory; fp32 operands split x = hi + lo (bf16 each), "
                "products hi*hi + hi*lo + lo*hi in that order; bf16 inputs exact; fixed 16-wide K steps"
              : "fp32 SIMT; dot products of length d in 4 partials over ascending groups of 4, (p0+p1)+(p2+p3)",
           s->out_dtype == GDN_BF16 ? "round to nearest even from fp32" : "fp32");
  return std::string(buf);
}

}  // namespace

extern "C" gdn_status gdn_cpr_policy_digest(const gdn_cpr_shape* shape, unsigned char digest[32], char* text,
                                            size_t text_len) {
  if (!shape || !digest) return GDN_ERR_INVALID_ARG;
  size_t bytes = 0;
  const gdn_status rc = gdn_cpr_workspace_size(shape, GDN_MODE_DECODE, nullptr, &bytes);
  if (rc != GDN_OK) return rc;
  const std::string t = policy_text(shape);
  sha256(reinterpret_cast<const unsigned char*>(t.data()), t.size(), digest);
  if (text && text_len > 0) {
    const size_t n = t.size() < text_len - 1 ? t.size() : text_len - 1;
    memcpy(text, t.data(), n);
    text[n] = '\0';
  }
  return GDN_OK;
}
