// Device-side building blocks shared by the library's kernels: the counter
// hash (SplitMix64 output function, MurmurHash3 fmix32), the Exp(1) draws,
// the vocabulary-pass partial record, and small PTX wrappers.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "dg.h"

namespace dg {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kGroup = 8;  // vocabulary indices per Gumbel group

enum : uint32_t {
  kTagGMin = 1, kTagGArg = 2, kTagGRest = 3, kTagRenoise = 4, kTagInit = 5,
  kTagSeg = 6,     // segmented rule: one draw per vocabulary segment
  kTagWithin = 7   // segmented rule: one draw per index of the winning segment
};

// SplitMix64 output function of the state x (Steele, Lea & Flood 2014).
__host__ __device__ __forceinline__ uint64_t mix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// MurmurHash3 32-bit finalizer.
__host__ __device__ __forceinline__ uint32_t fmix32(uint32_t h) {
  h ^= h >> 16;
  h *= 0x85EBCA6Bu;
  h ^= h >> 13;
  h *= 0xC2B2AE35u;
  h ^= h >> 16;
  return h;
}

// Key of (seed, request, rng_step, position); stream keys append the tag.
__device__ __forceinline__ uint64_t position_key(uint64_t seed, uint64_t req, uint64_t rstep,
                                                 uint64_t pos) {
  uint64_t k = mix64(seed);
  k = mix64(k ^ req);
  k = mix64(k ^ rstep);
  return mix64(k ^ pos);
}
__device__ __forceinline__ uint64_t stream_key(uint64_t pkey, uint32_t tag) {
  return mix64(pkey ^ (uint64_t)tag);
}

// floor(h * n / 2^32): an integer uniform in [0, n).
__device__ __forceinline__ uint32_t below(uint32_t h, uint32_t n) {
  return (uint32_t)(((uint64_t)h * (uint64_t)n) >> 32);
}

// -ln((h + 1/2) / 2^32); the upper half goes through log1p of the exact
// complement so that small values keep their relative precision.
__device__ __forceinline__ float exp1_draw(uint32_t h) {
  if (h < 0x80000000u) {
    // u <= 1/2: -ln u >= ln 2, so the absolute error of the fast logarithm
    // (about 2^-22 |ln u|) stays a relative error of about 2^-22.
    const float u = fmaf((float)h, 2.3283064365386963e-10f, 1.1641532182693481e-10f);
    return -__logf(u);
  }
  const float w = fmaf((float)(~h), 2.3283064365386963e-10f, 1.1641532182693481e-10f);
  return -log1pf(-w);
}

// The same Exp(1) draw -ln((h + 1/2) / 2^32) without a divergent branch, for
// code where every lane draws at once (a warp would otherwise run both sides
// of exp1_draw's branch).  x is the smaller of U and its complement W = 1 - U
// (both exact multiples of 2^-33 up to fp32 rounding, at most 1/2):
//   U <= 1/2:  -ln U = -ln 2 * log2 x;
//   U >  1/2:  -ln(1 - W) = W + W^2/2 + W^3/3 + W^4/4 + W^5/5 + ... for
//              W <= 1/16 (truncated after five terms: relative error below
//              W^5 / 6 <= 2^-22), else -ln 2 * log2(1 - W), where 1 - W >= 1/2.
// Relative error a few 1e-6 at worst (the fast log2 near 1), against the
// 1e-4 near-tie window of the scores it enters.
__device__ __forceinline__ float exp1_draw_uniform(uint32_t h) {
  const bool upper = h >= 0x80000000u;
  const float x = fmaf((float)(upper ? ~h : h), 2.3283064365386963e-10f, 1.1641532182693481e-10f);
  const float big = -kLn2 * __log2f(upper ? 1.0f - x : x);
  const float series =
      x * fmaf(x, fmaf(x, fmaf(x, fmaf(x, 0.2f, 0.25f), 0.33333334f), 0.5f), 1.0f);
  return (upper && x <= 0.0625f) ? series : big;
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The softmax sums are kept relative to integer references (ceil of a
// maximum of z c, c = log2(e) / T), so that moving a sum from one reference
// to another multiplies it by 2^d with d a whole number: exact, where the
// fast exp2 of a fraction would leave an error of one sign in every entropy
// of a canvas.  pow2_int: 2^d for an integral d <= 0 (0 below 2^-126).
__device__ __forceinline__ float pow2_int(float d) {
  const int e = __float2int_rz(d);
  return e < -126 ? 0.f : __int_as_float((127 + e) << 23);
}

// 1/x by the hardware's approximate reciprocal (PTX rcp.approx.ftz.f32:
// at most 1 ulp from 1/x; +inf gives +0).
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Logit softcap c tanh(z / c), from tanh x = 1 - 2 / (e^(2x) + 1):
// c - 2c / (2^(z k) + 1) with k = 2 log2(e) / c.  +inf maps to c, -inf to
// c - 2c rcp(1) and NaN stays NaN.  The absolute error is a few 1e-7 c: the
// relative errors of ex2.approx and of the reciprocal (each within an ulp or
// two), times 2c / (e + 1) <= 2c.  Two MUFU operations per logit.
__device__ __forceinline__ float softcap_f(float z, float k, float c) {
  const float e = ex2_approx(__fmul_rn(z, k));
  return fmaf(-2.0f * c, rcp_approx(__fadd_rn(e, 1.0f)), c);
}
// The same on a pair with f32x2 arithmetic, bit for bit (each lane of a
// packed multiply, add or fma rounds as the scalar one does).
__device__ __forceinline__ float2 softcap2_f(float2 z, float k, float c) {
  const float2 t = __fmul2_rn(z, make_float2(k, k));
  const float2 x = __fadd2_rn(make_float2(ex2_approx(t.x), ex2_approx(t.y)), make_float2(1.f, 1.f));
  return __ffma2_rn(make_float2(rcp_approx(x.x), rcp_approx(x.y)),
                    make_float2(-2.0f * c, -2.0f * c), make_float2(c, c));
}

// Packed pairs of fp32 (Blackwell f32x2 arithmetic).
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float lo2(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi2(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Per (position, vocabulary chunk) result of the vocabulary pass.
//   zmax/am : largest stored logit of the chunk and its lowest index (-1 none)
//   s, t    : sum 2^a and sum a 2^a, a = z*c - ceil(zmax*c), c = log2(e)/T
//   b2/cand : best perturbed score (z*c - log2 E) and its lowest index
//   flags   : kPartNaN / kPartPInf / kPartBadT
struct alignas(16) Partial {
  float zmax;
  int32_t am;
  float s;
  float t;
  float b2;
  int32_t cand;
  uint32_t flags;
  uint32_t pad;
};
enum : uint32_t { kPartNaN = 1u, kPartPInf = 2u, kPartBadT = 4u, kPartFeed = 8u };
// The fused step (dg_denoise_step_feed): the vocabulary pass writes the
// feed's operand 2^(z c - R) as bf16 while it streams the logits, with R the
// whole number ceil(m' log2 e) + kFeedMargin from the position's previous
// maximum m' (dg_state.m before this step); a chunk that wrote all of its
// columns sets kPartFeed and leaves R in its record's pad word.  A position
// keeps that operand when its new maximum satisfies |zmax c - R| <= kFeedSpan:
// the largest term is then within 2^+-96 (bf16 spans 2^-133 .. 2^127), and no
// term that matters underflows.
constexpr float kFeedMargin = 32.f;
constexpr float kFeedSpan = 96.f;

// Chunking of the vocabulary for the vocabulary pass: a pure function of the
// sizes, shared by the workspace query and the launch.
struct VocabChunking {
  int32_t chunk;     // elements per chunk (a multiple of 1024)
  int32_t n_chunks;  // chunks per position
};
__host__ __device__ inline VocabChunking vocab_chunking(int64_t n_pos, int32_t V,
                                                        bool per_group) {
  // Few, long chunks: each warp's start (stream keys, the warm start of the
  // Gumbel screen, the first rounds' exact evaluations) is amortised over its
  // chunk, and a count that divides 8 keeps the eight warps of a CTA on whole
  // positions, so they share each position's screening bound.  The counts
  // follow timings of the pass on a GB300 at V = 262,144 for 256 to 32,768
  // positions (2, 4, 8 and 16 chunks tried at each): 8 chunks for up to 1,216
  // positions, 4 up to 9,728, 2 beyond; never below 2048 logits per chunk.
  // Rows that take the per-group path (fp32 logits, bf16 rows whose stride
  // is not a multiple of 16 bytes) load each group with plain loads; at few
  // positions they are latency-bound, and 16 requested chunks (13 at
  // V = 50,257) beat 8 by 13 % at 256 positions.
  int64_t nc = 2;
  if (n_pos <= 9728) nc = 4;
  if (n_pos <= 1216) nc = per_group ? 16 : 8;
  while (nc > 1 && ((int64_t)V + nc - 1) / nc < 2048) nc >>= 1;
  // chunks start on multiples of 1024 indices, so that every vocabulary
  // segment of the segmented Gumbel-max rule (32 indices inside one
  // superblock of 1024) lies in one chunk
  int64_t chunk = ((int64_t)V + nc - 1) / nc;
  chunk = (chunk + 1023) / 1024 * 1024;
  VocabChunking out;
  out.chunk = (int32_t)chunk;
  out.n_chunks = (int32_t)(((int64_t)V + chunk - 1) / chunk);
  return out;
}

}  // namespace dg
