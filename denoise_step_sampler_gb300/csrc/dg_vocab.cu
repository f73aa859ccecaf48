// K1 -- the fused vocabulary pass.
//
// One warp streams one contiguous chunk of one position's logit row exactly
// once and produces, without materialising probabilities:
//   * the clean argmax (largest stored logit, lowest index on ties);
//   * the online-softmax pair (s, t) in base 2 relative to the running maximum,
//     from which the entropy H = ln s - t/s follows ("DiffusionGemma
//     Explained", section "Sampling", step 2);
//   * the Gumbel-max candidate argmax(z/T + G) (vLLM blog, "Putting it
//     together": argmax(logits/T + gumbel_noise)).
// The Gumbel noise uses the library's exact group construction (8 indices per
// group share one minimum draw), so the common path costs one hash per 16-byte
// vector; a group is evaluated element by element only when it can still hold
// the winner (group minimum X/8 <= e^{max y - best}).  Chunks that hold a NaN,
// +inf or -inf logit are redone on a careful scalar path.
#include <cuda_bf16.h>

#include <atomic>

#include "dg_device.cuh"
#include "dg_internal.h"

namespace dg {
namespace {

constexpr int kWarps = 8;  // warps per CTA

struct Keys {
  uint32_t ka, kb, kc;  // low words of the GMIN / GARG / GREST stream keys
  uint32_t ks, kw;      // low words of the SEG / WITHIN stream keys (segmented rule)
};

// The softmax sums are kept in three levels so that no fp32 sum adds more
// than a few dozen terms: S/T collect one round of groups, BS/BT collect up
// to 16 rounds, ts/tt the rest of the chunk.
//
// The sums are taken relative to a reference m2 (base 2): an integer, so
// that moving the sums to a new reference is exact (pow2_int).  With
// a = z c - m2, s = sum 2^a and t = sum a 2^a give the same entropy
// log2 s - t/s for every choice of m2; the reference only keeps the terms in
// range.
struct Lane {
  float zmax;   // running max of stored logits
  int32_t am;   // its lowest index (-1 until known)
  float m2;     // reference of the sums (-inf while they are empty)
  float2 S0, S1, T0, T1;        // round sums of 2^a and a 2^a, in pairs
  float2 BS, BT;                // block sums
  float ts, tt;                 // chunk totals
  float b2;     // best perturbed score, base 2 (segmented rule: best segment score)
  int32_t cand;  // its index (segmented rule: the segment's id until the inner draw)
  float pseg;   // segmented rule: sum of 2^a over the pending segment, reference m2
  int32_t pk;   // segmented rule: pending segment id (-1 none)
};

__device__ __forceinline__ void lane_init(Lane &L) {
  L.zmax = -INFINITY;
  L.am = -1;
  L.m2 = -INFINITY;
  L.S0 = L.S1 = L.T0 = L.T1 = make_float2(0.f, 0.f);
  L.BS = L.BT = make_float2(0.f, 0.f);
  L.ts = L.tt = 0.f;
  L.b2 = -INFINITY;
  L.cand = -1;
  L.pseg = 0.f;
  L.pk = -1;
}

// Round sums into the block sums.
__device__ __forceinline__ void fold_round(Lane &L) {
  L.BS = __fadd2_rn(L.BS, __fadd2_rn(L.S0, L.S1));
  L.BT = __fadd2_rn(L.BT, __fadd2_rn(L.T0, L.T1));
  L.S0 = L.S1 = L.T0 = L.T1 = make_float2(0.f, 0.f);
}
// Block sums into the chunk totals.
// Block sums into the chunk totals.
__device__ __forceinline__ void fold_block_sums(Lane &L) {
  L.ts += L.BS.x + L.BS.y;
  L.tt += L.BT.x + L.BT.y;
  L.BS = L.BT = make_float2(0.f, 0.f);
}
__device__ __forceinline__ void fold_block(Lane &L) {
  fold_round(L);
  fold_block_sums(L);
}

__device__ __forceinline__ void sums(Lane &L, float &s, float &t) {
  fold_block(L);
  s = L.ts;
  t = L.tt;
}

// Move the reference of the sums from L.m2 up to m2n: rescale every level
// (s' = s 2^d, t' = (t + d s) 2^d with d = m2 - m2n <= 0).
__device__ __forceinline__ void rescale(Lane &L, float m2n) {
  if (L.m2 == -INFINITY) {
    L.S0 = L.S1 = L.T0 = L.T1 = make_float2(0.f, 0.f);
    L.BS = L.BT = make_float2(0.f, 0.f);
    L.ts = L.tt = 0.f;
    L.pseg = 0.f;
    L.m2 = m2n;
    return;
  }
  const float d = L.m2 - m2n;  // integral, <= 0
  const float f = pow2_int(d);
  auto one = [&](float2 &S, float2 &T) {
    T.x = fmaf(d, S.x, T.x) * f;
    T.y = fmaf(d, S.y, T.y) * f;
    S.x *= f;
    S.y *= f;
  };
  one(L.S0, L.T0);
  one(L.S1, L.T1);
  one(L.BS, L.BT);
  L.tt = fmaf(d, L.ts, L.tt) * f;
  L.ts *= f;
  L.pseg *= f;
  L.m2 = m2n;
}

// ---- segmented Gumbel-max rule ("DiffusionGemma: the first dLLM natively
// supported in vLLM", "Putting it together": argmax(logits/T + gumbel_noise),
// drawn in two levels).  Segment k = 32 j + l holds the indices
// 1024 j + 256 u + 8 l + t (u < 4, t < 8), so the 8-index group g lies in
// segment 32 (g >> 7) + (g & 31): with chunks starting on multiples of 1024,
// lane l of a warp only ever sees groups of its own segments.

__device__ __forceinline__ int32_t segment_of_group(uint32_t g) {
  return (int32_t)(32u * (g >> 7) + (g & 31u));
}

// Score the pending segment: its base-2 score m2 + log2(sum 2^a) - log2(E_k),
// E_k = X(draw32(K_SEG, k)); keep the best (lowest id on ties).
__device__ __forceinline__ void seg_close(Lane &L, const Keys &K) {
  if (L.pk >= 0 && L.pseg > 0.f) {
    const float E = exp1_draw_uniform(fmix32(K.ks ^ (uint32_t)L.pk));
    const float sc = L.m2 + (__log2f(L.pseg) - __log2f(E));
    if (sc > L.b2 || (sc == L.b2 && L.pk < L.cand)) {
      L.b2 = sc;
      L.cand = L.pk;
    }
  }
  L.pk = -1;
  L.pseg = 0.f;
}
// Score segment k of total mass `mass` (relative to L.m2) at once, when no
// segment is pending: the same as seg_add(k, mass) then seg_close.  The
// segment beats the best score b2 only if its draw E is below
// tau = mass 2^(m2 - b2), and E >= W = 1 - U = (~h + 1/2) 2^-32 (as
// -ln U >= 1 - U), so a segment whose W is above tau (with a 0.1 % margin
// for rounding) is skipped without its logarithms.
__device__ __forceinline__ void seg_score(Lane &L, int32_t k, float mass, const Keys &K) {
  const uint32_t h = fmix32(K.ks ^ (uint32_t)k);
  const float tau = mass * ex2_approx(L.m2 - L.b2);
  if ((float)(~h) * 2.3283064365386963e-10f <= tau * 1.001f && mass > 0.f) {
    const float E = exp1_draw_uniform(h);
    const float sc = L.m2 + (__log2f(mass) - __log2f(E));
    if (sc > L.b2 || (sc == L.b2 && k < L.cand)) {
      L.b2 = sc;
      L.cand = k;
    }
  }
}
// Add the mass (relative to L.m2) of some indices of segment k.
__device__ __forceinline__ void seg_add(Lane &L, int32_t k, float mass, const Keys &K) {
  if (k != L.pk) {
    seg_close(L, K);
    L.pk = k;
  }
  L.pseg += mass;
}

// Rounds of the bf16 path stream through a per-warp ring in shared memory
// (cp.async, bypassing L1): while a warp works on round r, rounds r+1 and
// r+2 are in flight, without holding registers.
constexpr int kStages = 3;
constexpr int kRingBytes = kWarps * kStages * 128 * 16;  // 48 KB per CTA
__device__ __forceinline__ void cp_async16s(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ uint4 ld_shared16(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Element-wise evaluation of group g (n members, z[0..n) finite or -inf)
// against the screening bound sb (a score some element already attains).
// Only members whose own bound E_j >= X/n can still reach sb draw their
// exponential and take a logarithm.
__device__ __forceinline__ void gumbel_group_exact(const float *z, int n, uint32_t g, uint32_t h,
                                                   float c, float sb, const Keys &K, Lane &L) {
  const float X = exp1_draw(h);
  const float base = X / (float)n;
  const uint32_t J = below(fmix32(K.kb ^ g), (uint32_t)n);
  for (int j = 0; j < n; ++j) {
    // E_j >= base, so score_j <= z_j c - log2(base); skip if that is below sb
    if (base > ex2_approx(fmaf(z[j], c, -sb)) * 1.001f) continue;
    float E = base;
    if ((uint32_t)j != J) E += exp1_draw(fmix32(K.kc ^ (g * kGroup + (uint32_t)j)));
    const float sc = fmaf(z[j], c, -__log2f(E));
    if (sc > L.b2) {
      L.b2 = sc;
      L.cand = (int32_t)(g * kGroup + j);
    }
  }
}

// Fast path for a full group of 8 finite logits: max / argmax and the
// softmax sums; returns whether the group passes the Gumbel screen against sb
// (its minimum exponential X/8 <= 2^(vmax*c - sb); X >= W = 1 - U with W
// from ~h), with the group's draw in h.
__device__ __forceinline__ bool group8(const float (&z)[8], uint32_t g, float c, float sb,
                                       const Keys &K, Lane &L, uint32_t &h) {
  const float vmax = fmaxf(fmaxf(fmaxf(z[0], z[1]), fmaxf(z[2], z[3])),
                           fmaxf(fmaxf(z[4], z[5]), fmaxf(z[6], z[7])));
  if (vmax > L.zmax) {
    int j = 7;
#pragma unroll
    for (int jj = 6; jj >= 0; --jj)
      if (z[jj] == vmax) j = jj;
    const float m2n = ceilf(vmax * c);
    rescale(L, m2n);
    L.zmax = vmax;
    L.am = (int32_t)(g * kGroup + j);
    L.m2 = m2n;
  }
  const float2 cc = make_float2(c, c);
  const float2 mm = make_float2(-L.m2, -L.m2);
  {
    const float2 a0 = __ffma2_rn(make_float2(z[0], z[1]), cc, mm);
    const float2 a1 = __ffma2_rn(make_float2(z[2], z[3]), cc, mm);
    const float2 a2 = __ffma2_rn(make_float2(z[4], z[5]), cc, mm);
    const float2 a3 = __ffma2_rn(make_float2(z[6], z[7]), cc, mm);
    const float2 e0 = make_float2(ex2_approx(a0.x), ex2_approx(a0.y));
    const float2 e1 = make_float2(ex2_approx(a1.x), ex2_approx(a1.y));
    const float2 e2 = make_float2(ex2_approx(a2.x), ex2_approx(a2.y));
    const float2 e3 = make_float2(ex2_approx(a3.x), ex2_approx(a3.y));
    L.S0 = __fadd2_rn(L.S0, e0);
    L.S1 = __fadd2_rn(L.S1, e1);
    L.T0 = __ffma2_rn(a0, e0, L.T0);
    L.T1 = __ffma2_rn(a1, e1, L.T1);
    L.S0 = __fadd2_rn(L.S0, e2);
    L.S1 = __fadd2_rn(L.S1, e3);
    L.T0 = __ffma2_rn(a2, e2, L.T0);
    L.T1 = __ffma2_rn(a3, e3, L.T1);
  }
  h = fmix32(K.ka ^ g);
  const float w = (float)(~h) * 2.3283064365386963e-10f;
  const float thr = 8.0f * ex2_approx(fmaf(vmax, c, -sb));
  return w <= thr * 1.001f;
}

// The segmented rule's form of group8: max / argmax and the softmax sums of a
// full group of 8 finite logits; returns the group's mass sum 2^(z c - m2)
// (no Gumbel screen: the rule draws once per segment).
__device__ __forceinline__ float group8_seg(const float (&z)[8], uint32_t g, float c, Lane &L) {
  const float vmax = fmaxf(fmaxf(fmaxf(z[0], z[1]), fmaxf(z[2], z[3])),
                           fmaxf(fmaxf(z[4], z[5]), fmaxf(z[6], z[7])));
  if (vmax > L.zmax) {
    int j = 7;
#pragma unroll
    for (int jj = 6; jj >= 0; --jj)
      if (z[jj] == vmax) j = jj;
    const float m2n = ceilf(vmax * c);
    rescale(L, m2n);
    L.zmax = vmax;
    L.am = (int32_t)(g * kGroup + j);
    L.m2 = m2n;
  }
  const float2 cc = make_float2(c, c);
  const float2 mm = make_float2(-L.m2, -L.m2);
  const float2 a0 = __ffma2_rn(make_float2(z[0], z[1]), cc, mm);
  const float2 a1 = __ffma2_rn(make_float2(z[2], z[3]), cc, mm);
  const float2 a2 = __ffma2_rn(make_float2(z[4], z[5]), cc, mm);
  const float2 a3 = __ffma2_rn(make_float2(z[6], z[7]), cc, mm);
  const float2 e0 = make_float2(ex2_approx(a0.x), ex2_approx(a0.y));
  const float2 e1 = make_float2(ex2_approx(a1.x), ex2_approx(a1.y));
  const float2 e2 = make_float2(ex2_approx(a2.x), ex2_approx(a2.y));
  const float2 e3 = make_float2(ex2_approx(a3.x), ex2_approx(a3.y));
  L.S0 = __fadd2_rn(L.S0, e0);
  L.S1 = __fadd2_rn(L.S1, e1);
  L.T0 = __ffma2_rn(a0, e0, L.T0);
  L.T1 = __ffma2_rn(a1, e1, L.T1);
  L.S0 = __fadd2_rn(L.S0, e2);
  L.S1 = __fadd2_rn(L.S1, e3);
  L.T0 = __ffma2_rn(a2, e2, L.T0);
  L.T1 = __ffma2_rn(a3, e3, L.T1);
  const float2 es = __fadd2_rn(__fadd2_rn(e0, e1), __fadd2_rn(e2, e3));
  return es.x + es.y;
}

// Exact evaluation of the groups that passed the screen, deferred through a
// per-warp queue in shared memory so that it always runs in full batches:
// four queued groups at a time, eight lanes per group and one member per
// lane, so the rare exact draws run convergently and no batch is mostly idle.
// Each evaluating lane keeps the best (score, index) it saw; the warp merge at
// the end takes the overall maximum, lowest index on ties.  Groups are
// screened against the bound known when they were queued and evaluated
// against the (tighter) bound known when their batch runs; both are scores
// some member of the position attains, so no possible winner is skipped.
struct QEntry {
  float z[8];
  uint32_t g, h, pad0, pad1;
};
constexpr int kQueue = 64;  // entries per warp (at most 3 + 32 are ever pending)

struct Queue {
  QEntry *q;  // this warp's ring
  int head, count;  // warp-uniform
};

// Exact perturbed score (base 2) of member j of the full group g, with the
// same operations as the batched evaluation below (so equal members score
// equally wherever they are evaluated).
__device__ __forceinline__ float exact_score8(float zj, uint32_t g, uint32_t j, float c,
                                              const Keys &K) {
  const float base = exp1_draw(fmix32(K.ka ^ g)) * 0.125f;
  const uint32_t J = below(fmix32(K.kb ^ g), 8u);
  float E = base;
  if (j != J) E += exp1_draw(fmix32(K.kc ^ (g * kGroup + j)));
  return fmaf(zj, c, -__log2f(E));
}

__device__ __forceinline__ void run_batch(Queue &Q, int cnt, float c, float &wb, const Keys &K,
                                          Lane &L, int lane) {
  const int slot = lane >> 3, j = lane & 7;
  const float sb = wb;
  if (slot < cnt) {
    const QEntry &e = Q.q[(Q.head + slot) & (kQueue - 1)];
    const float zj = e.z[j];
    const uint32_t gg = e.g, hh = e.h;
    const float base = exp1_draw(hh) * 0.125f;
    // E_j >= X/8, so score_j <= z_j c - log2(X/8): skip if below sb
    if (!(base > ex2_approx(fmaf(zj, c, -sb)) * 1.001f)) {
      const uint32_t J = below(fmix32(K.kb ^ gg), 8u);
      float E = base;
      if ((uint32_t)j != J) E += exp1_draw(fmix32(K.kc ^ (gg * kGroup + (uint32_t)j)));
      const float sc = fmaf(zj, c, -__log2f(E));
      const int32_t idx = (int32_t)(gg * kGroup + (uint32_t)j);
      if (sc > L.b2 || (sc == L.b2 && (uint32_t)idx < (uint32_t)L.cand)) {
        L.b2 = sc;
        L.cand = idx;
      }
    }
  }
  Q.head = (Q.head + cnt) & (kQueue - 1);
  Q.count -= cnt;
  wb = fmaxf(wb, L.b2);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) wb = fmaxf(wb, __shfl_xor_sync(0xFFFFFFFFu, wb, off));
}

// All 32 lanes call this after screening one group each.
__device__ __forceinline__ void coop_eval(bool pass, const float (&z)[8], uint32_t g, uint32_t h,
                                          float c, float &wb, const Keys &K, Lane &L, int lane,
                                          Queue &Q) {
  const uint32_t mask = __ballot_sync(0xFFFFFFFFu, pass);
  if (mask == 0u) return;
  if (pass) {
    const int pos = Q.head + Q.count + __popc(mask & ((1u << lane) - 1u));
    QEntry &e = Q.q[pos & (kQueue - 1)];
    *reinterpret_cast<float4 *>(&e.z[0]) = make_float4(z[0], z[1], z[2], z[3]);
    *reinterpret_cast<float4 *>(&e.z[4]) = make_float4(z[4], z[5], z[6], z[7]);
    e.g = g;
    e.h = h;
  }
  Q.count += __popc(mask);
  __syncwarp();
  while (Q.count >= 4) run_batch(Q, 4, c, wb, K, L, lane);
  __syncwarp();
}

__device__ __forceinline__ void flush_queue(Queue &Q, float c, float &wb, const Keys &K, Lane &L,
                                            int lane) {
  __syncwarp();
  while (Q.count > 0) run_batch(Q, Q.count < 4 ? Q.count : 4, c, wb, K, L, lane);
  __syncwarp();
}

// Order-preserving map of floats to signed integers (for atomicMax).
__device__ __forceinline__ int32_t f2ord(float f) {
  const int32_t i = __float_as_int(f);
  return i >= 0 ? i : (i ^ 0x7FFFFFFF);
}
__device__ __forceinline__ float ord2f(int32_t i) {
  return __int_as_float(i >= 0 ? i : (i ^ 0x7FFFFFFF));
}
// The warps of a CTA that work on chunks of the same position share the best
// attained score through shared memory: publish this warp's bound and take
// the position's.
__device__ __forceinline__ void share_bound(int32_t *slot, float &wb, int lane) {
  int32_t v = 0;
  if (lane == 0) v = atomicMax(slot, f2ord(wb));
  wb = fmaxf(wb, ord2f(__shfl_sync(0xFFFFFFFFu, v, 0)));
}

// Careful path for any group (n <= 8 members, any values): flags NaN / +inf,
// skips -inf, evaluates every finite member's Gumbel score exactly (grouped
// rule) or adds the group's mass to its segment (segmented rule).
template <bool SEG>
__device__ void group_careful(const float *z, int n, uint32_t g, float c, const Keys &K, Lane &L,
                              uint32_t &flags) {
  float zz[8];
  float vmax = -INFINITY;
  int jm = -1;
  for (int j = 0; j < n; ++j) {
    float v = z[j];
    if (isnan(v)) {
      flags |= kPartNaN;
      v = -INFINITY;
    } else if (v == INFINITY) {
      flags |= kPartPInf;
      v = -INFINITY;
    }
    zz[j] = v;
    if (v > vmax) {
      vmax = v;
      jm = j;
    }
  }
  if (vmax == -INFINITY) return;  // nothing finite in this group
  if (vmax > L.zmax) {
    const float m2n = ceilf(vmax * c);
    rescale(L, m2n);
    L.zmax = vmax;
    L.am = (int32_t)(g * kGroup + jm);
    L.m2 = m2n;
  }
  float s = 0.f, t = 0.f;
  for (int j = 0; j < n; ++j) {
    if (zz[j] == -INFINITY) continue;
    const float a = fmaf(zz[j], c, -L.m2);
    const float e = ex2_approx(a);
    s += e;
    t = fmaf(a, e, t);
  }
  L.S0.x += s;
  L.T0.x += t;
  if ((g & 15u) == 15u) fold_block(L); else fold_round(L);
  if constexpr (SEG)
    seg_add(L, segment_of_group(g), s, K);
  else
    gumbel_group_exact(zz, n, g, fmix32(K.ka ^ g), c, L.b2, K, L);
}

// Largest of the 32 bf16 values of a round (NaN values are ignored; the sums
// catch them).
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162 *>(&a);
  __nv_bfloat162 y = *reinterpret_cast<const __nv_bfloat162 *>(&b);
  __nv_bfloat162 r = __hmax2(x, y);
  return *reinterpret_cast<uint32_t *>(&r);
}
__device__ __forceinline__ float round_max_bf16(const uint4 (&v)[4]) {
  uint32_t m[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) m[u] = bmax2(bmax2(v[u].x, v[u].y), bmax2(v[u].z, v[u].w));
  const uint32_t r = bmax2(bmax2(m[0], m[1]), bmax2(m[2], m[3]));
  return fmaxf(__uint_as_float(r << 16), __uint_as_float(r & 0xFFFF0000u));
}
// float -> uint32, truncating, saturating (NaN -> 0).
__device__ __forceinline__ uint32_t f2u_sat(float x) {
  uint32_t r;
  asm("cvt.rzi.sat.u32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
// The sums' reference moves only when the maximum of z c passes it by more
// than this, so terms stay below 2^4.  A wider margin saved nothing: a term
// far above the reference left the small terms added after it below half
// a unit in the last place of their sum, where rounding drops them, and the
// entropies came out low by up to a few 1e-7.
constexpr float kLazyRef = 4.f;

__device__ __forceinline__ void unpack_bf16x8(const uint4 &v, float (&z)[8]) {
  z[0] = __uint_as_float(v.x << 16);
  z[1] = __uint_as_float(v.x & 0xFFFF0000u);
  z[2] = __uint_as_float(v.y << 16);
  z[3] = __uint_as_float(v.y & 0xFFFF0000u);
  z[4] = __uint_as_float(v.z << 16);
  z[5] = __uint_as_float(v.z & 0xFFFF0000u);
  z[6] = __uint_as_float(v.w << 16);
  z[7] = __uint_as_float(v.w & 0xFFFF0000u);
}

// unpack_bf16x8, then (CAP) the softcap on every value.
template <bool CAP>
__device__ __forceinline__ void unpack8c(const uint4 &v, float (&z)[8], float cap_k, float cap_c) {
  unpack_bf16x8(v, z);
  if (CAP) {
#pragma unroll
    for (int j = 0; j < 8; ++j) z[j] = softcap_f(z[j], cap_k, cap_c);
  }
}

template <int DT>
__device__ __forceinline__ float load_scalar(const void *row, int64_t v) {
  if (DT == DG_BF16) {
    const unsigned short b = __ldg(reinterpret_cast<const unsigned short *>(row) + v);
    return __uint_as_float((uint32_t)b << 16);
  } else {
    return __ldg(reinterpret_cast<const float *>(row) + v);
  }
}

template <int DT>
__device__ __forceinline__ void load_group_scalar(const void *row, int64_t v, int n, float *z) {
  for (int j = 0; j < n; ++j) z[j] = load_scalar<DT>(row, v + j);
}
// The n (<= 8) logits of the group starting at column v (a multiple of 8) as
// fp32, softcapped when CAP ("The Annotated DiffusionGemma", "Logit
// Softcapping": every later step reads the capped value).  Whole groups of a
// 16-byte-aligned row take vector loads.
template <int DT, bool CAP>
__device__ __forceinline__ void load_group(const void *row, bool aligned, int64_t v, int n,
                                           float *z, float cap_k, float cap_c) {
  if (aligned && n == 8) {
    if (DT == DG_BF16) {
      float w[8];
      unpack_bf16x8(ld_stream(reinterpret_cast<const uint4 *>(
                        reinterpret_cast<const uint16_t *>(row) + v)),
                    w);
#pragma unroll
      for (int j = 0; j < 8; ++j) z[j] = w[j];
    } else {
      const uint4 *p = reinterpret_cast<const uint4 *>(reinterpret_cast<const float *>(row) + v);
      const uint4 a = ld_stream(p), b = ld_stream(p + 1);
      z[0] = __uint_as_float(a.x); z[1] = __uint_as_float(a.y);
      z[2] = __uint_as_float(a.z); z[3] = __uint_as_float(a.w);
      z[4] = __uint_as_float(b.x); z[5] = __uint_as_float(b.y);
      z[6] = __uint_as_float(b.z); z[7] = __uint_as_float(b.w);
    }
  } else {
    load_group_scalar<DT>(row, v, n, z);
  }
  if (CAP)
    for (int j = 0; j < n; ++j) z[j] = softcap_f(z[j], cap_k, cap_c);
}

// Merge the 32 lanes' records; every lane ends with the warp result, its sums
// relative to ceil(zmax c).  Each lane's sums come relative to its own
// (integral) reference m2.
__device__ __forceinline__ void warp_merge(float c, float m2, float &zmax, int32_t &am, float &s,
                                           float &t, float &b2, int32_t &cand) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float om2 = __shfl_xor_sync(0xFFFFFFFFu, m2, off);
    const float oz = __shfl_xor_sync(0xFFFFFFFFu, zmax, off);
    const int32_t oam = __shfl_xor_sync(0xFFFFFFFFu, am, off);
    const float os = __shfl_xor_sync(0xFFFFFFFFu, s, off);
    const float ot = __shfl_xor_sync(0xFFFFFFFFu, t, off);
    const float ob = __shfl_xor_sync(0xFFFFFFFFu, b2, off);
    const int32_t oc = __shfl_xor_sync(0xFFFFFFFFu, cand, off);
    // softmax sums, relative to ceil(zmax * c) on each side
    const float nz = fmaxf(zmax, oz);
    if (nz != -INFINITY) {
      const float M2 = ceilf(nz * c);
      float ns = 0.f, nt = 0.f;
      if (s > 0.f) {
        const float d = m2 - M2;
        const float f = pow2_int(d);
        ns += s * f;
        nt += fmaf(d, s, t) * f;
      }
      if (os > 0.f) {
        const float d = om2 - M2;
        const float f = pow2_int(d);
        ns += os * f;
        nt += fmaf(d, os, ot) * f;
      }
      s = ns;
      t = nt;
      m2 = M2;
    }
    if (oz > zmax || (oz == zmax && oam >= 0 && (am < 0 || oam < am))) {
      zmax = oz;
      am = oam;
    }
    if (ob > b2 || (ob == b2 && oc >= 0 && (cand < 0 || oc < cand))) {
      b2 = ob;
      cand = oc;
    }
  }
}

// The segmented rule's inner draw: the warp's best segment k (warp-uniform)
// has 32 indices, one per lane; the candidate is the index maximising
// z c - log2(E_v), E_v = X(draw32(K_WITHIN, v)), lowest index on ties.
template <int DT, bool CAP>
__device__ __forceinline__ int32_t segment_inner_draw(const void *row, int32_t V, int32_t k,
                                                      float c, const Keys &K, float cap_k,
                                                      float cap_c, int lane) {
  const int64_t v = 1024 * (int64_t)(k >> 5) + 256 * (lane >> 3) + 8 * (k & 31) + (lane & 7);
  float sc = -INFINITY;
  int32_t idx = -1;
  if (v < V) {
    float z = load_scalar<DT>(row, v);
    if (CAP) z = softcap_f(z, cap_k, cap_c);
    if (z > -INFINITY && z < INFINITY) {
      const float E = exp1_draw_uniform(fmix32(K.kw ^ (uint32_t)v));
      sc = fmaf(z, c, -__log2f(E));
      idx = (int32_t)v;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float os = __shfl_xor_sync(0xFFFFFFFFu, sc, off);
    const int32_t oi = __shfl_xor_sync(0xFFFFFFFFu, idx, off);
    if (os > sc || (os == sc && oi >= 0 && (idx < 0 || oi < idx))) {
      sc = os;
      idx = oi;
    }
  }
  return idx;
}

// CAP: logits pass through the softcap (cap_k = 2 log2(e) / c, cap_c = c)
// before any other use (on 16-byte-aligned bf16 rows in the ring, in
// registers).  SEG: the candidate follows the segmented rule (no Gumbel
// screen, queue or shared bound; one draw per segment of 32 indices, then the
// inner draw).
template <int DT, bool CAP, bool SEG, bool FEED>
// bf16 kernels run 3 CTAs of 8 warps per SM (the ring and the queues fill
// shared memory), at most 80 registers per thread; fp32 ones 4 CTAs at 64.
__global__ void __launch_bounds__(kWarps * 32, DT == DG_BF16 ? 3 : 4)
    vocab_pass_kernel(const void *__restrict__ logits, int64_t ld, int32_t V, int32_t C,
                      int64_t n_pos, int32_t chunk, int32_t n_chunks, uint64_t seed,
                      float cap_k, float cap_c,
                      const uint8_t *__restrict__ phase, const uint64_t *__restrict__ request_id,
                      const float *__restrict__ temperature, const uint64_t *__restrict__ rng_step,
                      Partial *__restrict__ part, uint32_t *__restrict__ status,
                      uint4 *__restrict__ feed_p, int64_t feed_ld8,
                      const float *__restrict__ m_prev) {
  __shared__ int32_t s_bound[kWarps];  // best score per position handled by this CTA
  __shared__ QEntry s_queue[kWarps][SEG ? 1 : kQueue];
  extern __shared__ uint4 s_ring[];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  if (lane == 0) s_bound[warp] = f2ord(-INFINITY);
  __syncthreads();
  const int64_t wg = (int64_t)blockIdx.x * kWarps + warp;
  if (wg >= n_pos * (int64_t)n_chunks) return;
  const int64_t pos = wg / n_chunks;
  const int32_t ch = (int32_t)(wg - pos * n_chunks);
  const int64_t r = pos / C;
  const int64_t i = pos - r * C;
  if (phase[r] != DG_PHASE_DENOISE) return;
  // slot of this position among the positions the CTA covers
  const int64_t pos0 = ((int64_t)blockIdx.x * kWarps) / n_chunks;
  int32_t *slot = &s_bound[(int)(pos - pos0)];
  Partial *out = part + wg;

  const float T = temperature[r];
  if (!(T > 0.f) || !isfinite(T)) {
    if (lane == 0) {
      Partial P;
      P.zmax = -INFINITY;
      P.am = -1;
      P.s = 0.f;
      P.t = 0.f;
      P.b2 = -INFINITY;
      P.cand = -1;
      P.flags = kPartBadT;
      P.pad = 0;
      *out = P;
      if (ch == 0) atomicOr(status, (uint32_t)DG_DEV_BAD_TEMPERATURE);
    }
    return;
  }
  const float c = kLog2e / T;

  const uint64_t pk = position_key(seed, request_id[r], rng_step[r], (uint64_t)i);
  Keys K;
  K.ka = (uint32_t)stream_key(pk, kTagGMin);
  K.kb = (uint32_t)stream_key(pk, kTagGArg);
  K.kc = (uint32_t)stream_key(pk, kTagGRest);
  if constexpr (SEG) {
    K.ks = (uint32_t)stream_key(pk, kTagSeg);
    K.kw = (uint32_t)stream_key(pk, kTagWithin);
  }

  const int64_t v0 = (int64_t)ch * chunk;
  const int64_t v1 = min((int64_t)V, v0 + chunk);
  const size_t esz = (DT == DG_BF16) ? 2 : 4;
  const char *row = reinterpret_cast<const char *>(logits) + (size_t)pos * (size_t)ld * esz;
  const int32_t n_full = (int32_t)((v1 - v0) / kGroup);
  const uint32_t g0 = (uint32_t)(v0 / kGroup);
  const int tail_n = (int)((v1 - v0) - (int64_t)n_full * kGroup);
  const bool aligned = ((reinterpret_cast<uintptr_t>(row) & 15u) == 0);

  Lane L;
  lane_init(L);
  uint32_t flags = 0;
  bool feed_ok = false;  // FEED: this lane wrote every operand slot of its share
  float feed_R = 0.f;

  // ---- fast path over full groups.  Lanes walk the chunk in warp-uniform
  // rounds (every lane runs the same number of iterations, partial rounds are
  // predicated per lane), so the warp-cooperative steps are reached by all 32
  // lanes.
  float wb = -INFINITY;  // best score attained anywhere in the warp so far
  Queue Q;
  Q.q = &s_queue[threadIdx.x >> 5][0];
  Q.head = 0;
  Q.count = 0;
  if (aligned && DT == DG_BF16) {
    const uint4 *vrow = reinterpret_cast<const uint4 *>(row) + g0;
    const int rounds = n_full / 128;
    // Per round each lane holds 4 groups (32 logits).  The round's maximum
    // (a packed bf16 max) serves three things at once: the running maximum
    // (whose index is found once, at the end, from the round that set it),
    // the reference of the sums (moved only when the maximum passes it by
    // more than kLazyRef), and one Gumbel screening threshold for all four
    // groups.
    const float2 cc = make_float2(c, c);
    int am_round = -1;
    if (!SEG && rounds > 0) {
      // Warm start: each lane scores the largest logit of its first round
      // exactly, so that the first round is already screened against a
      // finite bound instead of queueing every group.
      float zb = -INFINITY;
      uint32_t ib = 0;
#pragma unroll
      for (int u = 3; u >= 0; --u) {
        float z[8];
        unpack8c<CAP>(ld_stream(vrow + lane + u * 32), z, cap_k, cap_c);
#pragma unroll
        for (int j = 7; j >= 0; --j)
          if (z[j] >= zb) {
            zb = z[j];
            ib = (uint32_t)(u * 8 + j);
          }
      }
      if (zb > -INFINITY && zb < INFINITY) {  // NaN/inf chunks take the careful path anyway
        const uint32_t g = g0 + (uint32_t)lane + (ib >> 3) * 32u;
        const float sc = exact_score8(zb, g, ib & 7u, c, K);
        if (sc > L.b2) {
          L.b2 = sc;
          L.cand = (int32_t)(g * kGroup + (ib & 7u));
        }
      }
      wb = L.b2;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) wb = fmaxf(wb, __shfl_xor_sync(0xFFFFFFFFu, wb, off));
      share_bound(slot, wb, lane);
    }
    // this lane's slots of the warp's ring (a shared-memory address), and
    // the next round to issue
    const uint32_t ring = (uint32_t)__cvta_generic_to_shared(
        s_ring + (size_t)(threadIdx.x >> 5) * (kStages * 128) + lane);
    const uint4 *nxt = vrow + lane;
    // FEED: this lane's first 16-byte slot of the feed operand row, and
    // the row's reference R; feed_f = 2^(m2 - R) turns a sum term 2^(z c - m2)
    // into the operand's 2^(z c - R)
    uint4 *frow = nullptr;
    if constexpr (FEED) {
      const float mp = m_prev[pos];
      feed_ok = isfinite(mp);
      feed_R = feed_ok ? ceilf(mp * kLog2e) + kFeedMargin : 0.f;
      frow = feed_p + (size_t)pos * (size_t)feed_ld8 + g0 + lane;
    }
    float feed_f = 0.f;
#pragma unroll
    for (int r = 0; r < kStages - 1; ++r) {
      if (r < rounds) {
#pragma unroll
        for (int u = 0; u < 4; ++u) cp_async16s(ring + (r * 128 + u * 32) * 16, nxt + u * 32);
      }
      nxt += 128;
      cp_async_commit();
    }
    // Round rd is read from stage sc while round rd + 2 is issued into stage
    // si; both counters rotate, so no round computes a modulo or a 64-bit
    // source address.
    // the segment of round 0 (superblock v0 / 1024): each round is one
    // segment per lane, 32 segments on
    int32_t segk = (int32_t)(32u * (uint32_t)(v0 / 1024) + (uint32_t)lane);
    int sc = 0, si = kStages - 1;
    for (int rd = 0; rd < rounds;
         ++rd, sc = (sc == kStages - 1) ? 0 : sc + 1, si = (si == kStages - 1) ? 0 : si + 1) {
      if (rd + kStages - 1 < rounds) {
#pragma unroll
        for (int u = 0; u < 4; ++u) cp_async16s(ring + (si * 128 + u * 32) * 16, nxt + u * 32);
      }
      nxt += 128;
      cp_async_commit();
      cp_async_wait<kStages - 1>();
      const uint32_t cur = ring + sc * 128 * 16;
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = ld_shared16(cur + u * 32 * 16);
      // the softcap is increasing, so the round's capped maximum is the cap
      // of its raw maximum
      float rmax = round_max_bf16(v);
      if (CAP) rmax = softcap_f(rmax, cap_k, cap_c);
      if (rmax > L.zmax) am_round = rd;
      L.zmax = fmaxf(L.zmax, rmax);
      // L.m2 + kLazyRef is a whole number, so comparing rmax c with it
      // decides the same as comparing its ceiling
      const float xr = rmax * c;
      if (xr > L.m2 + kLazyRef) rescale(L, ceilf(xr));  // the first finite round sets it
      const float2 mm = make_float2(-L.m2, -L.m2);
      if constexpr (FEED) {
        // terms above 2^(R + 96) could overflow the operand: the position
        // will take the fallback (its new maximum fails the span test)
        if (L.m2 - feed_R > kFeedSpan) feed_ok = false;
        feed_f = pow2_int(fmaxf(L.m2 - feed_R, -127.f));
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
        uint32_t pw[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float zl = __uint_as_float(w[k] << 16), zh = __uint_as_float(w[k] & 0xFFFF0000u);
          if (CAP) {
            const float2 zc = softcap2_f(make_float2(zl, zh), cap_k, cap_c);
            zl = zc.x;
            zh = zc.y;
          }
          const float2 a = __ffma2_rn(make_float2(zl, zh), cc, mm);
          const float2 e = make_float2(ex2_approx(a.x), ex2_approx(a.y));
          if constexpr (FEED) {
            const float2 pf = __fmul2_rn(e, make_float2(feed_f, feed_f));
            const __nv_bfloat162 pb = __floats2bfloat162_rn(pf.x, pf.y);
            pw[k] = *reinterpret_cast<const uint32_t *>(&pb);
          }
          if (SEG && u == 0 && k < 2) {
            // the segmented rule's round sums start from the round's first
            // pairs instead of from zeros (the same values: 0 + e = e)
            if (k & 1) {
              L.S1 = e;
              L.T1 = __fmul2_rn(a, e);
            } else {
              L.S0 = e;
              L.T0 = __fmul2_rn(a, e);
            }
          } else if (k & 1) {
            L.S1 = __fadd2_rn(L.S1, e);
            L.T1 = __ffma2_rn(a, e, L.T1);
          } else {
            L.S0 = __fadd2_rn(L.S0, e);
            L.T0 = __ffma2_rn(a, e, L.T0);
          }
        }
        if constexpr (FEED) frow[(size_t)rd * 128 + u * 32] = make_uint4(pw[0], pw[1], pw[2], pw[3]);
      }
      if constexpr (SEG) {
        // the round is lane's whole segment of superblock (v0 / 1024 + rd):
        // its mass is the round's sums, scored at once
        const float2 es = __fadd2_rn(L.S0, L.S1);
        seg_score(L, segk, es.x + es.y, K);
        segk += 32;
        L.BS = __fadd2_rn(L.BS, es);
        L.BT = __fadd2_rn(L.BT, __fadd2_rn(L.T0, L.T1));
        if ((rd & 15) == 15) fold_block_sums(L);
        continue;
      }
      // Gumbel screen: group g can hold a score >= wb only if its W_g
      // (= (~h + 1/2) 2^-32) <= 8 2^(vmax c - wb); with the round maximum for
      // vmax and a 0.1 % margin that is ~h <= 2^(rmax c - wb + 35.00144).
      const uint32_t lim = ~f2u_sat(ex2_approx(fmaf(rmax, c, -wb) + 35.0014415f));
      const uint32_t gq = g0 + (uint32_t)(rd * 128 + lane);
      bool any = false;
#pragma unroll
      for (int u = 0; u < 4; ++u) any |= fmix32(K.ka ^ (gq + 32u * u)) >= lim;
      if (__any_sync(0xFFFFFFFFu, any)) {
        // rare: reread the round from the ring and queue the passing groups
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t g = gq + 32u * u;
          const uint32_t h = fmix32(K.ka ^ g);
          float z[8];
          unpack8c<CAP>(ld_shared16(cur + u * 32 * 16), z, cap_k, cap_c);
          coop_eval(h >= lim, z, g, h, c, wb, K, L, lane, Q);
        }
      }
      if ((rd & 15) == 15) fold_block(L); else fold_round(L);
      share_bound(slot, wb, lane);
    }
    if constexpr (FEED) {
      // columns outside whole rounds get no operand: the position falls back
      if (rounds * 128 != n_full || tail_n > 0) feed_ok = false;
    }
    // the segmented rule's round sums hold the last round's values (already
    // folded); the paths after the ring add to them from zero
    if constexpr (SEG) L.S0 = L.S1 = L.T0 = L.T1 = make_float2(0.f, 0.f);
    cp_async_wait<0>();
    if (am_round >= 0) {
      // lowest index holding the lane's maximum, in the round that set it
      const int q = am_round * 128 + lane;
      int32_t best = -1;
#pragma unroll
      for (int u = 3; u >= 0; --u) {
        float z[8];
        unpack8c<CAP>(ld_stream(vrow + q + u * 32), z, cap_k, cap_c);
#pragma unroll
        for (int j = 7; j >= 0; --j)
          if (z[j] == L.zmax) best = (int32_t)((g0 + (uint32_t)(q + u * 32)) * kGroup + j);
      }
      L.am = best;
    }
    for (int base = rounds * 128; base < n_full; base += 32) {
      const int q = base + lane;
      float z[8];
      uint32_t h = 0;
      bool pass = false;
      if constexpr (SEG) {
        if (q < n_full) {
          unpack8c<CAP>(ld_stream(vrow + q), z, cap_k, cap_c);
          const uint32_t g = g0 + (uint32_t)q;
          seg_add(L, segment_of_group(g), group8_seg(z, g, c, L), K);
        }
        continue;
      }
      if (q < n_full) {
        unpack8c<CAP>(ld_stream(vrow + q), z, cap_k, cap_c);
        pass = group8(z, g0 + (uint32_t)q, c, wb, K, L, h);
      }
      coop_eval(pass, z, g0 + (uint32_t)q, h, c, wb, K, L, lane, Q);
    }
  } else if (!CAP && aligned) {
    const uint4 *vrow = reinterpret_cast<const uint4 *>(row) + 2 * (size_t)g0;
    const int rounds = n_full / 64;
    for (int rd = 0; rd < rounds; ++rd) {
      const int q = rd * 64 + lane;
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        v[2 * u] = ld_stream(vrow + 2 * (q + u * 32));
        v[2 * u + 1] = ld_stream(vrow + 2 * (q + u * 32) + 1);
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        float z[8] = {__uint_as_float(v[2 * u].x),     __uint_as_float(v[2 * u].y),
                      __uint_as_float(v[2 * u].z),     __uint_as_float(v[2 * u].w),
                      __uint_as_float(v[2 * u + 1].x), __uint_as_float(v[2 * u + 1].y),
                      __uint_as_float(v[2 * u + 1].z), __uint_as_float(v[2 * u + 1].w)};
        const uint32_t g = g0 + (uint32_t)(q + u * 32);
        if constexpr (SEG) {
          seg_add(L, segment_of_group(g), group8_seg(z, g, c, L), K);
        } else {
          uint32_t h;
          const bool pass = group8(z, g, c, wb, K, L, h);
          coop_eval(pass, z, g, h, c, wb, K, L, lane, Q);
        }
      }
      if ((rd & 15) == 15) fold_block(L); else fold_round(L);
      if (!SEG) share_bound(slot, wb, lane);
    }
    for (int base = rounds * 64; base < n_full; base += 32) {
      const int q = base + lane;
      float z[8];
      uint32_t h = 0;
      bool pass = false;
      if (q < n_full) {
        const uint4 a = ld_stream(vrow + 2 * q), b = ld_stream(vrow + 2 * q + 1);
        z[0] = __uint_as_float(a.x); z[1] = __uint_as_float(a.y);
        z[2] = __uint_as_float(a.z); z[3] = __uint_as_float(a.w);
        z[4] = __uint_as_float(b.x); z[5] = __uint_as_float(b.y);
        z[6] = __uint_as_float(b.z); z[7] = __uint_as_float(b.w);
        if constexpr (SEG)
          seg_add(L, segment_of_group(g0 + (uint32_t)q), group8_seg(z, g0 + (uint32_t)q, c, L), K);
        else
          pass = group8(z, g0 + (uint32_t)q, c, wb, K, L, h);
      }
      if (!SEG) coop_eval(pass, z, g0 + (uint32_t)q, h, c, wb, K, L, lane, Q);
    }
  } else {
    for (int base = 0; base < n_full; base += 32) {  // warp-uniform trip count
      const int q = base + lane;
      float z[8];
      uint32_t h = 0;
      bool pass = false;
      if (q < n_full) {
        load_group<DT, CAP>(row, aligned, v0 + (int64_t)q * kGroup, 8, z, cap_k, cap_c);
        if constexpr (SEG)
          seg_add(L, segment_of_group(g0 + (uint32_t)q), group8_seg(z, g0 + (uint32_t)q, c, L), K);
        else
          pass = group8(z, g0 + (uint32_t)q, c, wb, K, L, h);
      }
      if (!SEG) coop_eval(pass, z, g0 + (uint32_t)q, h, c, wb, K, L, lane, Q);
      if ((base & 511) == 480) fold_block(L); else if ((base & 127) == 96) fold_round(L);
      if (!SEG && (base & 127) == 96) share_bound(slot, wb, lane);
    }
  }

  if (!SEG) flush_queue(Q, c, wb, K, L, lane);
  float s, t;
  sums(L, s, t);
  const bool bad = !(isfinite(s) && isfinite(t));
  if (__any_sync(0xFFFFFFFFu, bad)) {
    // ---- careful path: redo the whole chunk
    feed_ok = false;
    lane_init(L);
    for (int q = lane; q < n_full; q += 32) {
      float z[8];
      load_group<DT, CAP>(row, aligned, v0 + (int64_t)q * kGroup, 8, z, cap_k, cap_c);
      group_careful<SEG>(z, 8, g0 + (uint32_t)q, c, K, L, flags);
    }
  }
  if (tail_n > 0 && lane == (n_full & 31)) {
    float z[8];
    load_group<DT, CAP>(row, false, v0 + (int64_t)n_full * kGroup, tail_n, z, cap_k, cap_c);
    group_careful<SEG>(z, tail_n, g0 + (uint32_t)n_full, c, K, L, flags);
  }
  sums(L, s, t);
  if (SEG) seg_close(L, K);

  float zmax = L.zmax, b2 = L.b2;
  int32_t am = L.am, cand = L.cand;
  warp_merge(c, L.m2, zmax, am, s, t, b2, cand);
  // segmented rule: cand is the warp's best segment (warp-uniform after the
  // merge); draw the index inside it
  if (SEG && b2 > -INFINITY)
    cand = segment_inner_draw<DT, CAP>(row, V, cand, c, K, cap_k, cap_c, lane);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) flags |= __shfl_xor_sync(0xFFFFFFFFu, flags, off);
  if (FEED && __all_sync(0xFFFFFFFFu, feed_ok)) flags |= kPartFeed;
  if (lane == 0) {
    Partial P;
    P.zmax = zmax;
    P.am = am;
    P.s = s;
    P.t = t;
    P.b2 = b2;
    P.cand = cand;
    P.flags = flags;
    P.pad = FEED ? __float_as_uint(feed_R) : 0u;
    *out = P;
  }
}

}  // namespace

cudaError_t launch_vocab_pass(const dg_params &p, const void *logits, const dg_state &st,
                              Partial *part, int32_t chunk, int32_t n_chunks, cudaStream_t s) {
  const int64_t n_pos = (int64_t)p.batch * p.canvas_len;
  const int64_t warps = n_pos * n_chunks;
  const int64_t blocks = (warps + kWarps - 1) / kWarps;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  {
    static std::atomic<bool> attr_set[64];  // the shared-memory limit is raised once per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_set[dev].load(std::memory_order_relaxed)) {
      e = cudaFuncSetAttribute(vocab_pass_kernel<DG_BF16, false, false, false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kRingBytes);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(vocab_pass_kernel<DG_BF16, false, true, false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kRingBytes);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(vocab_pass_kernel<DG_BF16, true, false, false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kRingBytes);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(vocab_pass_kernel<DG_BF16, true, true, false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kRingBytes);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(vocab_pass_kernel<DG_BF16, false, true, true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kRingBytes);
      if (e != cudaSuccess) return e;
      if (dev >= 0 && dev < 64) attr_set[dev].store(true, std::memory_order_relaxed);
    }
  }
  const bool cap = p.softcap > 0.f;
  const float cap_k = cap ? 2.0f * kLog2e / p.softcap : 0.f;
  const float cap_c = cap ? p.softcap : 0.f;
#define DG_VOCAB_LAUNCH(DT, CAP, SEG)                                                         \
  vocab_pass_kernel<DT, CAP, SEG, false><<<(unsigned)blocks, kWarps * 32,                    \
                                           DT == DG_BF16 ? kRingBytes : 0, s>>>(              \
      logits, p.logits_ld, p.vocab, p.canvas_len, n_pos, chunk, n_chunks, p.seed, cap_k, cap_c, \
      st.phase, st.request_id, st.temperature, st.rng_step, part, st.device_status, nullptr, 0, \
      nullptr)
  const bool seg = p.sample_rule == DG_SAMPLE_SEGMENTED;
  if (p.logits_dtype == DG_BF16) {
    if (cap) {
      if (seg) DG_VOCAB_LAUNCH(DG_BF16, true, true);
      else DG_VOCAB_LAUNCH(DG_BF16, true, false);
    } else {
      if (seg) DG_VOCAB_LAUNCH(DG_BF16, false, true);
      else DG_VOCAB_LAUNCH(DG_BF16, false, false);
    }
  } else {
    if (cap) {
      if (seg) DG_VOCAB_LAUNCH(DG_F32, true, true);
      else DG_VOCAB_LAUNCH(DG_F32, true, false);
    } else {
      if (seg) DG_VOCAB_LAUNCH(DG_F32, false, true);
      else DG_VOCAB_LAUNCH(DG_F32, false, false);
    }
  }
#undef DG_VOCAB_LAUNCH
  return cudaGetLastError();
}

namespace {
template <bool CAP>
cudaError_t vocab_pass_feed_launch(const dg_params &p, const void *logits, const dg_state &st,
                                   Partial *part, int32_t chunk, int32_t n_chunks, uint4 *feed_p,
                                   int64_t feed_ld8, cudaStream_t s) {
  const int64_t n_pos = (int64_t)p.batch * p.canvas_len;
  const int64_t warps = n_pos * n_chunks;
  const int64_t blocks = (warps + kWarps - 1) / kWarps;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  static std::atomic<bool> attr_set[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev].load(std::memory_order_relaxed)) {
    e = cudaFuncSetAttribute(vocab_pass_kernel<DG_BF16, CAP, true, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kRingBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev].store(true, std::memory_order_relaxed);
  }
  const float cap_k = CAP ? 2.0f * kLog2e / p.softcap : 0.f;
  const float cap_c = CAP ? p.softcap : 0.f;
  vocab_pass_kernel<DG_BF16, CAP, true, true><<<(unsigned)blocks, kWarps * 32, kRingBytes, s>>>(
      logits, p.logits_ld, p.vocab, p.canvas_len, n_pos, chunk, n_chunks, p.seed, cap_k, cap_c,
      st.phase, st.request_id, st.temperature, st.rng_step, part, st.device_status, feed_p,
      feed_ld8, st.m);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_vocab_pass_feed(const dg_params &p, const void *logits, const dg_state &st,
                                   Partial *part, int32_t chunk, int32_t n_chunks,
                                   uint4 *feed_p, int64_t feed_ld8, cudaStream_t s) {
  // the caller has checked: bf16 rows on 16-byte boundaries, segmented rule
  return p.softcap > 0.f
             ? vocab_pass_feed_launch<true>(p, logits, st, part, chunk, n_chunks, feed_p, feed_ld8, s)
             : vocab_pass_feed_launch<false>(p, logits, st, part, chunk, n_chunks, feed_p, feed_ld8,
                                             s);
}

}  // namespace dg
