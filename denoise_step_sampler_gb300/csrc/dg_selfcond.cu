// K4 -- the self-conditioning contraction out = softmax(z/T) . E on the
// Blackwell tensor cores (Technical Report section 3.2, eq. 6: the p0 E inside
// FFW(p0 E)).
//
// The probabilities are never stored: each 256 x 64 tile of bf16 logits
// arrives by TMA in the 128-byte-swizzled K-major layout the MMA reads, and
// eight producer warps turn it into p in place,
// p = 2^(z*log2(e)/T - (m*log2(e) + log2 s)), from the per-position (m, s)
// the sampler step wrote (fp32 or unaligned logits are loaded by the producers
// instead).  The E tile (64 vocabulary rows x 256 embedding columns, bf16,
// N-major, 128-byte swizzle) arrives by TMA and serves two M=128 MMAs (the two
// row halves), so each staged byte of E feeds 256 rows of work.  A tiled TMA
// copy holds the thread that issues it for a time that grows with the box's
// row count, so tiles are 128 bytes wide (half the rows per byte of 64-byte
// tiles) and are issued by four warps: two for the logits halves, two for E.  One thread
// issues the tcgen05.mma (M=128, N=256, K=16, bf16 x bf16 -> fp32) into two
// 256-column TMEM accumulators; the epilogue reads them back with tcgen05.ld.
// Small batches split the vocabulary (K) across CTAs and reduce the fp32
// partial sums in a second kernel.  Every wait is bounded: a wait that gives up
// sets DG_DEV_WAIT_TIMEOUT, the CTA drains what it issued and returns.
#include <cuda.h>
#include <cuda_bf16.h>

#include <atomic>

#include <cstring>
#include <algorithm>

#include "dg_device.cuh"
#include "dg_internal.h"

namespace dg {
namespace {

constexpr int BM = 256;  // rows per CTA: two M=128 MMAs share every E tile
constexpr int BN = 256;  // embedding columns per CTA (one N=256 MMA per row half)
constexpr int BK = 64;   // one 128-byte swizzle row of bf16
// Two operand rings that advance separately: E tiles (mostly from DRAM, the
// slow ones to land) run one stage deeper than the logits tiles, which also
// wait for the p rebuild.
constexpr int NE = 4;    // E stages of 32 KB
constexpr int NA = 3;    // logits / p stages of 32 KB
constexpr int kProdWarps = 16;  // four per scheduler: the p rebuild is latency-bound
constexpr int kAIssuers = 2;  // TMA warps that each load one 128-row half of the logits tile
constexpr int kFirstAWarp = 2 + kProdWarps;
#ifndef DG_K4_E_ISSUERS
#define DG_K4_E_ISSUERS 1
#endif
// TMA warps for the E tile: a tiled copy holds its issuing thread for a time
// that grows with the box's rows, so the four boxes of a stage may be split
// between two warps (warp 0 and the last warp).
constexpr int kEIssuers = DG_K4_E_ISSUERS;
static_assert(kEIssuers == 1 || kEIssuers == 2, "one or two E warps");
#ifndef DG_K4_E3D
#define DG_K4_E3D 1
#endif
constexpr int kSecondEWarp = kEIssuers == 2 ? kFirstAWarp + kAIssuers : -1;
// warp 0 E-tile TMA, warp 1 MMA, 16 producer/epilogue warps, 2 logits TMA
// warps, optionally a second E warp (at 96 registers a thread, 21 warps fit)
constexpr int kThreads = 32 * (kFirstAWarp + kAIssuers + kEIssuers - 1);
constexpr uint32_t kABytes = BM * BK * 2;  // 32 KB
constexpr uint32_t kAHalf = 128 * BK * 2;  // 16 KB: one M=128 operand
constexpr uint32_t kBBoxBytes = BK * 128;  // one 64-column box of E: 64 rows x 128 B
constexpr uint32_t kBBytes = BK * BN * 2;  // 32 KB
constexpr uint32_t kSharedBytes = 1024;  // barriers + per-row flags, after the stages
constexpr uint32_t kSmemBytes = NE * kBBytes + NA * kABytes + kSharedBytes + 1024;  // + alignment
static_assert(kSmemBytes <= 232448, "over the 227 KB per-CTA shared memory limit");
// E tiles come mostly from DRAM, logits tiles mostly from L2 (the column tiles
// of a row block run side by side), so the CTAs of even row tiles ask L2 for
// the E tile this many k-blocks before it is loaded (the odd row tile next to
// each, which runs at the same time on the same E tile, finds it there).
constexpr int kPrefetchKb = 4;
#ifndef DG_WAIT_NS
#define DG_WAIT_NS 2000000000ull
#endif
// Bound on any single pipeline wait.  Waits for copies or MMAs already issued
// (before a CTA exits or frees its TMEM) always keep the 2 s bound: those
// complete on their own, so the CTA never leaves with work in flight.
constexpr unsigned long long kWaitNs = DG_WAIT_NS;
constexpr unsigned long long kDrainNs = 2000000000ull;
// DG_TEST_WITHHOLD_E_STAGE (test builds only): the E warps stop before
// issuing that k-block's copies, so the MMA issuer's wait for it can only run
// out, which exercises the bounded-wait exit path without faulting anything.

struct Shared {
  uint64_t full[NE];     // TMA bytes of the stage's E tile landed
  uint64_t empty[NE];    // the MMAs reading the E stage completed
  uint64_t a_full[NA];   // TMA bytes of the stage's logits tile landed
  uint64_t a_ready[NA];  // producers wrote p into the A tile
  uint64_t a_empty[NA];  // the MMAs reading the A stage completed
  uint64_t tmem_full;
  uint64_t mma_done;
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t any_valid;
  uint8_t row_ok[BM];
};
static_assert(sizeof(Shared) <= kSharedBytes, "barrier block outgrew its reservation");

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint64_t *b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t *b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
}  // namespace

// First wait that gave up since load (diagnostics): {set, block, where, parity}.
// where = role << 28 | barrier << 24 | stage << 16 | k-iteration (low 16 bits);
// roles 0 TMA, 1 MMA, 2 producer, 3 epilogue; barriers 0 full, 1 a_ready,
// 2 empty (E), 3 tmem_full, 4 a_full, 5 a_empty.
__device__ uint32_t g_wait_record[4];

namespace {

__device__ __forceinline__ uint32_t where_code(uint32_t role, uint32_t bar, int stage, int iter) {
  return (role << 28) | (bar << 24) | ((uint32_t)stage << 16) | ((uint32_t)iter & 0xFFFFu);
}

// Bounded wait; false if it gave up or another role aborted.
__device__ __forceinline__ bool mbar_wait_flag(uint64_t *b, uint32_t parity, int32_t *abort_flag,
                                            uint32_t *status, uint32_t where) {
  // Poll the barrier; only every 256th failed poll looks at the abort flag and
  // the clock, so a completed phase is noticed at once.
  uint64_t t0 = 0;
  for (uint32_t it = 1;; ++it) {
    if (mbar_try(b, parity)) return true;
    if ((it & 255u) != 0u) continue;
    if (*(volatile int32_t *)abort_flag) return false;
    const uint64_t now = globaltimer();
    if (t0 == 0) {
      t0 = now;
    } else if (now - t0 > kWaitNs) {
      *(volatile int32_t *)abort_flag = 1;
      atomicOr(status, (uint32_t)DG_DEV_WAIT_TIMEOUT);
      if (atomicCAS(&g_wait_record[0], 0u, 1u) == 0u) {
        g_wait_record[1] = blockIdx.x;
        g_wait_record[2] = where;
        g_wait_record[3] = parity;
      }
      return false;
    }
  }
}
template <class SH>
__device__ __forceinline__ bool mbar_wait(uint64_t *b, uint32_t parity, SH *sh, uint32_t *status,
                                          uint32_t where) {
  return mbar_wait_flag(b, parity, &sh->abort_flag, status, where);
}
// Bounded wait used while draining after an abort (ignores the abort flag).
__device__ __noinline__ void mbar_drain(uint64_t *b, uint32_t parity) {
  uint64_t t0 = 0;
  for (uint32_t it = 1;; ++it) {
    if (mbar_try(b, parity)) return;
    if ((it & 255u) != 0u) continue;
    const uint64_t now = globaltimer();
    if (t0 == 0) t0 = now;
    else if (now - t0 > kDrainNs) return;
  }
}

__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *map, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// One 3D box: the four 64-column blocks of a stage's E tile in one copy
// (dimensions: column within a block, vocabulary row, block).
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int32_t x, int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory matrix descriptor (tcgen05 format); swz: 2 = 128-byte,
// 4 = 64-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t swz) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version
  d |= (uint64_t)swz << 61;
  return d;
}

// Instruction descriptor: bf16 x bf16 -> fp32, A K-major, B N-major, M=128, N=256
// (each MMA covers one 128-row half of the CTA's 256 rows).
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) |
                            ((uint32_t)(256 >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate));
}
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

struct GemmArgs {
  const void *logits;
  int64_t ld;
  int32_t V, C, d, dtype;
  int64_t rows;  // B*C
  int32_t m_tiles, n_tiles, splits, k_blocks, kb_per_split;
  int32_t tma_a;  // 1: bf16 logits tiles arrive by TMA; 0: producers load them
  int32_t e3d;    // 1: tmap_e is 3D and a stage's E tile is one copy; 0: 2D, one copy per block
  const uint8_t *phase;
  const uint8_t *sc_valid;
  const float *temperature;
  const float *m;
  const float *s;
  void *out;
  int32_t out_dtype;
  float *partial;  // [splits][rows][d] when splits > 1
  uint32_t *status;
  float cap_k, cap_c;  // logit softcap: 2 log2(e) / c and c (capped kernels only)
  float scale;         // factor on the output (the embedding scale; 1 = none)
  // fused step (else null): per row, the reference R of the operand the
  // vocabulary pass wrote (the A rows hold 2^(z c - R)), or NaN for rows the
  // materialisation pass wrote as p itself
  const float *feed_R;
};

__device__ __forceinline__ bool row_feeds(const GemmArgs &a, int64_t q, float &c, float &l2) {
  if (q >= a.rows) return false;
  const int64_t r = q / a.C;
  if (a.sc_valid[r] != 1 || a.phase[r] != DG_PHASE_DENOISE) return false;
  const float m = a.m[q], s = a.s[q], T = a.temperature[r];
  if (!(isfinite(m) && s > 0.f && isfinite(s) && T > 0.f && isfinite(T))) return false;
  c = kLog2e / T;
  l2 = fmaf(m, kLog2e, __log2f(s));
  return true;
}

// 8 consecutive logits of one row from global memory, as raw words: bf16
// pairs (w[0..3]) or fp32 (w[0..7]); columns >= V come back as -inf.
struct Raw8 {
  uint32_t w[8];
};
__device__ __forceinline__ Raw8 load_raw8(const GemmArgs &a, const char *rowp, int64_t k) {
  Raw8 r;
  const bool vec_ok = ((reinterpret_cast<uintptr_t>(rowp) & 15u) == 0) && (k + 8 <= a.V);
  if (a.dtype == DG_BF16) {
    if (vec_ok) {
      const uint4 v = __ldg(reinterpret_cast<const uint4 *>(rowp + k * 2));
      r.w[0] = v.x; r.w[1] = v.y; r.w[2] = v.z; r.w[3] = v.w;
    } else {
      const unsigned short *b = reinterpret_cast<const unsigned short *>(rowp);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t lo = (k + 2 * j < a.V) ? (uint32_t)__ldg(b + k + 2 * j) : 0xFF80u;
        const uint32_t hi = (k + 2 * j + 1 < a.V) ? (uint32_t)__ldg(b + k + 2 * j + 1) : 0xFF80u;
        r.w[j] = lo | (hi << 16);
      }
    }
  } else {
    if (vec_ok) {
      const uint4 u = __ldg(reinterpret_cast<const uint4 *>(rowp + k * 4));
      const uint4 v = __ldg(reinterpret_cast<const uint4 *>(rowp + k * 4 + 16));
      r.w[0] = u.x; r.w[1] = u.y; r.w[2] = u.z; r.w[3] = u.w;
      r.w[4] = v.x; r.w[5] = v.y; r.w[6] = v.z; r.w[7] = v.w;
    } else {
      const uint32_t *f = reinterpret_cast<const uint32_t *>(rowp);
#pragma unroll
      for (int j = 0; j < 8; ++j) r.w[j] = (k + j < a.V) ? __ldg(f + k + j) : 0xFF800000u;
    }
  }
  return r;
}

// p for 8 logits (bf16 pairs or fp32), packed to bf16; columns at or past V
// (given by `valid`, a count from the chunk start) become exactly 0.
__device__ __forceinline__ uint4 p_from_bf16(const uint32_t (&w)[4], float c, float l2,
                                             int valid) {
  float z[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    z[2 * j] = __uint_as_float(w[j] << 16);
    z[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
  }
  float p[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) p[j] = (j < valid) ? ex2_approx(fmaf(z[j], c, -l2)) : 0.f;
  return make_uint4(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]), pack_bf16x2(p[4], p[5]),
                    pack_bf16x2(p[6], p[7]));
}
// Same as p_from_bf16 for a chunk wholly inside the vocabulary (no bounds
// checks), with the exponent arguments formed by packed f32x2 FMAs.
__device__ __forceinline__ uint4 p_from_bf16_full(const uint4 &v, uint64_t cc, uint64_t nl) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t out[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint64_t z = pack2(__uint_as_float(w[j] << 16), __uint_as_float(w[j] & 0xFFFF0000u));
    const uint64_t arg = fma2(z, cc, nl);
    out[j] = pack_bf16x2(ex2_approx(lo2(arg)), ex2_approx(hi2(arg)));
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}
__device__ __forceinline__ uint4 p_from_f32(const uint32_t (&w)[8], float c, float l2,
                                            int valid) {
  float p[8];
#pragma unroll
  for (int j = 0; j < 8; ++j)
    p[j] = (j < valid) ? ex2_approx(fmaf(__uint_as_float(w[j]), c, -l2)) : 0.f;
  return make_uint4(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]), pack_bf16x2(p[4], p[5]),
                    pack_bf16x2(p[6], p[7]));
}

// p from softcapped logits ("The Annotated DiffusionGemma", "Logit
// Softcapping"): the same rebuild on c tanh(z / c) for the first `valid` of 8
// bf16 (w[0..3]) or fp32 (w[0..7]) logits.
__device__ __forceinline__ uint4 p_from_bf16_cap(const uint32_t (&w)[4], float c, float l2,
                                                 int valid, float cap_k, float cap_c) {
  float p[8];
#pragma unroll
  for (int j = 0; j < 8; j += 2) {
    const float2 zc = softcap2_f(make_float2(__uint_as_float(w[j >> 1] << 16),
                                             __uint_as_float(w[j >> 1] & 0xFFFF0000u)),
                                 cap_k, cap_c);
    p[j] = (j < valid) ? ex2_approx(fmaf(zc.x, c, -l2)) : 0.f;
    p[j + 1] = (j + 1 < valid) ? ex2_approx(fmaf(zc.y, c, -l2)) : 0.f;
  }
  return make_uint4(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]), pack_bf16x2(p[4], p[5]),
                    pack_bf16x2(p[6], p[7]));
}
__device__ __forceinline__ uint4 p_from_f32_cap(const uint32_t (&w)[8], float c, float l2,
                                                int valid, float cap_k, float cap_c) {
  float p[8];
#pragma unroll
  for (int j = 0; j < 8; ++j)
    p[j] = (j < valid)
               ? ex2_approx(fmaf(softcap_f(__uint_as_float(w[j]), cap_k, cap_c), c, -l2))
               : 0.f;
  return make_uint4(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]), pack_bf16x2(p[4], p[5]),
                    pack_bf16x2(p[6], p[7]));
}

// Byte offset of 16-byte chunk `ch` (0..7) of row `r` in a 128-byte-swizzled
// K-major tile (8-row atoms of 1024 bytes).
__device__ __forceinline__ uint32_t a_off(int r, int ch) {
  return (uint32_t)(r * 128 + ((ch ^ (r & 7)) << 4));
}

// One CTA per (column tile, row tile, vocabulary split), numbered with the
// column tile fastest and the row tile next, so the CTAs that read the same
// logits tile (all column tiles of a row tile) and those that read the same E
// tile (all row tiles of a column tile and split) run at the same time and
// share both through L2.  PRE: the A tiles are probabilities already
// (materialised once by selfcond_pmat_kernel), so the producers rebuild
// nothing and the MMA waits for the copies alone.
template <bool PRE>
__global__ void __launch_bounds__(kThreads, 1)
    selfcond_gemm_kernel(const __grid_constant__ CUtensorMap tmap_e,
                         const __grid_constant__ CUtensorMap tmap_z,
                         const __grid_constant__ CUtensorMap tmap_ep, GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  uint8_t *sB = smem;                  // NE x 32 KB (1024-aligned)
  uint8_t *sA = smem + NE * kBBytes;   // NA x 32 KB
  Shared *sh = reinterpret_cast<Shared *>(smem + NE * kBBytes + NA * kABytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_t = blockIdx.x % a.n_tiles;
  const int rest = blockIdx.x / a.n_tiles;
  const int m_t = rest % a.m_tiles;
  const int split = rest / a.m_tiles;
  const int64_t row0 = (int64_t)m_t * BM;
  const int n0 = n_t * BN;
  const int kb0 = split * a.kb_per_split;
  const int kb1 = min(a.k_blocks, kb0 + a.kb_per_split);
  const int nkb = max(0, kb1 - kb0);
  const int n_box = min(BN / 64, (a.d - n0 + 63) / 64);  // E boxes per stage

  if (threadIdx.x == 0) {
    for (int s = 0; s < NE; ++s) {
      mbar_init(&sh->full[s], kEIssuers);  // one expect-tx arrival per E warp
      mbar_init(&sh->empty[s], 1);  // the MMA commit
    }
    for (int s = 0; s < NA; ++s) {
      mbar_init(&sh->a_full[s], kAIssuers);
      mbar_init(&sh->a_ready[s], kProdWarps);
      mbar_init(&sh->a_empty[s], 1);  // this CTA's MMA commit
    }
    mbar_init(&sh->tmem_full, 1);
    mbar_init(&sh->mma_done, 1);
    sh->abort_flag = 0;
    sh->any_valid = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp >= 2 && threadIdx.x - 64 < BM) {
    const int t = threadIdx.x - 64;  // 0..255: one row each
    float c, l2;
    const bool ok = row_feeds(a, row0 + t, c, l2);
    sh->row_ok[t] = ok ? 1 : 0;
    if (ok) atomicOr(&sh->any_valid, 1);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&sh->tmem_base)),
                 "r"(2 * BN));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;
  // the pipeline runs if the CTA has a row to feed
  const bool run = sh->any_valid != 0 && nkb > 0;

  if (run) {
    if (warp == 0 || warp == kSecondEWarp) {
      // ------------------------------------------------ E ring (TMA)
      // Each E warp posts the bytes of its own boxes (box j belongs to E warp
      // j % kEIssuers) and loads them; the first also prefetches E into L2
      // on even row tiles.
      const int ew = warp == 0 ? 0 : 1;
      const bool prefetch = ew == 0 && (m_t & 1) == 0;
      if (lane == 0) {
        const int my_boxes = (n_box - ew + kEIssuers - 1) / kEIssuers;
        // a 3D copy always fills the whole stage (blocks past d read as zeros)
        const uint32_t my_tx = a.e3d ? (ew == 0 ? kBBytes : 0u) : (uint32_t)my_boxes * kBBoxBytes;
        if (prefetch)
          for (int i = 0; i < min(kPrefetchKb, nkb); ++i)
            tma_prefetch_2d(&tmap_ep, n0, (kb0 + i) * BK);
        int issued = 0;
        for (int i = 0; i < nkb; ++i) {
          const int s = i % NE;
          const uint32_t use = (uint32_t)(i / NE);
          if (i >= NE &&
              !mbar_wait(&sh->empty[s], (use - 1) & 1u, sh, a.status, where_code(0, 2, s, i)))
            break;
#ifdef DG_TEST_WITHHOLD_E_STAGE
          if (i == DG_TEST_WITHHOLD_E_STAGE) break;
#endif
          const int32_t kv = (kb0 + i) * BK;
          mbar_expect_tx(&sh->full[s], my_tx);
          uint8_t *dstB = sB + s * kBBytes;
          if (a.e3d) {
            if (ew == 0) tma_load_3d(dstB, &tmap_e, &sh->full[s], 0, kv, n0 / 64);
          } else {
            for (int j = ew; j < n_box; j += kEIssuers)
              tma_load_2d(dstB + j * kBBoxBytes, &tmap_e, &sh->full[s], n0 + j * 64, kv);
          }
          if (prefetch && i + kPrefetchKb < nkb)
            tma_prefetch_2d(&tmap_ep, n0, (kb0 + i + kPrefetchKb) * BK);
          issued = i + 1;
        }
        // every issued copy must land before the CTA may exit
        for (int i = max(0, issued - NE); i < issued; ++i)
          mbar_drain(&sh->full[i % NE], (uint32_t)(i / NE) & 1u);
      }
    } else if (warp >= kFirstAWarp) {
      // ------------------------------------------------ logits ring (TMA)
      // Warp kFirstAWarp + h loads the 128-row half h of the logits tile.
      const int h = warp - kFirstAWarp;
      if (lane == 0 && a.tma_a) {
        int issued = 0;
        for (int i = 0; i < nkb; ++i) {
          const int s = i % NA;
          const uint32_t use = (uint32_t)(i / NA);
          if (i >= NA &&
              !mbar_wait(&sh->a_empty[s], (use - 1) & 1u, sh, a.status, where_code(0, 5, s, i)))
            break;
          mbar_expect_tx(&sh->a_full[s], kAHalf);
          tma_load_2d(sA + s * kABytes + h * kAHalf, &tmap_z, &sh->a_full[s], (kb0 + i) * BK,
                      (int32_t)(row0 + h * 128));
          issued = i + 1;
        }
        for (int i = max(0, issued - NA); i < issued; ++i)
          mbar_drain(&sh->a_full[i % NA], (uint32_t)(i / NA) & 1u);
      }
    } else if (warp == 1) {
      // ------------------------------------------------ MMA issuer
      if (lane == 0) {
        for (int i = 0; i < nkb; ++i) {
          const int s = i % NE, sa = i % NA;
          if (!mbar_wait(&sh->full[s], (uint32_t)(i / NE) & 1u, sh, a.status,
                         where_code(1, 0, s, i)))
            break;
          if (!mbar_wait(PRE ? &sh->a_full[sa] : &sh->a_ready[sa], (uint32_t)(i / NA) & 1u, sh, a.status,
                         where_code(1, 1, sa, i)))
            break;
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + sa * kABytes);
          const uint32_t b_base = smem_u32(sB + s * kBBytes);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t bd = smem_desc(b_base + kk * 2048, kBBoxBytes, 1024, 2);
#pragma unroll
            for (int mh = 0; mh < 2; ++mh) {
              const uint64_t ad = smem_desc(a_base + mh * kAHalf + kk * 32, 16, 1024, 2);
              mma_bf16(tmem + (uint32_t)(mh * BN), ad, bd, (i > 0 || kk > 0) ? 1u : 0u);
            }
          }
          mma_commit(&sh->empty[s]);    // the E warps may reuse E stage s
          mma_commit(&sh->a_empty[sa]);  // the logits warps may reuse A stage sa
        }
        mma_commit(&sh->tmem_full);
        mma_commit(&sh->mma_done);
      }
    } else {
      // ------------------------------------------------ p producers
      const int t = threadIdx.x - 64;  // 0..511
      // Four (row, 16-byte chunk) units per thread, fixed across stages:
      // unit j is row (t >> 3) + 64 j, chunk t & 7, so each unit index of a
      // warp covers four whole 128-byte rows (no bank conflicts).
      const int ch = t & 7;
      uint32_t okm = 0;  // bit j: the row of unit j feeds the next step
      uint64_t cc2[4], nl2[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float c = 0.f, l2 = 0.f;
        if (row_feeds(a, row0 + (t >> 3) + 64 * j, c, l2)) okm |= 1u << j;
        cc2[j] = pack2(c, c);
        nl2[j] = pack2(-l2, -l2);
      }
      uint32_t off[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) off[j] = a_off((t >> 3) + 64 * j, ch);
      if constexpr (PRE) {
        // the tiles arrive as probabilities: nothing to rebuild
      } else if (a.tma_a) {
        for (int i = 0; i < nkb; ++i) {
          const int s = i % NA;
          const uint32_t par = (uint32_t)(i / NA) & 1u;
          // the whole warp leaves together if the wait gives up
          if (!__all_sync(0xFFFFFFFFu,
                          mbar_wait(&sh->a_full[s], par, sh, a.status, where_code(2, 4, s, i))))
            break;
          uint8_t *tileA = sA + s * kABytes;
          uint4 v[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) v[j] = *reinterpret_cast<const uint4 *>(tileA + off[j]);
          if ((int64_t)(kb0 + i + 1) * BK <= (int64_t)a.V) {  // warp-uniform: block inside V
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint4 pv = make_uint4(0u, 0u, 0u, 0u);
              if ((okm >> j) & 1u) {
                pv = p_from_bf16_full(v[j], cc2[j], nl2[j]);
              }
              *reinterpret_cast<uint4 *>(tileA + off[j]) = pv;
            }
          } else {
            const int64_t rem = (int64_t)a.V - ((int64_t)(kb0 + i) * BK + ch * 8);
            const int valid = rem >= 8 ? 8 : (rem <= 0 ? 0 : (int)rem);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
              uint4 pv = make_uint4(0u, 0u, 0u, 0u);
              if ((okm >> j) & 1u)
                pv = p_from_bf16(w, lo2(cc2[j]), -lo2(nl2[j]), valid);
              *reinterpret_cast<uint4 *>(tileA + off[j]) = pv;
            }
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh->a_ready[s]);
        }
      } else {
        // The producers load the logits themselves, one stage ahead.
        const size_t esz = (a.dtype == DG_BF16) ? 2 : 4;
        const char *rowp = reinterpret_cast<const char *>(a.logits) +
                           (size_t)(row0 + (t >> 3)) * (size_t)a.ld * esz;
        const size_t jstride = (size_t)64 * (size_t)a.ld * esz;  // unit j's row: rowp + j * jstride
        Raw8 x[4];
        if (nkb > 0) {
          const int64_t k = (int64_t)kb0 * BK + ch * 8;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if ((okm >> j) & 1u) x[j] = load_raw8(a, rowp + (size_t)j * jstride, k);
        }
        for (int i = 0; i < nkb; ++i) {
          const int s = i % NA;
          const uint32_t use = (uint32_t)(i / NA);
          if (i >= NA &&
              !__all_sync(0xFFFFFFFFu, mbar_wait(&sh->a_empty[s], (use - 1) & 1u, sh, a.status,
                                                 where_code(2, 5, s, i))))
            break;
          uint8_t *tileA = sA + s * kABytes;
          const int64_t k = (int64_t)(kb0 + i) * BK + ch * 8;
          const int64_t rem = (int64_t)a.V - k;
          const int valid = rem >= 8 ? 8 : (rem <= 0 ? 0 : (int)rem);
          uint4 pv[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            pv[j] = make_uint4(0u, 0u, 0u, 0u);
            if ((okm >> j) & 1u) {
              if (a.dtype == DG_BF16) {
                const uint32_t w[4] = {x[j].w[0], x[j].w[1], x[j].w[2], x[j].w[3]};
                pv[j] = p_from_bf16(w, lo2(cc2[j]), -lo2(nl2[j]), valid);
              } else {
                pv[j] = p_from_f32(x[j].w, lo2(cc2[j]), -lo2(nl2[j]), valid);
              }
            }
          }
          // prefetch the next stage's logits while this one is consumed
          if (i + 1 < nkb) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if ((okm >> j) & 1u) x[j] = load_raw8(a, rowp + (size_t)j * jstride, k + BK);
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) *reinterpret_cast<uint4 *>(tileA + off[j]) = pv[j];
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh->a_ready[s]);
        }
      }
    }
  }

  // ---------------------------------------------------- epilogue
  if (warp >= 2 && warp < kFirstAWarp) {
    const int ew = warp - 2;             // 0..15
    const int quarter = warp & 3;        // TMEM lane quarter this warp may access
    const int mh = (ew >> 2) & 1;        // which 128-row half (and accumulator)
    const int cbase = (ew >> 3) * (BN / 2);  // which half of the columns
    const int r = mh * 128 + quarter * 32 + lane;
    const int64_t q = row0 + r;
    bool have = false;
    if (run) have = mbar_wait(&sh->tmem_full, 0, sh, a.status, where_code(3, 3, 0, 0));
    have = __all_sync(0xFFFFFFFFu, have);
    tc_fence_after();
    const bool ok = have && sh->row_ok[r] != 0;
    // fused step: rows the vocabulary pass wrote hold 2^(z c - R); times
    // 2^(R - l2) they are p
    float g = 1.f;
    if (ok && a.feed_R) {
      float c_, l2_;
      row_feeds(a, q, c_, l2_);
      const float R = a.feed_R[q];
      if (isfinite(R)) g = exp2f(R - l2_);
    }
    for (int cb = cbase; cb < cbase + BN / 2; cb += 32) {
      const int col0 = n0 + cb;
      if (col0 >= a.d) break;  // warp-uniform
      float v[32];
      if (have) {
        tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(mh * BN + cb), v);
      }
      // per-lane conditions guard only the stores, never the warp-wide TMEM loads
      const int ncol = min(32, a.d - col0);
      if (!ok) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0.f;
      } else {  // split partials get the embedding scale in the reduction
        const float f = a.splits == 1 ? a.scale * g : g;
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] *= f;
      }
      if (q < a.rows && a.splits > 1 && run) {
        // (rows that do not feed get zeros from the reduction)
        float *dst = a.partial + ((size_t)split * a.rows + q) * a.d + col0;
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          if (j < ncol) *reinterpret_cast<float4 *>(dst + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
      } else if (q < a.rows && a.splits == 1 && a.out_dtype == DG_F32) {
        float *dst = reinterpret_cast<float *>(a.out) + (size_t)q * a.d + col0;
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          if (j < ncol) *reinterpret_cast<float4 *>(dst + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
      } else if (q < a.rows && a.splits == 1) {
        __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(a.out) + (size_t)q * a.d + col0;
#pragma unroll
        for (int j = 0; j < 32; j += 8)
          if (j < ncol)
            *reinterpret_cast<uint4 *>(dst + j) =
                make_uint4(pack_bf16x2(v[j], v[j + 1]), pack_bf16x2(v[j + 2], v[j + 3]),
                           pack_bf16x2(v[j + 4], v[j + 5]), pack_bf16x2(v[j + 6], v[j + 7]));
      }
    }
  }

  // ---------------------------------------------------- teardown
  if (run && warp == 1 && lane == 0) mbar_drain(&sh->mma_done, 0);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * BN));
  }
}

// The feed's probabilities, materialised once:
//   p[q, v] = 2^(z'_{q,v} c - l2_q)  (bf16), z' = cap(z) for a softcapped feed
// so that the GEMM's tiles need no rebuild.  Used where the rebuild would be
// slow: softcapped feeds (rebuilt in the GEMM, every column tile, 11 at
// d = 2,816, would cap each logit again, three transcendental operations per
// element each time), logits the GEMM cannot copy by TMA (fp32, or bf16 rows
// whose stride is not a multiple of 16 bytes), which its producers would
// otherwise load one stage ahead with plain loads, and batches of four row
// tiles and more, where the rebuild's shared-memory traffic costs the GEMM
// more than this pass costs.  One CTA per row; each
// thread keeps four 16-byte loads in flight.  Rows that do not feed are not
// written: the GEMM's epilogue writes zeros for them whatever their A rows
// hold (row q of the product depends on row q of p alone).
template <int DT, bool CAP>
__device__ __forceinline__ uint4 pmat8(const GemmArgs &a, const Raw8 &r, float c, float l2,
                                       int valid) {
  if constexpr (DT == DG_BF16) {
    const uint32_t w[4] = {r.w[0], r.w[1], r.w[2], r.w[3]};
    if constexpr (CAP) return p_from_bf16_cap(w, c, l2, valid, a.cap_k, a.cap_c);
    else return p_from_bf16(w, c, l2, valid);
  } else {
    if constexpr (CAP) return p_from_f32_cap(r.w, c, l2, valid, a.cap_k, a.cap_c);
    else return p_from_f32(r.w, c, l2, valid);
  }
}
template <int DT, bool CAP>
__global__ void __launch_bounds__(256) selfcond_pmat_kernel(GemmArgs a, uint4 *p, int64_t p_ld) {
  const int64_t q = blockIdx.x;
  float c = 0.f, l2 = 0.f;
  if (!row_feeds(a, q, c, l2)) return;
  if (a.feed_R && isfinite(a.feed_R[q])) return;  // the vocabulary pass wrote this row
  constexpr size_t esz = DT == DG_BF16 ? 2 : 4;
  const char *rowp = reinterpret_cast<const char *>(a.logits) + (size_t)q * (size_t)a.ld * esz;
  uint4 *prow = p + (size_t)q * (size_t)(p_ld / 8);
  const int64_t n8 = ((int64_t)a.V + 7) / 8;
  constexpr int U = 4;
  const int64_t step = blockDim.x;
  int64_t g = threadIdx.x;
  for (; g + (U - 1) * step < n8; g += U * step) {
    Raw8 r[U];
#pragma unroll
    for (int u = 0; u < U; ++u) r[u] = load_raw8(a, rowp, (g + u * step) * 8);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t k = (g + u * step) * 8;
      prow[g + u * step] = pmat8<DT, CAP>(a, r[u], c, l2, (int)min((int64_t)8, (int64_t)a.V - k));
    }
  }
  for (; g < n8; g += step) {
    const int64_t k = g * 8;
    prow[g] = pmat8<DT, CAP>(a, load_raw8(a, rowp, k), c, l2, (int)min((int64_t)8, (int64_t)a.V - k));
  }
}

// out[q, :] = sum over splits of the partial sums, zeros for rows that do
// not feed the next step.
__global__ void selfcond_reduce_kernel(GemmArgs a) {
  const int64_t n4 = a.rows * (int64_t)(a.d / 4);
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n4;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t q = e / (a.d / 4);
    const int64_t col = (e - q * (a.d / 4)) * 4;
    float c, l2;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (row_feeds(a, q, c, l2)) {
      for (int sp = 0; sp < a.splits; ++sp) {
        const float4 v =
            *reinterpret_cast<const float4 *>(a.partial + ((size_t)sp * a.rows + q) * a.d + col);
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
      acc.x *= a.scale;
      acc.y *= a.scale;
      acc.z *= a.scale;
      acc.w *= a.scale;
    }
    if (a.out_dtype == DG_F32) {
      *reinterpret_cast<float4 *>(reinterpret_cast<float *>(a.out) + q * a.d + col) = acc;
    } else {
      __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(a.out) + q * a.d + col;
      *reinterpret_cast<uint32_t *>(dst) = pack_bf16x2(acc.x, acc.y);
      *reinterpret_cast<uint32_t *>(dst + 2) = pack_bf16x2(acc.z, acc.w);
    }
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

}  // namespace

cudaError_t dg_selfcond_wait_record(uint32_t out[4]) {
  return cudaMemcpyFromSymbol(out, g_wait_record, sizeof(uint32_t) * 4);
}

SelfcondPlan selfcond_plan(int64_t rows, int32_t V, int32_t d, int32_t n_sms, int64_t l2_bytes,
                           bool materialise) {
  SelfcondPlan pl;
  pl.m_tiles = (int32_t)((rows + BM - 1) / BM);
  pl.n_tiles = (d + BN - 1) / BN;
  pl.k_blocks = (V + BK - 1) / BK;
  const int64_t tiles = (int64_t)pl.m_tiles * pl.n_tiles;
  const int64_t sms = n_sms > 0 ? n_sms : 1;
  // Choose the split count of least estimated time, in units of one CTA's
  // k-block (waves of one CTA per SM, at least 16 k-blocks per split):
  //   waves * (k-blocks per split + kCtaFixedKb) + the reduction's traffic.
  // A CTA's fixed cost (barriers and TMEM set up, the rings filled, the
  // accumulator drained) came to ~25 us, about 38 k-blocks of tensor work,
  // in measured sweeps on a GB300; the reduction moves 8 bytes per partial
  // sum, ~4.4 MB per k-block's time at the copy rate.  At one canvas this
  // picks 13 splits (one wave) where filling whole waves picked 55: 22 %
  // less time for the step.
  constexpr double kCtaFixedKb = 38.0;
  constexpr double kReduceBytesPerKb = 4.4e6;
  int best = 1;
  double best_cost = 0.0;
  for (int sp = 1; sp <= 64; ++sp) {
    if (sp > 1 && pl.k_blocks / sp < 16) break;
    const int64_t waves = (tiles * sp + sms - 1) / sms;
    const int64_t kbps = (pl.k_blocks + sp - 1) / sp;
    const double red = sp > 1 ? 8.0 * (double)sp * (double)rows * (double)d / kReduceBytesPerKb : 0.0;
    const double cost = (double)waves * ((double)kbps + kCtaFixedKb) + red;
    if (sp == 1 || cost < best_cost) {
      best_cost = cost;
      best = sp;
    }
  }
  // With many row tiles every E slice is read by CTAs of several waves, which
  // drift apart and reread it from DRAM.  Splitting further until one
  // split's E slice fits in L2 cut the step's time by ~2 % at 128 row tiles
  // (V = 262,144, d = 2,816: 11 or 12 splits instead of 3 on a GB300, whose
  // L2 holds 129 MiB); at 32 and 64 row tiles more splits were slower, so the
  // rule starts above 64.
  if (pl.m_tiles > 64 && l2_bytes > 0) {
    const int64_t e_bytes = (int64_t)pl.k_blocks * BK * d * 2;
    while (best < 64 && e_bytes / best > l2_bytes && pl.k_blocks / (best + 1) >= 16) ++best;
  }
  const int32_t kbps = (pl.k_blocks + best - 1) / best;
  pl.kb_per_split = kbps;
  pl.splits = (pl.k_blocks + kbps - 1) / kbps;
  pl.n_sms = (int32_t)sms;
  // a materialised p (softcapped feeds, logits the GEMM cannot copy by TMA):
  // rows of p_ld (V rounded up to 8) bf16, 256-byte aligned, ahead of the
  // split-K partial sums
  pl.p_ld = materialise ? ((int64_t)V + 7) / 8 * 8 : 0;
  pl.p_bytes = materialise ? ((size_t)rows * (size_t)pl.p_ld * 2 + 255) / 256 * 256 : 0;
  pl.ws_bytes = pl.p_bytes +
                (pl.splits > 1 ? (size_t)pl.splits * (size_t)rows * (size_t)d * sizeof(float) : 0);
  return pl;
}

namespace {
template <bool PRE>
cudaError_t launch_gemm(const CUtensorMap &map_e, const CUtensorMap &map_z,
                        const CUtensorMap &map_ep, const GemmArgs &a, int64_t grid,
                        cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::atomic<bool> attr_set[64];  // the shared-memory limit is raised once per device
  if (dev < 0 || dev >= 64 || !attr_set[dev].load(std::memory_order_relaxed)) {
    e = cudaFuncSetAttribute(selfcond_gemm_kernel<PRE>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev].store(true, std::memory_order_relaxed);
  }
  selfcond_gemm_kernel<PRE><<<(unsigned)grid, kThreads, kSmemBytes, s>>>(map_e, map_z, map_ep, a);
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_selfcond(const dg_params &p, const void *logits, const dg_state &st,
                            const void *E, int32_t d, int64_t ld_E, void *out, int32_t out_dtype,
                            void *ws, const SelfcondPlan &plan, cudaStream_t s,
                            const float *feed_R) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const int64_t rows = (int64_t)p.batch * p.canvas_len;
  CUtensorMap map_e, map_z, map_ep;
  // With d a multiple of 64, E is also a 3D tensor (column within a 64-column
  // block, vocabulary row, block), and a stage's four blocks are one copy:
  // a copy holds its issuing thread for a time that grows with its rows, and
  // one 3D copy of 4 x 64 rows holds it for less than four 2D copies of 64.
  // Every element of the 3D view lies inside E (blocks past d are outside
  // the tensor and read as zeros).
  bool e3d = DG_K4_E3D && d % 64 == 0;
  if (e3d) {
    const cuuint64_t dims[3] = {64, (cuuint64_t)p.vocab, (cuuint64_t)(d / 64)};
    const cuuint64_t strides[2] = {(cuuint64_t)ld_E * 2, 128};
    const cuuint32_t box[3] = {64, (cuuint32_t)BK, (cuuint32_t)(BN / 64)};
    const cuuint32_t estr[3] = {1, 1, 1};
    e3d = enc(&map_e, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(E), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  if (!e3d) {
    const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)p.vocab};
    const cuuint64_t strides[1] = {(cuuint64_t)ld_E * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)BK};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&map_e, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(E), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // the same E, one 256-column x BK-row box per k-block, for L2 prefetches only
    const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)p.vocab};
    const cuuint64_t strides[1] = {(cuuint64_t)ld_E * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BN, (cuuint32_t)BK};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&map_ep, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(E), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  // Softcapped calls, and logits that the GEMM cannot copy by TMA (fp32, or
  // bf16 rows whose stride is not a multiple of 16 bytes), materialise p once
  // in the workspace (plan.p_bytes, rows of plan.p_ld bf16), and the GEMM's
  // A tiles come from there.
  const bool pre = plan.p_bytes > 0;
  const bool tma_a = pre || (p.logits_dtype == DG_BF16 &&
                             (reinterpret_cast<uintptr_t>(logits) % 16) == 0 &&
                             (p.logits_ld * 2) % 16 == 0);
  memset(&map_z, 0, sizeof(map_z));
  if (tma_a) {
    const cuuint64_t dims[2] = {(cuuint64_t)p.vocab, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)(pre ? plan.p_ld : p.logits_ld) * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, 128u};  // 64 columns x 128 rows (half a tile)
    const cuuint32_t estr[2] = {1, 1};
    void *base = pre ? ws : const_cast<void *>(logits);
    if (enc(&map_z, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }

  GemmArgs a;
  a.logits = logits;
  a.ld = p.logits_ld;
  a.V = p.vocab;
  a.C = p.canvas_len;
  a.d = d;
  a.dtype = p.logits_dtype;
  a.rows = rows;
  a.m_tiles = plan.m_tiles;
  a.n_tiles = plan.n_tiles;
  a.splits = plan.splits;
  a.k_blocks = plan.k_blocks;
  a.kb_per_split = plan.kb_per_split;
  a.tma_a = tma_a ? 1 : 0;
  a.e3d = e3d ? 1 : 0;
  a.phase = st.phase;
  a.sc_valid = st.sc_valid;
  a.temperature = st.temperature;
  a.m = st.m;
  a.s = st.s;
  a.out = out;
  a.out_dtype = out_dtype;
  a.partial = reinterpret_cast<float *>(reinterpret_cast<char *>(ws) + plan.p_bytes);
  a.status = st.device_status;
  const bool cap = p.softcap > 0.f;
  a.cap_k = cap ? 2.0f * kLog2e / p.softcap : 0.f;
  a.cap_c = cap ? p.softcap : 0.f;
  a.scale = p.embed_scale > 0.f ? p.embed_scale : 1.0f;
  a.feed_R = feed_R;

  cudaError_t e;
  if (pre) {
    uint4 *pw = reinterpret_cast<uint4 *>(ws);
    if (p.logits_dtype == DG_BF16) {
      if (cap) selfcond_pmat_kernel<DG_BF16, true><<<(unsigned)rows, 256, 0, s>>>(a, pw, plan.p_ld);
      else selfcond_pmat_kernel<DG_BF16, false><<<(unsigned)rows, 256, 0, s>>>(a, pw, plan.p_ld);
    } else {
      if (cap) selfcond_pmat_kernel<DG_F32, true><<<(unsigned)rows, 256, 0, s>>>(a, pw, plan.p_ld);
      else selfcond_pmat_kernel<DG_F32, false><<<(unsigned)rows, 256, 0, s>>>(a, pw, plan.p_ld);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const int64_t grid = (int64_t)plan.m_tiles * plan.n_tiles * plan.splits;
  e = pre ? launch_gemm<true>(map_e, map_z, map_ep, a, grid, s)
          : launch_gemm<false>(map_e, map_z, map_ep, a, grid, s);
  if (e != cudaSuccess) return e;
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (plan.splits > 1) {
    // a grid-stride loop over float4 columns: 16 CTAs of 256 threads per SM
    const int64_t n4 = a.rows * (d / 4);
    const int64_t blocks = std::min<int64_t>((n4 + 255) / 256, (int64_t)plan.n_sms * 16);
    selfcond_reduce_kernel<<<(unsigned)blocks, 256, 0, s>>>(a);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace dg
