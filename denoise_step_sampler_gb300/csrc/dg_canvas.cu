// K2 -- one CTA per request slot: the per-canvas half of the sampler step.
//
// DENOISE rows: merge the vocabulary-pass partials of each position into
// (m, s, H, argmax, cand); then, under the entropy-budget rule, accept the
// positions of the ascending (H, i) order while the exclusive prefix sum of
// their entropies stays within the budget (the first always) -- "DiffusionGemma
// Explained", section "Sampling", step 3.  The order is never materialised:
// each position counts the pairs ranked before it and sums their entropies
// in 2^-40 fixed point (exact integer sums).  Re-noise rejected positions to
// uniform tokens (Technical Report section 3.3).  Under the monotone rule
// ("DiffusionGemma-Lite DIFFUSION.html", section 4.2) each position commits
// on an unchanged argmax or a confidence 1/s no lower than the last step's,
// committed tokens stay frozen, the rest are re-noised.  Then the convergence
// test of the stop rule and the phase update (vLLM blog, "Entropy-bounded
// denoising" and "Putting it together"; Lite section 4.4).
// PREFILL rows: a fresh uniform canvas.  COMMIT rows: emit the clean argmax
// canvas (monotone rule: the committed tokens and the last candidates
// elsewhere), then a fresh canvas and reset counters.  IDLE rows: untouched.
#include "dg_device.cuh"
#include "dg_internal.h"

namespace dg {
namespace {

constexpr int kMaxC = 1024;

__device__ __forceinline__ long long warp_sum(long long x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, off);
  return x;
}

// An entropy in 2^-40 fixed point: exact for every fp32 value >= 2^-16, so
// sums of a canvas's entropies are exact integer sums.
__device__ __forceinline__ long long hfix(float h) { return __float2ll_rn(h * 0x1p40f); }

struct CanvasArgs {
  int32_t B, C, V;
  uint64_t seed;
  float budget, thr;
  int32_t stable_k, step_cap;
  int32_t stop_rule, accept_rule;
  dg_state st;
  const Partial *part;
  int32_t n_chunks;
  int32_t merge_threads;  // threads per position in the chunk merge (1, 2 or 4)
  int mode;
  const uint8_t *row_mask;
  float *feed_R;  // fused step: per position, the operand's reference R, or NaN (fall back)
};

__global__ void __launch_bounds__(kMaxC) canvas_step_kernel(CanvasArgs a) {
  __shared__ float skey[kMaxC];
  __shared__ long long sfix[kMaxC];
  __shared__ long long swarp[32];
  __shared__ float sH[kMaxC], sS[kMaxC];
  __shared__ int32_t sAm[kMaxC], sCand[kMaxC];

  const int r = blockIdx.x;
  const int tid = threadIdx.x;
  const int nt = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nwarps = nt >> 5;
  const int C = a.C, V = a.V;
  const dg_state &st = a.st;

  const uint8_t ph = st.phase[r];
  bool do_init = false, do_commit = false;
  if (a.mode == 0) {
    if (ph == DG_PHASE_IDLE) return;
    if (ph > DG_PHASE_IDLE) {
      if (tid == 0) atomicOr(st.device_status, (uint32_t)DG_DEV_BAD_PHASE);
      return;
    }
    do_init = (ph == DG_PHASE_PREFILL);
    do_commit = (ph == DG_PHASE_COMMIT);
  } else {
    if (!a.row_mask[r]) return;
    do_init = (a.mode == 1);
    do_commit = (a.mode == 2);
  }
  const uint64_t rid = st.request_id[r];
  const uint64_t rs = st.rng_step[r];
  const int64_t base = (int64_t)r * C;

  const bool monotone = a.accept_rule == DG_ACCEPT_MONOTONE;
  if (do_init || do_commit) {
    for (int i = tid; i < C; i += nt) {
      if (do_commit) {
        int32_t tok = st.argmax_prev[base + i];
        if (monotone) tok = st.committed[base + i] ? st.canvas[base + i] : st.cand[base + i];
        if (tok < 0 || tok >= V) {
          atomicOr(st.device_status, (uint32_t)DG_DEV_BAD_TOKEN);
          tok = 0;
        }
        st.emitted[base + i] = tok;
      }
      const uint64_t pk = position_key(a.seed, rid, rs, (uint64_t)i);
      st.canvas[base + i] =
          (int32_t)below((uint32_t)(stream_key(pk, kTagInit) >> 32), (uint32_t)V);
      if (monotone) {  // a block starts with nothing committed and no confidence
        st.committed[base + i] = 0;
        st.prev_conf[base + i] = INFINITY;
      }
    }
    __syncthreads();
    if (tid == 0) {
      st.step[r] = 0;
      st.stable[r] = 0;
      st.num_sampled[r] = do_commit ? C : 0;
      st.num_rejected[r] = 0;
      st.sc_valid[r] = 0;
      st.converged[r] = 0;
      st.phase[r] = DG_PHASE_DENOISE;
      st.rng_step[r] = rs + 1;
    }
    return;
  }

  // ------------------------------------------------------------ DENOISE
  // Merge the chunk records of each position: mt threads per position (the
  // blockDim.x / CP2 adjacent lanes), each over a strided subset of chunks,
  // with the sums rescaled to a running maximum in fp32, then a shuffle merge.
  const float T = st.temperature[r];
  const float c = kLog2e / T;
  const int mt = a.merge_threads;
  {
    const int i = tid / mt, sub = tid % mt;
    uint32_t fl = 0;
    float zmax = -INFINITY, b2 = -INFINITY, S = 0.f, Tt = 0.f;
    int32_t pam = -1, pcand = -1;
    int feed_all = 1;           // every chunk wrote its operand columns
    float feed_R = -INFINITY;   // their common reference
    if (i < C) {
      const Partial *P = a.part + (size_t)(base + i) * a.n_chunks;
      for (int ch = sub; ch < a.n_chunks; ch += mt) {
        const Partial q = P[ch];
        fl |= q.flags;
        if ((q.flags & kPartFeed) == 0) feed_all = 0;
        feed_R = fmaxf(feed_R, __uint_as_float(q.pad));
        if (q.zmax > zmax || (q.zmax == zmax && q.am >= 0 && (pam < 0 || q.am < pam))) {
          if (q.zmax > zmax && S > 0.f) {  // the running maximum grows
            const float d = ceilf(zmax * c) - ceilf(q.zmax * c);
            const float f = pow2_int(d);
            Tt = fmaf(d, S, Tt) * f;
            S *= f;
          }
          zmax = q.zmax;
          pam = q.am;
        }
        if (q.s > 0.f) {
          const float d = ceilf(q.zmax * c) - ceilf(zmax * c);
          const float f = pow2_int(d);
          S = fmaf(q.s, f, S);
          Tt = fmaf(fmaf(d, q.s, q.t), f, Tt);
        }
        if (q.b2 > b2 || (q.b2 == b2 && q.cand >= 0 && (pcand < 0 || q.cand < pcand))) {
          b2 = q.b2;
          pcand = q.cand;
        }
      }
    }
    for (int off = 1; off < mt; off <<= 1) {
      const float oz = __shfl_xor_sync(0xFFFFFFFFu, zmax, off);
      const int32_t oam = __shfl_xor_sync(0xFFFFFFFFu, pam, off);
      const float os = __shfl_xor_sync(0xFFFFFFFFu, S, off);
      const float ot = __shfl_xor_sync(0xFFFFFFFFu, Tt, off);
      const float ob = __shfl_xor_sync(0xFFFFFFFFu, b2, off);
      const int32_t oc = __shfl_xor_sync(0xFFFFFFFFu, pcand, off);
      fl |= __shfl_xor_sync(0xFFFFFFFFu, fl, off);
      feed_all &= __shfl_xor_sync(0xFFFFFFFFu, feed_all, off);
      feed_R = fmaxf(feed_R, __shfl_xor_sync(0xFFFFFFFFu, feed_R, off));
      const float nz = fmaxf(zmax, oz);
      if (nz != -INFINITY) {
        float ns = 0.f, nt2 = 0.f;
        if (S > 0.f) {
          const float d = ceilf(zmax * c) - ceilf(nz * c);
          const float f = pow2_int(d);
          ns = S * f;
          nt2 = fmaf(d, S, Tt) * f;
        }
        if (os > 0.f) {
          const float d = ceilf(oz * c) - ceilf(nz * c);
          const float f = pow2_int(d);
          ns = fmaf(os, f, ns);
          nt2 = fmaf(fmaf(d, os, ot), f, nt2);
        }
        S = ns;
        Tt = nt2;
      }
      if (oz > zmax || (oz == zmax && oam >= 0 && (pam < 0 || oam < pam))) {
        zmax = oz;
        pam = oam;
      }
      if (ob > b2 || (ob == b2 && oc >= 0 && (pcand < 0 || oc < pcand))) {
        b2 = ob;
        pcand = oc;
      }
    }
    if (i < C && sub == 0) {
      bool ok = !(fl & (kPartNaN | kPartPInf | kPartBadT)) && zmax != -INFINITY && pam >= 0 &&
                pcand >= 0 && S > 0.f && isfinite(S) && isfinite(Tt);
      float Hf = NAN, m_out = NAN, s_out = NAN;
      if (ok) {  // S, Tt relative to ceil(zmax c): H does not depend on the reference
        Hf = 0.69314718f * (log2f(S) - __fdiv_rn(Tt, S));
        m_out = zmax / T;
        // s relative to the maximum itself: times 2^(ceil(zmax c) - zmax c)
        s_out = S * exp2f(ceilf(zmax * c) - zmax * c);
      } else if (!(fl & kPartBadT)) {
        atomicOr(st.device_status, (uint32_t)DG_DEV_NONFINITE_LOGITS);
      }
      sH[i] = ok ? Hf : NAN;
      sS[i] = ok ? s_out : NAN;
      sAm[i] = ok ? pam : 0;
      sCand[i] = ok ? pcand : 0;
      st.m[base + i] = m_out;
      st.s[base + i] = s_out;
      st.entropy[base + i] = Hf;
      st.argmax[base + i] = ok ? pam : 0;
      st.cand[base + i] = ok ? pcand : 0;
      if (a.feed_R) {
        // the operand 2^(z c - R) holds this position's distribution when its
        // maximum term lies within 2^+-kFeedSpan
        const bool fok = ok && feed_all && fabsf(zmax * c - feed_R) <= kFeedSpan;
        a.feed_R[base + i] = fok ? feed_R : NAN;
      }
    }
  }
  __syncthreads();
  const bool valid = (tid < C) && !isnan(sH[tid]);
  const float H = (tid < C) ? sH[tid] : NAN;
  const int32_t am = (tid < C) ? sAm[tid] : 0;
  const int32_t cand = (tid < C) ? sCand[tid] : 0;

  const int32_t step0 = st.step[r];
  int same = 1;
  long long hsum = 0;  // this position's entropy in fixed point (valid ones)
  bool bad = false;    // an invalid position makes the mean NaN
  if (monotone) {
    if (tid < C) {
      const int32_t prev_am = st.argmax_prev[base + tid];
      const bool was = st.committed[base + tid] != 0;
      const float conf = valid ? 1.f / sS[tid] : NAN;
      const float pc = st.prev_conf[base + tid];
      const bool unchanged = step0 > 0 && prev_am == am;
      const bool nw = valid && (unchanged || conf >= pc) && !was;
      int32_t tok = cand;
      if (!nw) {
        if (was) {
          tok = st.canvas[base + tid];
        } else {
          const uint64_t pk = position_key(a.seed, rid, rs, (uint64_t)tid);
          tok = (int32_t)below((uint32_t)(stream_key(pk, kTagRenoise) >> 32), (uint32_t)V);
        }
      }
      st.canvas[base + tid] = tok;
      st.committed[base + tid] = (was || nw) ? 1 : 0;
      if (valid) st.prev_conf[base + tid] = conf;
      st.accept[base + tid] = nw ? 1 : 0;
      same = (prev_am == am) ? 1 : 0;
      st.argmax_prev[base + tid] = am;
      hsum = valid ? hfix(H) : 0;
      bad = !valid;
    }
  } else {
    // rank (H, i) ascending among the canvas (invalid positions last, as
    // +inf) and sum the entropies ranked before each position
    const float key = valid ? H : INFINITY;
    if (tid < C) {
      skey[tid] = key;
      sfix[tid] = valid ? hfix(key) : 0;
    }
    __syncthreads();
    bool acc_me = false;
    if (tid < C && valid) {
      long long before = 0;  // entropies ranked before this position
      bool first = true;     // nothing ranked before it
      for (int j = 0; j < C; ++j) {  // every thread reads the same word: a broadcast
        const float kj = skey[j];
        if (kj < key || (kj == key && j < tid)) {
          first = false;
          before += sfix[j];
        }
      }
      const float bf = a.budget * 0x1p40f;  // the budget in the same fixed point
      const long long bfix = bf >= 0x1p62f ? 0x3FFFFFFFFFFFFFFFll : __float2ll_rd(bf);
      acc_me = first || before <= bfix;
    }

    // re-noise, accept mask
    if (tid < C) {
      const bool acc = acc_me;
      st.accept[base + tid] = acc ? 1 : 0;
      int32_t tok = cand;
      if (!acc) {
        const uint64_t pk = position_key(a.seed, rid, rs, (uint64_t)tid);
        tok = (int32_t)below((uint32_t)(stream_key(pk, kTagRenoise) >> 32), (uint32_t)V);
      }
      st.canvas[base + tid] = tok;
      same = (st.argmax_prev[base + tid] == am) ? 1 : 0;
      st.argmax_prev[base + tid] = am;
      hsum = valid ? hfix(H) : 0;
      bad = !valid;
    }
  }
  // convergence
  const int all_same = __syncthreads_and(same);
  const int any_bad = __syncthreads_or(bad);
  const long long wsum = warp_sum(hsum);
  if (lane == 0) swarp[warp] = wsum;
  __syncthreads();
  if (tid == 0) {
    long long tot = 0;
    for (int w = 0; w < nwarps; ++w) tot += swarp[w];
    const double hbar = any_bad ? (double)NAN : (double)tot * 0x1p-40 / (double)C;
    const int32_t step1 = step0 + 1;
    int32_t stable;
    bool conv;
    if (a.stop_rule == DG_STOP_ENTROPY) {
      stable = hbar < (double)a.thr ? st.stable[r] + 1 : 0;
      conv = stable >= a.stable_k || step1 >= a.step_cap;
    } else {
      const bool same_row = (step0 > 0) && all_same;
      stable = same_row ? st.stable[r] + 1 : 0;
      conv = (stable >= a.stable_k && hbar < (double)a.thr) || step1 >= a.step_cap;
    }
    st.stable[r] = stable;
    st.step[r] = step1;
    st.mean_entropy[r] = (float)hbar;
    st.converged[r] = conv ? 1 : 0;
    st.sc_valid[r] = conv ? 0 : 1;
    st.phase[r] = conv ? DG_PHASE_COMMIT : DG_PHASE_DENOISE;
    st.num_sampled[r] = 0;
    st.num_rejected[r] = C;
    st.rng_step[r] = rs + 1;
  }
}

}  // namespace

cudaError_t launch_canvas_step(const dg_params &p, const dg_state &st, const Partial *part,
                               int32_t n_chunks, int mode, const uint8_t *row_mask,
                               cudaStream_t s, float *feed_R) {
  int threads = 32;
  while (threads < p.canvas_len) threads <<= 1;
  // spread the chunk merge over up to 4 threads per position when there are
  // many chunks per position
  int mt = 1;
  while (mode == 0 && mt < 4 && n_chunks >= 8 * mt && threads * 2 <= 1024) {
    mt <<= 1;
    threads <<= 1;
  }
  CanvasArgs a;
  a.B = p.batch;
  a.C = p.canvas_len;
  a.V = p.vocab;
  a.seed = p.seed;
  a.budget = p.entropy_budget;
  a.thr = p.conf_threshold;
  a.stable_k = p.stable_k;
  a.step_cap = p.step_cap;
  a.stop_rule = p.stop_rule;
  a.accept_rule = p.accept_rule;
  a.st = st;
  a.part = part;
  a.n_chunks = n_chunks;
  a.merge_threads = mt;
  a.mode = mode;
  a.row_mask = row_mask;
  a.feed_R = feed_R;
  canvas_step_kernel<<<p.batch, threads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace dg
