// C-ABI front end: argument validation (no side effect on failure), the
// workspace query, and the launches of the sampler kernels on the caller's
// stream.  Nothing here allocates, frees or synchronises.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "dg_device.cuh"
#include "dg_internal.h"

namespace dg {

bool params_ok(const dg_params *p) {
  if (!p) return false;
  if (p->batch < 1 || p->canvas_len < 1 || p->canvas_len > 1024) return false;
  if (p->vocab < 2) return false;
  if (p->logits_dtype != DG_F32 && p->logits_dtype != DG_BF16) return false;
  if (p->logits_ld < p->vocab) return false;
  if (!std::isfinite(p->entropy_budget) || p->entropy_budget < 0.f) return false;
  if (std::isnan(p->conf_threshold)) return false;
  if (p->stable_k < 1 || p->step_cap < 1) return false;
  if (p->stop_rule != DG_STOP_ARGMAX_STABLE && p->stop_rule != DG_STOP_ENTROPY) return false;
  if (p->accept_rule != DG_ACCEPT_ENTROPY_BUDGET && p->accept_rule != DG_ACCEPT_MONOTONE)
    return false;
  if (!std::isfinite(p->softcap) || p->softcap < 0.f) return false;
  if (!std::isfinite(p->embed_scale) || p->embed_scale < 0.f) return false;
  if (p->sample_rule != DG_SAMPLE_GROUPED && p->sample_rule != DG_SAMPLE_SEGMENTED) return false;
  // positions and partial records must be addressable
  const int64_t n_pos = (int64_t)p->batch * p->canvas_len;
  if (n_pos > ((int64_t)1 << 40)) return false;
  return true;
}

bool aligned(const void *ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

namespace {
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
}  // namespace

size_t denoise_ws_bytes(const dg_params *p) {
  const int64_t n_pos = (int64_t)p->batch * p->canvas_len;
  const VocabChunking vc = vocab_chunking(n_pos, p->vocab, vocab_per_group(*p));
  return round_up((size_t)n_pos * (size_t)vc.n_chunks * sizeof(Partial), 256);
}

namespace {
// An attribute of the current device, cached per device; `fallback` when no
// device can be queried (host-only callers of the workspace query).
int64_t device_attr(cudaDeviceAttr attr, std::atomic<int64_t> (&cache)[64], int64_t fallback) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return fallback;
  }
  if (dev >= 0 && dev < 64) {
    const int64_t c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, attr, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return fallback;
  }
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}
std::atomic<int64_t> g_sm_cache[64], g_l2_cache[64];  // 0 = not yet queried
}  // namespace

int32_t device_sm_count() {
  return (int32_t)device_attr(cudaDevAttrMultiProcessorCount, g_sm_cache, 152);
}
int64_t device_l2_bytes() {
  return device_attr(cudaDevAttrL2CacheSize, g_l2_cache, kGB300L2Bytes);
}

// The device must be an sm_103 part (GB300); checked once per device.
int device_ok() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return DG_ERR_CUDA;
  }
  static std::atomic<int> cache[64];  // 0 unknown, 1 ok, 2 unsupported
  if (dev >= 0 && dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c) return c == 1 ? DG_OK : DG_ERR_UNSUPPORTED;
  }
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return DG_ERR_CUDA;
  }
  const bool ok = (major == 10 && minor == 3);
  if (dev >= 0 && dev < 64) cache[dev].store(ok ? 1 : 2, std::memory_order_relaxed);
  return ok ? DG_OK : DG_ERR_UNSUPPORTED;
}

bool state_ok_phase_machine(const dg_state *st) {
  return st && st->phase && st->request_id && st->rng_step && st->step && st->stable &&
         st->canvas && st->converged && st->sc_valid && st->num_sampled && st->num_rejected &&
         st->device_status;
}

bool state_ok_full(const dg_state *st) {
  return state_ok_phase_machine(st) && st->temperature && st->argmax_prev && st->cand &&
         st->argmax && st->accept && st->m && st->s && st->entropy && st->mean_entropy &&
         st->emitted;
}

// The monotone commit rule keeps per-position commit state.
bool rule_state_ok(const dg_params *p, const dg_state *st) {
  return p->accept_rule != DG_ACCEPT_MONOTONE || (st->committed && st->prev_conf);
}

int denoise_args_ok(const dg_params *p, const void *logits, const dg_state *st) {
  if (!params_ok(p) || !state_ok_full(st) || !logits || !rule_state_ok(p, st))
    return DG_ERR_INVALID_ARG;
  const size_t esz = p->logits_dtype == DG_BF16 ? 2 : 4;
  if (!aligned(logits, esz)) return DG_ERR_INVALID_ARG;
  return DG_OK;
}

}  // namespace dg

using namespace dg;

extern "C" {

size_t dg_workspace_bytes(const dg_params *p, int32_t d) {
  if (!params_ok(p) || d < 0) return 0;
  size_t ws = denoise_ws_bytes(p);
  if (d > 0) {
    const SelfcondPlan pl = selfcond_plan((int64_t)p->batch * p->canvas_len, p->vocab, d,
                                          device_sm_count(), device_l2_bytes(),
                                          selfcond_materialises(*p));
    if (pl.ws_bytes > ws) ws = pl.ws_bytes;
  }
  return ws;
}

int dg_init_canvas(const dg_params *p, const dg_state *st, const uint8_t *row_mask,
                   cudaStream_t stream) {
  if (!params_ok(p) || !state_ok_phase_machine(st) || !row_mask || !rule_state_ok(p, st))
    return DG_ERR_INVALID_ARG;
  const int dv = device_ok();
  if (dv != DG_OK) return dv;
  cudaGetLastError();
  if (launch_canvas_step(*p, *st, nullptr, 0, 1, row_mask, stream) != cudaSuccess)
    return DG_ERR_CUDA;
  return DG_OK;
}

int dg_commit(const dg_params *p, const dg_state *st, const uint8_t *row_mask,
              cudaStream_t stream) {
  if (!params_ok(p) || !state_ok_phase_machine(st) || !row_mask || !st->argmax_prev ||
      !st->emitted || !rule_state_ok(p, st) ||
      (p->accept_rule == DG_ACCEPT_MONOTONE && !st->cand))
    return DG_ERR_INVALID_ARG;
  const int dv = device_ok();
  if (dv != DG_OK) return dv;
  cudaGetLastError();
  if (launch_canvas_step(*p, *st, nullptr, 0, 2, row_mask, stream) != cudaSuccess)
    return DG_ERR_CUDA;
  return DG_OK;
}

int dg_anneal_temperature(const dg_params *p, const int32_t *step, float *temperature,
                          float t_max, float t_min, int32_t n_steps, const uint8_t *row_mask,
                          cudaStream_t stream) {
  if (!params_ok(p) || !step || !temperature || n_steps < 1) return DG_ERR_INVALID_ARG;
  if (!(t_max > 0.f) || !(t_min > 0.f) || !std::isfinite(t_max) || !std::isfinite(t_min))
    return DG_ERR_INVALID_ARG;
  if (!aligned(step, 4) || !aligned(temperature, 4)) return DG_ERR_INVALID_ARG;
  const int dv = device_ok();
  if (dv != DG_OK) return dv;
  cudaGetLastError();
  if (launch_anneal(p->batch, step, temperature, t_max, t_min, n_steps, row_mask, stream) !=
      cudaSuccess)
    return DG_ERR_CUDA;
  return DG_OK;
}

int dg_denoise_step(const dg_params *p, const void *logits, const dg_state *st, void *ws,
                    size_t ws_bytes, cudaStream_t stream) {
  const int rc = denoise_args_ok(p, logits, st);
  if (rc != DG_OK) return rc;
  const size_t need = denoise_ws_bytes(p);
  if (!ws || ws_bytes < need || !aligned(ws, 16)) return DG_ERR_WORKSPACE;
  const int dv = device_ok();
  if (dv != DG_OK) return dv;
  cudaGetLastError();
  const int64_t n_pos = (int64_t)p->batch * p->canvas_len;
  const VocabChunking vc = vocab_chunking(n_pos, p->vocab, vocab_per_group(*p));
  Partial *part = reinterpret_cast<Partial *>(ws);
  if (launch_vocab_pass(*p, logits, *st, part, vc.chunk, vc.n_chunks, stream) != cudaSuccess)
    return DG_ERR_CUDA;
  if (launch_canvas_step(*p, *st, part, vc.n_chunks, 0, nullptr, stream) != cudaSuccess)
    return DG_ERR_CUDA;
  return DG_OK;
}

int dg_selfcond_embed(const dg_params *p, const void *logits, const dg_state *st, const void *E,
                      int32_t d, int64_t ld_E, void *out, int32_t out_dtype, void *ws,
                      size_t ws_bytes, cudaStream_t stream) {
  if (!params_ok(p) || !st || !logits || !E || !out) return DG_ERR_INVALID_ARG;
  if (!st->phase || !st->sc_valid || !st->temperature || !st->m || !st->s || !st->device_status)
    return DG_ERR_INVALID_ARG;
  if (d < 16 || d % 16 != 0 || ld_E < d || (ld_E * 2) % 16 != 0) return DG_ERR_INVALID_ARG;
  if (out_dtype != DG_F32 && out_dtype != DG_BF16) return DG_ERR_INVALID_ARG;
  const size_t esz = p->logits_dtype == DG_BF16 ? 2 : 4;
  if (!aligned(logits, esz) || !aligned(E, 16) || !aligned(out, 16)) return DG_ERR_INVALID_ARG;
  const int64_t rows = (int64_t)p->batch * p->canvas_len;
  const SelfcondPlan pl = selfcond_plan(rows, p->vocab, d, device_sm_count(), device_l2_bytes(),
                                        selfcond_materialises(*p));
  if (pl.ws_bytes > 0 && (!ws || ws_bytes < pl.ws_bytes || !aligned(ws, 16)))
    return DG_ERR_WORKSPACE;
  const int dv = device_ok();
  if (dv != DG_OK) return dv;
  cudaGetLastError();
  if (launch_selfcond(*p, logits, *st, E, d, ld_E, out, out_dtype, ws, pl, stream) !=
      cudaSuccess)
    return DG_ERR_CUDA;
  return DG_OK;
}

namespace {
// The fused step writes the feed's operand from the vocabulary pass for bf16
// rows on 16-byte boundaries under the segmented rule (softcapped or not);
// other inputs run the two calls in turn.
bool feed_fusable(const dg_params &p, const void *logits) {
  return p.logits_dtype == DG_BF16 && p.sample_rule == DG_SAMPLE_SEGMENTED &&
         (p.logits_ld * 2) % 16 == 0 && aligned(logits, 16);
}
// Workspace of the fused step: [vocabulary-pass records][per-position R]
// [the operand rows (the self-cond plan's p) | split-K partial sums].
struct FeedLayout {
  size_t off_R, off_sc, total;
  SelfcondPlan plan;
};
FeedLayout feed_layout(const dg_params &p, int32_t d) {
  FeedLayout f;
  const int64_t rows = (int64_t)p.batch * p.canvas_len;
  f.off_R = denoise_ws_bytes(&p);
  f.off_sc = round_up(f.off_R + (size_t)rows * sizeof(float), 256);
  f.plan = selfcond_plan(rows, p.vocab, d, device_sm_count(), device_l2_bytes(), true);
  f.total = f.off_sc + f.plan.ws_bytes;
  return f;
}
}  // namespace

size_t dg_workspace_bytes_feed(const dg_params *p, int32_t d) {
  if (!params_ok(p) || d < 16 || d % 16 != 0) return 0;
  const size_t fused = feed_layout(*p, d).total;
  const size_t apart = dg_workspace_bytes(p, d);
  return fused > apart ? fused : apart;
}

int dg_denoise_step_feed(const dg_params *p, const void *logits, const dg_state *st,
                         const void *E, int32_t d, int64_t ld_E, void *out, int32_t out_dtype,
                         void *ws, size_t ws_bytes, cudaStream_t stream) {
  const int rc = denoise_args_ok(p, logits, st);
  if (rc != DG_OK) return rc;
  if (!E || !out || d < 16 || d % 16 != 0 || ld_E < d || (ld_E * 2) % 16 != 0)
    return DG_ERR_INVALID_ARG;
  if (out_dtype != DG_F32 && out_dtype != DG_BF16) return DG_ERR_INVALID_ARG;
  if (!aligned(E, 16) || !aligned(out, 16)) return DG_ERR_INVALID_ARG;
  if (!st->sc_valid || !st->m || !st->s) return DG_ERR_INVALID_ARG;
  if (!ws || ws_bytes < dg_workspace_bytes_feed(p, d) || !aligned(ws, 16)) return DG_ERR_WORKSPACE;
  const int dv = device_ok();
  if (dv != DG_OK) return dv;
  if (!feed_fusable(*p, logits)) {
    const int r1 = dg_denoise_step(p, logits, st, ws, ws_bytes, stream);
    if (r1 != DG_OK) return r1;
    return dg_selfcond_embed(p, logits, st, E, d, ld_E, out, out_dtype, ws, ws_bytes, stream);
  }
  cudaGetLastError();
  const FeedLayout f = feed_layout(*p, d);
  char *w = reinterpret_cast<char *>(ws);
  Partial *part = reinterpret_cast<Partial *>(w);
  float *feed_R = reinterpret_cast<float *>(w + f.off_R);
  void *ws_sc = w + f.off_sc;
  const int64_t n_pos = (int64_t)p->batch * p->canvas_len;
  const VocabChunking vc = vocab_chunking(n_pos, p->vocab, false);
  if (launch_vocab_pass_feed(*p, logits, *st, part, vc.chunk, vc.n_chunks,
                             reinterpret_cast<uint4 *>(ws_sc), f.plan.p_ld / 8,
                             stream) != cudaSuccess)
    return DG_ERR_CUDA;
  if (launch_canvas_step(*p, *st, part, vc.n_chunks, 0, nullptr, stream, feed_R) != cudaSuccess)
    return DG_ERR_CUDA;
  if (launch_selfcond(*p, logits, *st, E, d, ld_E, out, out_dtype, ws_sc, f.plan, stream,
                      feed_R) != cudaSuccess)
    return DG_ERR_CUDA;
  return DG_OK;
}

int dg_debug_wait_record(uint32_t out[4]) {
  if (!out) return DG_ERR_INVALID_ARG;
  if (dg_selfcond_wait_record(out) != cudaSuccess) return DG_ERR_CUDA;
  return DG_OK;
}

const char *dg_status_string(int code) {
  switch (code) {
    case DG_OK:
      return "ok";
    case DG_ERR_INVALID_ARG:
      return "invalid argument";
    case DG_ERR_UNSUPPORTED:
      return "unsupported device or configuration (needs sm_103)";
    case DG_ERR_WORKSPACE:
      return "workspace missing or too small";
    case DG_ERR_CUDA:
      return "CUDA error";
    case DG_ERR_SCRATCH_LIMIT:
      return "problem larger than the fixed scratch of dg_denoise_step_noalloc";
    default:
      return "unknown status";
  }
}

}  // extern "C"
