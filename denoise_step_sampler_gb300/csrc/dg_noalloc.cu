// dg_denoise_step_noalloc: the sampler step for callers that cannot allocate
// device memory.  Some callers cannot call cudaMalloc or hand out a scratch
// buffer: an engine whose device memory is entirely pre-planned by its own
// pool and lends none to plug-ins, or a host application whose CUDA
// allocations belong to another framework's allocator.  This entry point runs
// the same two kernels as dg_denoise_step, but its per-(position, vocabulary
// chunk) partial records live in a fixed array compiled into the library
// instead of a caller workspace.
//
// The array is static device memory: every GPU that loads the library holds
// it until the process exits.  All calls share it and it keeps the previous
// call's contents; nothing needs clearing, because the vocabulary pass writes
// every record that the canvas kernel later reads.  Two calls whose kernels
// overlap on the GPU (different streams, no ordering) race on the array.
#include <cstdint>

#include "dg_device.cuh"
#include "dg_internal.h"

namespace {

constexpr size_t kScratchRecords = 65536;  // 2 MiB of 32-byte partial records
static __device__ __align__(256) dg::Partial g_noalloc_scratch[kScratchRecords];

// Device address of the array, looked up once per device.  In host code the
// array's name is only a host-side stand-in, so its device address comes
// from cudaGetSymbolAddress with that device current.
constexpr int kMaxDevices = 64;
dg::Partial *g_scratch_ptr[kMaxDevices] = {nullptr};

int scratch_for_current_device(dg::Partial **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return DG_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return DG_ERR_UNSUPPORTED;
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return DG_ERR_CUDA;
    }
    g_scratch_ptr[dev] = reinterpret_cast<dg::Partial *>(p);
  }
  *out = g_scratch_ptr[dev];
  return DG_OK;
}

bool params_ok(const dg_params *p) {
  if (!p) return false;
  if (p->batch < 1 || p->canvas_len < 1 || p->canvas_len > 1024) return false;
  if (p->vocab < 2) return false;
  if (p->logits_dtype != DG_F32 && p->logits_dtype != DG_BF16) return false;
  if (p->logits_ld < p->vocab) return false;
  if (!(p->entropy_budget >= 0.f) || p->entropy_budget > 3.0e38f) return false;
  if (p->conf_threshold != p->conf_threshold) return false;
  if (p->stable_k < 1 || p->step_cap < 1) return false;
  if (p->stop_rule != DG_STOP_ARGMAX_STABLE && p->stop_rule != DG_STOP_ENTROPY) return false;
  if (p->accept_rule != DG_ACCEPT_ENTROPY_BUDGET && p->accept_rule != DG_ACCEPT_MONOTONE)
    return false;
  if (!(p->softcap >= 0.f) || p->softcap > 3.0e38f) return false;
  if (!(p->embed_scale >= 0.f) || p->embed_scale > 3.0e38f) return false;
  return true;
}

bool state_ok(const dg_params *p, const dg_state *st) {
  return st && st->phase && st->request_id && st->temperature && st->rng_step && st->step &&
         st->stable && st->canvas && st->argmax_prev && st->cand && st->argmax && st->accept &&
         st->m && st->s && st->entropy && st->mean_entropy && st->converged && st->sc_valid &&
         st->num_sampled && st->num_rejected && st->emitted && st->device_status &&
         (p->accept_rule != DG_ACCEPT_MONOTONE || (st->committed && st->prev_conf));
}

}  // namespace

extern "C" int dg_denoise_step_noalloc(const dg_params *p, const void *logits, const dg_state *st,
                                       cudaStream_t stream) {
  if (!params_ok(p) || !state_ok(p, st) || !logits) return DG_ERR_INVALID_ARG;
  const size_t esz = p->logits_dtype == DG_BF16 ? 2 : 4;
  if (reinterpret_cast<uintptr_t>(logits) % esz != 0) return DG_ERR_INVALID_ARG;
  const int64_t n_pos = (int64_t)p->batch * p->canvas_len;
  const dg::VocabChunking vc = dg::vocab_chunking(n_pos, p->vocab);
  if (n_pos * (int64_t)vc.n_chunks > (int64_t)kScratchRecords) return DG_ERR_SCRATCH_LIMIT;
  int major = 0, minor = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return DG_ERR_CUDA;
  }
  if (major != 10 || minor != 3) return DG_ERR_UNSUPPORTED;
  dg::Partial *part = nullptr;
  const int rc = scratch_for_current_device(&part);
  if (rc != DG_OK) return rc;
  cudaGetLastError();
  if (dg::launch_vocab_pass(*p, logits, *st, part, vc.chunk, vc.n_chunks, stream) != cudaSuccess)
    return DG_ERR_CUDA;
  if (dg::launch_canvas_step(*p, *st, part, vc.n_chunks, 0, nullptr, stream) != cudaSuccess)
    return DG_ERR_CUDA;
  return DG_OK;
}
