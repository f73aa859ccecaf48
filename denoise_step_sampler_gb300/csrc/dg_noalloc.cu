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
#include <cuda.h>

#include <cstdint>
#include <mutex>

#include "dg_device.cuh"
#include "dg_internal.h"

namespace {

constexpr size_t kScratchRecords = 65536;  // 2 MiB of 32-byte partial records
static __device__ __align__(256) dg::Partial g_noalloc_scratch[kScratchRecords];

// Device address of the array, looked up once per device with that device
// current (in host code the array's name is only a host-side stand-in).  A
// context created after cudaDeviceReset loads the module again, possibly at
// another address, so each entry remembers the context it was looked up in
// (by its unique id) and is looked up again when the current context differs.
typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

template <class F>
F driver_fn(const char *name) {
  void *fp = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &fp, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return reinterpret_cast<F>(fp);
}

constexpr int kMaxDevices = 64;
struct ScratchEntry {
  unsigned long long ctx_id;
  dg::Partial *ptr;
};
std::mutex g_scratch_mu;
ScratchEntry g_scratch[kMaxDevices] = {};

int scratch_for_current_device(dg::Partial **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return DG_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return DG_ERR_UNSUPPORTED;
  static const CtxGetCurrentFn get_ctx = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  if (!get_ctx || !get_id) return DG_ERR_CUDA;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_ctx(&ctx) != CUDA_SUCCESS) return DG_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchEntry &e = g_scratch[dev];
  if (ctx && get_id(ctx, &id) == CUDA_SUCCESS && e.ptr && e.ctx_id == id) {
    *out = e.ptr;
    return DG_OK;
  }
  // first call on this device, or a new context: look the address up (this
  // also makes the device's primary context current if none was)
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
    cudaGetLastError();
    return DG_ERR_CUDA;
  }
  if (get_ctx(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
    return DG_ERR_CUDA;
  e.ptr = reinterpret_cast<dg::Partial *>(p);
  e.ctx_id = id;
  *out = e.ptr;
  return DG_OK;
}

}  // namespace

extern "C" int dg_denoise_step_noalloc(const dg_params *p, const void *logits, const dg_state *st,
                                       cudaStream_t stream) {
  // the same argument checks as dg_denoise_step, in the same order
  const int rc = dg::denoise_args_ok(p, logits, st);
  if (rc != DG_OK) return rc;
  const int64_t n_pos = (int64_t)p->batch * p->canvas_len;
  const dg::VocabChunking vc = dg::vocab_chunking(n_pos, p->vocab, dg::vocab_per_group(*p));
  if (n_pos * (int64_t)vc.n_chunks > (int64_t)kScratchRecords) return DG_ERR_SCRATCH_LIMIT;
  const int dv = dg::device_ok();
  if (dv != DG_OK) return dv;
  dg::Partial *part = nullptr;
  const int sc = scratch_for_current_device(&part);
  if (sc != DG_OK) return sc;
  cudaGetLastError();
  if (dg::launch_vocab_pass(*p, logits, *st, part, vc.chunk, vc.n_chunks, stream) != cudaSuccess)
    return DG_ERR_CUDA;
  if (dg::launch_canvas_step(*p, *st, part, vc.n_chunks, 0, nullptr, stream) != cudaSuccess)
    return DG_ERR_CUDA;
  return DG_OK;
}
