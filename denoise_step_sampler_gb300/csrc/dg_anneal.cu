// Linear temperature anneal across the denoising steps of a block, on the
// device so that a captured decode loop needs no host round trip:
// T_r = t_max + k (t_min - t_max) / N with k the row's block-local step,
// clamped to [0, N].  "DiffusionGemma Explained" (ML@Berkeley), section
// "Sampling": the `denoise` loop starts at t_max and moves by
// (t_min - t_max) / max_denoising_steps after each step;
// "DiffusionGemma-Lite DIFFUSION.html", section 4.2 item 4.  The closed form is
// evaluated in fp64 and rounded once to fp32.
#include "dg_internal.h"

namespace dg {
namespace {

__global__ void anneal_kernel(int32_t B, const int32_t *__restrict__ step,
                              float *__restrict__ temperature, double t_max, double t_min,
                              int32_t n_steps, const uint8_t *__restrict__ row_mask) {
  const int32_t r = (int32_t)(blockIdx.x * blockDim.x + threadIdx.x);
  if (r >= B) return;
  if (row_mask && !row_mask[r]) return;
  int32_t k = step[r];
  k = k < 0 ? 0 : (k > n_steps ? n_steps : k);
  temperature[r] = (float)(t_max + (double)k * (t_min - t_max) / (double)n_steps);
}

}  // namespace

cudaError_t launch_anneal(int32_t B, const int32_t *step, float *temperature, float t_max,
                          float t_min, int32_t n_steps, const uint8_t *row_mask,
                          cudaStream_t s) {
  if (B <= 0) return cudaSuccess;
  anneal_kernel<<<(B + 255) / 256, 256, 0, s>>>(B, step, temperature, (double)t_max,
                                                 (double)t_min, n_steps, row_mask);
  return cudaGetLastError();
}

}  // namespace dg
