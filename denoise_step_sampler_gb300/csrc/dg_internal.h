// Host-side launchers shared between the C-ABI front end (dg_api.cu) and the
// kernel translation units.  Not part of the public interface.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "dg.h"

namespace dg {

struct Partial;

// Host-side argument checks shared by the entry points (dg_api.cu).  None has
// a side effect.
bool params_ok(const dg_params *p);             // sizes, enums, finite scalars
bool aligned(const void *ptr, size_t a);
bool state_ok_phase_machine(const dg_state *st);  // arrays the phase machine writes
bool state_ok_full(const dg_state *st);           // every array of a denoise step
bool rule_state_ok(const dg_params *p, const dg_state *st);  // monotone-rule arrays
// Every check of dg_denoise_step that precedes its workspace check:
// DG_OK or DG_ERR_INVALID_ARG.
int denoise_args_ok(const dg_params *p, const void *logits, const dg_state *st);
// Bytes of partial records the vocabulary pass writes for these sizes.
size_t denoise_ws_bytes(const dg_params *p);
// DG_OK on an sm_103 device, else DG_ERR_UNSUPPORTED or DG_ERR_CUDA.
int device_ok();

// K1: fused vocabulary pass -> per (position, chunk) partial records.
cudaError_t launch_vocab_pass(const dg_params &p, const void *logits, const dg_state &st,
                              Partial *part, int32_t chunk, int32_t n_chunks, cudaStream_t s);

// K2: per-canvas merge + acceptance + re-noise + convergence + phase machine.
// mode 0: every row by its phase; 1: init rows in row_mask; 2: commit rows in row_mask.
// The fused step's vocabulary pass: as launch_vocab_pass (bf16 rows on
// 16-byte boundaries, segmented rule, no softcap) and it also writes the
// feed's operand, rows of feed_ld8 16-byte words at feed_p.
cudaError_t launch_vocab_pass_feed(const dg_params &p, const void *logits, const dg_state &st,
                                   Partial *part, int32_t chunk, int32_t n_chunks,
                                   uint4 *feed_p, int64_t feed_ld8, cudaStream_t s);
// feed_R (fused step only, else null): per position, the reference R of the
// operand the vocabulary pass wrote, or NaN where the position must fall back.
cudaError_t launch_canvas_step(const dg_params &p, const dg_state &st, const Partial *part,
                               int32_t n_chunks, int mode, const uint8_t *row_mask,
                               cudaStream_t s, float *feed_R = nullptr);

// K4: self-conditioning GEMM (tcgen05 / TMEM).
struct SelfcondPlan {
  int32_t m_tiles;   // ceil(B*C / BM)
  int32_t n_tiles;   // ceil(d / BN)
  int32_t splits;    // K splits over the vocabulary
  int32_t k_blocks;  // ceil(V / BK)
  int32_t kb_per_split;  // k-blocks per split (every split non-empty)
  int32_t n_sms;     // SMs the plan fills in whole waves
  int64_t p_ld;      // materialised p: elements per row (else 0)
  size_t p_bytes;    // materialised p: bytes (else 0)
  size_t ws_bytes;   // materialised p + split-K partial sums (splits > 1)
};
// The split count depends on the sizes, on the number of SMs (n_sms) and, for
// more than 64 row tiles, on the L2 size (l2_bytes); with `materialise` (see
// selfcond_materialises) the plan also holds the materialised p.
SelfcondPlan selfcond_plan(int64_t rows, int32_t V, int32_t d, int32_t n_sms, int64_t l2_bytes,
                           bool materialise);
// Whether the vocabulary pass reads its rows group by group with plain loads
// (fp32 logits, or bf16 rows whose stride is not a multiple of 16 bytes)
// rather than through its load ring; the chunk count depends on it.
inline bool vocab_per_group(const dg_params &p) {
  return p.logits_dtype != DG_BF16 || (p.logits_ld * 2) % 16 != 0;
}
// Whether the self-conditioning call materialises p before the GEMM: a
// softcapped feed, logits the GEMM cannot copy by TMA (fp32, or bf16 rows
// whose stride is not a multiple of 16 bytes), or 1,024 positions (four row
// tiles) and more.  At V = 262,144, d = 2,816 the pass that writes p plus the
// GEMM on it (no rebuild in its producers) took 2 % (4 canvases) to 8 %
// (64 canvases) less than the rebuilding GEMM alone, and 4 % less at 128;
// at 1 and 2 canvases, where the GEMM waits on the E reads, it took 4-9 %
// more.
inline bool selfcond_materialises(const dg_params &p) {
  return p.softcap > 0.f || p.logits_dtype != DG_BF16 || (p.logits_ld * 2) % 16 != 0 ||
         (int64_t)p.batch * p.canvas_len >= 1024;
}

// SMs of the current device (cached per device); 152, the GB300's count, when
// no device can be queried (host-only callers of the workspace query).
int32_t device_sm_count();
// L2 bytes of the current device (cached per device); the GB300's when no
// device can be queried.
constexpr int64_t kGB300L2Bytes = 135528448;
int64_t device_l2_bytes();
// feed_R (fused step only, else null): the GEMM's A rows are the operand the
// vocabulary pass wrote at the start of `ws` (see launch_vocab_pass_feed),
// which the materialisation pass completes for rows where feed_R is NaN.
cudaError_t launch_selfcond(const dg_params &p, const void *logits, const dg_state &st,
                            const void *E, int32_t d, int64_t ld_E, void *out, int32_t out_dtype,
                            void *ws, const SelfcondPlan &plan, cudaStream_t s,
                            const float *feed_R = nullptr);

// Copies the self-cond GEMM's first wait-timeout record to host memory
// (synchronous; diagnostics only).
cudaError_t dg_selfcond_wait_record(uint32_t out[4]);

// Temperature anneal over the rows of the batch (see dg_anneal_temperature).
cudaError_t launch_anneal(int32_t B, const int32_t *step, float *temperature, float t_max,
                          float t_min, int32_t n_steps, const uint8_t *row_mask,
                          cudaStream_t s);

}  // namespace dg
