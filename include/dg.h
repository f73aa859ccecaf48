/*
 * dg.h -- C ABI of the GB300 (sm_103a) denoise-step sampler and
 * self-conditioning feed of a uniform-state block-diffusion language model.
 *
 * One call of dg_denoise_step processes every request slot of a batch by its
 * phase (prefill / denoise / commit / idle), as the single vectorised sample
 * step of the vLLM blog "DiffusionGemma: the first dLLM natively supported in
 * vLLM" (section "Putting it together: DiffusionGemmaModelState and
 * DiffusionSampler") does.  dg_selfcond_embed computes the probability-weighted
 * embedding softmax(z/T) . E of "DiffusionGemma Technical Report -- part 2/6",
 * section 3.2, eq. 6.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *     never allocates, frees or synchronises, and keeps no pointer after a call
 *     returns.  Scratch memory is the caller's workspace (dg_workspace_bytes).
 *   - DG_OK means "enqueued on `stream`".  Launch failures are reported as
 *     DG_ERR_CUDA (from cudaGetLastError).  Kernels never trap: conditions only
 *     the device can see set bits in state->device_status (DG_DEV_*).
 *   - Arguments are validated on the host before anything is enqueued; an
 *     invalid call returns an error code and has no side effect.
 *   - No host synchronisation: every call can be captured in a CUDA graph.
 *   - Layouts: B = batch (request slots), C = canvas length, V = vocabulary.
 *     logits are [B][C][ld] row-major, position (r, i) at row r*C + i, with
 *     ld >= V elements between consecutive positions.  Per-position state
 *     arrays are [B*C] at index r*C + i; per-request arrays are [B].
 *   - Random numbers: a counter-based hash of (seed, request_id, rng_step,
 *     position, tag) -- SplitMix64 key chain and MurmurHash3 fmix32 draws --
 *     so a step is reproducible from its inputs alone.
 */
#ifndef DG_H
#define DG_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
typedef enum {
  DG_OK = 0,
  DG_ERR_INVALID_ARG = 1, /* null pointer, bad size, bad alignment, bad enum   */
  DG_ERR_UNSUPPORTED = 2, /* device is not sm_103 / unsupported dtype combo    */
  DG_ERR_WORKSPACE = 3,   /* workspace pointer null or smaller than required   */
  DG_ERR_CUDA = 4,        /* a CUDA runtime call or a launch failed            */
  DG_ERR_SCRATCH_LIMIT = 5 /* too large for dg_denoise_step_noalloc's fixed scratch */
} dg_status;

/* Sticky bits OR-ed into state->device_status[0] by the kernels. */
enum {
  DG_DEV_NONFINITE_LOGITS = 1u, /* a denoise position held NaN / +inf or was all -inf */
  DG_DEV_BAD_TEMPERATURE = 2u,  /* a denoise row had T <= 0 or non-finite             */
  DG_DEV_BAD_TOKEN = 4u,        /* a committed token was outside [0, V)               */
  DG_DEV_WAIT_TIMEOUT = 8u,     /* a bounded wait in the self-cond GEMM gave up       */
  DG_DEV_BAD_PHASE = 16u        /* a phase value outside DG_PHASE_*                  */
};

/* Request phases (vLLM blog, "Putting it together": prefill, denoise, commit). */
enum { DG_PHASE_PREFILL = 0, DG_PHASE_DENOISE = 1, DG_PHASE_COMMIT = 2, DG_PHASE_IDLE = 3 };

/* Element types. */
enum { DG_F32 = 0, DG_BF16 = 1 };

/* Convergence rules (dg_params.stop_rule).
 * DG_STOP_ARGMAX_STABLE: the argmax canvas unchanged for stable_k consecutive
 *   steps and the mean entropy below conf_threshold ("DiffusionGemma
 *   Explained", "Sampling"; vLLM blog, "Entropy-bounded denoising");
 * DG_STOP_ENTROPY: the mean entropy below conf_threshold for stable_k
 *   consecutive steps ("DiffusionGemma-Lite DIFFUSION.html", section 4.4).
 * Either rule also stops at step_cap. */
enum { DG_STOP_ARGMAX_STABLE = 0, DG_STOP_ENTROPY = 1 };

/* Acceptance rules (dg_params.accept_rule).
 * DG_ACCEPT_ENTROPY_BUDGET: positions by ascending (H, i) accepted while the
 *   exclusive prefix sum of entropies is <= entropy_budget, the first always;
 *   the rest re-noised ("DiffusionGemma Explained", "Sampling", step 3).
 * DG_ACCEPT_MONOTONE: unchanged-or-stronger commits ("DiffusionGemma-Lite
 *   DIFFUSION.html", section 4.2): a position commits when its argmax equals
 *   the previous step's or its confidence (largest probability, 1/s) is >=
 *   the previous step's; a newly committed position takes the Gumbel-max
 *   candidate, an earlier committed one keeps its token, every other one is
 *   re-noised.  A block starts with nothing committed and prev_conf = +inf
 *   (so its first step commits nothing); commit rows emit the committed tokens
 *   and the last candidates elsewhere.  Needs dg_state.committed / prev_conf. */
enum { DG_ACCEPT_ENTROPY_BUDGET = 0, DG_ACCEPT_MONOTONE = 1 };

/* Gumbel-max sampling rules for the candidate (dg_params.sample_rule).  Both
 * draw the candidate exactly from softmax(z/T) (vLLM blog, "Putting it
 * together": argmax(logits/T + gumbel_noise)); they use different random
 * numbers, so their candidates differ draw by draw.
 * DG_SAMPLE_GROUPED: argmax_v(z_v/T + G_v) with one Gumbel per index, from
 *   the library's group construction (8 indices share one minimum draw).
 * DG_SAMPLE_SEGMENTED: the chunk-level variant.  The vocabulary is cut into
 *   segments of 32 indices (superblock j = [1024 j, 1024 j + 1024); its
 *   segment l holds the four groups of 8 at offsets 8 l + 256 u, u < 4).  A
 *   segment wins by Gumbel-max over ln(sum of its exp(z/T)) with one Gumbel
 *   per segment; the candidate is the Gumbel-max index inside it (one Gumbel
 *   per index of that segment only).  By the max-stability of the Gumbel law
 *   the result has the same distribution; the pass hashes once per 32
 *   indices instead of screening every group of 8. */
enum { DG_SAMPLE_GROUPED = 0, DG_SAMPLE_SEGMENTED = 1 };

/* Scalar parameters of a call (host memory, read during the call only). */
typedef struct {
  int32_t batch;          /* B >= 1 request slots                                */
  int32_t canvas_len;     /* C, 1 <= C <= 1024 (the pages use 256)               */
  int32_t vocab;          /* V, 2 <= V < 2^31                                    */
  int32_t logits_dtype;   /* DG_F32 or DG_BF16                                   */
  int64_t logits_ld;      /* elements between consecutive positions, >= V       */
  uint64_t seed;          /* random-number seed of the whole run                 */
  float entropy_budget;   /* nats, finite, >= 0 (acceptance budget)              */
  float conf_threshold;   /* nats; converge when mean entropy < this (not NaN)   */
  int32_t stable_k;       /* >= 1 consecutive steps the stop rule asks for       */
  int32_t step_cap;       /* >= 1 maximum denoise steps per block                */
  int32_t stop_rule;      /* DG_STOP_* (0 = argmax-stable)                       */
  int32_t accept_rule;    /* DG_ACCEPT_* (0 = entropy budget)                    */
  float softcap;          /* c of the logit softcap z <- c tanh(z / c), applied to
                             every stored logit before any other use ("The
                             Annotated DiffusionGemma", "Logit Softcapping"):
                             m, s, H, the argmax, the candidate and the
                             self-conditioning softmax all see capped logits.
                             0 = off; finite, >= 0                              */
  float embed_scale;      /* factor on dg_selfcond_embed's output (the model's
                             embedding scale on the probability-weighted
                             embedding, "The Annotated DiffusionGemma", the
                             forward pass); 0 = 1; finite, >= 0                 */
  int32_t sample_rule;    /* DG_SAMPLE_* (0 = grouped)                           */
} dg_params;

/* Per-request state: device arrays, preallocated by the caller and updated in
 * place (vLLM blog, "Putting it together": per-request state lives in
 * preallocated GPU tensors).  Shapes [B] or [B*C].  All fields are required
 * by dg_denoise_step; dg_init_canvas / dg_commit use the subset they touch. */
typedef struct {
  uint8_t *phase;              /* [B]   in/out DG_PHASE_*                            */
  const uint64_t *request_id;  /* [B]   in   identity of the slot for the hash       */
  const float *temperature;    /* [B]   in   T_r > 0 (caller anneals it if wanted)   */
  uint64_t *rng_step;          /* [B]   in/out +1 per processed call, never reset    */
  int32_t *step;               /* [B]   in/out denoise steps in the current block    */
  int32_t *stable;             /* [B]   in/out consecutive steps meeting the stop rule */
  int32_t *canvas;             /* [B*C] out  next tokens (accepted cand or re-noise) */
  int32_t *argmax_prev;        /* [B*C] in/out argmax canvas of the last step        */
  int32_t *cand;               /* [B*C] out  Gumbel-max candidates                   */
  int32_t *argmax;             /* [B*C] out  clean argmax of this step               */
  uint8_t *accept;             /* [B*C] out  1 = accepted (newly committed) position */
  float *m;                    /* [B*C] out  max_v z_v / T   (NaN if invalid; z after
                                  the softcap when dg_params.softcap > 0)           */
  float *s;                    /* [B*C] out  sum_v exp(z_v/T - m)                   */
  float *entropy;              /* [B*C] out  H in nats      (NaN if invalid)        */
  float *mean_entropy;         /* [B]   out  mean of H over the canvas              */
  uint8_t *converged;          /* [B]   out  1 = converged this step                */
  uint8_t *sc_valid;           /* [B]   out  1 = row feeds self-conditioning next    */
  int32_t *num_sampled;        /* [B]   out  0 (prefill/denoise) or C (commit)       */
  int32_t *num_rejected;       /* [B]   out  C (denoise) or 0                        */
  int32_t *emitted;            /* [B*C] out  tokens emitted by commit rows           */
  uint32_t *device_status;     /* [1]   in/out sticky DG_DEV_* bits                  */
  uint8_t *committed;          /* [B*C] in/out frozen positions (DG_ACCEPT_MONOTONE;
                                  may be NULL under the other rule)                 */
  float *prev_conf;            /* [B*C] in/out last step's confidence (same)        */
} dg_state;

/* Bytes of caller workspace needed by dg_denoise_step and, if d > 0, by
 * dg_selfcond_embed with embedding width d (one buffer serves both, as the
 * calls are ordered on one stream).  Returns 0 if `p` is invalid.  Depends on
 * the sizes in `p`, on d and on the SM count and L2 size of the current
 * device (the self-conditioning GEMM splits the vocabulary by a cost model of
 * its waves of CTAs and of the split-K reduction and, for more than 64 row
 * tiles of 256 positions, further until one split's slice of E fits in L2;
 * the partial sums take splits*B*C*d*4 bytes); query it with the device
 * current that the calls will run on.  With d > 0 it includes the feed's
 * materialised probabilities, B*C rows of V rounded up to
 * 8 bf16 (about B*C*V*2 bytes: 1.07 GB for 8 x 256 positions at V = 262,144,
 * 17.2 GB for 128 x 256), when B*C >= 1024, when p->softcap > 0, or when the
 * logits are fp32 or bf16 rows whose stride (logits_ld * 2 bytes) is not a
 * multiple of 16. */
size_t dg_workspace_bytes(const dg_params *p, int32_t d);

/* Stand-alone canvas initialisation (the prefill case) of the rows r with
 * row_mask[r] != 0 (device [B] uint8): canvas = uniform random tokens, counters
 * reset, phase = DENOISE, rng_step += 1.  Technical Report section 3.2
 * "Canvas initialization"; vLLM blog, prefill bullet.  Uses phase, request_id,
 * rng_step, step, stable, canvas, converged, sc_valid, num_sampled,
 * num_rejected. */
int dg_init_canvas(const dg_params *p, const dg_state *st, const uint8_t *row_mask,
                   cudaStream_t stream);

/* One sampler step over the whole batch, each row by its phase:
 *   PREFILL -> as dg_init_canvas;  COMMIT -> as dg_commit;  IDLE -> untouched;
 *   DENOISE -> per position: y = z/T, (m, s), entropy, clean argmax, Gumbel-max
 *   candidate argmax(y + G); per canvas: entropy-bounded acceptance (positions
 *   by ascending (H, i), accepted while the exclusive prefix sum of entropies
 *   is <= budget, the first always), re-noise of rejected positions to uniform
 *   tokens, convergence ((stable >= k and mean H < thr) or step >= cap) which
 *   moves the row to COMMIT.
 * Sources: "DiffusionGemma Explained" (ML@Berkeley), section "Sampling",
 * steps 1-4; Technical Report section 3.3; vLLM blog sections "Entropy-bounded
 * denoising" and "Putting it together".
 * `logits`: device [B][C][logits_ld] of p->logits_dtype, aligned to its
 * element size; only DENOISE rows are read.  `ws`: workspace of at least
 * dg_workspace_bytes(p, 0) bytes.  Two kernel launches. */
int dg_denoise_step(const dg_params *p, const void *logits, const dg_state *st,
                    void *ws, size_t ws_bytes, cudaStream_t stream);

/* Self-conditioning feed, Technical Report section 3.2 eq. 6 (the p0 E inside
 * FFW(p0 E)); "DiffusionGemma Explained", section "Self-conditioning":
 *   out[r*C + i, :] = sum_v softmax(z_{r,i} / T_r)_v * E[v, :]
 * for rows with sc_valid[r] = 1 and phase[r] = DENOISE and positions whose
 * entropy is finite; every other output row is written as zeros (first
 * decode step and encoder passes see zero self-conditioning: vLLM blog,
 * "Self-conditioning").  Must follow dg_denoise_step on the same stream (it
 * reads the m and s that step wrote) and use the same logits.
 * `E`: device bf16 [V][ld_E], 16-byte aligned, ld_E >= d, ld_E*2 % 16 == 0.
 * `d`: 16 <= d, d % 16 == 0.  `out`: device [B*C][d] of out_dtype (DG_F32 or
 * DG_BF16).  `ws`: at least dg_workspace_bytes(p, d) bytes.  Products run on
 * the tensor cores in bf16 with fp32 accumulation.  One to three kernel
 * launches: from 1,024 positions on, for a softcapped feed, for fp32 logits,
 * or for bf16 rows whose stride is not a multiple of 16 bytes, a first kernel
 * writes the probabilities to `ws` once and the GEMM reads them from there
 * (otherwise the GEMM rebuilds them from the logits tile by tile); the GEMM;
 * a split-K reduction when the vocabulary is split. */
int dg_selfcond_embed(const dg_params *p, const void *logits, const dg_state *st,
                      const void *E, int32_t d, int64_t ld_E, void *out, int32_t out_dtype,
                      void *ws, size_t ws_bytes, cudaStream_t stream);

/* The sampler step and the self-conditioning feed in one call: the same
 * results as dg_denoise_step followed by dg_selfcond_embed on the same
 * stream (outputs equal; the feed within the same tolerance), with the
 * logits read once for both where the inputs allow.  For bf16 logits whose
 * rows start on 16-byte boundaries, under DG_SAMPLE_SEGMENTED (with or
 * without a softcap; with one, z below is the capped logit), the vocabulary
 * pass also writes the feed's operand
 * 2^(z c - R) (bf16, c = log2(e)/T) into the workspace as it streams the
 * logits, with R = ceil(m' log2 e) + 32 from each position's previous
 * maximum m' (st->m before the call); positions whose new maximum z_max
 * leaves |z_max c - R| > 96 (the first step of a request, large jumps), or
 * whose logits are not finite, get p written by a separate pass instead.
 * The GEMM then reads the operand without rebuilding it, and each output row
 * is scaled by 2^(R - log2 sum 2^(z c)).  Other inputs run the two calls in
 * turn.  Arguments as for the two calls; `ws`: at least
 * dg_workspace_bytes_feed(p, d) bytes (about B*C*V*2 bytes more than
 * dg_workspace_bytes(p, d) below 1,024 positions).  Three to five kernel
 * launches.  The pages describe the two steps apart; the fusion is this
 * library's. */
size_t dg_workspace_bytes_feed(const dg_params *p, int32_t d);
int dg_denoise_step_feed(const dg_params *p, const void *logits, const dg_state *st,
                         const void *E, int32_t d, int64_t ld_E, void *out, int32_t out_dtype,
                         void *ws, size_t ws_bytes, cudaStream_t stream);

/* Stand-alone commit (the commit case) of the rows with row_mask[r] != 0:
 * emitted = argmax_prev (the clean argmax canvas, vLLM blog "Entropy-bounded
 * denoising"), num_sampled = C, num_rejected = 0, a fresh random canvas,
 * counters reset, phase = DENOISE, rng_step += 1. */
int dg_commit(const dg_params *p, const dg_state *st, const uint8_t *row_mask,
              cudaStream_t stream);

/* Linear temperature anneal over the denoising steps of a block:
 *   temperature[r] = t_max + k (t_min - t_max) / n_steps,
 * k = step[r] (the row's block-local step counter, dg_state.step) clamped to
 * [0, n_steps], evaluated in fp64 and rounded once to fp32.
 * Sources: "DiffusionGemma Explained" (ML@Berkeley), section "Sampling" (the
 * denoise loop starts at t_max and moves by (t_min - t_max) / N per step);
 * "DiffusionGemma-Lite DIFFUSION.html", section 4.2 item 4.
 * Call it before dg_denoise_step so that the vocabulary pass, the canvas step
 * and the self-conditioning feed of that step all read the same temperature.
 * `step`: device [B] int32 (in), `temperature`: device [B] fp32 (out), both
 * owned by the caller; `row_mask`: device [B] (nonzero = update the row) or
 * NULL for every row.  t_max, t_min > 0 and finite, n_steps >= 1, else
 * DG_ERR_INVALID_ARG with nothing enqueued.  One kernel launch; no
 * counterpart to the state layout: the pages anneal on the host. */
int dg_anneal_temperature(const dg_params *p, const int32_t *step, float *temperature,
                          float t_max, float t_min, int32_t n_steps,
                          const uint8_t *row_mask, cudaStream_t stream);

/* dg_denoise_step without a workspace, for callers that cannot allocate
 * device memory (an engine whose device memory is all pre-planned by its own
 * pool, or a host application whose allocations belong to another
 * framework's allocator).  The sources describe no such variant; it exists
 * for deployment only.  Same arguments, semantics and results as
 * dg_denoise_step; the scratch it needs (one 32-byte record per position and
 * vocabulary chunk) lives in a 2 MiB array inside the library that every GPU
 * loading the library keeps until the process exits.  Limit: batch *
 * canvas_len * chunks <= 65536 records (V = 262144 takes 8 chunks per
 * position up to 1216 positions, 4 up to 9728 and 2 beyond, so up to 32768
 * positions fit); larger problems return DG_ERR_SCRATCH_LIMIT before
 * anything is enqueued.  The first call on a device, and the first call in a
 * new context of that device (after cudaDeviceReset), looks up the array's
 * device address (cudaGetSymbolAddress) with that device current; make that
 * first call before any stream capture.  Calls share the array, so two calls
 * whose kernels may overlap on the GPU race: order them on one stream.
 * Allocates and frees nothing. */
int dg_denoise_step_noalloc(const dg_params *p, const void *logits, const dg_state *st,
                            cudaStream_t stream);

/* Diagnostics: copies to host memory the first bounded wait of the self-cond
 * GEMM that gave up since the library was loaded, as {set, block, where,
 * parity}; set = 0 if none did.  where = role << 28 | barrier << 24 |
 * stage << 16 | k-iteration (roles 0 TMA, 1 MMA, 2 producer, 3 epilogue;
 * barriers 0 E tile landed, 1 a_ready, 2 E stage free, 3 tmem_full, 4 logits
 * tile landed, 5 logits stage free).  Synchronous; not for
 * use inside a captured graph. */
int dg_debug_wait_record(uint32_t out[4]);

/* Static description of a return code. */
const char *dg_status_string(int code);

#ifdef __cplusplus
}
#endif
#endif /* DG_H */
