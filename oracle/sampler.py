"""fp64 oracle of one sampler step (test infrastructure; see the package
docstring).

Every row r of the batch carries a phase and is processed by it, as in the
vLLM blog's single vectorised sample step (section "Putting it together:
DiffusionGemmaModelState and DiffusionSampler"):

* PREFILL -- the canvas becomes uniform random tokens; nothing is sampled.
* DENOISE -- per position i: tempered logits y = z / T, softmax p, entropy
  H = -sum p ln p ("DiffusionGemma Explained", "Sampling", step 2), clean
  argmax of z, Gumbel-max candidate argmax(y + G) (vLLM blog, sampler
  bullet "denoising").  Then entropy-bounded acceptance: positions sorted by
  (H, i) ascending are accepted while the exclusive prefix sum of entropies
  stays within the budget ("DiffusionGemma Explained", "Sampling", step 3;
  Technical Report section 3.3 "Entropy-bounded token refinement"); the first
  is always accepted.  Rejected positions are re-noised to uniform tokens
  (Technical Report section 3.3).  Convergence: the argmax canvas equal to
  the previous step's for ``stable_k`` consecutive steps and mean entropy
  below the threshold, or the step cap (vLLM blog, same section; Technical
  Report section 3.3 "Adaptive stopping heuristic").
* COMMIT  -- emit the clean argmax canvas of the last denoise step, re-draw
  the canvas for the next block and reset the per-request counters (vLLM
  blog, sampler bullet "commit").
* IDLE    -- untouched.

Where the pages are silent or disagree, the reading taken is stated next to
the code that depends on it.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

from . import rng

PHASE_PREFILL = 0
PHASE_DENOISE = 1
PHASE_COMMIT = 2
PHASE_IDLE = 3

NEAR_TIE = 1e-4  # gap below which an index decision is flagged, not compared

# convergence rules
STOP_ARGMAX_STABLE = 0   # argmax canvas unchanged for k steps and mean entropy below thr
STOP_ENTROPY = 1         # mean entropy below thr for k consecutive steps
# acceptance rules
ACCEPT_ENTROPY_BUDGET = 0  # lowest-entropy positions within the entropy budget
ACCEPT_MONOTONE = 1        # unchanged-or-stronger commits, frozen once committed
# Gumbel-max sampling rules (both draw the candidate exactly from softmax(y))
SAMPLE_GROUPED = 0    # argmax(y + G) with per-index G from the group construction
SAMPLE_SEGMENTED = 1  # a segment by Gumbel-max over segment masses, then an index in it


@dataclass
class Params:
    batch: int
    canvas_len: int
    vocab: int
    seed: int
    entropy_budget: float
    conf_threshold: float
    stable_k: int
    step_cap: int
    stop_rule: int = STOP_ARGMAX_STABLE
    accept_rule: int = ACCEPT_ENTROPY_BUDGET
    softcap: float = 0.0       # c of the logit softcap; 0 = logits used as stored
    embed_scale: float = 0.0   # factor on the self-conditioning feed; 0 = 1
    sample_rule: int = SAMPLE_GROUPED


@dataclass
class State:
    """Per-request state; arrays are numpy, shapes [B] or [B, C]."""

    phase: np.ndarray          # uint8 [B]
    request_id: np.ndarray     # uint64 [B]
    temperature: np.ndarray    # float [B]
    rng_step: np.ndarray       # uint64 [B]
    step: np.ndarray           # int32 [B]
    stable: np.ndarray         # int32 [B]
    canvas: np.ndarray         # int32 [B, C]
    argmax_prev: np.ndarray    # int32 [B, C]
    cand: np.ndarray = None    # int32 [B, C]
    argmax: np.ndarray = None  # int32 [B, C]
    accept: np.ndarray = None  # uint8 [B, C]
    m: np.ndarray = None       # float64 [B, C]
    s: np.ndarray = None       # float64 [B, C]
    entropy: np.ndarray = None  # float64 [B, C]
    mean_entropy: np.ndarray = None  # float64 [B]
    converged: np.ndarray = None     # uint8 [B]
    sc_valid: np.ndarray = None      # uint8 [B]
    num_sampled: np.ndarray = None   # int32 [B]
    num_rejected: np.ndarray = None  # int32 [B]
    emitted: np.ndarray = None       # int32 [B, C]
    committed: np.ndarray = None     # uint8 [B, C] (monotone rule)
    prev_conf: np.ndarray = None     # float64 [B, C] (monotone rule)

    def copy(self):
        out = State(**{k: (None if v is None else np.array(v, copy=True))
                       for k, v in self.__dict__.items()})
        return out


@dataclass
class Flags:
    """Near-tie flags: where fp64 and any fp32 evaluation may legitimately
    take a different discrete decision (gap or distance below 1e-4)."""

    cand: np.ndarray = None      # bool [B, C]: top-2 perturbed-score gap < 1e-4
    accept: np.ndarray = None    # bool [B]: acceptance cut within 1e-4
    converged: np.ndarray = None  # bool [B]: |mean H - thr| < 1e-4 where thr decides
    gaps: np.ndarray = None      # float64 [B, C]
    commit: np.ndarray = None    # bool [B, C]: |conf - prev_conf| < 1e-4 (monotone rule)


# --------------------------------------------------------------------------
# per position


@dataclass
class PositionResult:
    valid: bool
    m: float
    s: float
    entropy: float
    argmax: int
    cand: int
    gap: float


def softcap(z, c):
    """Logit softcapping ("The Annotated DiffusionGemma", "Putting Them
    together" / "Logit Softcapping"): z_capped = c tanh(z / c), applied to the
    final logits before anything reads them.  float64; c = 0 leaves ``z``
    unchanged.  tanh maps +-inf to +-1, so infinite logits become +-c; NaN
    stays NaN."""
    z = np.asarray(z, dtype=np.float64)
    if c == 0:
        return z
    return c * np.tanh(z / c)


def gumbel_keys(seed, request_id, rng_step, position):
    p = rng.position_key(seed, request_id, rng_step, position)
    return (rng.stream_key(p, rng.TAG_GMIN), rng.stream_key(p, rng.TAG_GARG),
            rng.stream_key(p, rng.TAG_GREST))


def segment_keys(seed, request_id, rng_step, position):
    """Stream keys (K_SEG, K_WITHIN) of the segmented rule at one position."""
    p = rng.position_key(seed, request_id, rng_step, position)
    return rng.stream_key(p, rng.TAG_SEG), rng.stream_key(p, rng.TAG_WITHIN)


def segmented_candidate(y, ks, kw):
    """Hierarchical Gumbel-max (the chunk-level variant of the vLLM blog's
    argmax(logits/T + gumbel_noise), section "Putting it together").

    Step 1: each segment k (rng.segment_of) has mass W_k = sum_{v in k}
    exp(y_v - m); the winning segment is argmax_k (ln W_k + G_k), G_k =
    -ln exp1(draw32(K_SEG, k)) standard Gumbel, lowest k on ties.  By
    Gumbel-max, P(k) = W_k / sum W.  Step 2: inside it, the candidate is
    argmax_v (y_v + G'_v), G'_v = -ln exp1(draw32(K_WITHIN, v)), lowest v on
    ties, so P(v | k) = exp(y_v) / W_k and P(v) = softmax(y)_v exactly.
    Returns (candidate, gap): gap is the smaller of the two top-2 score gaps
    (segments, and indices inside the winning segment)."""
    y = np.asarray(y, dtype=np.float64)
    V = y.size
    m = float(np.max(y))
    e = np.exp(y - m)
    seg = rng.segment_of(np.arange(V))
    W = np.bincount(seg, weights=e)
    k_all = np.arange(W.size)
    E = rng.exp1(rng.draw32(ks, k_all.astype(np.uint32)))
    with np.errstate(divide="ignore"):
        score = np.log(W) - np.log(E)
    k = int(np.argmax(score))
    gap_seg = float(score[k] - np.max(np.delete(score, k))) if W.size > 1 else math.inf
    members = rng.segment_members(k, V)
    Ew = rng.exp1(rng.draw32(kw, members.astype(np.uint32)))
    s2 = y[members] - np.log(Ew)
    i = int(np.argmax(s2))
    gap_in = float(s2[i] - np.max(np.delete(s2, i))) if members.size > 1 else math.inf
    return int(members[i]), min(gap_seg, gap_in)


def vocab_pass(z, T, ka, kb, kc, sample_rule=SAMPLE_GROUPED, seg_keys=None) -> PositionResult:
    """All per-position quantities of one logit row ``z`` (float64, the stored
    logits widened exactly) at temperature ``T``.  The candidate follows
    ``sample_rule``: SAMPLE_GROUPED uses the Gumbel keys (ka, kb, kc),
    SAMPLE_SEGMENTED the segment keys ``seg_keys`` = (K_SEG, K_WITHIN).

    Validity (a reading; the pages are silent): a row holding a NaN or a +inf
    logit, a row whose logits are all -inf, or a non-positive / non-finite
    temperature is invalid: entropy, m and s are NaN, argmax = cand = 0.
    -inf logits in a valid row are tokens of probability zero.
    """
    z = np.asarray(z, dtype=np.float64)
    V = z.size
    bad = (not (T > 0.0 and math.isfinite(T)) or np.isnan(z).any()
           or np.isposinf(z).any() or not np.isfinite(z).any())
    if bad:
        return PositionResult(False, math.nan, math.nan, math.nan, 0, 0, math.inf)
    # temperature (Technical Report eq. 6: Softmax(L_t / tau_t))
    y = z / T
    # softmax with max subtraction: p_v = exp(y_v - m) / s
    m = float(np.max(y))
    e = np.exp(y - m)
    s = float(np.sum(e))
    p = e / s
    # entropy -sum p ln p over the support ("DiffusionGemma Explained", step 2)
    nz = p > 0
    H = float(-np.sum(p[nz] * np.log(p[nz])))
    # clean argmax, lowest index on ties (vLLM blog: the argmax canvas)
    am = int(np.argmax(z))
    if sample_rule == SAMPLE_SEGMENTED:
        cand, gap = segmented_candidate(y, *seg_keys)
        return PositionResult(True, m, s, H, am, cand, gap)
    # Gumbel-max candidate argmax(y + G), lowest index on ties
    G = rng.gumbel_noise(V, ka, kb, kc)
    score = y + G
    cand = int(np.argmax(score))
    if V > 1:
        rest = np.delete(score, cand)
        gap = float(score[cand] - np.max(rest))
    else:
        gap = math.inf
    return PositionResult(True, m, s, H, am, cand, gap)


# --------------------------------------------------------------------------
# per canvas


def accept_mask(H, budget):
    """Entropy-bounded acceptance of one canvas.

    Positions sorted by (H_i, i) ascending (invalid positions, H = NaN, sort
    last as +inf); the k-th in that order is accepted iff k = 0 or the sum of
    the entropies before it is <= budget ("DiffusionGemma Explained",
    "Sampling", step 3: the largest prefix whose exclusive sum stays within
    the bound).  Invalid positions (a reading; the pages are silent) are
    never accepted, so a canvas with no valid position accepts nothing.
    Returns (accept[C] bool, flagged) where ``flagged`` says that the cut
    lies within 1e-4 of a decision boundary.
    """
    H = np.asarray(H, dtype=np.float64)
    C = H.size
    key = np.where(np.isnan(H), np.inf, H)
    order = sorted(range(C), key=lambda i: (key[i], i))
    acc = np.zeros(C, dtype=bool)
    prefix = 0.0
    flagged = False
    for k, i in enumerate(order):
        if k > 0 and abs(prefix - budget) < NEAR_TIE:
            flagged = True
        if np.isfinite(key[i]) and (k == 0 or prefix <= budget):
            acc[i] = True
        prefix = prefix + key[i]
    n_acc = int(acc.sum())
    if 0 < n_acc < C:
        a, b = key[order[n_acc - 1]], key[order[n_acc]]
        if abs(b - a) < NEAR_TIE:
            flagged = True
    return acc, flagged


def renoise_tokens(seed, request_id, rng_step, C, V):
    p = rng.position_key(seed, request_id, rng_step, np.arange(C, dtype=np.uint64))
    return rng.uniform_token(rng.stream_key(p, rng.TAG_RENOISE), V).astype(np.int32)


def init_tokens(seed, request_id, rng_step, C, V):
    p = rng.position_key(seed, request_id, rng_step, np.arange(C, dtype=np.uint64))
    return rng.uniform_token(rng.stream_key(p, rng.TAG_INIT), V).astype(np.int32)


def _ensure_outputs(st: State, B, C):
    def z(shape, dt, fill=0):
        return np.full(shape, fill, dtype=dt)
    if st.cand is None: st.cand = z((B, C), np.int32)
    if st.argmax is None: st.argmax = z((B, C), np.int32)
    if st.accept is None: st.accept = z((B, C), np.uint8)
    if st.m is None: st.m = z((B, C), np.float64, np.nan)
    if st.s is None: st.s = z((B, C), np.float64, np.nan)
    if st.entropy is None: st.entropy = z((B, C), np.float64, np.nan)
    if st.mean_entropy is None: st.mean_entropy = z((B,), np.float64, np.nan)
    if st.converged is None: st.converged = z((B,), np.uint8)
    if st.sc_valid is None: st.sc_valid = z((B,), np.uint8)
    if st.num_sampled is None: st.num_sampled = z((B,), np.int32)
    if st.num_rejected is None: st.num_rejected = z((B,), np.int32)
    if st.emitted is None: st.emitted = z((B, C), np.int32)
    if st.committed is None: st.committed = z((B, C), np.uint8)
    if st.prev_conf is None: st.prev_conf = z((B, C), np.float64, np.inf)


def _reset_commit_state(p: Params, st: State, r: int):
    """Start of a block under the monotone rule: nothing frozen, and no
    previous confidence (reading: +inf, so that the first step commits
    nothing -- it has no previous mode to compare with either)."""
    if p.accept_rule == ACCEPT_MONOTONE:
        st.committed[r] = 0
        st.prev_conf[r] = np.inf


def prefill_row(p: Params, st: State, r: int):
    """Canvas of uniform random tokens (Technical Report section 3.2 "Canvas
    initialization"; vLLM blog: prefill initialises the canvas and samples
    nothing).  num_rejected = 0 is a reading (the blog names only
    num_sampled)."""
    C, V = p.canvas_len, p.vocab
    st.canvas[r] = init_tokens(p.seed, st.request_id[r], st.rng_step[r], C, V)
    st.step[r] = 0
    st.stable[r] = 0
    st.num_sampled[r] = 0
    st.num_rejected[r] = 0
    st.sc_valid[r] = 0
    st.converged[r] = 0
    st.phase[r] = PHASE_DENOISE
    st.rng_step[r] = st.rng_step[r] + np.uint64(1)
    _reset_commit_state(p, st, r)


def commit_row(p: Params, st: State, r: int):
    """Emit the clean argmax canvas of the last denoise step (vLLM blog: the
    committed tokens are the clean argmax prediction), then start the next
    block from a fresh random canvas with reset counters.

    Under the monotone rule the block's result is the frozen tokens where a
    position committed and the last step's draw elsewhere
    ("DiffusionGemma-Lite DIFFUSION.html", section 4.2 item 5: every position
    ends with its best posterior guess even if it never committed)."""
    C, V = p.canvas_len, p.vocab
    if p.accept_rule == ACCEPT_MONOTONE:
        st.emitted[r] = np.where(st.committed[r] != 0, st.canvas[r], st.cand[r])
    else:
        st.emitted[r] = st.argmax_prev[r]
    st.num_sampled[r] = C
    st.num_rejected[r] = 0
    st.canvas[r] = init_tokens(p.seed, st.request_id[r], st.rng_step[r], C, V)
    st.step[r] = 0
    st.stable[r] = 0
    st.sc_valid[r] = 0
    st.converged[r] = 0
    st.phase[r] = PHASE_DENOISE
    st.rng_step[r] = st.rng_step[r] + np.uint64(1)
    _reset_commit_state(p, st, r)


def _vocab_job(args):
    """One position's vocabulary pass (a picklable unit for a process pool).
    The softcap, when set, is applied to the stored logits first."""
    z, T, seed, rid, rstep, i, cap, rule = args
    ka, kb, kc = gumbel_keys(seed, rid, rstep, i)
    sk = segment_keys(seed, rid, rstep, i) if rule == SAMPLE_SEGMENTED else None
    return vocab_pass(softcap(z, cap), T, ka, kb, kc, rule, sk)


def denoise_row(p: Params, st: State, r: int, logits_row, flags: Flags, mapper=map):
    """One denoise step of row r from its logits ``logits_row`` [C, V].
    ``mapper`` evaluates the independent per-position passes (``map`` or a
    process pool's ``map``)."""
    C, V = p.canvas_len, p.vocab
    T = float(st.temperature[r])
    jobs = [(logits_row[i], T, p.seed, st.request_id[r], st.rng_step[r], i, p.softcap,
             p.sample_rule) for i in range(C)]
    H = np.empty(C)
    for i, res in enumerate(mapper(_vocab_job, jobs)):
        st.m[r, i] = res.m
        st.s[r, i] = res.s
        st.entropy[r, i] = res.entropy
        st.argmax[r, i] = res.argmax
        st.cand[r, i] = res.cand
        flags.gaps[r, i] = res.gap
        flags.cand[r, i] = res.gap < NEAR_TIE
        H[i] = res.entropy
    R = renoise_tokens(p.seed, st.request_id[r], st.rng_step[r], C, V)
    if p.accept_rule == ACCEPT_MONOTONE:
        monotone_commit(st, r, H, R, flags)
    else:
        acc, aflag = accept_mask(H, p.entropy_budget)
        flags.accept[r] = aflag
        st.accept[r] = acc.astype(np.uint8)
        st.canvas[r] = np.where(acc, st.cand[r], R)
    # convergence (vLLM blog; Technical Report "Adaptive stopping heuristic")
    same = bool(st.step[r] > 0 and np.all(st.argmax[r] == st.argmax_prev[r]))
    Hbar = float(np.sum(H) / C)
    if p.stop_rule == STOP_ENTROPY:
        # "DiffusionGemma-Lite DIFFUSION.html", section 4.4: stop once the mean
        # entropy has stayed below the threshold for stability_steps steps
        st.stable[r] = st.stable[r] + 1 if Hbar < p.conf_threshold else 0
    else:
        st.stable[r] = st.stable[r] + 1 if same else 0
    st.mean_entropy[r] = Hbar
    st.step[r] = st.step[r] + 1
    st.argmax_prev[r] = st.argmax[r]
    if p.stop_rule == STOP_ENTROPY:
        conv = st.stable[r] >= p.stable_k or st.step[r] >= p.step_cap
    else:
        conv = (st.stable[r] >= p.stable_k and Hbar < p.conf_threshold) or st.step[r] >= p.step_cap
    # Near-tie flag of the convergence decision (a reading of the near-tie
    # rule for the mean-entropy threshold): the mean entropy lies within 1e-4
    # of the threshold AND the threshold decides something.  Under the
    # entropy-only stop it decides the stable counter itself; under the
    # argmax-stable rule only a row whose argmax has been stable for stable_k
    # steps and that is below the step cap depends on it.
    near = (not math.isnan(Hbar)) and abs(Hbar - p.conf_threshold) < NEAR_TIE
    if p.stop_rule == STOP_ENTROPY:
        flags.converged[r] = near
    else:
        flags.converged[r] = near and st.stable[r] >= p.stable_k and st.step[r] < p.step_cap
    st.converged[r] = 1 if conv else 0
    st.sc_valid[r] = 0 if conv else 1
    st.phase[r] = PHASE_COMMIT if conv else PHASE_DENOISE
    st.num_sampled[r] = 0
    st.num_rejected[r] = C
    st.rng_step[r] = st.rng_step[r] + np.uint64(1)


def monotone_commit(st: State, r: int, H, R, flags: Flags):
    """The unchanged-or-stronger commit rule ("DiffusionGemma-Lite
    DIFFUSION.html", section 4.2): a position commits when its posterior mode
    equals the previous step's or its confidence (the largest probability,
    1/s with s = sum exp(y - max y)) did not fall; a newly committed position
    takes the step's draw, a position committed earlier keeps its token (never
    overwritten), and every other position is re-noised to a uniform token.
    Readings: on the first step of a block there is no previous mode (its
    comparison is false) and the previous confidence is +inf, so nothing
    commits; positions with an invalid distribution never commit and keep their
    previous confidence.  ``accept`` marks the newly committed positions.
    Called before argmax_prev is replaced by this step's argmax."""
    valid = ~np.isnan(H)
    conf = np.where(valid, 1.0 / np.where(valid, st.s[r], 1.0), np.nan)
    first = st.step[r] == 0
    unchanged = np.zeros_like(valid) if first else (st.argmax[r] == st.argmax_prev[r])
    prev = st.prev_conf[r].astype(np.float64)
    stronger = valid & (conf >= prev)
    commit = valid & (unchanged | stronger)
    was = st.committed[r] != 0
    new = commit & ~was
    st.canvas[r] = np.where(new, st.cand[r], np.where(was, st.canvas[r], R))
    st.committed[r] = (was | new).astype(np.uint8)
    st.prev_conf[r] = np.where(valid, conf, prev)
    st.accept[r] = new.astype(np.uint8)
    # the confidence comparison decides only where the mode changed
    flags.commit[r] = valid & ~unchanged & ~was & (np.abs(conf - prev) < NEAR_TIE)


def step(p: Params, st_in: State, logits, rows=None, mapper=map):
    """One sampler call over the whole batch: each row by its phase.

    ``logits`` is indexable as logits[r] -> [C, V] float64 (or convertible);
    rows other than DENOISE rows are not read.  ``rows`` optionally limits
    which DENOISE rows are evaluated (the others are left untouched, which is
    how large configurations are checked on a sample).  Returns the new
    state and the near-tie flags; ``st_in`` is not modified.
    """
    B, C = p.batch, p.canvas_len
    st = st_in.copy()
    _ensure_outputs(st, B, C)
    flags = Flags(cand=np.zeros((B, C), bool), accept=np.zeros(B, bool),
                  converged=np.zeros(B, bool), gaps=np.full((B, C), np.inf),
                  commit=np.zeros((B, C), bool))
    for r in range(B):
        ph = int(st.phase[r])
        if ph == PHASE_PREFILL:
            prefill_row(p, st, r)
        elif ph == PHASE_COMMIT:
            commit_row(p, st, r)
        elif ph == PHASE_DENOISE:
            if rows is not None and r not in rows:
                continue
            denoise_row(p, st, r, np.asarray(logits[r], dtype=np.float64), flags, mapper)
    return st, flags


def init_rows(p: Params, st_in: State, row_mask):
    """Stand-alone canvas initialisation of the masked rows (prefill form)."""
    st = st_in.copy()
    _ensure_outputs(st, p.batch, p.canvas_len)
    for r in range(p.batch):
        if row_mask[r]:
            prefill_row(p, st, r)
    return st


def commit_rows(p: Params, st_in: State, row_mask):
    """Stand-alone commit of the masked rows."""
    st = st_in.copy()
    _ensure_outputs(st, p.batch, p.canvas_len)
    for r in range(p.batch):
        if row_mask[r]:
            commit_row(p, st, r)
    return st


def anneal_temperature(step, temperature, t_max, t_min, n_steps, row_mask=None):
    """Linear temperature anneal over the denoising steps of a block.

    "DiffusionGemma Explained" (ML@Berkeley), section "Sampling", the
    ``denoise`` listing: the temperature starts at t_max and moves by
    (t_min - t_max) / max_denoising_steps after every step, so step k of the
    block divides the logits by t_max + k (t_min - t_max) / N.
    "DiffusionGemma-Lite DIFFUSION.html", section 4.2 item 4: tau(k) is
    annealed linearly from temp_start to temp_end across the schedule.

    Readings: k is the row's block-local step counter (0 at the first denoise
    step of a block), clamped to [0, N] so that steps past the schedule keep
    t_min; the value is the closed form in fp64, rounded once to fp32 (the
    listing's repeated addition differs only below fp32 resolution).  Rows
    with row_mask[r] == 0 keep their temperature.  Returns a new fp32 array.
    """
    out = np.asarray(temperature, dtype=np.float32).copy()
    t_max = float(np.float32(t_max))
    t_min = float(np.float32(t_min))
    for r in range(out.shape[0]):
        if row_mask is not None and not row_mask[r]:
            continue
        k = min(max(int(step[r]), 0), int(n_steps))
        out[r] = np.float32(t_max + k * (t_min - t_max) / n_steps)
    return out


def new_state(p: Params, phase, request_id, temperature, rng_step=None):
    B, C = p.batch, p.canvas_len
    st = State(
        phase=np.asarray(phase, dtype=np.uint8).copy(),
        request_id=np.asarray(request_id, dtype=np.uint64).copy(),
        temperature=np.asarray(temperature, dtype=np.float64).copy(),
        rng_step=(np.zeros(B, np.uint64) if rng_step is None
                  else np.asarray(rng_step, dtype=np.uint64).copy()),
        step=np.zeros(B, np.int32), stable=np.zeros(B, np.int32),
        canvas=np.zeros((B, C), np.int32), argmax_prev=np.zeros((B, C), np.int32))
    _ensure_outputs(st, B, C)
    return st
