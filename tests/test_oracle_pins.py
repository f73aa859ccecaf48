"""Pins of the fp64 oracle against what the pages and the mathematics fix:
published hash test vectors, closed forms, library routines, brute force and
statistical laws.  CPU only."""

import math
import os

import numpy as np
import pytest
from scipy import special, stats

from oracle import forward, rng, sampler, selfcond

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _keys(seed, r, k, i):
    return sampler.gumbel_keys(seed, r, k, i)


def _read_vectors(name):
    out = []
    with open(os.path.join(GOLDEN, "hash_vectors.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            fn, x, y = line.split()
            if fn == name:
                out.append((int(x, 16), int(y, 16)))
    return out


# ---------------------------------------------------------------- hashing

def test_splitmix64_published_outputs():
    vecs = _read_vectors("splitmix64")
    assert len(vecs) == 3
    for x, y in vecs:
        assert int(rng.mix64(np.uint64(x))) == y


def test_fmix32_published_outputs():
    vecs = _read_vectors("fmix32")
    assert len(vecs) == 3
    for x, y in vecs:
        assert int(rng.fmix32(np.uint32(x))) == y


def test_below_exact_against_bigint():
    g = np.random.default_rng(1)
    h = g.integers(0, 2 ** 32, 5000, dtype=np.uint64).astype(np.uint32)
    for n in (1, 2, 7, 8, 50257, 262144, 2 ** 31 + 11):
        got = rng.below(h, n)
        want = np.array([(int(x) * n) >> 32 for x in h])
        assert np.array_equal(got, want)
        assert got.min() >= 0 and got.max() < n


def test_uniform_open_interval_and_exp1_branches():
    h = np.array([0, 1, 2 ** 31 - 1, 2 ** 31, 2 ** 32 - 2, 2 ** 32 - 1], dtype=np.uint32)
    u = rng.uniform(h)
    assert np.all(u > 0) and np.all(u < 1)
    e = rng.exp1(h)
    # both branches agree with the exact -ln u computed from the rational u
    want = np.array([-math.log((int(x) + 0.5) / 2 ** 32) if x < 2 ** 31 else
                     -math.log1p(-((2 ** 32 - 1 - int(x)) + 0.5) / 2 ** 32) for x in h])
    assert np.allclose(e, want, rtol=1e-15, atol=0)
    # the largest draw gives the smallest Exp(1) value 2^-33 (to first order)
    assert abs(e[-1] - 2.0 ** -33) < 1e-20


# ------------------------------------------------------- forward process

@pytest.mark.parametrize("V", [8, 50257, 262144])
@pytest.mark.parametrize("kappa", [0.0, 0.25, 1.0])
def test_forward_row_is_a_distribution(V, kappa):
    row = forward.transition_row(3, kappa, V)
    assert abs(row.sum() - 1.0) < 1e-12
    assert abs(row[3] - (kappa + (1 - kappa) / V)) < 1e-15


# ------------------------------------------------------------- entropy

@pytest.mark.parametrize("V", [8, 1000, 50257])
def test_uniform_logits_entropy_is_lnV(V):
    ka, kb, kc = _keys(1, 0, 0, 0)
    res = sampler.vocab_pass(np.ones(V), 0.7, ka, kb, kc)
    assert abs(res.entropy - math.log(V)) < 1e-12
    assert res.argmax == 0  # lowest index on exact ties
    assert abs(res.s - V) < 1e-9


def test_one_hot_entropy_is_zero():
    ka, kb, kc = _keys(1, 0, 0, 0)
    z = np.full(64, -np.inf)
    z[17] = 3.0
    res = sampler.vocab_pass(z, 1.0, ka, kb, kc)
    assert res.valid and res.entropy == 0.0 and res.argmax == 17 and res.cand == 17
    z = np.zeros(64)
    z[5] = 1000.0
    res = sampler.vocab_pass(z, 1.0, ka, kb, kc)
    assert res.entropy < 1e-300 * 0 + 1e-12 and res.cand == 5


@pytest.mark.parametrize("delta,T", [(0.0, 1.0), (1.0, 1.0), (3.0, 0.5), (-2.0, 2.0)])
def test_binary_entropy_closed_form(delta, T):
    ka, kb, kc = _keys(2, 0, 0, 0)
    res = sampler.vocab_pass(np.array([0.0, delta]), T, ka, kb, kc)
    q = special.expit(delta / T)
    want = -(q * math.log(q) + (1 - q) * math.log(1 - q))
    assert abs(res.entropy - want) < 1e-12


def test_entropy_matches_library_and_the_streaming_identity():
    g = np.random.default_rng(3)
    for V in (2, 9, 1000, 4097):
        z = g.normal(0, 2, V)
        z[g.integers(V)] += 9.0
        T = float(g.uniform(0.5, 1.5))
        res = sampler.vocab_pass(z, T, *_keys(3, V, 0, 0))
        p = special.softmax(z / T)
        assert abs(res.entropy - stats.entropy(p)) < 1e-12
        # H = ln s - t/s with s = sum e^{y-m}, t = sum (y-m) e^{y-m}
        y = z / T
        m = y.max()
        e = np.exp(y - m)
        assert abs(res.entropy - (math.log(e.sum()) - np.sum((y - m) * e) / e.sum())) < 1e-11
        # (m, s) reproduce the log-partition function
        assert abs(res.m + math.log(res.s) - special.logsumexp(y)) < 1e-12


def test_entropy_shift_invariance():
    g = np.random.default_rng(4)
    z = g.normal(0, 2, 777)
    a = sampler.vocab_pass(z, 0.9, *_keys(4, 0, 0, 0))
    b = sampler.vocab_pass(z + 123.25, 0.9, *_keys(4, 0, 0, 0))
    assert abs(a.entropy - b.entropy) < 1e-11
    assert a.argmax == b.argmax


def test_neg_inf_tokens_have_zero_mass_and_invalid_rows():
    g = np.random.default_rng(5)
    z = g.normal(0, 1, 100)
    z[::3] = -np.inf
    res = sampler.vocab_pass(z, 1.0, *_keys(5, 0, 0, 0))
    finite = z[np.isfinite(z)]
    assert abs(res.entropy - stats.entropy(special.softmax(finite))) < 1e-12
    assert np.isfinite(z[res.cand]) and np.isfinite(z[res.argmax])
    for bad in (np.array([0.0, np.nan, 1.0]), np.array([0.0, np.inf]), np.full(4, -np.inf)):
        r = sampler.vocab_pass(bad, 1.0, *_keys(5, 0, 0, 0))
        assert not r.valid and math.isnan(r.entropy) and r.cand == 0 and r.argmax == 0
    r = sampler.vocab_pass(np.zeros(4), 0.0, *_keys(5, 0, 0, 0))
    assert not r.valid


# ------------------------------------------------------------- Gumbel

def test_group_exponentials_are_iid_exp1():
    """Marginal law Exp(1) (KS), zero correlation inside groups, minimum of a
    full group ~ Exp(rate 8), argmin uniform over the 8 slots."""
    V = 400_003  # ragged last group
    ka, kb, kc = _keys(6, 1, 2, 3)
    E = rng.gumbel_exponentials(V, ka, kb, kc)
    assert np.all(E > 0)
    assert stats.kstest(E, "expon").pvalue > 1e-3
    full = E[: (V // 8) * 8].reshape(-1, 8)
    assert stats.kstest(full.min(axis=1) * 8.0, "expon").pvalue > 1e-3
    counts = np.bincount(full.argmin(axis=1), minlength=8)
    assert stats.chisquare(counts).pvalue > 1e-3
    for a, b in ((0, 1), (3, 7), (2, 5)):
        r = np.corrcoef(full[:, a], full[:, b])[0, 1]
        assert abs(r) < 4.0 / math.sqrt(full.shape[0])
    G = rng.gumbel_noise(V, ka, kb, kc)
    assert stats.kstest(G, "gumbel_r").pvalue > 1e-3


def test_planted_group_mistake_is_caught():
    """A plausible slip (forgetting to divide the group minimum by the group
    size) must fail the marginal-law pin above."""
    V = 200_000
    ka, kb, kc = _keys(6, 1, 2, 3)
    v = np.arange(V)
    g = v // 8
    x = rng.exp1(rng.draw32(ka, np.arange(V // 8, dtype=np.uint32)))
    j = rng.below(rng.draw32(kb, np.arange(V // 8, dtype=np.uint32)), 8)
    rest = rng.exp1(rng.draw32(kc, v.astype(np.uint32)))
    wrong = x[g] + np.where(v - 8 * g == j[g], 0.0, rest)  # no division by n_g
    assert stats.kstest(wrong, "expon").pvalue < 1e-6


def _cand_frequencies(z, T, n, seed):
    counts = np.zeros(z.size, dtype=np.int64)
    for r in range(n):
        res = sampler.vocab_pass(z, T, *_keys(seed, r, 0, 0))
        counts[res.cand] += 1
    return counts


@pytest.mark.parametrize("V,T", [(8, 0.5), (8, 1.0), (8, 2.0), (13, 1.0)])
def test_gumbel_max_frequencies_follow_softmax(V, T):
    z = np.random.default_rng(7 + V).normal(0, 1, V)
    n = 20000
    counts = _cand_frequencies(z, T, n, seed=11)
    p = special.softmax(z / T)
    assert stats.chisquare(counts, n * p).pvalue > 1e-3


def test_gumbel_max_tail_on_larger_vocab():
    V, n = 1000, 4000
    z = np.random.default_rng(8).normal(0, 1, V)
    z[:4] += np.array([6.0, 5.0, 4.5, 4.0])
    counts = _cand_frequencies(z, 1.0, n, seed=12)
    p = special.softmax(z)
    head = np.concatenate([counts[:4], [counts[4:].sum()]])
    ph = np.concatenate([p[:4], [p[4:].sum()]])
    assert stats.chisquare(head, n * ph).pvalue > 1e-3


def test_low_temperature_candidate_is_the_argmax():
    g = np.random.default_rng(9)
    for r in range(50):
        z = np.round(g.normal(0, 2, 300), 1)
        z[g.integers(300)] += 0.5
        res = sampler.vocab_pass(z, 1e-3, *_keys(13, r, 0, 0))
        srt = np.sort(z)
        if srt[-1] - srt[-2] > 0.05:
            assert res.cand == res.argmax


# --------------------------------------------------- uniform tokens

@pytest.mark.parametrize("V", [8, 50257])
def test_init_and_renoise_tokens_are_uniform(V):
    toks = np.concatenate([sampler.init_tokens(21, r, 0, 256, V) for r in range(400)])
    ren = np.concatenate([sampler.renoise_tokens(21, r, 0, 256, V) for r in range(400)])
    for t in (toks, ren):
        assert t.min() >= 0 and t.max() < V
        bins = 8 if V == 8 else 64
        counts = np.bincount((t.astype(np.int64) * bins) // V, minlength=bins)
        assert stats.chisquare(counts).pvalue > 1e-3
    # different tags are different streams
    assert abs(np.corrcoef(toks, ren)[0, 1]) < 4.0 / math.sqrt(toks.size)


# ------------------------------------------------------- acceptance

def _brute_force_accept(H, b):
    """Over all 2^C subsets: the largest set that is down-closed in (H, i)
    order and whose members other than its last (in that order) sum <= b."""
    C = len(H)
    order = sorted(range(C), key=lambda i: (H[i], i))
    rank = {i: k for k, i in enumerate(order)}
    best = None
    for mask in range(1, 1 << C):
        members = [i for i in range(C) if mask >> i & 1]
        ranks = sorted(rank[i] for i in members)
        if ranks != list(range(len(ranks))):
            continue
        body = sum(H[order[k]] for k in range(len(ranks) - 1))
        if body <= b and (best is None or len(members) > len(best)):
            best = members
    out = np.zeros(C, bool)
    out[best] = True
    return out


@pytest.mark.parametrize("b", [0.0, 0.1, 1.0, 10.0, 1e9])
def test_accept_matches_brute_force(b):
    g = np.random.default_rng(int(b * 10) + 1)
    for _ in range(60):
        H = g.exponential(0.8, 8)
        if g.random() < 0.5:  # inject exact ties
            H[g.integers(8)] = H[g.integers(8)]
        acc, _ = sampler.accept_mask(H, b)
        assert np.array_equal(acc, _brute_force_accept(list(H), b))


def test_accept_zero_budget_and_monotone():
    g = np.random.default_rng(10)
    for _ in range(50):
        H = g.exponential(1.0, 16) + 1e-3
        acc0, _ = sampler.accept_mask(H, 0.0)
        assert acc0.sum() == 1 and acc0[np.argmin(H)]
        prev = 0
        for b in np.linspace(0, H.sum(), 25):
            n = sampler.accept_mask(H, b)[0].sum()
            assert n >= prev
            prev = n
        assert sampler.accept_mask(H, H.sum() - H.max() + 1e-9)[0].all()


def test_accept_invalid_positions_sort_last():
    H = np.array([0.5, np.nan, 0.1, 0.2])
    acc, _ = sampler.accept_mask(H, 100.0)
    assert list(acc) == [True, False, True, True]


# --------------------------------------------- convergence / phases

def _one_hot_logits(tokens, V, level=1000.0):
    z = np.zeros((len(tokens), V))
    z[np.arange(len(tokens)), tokens] = level
    return z


def test_phase_cycle_and_counters():
    C, V = 8, 16
    p = sampler.Params(batch=1, canvas_len=C, vocab=V, seed=5, entropy_budget=1.0,
                       conf_threshold=0.3, stable_k=2, step_cap=10)
    st = sampler.new_state(p, [sampler.PHASE_PREFILL], [42], [1.0])
    st, _ = sampler.step(p, st, None)
    assert st.phase[0] == sampler.PHASE_DENOISE and st.num_sampled[0] == 0
    assert np.array_equal(st.canvas[0], sampler.init_tokens(5, 42, 0, C, V))
    toks = np.arange(C) % V
    seq = [toks, toks, toks, toks]
    want_stable = [0, 1, 2]
    for k in range(3):
        st, _ = sampler.step(p, st, _one_hot_logits(seq[k], V)[None])
        assert st.stable[0] == want_stable[k] and st.step[0] == k + 1
        assert st.num_sampled[0] == 0 and st.num_rejected[0] == C
        # one-hot rows: H = 0, every position accepted, canvas = argmax
        assert st.accept[0].all() and np.array_equal(st.canvas[0], toks)
    assert st.converged[0] == 1 and st.phase[0] == sampler.PHASE_COMMIT and st.sc_valid[0] == 0
    st, _ = sampler.step(p, st, None)
    assert np.array_equal(st.emitted[0], toks) and st.num_sampled[0] == C
    assert st.phase[0] == sampler.PHASE_DENOISE and st.step[0] == 0 and st.stable[0] == 0
    assert st.rng_step[0] == 5


def test_unstable_argmax_resets_and_cap_is_exact():
    C, V = 8, 16
    for cap in (1, 3, 6):
        p = sampler.Params(1, C, V, 9, 1.0, 0.3, 1, cap)
        st = sampler.new_state(p, [sampler.PHASE_DENOISE], [1], [1.0])
        steps = 0
        while st.phase[0] == sampler.PHASE_DENOISE:
            toks = (np.arange(C) + steps) % V  # argmax changes every step
            st, _ = sampler.step(p, st, _one_hot_logits(toks, V)[None])
            steps += 1
            assert st.stable[0] == 0
        assert steps == cap


def test_threshold_below_zero_runs_to_cap():
    """'adaptive off' is the fixed schedule: thr < 0 never converges early."""
    C, V = 8, 16
    p = sampler.Params(1, C, V, 9, 1.0, -1.0, 1, 5)
    st = sampler.new_state(p, [sampler.PHASE_DENOISE], [1], [1.0])
    n = 0
    while st.phase[0] == sampler.PHASE_DENOISE:
        st, _ = sampler.step(p, st, _one_hot_logits(np.arange(C), V)[None])
        n += 1
    assert n == 5


def test_mean_entropy_threshold_gates_convergence():
    C, V = 8, 16
    p = sampler.Params(1, C, V, 9, 100.0, 0.3, 1, 50)
    st = sampler.new_state(p, [sampler.PHASE_DENOISE], [1], [1.0])
    flat = np.zeros((C, V))
    flat[np.arange(C), np.arange(C)] = 1.0  # stable argmax, high entropy
    for _ in range(5):
        st, _ = sampler.step(p, st, flat[None])
        assert st.phase[0] == sampler.PHASE_DENOISE and st.mean_entropy[0] > 2.0
    st, _ = sampler.step(p, st, _one_hot_logits(np.arange(C), V)[None])
    assert st.phase[0] == sampler.PHASE_COMMIT


def test_idle_rows_untouched_and_mixed_batch():
    C, V = 8, 32
    p = sampler.Params(4, C, V, 3, 2.0, 0.3, 1, 4)
    st = sampler.new_state(p, [0, 1, 2, 3], [10, 11, 12, 13], [1.0, 0.8, 1.0, 1.0])
    st.argmax_prev[2] = np.arange(C)
    g = np.random.default_rng(0)
    logits = g.normal(0, 2, (4, C, V))
    st2, _ = sampler.step(p, st, logits)
    assert st2.phase.tolist() == [1, 1, 1, 3]
    assert np.array_equal(st2.emitted[2], np.arange(C))
    assert np.array_equal(st2.canvas[3], st.canvas[3]) and st2.rng_step[3] == 0
    assert st2.rng_step[:3].tolist() == [1, 1, 1]


# --------------------------------------------------------- self-cond

def test_selfcond_one_hot_returns_embedding_row():
    g = np.random.default_rng(11)
    V, d = 50, 12
    E = g.normal(0, 0.02, (V, d))
    z = np.full((3, V), -np.inf)
    z[0, 7] = 0.0
    z[1, 0] = 5.0
    z[2, 49] = -3.0
    out = selfcond.selfcond_rows(z, 1.0, E)
    assert np.array_equal(out, E[[7, 0, 49]])


def test_selfcond_uniform_gives_column_means_and_linearity():
    g = np.random.default_rng(12)
    V, d = 64, 9
    E = g.normal(0, 0.02, (V, d))
    out = selfcond.selfcond_rows(np.zeros((1, V)), 0.7, E)
    assert np.allclose(out[0], E.mean(axis=0), atol=1e-15)
    a = 0.3
    z = np.full((1, V), -np.inf)
    z[0, 3] = math.log(a)
    z[0, 40] = math.log(1 - a)
    out = selfcond.selfcond_rows(z, 1.0, E)
    assert np.allclose(out[0], a * E[3] + (1 - a) * E[40], atol=1e-15)


def test_selfcond_non_feeding_rows_are_zero():
    g = np.random.default_rng(13)
    B, C, V, d = 3, 4, 20, 5
    E = g.normal(0, 0.02, (V, d))
    logits = g.normal(0, 2, (B, C, V))
    out = selfcond.selfcond(logits, np.ones(B), E, np.array([True, False, True]))
    assert np.all(out[C:2 * C] == 0) and np.any(out[:C] != 0)


# ---- temperature anneal ("DiffusionGemma Explained", "Sampling", the denoise
# listing; "DiffusionGemma-Lite DIFFUSION.html", section 4.2 item 4)

def test_anneal_endpoints_and_clamping():
    from oracle import sampler as osam
    steps = np.array([0, 24, 40, -3], dtype=np.int32)
    T = osam.anneal_temperature(steps, np.zeros(4, np.float32), 0.8, 0.4, 24)
    assert T[0] == np.float32(0.8) and T[3] == np.float32(0.8)
    assert T[1] == np.float32(0.4) and T[2] == np.float32(0.4)


def test_anneal_matches_the_listing_by_repeated_addition():
    # the listing's loop: t = t_max, then t += (t_min - t_max) / N after each step
    from oracle import sampler as osam
    for t_max, t_min, N in [(0.8, 0.4, 24), (1.2, 0.6, 32), (0.5, 1.5, 7)]:
        t = float(np.float32(t_max))
        dt = (float(np.float32(t_min)) - t) / N
        steps = np.arange(N + 1, dtype=np.int32)
        T = osam.anneal_temperature(steps, np.zeros(N + 1, np.float32), t_max, t_min, N)
        for k in range(N + 1):
            assert abs(float(T[k]) - t) <= float(np.spacing(np.float32(t))), (t_max, t_min, N, k)
            t += dt
        d = np.diff(T.astype(np.float64))
        assert np.all(d <= 0) if t_max > t_min else np.all(d >= 0)


def test_anneal_leaves_masked_rows():
    from oracle import sampler as osam
    T0 = np.array([0.7, 0.9, 1.1], np.float32)
    T = osam.anneal_temperature(np.array([5, 5, 5]), T0, 1.0, 0.5, 10, row_mask=[1, 0, 1])
    assert T[1] == T0[1] and T[0] == np.float32(0.75) and T[2] == np.float32(0.75)


# ---- rule variants ("DiffusionGemma-Lite DIFFUSION.html": section 4.2, the
# unchanged-or-stronger commit rule; section 4.4, entropy-only adaptive stop)

def _peaked(C, V, hot, height):
    """[C, V] logits: zeros except `height` at token hot[i] of position i."""
    z = np.zeros((C, V))
    z[np.arange(C), hot] = height
    return z


def test_entropy_stop_converges_on_entropy_alone():
    # the argmax moves every step, so the argmax-stable rule never converges
    # before the cap, while the entropy rule stops after stable_k low-entropy
    # steps: steps 0, 1 are flat (mean H = ln V > thr), 2, 3, 4 are sharp
    from oracle import sampler as osam
    C, V, k = 4, 16, 3
    for rule, expect in [(osam.STOP_ENTROPY, 5), (osam.STOP_ARGMAX_STABLE, 8)]:
        p = osam.Params(batch=1, canvas_len=C, vocab=V, seed=3, entropy_budget=100.0,
                        conf_threshold=0.3, stable_k=k, step_cap=8, stop_rule=rule)
        st = osam.new_state(p, [osam.PHASE_DENOISE], [1], [1.0])
        for t in range(8):
            z = np.zeros((C, V)) if t < 2 else _peaked(C, V, (np.arange(C) + t) % V, 40.0)
            st, _ = osam.step(p, st, [z])
            if st.converged[0]:
                break
        assert t + 1 == expect, (rule, t + 1)
        if rule == osam.STOP_ENTROPY:
            assert st.stable[0] == k


def test_monotone_first_step_commits_nothing():
    from oracle import sampler as osam
    C, V = 6, 32
    p = osam.Params(batch=1, canvas_len=C, vocab=V, seed=5, entropy_budget=0.0,
                    conf_threshold=0.0, stable_k=3, step_cap=10, accept_rule=osam.ACCEPT_MONOTONE)
    st = osam.new_state(p, [osam.PHASE_PREFILL], [2], [1.0])
    st, _ = osam.step(p, st, [None])
    assert np.all(st.committed[0] == 0) and np.all(np.isinf(st.prev_conf[0]))
    st1, _ = osam.step(p, st, [_peaked(C, V, np.arange(C), 30.0)])
    assert np.all(st1.committed[0] == 0) and np.all(st1.accept[0] == 0)
    R = osam.renoise_tokens(p.seed, st.request_id[0], st.rng_step[0], C, V)
    assert np.array_equal(st1.canvas[0], R)


def test_monotone_unchanged_or_stronger_by_hand():
    # position 0: same mode, confidence falls -> commits (unchanged)
    # position 1: new mode, confidence rises  -> commits (stronger)
    # position 2: new mode, confidence falls  -> stays open, re-noised
    from oracle import sampler as osam
    C, V = 3, 8
    p = osam.Params(batch=1, canvas_len=C, vocab=V, seed=9, entropy_budget=0.0,
                    conf_threshold=-1.0, stable_k=3, step_cap=10, accept_rule=osam.ACCEPT_MONOTONE)
    st = osam.new_state(p, [osam.PHASE_DENOISE], [4], [1.0])
    z0 = np.zeros((C, V)); z0[0, 1] = 5.0; z0[1, 2] = 1.0; z0[2, 3] = 5.0
    st, _ = osam.step(p, st, [z0])              # first step: nothing commits
    z1 = np.zeros((C, V)); z1[0, 1] = 2.0; z1[1, 5] = 6.0; z1[2, 6] = 1.0
    st2, _ = osam.step(p, st, [z1])
    # confidences by hand: max p = e^a / (e^a + V - 1)
    conf = lambda a: math.exp(a) / (math.exp(a) + V - 1)
    assert abs(st2.prev_conf[0, 1] - conf(6.0)) < 1e-12
    assert st.prev_conf[0, 1] == conf(1.0) or abs(st.prev_conf[0, 1] - conf(1.0)) < 1e-12
    assert list(st2.committed[0]) == [1, 1, 0]
    assert list(st2.accept[0]) == [1, 1, 0]
    assert st2.canvas[0, 0] == st2.cand[0, 0] and st2.canvas[0, 1] == st2.cand[0, 1]
    R = osam.renoise_tokens(p.seed, st.request_id[0], st.rng_step[0], C, V)
    assert st2.canvas[0, 2] == R[2]


def test_monotone_frozen_tokens_never_change_and_emission():
    from oracle import sampler as osam
    rs = np.random.default_rng(1)
    C, V = 16, 24
    p = osam.Params(batch=1, canvas_len=C, vocab=V, seed=11, entropy_budget=0.0,
                    conf_threshold=-1.0, stable_k=99, step_cap=6, accept_rule=osam.ACCEPT_MONOTONE)
    st = osam.new_state(p, [osam.PHASE_DENOISE], [7], [0.9])
    frozen = {}
    for t in range(6):
        z = rs.normal(0, 1.5, (C, V)); z[:, 3] += 0.3 * t   # confidence tends to rise
        prev = st
        st, _ = osam.step(p, st, [z])
        assert np.all(st.committed[0] >= prev.committed[0])
        for i, tok in frozen.items():
            assert st.canvas[0, i] == tok
        for i in np.flatnonzero((st.committed[0] == 1) & (prev.committed[0] == 0)):
            assert st.canvas[0, i] == st.cand[0, i]
            frozen[i] = st.canvas[0, i]
    assert st.phase[0] == osam.PHASE_COMMIT and frozen
    out, _ = osam.step(p, st, [None])
    want = np.where(st.committed[0] == 1, st.canvas[0], st.cand[0])
    assert np.array_equal(out.emitted[0], want)
    assert np.all(out.committed[0] == 0) and np.all(np.isinf(out.prev_conf[0]))


# ---- logit softcap and embedding scale ("The Annotated DiffusionGemma",
# "Logit Softcapping" and the model's forward)

def _tanh_by_exp(x):
    """tanh from its exponential definition, (e^2x - 1) / (e^2x + 1)."""
    e = math.exp(2.0 * x)
    return (e - 1.0) / (e + 1.0)


@pytest.mark.parametrize("c", [30.0, 5.0, 0.75])
def test_softcap_closed_forms(c):
    # at z = +-c the cap is +-c tanh(1); at z = c/2 it is c tanh(1/2)
    z = np.array([c, -c, 0.5 * c, 0.0])
    got = sampler.softcap(z, c)
    want = [c * _tanh_by_exp(1.0), -c * _tanh_by_exp(1.0), c * _tanh_by_exp(0.5), 0.0]
    assert np.allclose(got, want, rtol=1e-14, atol=0)
    # small logits are essentially unchanged: z - z^3 / (3 c^2) to third order
    small = np.array([1e-3, -2e-3, 5e-4]) * c
    assert np.allclose(sampler.softcap(small, c), small - small ** 3 / (3 * c * c), rtol=1e-11)
    # large logits approach +-c, infinite ones reach it; NaN stays NaN
    big = sampler.softcap(np.array([1e6 * c, -1e6 * c, np.inf, -np.inf, np.nan]), c)
    assert big[0] == c and big[1] == -c and big[2] == c and big[3] == -c and np.isnan(big[4])


def test_softcap_is_odd_monotone_and_bounded():
    g = np.random.default_rng(21)
    c = 30.0
    z = np.sort(g.normal(0, 40, 4001))
    y = sampler.softcap(z, c)
    assert np.all(np.diff(y) >= 0)
    assert np.array_equal(sampler.softcap(-z, c), -y)
    assert np.all(np.abs(y) <= np.minimum(np.abs(z), c))
    assert np.array_equal(sampler.softcap(z, 0.0), z)  # c = 0: no cap


def test_step_with_softcap_equals_step_on_capped_logits():
    """The sampler reads the capped logits and nothing else: a capped step is
    an uncapped step on c tanh(z / c) (built here from the exponential form)."""
    g = np.random.default_rng(22)
    C, V, c = 8, 40, 3.0
    z = g.normal(0, 4, (2, C, V))
    zc = np.vectorize(lambda x: c * _tanh_by_exp(x / c))(z)
    base = dict(batch=2, canvas_len=C, vocab=V, seed=77, entropy_budget=12.0,
                conf_threshold=0.3, stable_k=2, step_cap=8)
    pc = sampler.Params(**base, softcap=c)
    p0 = sampler.Params(**base)
    st = sampler.new_state(pc, [sampler.PHASE_DENOISE] * 2, [4, 5], [0.9, 1.3])
    a, _ = sampler.step(pc, st, z)
    b, _ = sampler.step(p0, st, zc)
    for k in ("canvas", "cand", "argmax", "accept", "stable", "phase"):
        assert np.array_equal(getattr(a, k), getattr(b, k)), k
    for k in ("m", "s", "entropy", "mean_entropy"):
        assert np.allclose(getattr(a, k), getattr(b, k), rtol=1e-13, atol=1e-13), k
    # the cap changes the result: c = 3 squeezes these logits hard
    u, _ = sampler.step(p0, st, z)
    assert not np.allclose(u.entropy, a.entropy)


def test_selfcond_softcap_and_scale_by_hand():
    # V = 3, one row: p = exp(cap(z)) / sum, done term by term
    c, T, scale = 2.0, 0.5, math.sqrt(7.0)
    z = np.array([[1.0, -3.0, 0.25]])
    E = np.array([[1.0, 0.0], [0.0, 2.0], [-1.0, 1.0]])
    w = [math.exp(c * _tanh_by_exp(x / c) / T) for x in z[0]]
    s = sum(w)
    want = [scale * (w[0] * 1.0 + w[2] * -1.0) / s, scale * (w[1] * 2.0 + w[2] * 1.0) / s]
    got = selfcond.selfcond_rows(z, T, E, cap=c, scale=scale)
    assert np.allclose(got[0], want, rtol=1e-14)
    # scale 0 means 1; the scale is linear
    g = np.random.default_rng(23)
    L, E2 = g.normal(0, 3, (2, 4, 30)), g.normal(0, 0.02, (30, 6))
    one = selfcond.selfcond(L, np.ones(2), E2, np.array([True, True]), cap=5.0)
    assert np.array_equal(one, selfcond.selfcond(L, np.ones(2), E2, np.array([True, True]),
                                                 cap=5.0, scale=1.0))
    assert np.allclose(selfcond.selfcond(L, np.ones(2), E2, np.array([True, True]), cap=5.0,
                                         scale=3.5), 3.5 * one, rtol=1e-15, atol=0)


def test_softcap_large_c_reduces_to_the_uncapped_step():
    # c tanh(z / c) -> z as c grows: with |z| <= ~20 and c = 1e6 the cap moves
    # each logit by < z^3 / (3 c^2) ~ 3e-9, so the step is unchanged
    g = np.random.default_rng(24)
    C, V = 8, 50
    z = g.normal(0, 4, (1, C, V))
    base = dict(batch=1, canvas_len=C, vocab=V, seed=91, entropy_budget=6.0,
                conf_threshold=0.3, stable_k=2, step_cap=8)
    st = sampler.new_state(sampler.Params(**base), [sampler.PHASE_DENOISE], [7], [0.8])
    a, _ = sampler.step(sampler.Params(**base, softcap=1e6), st, z)
    b, _ = sampler.step(sampler.Params(**base), st, z)
    for k in ("canvas", "cand", "argmax", "accept"):
        assert np.array_equal(getattr(a, k), getattr(b, k)), k
    assert np.allclose(a.entropy, b.entropy, rtol=0, atol=1e-7)
