"""Pins of the oracle's near-tie flags: the decisions it marks as "not compared
exactly" because a result 1e-4 away would decide them the other way.

The rule (the near-tie definition of the method's parity contract): a
Gumbel-max candidate whose top-2 perturbed scores differ by less than 1e-4,
an acceptance cut where some exclusive prefix of the sorted entropies lies
within 1e-4 of the budget ("DiffusionGemma Explained", "Sampling", step 3),
or where the two entropies either side of the cut lie within 1e-4, a mean
entropy within 1e-4 of the convergence threshold where that threshold decides
the outcome (vLLM blog, "Entropy-bounded denoising"), and, under the
unchanged-or-stronger rule ("DiffusionGemma-Lite DIFFUSION.html", section
4.2), a confidence within 1e-4 of the previous one where the mode changed.

Every case below is built by hand so that its answer is known from the
construction: distances of 5e-5 must flag, 2e-4 must not, exact ties must,
and a distance of exactly 1e-4 must not (the rule is strict).  The last
tests plant plausible slips in copies of the oracle's functions and check
that these pins catch each one.  CPU only."""

import inspect
import math
import textwrap

import numpy as np
import pytest

from oracle import rng, sampler


# ------------------------------------------------------------ candidate gap

def _vocab_pass_with_noise(monkeypatch, z, T, G, fn=None):
    """The oracle's vocabulary pass with the Gumbel noise replaced by ``G``
    (dyadic values, so every perturbed score below is exact)."""
    monkeypatch.setattr(rng, "gumbel_noise", lambda V, ka, kb, kc: np.asarray(G, np.float64))
    return (fn or sampler.vocab_pass)(np.asarray(z, np.float64), T, 1, 2, 3)


def _gap_pins(monkeypatch, fn=None):
    """Failures of the candidate-gap pins for vocabulary-pass function ``fn``."""
    bad = []
    flag = lambda res: res.gap < sampler.NEAR_TIE

    # perturbed scores 0, 1, 1 - 5e-5, -1 (T = 1, no noise): flagged, cand 1
    r = _vocab_pass_with_noise(monkeypatch, [0.0, 1.0, 1.0 - 5e-5, -1.0], 1.0, [0] * 4, fn)
    if not (r.cand == 1 and flag(r) and abs(r.gap - 5e-5) < 1e-12):
        bad.append("gap 5e-5")
    # 2e-4 apart: not flagged
    r = _vocab_pass_with_noise(monkeypatch, [0.0, 1.0, 1.0 - 2e-4, -1.0], 1.0, [0] * 4, fn)
    if not (r.cand == 1 and not flag(r)):
        bad.append("gap 2e-4")
    # an exact tie of the best score: lowest index, gap exactly 0, flagged
    r = _vocab_pass_with_noise(monkeypatch, [0.5, 1.0, 1.0, -1.0], 1.0, [0] * 4, fn)
    if not (r.cand == 1 and r.gap == 0.0 and flag(r)):
        bad.append("exact tie")
    # a tie below the best is no near-tie
    r = _vocab_pass_with_noise(monkeypatch, [1.0, 0.5, 0.5, -1.0], 1.0, [0] * 4, fn)
    if not (r.cand == 0 and r.gap == 0.5 and not flag(r)):
        bad.append("tie below the best")
    # the gap is taken on y + G with y = z / T: T = 1/2 doubles z, and the
    # noise [1/4, -1/2, 0, 1/8] brings the scores to 0, 1, 1 - 5e-5, -1
    G = [0.25, -0.5, 0.0, 0.125]
    z = [(0.0 - 0.25) / 2, (1.0 + 0.5) / 2, (1.0 - 5e-5) / 2, (-1.0 - 0.125) / 2]
    r = _vocab_pass_with_noise(monkeypatch, z, 0.5, G, fn)
    if not (r.cand == 1 and flag(r) and abs(r.gap - 5e-5) < 1e-12):
        bad.append("perturbed, tempered scores")
    # close clean logits, far perturbed scores: not flagged
    r = _vocab_pass_with_noise(monkeypatch, [1.0, 1.0 + 5e-5, -3.0, -3.0], 1.0,
                               [0.0, 0.5, 0.0, 0.0], fn)
    if not (r.cand == 1 and abs(r.gap - (0.5 + 5e-5)) < 1e-12 and not flag(r)):
        bad.append("clean logits close")
    # a -inf token never takes part: V = 2 with one finite logit has no rival
    r = _vocab_pass_with_noise(monkeypatch, [-math.inf, 0.3], 1.0, [0.0, 0.0], fn)
    if not (r.cand == 1 and not flag(r)):
        bad.append("-inf rival")
    return bad


def test_candidate_gap_flag(monkeypatch):
    assert _gap_pins(monkeypatch) == []


# ---------------------------------------------------------- acceptance cut

# entropies in a scrambled position order; sorted: .1 .2 .3 .4 1 2 3 4,
# exclusive prefixes 0 .1 .3 .6 1 2 4 7, total 11
_H8 = np.array([2.0, 0.3, 4.0, 0.1, 1.0, 0.4, 3.0, 0.2])


def _accept_pins(fn=None):
    """Failures of the acceptance-flag pins for accept-mask function ``fn``."""
    fn = fn or sampler.accept_mask
    bad = []

    def check(name, H, b, n_acc, flagged):
        acc, fl = fn(np.asarray(H, np.float64), b)
        if int(acc.sum()) != n_acc or bool(fl) != flagged:
            bad.append(f"{name}: accepted {int(acc.sum())} flagged {bool(fl)}")

    # an exclusive prefix (1.0, before the 5th position) at the budget +- 5e-5
    check("prefix +5e-5", _H8, 1.0 + 5e-5, 5, True)
    check("prefix -5e-5", _H8, 1.0 - 5e-5, 4, True)
    # ... and +- 2e-4 away
    check("prefix +2e-4", _H8, 1.0 + 2e-4, 5, False)
    check("prefix -2e-4", _H8, 1.0 - 2e-4, 4, False)
    # the first position is always accepted, whatever the budget: its (empty)
    # prefix 0 is no decision, so a budget of 5e-5 is not near a tie
    check("first position", _H8, 5e-5, 1, False)
    # an inclusive sum of all 8 (11.0) is no exclusive prefix
    check("total +5e-5", _H8, 11.0 + 5e-5, 8, False)
    check("total -5e-5", _H8, 11.0 - 5e-5, 8, False)
    # neighbours across the cut within 5e-5: 1.0 accepted, 1.00005 rejected
    H = np.array([0.1, 0.2, 0.3, 0.4, 1.0, 1.0 + 5e-5, 3.0, 4.0])[[5, 0, 7, 2, 4, 1, 6, 3]]
    check("neighbours 5e-5", H, 1.5, 5, True)
    H = np.array([0.1, 0.2, 0.3, 0.4, 1.0, 1.0 + 2e-4, 3.0, 4.0])
    check("neighbours 2e-4", H, 1.5, 5, False)
    # close neighbours both accepted (no cut between them): no flag
    H = np.array([0.1, 0.1 + 3e-5, 0.3, 0.4, 1.0, 2.0, 3.0, 4.0])
    check("close pair inside", H, 1.5, 5, False)
    # close neighbours both rejected: no flag
    H = np.array([0.1, 0.2, 0.3, 0.4, 1.0, 2.0, 3.0, 3.0 + 3e-5])
    check("close pair outside", H, 1.5, 5, False)
    # exact ties across the cut (equal entropies): flagged
    H = np.array([0.1, 0.2, 0.3, 0.4, 1.0, 1.0, 3.0, 4.0])
    check("tie across cut", H, 1.5, 5, True)
    # distance exactly 1e-4 (2e-4 - 1e-4 is exact in binary64): the rule is
    # strict, so neither the neighbours nor the prefix 1e-4 vs budget 0 flag
    H = np.array([1e-4, 2e-4, 5.0, 5.0, 5.0, 5.0, 5.0, 5.0])
    check("exactly 1e-4", H, 0.0, 1, False)
    # every position accepted: no cut, no flag
    check("all accepted", _H8, 100.0, 8, False)
    # invalid positions (NaN) sort last and are never accepted; no flag from
    # the infinite key
    H = np.array([0.1, np.nan, 0.2, np.nan])
    check("invalid tail", H, 100.0, 2, False)
    return bad


def test_acceptance_flag():
    assert _accept_pins() == []


# ------------------------------------------------------- convergence flag

def _conv_case(stop_rule, thr_offset, stable_before, step_before, cap, k=2, fn_step=None):
    """One denoise step of one C = 4 canvas whose argmax equals argmax_prev;
    the threshold is the step's mean entropy + thr_offset.  Returns the
    convergence flag."""
    C, V = 4, 16
    z = np.zeros((C, V))
    z[np.arange(C), [3, 5, 7, 9]] = [2.0, 2.5, 3.0, 3.5]
    p = sampler.Params(batch=1, canvas_len=C, vocab=V, seed=3, entropy_budget=10.0,
                       conf_threshold=0.0, stable_k=k, step_cap=cap, stop_rule=stop_rule)
    st = sampler.new_state(p, [sampler.PHASE_DENOISE], [1], [1.0])
    st.argmax_prev[0] = [3, 5, 7, 9]
    st.stable[0] = stable_before
    st.step[0] = step_before
    probe, _ = sampler.step(p, st, [z])
    p.conf_threshold = float(probe.mean_entropy[0]) + thr_offset
    _, fl = (fn_step or sampler.step)(p, st, [z])
    return bool(fl.converged[0])


def _conv_pins(fn_step=None):
    bad = []
    A, E = sampler.STOP_ARGMAX_STABLE, sampler.STOP_ENTROPY
    cases = [
        # (name, rule, offset, stable_before, step_before, cap, want)
        ("stable, +5e-5", A, 5e-5, 1, 1, 10, True),
        ("stable, -5e-5", A, -5e-5, 1, 1, 10, True),
        ("stable, +2e-4", A, 2e-4, 1, 1, 10, False),
        ("stable, -2e-4", A, -2e-4, 1, 1, 10, False),
        # the argmax not yet stable for k steps: the threshold decides nothing
        ("not yet stable", A, 5e-5, 0, 1, 10, False),
        # first step of a block never counts as stable
        ("first step", A, 5e-5, 5, 0, 10, False),
        # the step cap converges the row whatever the entropy
        ("at the cap", A, 5e-5, 1, 9, 10, False),
        # entropy-only stop: the threshold decides the stable counter itself
        ("entropy stop, +5e-5", E, 5e-5, 0, 1, 10, True),
        ("entropy stop, -5e-5", E, -5e-5, 0, 1, 10, True),
        ("entropy stop, 2e-4", E, 2e-4, 0, 1, 10, False),
    ]
    for name, rule, off, stb, stp, cap, want in cases:
        if _conv_case(rule, off, stb, stp, cap, fn_step=fn_step) != want:
            bad.append(name)
    return bad


def test_convergence_flag():
    assert _conv_pins() == []


# ------------------------------------------------- monotone commit flag

def _monotone_case(conf_offset, mode_changed, committed):
    """One position (V = 2, T = 1, z = [a, 0]: confidence sigmoid(a)) under
    the unchanged-or-stronger rule, with prev_conf = sigmoid(a) + offset."""
    a = 1.3
    conf = 1.0 / (1.0 + math.exp(-a))
    p = sampler.Params(batch=1, canvas_len=1, vocab=2, seed=8, entropy_budget=0.0,
                       conf_threshold=-1.0, stable_k=3, step_cap=10,
                       accept_rule=sampler.ACCEPT_MONOTONE)
    st = sampler.new_state(p, [sampler.PHASE_DENOISE], [4], [1.0])
    st.step[0] = 1
    st.argmax_prev[0] = [1 if mode_changed else 0]
    st.prev_conf[0] = [conf + conf_offset]
    st.committed[0] = [1 if committed else 0]
    out, fl = sampler.step(p, st, [np.array([[a, 0.0]])])
    return bool(fl.commit[0, 0]), out


def test_monotone_commit_flag():
    # confidence within 5e-5 of the previous one, mode changed: the decision
    # is the confidence comparison, flagged
    for off in (5e-5, -5e-5):
        fl, out = _monotone_case(off, True, False)
        assert fl, off
        assert bool(out.committed[0, 0]) == (off <= 0)  # conf >= prev commits
    # 2e-4 away: decided, not flagged
    for off in (2e-4, -2e-4):
        assert not _monotone_case(off, True, False)[0], off
    # mode unchanged: it commits whatever the confidence, not flagged
    fl, out = _monotone_case(5e-5, False, False)
    assert not fl and out.committed[0, 0] == 1
    # committed earlier: frozen, not flagged
    fl, out = _monotone_case(5e-5, True, True)
    assert not fl and out.committed[0, 0] == 1


# ------------------------------------------------ planted slips are caught

def _mutant(fn, old, new):
    """A copy of oracle function ``fn`` with ``old`` replaced by ``new`` in
    its source, compiled in the oracle module's namespace."""
    src = textwrap.dedent(inspect.getsource(fn))
    assert src.count(old) == 1, old
    ns = dict(vars(inspect.getmodule(fn)))
    exec(compile(src.replace(old, new), "<mutant>", "exec"), ns)
    return ns[fn.__name__]


ACCEPT_SLIPS = {
    # the flag compares the inclusive prefix (the sum including position k)
    "inclusive prefix": ("if k > 0 and abs(prefix - budget) < NEAR_TIE:",
                         "if abs(prefix + key[i] - budget) < NEAR_TIE:"),
    # the first position's empty prefix is flagged against the budget
    "first position flagged": ("if k > 0 and abs(prefix - budget) < NEAR_TIE:",
                               "if abs(prefix - budget) < NEAR_TIE:"),
    # non-strict comparisons
    "<= on the prefix": ("if k > 0 and abs(prefix - budget) < NEAR_TIE:",
                         "if k > 0 and abs(prefix - budget) <= NEAR_TIE:"),
    "<= on the neighbours": ("if abs(b - a) < NEAR_TIE:", "if abs(b - a) <= NEAR_TIE:"),
    # neighbours taken one step off the cut
    "neighbours off by one": ("a, b = key[order[n_acc - 1]], key[order[n_acc]]",
                              "a, b = key[order[n_acc - 2]], key[order[n_acc - 1]]"),
    # no neighbour test at all
    "no neighbour test": ("if abs(b - a) < NEAR_TIE:", "if False:"),
}


@pytest.mark.parametrize("slip", sorted(ACCEPT_SLIPS))
def test_acceptance_pins_catch_slip(slip):
    old, new = ACCEPT_SLIPS[slip]
    mutant = _mutant(sampler.accept_mask, old, new)
    try:
        bad = _accept_pins(mutant)
    except IndexError:
        bad = ["raised"]
    assert bad, slip


GAP_SLIPS = {
    # the gap measured on the clean logits instead of the perturbed scores
    "clean-logit gap": ("rest = np.delete(score, cand)\n        gap = float(score[cand] - np.max(rest))",
                        "zz = np.sort(z)\n        gap = float(zz[-1] - zz[-2])"),
    # the gap to the best score strictly below the winner (wrong under ties)
    "gap below ties": ("rest = np.delete(score, cand)",
                       "rest = score[score < score[cand]] if np.any(score < score[cand]) else score"),
    # the gap on the tempered logits without the noise
    "noise-free gap": ("rest = np.delete(score, cand)\n        gap = float(score[cand] - np.max(rest))",
                       "ys = np.sort(y)\n        gap = float(ys[-1] - ys[-2])"),
}


@pytest.mark.parametrize("slip", sorted(GAP_SLIPS))
def test_gap_pins_catch_slip(slip, monkeypatch):
    old, new = GAP_SLIPS[slip]
    mutant = _mutant(sampler.vocab_pass, old, new)
    assert _gap_pins(monkeypatch, mutant), slip


CONV_SLIPS = {
    # the flag set whenever the mean entropy is near, relevant or not
    "always relevant": ("flags.converged[r] = near and st.stable[r] >= p.stable_k and st.step[r] < p.step_cap",
                        "flags.converged[r] = near"),
    # a window wider than the rule's 1e-4
    "window too wide": ("abs(Hbar - p.conf_threshold) < NEAR_TIE",
                        "abs(Hbar - p.conf_threshold) < 3 * NEAR_TIE"),
}


@pytest.mark.parametrize("slip", sorted(CONV_SLIPS))
def test_convergence_pins_catch_slip(slip, monkeypatch):
    old, new = CONV_SLIPS[slip]
    mutant = _mutant(sampler.denoise_row, old, new)
    monkeypatch.setattr(sampler, "denoise_row", mutant)
    assert _conv_pins(), slip
