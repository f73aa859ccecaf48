"""Pins of the oracle's segmented (hierarchical) Gumbel-max rule: a segment
drawn by Gumbel-max over segment masses, then an index drawn by Gumbel-max
inside it.  By the max-stability of the Gumbel law this is an exact draw from
softmax(y), the same law as the flat argmax(y + G) (vLLM blog, "Putting it
together": argmax(logits/T + gumbel_noise)).  The pins check the partition,
the law of the draw by chi-square against scipy's softmax (over segments,
inside a segment and over indices), the low-temperature limit, and that a
planted slip fails them.  CPU only."""

import numpy as np
import pytest
from scipy import special, stats

from oracle import rng, sampler


def _draws(z, T, n, seed, fn=None):
    fn = fn or sampler.segmented_candidate
    counts = np.zeros(z.size, dtype=np.int64)
    y = np.asarray(z, np.float64) / T
    for r in range(n):
        ks, kw = sampler.segment_keys(seed, r, 3, 5)
        counts[fn(y, ks, kw)[0]] += 1
    return counts


@pytest.mark.parametrize("V", [1, 8, 300, 1024, 1300, 4099])
def test_segments_partition_the_vocabulary(V):
    v = np.arange(V)
    seg = rng.segment_of(v)
    seen = np.zeros(V, dtype=np.int64)
    for k in np.unique(seg):
        mem = rng.segment_members(k, V)
        assert np.all(rng.segment_of(mem) == k)
        assert mem.size <= 32 and np.all(np.diff(mem) > 0)
        seen[mem] += 1
    assert np.all(seen == 1)
    # full superblocks hold 32 segments of 32 indices each
    for k in range(32 * (V // 1024)):
        assert rng.segment_members(k, V).size == 32
    # the lane layout: index 1024 j + 256 u + 8 l + t is in segment 32 j + l
    assert rng.segment_of(1024 * 3 + 256 * 2 + 8 * 5 + 7) == 32 * 3 + 5


def test_law_over_indices_in_several_segments():
    # mass on 12 indices spread over segments of two superblocks (the rest -inf)
    V = 1300
    z = np.full(V, -np.inf)
    hot = np.array([3, 7, 9, 260, 300, 517, 1030, 1031, 1100, 1299, 40, 41])
    z[hot] = np.random.default_rng(1).normal(0, 1, hot.size)
    n = 20000
    c = _draws(z, 1.0, n, seed=21)
    assert c[np.setdiff1d(np.arange(V), hot)].sum() == 0
    p = special.softmax(z[hot])
    assert stats.chisquare(c[hot], n * p).pvalue > 1e-3


@pytest.mark.parametrize("T", [0.6, 1.0, 1.7])
def test_law_with_finite_logits(T):
    V = 2048
    g = np.random.default_rng(2)
    z = g.normal(0, 1, V)
    z[[5, 700, 1500, 1501]] += [4.0, 3.5, 3.0, 2.5]
    n = 12000
    c = _draws(z, T, n, seed=22)
    p = special.softmax(z / T)
    head = [5, 700, 1500, 1501]
    obs = np.concatenate([c[head], [n - c[head].sum()]])
    exp = n * np.concatenate([p[head], [1 - p[head].sum()]])
    assert stats.chisquare(obs, exp).pvalue > 1e-3
    # the segment of the draw follows the segment masses
    seg = rng.segment_of(np.arange(V))
    W = np.bincount(seg, weights=p)
    cs = np.bincount(seg, weights=c)
    big = W * n > 40
    obs, exp = cs[big], n * W[big]
    if (~big).any():
        obs = np.concatenate([obs, [cs[~big].sum()]])
        exp = np.concatenate([exp, [n * W[~big].sum()]])
    assert stats.chisquare(obs, exp).pvalue > 1e-3


def test_law_inside_one_segment():
    # all the mass in one segment: the inner draw alone follows softmax
    V = 1024
    z = np.full(V, -np.inf)
    mem = rng.segment_members(9, V)
    z[mem] = np.random.default_rng(3).normal(0, 1, mem.size)
    n = 16000
    c = _draws(z, 1.0, n, seed=23)
    assert stats.chisquare(c[mem], n * special.softmax(z[mem])).pvalue > 1e-3


def test_low_temperature_gives_the_argmax():
    g = np.random.default_rng(4)
    for r in range(30):
        z = np.round(g.normal(0, 2, 3000), 1)
        z[g.integers(3000)] += 0.5
        srt = np.sort(z)
        if srt[-1] - srt[-2] < 0.05:
            continue
        ks, kw = sampler.segment_keys(9, r, 0, 0)
        cand, _ = sampler.segmented_candidate(z / 1e-3, ks, kw)
        assert cand == int(np.argmax(z))


def test_vocab_pass_routes_the_rule_and_keeps_the_rest():
    z = np.random.default_rng(5).normal(0, 2, 5000)
    keys = sampler.gumbel_keys(1, 2, 3, 4)
    sk = sampler.segment_keys(1, 2, 3, 4)
    a = sampler.vocab_pass(z, 0.8, *keys)
    b = sampler.vocab_pass(z, 0.8, *keys, sampler.SAMPLE_SEGMENTED, sk)
    assert (a.m, a.s, a.entropy, a.argmax) == (b.m, b.s, b.entropy, b.argmax)
    cand, gap = sampler.segmented_candidate(z / 0.8, *sk)
    assert (b.cand, b.gap) == (cand, gap)


def test_planted_slip_is_caught():
    """Taking the winning segment's largest logit instead of drawing inside
    it (a plausible slip) must fail the law."""
    import inspect
    import textwrap
    src = textwrap.dedent(inspect.getsource(sampler.segmented_candidate))
    old = "s2 = y[members] - np.log(Ew)"
    assert src.count(old) == 1
    ns = dict(vars(sampler))
    exec(compile(src.replace(old, "s2 = y[members] + 0.0 * Ew"), "<mutant>", "exec"), ns)
    V = 1024
    z = np.full(V, -np.inf)
    mem = rng.segment_members(9, V)
    z[mem] = np.random.default_rng(3).normal(0, 1, mem.size)
    n = 4000
    c = _draws(z, 1.0, n, seed=23, fn=ns["segmented_candidate"])
    assert stats.chisquare(c[mem], n * special.softmax(z[mem])).pvalue < 1e-6
