"""Counter-based random numbers of the sampler, written from their published
definitions (test infrastructure; see the package docstring).

The pages fix no generator: the ML@Berkeley walkthrough ("DiffusionGemma
Explained", section "Sampling") draws with torch's stateful RNG and the vLLM
blog (section "DiffusionGemma sampler") adds unspecified ``gumbel_noise``.
This module is the library's own definition, keyed by
(seed, request_id, rng_step, position, tag) so that any implementation can
reproduce a draw bit for bit:

* ``mix64``   -- the SplitMix64 output function (Steele, Lea & Flood,
  "Fast splittable pseudorandom number generators", OOPSLA 2014).
* ``fmix32``  -- the 32-bit finalizer of MurmurHash3 (Appleby, public domain).
* ``position_key`` / ``stream_key`` -- the key chain
  P = mix64(mix64(mix64(mix64(seed) ^ request) ^ rng_step) ^ position),
  K_tag = mix64(P ^ tag).
* ``draw32(K, x)`` = fmix32(lo32(K) ^ x) for a 32-bit counter x.
* ``uniform(h)`` = (h + 1/2) / 2^32, in (0, 1), never 0 or 1.
* ``exp1(h)``   = -ln uniform(h), an Exp(1) variate.
* ``below(h, n)`` = floor(h * n / 2^32), an integer in [0, n).

Gumbel noise (tags GMIN, GARG, GREST) uses the exact group construction of
iid Exp(1) variables by the memoryless property: for a group of n iid Exp(1)
variables the minimum is Exp(1)/n, its position is uniform and independent,
and every other member is the minimum plus a fresh Exp(1).  Groups are the
8 consecutive vocabulary indices [8g, 8g+8) (the last one ragged):

    X_g = exp1(draw32(K_GMIN, g)),   J_g = below(draw32(K_GARG, g), n_g),
    E_v = X_g / n_g + [v - 8g != J_g] * exp1(draw32(K_GREST, v)),
    G_v = -ln E_v  (standard Gumbel).

The segmented (hierarchical) Gumbel-max rule uses tags SEG and WITHIN over a
fixed partition of the vocabulary into segments of 32 indices: superblock j
holds the indices [1024 j, 1024 j + 1024), and its segment l (0 <= l < 32)
the four groups of 8 at offsets 8 l, 256 + 8 l, 512 + 8 l and 768 + 8 l, so
segment k = 32 j + l holds {1024 j + 256 u + 8 l + t : 0 <= u < 4,
0 <= t < 8} (indices >= V left out).
"""

from __future__ import annotations

import numpy as np

TAG_GMIN = 1
TAG_GARG = 2
TAG_GREST = 3
TAG_RENOISE = 4
TAG_INIT = 5
TAG_SEG = 6      # one Exp(1) per vocabulary segment (segmented rule)
TAG_WITHIN = 7   # one Exp(1) per index, used inside the winning segment

GROUP = 8
SUPERBLOCK = 1024  # indices per superblock: 32 segments of 4 groups of 8
SEGMENTS_PER_SUPERBLOCK = 32

_U64 = np.uint64
_GOLDEN = _U64(0x9E3779B97F4A7C15)
_SM_M1 = _U64(0xBF58476D1CE4E5B9)
_SM_M2 = _U64(0x94D049BB133111EB)
_MASK32 = _U64(0xFFFFFFFF)


def mix64(x):
    """SplitMix64 output function of the state ``x`` (uint64, vectorised).

    z = x + 0x9E3779B97F4A7C15; z = (z ^ z>>30) * 0xBF58476D1CE4E5B9;
    z = (z ^ z>>27) * 0x94D049BB133111EB; return z ^ z>>31  (all mod 2^64).
    """
    x = np.asarray(x, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = x + _GOLDEN
        z = (z ^ (z >> _U64(30))) * _SM_M1
        z = (z ^ (z >> _U64(27))) * _SM_M2
    return z ^ (z >> _U64(31))


def fmix32(h):
    """MurmurHash3 32-bit finalizer (uint32, vectorised).

    h ^= h>>16; h *= 0x85EBCA6B; h ^= h>>13; h *= 0xC2B2AE35; h ^= h>>16.
    """
    h = np.asarray(h, dtype=np.uint32)
    with np.errstate(over="ignore"):
        h = h ^ (h >> np.uint32(16))
        h = h * np.uint32(0x85EBCA6B)
        h = h ^ (h >> np.uint32(13))
        h = h * np.uint32(0xC2B2AE35)
        h = h ^ (h >> np.uint32(16))
    return h


def _u64(v):
    return np.asarray(v).astype(np.uint64) if np.asarray(v).dtype != np.uint64 else np.asarray(v)


def position_key(seed, request_id, rng_step, position):
    """P = mix64(mix64(mix64(mix64(seed) ^ request_id) ^ rng_step) ^ position).

    All arguments are taken modulo 2^64 and broadcast against each other.
    """
    k = mix64(_u64(seed))
    k = mix64(k ^ _u64(request_id))
    k = mix64(k ^ _u64(rng_step))
    k = mix64(k ^ _u64(position))
    return k


def stream_key(pkey, tag):
    """K_tag = mix64(P ^ tag)."""
    return mix64(_u64(pkey) ^ _U64(tag))


def lo32(k):
    return (np.asarray(k, dtype=np.uint64) & _MASK32).astype(np.uint32)


def hi32(k):
    return (np.asarray(k, dtype=np.uint64) >> _U64(32)).astype(np.uint32)


def draw32(key, x):
    """fmix32(lo32(key) ^ x); ``key`` broadcasts against the counters ``x``."""
    return fmix32(lo32(key) ^ np.asarray(x, dtype=np.uint32))


def uniform(h):
    """(h + 1/2) / 2^32 as float64 (exact), in (0, 1)."""
    return (np.asarray(h, dtype=np.uint32).astype(np.float64) + 0.5) * 2.0 ** -32


def exp1(h):
    """-ln U(h).  For U > 1/2 it is evaluated as -log1p(-W) with the exact
    complement W = 1 - U = (2^32 - 1 - h + 1/2) / 2^32, so that tiny values
    keep full relative precision."""
    h = np.asarray(h, dtype=np.uint32)
    u = uniform(h)
    w = uniform(~h)
    return np.where(h < np.uint32(1 << 31), -np.log(u), -np.log1p(-w))


def below(h, n):
    """floor(h * n / 2^32) for n < 2^32, computed exactly in integers."""
    h = np.asarray(h, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return ((h * _u64(n)) >> _U64(32)).astype(np.int64)


def gumbel_exponentials(V, ka, kb, kc):
    """The iid Exp(1) variables E_v, v in [0, V), of one position whose Gumbel
    stream keys are (K_GMIN, K_GARG, K_GREST) = (ka, kb, kc)."""
    v = np.arange(V, dtype=np.int64)
    g = v // GROUP
    ng = np.minimum(GROUP, V - GROUP * np.arange((V + GROUP - 1) // GROUP))
    x_g = exp1(draw32(ka, np.arange(ng.size, dtype=np.uint32)))
    j_g = below(draw32(kb, np.arange(ng.size, dtype=np.uint32)), ng)
    rest = exp1(draw32(kc, v.astype(np.uint32)))
    is_min = (v - GROUP * g) == j_g[g]
    return x_g[g] / ng[g] + np.where(is_min, 0.0, rest)


def segment_of(v):
    """Segment index of vocabulary index v (vectorised):
    32 * (v // 1024) + (v mod 256) // 8."""
    v = np.asarray(v, dtype=np.int64)
    return SEGMENTS_PER_SUPERBLOCK * (v // SUPERBLOCK) + (v % 256) // GROUP


def segment_members(k, V):
    """The vocabulary indices of segment k, ascending (those < V)."""
    j, lane = divmod(int(k), SEGMENTS_PER_SUPERBLOCK)
    v = np.array([SUPERBLOCK * j + 256 * u + GROUP * lane + t
                  for u in range(4) for t in range(GROUP)], dtype=np.int64)
    return v[v < V]


def gumbel_noise(V, ka, kb, kc):
    """G_v = -ln E_v, standard Gumbel variates."""
    return -np.log(gumbel_exponentials(V, ka, kb, kc))


def uniform_token(key, V):
    """A token uniform in [0, V) from the high half of a 64-bit stream key
    (used for re-noising and for canvas initialisation)."""
    return below(hi32(key), V)
