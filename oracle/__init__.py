"""Plain fp64 CPU oracle of the per-denoise-step sampler and self-conditioning feed.

TEST INFRASTRUCTURE ONLY.  Nothing in the product (the CUDA library and its
Python binding) imports, calls or links this package.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg use it.

It is written from the method's definitions, step by step, in float64 with
numpy, with no blocking, fusion or reordering beyond what the definitions
state:

* ``rng``       -- the counter-based random numbers (SplitMix64 key chain,
                   MurmurHash3 fmix32 draws, exact Exp(1) groups).
* ``sampler``   -- temperature, softmax, entropy, clean argmax, Gumbel-max
                   candidate, entropy-bounded acceptance, re-noise,
                   convergence and the prefill / denoise / commit phases.
* ``selfcond``  -- the probability-weighted embedding softmax(z/T) . E.
* ``forward``   -- the forward-process transition row (used as a pin).

Sources ("DiffusionGemma Technical Report -- part 2/6", "DiffusionGemma
Explained" (ML@Berkeley), the vLLM blog "DiffusionGemma: the first dLLM
natively supported in vLLM") are cited per function.

Parity status: every function here is pinned by tests in
``tests/test_oracle_pins.py`` against closed forms, library routines,
brute force or statistical laws; the pages print no numeric worked example
of the sampler, so no pin compares against a printed value.
"""

from . import rng, sampler, selfcond, forward  # noqa: F401
