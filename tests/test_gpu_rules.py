"""Parity of the rule variants with the oracle: the entropy-only stop rule
and the unchanged-or-stronger monotone commit rule ("DiffusionGemma-Lite
DIFFUSION.html", sections 4.4 and 4.2), over multi-step loops that reach the
commit, and with mixed phases."""

import numpy as np
import pytest
import torch

import denoise_step_sampler_gb300 as dg
from denoise_step_sampler_gb300 import synthetic as syn

from _gpu_common import denoise_and_compare, make_state

pytestmark = pytest.mark.gpu


def _loop(p, rids, temps, steps, V):
    st = make_state(p, [dg.DG_PHASE_PREFILL] * p.batch, request_ids=rids, temperatures=temps)
    seen_commit = 0
    flagged = 0
    for k in range(steps):
        logits = torch.stack([syn.loop_logits(p.canvas_len, V, seed=p.seed, request=r, step=k,
                                              device="cuda") for r in rids]).reshape(-1)
        before_phase = st.phase.cpu().numpy().copy()
        _, after, _, _, n = denoise_and_compare(p, st, logits)
        flagged += n["accept"]
        seen_commit += int(np.sum(before_phase == dg.DG_PHASE_COMMIT))
    return st, seen_commit, flagged


@pytest.mark.parametrize("stop_rule,accept_rule", [
    (dg.DG_STOP_ENTROPY, dg.DG_ACCEPT_ENTROPY_BUDGET),
    (dg.DG_STOP_ARGMAX_STABLE, dg.DG_ACCEPT_MONOTONE),
    (dg.DG_STOP_ENTROPY, dg.DG_ACCEPT_MONOTONE),
])
def test_rule_loop_matches_oracle(stop_rule, accept_rule):
    B, C, V = 3, 128, 4096
    p = dg.Params(batch=B, canvas_len=C, vocab=V, logits_dtype=dg.DG_BF16, seed=0xD1FF0007,
                  entropy_budget=24.0, conf_threshold=1.5, stable_k=2, step_cap=7,
                  stop_rule=stop_rule, accept_rule=accept_rule)
    st, commits, flagged = _loop(p, [21, 22, 23], [0.7, 1.0, 1.2], 12, V)
    assert commits >= B, commits          # every request reached its commit at least once
    if accept_rule == dg.DG_ACCEPT_MONOTONE:
        assert flagged <= B * C            # near ties stay rare


def test_monotone_with_mixed_phases_and_noalloc():
    # one row of each phase; the monotone state of prefill and commit rows is
    # reset, and the allocation-free entry gives the same state
    B, C, V = 4, 64, 2048
    p = dg.Params(batch=B, canvas_len=C, vocab=V, logits_dtype=dg.DG_F32, seed=31,
                  entropy_budget=8.0, conf_threshold=0.5, stable_k=2, step_cap=5,
                  accept_rule=dg.DG_ACCEPT_MONOTONE)
    phases = [dg.DG_PHASE_PREFILL, dg.DG_PHASE_DENOISE, dg.DG_PHASE_COMMIT, dg.DG_PHASE_IDLE]
    st = make_state(p, phases, request_ids=[1, 2, 3, 4], temperatures=[1.0] * B,
                    argmax_prev=np.arange(B * C) % V)
    g = torch.Generator(device="cpu").manual_seed(3)
    st.committed.copy_(torch.randint(0, 2, (B * C,), generator=g, dtype=torch.uint8))
    st.prev_conf.copy_(torch.rand(B * C, generator=g))
    st.cand.copy_(torch.randint(0, V, (B * C,), generator=g, dtype=torch.int32))
    logits = syn.boosted_logits(B * C, V, seed=5, dtype=torch.float32, device="cuda").reshape(-1)
    st2 = make_state(p, phases, request_ids=[1, 2, 3, 4], temperatures=[1.0] * B,
                     argmax_prev=np.arange(B * C) % V)
    for name in ("committed", "prev_conf", "cand", "canvas"):
        getattr(st2, name).copy_(getattr(st, name))
    denoise_and_compare(p, st, logits)
    dg.dg_denoise_step_noalloc(p, logits, st2)
    torch.cuda.synchronize()
    a, b = st.snapshot(), st2.snapshot()
    for k in a:
        assert np.array_equal(a[k], b[k], equal_nan=True) if a[k].dtype.kind == "f" else \
            np.array_equal(a[k], b[k]), k
