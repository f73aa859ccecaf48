"""Parity of the on-device temperature anneal with the oracle, alone and
inside a multi-step denoise loop."""

import numpy as np
import pytest
import torch

import denoise_step_sampler_gb300 as dg
from denoise_step_sampler_gb300 import synthetic as syn
from oracle import sampler as osam

from _gpu_common import denoise_and_compare, make_state

pytestmark = pytest.mark.gpu


def test_anneal_is_bit_exact():
    B, C, V = 7, 8, 64
    p = dg.Params(batch=B, canvas_len=C, vocab=V, logits_dtype=dg.DG_F32, seed=1)
    st = make_state(p, [dg.DG_PHASE_DENOISE] * B, temperatures=np.full(B, 0.9))
    steps = np.array([0, 1, 12, 23, 24, 40, -2], np.int32)
    st.step.copy_(torch.as_tensor(steps))
    mask = np.array([1, 1, 1, 1, 1, 1, 0], np.uint8)
    for t_max, t_min, N in [(0.8, 0.4, 24), (1.3, 0.55, 7), (0.5, 1.5, 24)]:
        before = st.temperature.cpu().numpy()
        dg.dg_anneal_temperature(p, st, t_max, t_min, N, row_mask=torch.as_tensor(mask, device="cuda"))
        torch.cuda.synchronize()
        got = st.temperature.cpu().numpy()
        want = osam.anneal_temperature(steps, before, t_max, t_min, N, row_mask=mask)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), (t_max, t_min, N, got, want)
    # without a mask every row is updated
    dg.dg_anneal_temperature(p, st, 1.0, 0.5, 10)
    torch.cuda.synchronize()
    want = osam.anneal_temperature(steps, np.zeros(B, np.float32), 1.0, 0.5, 10)
    assert np.array_equal(st.temperature.cpu().numpy().view(np.uint32), want.view(np.uint32))


def test_annealed_denoise_loop_matches_oracle():
    # every step: anneal from the block-local step counter, then one denoise
    # step compared with the oracle from the same prior state
    B, C, V, N = 2, 64, 4096, 6
    p = dg.Params(batch=B, canvas_len=C, vocab=V, logits_dtype=dg.DG_BF16, seed=0xD1FF0003,
                  entropy_budget=12.0, conf_threshold=0.3, stable_k=3, step_cap=N)
    st = make_state(p, [dg.DG_PHASE_DENOISE] * B, request_ids=[11, 12], temperatures=[1.0, 1.0])
    for k in range(N):
        step_before = st.step.cpu().numpy().copy()
        T_before = st.temperature.cpu().numpy().copy()
        dg.dg_anneal_temperature(p, st, 1.2, 0.6, N)
        torch.cuda.synchronize()
        want = osam.anneal_temperature(step_before, T_before, 1.2, 0.6, N)
        assert np.array_equal(st.temperature.cpu().numpy().view(np.uint32), want.view(np.uint32)), k
        logits = torch.stack([syn.loop_logits(C, V, seed=p.seed, request=r, step=k, device="cuda")
                              for r in (11, 12)]).reshape(-1)
        denoise_and_compare(p, st, logits)
