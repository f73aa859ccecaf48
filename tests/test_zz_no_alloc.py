"""The allocation-free sampler step, for callers that cannot allocate device
memory (an engine whose device memory is all pre-planned by its own pool, or a
host application whose allocations belong to another framework's allocator).

dg_denoise_step_noalloc must give the same results as dg_denoise_step, which
takes a caller workspace, over two calls in a row (the second call starts from
the state the first one left and reuses the library's fixed scratch).  This
file is collected last so a first failure here does not hide the others."""

import ctypes

import numpy as np
import pytest
import torch

import denoise_step_sampler_gb300 as dg
from denoise_step_sampler_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

ENT_TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    from denoise_step_sampler_gb300 import build
    build.build()
    dg.lib()


def _state(p, temps):
    st = dg.State(p.batch, p.canvas_len, "cuda")
    st.phase.fill_(dg.DG_PHASE_DENOISE)
    st.phase[0] = dg.DG_PHASE_PREFILL
    st.temperature.copy_(torch.tensor(temps, dtype=torch.float32))
    st.request_id.copy_(torch.arange(p.batch) + 40)
    return st


def _compare(a, b):
    for k in ("canvas", "cand", "argmax", "argmax_prev", "accept", "phase", "step", "stable",
              "rng_step", "converged", "sc_valid", "num_sampled", "num_rejected", "emitted",
              "device_status"):
        assert np.array_equal(a[k], b[k]), k
    for k in ("entropy", "m", "mean_entropy"):
        ok = np.isnan(a[k]) == np.isnan(b[k])
        assert ok.all(), k
        f = ~np.isnan(a[k])
        assert np.all(np.abs(a[k][f] - b[k][f]) <= ENT_TOL), k
    assert np.allclose(a["s"], b["s"], rtol=1e-5, atol=0.0, equal_nan=True)
    # the unchanged-or-stronger rule's per-position state
    assert np.array_equal(a["committed"], b["committed"])
    assert np.allclose(a["prev_conf"], b["prev_conf"], rtol=1e-5, atol=0.0, equal_nan=True)


@pytest.mark.parametrize("B,C,V,dt,rule", [
    (3, 256, 50257, dg.DG_BF16, dg.DG_ACCEPT_ENTROPY_BUDGET),
    (2, 64, 3001, dg.DG_F32, dg.DG_ACCEPT_ENTROPY_BUDGET),
    (3, 128, 4099, dg.DG_BF16, dg.DG_ACCEPT_MONOTONE),
])
def test_noalloc_step_matches_workspace_step_twice(B, C, V, dt, rule):
    p = dg.Params(batch=B, canvas_len=C, vocab=V, logits_dtype=dt, seed=77,
                  entropy_budget=40.0, conf_threshold=0.3, stable_k=1, step_cap=8,
                  accept_rule=rule)
    temps = list(np.linspace(0.7, 1.2, B))
    tdt = torch.bfloat16 if dt == dg.DG_BF16 else torch.float32
    ref, new = _state(p, temps), _state(p, temps)
    ws = torch.empty(dg.dg_workspace_bytes(p, 0), dtype=torch.uint8, device="cuda")
    L = dg.lib()
    for step in range(2):
        logits = syn.boosted_logits(B * C, V, seed=1000 + step, dtype=tdt, device="cuda").reshape(-1)
        dg.dg_denoise_step(p, logits, ref, ws)
        rc = L.dg_denoise_step_noalloc(ctypes.byref(p.c()), ctypes.c_void_p(logits.data_ptr()),
                                       ctypes.byref(new.c()),
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == dg.DG_OK, dg.dg_status_string(rc)
        torch.cuda.synchronize()
        _compare(new.snapshot(), ref.snapshot())


def test_noalloc_rejects_problems_beyond_its_scratch():
    p = dg.Params(batch=512, canvas_len=256, vocab=262144, logits_dtype=dg.DG_BF16)
    # the size check comes before any pointer is used
    fake = dg._CState(*([0x1000] * len(dg._STATE_FIELDS)))
    rc = dg.lib().dg_denoise_step_noalloc(ctypes.byref(p.c()), ctypes.c_void_p(0x10000),
                                          ctypes.byref(fake), None)
    assert rc == dg.DG_ERR_SCRATCH_LIMIT
    assert "scratch" in dg.dg_status_string(rc)
