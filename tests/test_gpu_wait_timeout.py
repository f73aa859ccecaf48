"""A bounded wait of the self-conditioning GEMM runs out, on purpose, and the
call still ends with its error reported and the context usable.

The library's test build (libdg_waittest.so, same sources) bounds its
pipeline waits at 1 ms and withholds the E copies of the third k-block, so
the wait for them can only run out.  Nothing faults, traps or waits without
a bound: waits for copies or MMAs already issued keep their 2 s bound, so
no CTA exits or frees its TMEM with work in flight.  The test checks that
the call returns promptly, that DG_DEV_WAIT_TIMEOUT is set, that the wait
record names a real wait, and that the default build then computes the
same call correctly in the same context."""

import ctypes
import time

import numpy as np
import pytest
import torch

import denoise_step_sampler_gb300 as dg
from denoise_step_sampler_gb300 import build
from denoise_step_sampler_gb300 import synthetic as syn

from _gpu_common import make_state, oracle_selfcond_rows, selfcond_check

pytestmark = pytest.mark.gpu

ROLES = {0: "TMA", 1: "MMA", 2: "producer", 3: "epilogue"}
BARRIERS = {0: "E landed", 1: "p ready", 2: "E stage free", 3: "accumulator full",
            4: "logits landed", 5: "logits stage free"}


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    dg.lib()


def test_selfcond_wait_runs_out_and_the_context_stays_usable():
    B, C, V, d = 2, 256, 8192, 512
    p = dg.Params(batch=B, canvas_len=C, vocab=V, logits_dtype=dg.DG_BF16, seed=77,
                  entropy_budget=50.0, conf_threshold=-1.0, stable_k=3, step_cap=1000)
    temps = [0.8, 1.1]
    st = make_state(p, [dg.DG_PHASE_DENOISE] * B, temperatures=temps)
    logits = syn.boosted_logits(B * C, V, seed=9, device="cuda").reshape(-1)
    E = syn.embedding(V, d, seed=10, device="cuda")
    ws = torch.empty(max(16, dg.dg_workspace_bytes(p, d)), dtype=torch.uint8, device="cuda")
    dg.dg_denoise_step(p, logits, st, ws)
    torch.cuda.synchronize()
    assert int(st.device_status.item()) == 0

    L = dg.load(build.WAIT_TEST_LIB)
    rec0 = (ctypes.c_uint32 * 4)()
    assert L.dg_debug_wait_record(ctypes.cast(rec0, ctypes.c_void_p)) == dg.DG_OK
    assert rec0[0] == 0  # no wait has given up in this build yet
    out = torch.zeros((B * C, d), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    t0 = time.perf_counter()
    rc = L.dg_selfcond_embed(ctypes.byref(p.c()), ctypes.c_void_p(logits.data_ptr()),
                             ctypes.byref(st.c()), ctypes.c_void_p(E.data_ptr()), d,
                             E.stride(0), ctypes.c_void_p(out.data_ptr()), dg.DG_F32,
                             ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                             ctypes.c_void_p(stream.cuda_stream))
    assert rc == dg.DG_OK
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert elapsed < 1.5, elapsed  # the 1 ms bound ended the call, not the 2 s drains
    status = int(st.device_status.item())
    assert status & dg.DG_DEV_WAIT_TIMEOUT, status
    rec = (ctypes.c_uint32 * 4)()
    assert L.dg_debug_wait_record(ctypes.cast(rec, ctypes.c_void_p)) == dg.DG_OK
    assert rec[0] == 1
    where = rec[2]
    role, bar, it = where >> 28, (where >> 24) & 0xF, where & 0xFFFF
    assert role in ROLES and bar in BARRIERS, hex(where)
    # the first wait to give up waits on the withheld k-block or on work
    # that waits for it (the pipeline runs at most a ring's depth ahead)
    assert it <= 2 + 4, (ROLES[role], BARRIERS[bar], it)

    # the default build, same context, same inputs: correct and clean
    st.device_status.zero_()
    out2 = torch.full((B * C, d), float("nan"), dtype=torch.float32, device="cuda")
    dg.dg_selfcond_embed(p, logits, st, E, out2, ws)
    torch.cuda.synchronize()
    assert int(st.device_status.item()) == 0
    got = out2.cpu().numpy()
    zh = logits.view(B, C, V).float().cpu().numpy()
    Eh = E.float().cpu().numpy().astype(np.float64)
    for r in range(B):
        rows = np.arange(0, C, 17)
        ref = oracle_selfcond_rows(zh[r, rows].astype(np.float64), float(np.float32(temps[r])), Eh)
        selfcond_check(got[r * C + rows], ref)
