"""GPU parity of the fused step dg_denoise_step_feed: the sampler step and
the self-conditioning feed in one call, the vocabulary pass writing the
feed's operand 2^(z c - R) as it streams the logits.  Against the two calls
dg_denoise_step + dg_selfcond_embed run on a copy of the same state: every
sampler output bit for bit (the vocabulary pass's arithmetic is the same),
and the feed against the fp64 oracle within the feed tolerance.  Covered:
first and second steps; positions whose previous maximum is far from the new
one (the operand would leave bf16's range: p is written by a separate pass
instead); rows that do not feed; the softcap with the embedding scale; and
inputs the fusion does not take (unaligned rows, the grouped rule), which run
the two calls."""

import numpy as np
import pytest
import torch

import denoise_step_sampler_gb300 as dg
from denoise_step_sampler_gb300 import synthetic as syn

from _gpu_common import make_state, oracle_selfcond_rows, selfcond_check
from oracle import selfcond as osc

pytestmark = pytest.mark.gpu

FIELDS = ("canvas", "argmax_prev", "cand", "argmax", "accept", "m", "s", "entropy", "step",
          "stable", "mean_entropy", "converged", "sc_valid", "phase", "rng_step",
          "num_sampled", "num_rejected", "device_status")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from denoise_step_sampler_gb300 import build
    build.build()
    dg.lib()


def _clone(st: dg.State) -> dg.State:
    c = dg.State(st.batch, st.canvas_len, "cuda")
    for k, v in vars(st).items():
        if isinstance(v, torch.Tensor):
            getattr(c, k).copy_(v)
    return c


def _check_feed(got, logits2d, T, Eh, rows, C, cap=0.0, scale=0.0):
    # rows grouped by canvas (one temperature each), one fp64 product per group
    rows = np.asarray(rows)
    for r in np.unique(rows // C):
        sel = rows[rows // C == r]
        z = logits2d[torch.as_tensor(sel, device=logits2d.device)].float().cpu().numpy()
        if cap > 0 or scale > 0:
            ref = osc.selfcond_rows(z.astype(np.float64), float(np.float32(T[r])), Eh,
                                    cap=float(np.float32(cap)), scale=float(np.float32(scale)))
        else:
            ref = oracle_selfcond_rows(z.astype(np.float64), float(np.float32(T[r])), Eh)
        selfcond_check(got[sel], ref)


def _steps(p, phases, logits, E, temps, n_steps=2, m_init=None, out_dtype=torch.float32,
           sample_rows=None):
    st_a = make_state(p, phases, temperatures=temps)
    if m_init is not None:
        st_a.m.copy_(m_init)
    st_b = _clone(st_a)
    d = E.shape[1]
    Eh = E.float().cpu().numpy().astype(np.float64)
    ws_a = torch.empty(max(16, dg.dg_workspace_bytes(p, d)), dtype=torch.uint8, device="cuda")
    ws_b = torch.full((dg.dg_workspace_bytes_feed(p, d),), 0xFF, dtype=torch.uint8, device="cuda")
    n = p.batch * p.canvas_len
    for step in range(n_steps):
        out_a = torch.full((n, d), float("nan"), dtype=out_dtype, device="cuda")
        out_b = torch.full((n, d), float("nan"), dtype=out_dtype, device="cuda")
        dg.dg_denoise_step(p, logits, st_a, ws_a)
        dg.dg_selfcond_embed(p, logits, st_a, E, out_a, ws_a)
        dg.dg_denoise_step_feed(p, logits, st_b, E, out_b, ws_b)
        torch.cuda.synchronize()
        sa, sb = st_a.snapshot(), st_b.snapshot()
        for k in FIELDS:
            assert np.array_equal(np.asarray(sa[k]), np.asarray(sb[k]), equal_nan=True), (step, k)
        assert int(sb["device_status"][0]) == 0
        ga, gb = out_a.float().cpu().numpy(), out_b.float().cpu().numpy()
        feeding = np.repeat(np.asarray(sb["sc_valid"]) != 0, p.canvas_len)
        assert np.all(gb[~feeding] == 0.0) and np.all(ga[~feeding] == 0.0)
        rows = np.nonzero(feeding)[0]
        if sample_rows is not None and len(rows) > sample_rows:
            rows = rows[np.linspace(0, len(rows) - 1, sample_rows).astype(int)]
        ldv = logits.numel() // n
        _check_feed(gb, logits.view(n, ldv)[:, :p.vocab], temps_arr(temps, p.batch), Eh, rows,
                    p.canvas_len, cap=p.softcap, scale=p.embed_scale)
    return st_b


def temps_arr(temps, B):
    return np.asarray(temps, np.float32) if temps is not None else np.ones(B, np.float32)


@pytest.mark.parametrize("B,C,V,d", [(2, 256, 8192, 256), (3, 128, 4096, 128), (1, 64, 2048, 64)],
                         ids=["B2V8192", "B3V4096", "B1V2048"])
def test_feed_matches_the_two_calls_and_the_oracle(B, C, V, d):
    p = dg.Params(batch=B, canvas_len=C, vocab=V, logits_dtype=dg.DG_BF16, seed=31,
                  entropy_budget=40.0, conf_threshold=-1.0, stable_k=3, step_cap=1000,
                  sample_rule=dg.DG_SAMPLE_SEGMENTED)
    temps = list(np.linspace(0.7, 1.2, B))
    logits = syn.boosted_logits(B * C, V, seed=V + B, device="cuda").reshape(-1)
    E = syn.embedding(V, d, seed=d, device="cuda")
    _steps(p, [dg.DG_PHASE_DENOISE] * B, logits, E, temps, n_steps=3, sample_rows=48)


def test_feed_falls_back_where_the_previous_maximum_is_far():
    # canvas 0's previous maxima are far above the new ones (the operand would
    # underflow), canvas 1's far below (it would overflow bf16), canvas 2 has
    # NaN: all three take the separate p pass; canvas 3 keeps the operand
    B, C, V, d = 4, 128, 8192, 128
    p = dg.Params(batch=B, canvas_len=C, vocab=V, logits_dtype=dg.DG_BF16, seed=5,
                  entropy_budget=40.0, conf_threshold=-1.0, stable_k=3, step_cap=1000,
                  sample_rule=dg.DG_SAMPLE_SEGMENTED)
    m0 = torch.zeros(B * C, dtype=torch.float32, device="cuda")
    m0[:C] = 500.0
    m0[C:2 * C] = -300.0
    m0[2 * C:3 * C] = float("nan")
    logits = syn.boosted_logits(B * C, V, seed=3, device="cuda").reshape(-1)
    E = syn.embedding(V, d, seed=4, device="cuda")
    _steps(p, [dg.DG_PHASE_DENOISE] * B, logits, E, [0.8] * B, n_steps=1, m_init=m0)


def test_feed_rows_that_do_not_feed_and_bf16_output():
    B, C, V, d = 4, 64, 4096, 64
    p = dg.Params(batch=B, canvas_len=C, vocab=V, logits_dtype=dg.DG_BF16, seed=4,
                  entropy_budget=50.0, conf_threshold=-1.0, stable_k=1, step_cap=3,
                  sample_rule=dg.DG_SAMPLE_SEGMENTED)
    logits = syn.boosted_logits(B * C, V, seed=1, device="cuda").reshape(-1)
    E = syn.embedding(V, d, seed=6, device="cuda")
    phases = [dg.DG_PHASE_DENOISE, dg.DG_PHASE_PREFILL, dg.DG_PHASE_IDLE, dg.DG_PHASE_DENOISE]
    _steps(p, phases, logits, E, [0.9, 1.0, 1.0, 1.1], n_steps=3, out_dtype=torch.bfloat16)


@pytest.mark.parametrize("kind", ["unaligned", "grouped"])
def test_feed_inputs_that_take_the_two_calls(kind):
    B, C, V, d = 2, 128, 5000, 128
    kw = dict(batch=B, canvas_len=C, vocab=V, logits_dtype=dg.DG_BF16, seed=9,
              entropy_budget=40.0, conf_threshold=-1.0, stable_k=3, step_cap=1000,
              sample_rule=dg.DG_SAMPLE_SEGMENTED)
    if kind == "grouped":
        kw["sample_rule"] = dg.DG_SAMPLE_GROUPED
    p = dg.Params(**kw)
    src = syn.boosted_logits(B * C, V, seed=2, device="cuda").reshape(-1)
    if kind == "unaligned":
        flat = torch.empty(src.numel() + 8, dtype=torch.bfloat16, device="cuda")
        logits = flat[1:1 + src.numel()]
        logits.copy_(src)
    else:
        logits = src
    E = syn.embedding(V, d, seed=7, device="cuda")
    st_a = make_state(p, [dg.DG_PHASE_DENOISE] * B, temperatures=[0.8, 1.1])
    st_b = _clone(st_a)
    ws_a = torch.empty(max(16, dg.dg_workspace_bytes(p, d)), dtype=torch.uint8, device="cuda")
    ws_b = torch.empty(dg.dg_workspace_bytes_feed(p, d), dtype=torch.uint8, device="cuda")
    out_a = torch.empty((B * C, d), dtype=torch.float32, device="cuda")
    out_b = torch.empty((B * C, d), dtype=torch.float32, device="cuda")
    dg.dg_denoise_step(p, logits, st_a, ws_a)
    dg.dg_selfcond_embed(p, logits, st_a, E, out_a, ws_a)
    dg.dg_denoise_step_feed(p, logits, st_b, E, out_b, ws_b)
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b)  # the same two calls
    sa, sb = st_a.snapshot(), st_b.snapshot()
    for k in FIELDS:
        assert np.array_equal(np.asarray(sa[k]), np.asarray(sb[k]), equal_nan=True), k


@pytest.mark.parametrize("B,C,V,d,cap,scale",
                         [(2, 256, 8192, 256, 30.0, 16.0), (3, 128, 4096, 128, 15.0, 0.0),
                          (2, 64, 2048, 64, 50.0, 8.0)],
                         ids=["B2V8192c30", "B3V4096c15", "B2V2048c50"])
def test_feed_softcap_matches_the_two_calls_and_the_oracle(B, C, V, d, cap, scale):
    # the vocabulary pass writes 2^(c_cap tanh(z / c_cap) c - R); the first
    # step has no previous maximum (every row takes the separate pass), the
    # later ones keep the operand
    p = dg.Params(batch=B, canvas_len=C, vocab=V, logits_dtype=dg.DG_BF16, seed=77,
                  entropy_budget=40.0, conf_threshold=-1.0, stable_k=3, step_cap=1000,
                  sample_rule=dg.DG_SAMPLE_SEGMENTED, softcap=cap, embed_scale=scale)
    temps = list(np.linspace(0.6, 1.3, B))
    logits = syn.boosted_logits(B * C, V, seed=V + 5, device="cuda", boost_hi=24.0).reshape(-1)
    E = syn.embedding(V, d, seed=d + 1, device="cuda")
    _steps(p, [dg.DG_PHASE_DENOISE] * B, logits, E, temps, n_steps=3, sample_rows=48)


def test_feed_at_eight_canvases_full_vocabulary_softcap():
    B, C, V, d = 8, 256, 262144, 2816
    p = dg.Params(batch=B, canvas_len=C, vocab=V, logits_dtype=dg.DG_BF16, seed=0xD1FF000C,
                  entropy_budget=96.0, conf_threshold=0.3, stable_k=3, step_cap=32,
                  sample_rule=dg.DG_SAMPLE_SEGMENTED, softcap=30.0, embed_scale=53.066)
    logits = syn.boosted_logits(B * C, V, seed=15, device="cuda").reshape(-1)
    E = syn.embedding(V, d, seed=16, device="cuda")
    _steps(p, [dg.DG_PHASE_DENOISE] * B, logits, E, [0.8] * B, n_steps=2, sample_rows=16)


def test_feed_at_one_canvas_full_vocabulary():
    # one wave of 143 GEMM CTAs (13 vocabulary splits), the operand from the
    # vocabulary pass after the first step
    B, C, V, d = 1, 256, 262144, 2816
    p = dg.Params(batch=B, canvas_len=C, vocab=V, logits_dtype=dg.DG_BF16, seed=0xD1FF000D,
                  entropy_budget=96.0, conf_threshold=0.3, stable_k=3, step_cap=32,
                  sample_rule=dg.DG_SAMPLE_SEGMENTED)
    logits = syn.boosted_logits(B * C, V, seed=17, device="cuda").reshape(-1)
    E = syn.embedding(V, d, seed=18, device="cuda")
    _steps(p, [dg.DG_PHASE_DENOISE] * B, logits, E, [0.8] * B, n_steps=2, sample_rows=16)


def test_feed_at_eight_canvases_full_vocabulary():
    B, C, V, d = 8, 256, 262144, 2816
    p = dg.Params(batch=B, canvas_len=C, vocab=V, logits_dtype=dg.DG_BF16, seed=0xD1FF000A,
                  entropy_budget=96.0, conf_threshold=0.3, stable_k=3, step_cap=32,
                  sample_rule=dg.DG_SAMPLE_SEGMENTED)
    logits = syn.boosted_logits(B * C, V, seed=11, device="cuda").reshape(-1)
    E = syn.embedding(V, d, seed=12, device="cuda")
    _steps(p, [dg.DG_PHASE_DENOISE] * B, logits, E, [0.8] * B, n_steps=2, sample_rows=16)


def test_feed_at_128_canvases_full_vocabulary():
    # the benchmark's default workload: 11 vocabulary splits, a 17 GB operand
    B, C, V, d = 128, 256, 262144, 2816
    p = dg.Params(batch=B, canvas_len=C, vocab=V, logits_dtype=dg.DG_BF16, seed=0xD1FF000B,
                  entropy_budget=128.0, conf_threshold=0.3, stable_k=3, step_cap=32,
                  sample_rule=dg.DG_SAMPLE_SEGMENTED)
    logits = syn.boosted_logits(B * C, V, seed=13, device="cuda").reshape(-1)
    E = syn.embedding(V, d, seed=14, device="cuda")
    _steps(p, [dg.DG_PHASE_DENOISE] * B, logits, E, [0.8] * B, n_steps=2, sample_rows=24)
