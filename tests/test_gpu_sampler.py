"""GPU parity of dg_denoise_step / dg_init_canvas / dg_commit against the fp64
oracle on seeded synthetic inputs: several vocabulary sizes and tile counts,
ragged tails, unaligned rows, both logit dtypes, mixed phases, non-finite
logits, and multi-step loops compared step by step from the GPU's state."""

import numpy as np
import pytest
import torch

import denoise_step_sampler_gb300 as dg
from denoise_step_sampler_gb300 import synthetic as syn

from _gpu_common import compare_step, denoise_and_compare, make_state, run_oracle_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from denoise_step_sampler_gb300 import build
    build.build()
    dg.lib()


def _logits(B, C, V, dtype, seed, ld=None, boost_hi=12.0):
    t = torch.bfloat16 if dtype == dg.DG_BF16 else torch.float32
    return syn.boosted_logits(B * C, V, seed=seed, dtype=t, device="cuda", boost_hi=boost_hi,
                              ld=ld).reshape(-1)


CASES = [
    # (B, C, V, dtype, ld, budget, T)
    (2, 8, 8, dg.DG_F32, None, 1.0, [1.0, 0.5]),
    (2, 8, 64, dg.DG_BF16, None, 2.0, [0.8, 1.3]),
    (3, 8, 1000, dg.DG_F32, 1003, 3.0, [1.0, 0.7, 1.9]),       # unaligned fp32 rows
    (2, 256, 1000, dg.DG_BF16, None, 96.0, [0.8, 1.0]),
    (1, 256, 50257, dg.DG_F32, None, 64.0, [1.0]),              # ragged last group, unaligned
    (2, 64, 50257, dg.DG_BF16, 50264, 30.0, [0.9, 1.1]),        # aligned bf16 rows, ragged V
    (2, 32, 4099, dg.DG_BF16, 4099, 20.0, [1.2, 0.6]),          # 2-byte aligned bf16 rows
    (1, 100, 2048, dg.DG_F32, None, 5.0, [1.0]),                # C not a power of two
    (1, 8, 8192, dg.DG_BF16, None, 2.0, [0.9]),                 # one bf16 round per chunk
    (1, 8, 16384, dg.DG_BF16, None, 2.0, [0.9]),                # two rounds (fewer than the ring)
    (1, 16, 2, dg.DG_F32, None, 1.0, [1.0]),                    # smallest vocabulary
    (3, 1, 300, dg.DG_BF16, None, 0.5, [0.8, 1.0, 1.2]),        # one position per canvas
    (1, 1024, 4096, dg.DG_BF16, None, 300.0, [1.0]),            # largest canvas
]


RULES = [dg.DG_SAMPLE_GROUPED, dg.DG_SAMPLE_SEGMENTED]


@pytest.mark.parametrize("rule", RULES, ids=["grouped", "segmented"])
@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}C{c[1]}V{c[2]}dt{c[3]}ld{c[4]}" for c in CASES])
def test_denoise_step_matches_oracle(case, rule):
    B, C, V, dt, ld, budget, T = case
    p = dg.Params(batch=B, canvas_len=C, vocab=V, logits_dtype=dt, logits_ld=ld, seed=0xD1FF0001,
                  entropy_budget=budget, conf_threshold=0.3, stable_k=3, step_cap=32,
                  sample_rule=rule)
    st = make_state(p, [dg.DG_PHASE_DENOISE] * B, request_ids=np.arange(B) + 17, temperatures=T,
                    rng_step=np.arange(B) * 5)
    logits = _logits(B, C, V, dt, seed=B * 1000 + V, ld=ld)
    _, after, ost, flags, n = denoise_and_compare(p, st, logits)
    assert after["device_status"][0] == 0
    total = B * C
    assert n["cand"] <= max(2, total // 50), n


def test_mixed_phases_in_one_batch():
    B, C, V = 6, 64, 3000
    p = dg.Params(batch=B, canvas_len=C, vocab=V, logits_dtype=dg.DG_BF16, seed=7,
                  entropy_budget=20.0, conf_threshold=0.3, stable_k=1, step_cap=4)
    phases = [dg.DG_PHASE_PREFILL, dg.DG_PHASE_DENOISE, dg.DG_PHASE_COMMIT, dg.DG_PHASE_IDLE,
              dg.DG_PHASE_DENOISE, dg.DG_PHASE_COMMIT]
    prev = np.random.default_rng(1).integers(0, V, (B, C))
    st = make_state(p, phases, request_ids=[5, 6, 7, 8, 9, 10],
                    temperatures=[1.0, 0.9, 1.0, 1.0, 1.1, 1.0], rng_step=[0, 3, 9, 2, 1, 4],
                    argmax_prev=prev)
    st.step[4] = 3  # this row reaches the cap in this step
    st.canvas.copy_(torch.arange(B * C, dtype=torch.int32, device="cuda"))
    logits = _logits(B, C, V, dg.DG_BF16, seed=99)
    _, after, ost, flags, _ = denoise_and_compare(p, st, logits)
    assert after["phase"].tolist() == [1, 1, 1, 3, 2, 1]
    assert after["num_sampled"].tolist() == [0, 0, C, 0, 0, C]


@pytest.mark.parametrize("rule", RULES, ids=["grouped", "segmented"])
def test_nonfinite_and_masked_rows(rule):
    B, C, V = 3, 16, 700
    p = dg.Params(batch=B, canvas_len=C, vocab=V, logits_dtype=dg.DG_F32, seed=3,
                  entropy_budget=10.0, conf_threshold=0.3, stable_k=1, step_cap=8,
                  sample_rule=rule)
    st = make_state(p, [1, 1, 1], temperatures=[1.0, 1.0, 0.0])
    logits = _logits(B, C, V, dg.DG_F32, seed=5).view(B, C, V)
    logits[0, 1, 10] = float("nan")
    logits[0, 2, 20] = float("inf")
    logits[0, 3, :] = float("-inf")
    logits[0, 4, ::3] = float("-inf")        # masked tokens, still valid
    logits[1, :, 100:600] = float("-inf")    # heavy masking in every chunk
    _, after, ost, flags, _ = denoise_and_compare(p, st, logits.reshape(-1))
    ent = after["entropy"].reshape(B, C)
    assert np.isnan(ent[0, 1:4]).all() and np.isfinite(ent[0, 4]) and np.isfinite(ent[1]).all()
    assert np.isnan(ent[2]).all()
    acc = after["accept"].reshape(B, C)
    assert acc[0, 1:4].sum() == 0 and acc[2].sum() == 0
    status = int(after["device_status"][0])
    assert status & dg.DG_DEV_NONFINITE_LOGITS and status & dg.DG_DEV_BAD_TEMPERATURE
    cand = after["cand"].reshape(B, C)
    assert np.all((cand[1] < 100) | (cand[1] >= 600))


def test_init_and_commit_entry_points():
    B, C, V = 4, 32, 5000
    p = dg.Params(batch=B, canvas_len=C, vocab=V, seed=11)
    prev = np.random.default_rng(2).integers(0, V, (B, C))
    st = make_state(p, [dg.DG_PHASE_IDLE, dg.DG_PHASE_COMMIT, dg.DG_PHASE_DENOISE, dg.DG_PHASE_IDLE],
                    request_ids=[1, 2, 3, 4], rng_step=[0, 1, 2, 3], argmax_prev=prev)
    from oracle import sampler as osam
    from _gpu_common import oracle_params, oracle_state
    before = st.snapshot()
    mask = torch.tensor([1, 0, 1, 0], dtype=torch.uint8, device="cuda")
    dg.dg_init_canvas(p, st, mask)
    torch.cuda.synchronize()
    after = st.snapshot()
    ost = osam.init_rows(oracle_params(p), oracle_state(before, p), [1, 0, 1, 0])
    assert np.array_equal(after["canvas"].reshape(B, C), ost.canvas)
    assert np.array_equal(after["rng_step"], ost.rng_step)
    assert after["phase"].tolist() == [1, 2, 1, 3]
    before = after
    mask = torch.tensor([0, 1, 0, 1], dtype=torch.uint8, device="cuda")
    dg.dg_commit(p, st, mask)
    torch.cuda.synchronize()
    after = st.snapshot()
    ost = osam.commit_rows(oracle_params(p), oracle_state(before, p), [0, 1, 0, 1])
    assert np.array_equal(after["emitted"].reshape(B, C), ost.emitted)
    assert np.array_equal(after["canvas"].reshape(B, C), ost.canvas)
    assert after["num_sampled"].tolist() == [0, C, 0, C]
    assert after["phase"].tolist() == [1, 1, 1, 1]


def test_bad_token_and_phase_set_status_without_trapping():
    B, C, V = 2, 8, 50
    p = dg.Params(batch=B, canvas_len=C, vocab=V, seed=1)
    st = make_state(p, [dg.DG_PHASE_COMMIT, 7], argmax_prev=np.full((B, C), 9999))
    ws = torch.empty(dg.dg_workspace_bytes(p, 0), dtype=torch.uint8, device="cuda")
    logits = torch.zeros(B * C * V, dtype=torch.bfloat16, device="cuda")
    dg.dg_denoise_step(p, logits, st, ws)
    torch.cuda.synchronize()
    snap = st.snapshot()
    assert snap["device_status"][0] & dg.DG_DEV_BAD_TOKEN
    assert snap["device_status"][0] & dg.DG_DEV_BAD_PHASE
    assert np.all(snap["emitted"][:C] == 0)


@pytest.mark.parametrize("rule", RULES, ids=["grouped", "segmented"])
def test_multistep_loop_until_every_request_commits(rule):
    """A mixed-phase loop (prefill, denoise, commit requests) with rising
    confidence; every step is compared from the GPU's prior state."""
    B, C, V = 6, 64, 1000
    p = dg.Params(batch=B, canvas_len=C, vocab=V, logits_dtype=dg.DG_BF16, seed=0xD1FF0003,
                  entropy_budget=96.0, conf_threshold=0.3, stable_k=3, step_cap=12,
                  sample_rule=rule)
    temps = syn.temperatures(B, seed=3, device="cpu").numpy()
    phases = [0, 0, 1, 1, 1, 2]
    st = make_state(p, phases, request_ids=np.arange(B), temperatures=temps)
    committed = np.zeros(B, bool)
    logits = torch.empty(B, C, V, dtype=torch.bfloat16, device="cuda")
    for s in range(40):
        for r in range(B):
            syn.loop_logits(C, V, seed=p.seed, request=r, step=s, out=logits[r], device="cuda")
        committed |= st.snapshot()["phase"] == dg.DG_PHASE_COMMIT
        if committed.all():
            break
        denoise_and_compare(p, st, logits.reshape(-1))
    assert committed.all()


@pytest.mark.gpu
@pytest.mark.parametrize("rule", RULES, ids=["grouped", "segmented"])
@pytest.mark.parametrize("T", [1.0, 0.5])
def test_large_logit_jumps_move_the_sum_reference(T, rule):
    """Spikes far above the running maximum (more than 2^32 in base 2) at early,
    middle and late vocabulary indices force the vocabulary pass to move the
    reference of its softmax sums mid-chunk; the results must still match."""
    B, C, V = 1, 16, 262144
    p = dg.Params(batch=B, canvas_len=C, vocab=V, logits_dtype=dg.DG_BF16, seed=99,
                  entropy_budget=8.0, conf_threshold=0.3, stable_k=3, step_cap=32,
                  sample_rule=rule)
    logits = _logits(B, C, V, dg.DG_BF16, seed=7).view(B, C, V)
    g = torch.Generator(device="cpu").manual_seed(5)
    for i in range(C):
        n = 1 + i % 3
        idx = torch.randint(0, V, (n,), generator=g).sort().values
        for k, v in enumerate(idx.tolist()):
            logits[0, i, v] = 20.0 + 30.0 * k + float(i)   # rising spikes
    st = make_state(p, [dg.DG_PHASE_DENOISE], request_ids=[3], temperatures=[T])
    denoise_and_compare(p, st, logits.reshape(-1))
