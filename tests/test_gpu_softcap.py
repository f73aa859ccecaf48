"""GPU parity of the logit softcap z <- c tanh(z / c) and the embedding scale
on the self-conditioning feed ("The Annotated DiffusionGemma", "Logit
Softcapping" and the model's forward pass) against the fp64 oracle: the
sampler step on bf16 and fp32 logits, aligned and unaligned rows, a mild and a
hard cap; infinite logits (capped to +-c) and NaN rows; the self-conditioning
feed through the TMA, materialised-p, split-K and single-pass plans; and the
scale alone, which must be an exact fp32 product."""

import numpy as np
import pytest
import torch

import denoise_step_sampler_gb300 as dg
from denoise_step_sampler_gb300 import synthetic as syn

from _gpu_common import denoise_and_compare, make_state, selfcond_check
from oracle import selfcond as osc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from denoise_step_sampler_gb300 import build
    build.build()
    dg.lib()


STEP_CASES = [
    # (B, C, V, dtype, ld, cap)
    (2, 128, 4096, dg.DG_BF16, None, 30.0),
    (2, 128, 4096, dg.DG_BF16, None, 3.0),
    (1, 96, 3001, dg.DG_BF16, 3003, 30.0),   # rows not 16-byte aligned, ragged tail
    (2, 64, 5000, dg.DG_F32, None, 30.0),
    (1, 200, 1003, dg.DG_F32, 1003, 2.5),    # fp32 rows not 16-byte aligned
]


@pytest.mark.parametrize("rule", [dg.DG_SAMPLE_GROUPED, dg.DG_SAMPLE_SEGMENTED],
                         ids=["grouped", "segmented"])
@pytest.mark.parametrize("case", STEP_CASES,
                         ids=[f"V{c[2]}-{'bf16' if c[3] else 'f32'}-ld{c[4]}-c{c[5]}" for c in STEP_CASES])
def test_softcap_step_matches_oracle(case, rule):
    B, C, V, dt, ld, cap = case
    p = dg.Params(batch=B, canvas_len=C, vocab=V, logits_dtype=dt, logits_ld=ld, seed=0xD1FF0011,
                  entropy_budget=0.25 * C, conf_threshold=0.3, stable_k=2, step_cap=8, softcap=cap,
                  sample_rule=rule)
    st = make_state(p, [dg.DG_PHASE_DENOISE] * B, request_ids=np.arange(B) + 5,
                    temperatures=np.linspace(0.7, 1.2, B))
    tdt = torch.bfloat16 if dt == dg.DG_BF16 else torch.float32
    logits = syn.boosted_logits(B * C, V, seed=V + int(cap), dtype=tdt, device="cuda", ld=ld,
                                boost_hi=24.0).reshape(-1)
    st2 = make_state(p, [dg.DG_PHASE_DENOISE] * B, request_ids=np.arange(B) + 5,
                     temperatures=np.linspace(0.7, 1.2, B))
    _, after, _, _, _ = denoise_and_compare(p, st, logits)
    assert after["device_status"][0] == 0
    # the allocation-free entry runs the same capped kernels
    dg.dg_denoise_step_noalloc(p, logits, st2)
    torch.cuda.synchronize()
    b = st2.snapshot()
    for k in after:
        assert np.array_equal(after[k], b[k], equal_nan=after[k].dtype.kind == "f"), k


def test_softcap_infinite_and_nan_logits():
    # +-inf logits become +-c (finite, no error bit); a NaN makes its position
    # invalid and sets the non-finite bit
    B, C, V, cap = 1, 64, 2048, 4.0
    p = dg.Params(batch=B, canvas_len=C, vocab=V, logits_dtype=dg.DG_F32, seed=3,
                  entropy_budget=16.0, conf_threshold=0.3, stable_k=2, step_cap=8, softcap=cap)
    st = make_state(p, [dg.DG_PHASE_DENOISE], temperatures=[0.9])
    z = syn.boosted_logits(C, V, seed=9, dtype=torch.float32, device="cuda").clone()
    z[0, 17] = float("inf")
    z[1, 3] = float("inf")
    z[1, 900] = float("inf")           # tie at +c: the lowest index is the argmax
    z[2, :] = float("-inf")
    z[2, 5] = float("inf")
    z[3, 100] = float("-inf")
    _, after, _, _, _ = denoise_and_compare(p, st, z.reshape(-1))
    assert after["argmax"][0] == 17 and after["argmax"][1] == 3
    assert after["device_status"][0] == 0
    st2 = make_state(p, [dg.DG_PHASE_DENOISE], temperatures=[0.9])
    z[4, 7] = float("nan")
    _, after2, _, _, _ = denoise_and_compare(p, st2, z.reshape(-1))
    assert np.isnan(after2["entropy"][4]) and after2["device_status"][0] != 0


SC_CASES = [
    # (B, C, V, dtype, ld, d, ldE, out, cap, scale)
    (2, 64, 64, dg.DG_F32, None, 16, 16, torch.float32, 3.0, 4.0),           # one split
    (2, 128, 5000, dg.DG_BF16, 5008, 256, 256, torch.float32, 30.0, 16.0),   # bf16 by TMA
    (2, 96, 3001, dg.DG_BF16, 3003, 208, 208, torch.bfloat16, 30.0, 0.0),    # producer loads
    (1, 200, 1003, dg.DG_F32, 1003, 272, 288, torch.float32, 2.5, 1.5),      # fp32 producers
    (1, 256, 20000, dg.DG_BF16, None, 512, 512, torch.float32, 30.0, 22.627417),  # split-K
]


@pytest.mark.parametrize("case", SC_CASES, ids=[f"V{c[2]}d{c[5]}c{c[8]}s{c[9]}" for c in SC_CASES])
def test_softcap_selfcond_matches_oracle(case):
    B, C, V, dt, ld, d, ldE, odt, cap, scale = case
    p = dg.Params(batch=B, canvas_len=C, vocab=V, logits_dtype=dt, logits_ld=ld, seed=21,
                  entropy_budget=50.0, conf_threshold=-1.0, stable_k=3, step_cap=1000,
                  softcap=cap, embed_scale=scale)
    temps = np.linspace(0.7, 1.3, B)
    st = make_state(p, [dg.DG_PHASE_DENOISE] * B, temperatures=temps)
    tdt = torch.bfloat16 if dt == dg.DG_BF16 else torch.float32
    logits = syn.boosted_logits(B * C, V, seed=V + d, dtype=tdt, device="cuda", ld=ld,
                                boost_hi=24.0).reshape(-1)
    E = syn.embedding(V, ldE, seed=d, device="cuda")[:, :d]
    ws = torch.empty(max(16, dg.dg_workspace_bytes(p, d)), dtype=torch.uint8, device="cuda")
    dg.dg_denoise_step(p, logits, st, ws)
    out = torch.full((B * C, d), float("nan"), dtype=odt, device="cuda")
    dg.dg_selfcond_embed(p, logits, st, E, out, ws)
    torch.cuda.synchronize()
    assert int(st.device_status.item()) == 0
    got = out.float().cpu().numpy()
    Eh = E.float().cpu().numpy().astype(np.float64)
    ldv = V if ld is None else ld
    zh = logits.view(B, C, ldv)[:, :, :V].float().cpu().numpy()
    for r in range(B):
        ref = osc.selfcond_rows(zh[r], float(np.float32(temps[r])), Eh,
                                cap=float(np.float32(cap)), scale=float(np.float32(scale)))
        selfcond_check(got[r * C:(r + 1) * C], ref)


@pytest.mark.parametrize("V,d", [(64, 16), (20000, 512)])
def test_embed_scale_is_an_exact_product(V, d):
    # same plan, same accumulation: the scaled feed is fl(scale * unscaled)
    B, C = 2, 256
    base = dict(batch=B, canvas_len=C, vocab=V, logits_dtype=dg.DG_BF16, seed=4,
                entropy_budget=50.0, conf_threshold=-1.0, step_cap=1000)
    logits = syn.boosted_logits(B * C, V, seed=11, dtype=torch.bfloat16, device="cuda").reshape(-1)
    E = syn.embedding(V, d, seed=12, device="cuda")
    outs = []
    for scale in (0.0, 2.75):
        p = dg.Params(**base, embed_scale=scale)
        st = make_state(p, [dg.DG_PHASE_DENOISE] * B, temperatures=[0.8, 1.1])
        ws = torch.empty(max(16, dg.dg_workspace_bytes(p, d)), dtype=torch.uint8, device="cuda")
        dg.dg_denoise_step(p, logits, st, ws)
        out = torch.empty((B * C, d), dtype=torch.float32, device="cuda")
        dg.dg_selfcond_embed(p, logits, st, E, out, ws)
        outs.append(out)
    torch.cuda.synchronize()
    assert torch.equal(outs[1], outs[0] * torch.tensor(2.75, dtype=torch.float32))


@pytest.mark.parametrize("splitk", [False, True], ids=["one-pass", "split-K"])
def test_softcap_rows_that_do_not_feed_are_zero_whatever_the_workspace_holds(splitk):
    # the materialised p of rows that do not feed is never written; the
    # workspace is filled with NaN bytes first, and those rows must still come
    # out as exact zeros while the feeding rows match the oracle
    B, C = 4, 64
    V, d = (60000, 256) if splitk else (500, 32)
    p = dg.Params(batch=B, canvas_len=C, vocab=V, logits_dtype=dg.DG_BF16, seed=4,
                  entropy_budget=50.0, conf_threshold=-1.0, stable_k=1, step_cap=2,
                  softcap=30.0, embed_scale=8.0)
    st = make_state(p, [dg.DG_PHASE_DENOISE, dg.DG_PHASE_PREFILL, dg.DG_PHASE_IDLE,
                        dg.DG_PHASE_DENOISE], temperatures=[0.9, 1, 1, 1])
    st.step[3] = 1  # reaches the cap: converges, does not feed
    logits = syn.boosted_logits(B * C, V, seed=1, device="cuda", boost_hi=24.0).reshape(-1)
    E = syn.embedding(V, d, seed=6, device="cuda")
    ws = torch.full((max(16, dg.dg_workspace_bytes(p, d)),), 0xFF, dtype=torch.uint8, device="cuda")
    dg.dg_denoise_step(p, logits, st, ws)
    ws.fill_(0xFF)
    out = torch.full((B * C, d), float("nan"), dtype=torch.float32, device="cuda")
    dg.dg_selfcond_embed(p, logits, st, E, out, ws)
    torch.cuda.synchronize()
    assert int(st.device_status.item()) == 0
    assert st.snapshot()["sc_valid"].tolist() == [1, 0, 0, 0]
    got = out.view(B, C, d)
    assert torch.count_nonzero(got[1:]).item() == 0
    zh = logits.view(B, C, V)[0].float().cpu().numpy().astype(np.float64)
    ref = osc.selfcond_rows(zh, float(np.float32(0.9)), E.float().cpu().numpy().astype(np.float64),
                            cap=30.0, scale=8.0)
    selfcond_check(got[0].cpu().numpy(), ref)
