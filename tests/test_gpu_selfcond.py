"""GPU parity of dg_selfcond_embed (the tcgen05 p.E contraction) against the
fp64 oracle: ragged M / N / K tiles, split-K and single-pass plans, both
logit dtypes, fp32 and bf16 outputs, padded E rows, the three ways the A
operand arrives (bf16 logits by TMA with the rebuild in the GEMM, p
materialised first for fp32 logits and strides off 16 bytes, and producer
loads for bf16 rows on a base off a 16-byte boundary), rows that do not feed
the next step, and the one-hot case that must return embedding rows exactly."""

import numpy as np
import pytest
import torch

import denoise_step_sampler_gb300 as dg
from denoise_step_sampler_gb300 import synthetic as syn

from _gpu_common import make_state, oracle_selfcond_rows, selfcond_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from denoise_step_sampler_gb300 import build
    build.build()
    dg.lib()


def _run(p, st, logits, E, out_dtype=torch.float32):
    d = E.shape[1]
    ws = torch.empty(max(16, dg.dg_workspace_bytes(p, d)), dtype=torch.uint8, device="cuda")
    dg.dg_denoise_step(p, logits, st, ws)
    out = torch.full((p.batch * p.canvas_len, d), float("nan"), dtype=out_dtype, device="cuda")
    dg.dg_selfcond_embed(p, logits, st, E, out, ws)
    torch.cuda.synchronize()
    return out


CASES = [
    # (B, C, V, dtype, ld, d, ldE, out)
    (2, 64, 64, dg.DG_F32, None, 16, 16, torch.float32),
    (2, 128, 1000, dg.DG_BF16, None, 64, 64, torch.float32),
    (1, 200, 1003, dg.DG_F32, 1003, 272, 288, torch.float32),
    (3, 64, 4096, dg.DG_BF16, None, 128, 128, torch.bfloat16),
    (1, 256, 20000, dg.DG_BF16, None, 512, 512, torch.float32),
    (4, 256, 3000, dg.DG_BF16, None, 768, 768, torch.float32),
    (3, 128, 2048, dg.DG_BF16, None, 128, 128, torch.float32),   # odd row-tile count
    (5, 256, 1024, dg.DG_F32, None, 1024, 1024, torch.float32),  # fp32, many row tiles
    (2, 128, 5000, dg.DG_BF16, 5008, 256, 256, torch.float32),   # bf16 by TMA, ld > V, ragged k
    (2, 96, 3001, dg.DG_BF16, 3003, 208, 208, torch.bfloat16),   # bf16 rows not 16-byte aligned
    (4, 256, 4096, dg.DG_BF16, None, 400, 400, torch.float32),   # several row tiles, 3 E boxes in the last column tile
    (3, 1, 300, dg.DG_BF16, None, 16, 16, torch.float32),        # one position per canvas
    (1, 16, 2, dg.DG_F32, None, 32, 32, torch.float32),          # smallest vocabulary
]


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}C{c[1]}V{c[2]}d{c[5]}" for c in CASES])
def test_selfcond_matches_oracle(case):
    B, C, V, dt, ld, d, ldE, odt = case
    p = dg.Params(batch=B, canvas_len=C, vocab=V, logits_dtype=dt, logits_ld=ld, seed=21,
                  entropy_budget=50.0, conf_threshold=-1.0, stable_k=3, step_cap=1000)
    temps = np.linspace(0.7, 1.3, B)
    st = make_state(p, [dg.DG_PHASE_DENOISE] * B, temperatures=temps)
    tdt = torch.bfloat16 if dt == dg.DG_BF16 else torch.float32
    logits = syn.boosted_logits(B * C, V, seed=V + d, dtype=tdt, device="cuda", ld=ld).reshape(-1)
    Efull = syn.embedding(V, ldE, seed=d, device="cuda")
    E = Efull[:, :d]
    out = _run(p, st, logits, E, odt)
    got = out.float().cpu().numpy()
    Eh = E.float().cpu().numpy().astype(np.float64)
    ldv = V if ld is None else ld
    zh = logits.view(B, C, ldv)[:, :, :V].float().cpu().numpy()
    for r in range(B):
        ref = oracle_selfcond_rows(zh[r], float(np.float32(temps[r])), Eh)
        selfcond_check(got[r * C:(r + 1) * C], ref)


def test_selfcond_one_hot_returns_embedding_rows_exactly():
    B, C, V, d = 1, 128, 777, 64
    p = dg.Params(batch=B, canvas_len=C, vocab=V, logits_dtype=dg.DG_F32, seed=2,
                  entropy_budget=50.0, conf_threshold=-1.0, step_cap=100)
    st = make_state(p, [dg.DG_PHASE_DENOISE], temperatures=[0.8])
    tok = torch.randint(0, V, (C,), device="cuda")
    logits = torch.full((C, V), float("-inf"), device="cuda")
    logits[torch.arange(C, device="cuda"), tok] = torch.randn(C, device="cuda")
    E = syn.embedding(V, d, seed=5, device="cuda")
    out = _run(p, st, logits.reshape(-1), E)
    assert torch.equal(out, E[tok].float())


def test_rows_that_do_not_feed_are_zero():
    B, C, V, d = 4, 64, 500, 32
    p = dg.Params(batch=B, canvas_len=C, vocab=V, logits_dtype=dg.DG_BF16, seed=4,
                  entropy_budget=50.0, conf_threshold=-1.0, stable_k=1, step_cap=2)
    st = make_state(p, [dg.DG_PHASE_DENOISE, dg.DG_PHASE_PREFILL, dg.DG_PHASE_IDLE,
                        dg.DG_PHASE_DENOISE], temperatures=[1, 1, 1, 1])
    st.step[3] = 1  # reaches the cap: converges, does not feed
    logits = syn.boosted_logits(B * C, V, seed=1, device="cuda").reshape(-1)
    E = syn.embedding(V, d, seed=6, device="cuda")
    out = _run(p, st, logits, E).view(B, C, d)
    assert torch.count_nonzero(out[1:]).item() == 0
    assert torch.count_nonzero(out[0]).item() > 0
    snap = st.snapshot()
    assert snap["sc_valid"].tolist() == [1, 0, 0, 0]


@pytest.mark.parametrize("split", [False, True], ids=["one-pass", "split-K"])
def test_selfcond_bf16_rows_off_a_16_byte_boundary(split):
    # a 16-byte-multiple stride on a base address 2 bytes past a 16-byte
    # boundary: the one input the GEMM's producers still load themselves
    # (fp32 logits and strides off 16 bytes materialise p first)
    B, C = 2, 128
    V, d, ld = (20000, 256, 20008) if split else (1000, 64, 1008)
    p = dg.Params(batch=B, canvas_len=C, vocab=V, logits_dtype=dg.DG_BF16, logits_ld=ld, seed=21,
                  entropy_budget=50.0, conf_threshold=-1.0, stable_k=3, step_cap=1000)
    temps = [0.75, 1.2]
    st = make_state(p, [dg.DG_PHASE_DENOISE] * B, temperatures=temps)
    src = syn.boosted_logits(B * C, V, seed=5, dtype=torch.bfloat16, device="cuda", ld=ld).reshape(-1)
    flat = torch.empty(src.numel() + 8, dtype=torch.bfloat16, device="cuda")
    logits = flat[1:1 + src.numel()]
    logits.copy_(src)
    assert logits.data_ptr() % 16 == 2
    E = syn.embedding(V, d, seed=7, device="cuda")
    out = _run(p, st, logits, E)
    assert int(st.device_status.item()) == 0
    got = out.cpu().numpy()
    Eh = E.float().cpu().numpy().astype(np.float64)
    zh = src.view(B, C, ld)[:, :, :V].float().cpu().numpy()
    for r in range(B):
        ref = oracle_selfcond_rows(zh[r], float(np.float32(temps[r])), Eh)
        selfcond_check(got[r * C:(r + 1) * C], ref)


@pytest.mark.parametrize("V,d", [(500, 32), (60000, 256)], ids=["one-pass", "split-K"])
def test_fp32_rows_that_do_not_feed_are_zero_whatever_the_workspace_holds(V, d):
    # fp32 logits take the materialised-p route, which never writes the p of
    # rows that do not feed; the workspace is filled with NaN bytes first
    B, C = 4, 64
    p = dg.Params(batch=B, canvas_len=C, vocab=V, logits_dtype=dg.DG_F32, seed=4,
                  entropy_budget=50.0, conf_threshold=-1.0, stable_k=1, step_cap=2)
    st = make_state(p, [dg.DG_PHASE_DENOISE, dg.DG_PHASE_PREFILL, dg.DG_PHASE_IDLE,
                        dg.DG_PHASE_DENOISE], temperatures=[0.9, 1, 1, 1])
    st.step[3] = 1  # reaches the cap: converges, does not feed
    logits = syn.boosted_logits(B * C, V, seed=1, dtype=torch.float32, device="cuda").reshape(-1)
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
    zh = logits.view(B, C, V)[0].cpu().numpy().astype(np.float64)
    ref = oracle_selfcond_rows(zh, float(np.float32(0.9)), E.float().cpu().numpy().astype(np.float64))
    selfcond_check(got[0].cpu().numpy(), ref)
