"""GPU parity at the benchmark workloads' full sizes, on sampled outputs the
fp64 oracle can compute one by one, in the launch configuration bench.py
times:

* 1 canvas x 256, V = 50257, fp32 logits (unaligned rows), d = 512: every
  position and every self-conditioning row;
* 8 canvases x 256, V = 262144, bf16, d = 2816, both sampling rules: one
  full canvas (acceptance and re-noise included), 64 random positions, two
  self-conditioning rows from every 256-row tile of the GEMM;
* the same with the logit softcap (c = 30) and the sqrt(d) embedding scale,
  at 8 and at 128 canvases;
* 1, 2, 4, 16, 32 and 64 canvases (the sweep sizes) and 128 canvases x 256 (17 GB of
  logits, both sampling rules): one full canvas, 64 random positions, two
  self-conditioning rows from every 256-row tile of the GEMM;
* the mixed-phase loop (32 requests: 8 prefill, 20 denoise, 4 commit) at
  V = 262144: the first two steps compared for three requests from the GPU's
  prior state, then run until every request has committed, checking the phase
  machine's counters on every step;
* the one-canvas loop of 24 denoise steps + commit captured in a CUDA graph:
  replay equals eager execution bit for bit, and its first and last steps
  match the oracle."""

import numpy as np
import pytest
import torch

import denoise_step_sampler_gb300 as dg
from denoise_step_sampler_gb300 import synthetic as syn

from _gpu_common import (ENT_TOL, S_RTOL, compare_step, make_state, oracle_params, oracle_state, pmap,
                         run_oracle_step, selfcond_check)
from oracle import sampler as osam
from oracle import selfcond as osc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from denoise_step_sampler_gb300 import build
    build.build()
    dg.lib()


def _positions_match(p, snap, host_logits, T, rid, rstep, idx):
    """Per-position outputs of sampled positions (flat indices) vs the oracle."""
    C = p.canvas_len
    jobs = [(host_logits[q].astype(np.float64), float(T[q // C]), p.seed, rid[q // C],
             rstep[q // C], q % C, p.softcap, p.sample_rule) for q in idx]
    res = pmap(osam._vocab_job, jobs)
    n_flag = 0
    for q, r in zip(idx, res):
        assert abs(snap["entropy"][q] - r.entropy) <= ENT_TOL, q
        assert snap["argmax"][q] == r.argmax, q
        if r.gap >= osam.NEAR_TIE:
            assert snap["cand"][q] == r.cand, q
        else:
            n_flag += 1
        assert abs(snap["m"][q] - r.m) <= 1e-4 and abs(snap["s"][q] / r.s - 1) <= S_RTOL, q
    return n_flag


def _selfcond_rows(out, host_logits, rows, T, E_host, C):
    for q in rows:
        ref = osc.selfcond_rows(host_logits[q:q + 1].astype(np.float64), float(T[q // C]), E_host)
        selfcond_check(out[q:q + 1], ref)


def _one_step(B, C, V, dt, T, budget, d, boost, seed, n_rand, n_sc, full_canvas=True,
              softcap=0.0, embed_scale=0.0, sample_rule=dg.DG_SAMPLE_GROUPED):
    """One step at full size: one whole canvas and n_rand sampled positions
    against the oracle, and n_sc self-conditioning rows from every 256-row
    tile of the GEMM (so every row tile, and both row halves of its MMAs,
    is checked).  Returns the compare_step counts of the whole canvas."""
    tdt = torch.bfloat16 if dt == dg.DG_BF16 else torch.float32
    p = dg.Params(batch=B, canvas_len=C, vocab=V, logits_dtype=dt, seed=seed,
                  entropy_budget=budget, conf_threshold=0.3, stable_k=3, step_cap=32,
                  softcap=softcap, embed_scale=embed_scale, sample_rule=sample_rule)
    st = make_state(p, [dg.DG_PHASE_DENOISE] * B, request_ids=np.arange(B) * 3 + 1,
                    temperatures=[T] * B, rng_step=np.arange(B))
    logits = syn.boosted_logits(B * C, V, seed=seed, dtype=tdt, device="cuda",
                                boost_hi=boost).reshape(-1)
    E = syn.embedding(V, d, seed=seed + 1, device="cuda")
    ws = torch.empty(max(16, dg.dg_workspace_bytes(p, d)), dtype=torch.uint8, device="cuda")
    before = st.snapshot()
    out = torch.empty((B * C, d), dtype=torch.float32, device="cuda")
    dg.dg_denoise_step(p, logits, st, ws)
    dg.dg_selfcond_embed(p, logits, st, E, out, ws)
    torch.cuda.synchronize()
    after = st.snapshot()
    assert after["device_status"][0] == 0
    rng = np.random.default_rng(seed)
    L2 = logits.view(B * C, V)
    counts = None
    if full_canvas:
        r = int(rng.integers(B))
        rows_host = {rr: (L2[rr * C:(rr + 1) * C].float().cpu().numpy() if rr == r else None)
                     for rr in range(B)}
        ost, flags = run_oracle_step(p, before, rows_host, rows=[r])
        counts = compare_step(p, before, after, ost, flags, rows=[r])
    idx = sorted(set(rng.integers(B * C, size=n_rand).tolist()))
    host = {q: L2[q].float().cpu().numpy() for q in idx}
    n_flag = _positions_match(p, after, host, after["temperature"], after["request_id"],
                              before["rng_step"], idx)
    assert n_flag <= max(2, len(idx) // 20)
    n_pos = B * C
    sc_rows = sorted({int(t0 + x) for t0 in range(0, n_pos, 256)
                      for x in rng.integers(min(256, n_pos - t0), size=n_sc)})
    E_host = E.float().cpu().numpy().astype(np.float64)
    got = out.cpu().numpy()
    sel = torch.tensor(sc_rows, device="cuda")
    ref = osc.selfcond_rows(L2[sel].float().cpu().numpy().astype(np.float64), float(np.float32(T)),
                            E_host, cap=float(np.float32(softcap)),
                            scale=float(np.float32(embed_scale)))
    selfcond_check(got[sc_rows], ref)
    return counts


def test_one_canvas_V50257_fp32_everything():
    B, C, V, d = 1, 256, 50257, 512
    p = dg.Params(batch=B, canvas_len=C, vocab=V, logits_dtype=dg.DG_F32, seed=0xD1FF0001,
                  entropy_budget=64.0, conf_threshold=0.3, stable_k=3, step_cap=32)
    st = make_state(p, [dg.DG_PHASE_DENOISE], request_ids=[0], temperatures=[1.0])
    logits = syn.boosted_logits(C, V, seed=p.seed, dtype=torch.float32, device="cuda",
                                boost_hi=12.0).reshape(-1)
    E = syn.embedding(V, d, seed=p.seed + 1, device="cuda")
    ws = torch.empty(max(16, dg.dg_workspace_bytes(p, d)), dtype=torch.uint8, device="cuda")
    before = st.snapshot()
    out = torch.empty((C, d), dtype=torch.float32, device="cuda")
    dg.dg_denoise_step(p, logits, st, ws)
    dg.dg_selfcond_embed(p, logits, st, E, out, ws)
    torch.cuda.synchronize()
    after = st.snapshot()
    host = logits.view(1, C, V).cpu().numpy()
    ost, flags = run_oracle_step(p, before, host)
    compare_step(p, before, after, ost, flags)
    ref = osc.selfcond(host.astype(np.float64), ost.temperature, E.float().cpu().numpy(),
                       ost.sc_valid.astype(bool))
    selfcond_check(out.cpu().numpy(), ref)


@pytest.mark.parametrize("rule", [dg.DG_SAMPLE_GROUPED, dg.DG_SAMPLE_SEGMENTED],
                         ids=["grouped", "segmented"])
def test_eight_canvases_V262144_bf16_sampled(rule):
    _one_step(8, 256, 262144, dg.DG_BF16, 0.8, 96.0, 2816, 16.0, 0xD1FF0002, 64, 2,
              sample_rule=rule)


@pytest.mark.parametrize("B,seed", [(1, 0xD1FF0011), (2, 0xD1FF0012), (4, 0xD1FF0013),
                                    (16, 0xD1FF0007), (32, 0xD1FF0006), (64, 0xD1FF0008)],
                         ids=["1", "2", "4", "16", "32", "64"])
def test_sweep_canvases_V262144_bf16_sampled(B, seed):
    # the sweep sizes: other split plans of the GEMM (on 152 SMs: 13 splits
    # at one canvas and 6 at two, one wave each, with p rebuilt in the GEMM;
    # 10 at four and 6 at 16 canvases, 3 from 32 on, on a materialised p) and
    # 8, 4 or 2 vocabulary chunks per position
    _one_step(B, 256, 262144, dg.DG_BF16, 0.8, 128.0, 2816, 16.0, seed, 64, 8 if B <= 2 else 2,
              sample_rule=dg.DG_SAMPLE_SEGMENTED)


def test_eight_canvases_softcap_and_embed_scale_sampled():
    # the softcapped path (c = 30) with the sqrt(d) embedding scale on the feed
    _one_step(8, 256, 262144, dg.DG_BF16, 0.8, 96.0, 2816, 16.0, 0xD1FF0005, 64, 2,
              softcap=30.0, embed_scale=float(np.sqrt(2816.0)))


def test_128_canvases_softcap_and_embed_scale_sampled():
    # the softcapped feed at the largest workload: a 17 GB materialised p in
    # the workspace and the GEMM's L2-fitted split count (11 on a GB300)
    _one_step(128, 256, 262144, dg.DG_BF16, 0.8, 128.0, 2816, 16.0, 0xD1FF0009, 64, 2,
              softcap=30.0, embed_scale=float(np.sqrt(2816.0)), sample_rule=dg.DG_SAMPLE_SEGMENTED)


@pytest.mark.parametrize("rule", [dg.DG_SAMPLE_SEGMENTED, dg.DG_SAMPLE_GROUPED],
                         ids=["segmented", "grouped"])
def test_128_canvases_V262144_bf16_sampled(rule):
    # the benchmark's default workload and rule, and the grouped rule
    _one_step(128, 256, 262144, dg.DG_BF16, 0.8, 128.0, 2816, 16.0, 0xD1FF0004, 64, 2,
              sample_rule=rule)


def test_mixed_phase_loop_full_vocab():
    B, C, V, d = 32, 256, 262144, 2816
    seed = 0xD1FF0003
    p = dg.Params(batch=B, canvas_len=C, vocab=V, logits_dtype=dg.DG_BF16, seed=seed,
                  entropy_budget=96.0, conf_threshold=0.3, stable_k=3, step_cap=32)
    temps = syn.temperatures(B, seed=seed, device="cpu").numpy()
    phases = [0] * 8 + [1] * 20 + [2] * 4
    prev = np.zeros((B, C), np.int64)
    for r in range(28, 32):  # commit rows emit the generator's clean argmax canvas
        prev[r] = syn.true_tokens(C, V, seed=seed, request=r).numpy()
    st = make_state(p, phases, request_ids=np.arange(B), temperatures=temps, argmax_prev=prev)
    E = syn.embedding(V, d, seed=seed + 1, device="cuda")
    ws = torch.empty(max(16, dg.dg_workspace_bytes(p, d)), dtype=torch.uint8, device="cuda")
    out = torch.empty((B * C, d), dtype=torch.float32, device="cuda")
    logits = torch.empty((B, C, V), dtype=torch.bfloat16, device="cuda")
    committed = np.zeros(B, bool)
    for s in range(40):
        for r in range(B):
            syn.loop_logits(C, V, seed=seed, request=r, step=s, out=logits[r], device="cuda")
        before = st.snapshot()
        committed |= before["phase"] == dg.DG_PHASE_COMMIT
        if committed.all():
            break
        dg.dg_denoise_step(p, logits.view(-1), st, ws)
        dg.dg_selfcond_embed(p, logits.view(-1), st, E, out, ws)
        torch.cuda.synchronize()
        after = st.snapshot()
        assert after["device_status"][0] == 0
        # phase-machine counters on every row, every step
        for r in range(B):
            ph = before["phase"][r]
            assert after["rng_step"][r] == before["rng_step"][r] + 1
            if ph == dg.DG_PHASE_COMMIT:
                assert after["num_sampled"][r] == C and after["phase"][r] == dg.DG_PHASE_DENOISE
                assert np.array_equal(after["emitted"][r * C:(r + 1) * C],
                                      before["argmax_prev"][r * C:(r + 1) * C])
            elif ph == dg.DG_PHASE_DENOISE:
                assert after["num_sampled"][r] == 0 and after["num_rejected"][r] == C
                assert after["step"][r] == before["step"][r] + 1
            else:
                assert after["phase"][r] == dg.DG_PHASE_DENOISE and after["step"][r] == 0
        # every step: three denoise requests in full, plus every prefill /
        # commit row
        sampled = [8, 19, 27]
        rows = sampled + [r for r in range(B)
                          if before["phase"][r] in (dg.DG_PHASE_PREFILL, dg.DG_PHASE_COMMIT)]
        host = {r: logits[r].float().cpu().numpy() for r in sampled}
        ost, flags = run_oracle_step(p, before, host, rows=sampled)
        compare_step(p, before, after, ost, flags, rows=rows)
    assert committed.all()


def test_one_canvas_loop_cuda_graph_equals_eager():
    C, V, d, steps = 256, 262144, 2816, 24
    seed = 0xD1FF0005
    p = dg.Params(batch=1, canvas_len=C, vocab=V, logits_dtype=dg.DG_BF16, seed=seed,
                  entropy_budget=96.0, conf_threshold=0.3, stable_k=3, step_cap=steps)
    T = float(syn.temperatures(1, seed=seed, device="cpu")[0])
    bufs = [syn.loop_logits(C, V, seed=seed, request=0, step=s, device="cuda").reshape(-1)
            for s in range(steps + 1)]
    E = syn.embedding(V, d, seed=seed + 1, device="cuda")
    ws = torch.empty(max(16, dg.dg_workspace_bytes(p, d)), dtype=torch.uint8, device="cuda")

    def fresh():
        return make_state(p, [dg.DG_PHASE_PREFILL], request_ids=[0], temperatures=[T])

    def run(st, out, stream):
        for s in range(steps + 1):
            dg.dg_denoise_step(p, bufs[s], st, ws, stream=stream)
            dg.dg_selfcond_embed(p, bufs[s], st, E, out, ws, stream=stream)

    # eager
    st_e = fresh()
    out_e = torch.empty((C, d), dtype=torch.float32, device="cuda")
    dg.dg_init_canvas(p, st_e, torch.ones(1, dtype=torch.uint8, device="cuda"))
    snaps = [st_e.snapshot()]
    for s in range(steps + 1):
        dg.dg_denoise_step(p, bufs[s], st_e, ws)
        dg.dg_selfcond_embed(p, bufs[s], st_e, E, out_e, ws)
        torch.cuda.synchronize()
        snaps.append(st_e.snapshot())
    assert any(sn["num_sampled"][0] == C for sn in snaps[1:])  # the block was committed
    # graph
    st_g = fresh()
    out_g = torch.empty((C, d), dtype=torch.float32, device="cuda")
    dg.dg_init_canvas(p, st_g, torch.ones(1, dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    s_cap = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s_cap):
        run(st_g, out_g, s_cap)
    g.replay()
    torch.cuda.synchronize()
    a = st_g.snapshot()
    for k in ("canvas", "cand", "argmax", "argmax_prev", "accept", "emitted", "phase", "step",
              "stable", "rng_step", "num_sampled", "entropy", "m", "s", "mean_entropy"):
        assert np.array_equal(a[k], snaps[-1][k], equal_nan=True) if a[k].dtype.kind == "f" \
            else np.array_equal(a[k], snaps[-1][k]), k
    assert torch.equal(out_g, out_e)
    # the first and the last denoise steps against the oracle
    den = [s for s in range(steps + 1) if snaps[s]["phase"][0] == dg.DG_PHASE_DENOISE]
    for s in (den[0], den[-1]):
        host = {0: bufs[s].view(C, V).float().cpu().numpy()}
        ost, flags = run_oracle_step(p, snaps[s], host)
        compare_step(p, snaps[s], snaps[s + 1], ost, flags)


def test_zz_report_prefix_error():
    """Prints the largest prefix errors of the sorted entropies met by the
    comparisons above (run with -s to see them)."""
    from _gpu_common import PREFIX_STATS
    print("largest |GPU - oracle| entropy prefix: at the acceptance cut %.3g, any prefix %.3g"
          % (PREFIX_STATS["cut"], PREFIX_STATS["all"]))
