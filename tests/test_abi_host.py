"""Host-side checks of the C ABI: the library builds for sm_103a, loads, exports
every entry point include/dg.h declares, and rejects invalid arguments on the
host before anything reaches a GPU.  No kernel is launched here."""

import ctypes
import os
import re
import shutil

import pytest
import torch

import denoise_step_sampler_gb300 as dg
from denoise_step_sampler_gb300 import build as dgbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dg.h")

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists(
    "/usr/local/cuda/bin/nvcc"), reason="nvcc not available")


@pytest.fixture(scope="module")
def L():
    dgbuild.build()
    return dg.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dg_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert set(names) >= {"dg_init_canvas", "dg_denoise_step", "dg_selfcond_embed", "dg_commit",
                          "dg_workspace_bytes", "dg_status_string"}
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    for code in range(5):
        assert dg.dg_status_string(code)
    assert dg.dg_status_string(99) == "unknown status"


def _params(**kw):
    base = dict(batch=2, canvas_len=256, vocab=1000, logits_dtype=dg.DG_F32, seed=1,
                entropy_budget=10.0, conf_threshold=0.3, stable_k=3, step_cap=8)
    base.update(kw)
    return dg.Params(**base)


def test_workspace_query(L):
    p = _params()
    a = dg.dg_workspace_bytes(p, 0)
    assert a > 0 and a % 256 == 0
    assert dg.dg_workspace_bytes(p, 64) >= a
    assert dg.dg_workspace_bytes(_params(batch=8), 0) >= a
    for bad in (dict(batch=0), dict(canvas_len=0), dict(canvas_len=2048), dict(vocab=1),
                dict(logits_dtype=7), dict(logits_ld=999), dict(entropy_budget=-1.0),
                dict(entropy_budget=float("inf")), dict(conf_threshold=float("nan")),
                dict(stable_k=0), dict(step_cap=0), dict(softcap=-1.0),
                dict(softcap=float("nan")), dict(softcap=float("inf")),
                dict(embed_scale=-2.0), dict(embed_scale=float("nan"))):
        assert dg.dg_workspace_bytes(_params(**bad), 0) == 0, bad
    assert L.dg_workspace_bytes(None, 0) == 0


def _fake_state():
    # distinct non-null fake device addresses; validation must fail before use
    st = dg._CState(*[0x1000 + 0x100 * i for i in range(len(dg._STATE_FIELDS))])
    return st


def test_invalid_arguments_are_rejected_on_host(L):
    p = _params().c()
    st = _fake_state()
    fake = ctypes.c_void_p(0x7000)
    ws = ctypes.c_void_p(0x9000)
    need = L.dg_workspace_bytes(ctypes.byref(p), 0)
    E = ctypes.c_void_p(0xA000)
    out = ctypes.c_void_p(0xB000)
    # null params / state / logits
    assert L.dg_denoise_step(None, fake, ctypes.byref(st), ws, need, None) == dg.DG_ERR_INVALID_ARG
    assert L.dg_denoise_step(ctypes.byref(p), fake, None, ws, need, None) == dg.DG_ERR_INVALID_ARG
    assert L.dg_denoise_step(ctypes.byref(p), None, ctypes.byref(st), ws, need, None) == dg.DG_ERR_INVALID_ARG
    # a null field in the state
    st2 = _fake_state()
    st2.entropy = None
    assert L.dg_denoise_step(ctypes.byref(p), fake, ctypes.byref(st2), ws, need, None) == dg.DG_ERR_INVALID_ARG
    # misaligned logits
    assert L.dg_denoise_step(ctypes.byref(p), ctypes.c_void_p(0x7001), ctypes.byref(st), ws, need,
                             None) == dg.DG_ERR_INVALID_ARG
    # workspace too small or missing
    assert L.dg_denoise_step(ctypes.byref(p), fake, ctypes.byref(st), ws, need - 1, None) == dg.DG_ERR_WORKSPACE
    assert L.dg_denoise_step(ctypes.byref(p), fake, ctypes.byref(st), None, need, None) == dg.DG_ERR_WORKSPACE
    # self-cond: bad widths, strides, dtypes, alignment
    for d, ldE, odt in ((0, 64, 0), (24, 24, 0), (64, 60, 0), (64, 68, 0), (64, 64, 5)):
        assert L.dg_selfcond_embed(ctypes.byref(p), fake, ctypes.byref(st), E, d, ldE, out, odt,
                                   ws, 1 << 30, None) == dg.DG_ERR_INVALID_ARG, (d, ldE, odt)
    assert L.dg_selfcond_embed(ctypes.byref(p), fake, ctypes.byref(st), ctypes.c_void_p(0xA008),
                               64, 64, out, 0, ws, 1 << 30, None) == dg.DG_ERR_INVALID_ARG
    # init / commit need a row mask
    assert L.dg_init_canvas(ctypes.byref(p), ctypes.byref(st), None, None) == dg.DG_ERR_INVALID_ARG
    assert L.dg_commit(ctypes.byref(p), ctypes.byref(st), None, None) == dg.DG_ERR_INVALID_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="only meaningful without a GPU")
def test_valid_call_without_gpu_reports_cuda_error(L):
    p = _params().c()
    st = _fake_state()
    need = L.dg_workspace_bytes(ctypes.byref(p), 0)
    rc = L.dg_denoise_step(ctypes.byref(p), ctypes.c_void_p(0x7000), ctypes.byref(st),
                           ctypes.c_void_p(0x9000), need, None)
    assert rc in (dg.DG_ERR_CUDA, dg.DG_ERR_UNSUPPORTED)


def test_binding_checks_shapes_before_calling():
    p = _params()
    with pytest.raises(ValueError):
        dg.dg_denoise_step(p, torch.zeros(10), dg.State.__new__(dg.State), torch.zeros(1))


def test_anneal_arguments_are_rejected_on_host(L):
    p = _params().c()
    step = ctypes.c_void_p(0x7100)
    temp = ctypes.c_void_p(0x7200)
    ok = (ctypes.byref(p), step, temp, 0.8, 0.4, 24, None, None)
    bad = [
        (None,) + ok[1:],
        ok[:1] + (None,) + ok[2:],
        ok[:2] + (None,) + ok[3:],
        ok[:3] + (0.0,) + ok[4:],
        ok[:3] + (float("nan"),) + ok[4:],
        ok[:4] + (-0.4,) + ok[5:],
        ok[:4] + (float("inf"),) + ok[5:],
        ok[:5] + (0,) + ok[6:],
        ok[:1] + (ctypes.c_void_p(0x7101),) + ok[2:],   # misaligned int32 array
    ]
    for args in bad:
        assert L.dg_anneal_temperature(*args) == dg.DG_ERR_INVALID_ARG, args


def test_workspace_follows_the_split_plan(L):
    # the self-conditioning workspace is the materialised p (bf16 rows of V
    # rounded up to 8, from 1,024 positions on, and for softcapped feeds)
    # followed by [splits][B*C][d] fp32 partial sums; on a 152-SM part with
    # 129 MiB of L2 (the values used when no device can be queried), the split
    # count of least cost waves * (k-blocks per split + 38) + reduction bytes /
    # 4.4 MB:
    #  - 1 and 2 canvases: 13 and 6 splits, one wave of 143 and 132 CTAs;
    #  - 8 and 64 canvases: 5 and 3 (three and fourteen waves);
    #  - 128 canvases (more than 64 row tiles of 256) split further, until one
    #    split's slice of E fits in L2: 11 splits (10 would leave 148 MB)
    V, d = 262144, 2816
    p_bytes = lambda B: (B * 256 * V * 2 + 255) // 256 * 256
    for B, splits in ((8, 5), (64, 3), (128, 11)):
        p = dg.Params(batch=B, canvas_len=256, vocab=V, logits_dtype=dg.DG_BF16)
        assert dg.dg_workspace_bytes(p, d) == p_bytes(B) + splits * B * 256 * d * 4, B
    assert V * d * 2 // 10 > 135528448 >= V * d * 2 // 11
    # one and two canvases rebuild p inside the GEMM: partial sums only
    one = dg.Params(batch=1, canvas_len=256, vocab=V, logits_dtype=dg.DG_BF16)
    assert dg.dg_workspace_bytes(one, d) == 13 * 256 * d * 4
    two = dg.Params(batch=2, canvas_len=256, vocab=V, logits_dtype=dg.DG_BF16)
    ws2 = dg.dg_workspace_bytes(two, d)
    assert ws2 == 6 * 2 * 256 * d * 4
    capped = dg.Params(batch=2, canvas_len=256, vocab=V, logits_dtype=dg.DG_BF16, softcap=30.0)
    assert dg.dg_workspace_bytes(capped, d) == p_bytes(2) + ws2


def test_fused_step_workspace_and_arguments_on_host(L):
    # dg_workspace_bytes_feed: 0 for invalid params or widths, else at least
    # the two calls' workspace (the fused call may fall back to them)
    for B in (1, 8):
        p = _params(batch=B, logits_dtype=dg.DG_BF16, vocab=4096,
                    sample_rule=dg.DG_SAMPLE_SEGMENTED)
        for d in (16, 256):
            assert dg.dg_workspace_bytes_feed(p, d) >= dg.dg_workspace_bytes(p, d) > 0
        for d in (0, 8, 24):
            assert dg.dg_workspace_bytes_feed(p, d) == 0, d
    assert dg.dg_workspace_bytes_feed(_params(batch=0), 64) == 0
    assert L.dg_workspace_bytes_feed(None, 64) == 0
    # dg_denoise_step_feed rejects bad arguments before any device work
    p = _params(logits_dtype=dg.DG_BF16, vocab=4096, sample_rule=dg.DG_SAMPLE_SEGMENTED).c()
    st = _fake_state()
    fake, E, out, ws = (ctypes.c_void_p(a) for a in (0x7000, 0xA000, 0xB000, 0x9000))
    d = 64
    need = L.dg_workspace_bytes_feed(ctypes.byref(p), d)
    ok = [ctypes.byref(p), fake, ctypes.byref(st), E, d, d, out, dg.DG_F32, ws, need, None]

    def call(**kw):
        args = list(ok)
        for k, v in kw.items():
            args[["p", "logits", "st", "E", "d", "ldE", "out", "odt", "ws", "n", "s"].index(k)] = v
        return L.dg_denoise_step_feed(*args)

    for kw in (dict(p=None), dict(logits=None), dict(st=None), dict(E=None), dict(out=None),
               dict(d=0), dict(d=24), dict(ldE=32), dict(ldE=68), dict(odt=5),
               dict(E=ctypes.c_void_p(0xA008)), dict(out=ctypes.c_void_p(0xB004)),
               dict(logits=ctypes.c_void_p(0x7001))):
        assert call(**kw) == dg.DG_ERR_INVALID_ARG, kw
    for field in ("sc_valid", "m", "s"):
        st2 = _fake_state()
        setattr(st2, field, None)
        assert call(st=ctypes.byref(st2)) == dg.DG_ERR_INVALID_ARG, field
    assert call(n=need - 1) == dg.DG_ERR_WORKSPACE
    assert call(ws=None) == dg.DG_ERR_WORKSPACE
    assert call(ws=ctypes.c_void_p(0x9008)) == dg.DG_ERR_WORKSPACE
    if not torch.cuda.is_available():
        assert call() in (dg.DG_ERR_CUDA, dg.DG_ERR_UNSUPPORTED)
