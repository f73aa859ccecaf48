"""Python binding of ``libdg`` -- the GB300 (sm_103a) denoise-step sampler and
self-conditioning feed of a uniform-state block-diffusion language model.

The functions carry the C ABI's names (``include/dg.h``) and only marshal
torch tensors into pointers, sizes and the current CUDA stream: every step of
the computation runs in the library's CUDA kernels.  There is no CPU path;
calling any entry point without the built library raises ``RuntimeError``.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

__all__ = [
    "DG_OK", "DG_ERR_INVALID_ARG", "DG_ERR_UNSUPPORTED", "DG_ERR_WORKSPACE", "DG_ERR_CUDA",
    "DG_PHASE_PREFILL", "DG_PHASE_DENOISE", "DG_PHASE_COMMIT", "DG_PHASE_IDLE",
    "DG_F32", "DG_BF16", "DG_DEV_NONFINITE_LOGITS", "DG_DEV_BAD_TEMPERATURE",
    "DG_DEV_BAD_TOKEN", "DG_DEV_WAIT_TIMEOUT", "DG_DEV_BAD_PHASE",
    "Params", "State", "DgError", "lib", "library_path",
    "dg_workspace_bytes", "dg_init_canvas", "dg_denoise_step", "dg_selfcond_embed",
    "dg_denoise_step_feed", "dg_workspace_bytes_feed",
    "dg_commit", "dg_status_string", "dg_debug_wait_record", "dg_denoise_step_noalloc",
    "DG_ERR_SCRATCH_LIMIT", "load",
]

DG_OK, DG_ERR_INVALID_ARG, DG_ERR_UNSUPPORTED, DG_ERR_WORKSPACE, DG_ERR_CUDA = 0, 1, 2, 3, 4
DG_ERR_SCRATCH_LIMIT = 5
DG_PHASE_PREFILL, DG_PHASE_DENOISE, DG_PHASE_COMMIT, DG_PHASE_IDLE = 0, 1, 2, 3
DG_F32, DG_BF16 = 0, 1
DG_STOP_ARGMAX_STABLE, DG_STOP_ENTROPY = 0, 1
DG_ACCEPT_ENTROPY_BUDGET, DG_ACCEPT_MONOTONE = 0, 1
DG_SAMPLE_GROUPED, DG_SAMPLE_SEGMENTED = 0, 1
DG_DEV_NONFINITE_LOGITS, DG_DEV_BAD_TEMPERATURE, DG_DEV_BAD_TOKEN = 1, 2, 4
DG_DEV_WAIT_TIMEOUT, DG_DEV_BAD_PHASE = 8, 16

_HERE = os.path.dirname(os.path.abspath(__file__))


def library_path() -> str:
    return os.path.join(_HERE, "libdg.so")


class _CParams(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("canvas_len", ctypes.c_int32), ("vocab", ctypes.c_int32),
        ("logits_dtype", ctypes.c_int32), ("logits_ld", ctypes.c_int64),
        ("seed", ctypes.c_uint64), ("entropy_budget", ctypes.c_float),
        ("conf_threshold", ctypes.c_float), ("stable_k", ctypes.c_int32),
        ("step_cap", ctypes.c_int32), ("stop_rule", ctypes.c_int32),
        ("accept_rule", ctypes.c_int32), ("softcap", ctypes.c_float),
        ("embed_scale", ctypes.c_float), ("sample_rule", ctypes.c_int32),
    ]


_STATE_FIELDS = [
    "phase", "request_id", "temperature", "rng_step", "step", "stable", "canvas",
    "argmax_prev", "cand", "argmax", "accept", "m", "s", "entropy", "mean_entropy",
    "converged", "sc_valid", "num_sampled", "num_rejected", "emitted", "device_status",
    "committed", "prev_conf",
]


class _CState(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _STATE_FIELDS]


class DgError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {dg_status_string(code)} (code {code})")
        self.code = code


_LIB = None


def load(path: str) -> ctypes.CDLL:
    """Load a build of the library at ``path`` with the C signatures declared
    (``lib()`` loads the default build; tests load the wait test build)."""
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built; run `python -m denoise_step_sampler_gb300.build`")
    L = ctypes.CDLL(path)
    P, S = ctypes.POINTER(_CParams), ctypes.POINTER(_CState)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    L.dg_workspace_bytes.argtypes, L.dg_workspace_bytes.restype = [P, i32], sz
    L.dg_init_canvas.argtypes, L.dg_init_canvas.restype = [P, S, vp, vp], ctypes.c_int
    L.dg_commit.argtypes, L.dg_commit.restype = [P, S, vp, vp], ctypes.c_int
    L.dg_denoise_step.argtypes = [P, vp, S, vp, sz, vp]
    L.dg_denoise_step.restype = ctypes.c_int
    L.dg_selfcond_embed.argtypes = [P, vp, S, vp, i32, i64, vp, i32, vp, sz, vp]
    L.dg_selfcond_embed.restype = ctypes.c_int
    L.dg_workspace_bytes_feed.argtypes, L.dg_workspace_bytes_feed.restype = [P, i32], sz
    L.dg_denoise_step_feed.argtypes = [P, vp, S, vp, i32, i64, vp, i32, vp, sz, vp]
    L.dg_denoise_step_feed.restype = ctypes.c_int
    L.dg_status_string.argtypes, L.dg_status_string.restype = [ctypes.c_int], ctypes.c_char_p
    L.dg_denoise_step_noalloc.argtypes = [P, vp, S, vp]
    L.dg_denoise_step_noalloc.restype = ctypes.c_int
    L.dg_debug_wait_record.argtypes = [vp]
    L.dg_debug_wait_record.restype = ctypes.c_int
    L.dg_anneal_temperature.argtypes = [P, vp, vp, ctypes.c_float, ctypes.c_float, i32, vp, vp]
    L.dg_anneal_temperature.restype = ctypes.c_int
    return L


def lib():
    """Load ``libdg.so`` (built in-tree by ``denoise_step_sampler_gb300.build``)."""
    global _LIB
    if _LIB is None:
        _LIB = load(library_path())
    return _LIB


@dataclass
class Params:
    """Scalar parameters of a call (``dg_params``)."""

    batch: int
    canvas_len: int
    vocab: int
    logits_dtype: int = DG_BF16
    logits_ld: int | None = None
    seed: int = 0
    entropy_budget: float = 96.0
    conf_threshold: float = 0.3
    stable_k: int = 3
    step_cap: int = 32
    stop_rule: int = DG_STOP_ARGMAX_STABLE
    accept_rule: int = DG_ACCEPT_ENTROPY_BUDGET
    softcap: float = 0.0      # logit softcap c (0 = off)
    embed_scale: float = 0.0  # factor on the self-conditioning feed (0 = 1)
    sample_rule: int = DG_SAMPLE_GROUPED  # Gumbel-max rule of the candidate

    def c(self) -> _CParams:
        return _CParams(self.batch, self.canvas_len, self.vocab, self.logits_dtype,
                        self.vocab if self.logits_ld is None else self.logits_ld,
                        self.seed & 0xFFFFFFFFFFFFFFFF, self.entropy_budget,
                        self.conf_threshold, self.stable_k, self.step_cap, self.stop_rule,
                        self.accept_rule, self.softcap, self.embed_scale, self.sample_rule)


class State:
    """Per-request sampler state as device tensors (``dg_state``).

    uint64 quantities (request ids, rng steps) are stored in int64 tensors and
    read by the library as their two's-complement bit patterns.
    """

    def __init__(self, batch: int, canvas_len: int, device="cuda"):
        B, C = batch, canvas_len
        dev = torch.device(device)
        z = lambda shape, dt: torch.zeros(shape, dtype=dt, device=dev)  # noqa: E731
        self.batch, self.canvas_len, self.device = B, C, dev
        self.phase = torch.full((B,), DG_PHASE_IDLE, dtype=torch.uint8, device=dev)
        self.request_id = torch.arange(B, dtype=torch.int64, device=dev)
        self.temperature = torch.ones(B, dtype=torch.float32, device=dev)
        self.rng_step = z(B, torch.int64)
        self.step = z(B, torch.int32)
        self.stable = z(B, torch.int32)
        self.canvas = z(B * C, torch.int32)
        self.argmax_prev = z(B * C, torch.int32)
        self.cand = z(B * C, torch.int32)
        self.argmax = z(B * C, torch.int32)
        self.accept = z(B * C, torch.uint8)
        self.m = z(B * C, torch.float32)
        self.s = z(B * C, torch.float32)
        self.entropy = z(B * C, torch.float32)
        self.mean_entropy = z(B, torch.float32)
        self.converged = z(B, torch.uint8)
        self.sc_valid = z(B, torch.uint8)
        self.num_sampled = z(B, torch.int32)
        self.num_rejected = z(B, torch.int32)
        self.emitted = z(B * C, torch.int32)
        self.device_status = z(1, torch.int32)
        self.committed = z(B * C, torch.uint8)
        self.prev_conf = torch.full((B * C,), float("inf"), dtype=torch.float32, device=dev)

    _EXPECT = {
        "phase": (torch.uint8, "B"), "request_id": (torch.int64, "B"),
        "temperature": (torch.float32, "B"), "rng_step": (torch.int64, "B"),
        "step": (torch.int32, "B"), "stable": (torch.int32, "B"),
        "canvas": (torch.int32, "BC"), "argmax_prev": (torch.int32, "BC"),
        "cand": (torch.int32, "BC"), "argmax": (torch.int32, "BC"),
        "accept": (torch.uint8, "BC"), "m": (torch.float32, "BC"), "s": (torch.float32, "BC"),
        "entropy": (torch.float32, "BC"), "mean_entropy": (torch.float32, "B"),
        "converged": (torch.uint8, "B"), "sc_valid": (torch.uint8, "B"),
        "num_sampled": (torch.int32, "B"), "num_rejected": (torch.int32, "B"),
        "emitted": (torch.int32, "BC"), "device_status": (torch.int32, "1"),
        "committed": (torch.uint8, "BC"), "prev_conf": (torch.float32, "BC"),
    }

    def c(self) -> _CState:
        vals = []
        for name in _STATE_FIELDS:
            t = getattr(self, name)
            dt, shape = self._EXPECT[name]
            n = {"B": self.batch, "BC": self.batch * self.canvas_len, "1": 1}[shape]
            if t.dtype != dt or t.numel() != n or not t.is_contiguous() or t.device.type != "cuda":
                raise ValueError(f"state.{name}: want contiguous cuda {dt} with {n} elements")
            vals.append(t.data_ptr())
        return _CState(*vals)

    def snapshot(self) -> dict:
        """Host copies of every field (numpy), uint64 fields reinterpreted."""
        out = {}
        for name in _STATE_FIELDS:
            a = getattr(self, name).detach().cpu().numpy()
            if name in ("request_id", "rng_step"):
                a = a.view("uint64")
            if name == "device_status":
                a = a.view("uint32")
            out[name] = a
        return out


def _stream_ptr(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(code: int, where: str):
    if code != DG_OK:
        raise DgError(code, where)


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def dg_status_string(code: int) -> str:
    return lib().dg_status_string(int(code)).decode()


def dg_debug_wait_record() -> list:
    """{set, block, where, parity} of the first self-cond GEMM wait that gave up
    since load (diagnostics; synchronous)."""
    rec = (ctypes.c_uint32 * 4)()
    _check(lib().dg_debug_wait_record(ctypes.cast(rec, ctypes.c_void_p)), "dg_debug_wait_record")
    return list(rec)


def dg_workspace_bytes(params: Params, d: int = 0) -> int:
    return int(lib().dg_workspace_bytes(ctypes.byref(params.c()), int(d)))


def _logits_ok(params: Params, logits: torch.Tensor):
    want = torch.bfloat16 if params.logits_dtype == DG_BF16 else torch.float32
    ld = params.vocab if params.logits_ld is None else params.logits_ld
    if logits.dtype != want or logits.device.type != "cuda" or not logits.is_contiguous():
        raise ValueError(f"logits: want contiguous cuda {want}")
    if logits.numel() != params.batch * params.canvas_len * ld:
        raise ValueError("logits: want batch * canvas_len * logits_ld elements")


def dg_init_canvas(params: Params, state: State, row_mask: torch.Tensor, stream=None):
    if row_mask.dtype != torch.uint8 or row_mask.numel() != params.batch:
        raise ValueError("row_mask: want uint8 [batch]")
    _check(lib().dg_init_canvas(ctypes.byref(params.c()), ctypes.byref(state.c()),
                                _ptr(row_mask), _stream_ptr(stream)), "dg_init_canvas")


def dg_commit(params: Params, state: State, row_mask: torch.Tensor, stream=None):
    if row_mask.dtype != torch.uint8 or row_mask.numel() != params.batch:
        raise ValueError("row_mask: want uint8 [batch]")
    _check(lib().dg_commit(ctypes.byref(params.c()), ctypes.byref(state.c()),
                           _ptr(row_mask), _stream_ptr(stream)), "dg_commit")


def dg_anneal_temperature(params: Params, state: State, t_max: float, t_min: float,
                          n_steps: int, row_mask: torch.Tensor | None = None, stream=None):
    """Write state.temperature[r] = t_max + k (t_min - t_max) / n_steps from the
    rows' block-local step counters k (clamped to [0, n_steps]); call it before
    dg_denoise_step."""
    if row_mask is not None and (row_mask.dtype != torch.uint8 or row_mask.numel() != params.batch):
        raise ValueError("row_mask: want uint8 [batch]")
    _check(lib().dg_anneal_temperature(ctypes.byref(params.c()), _ptr(state.step),
                                       _ptr(state.temperature), float(t_max), float(t_min),
                                       int(n_steps), _ptr(row_mask) if row_mask is not None else None,
                                       _stream_ptr(stream)), "dg_anneal_temperature")


def dg_denoise_step(params: Params, logits: torch.Tensor, state: State,
                    workspace: torch.Tensor, stream=None):
    _logits_ok(params, logits)
    _check(lib().dg_denoise_step(ctypes.byref(params.c()), _ptr(logits), ctypes.byref(state.c()),
                                 _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _stream_ptr(stream)), "dg_denoise_step")


def dg_denoise_step_noalloc(params: Params, logits: torch.Tensor, state: State, stream=None):
    """dg_denoise_step for callers that cannot allocate device memory: no
    workspace argument; the library's own fixed scratch is used instead (see
    include/dg.h for its limit and sharing rules)."""
    _logits_ok(params, logits)
    _check(lib().dg_denoise_step_noalloc(ctypes.byref(params.c()), _ptr(logits),
                                         ctypes.byref(state.c()), _stream_ptr(stream)),
           "dg_denoise_step_noalloc")


def dg_selfcond_embed(params: Params, logits: torch.Tensor, state: State, E: torch.Tensor,
                      out: torch.Tensor, workspace: torch.Tensor | None, stream=None):
    _logits_ok(params, logits)
    if E.dtype != torch.bfloat16 or E.dim() != 2 or E.stride(1) != 1 or E.shape[0] != params.vocab:
        raise ValueError("E: want bf16 [V, d] with unit column stride")
    d = E.shape[1]
    if out.dtype == torch.float32:
        odt = DG_F32
    elif out.dtype == torch.bfloat16:
        odt = DG_BF16
    else:
        raise ValueError("out: want float32 or bfloat16")
    if out.numel() != params.batch * params.canvas_len * d or not out.is_contiguous():
        raise ValueError("out: want contiguous [batch * canvas_len, d]")
    ws_ptr = _ptr(workspace)
    ws_n = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().dg_selfcond_embed(ctypes.byref(params.c()), _ptr(logits), ctypes.byref(state.c()),
                                   _ptr(E), int(d), int(E.stride(0)), _ptr(out), odt, ws_ptr, ws_n,
                                   _stream_ptr(stream)), "dg_selfcond_embed")


def dg_workspace_bytes_feed(params: Params, d: int) -> int:
    return int(lib().dg_workspace_bytes_feed(ctypes.byref(params.c()), int(d)))


def dg_denoise_step_feed(params: Params, logits: torch.Tensor, state: State, E: torch.Tensor,
                         out: torch.Tensor, workspace: torch.Tensor, stream=None):
    _logits_ok(params, logits)
    if E.dtype != torch.bfloat16 or E.dim() != 2 or E.stride(1) != 1 or E.shape[0] != params.vocab:
        raise ValueError("E: want bf16 [V, d] with unit column stride")
    d = E.shape[1]
    if out.dtype == torch.float32:
        odt = DG_F32
    elif out.dtype == torch.bfloat16:
        odt = DG_BF16
    else:
        raise ValueError("out: want float32 or bfloat16")
    if out.numel() != params.batch * params.canvas_len * d or not out.is_contiguous():
        raise ValueError("out: want contiguous [batch * canvas_len, d]")
    ws_n = workspace.numel() * workspace.element_size()
    _check(lib().dg_denoise_step_feed(ctypes.byref(params.c()), _ptr(logits),
                                      ctypes.byref(state.c()), _ptr(E), int(d), int(E.stride(0)),
                                      _ptr(out), odt, _ptr(workspace), ws_n, _stream_ptr(stream)),
           "dg_denoise_step_feed")
