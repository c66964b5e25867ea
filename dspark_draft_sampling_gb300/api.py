"""Thin ctypes binding of libdspark (``include/dspark.h``) over torch CUDA tensors.

Argument marshalling only: shapes, dtypes and device pointers are checked and passed
to the C ABI; every arithmetic step runs in the library's CUDA kernels.  There is no
CPU fallback: if ``libdspark.so`` is missing or a call fails, a ``DsparkError`` is
raised.
"""
from __future__ import annotations

import ctypes
import os
import threading
import time

import torch

from . import build as _build

_STATUS_NAMES = {0: "OK", 1: "INVALID", 2: "UNSUPPORTED", 3: "CUDA", 4: "TIMEOUT", 5: "INDEX"}
DSPARK_OK, DSPARK_ERR_INVALID, DSPARK_ERR_UNSUPPORTED = 0, 1, 2
DSPARK_ERR_CUDA, DSPARK_ERR_TIMEOUT, DSPARK_ERR_INDEX = 3, 4, 5

# Every symbol the header declares, with (restype, argtypes).
_P, _I, _U, _F, _Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "dspark_last_error": (ctypes.c_char_p, []),
    "dspark_version": (ctypes.c_char_p, []),
    "dspark_markov_workspace_bytes": (_Z, [_I, _I, _I, _I]),
    "dspark_markov_draft": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _Z, _P]),
    "dspark_markov_draft_kernel": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _Z, _I,
                                        _P]),
    "dspark_markov_kernel_for": (_I, [_I, _I, _I, _I]),
    "dspark_markov_status": (_I, [_P, _P]),
    "dspark_markov_draft_debug": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _Z, _U, _U, _P]),
    "dspark_markov_draft_noalloc": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P]),
    "dspark_markov_plan_create": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _Z,
                                       ctypes.POINTER(_P)]),
    "dspark_markov_plan_launch": (_I, [_P, _P]),
    "dspark_markov_plan_destroy": (None, [_P]),
    "dspark_draft_plan_create": (_I, [_P, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _Z, _P,
                                      _Z, ctypes.POINTER(_P)]),
    "dspark_draft_plan_launch": (_I, [_P, _P]),
    "dspark_draft_plan_destroy": (None, [_P]),
    "dspark_gated_draft_plan_create": (_I, [_P, _P, _I, _F, _F, _P, _P, _P, _P, _P, _P, _P, _I, _I,
                                            _I, _I, _P, _P, _Z, ctypes.POINTER(_P)]),
    "dspark_gated_draft_plan_launch": (_I, [_P, _P]),
    "dspark_gated_draft_plan_destroy": (None, [_P]),
    "dspark_conf_probe": (_I, [_P, _P, _F, _F, _I, _I, _P, _P, _P]),
    "dspark_conf_probe_split": (_I, [_P, _P, _I, ctypes.c_longlong, _P, _I, ctypes.c_longlong, _F, _F,
                                     _I, _P, _P, _P]),
    "dspark_ws_matvec_workspace_bytes": (_Z, [_I, _I, _I]),
    "dspark_ws_matvec": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _Z, _P]),
    "dspark_ws_matvec_status": (_I, [_P, _P]),
    "dspark_ws_matvec_grouped_workspace_bytes": (_Z, [_P, _I]),
    "dspark_ws_matvec_grouped": (_I, [_P, _I, _P, _Z, _P]),
    "dspark_ws_matvec_debug": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _Z, _U, _P]),
    "dspark_ws_matvec_q8_debug": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _Z, _U, _P]),
    "dspark_q8_0_repack": (_I, [_P, _P, _P, _I, _I, _P]),
    "dspark_markov_draft_host_scratch_bytes": (_Z, [_I, _I, _I, _I]),
    "dspark_markov_draft_host": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _Z, _P, _P]),
    "dspark_conf_probe_host_scratch_bytes": (_Z, [_I, _I]),
    "dspark_conf_probe_host": (_I, [_P, _P, _F, _F, _I, _I, _P, _P, _P, _Z, _P, _P]),
    "dspark_ws_matvec_host_scratch_bytes": (_Z, [_I, _I, _I]),
    "dspark_ws_matvec_host": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _Z, _P, _P]),
    "dspark_ws_matvec_grouped_host_scratch_bytes": (_Z, [_P, _I]),
    "dspark_ws_matvec_grouped_host": (_I, [_P, _I, _P, _Z, _P, _P]),
    "dspark_ws_matvec_q8_workspace_bytes": (_Z, [_I, _I, _I]),
    "dspark_ws_matvec_q8": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _Z, _P]),
    "dspark_ws_matvec_q8_grouped_workspace_bytes": (_Z, [_P, _I]),
    "dspark_ws_matvec_q8_grouped": (_I, [_P, _I, _P, _Z, _P]),
    "dspark_ws_matvec_q8_grouped_debug": (_I, [_P, _I, _P, _Z, _I, _U, _P]),
}

_lock = threading.Lock()
_lib = None


class DsparkError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__(f"libdspark {_STATUS_NAMES.get(status, status)}: {message}")


def lib_path() -> str:
    return _build.lib_file()


def load_library(path: str | None = None):
    """Load libdspark.so (built by ``dspark_draft_sampling_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or lib_path()
        if not os.path.exists(p):
            raise DsparkError(DSPARK_ERR_CUDA, f"{p} not found; build it with "
                              "`python -m dspark_draft_sampling_gb300.build`")
        lib = ctypes.CDLL(p)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib


def _err(lib) -> str:
    msg = lib.dspark_last_error()
    return msg.decode(errors="replace") if msg else ""


def _check(lib, status: int):
    if status != DSPARK_OK:
        raise DsparkError(status, _err(lib))


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t, name: str, *, dtypes=None, itemsize=None, allow_none=False, allow_pinned=False):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    pinned_ok = allow_pinned and isinstance(t, torch.Tensor) and not t.is_cuda and t.is_pinned()
    if not isinstance(t, torch.Tensor) or not (t.is_cuda or pinned_ok):
        raise ValueError(f"{name} must be a CUDA tensor" + (" or pinned host memory" if allow_pinned else ""))
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtypes is not None and t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if itemsize is not None and t.element_size() != itemsize:
        raise ValueError(f"{name} must have {itemsize}-byte elements")
    return ctypes.c_void_p(t.data_ptr())


_BITS16 = (torch.bfloat16, torch.int16, torch.float16)


def markov_workspace_bytes(num_reqs: int, k: int, vocab: int, rank: int) -> int:
    return int(load_library().dspark_markov_workspace_bytes(num_reqs, k, vocab, rank))


def new_markov_workspace(num_reqs: int, k: int, vocab: int, rank: int, device=None):
    n = markov_workspace_bytes(num_reqs, k, vocab, rank)
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


MARKOV_KERNELS = {"auto": 0, "grid": 1, "cluster": 2}


def markov_kernel_for(num_reqs, k, vocab, rank) -> str:
    """Which kernel ``markov_draft(kernel="auto")`` runs for these sizes on the current device
    (with a 16-byte aligned base): ``"grid"`` or ``"cluster"``."""
    lib = load_library()
    code = int(lib.dspark_markov_kernel_for(int(num_reqs), int(k), int(vocab), int(rank)))
    return {v: n for n, v in MARKOV_KERNELS.items()}[code]


def markov_draft(base, w1, w2, d2t, prev, *, out_ids=None, workspace=None, dbg_logits=None,
                 dbg_bias=None, stream=None, kernel="auto"):
    """k-step Markov block draft.  base [B,k,V] fp32, w1/w2 [V,R] bf16, d2t [V] int32 or
    None, prev [B] int64 (updated in place).  Returns out_ids [B,k] int64 (target ids).
    ``kernel``: "auto" (dspark_markov_draft), or "grid" / "cluster" to name the kernel
    (dspark_markov_draft_kernel)."""
    lib = load_library()
    if kernel not in MARKOV_KERNELS:
        raise ValueError(f"kernel must be one of {sorted(MARKOV_KERNELS)}")
    if base.dim() != 3:
        raise ValueError("base must be [num_reqs, k, vocab]")
    B, k, V = base.shape
    R = w2.shape[1] if w2.dim() == 2 else -1
    if out_ids is None:
        out_ids = torch.empty((B, k), dtype=torch.int64, device=base.device)
    if workspace is None:
        workspace = new_markov_workspace(B, k, V, R, base.device)
    args = [
        _ptr(base, "base", dtypes=(torch.float32,)),
        _ptr(w1, "markov_w1", itemsize=2, dtypes=_BITS16),
        _ptr(w2, "markov_w2", itemsize=2, dtypes=_BITS16),
        _ptr(d2t, "d2t", dtypes=(torch.int32,), allow_none=True),
        _ptr(prev, "prev", dtypes=(torch.int64,)),
        B, k, V, R,
        _ptr(out_ids, "out_ids", dtypes=(torch.int64,)),
        _ptr(dbg_logits, "dbg_logits", dtypes=(torch.float32,), allow_none=True),
        _ptr(dbg_bias, "dbg_bias", dtypes=(torch.float32,), allow_none=True),
        _ptr(workspace, "workspace"), workspace.numel() * workspace.element_size()]
    if kernel == "auto":
        st = lib.dspark_markov_draft(*args, _stream(stream))
    else:
        st = lib.dspark_markov_draft_kernel(*args, MARKOV_KERNELS[kernel], _stream(stream))
    _check(lib, st)
    return out_ids


def markov_status(workspace, stream=None) -> int:
    """Synchronize and return the device status of the last draft on ``workspace``
    (0 = OK, DSPARK_ERR_INDEX, DSPARK_ERR_TIMEOUT)."""
    lib = load_library()
    return int(lib.dspark_markov_status(_ptr(workspace, "workspace"), _stream(stream)))


def markov_draft_debug(base, w1, w2, d2t, prev, out_ids, workspace, *, missing_arrivals: int,
                       timeout_us: int, stream=None):
    """Fault-injection hook: see dspark_markov_draft_debug in dspark.h."""
    lib = load_library()
    B, k, V = base.shape
    R = w2.shape[1]
    st = lib.dspark_markov_draft_debug(
        _ptr(base, "base"), _ptr(w1, "markov_w1"), _ptr(w2, "markov_w2"),
        _ptr(d2t, "d2t", allow_none=True), _ptr(prev, "prev"), B, k, V, R,
        _ptr(out_ids, "out_ids"), _ptr(workspace, "workspace"), workspace.numel(),
        int(missing_arrivals), int(timeout_us), _stream(stream))
    _check(lib, st)


class MarkovPlan:
    """A Markov draft recorded once into a CUDA graph; ``launch()`` replays it."""

    def __init__(self, base, w1, w2, d2t, prev, out_ids=None, workspace=None):
        self._lib = lib = load_library()
        B, k, V = base.shape
        R = w2.shape[1]
        if out_ids is None:
            out_ids = torch.empty((B, k), dtype=torch.int64, device=base.device)
        if workspace is None:
            workspace = new_markov_workspace(B, k, V, R, base.device)
        # keep the tensors alive for the plan's lifetime
        self.tensors = (base, w1, w2, d2t, prev, out_ids, workspace)
        self.out_ids, self.workspace = out_ids, workspace
        handle = ctypes.c_void_p()
        st = lib.dspark_markov_plan_create(
            _ptr(base, "base", dtypes=(torch.float32,)),
            _ptr(w1, "markov_w1", itemsize=2, dtypes=_BITS16),
            _ptr(w2, "markov_w2", itemsize=2, dtypes=_BITS16),
            _ptr(d2t, "d2t", dtypes=(torch.int32,), allow_none=True),
            _ptr(prev, "prev", dtypes=(torch.int64,)), B, k, V, R,
            _ptr(out_ids, "out_ids", dtypes=(torch.int64,)),
            _ptr(workspace, "workspace"), workspace.numel(), ctypes.byref(handle))
        _check(lib, st)
        self._handle = handle

    def launch(self, stream=None):
        _check(self._lib, self._lib.dspark_markov_plan_launch(self._handle, _stream(stream)))
        return self.out_ids

    def close(self):
        if getattr(self, "_handle", None):
            self._lib.dspark_markov_plan_destroy(self._handle)
            self._handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class DraftPlan:
    """lm_head matvec (base logits written on the device) + Markov draft in one CUDA graph.

    lm_head fp16 [vocab, H]; hidden fp16 [num_reqs * k, H]; markov_w1/w2 bf16 [vocab, R];
    d2t int32 [vocab] or None; prev int64 [num_reqs] (updated on the device)."""

    def __init__(self, lm_head, hidden, w1, w2, d2t, prev, k: int):
        self._lib = lib = load_library()
        V, H = lm_head.shape
        B = prev.numel()
        R = w2.shape[1]
        if hidden.shape != (B * k, H):
            raise ValueError("hidden must be [num_reqs * k, hidden_dim]")
        dev = lm_head.device
        self.base = torch.empty((B, k, V), dtype=torch.float32, device=dev)
        self.out_ids = torch.empty((B, k), dtype=torch.int64, device=dev)
        self.markov_ws = new_markov_workspace(B, k, V, R, dev)
        self.ws_ws = new_ws_workspace(B * k, V, H, dev)
        self.tensors = (lm_head, hidden, w1, w2, d2t, prev)
        handle = ctypes.c_void_p()
        st = lib.dspark_draft_plan_create(
            _ptr(lm_head, "lm_head", itemsize=2, dtypes=_BITS16), _ptr(hidden, "hidden", itemsize=2,
                                                                        dtypes=_BITS16), H,
            _ptr(w1, "markov_w1", itemsize=2, dtypes=_BITS16),
            _ptr(w2, "markov_w2", itemsize=2, dtypes=_BITS16),
            _ptr(d2t, "d2t", dtypes=(torch.int32,), allow_none=True),
            _ptr(prev, "prev", dtypes=(torch.int64,)), B, k, V, R,
            _ptr(self.base, "base"), _ptr(self.out_ids, "out_ids"),
            _ptr(self.markov_ws, "markov_ws"), self.markov_ws.numel(),
            _ptr(self.ws_ws, "ws_ws"), self.ws_ws.numel(), ctypes.byref(handle))
        _check(lib, st)
        self._handle = handle

    def launch(self, stream=None):
        _check(self._lib, self._lib.dspark_draft_plan_launch(self._handle, _stream(stream)))
        return self.out_ids

    def close(self):
        if getattr(self, "_handle", None):
            self._lib.dspark_draft_plan_destroy(self._handle)
            self._handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class GatedDraftPlan:
    """Probe -> (if sigmoid(z) >= threshold) Markov draft, decided on the device, one graph."""

    def __init__(self, wq, probe_input, bias: float, threshold: float, base, w1, w2, d2t, prev):
        self._lib = lib = load_library()
        B, k, V = base.shape
        R = w2.shape[1]
        K = probe_input.numel()
        dev = base.device
        self.logit = torch.empty(1, dtype=torch.float32, device=dev)
        self.gate = torch.empty(1, dtype=torch.int32, device=dev)
        self.out_ids = torch.empty((B, k), dtype=torch.int64, device=dev)
        self.workspace = new_markov_workspace(B, k, V, R, dev)
        self.tensors = (wq, probe_input, base, w1, w2, d2t, prev)
        handle = ctypes.c_void_p()
        st = lib.dspark_gated_draft_plan_create(
            _ptr(wq, "wq", dtypes=(torch.uint8, torch.int8)),
            _ptr(probe_input, "probe_input", dtypes=(torch.float32,)), K, float(bias), float(threshold),
            _ptr(self.logit, "logit"), _ptr(self.gate, "gate"),
            _ptr(base, "base", dtypes=(torch.float32,)),
            _ptr(w1, "markov_w1", itemsize=2, dtypes=_BITS16),
            _ptr(w2, "markov_w2", itemsize=2, dtypes=_BITS16),
            _ptr(d2t, "d2t", dtypes=(torch.int32,), allow_none=True),
            _ptr(prev, "prev", dtypes=(torch.int64,)), B, k, V, R,
            _ptr(self.out_ids, "out_ids"), _ptr(self.workspace, "workspace"), self.workspace.numel(),
            ctypes.byref(handle))
        _check(lib, st)
        self._handle = handle

    def launch(self, stream=None):
        _check(self._lib, self._lib.dspark_gated_draft_plan_launch(self._handle, _stream(stream)))
        return self.out_ids

    def close(self):
        if getattr(self, "_handle", None):
            self._lib.dspark_gated_draft_plan_destroy(self._handle)
            self._handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def conf_probe(wq, hidden, bias: float, threshold: float, *, logit_out=None, gate_out=None,
               stream=None):
    """Q8_0 confidence probes.  wq uint8 [K/32*34], hidden fp32 [n, K] (or [K]).
    gate_out may be a pinned host tensor: the kernel then stores each 4-byte decision
    straight into host memory (the device reaches pinned memory by the same address).
    Returns (logit_out [n] fp32, gate_out [n] int32)."""
    lib = load_library()
    if hidden.dim() == 1:
        hidden = hidden.view(1, -1)
    n, K = hidden.shape
    if wq.numel() != (K // 32) * 34:
        raise ValueError("wq must hold K/32 Q8_0 blocks of 34 bytes")
    if gate_out is None:
        gate_out = torch.empty(n, dtype=torch.int32, device=hidden.device)
    if logit_out is None and gate_out.is_cuda:
        logit_out = torch.empty(n, dtype=torch.float32, device=hidden.device)
    st = lib.dspark_conf_probe(_ptr(wq, "wq", dtypes=(torch.uint8, torch.int8)),
                               _ptr(hidden, "hidden", dtypes=(torch.float32,)),
                               float(bias), float(threshold), K, n,
                               _ptr(logit_out, "logit_out", dtypes=(torch.float32,), allow_none=True),
                               _ptr(gate_out, "gate_out", dtypes=(torch.int32,), allow_pinned=True),
                               _stream(stream))
    _check(lib, st)
    return logit_out, gate_out


class ProbeCall:
    """Confidence probes prepared once for the latency path: the arguments are checked and
    marshalled at construction, so each ``launch()`` is one C call (dspark_conf_probe).  With
    ``gate_out`` in pinned host memory the kernel stores each 4-byte decision straight into
    host memory, and ``decide()`` launches and polls those words: no copy and no stream
    synchronization on the host path.  The tensors must stay alive and in place."""

    _PENDING = 2  # never a decision: the kernel writes 1, 0, or -1 after a wait that gave up

    def __init__(self, wq, hidden, bias: float, threshold: float, *, gate_out=None, logit_out=None,
                 stream=None):
        lib = load_library()
        if hidden.dim() == 1:
            hidden = hidden.view(1, -1)
        n, K = hidden.shape
        if wq.numel() != (K // 32) * 34:
            raise ValueError("wq must hold K/32 Q8_0 blocks of 34 bytes")
        if gate_out is None:
            gate_out = torch.empty(n, dtype=torch.int32).pin_memory()
        if gate_out.numel() < n:
            raise ValueError("gate_out holds fewer than n decisions")
        self.gate_out, self.logit_out, self.n = gate_out, logit_out, n
        self._keep = (wq, hidden)
        self._fn = lib.dspark_conf_probe
        self._lib = lib
        self._args = (_ptr(wq, "wq", dtypes=(torch.uint8, torch.int8)),
                      _ptr(hidden, "hidden", dtypes=(torch.float32,)),
                      ctypes.c_float(bias), ctypes.c_float(threshold), K, n,
                      _ptr(logit_out, "logit_out", dtypes=(torch.float32,), allow_none=True),
                      _ptr(gate_out, "gate_out", dtypes=(torch.int32,), allow_pinned=True),
                      _stream(stream))
        self._stream = stream
        self._gates = None if gate_out.is_cuda else gate_out.numpy()

    def launch(self):
        st = self._fn(*self._args)
        if st != DSPARK_OK:
            _check(self._lib, st)

    def decide(self, timeout_s: float = 1.0):
        """Launch and wait for the decisions in pinned host memory; returns them as a numpy
        int32 array (1: keep drafting, 0: stop, -1: the kernel gave up a wait).  After
        ``timeout_s`` the stream is synchronized and its error, if any, raised."""
        g = self._gates
        if g is None:
            raise ValueError("decide() needs gate_out in pinned host memory")
        n, pending = self.n, self._PENDING
        g[:n] = pending
        self.launch()
        t0 = time.perf_counter()
        i = 0  # the probes' stores land in any order; a word stays set once written
        while i < n:
            if g[i] != pending:
                i += 1
                continue
            if time.perf_counter() - t0 > timeout_s:
                (self._stream or torch.cuda.current_stream()).synchronize()
                if (g[:n] == pending).any():
                    raise DsparkError(DSPARK_ERR_TIMEOUT, "probe decisions did not arrive")
                break
        return g[:n].copy()


def conf_probe_split(wq, hidden, state, bias: float, threshold: float, *, logit_out=None,
                     gate_out=None, stream=None):
    """Probes over [hidden; state] given as two row-major tensors [n, K_hidden], [n, K_state]
    (any row strides that keep rows 16-byte aligned).  Returns (logit [n], gate [n])."""
    lib = load_library()
    n, Kh = hidden.shape
    n2, Ks = state.shape
    if n != n2:
        raise ValueError("hidden and state disagree on the number of probes")
    if wq.numel() != ((Kh + Ks) // 32) * 34:
        raise ValueError("wq must hold (K_hidden + K_state) / 32 Q8_0 blocks of 34 bytes")
    for t, name in ((hidden, "hidden"), (state, "state")):
        if not t.is_cuda or t.dtype != torch.float32 or t.stride(1) != 1:
            raise ValueError(f"{name} must be a CUDA float32 tensor with unit column stride")
    if gate_out is None:
        gate_out = torch.empty(n, dtype=torch.int32, device=hidden.device)
    if logit_out is None:
        logit_out = torch.empty(n, dtype=torch.float32, device=hidden.device)
    st = lib.dspark_conf_probe_split(_ptr(wq, "wq", dtypes=(torch.uint8, torch.int8)),
                                     ctypes.c_void_p(hidden.data_ptr()), Kh, hidden.stride(0),
                                     ctypes.c_void_p(state.data_ptr()), Ks, state.stride(0),
                                     float(bias), float(threshold), n,
                                     _ptr(logit_out, "logit_out", dtypes=(torch.float32,)),
                                     _ptr(gate_out, "gate_out", dtypes=(torch.int32,)),
                                     _stream(stream))
    _check(lib, st)
    return logit_out, gate_out


def ws_matvec_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load_library().dspark_ws_matvec_workspace_bytes(M, N, K))


def new_ws_workspace(M: int, N: int, K: int, device=None):
    """Zero-filled scratch for ws_matvec (the kernel leaves it zero-filled after each call)."""
    n = ws_matvec_workspace_bytes(M, N, K)
    if n == 0:
        raise DsparkError(DSPARK_ERR_CUDA, "could not size the ws_matvec workspace")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def ws_matvec(W, X, *, out=None, out_fp32: bool = False, workspace=None, stream=None):
    """Y = X W^T.  W fp16 [N, K], X fp16 [M, K]; returns Y [M, N] (fp16, or fp32)."""
    lib = load_library()
    N, K = W.shape
    M, K2 = X.shape
    if K != K2:
        raise ValueError("W and X disagree on K")
    w_p = _ptr(W, "W", itemsize=2, dtypes=_BITS16)
    x_p = _ptr(X, "X", itemsize=2, dtypes=_BITS16)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32 if out_fp32 else torch.float16,
                          device=W.device)
    if workspace is None:
        workspace = new_ws_workspace(M, N, K, W.device)
    y_fp32 = out.dtype == torch.float32
    st = lib.dspark_ws_matvec(w_p, x_p,
                              _ptr(out, "out", dtypes=(torch.float16, torch.float32)),
                              1 if y_fp32 else 0, M, N, K,
                              _ptr(workspace, "workspace"), workspace.numel(), _stream(stream))
    _check(lib, st)
    return out


def q8_0_repack(w_q8_0, N: int, K: int, *, stream=None):
    """Split Q8_0 blocks (uint8 [N * K/32 * 34], row-major by weight row) into
    (q int8 [N, K], d fp16-bit int16 [N, K/32]) on the device."""
    lib = load_library()
    if K <= 0 or K % 32:
        raise ValueError("K must be a positive multiple of 32")
    if w_q8_0.numel() != N * (K // 32) * 34:
        raise ValueError("w_q8_0 does not hold N * K/32 Q8_0 blocks")
    src = _ptr(w_q8_0, "w_q8_0", dtypes=(torch.uint8,))
    q = torch.empty((N, K), dtype=torch.int8, device=w_q8_0.device)
    d = torch.empty((N, K // 32), dtype=torch.int16, device=w_q8_0.device)
    st = lib.dspark_q8_0_repack(src, _ptr(q, "q"), _ptr(d, "d"), N, K, _stream(stream))
    _check(lib, st)
    return q, d


def ws_matvec_q8_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load_library().dspark_ws_matvec_q8_workspace_bytes(M, N, K))


def new_ws_q8_workspace(M: int, N: int, K: int, device=None):
    """Zero-filled scratch for ws_matvec_q8 (the kernel leaves it zero-filled after each call)."""
    n = ws_matvec_q8_workspace_bytes(M, N, K)
    if n == 0:
        raise DsparkError(DSPARK_ERR_CUDA, "could not size the ws_matvec_q8 workspace")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def ws_matvec_q8(Wq, Wd, X, *, out=None, out_fp32: bool = False, workspace=None, stream=None):
    """Y = X dequant(W)^T.  Wq int8 [N, K], Wd fp16 bits [N, K/32] (from q8_0_repack),
    X fp16 [M, K]; returns Y [M, N] (fp16, or fp32)."""
    lib = load_library()
    N, K = Wq.shape
    M, K2 = X.shape
    if K != K2:
        raise ValueError("Wq and X disagree on K")
    if tuple(Wd.shape) != (N, K // 32):
        raise ValueError("Wd must be [N, K/32]")
    q_p = _ptr(Wq, "Wq", dtypes=(torch.int8,))
    d_p = _ptr(Wd, "Wd", itemsize=2, dtypes=_BITS16)
    x_p = _ptr(X, "X", itemsize=2, dtypes=_BITS16)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32 if out_fp32 else torch.float16,
                          device=Wq.device)
    if workspace is None:
        workspace = new_ws_q8_workspace(M, N, K, Wq.device)
    y_fp32 = out.dtype == torch.float32
    st = lib.dspark_ws_matvec_q8(q_p, d_p, x_p,
                                 _ptr(out, "out", dtypes=(torch.float16, torch.float32)),
                                 1 if y_fp32 else 0, M, N, K,
                                 _ptr(workspace, "workspace"), workspace.numel(), _stream(stream))
    _check(lib, st)
    return out


class WsQ8Problem(ctypes.Structure):
    """dspark_ws_q8_problem."""
    _fields_ = [("Wq", ctypes.c_void_p), ("Wd", ctypes.c_void_p), ("X", ctypes.c_void_p),
                ("Y", ctypes.c_void_p), ("y_is_fp32", ctypes.c_int), ("M", ctypes.c_int),
                ("N", ctypes.c_int), ("K", ctypes.c_int)]


def new_ws_q8_grouped_workspace(device=None):
    """Zero-filled workspace for ws_matvec_q8_grouped on the current device."""
    n = int(load_library().dspark_ws_matvec_q8_grouped_workspace_bytes(None, 0))
    if n == 0:
        raise DsparkError(DSPARK_ERR_CUDA, "could not size the grouped ws_matvec_q8 workspace")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def _ws_q8_problems(problems):
    arr = (WsQ8Problem * len(problems))()
    for i, (Wq, Wd, X, Y) in enumerate(problems):
        N, K = Wq.shape
        M, K2 = X.shape
        if K != K2 or tuple(Y.shape) != (M, N) or tuple(Wd.shape) != (N, K // 32):
            raise ValueError(f"problem {i}: Wq [N,K], Wd [N,K/32], X [M,K] and Y [M,N] disagree")
        arr[i] = WsQ8Problem(_ptr(Wq, "Wq", dtypes=(torch.int8,)), _ptr(Wd, "Wd", itemsize=2, dtypes=_BITS16),
                             _ptr(X, "X", itemsize=2, dtypes=_BITS16),
                             _ptr(Y, "Y", dtypes=(torch.float16, torch.float32)),
                             1 if Y.dtype == torch.float32 else 0, M, N, K)
    return arr


def ws_matvec_q8_grouped(problems, *, workspace=None, stream=None):
    """Several independent Y = X dequant(W)^T in one launch.  problems: list of (Wq int8
    [N,K], Wd fp16 bits [N,K/32], X fp16 [M,K], Y [M,N] fp16 or fp32) device tensors; Y is
    written in place."""
    lib = load_library()
    arr = _ws_q8_problems(problems)
    if workspace is None:
        workspace = new_ws_q8_grouped_workspace(problems[0][0].device)
    st = lib.dspark_ws_matvec_q8_grouped(ctypes.cast(arr, ctypes.c_void_p), len(arr), _ptr(workspace, "workspace"),
                                         workspace.numel(), _stream(stream))
    _check(lib, st)
    return [p[3] for p in problems]


def ws_matvec_q8_grouped_debug(problems, workspace, *, withheld_cta: int, timeout_us: int, stream=None):
    """Fault-injection hook: see dspark_ws_matvec_q8_grouped_debug in dspark.h."""
    lib = load_library()
    arr = _ws_q8_problems(problems)
    st = lib.dspark_ws_matvec_q8_grouped_debug(ctypes.cast(arr, ctypes.c_void_p), len(arr),
                                               _ptr(workspace, "workspace"), workspace.numel(), int(withheld_cta),
                                               int(timeout_us), _stream(stream))
    _check(lib, st)


# ---- host-buffer forms: per-call inputs and outputs in (pinned) host memory ----

def _host_ptr(t, name: str, *, dtypes=None, itemsize=None, allow_none=False):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor, ideally pinned")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtypes is not None and t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if itemsize is not None and t.element_size() != itemsize:
        raise ValueError(f"{name} must have {itemsize}-byte elements")
    return ctypes.c_void_p(t.data_ptr())


def markov_draft_host_scratch_bytes(num_reqs: int, k: int, vocab: int, rank: int) -> int:
    return int(load_library().dspark_markov_draft_host_scratch_bytes(num_reqs, k, vocab, rank))


def conf_probe_host_scratch_bytes(K: int, n_probes: int) -> int:
    return int(load_library().dspark_conf_probe_host_scratch_bytes(K, n_probes))


def ws_matvec_host_scratch_bytes(M: int, N: int, K: int) -> int:
    return int(load_library().dspark_ws_matvec_host_scratch_bytes(M, N, K))


def _event(ev):
    """Raw handle of a torch.cuda.Event.  torch creates the CUDA event on its first record, so
    an event that was never recorded is recorded once here to create it (the library then
    records it again where it belongs)."""
    if ev is None:
        return None
    if not ev.cuda_event:
        ev.record(torch.cuda.current_stream())
    if not ev.cuda_event:
        raise DsparkError(DSPARK_ERR_CUDA, "could not create the CUDA event")
    return ctypes.c_void_p(ev.cuda_event)


def markov_draft_host(base_h, w1, w2, d2t, prev_h, out_ids_h, scratch, *, inputs_copied=None,
                      stream=None):
    """Markov draft from host inputs: base_h float [B,k,V] and prev_h int64 [B] (updated in
    place) on the host, w1/w2/d2t on the device; fills out_ids_h int64 [B,k] on the host
    once `stream` is synchronized."""
    lib = load_library()
    B, k, V = base_h.shape
    R = w2.shape[1]
    st = lib.dspark_markov_draft_host(
        _host_ptr(base_h, "base_h", dtypes=(torch.float32,)),
        _ptr(w1, "markov_w1", itemsize=2, dtypes=_BITS16), _ptr(w2, "markov_w2", itemsize=2, dtypes=_BITS16),
        _ptr(d2t, "d2t", dtypes=(torch.int32,), allow_none=True),
        _host_ptr(prev_h, "prev_h", dtypes=(torch.int64,)), B, k, V, R,
        _host_ptr(out_ids_h, "out_ids_h", dtypes=(torch.int64,)),
        _ptr(scratch, "scratch"), scratch.numel() * scratch.element_size(), _event(inputs_copied),
        _stream(stream))
    _check(lib, st)
    return out_ids_h


def conf_probe_host(wq, hidden_h, bias: float, threshold: float, gate_h, scratch, *, logit_h=None,
                    inputs_copied=None, stream=None):
    """Confidence probes from host inputs: hidden_h float [n, K] on the host, wq on the
    device; fills gate_h int32 [n] (and logit_h float [n]) on the host."""
    lib = load_library()
    n, K = hidden_h.shape
    st = lib.dspark_conf_probe_host(
        _ptr(wq, "wq", dtypes=(torch.uint8, torch.int8)), _host_ptr(hidden_h, "hidden_h", dtypes=(torch.float32,)),
        float(bias), float(threshold), K, n, _host_ptr(logit_h, "logit_h", dtypes=(torch.float32,), allow_none=True),
        _host_ptr(gate_h, "gate_h", dtypes=(torch.int32,)), _ptr(scratch, "scratch"),
        scratch.numel() * scratch.element_size(), _event(inputs_copied), _stream(stream))
    _check(lib, st)
    return gate_h


def ws_matvec_host(W, X_h, Y_h, scratch, *, inputs_copied=None, stream=None):
    """Y_h = X_h W^T with X_h fp16 [M, K] and Y_h [M, N] (fp16 or fp32) on the host, W on the
    device; `scratch` must be zero-filled before its first use."""
    lib = load_library()
    N, K = W.shape
    M = X_h.shape[0]
    st = lib.dspark_ws_matvec_host(
        _ptr(W, "W", itemsize=2, dtypes=_BITS16), _host_ptr(X_h, "X_h", itemsize=2, dtypes=_BITS16),
        _host_ptr(Y_h, "Y_h", dtypes=(torch.float16, torch.float32)), 1 if Y_h.dtype == torch.float32 else 0,
        M, N, K, _ptr(scratch, "scratch"), scratch.numel() * scratch.element_size(), _event(inputs_copied),
        _stream(stream))
    _check(lib, st)
    return Y_h


def ws_matvec_status(workspace, *, stream=None) -> int:
    """Status of a WS (fp16 or Q8_0) workspace after its calls: DSPARK_OK or
    DSPARK_ERR_TIMEOUT (reported once, then cleared)."""
    lib = load_library()
    return int(lib.dspark_ws_matvec_status(_ptr(workspace, "workspace"), _stream(stream)))


class WsProblem(ctypes.Structure):
    """Mirror of dspark_ws_problem."""
    _fields_ = [("W", ctypes.c_void_p), ("X", ctypes.c_void_p), ("Y", ctypes.c_void_p),
                ("y_is_fp32", ctypes.c_int), ("M", ctypes.c_int), ("N", ctypes.c_int), ("K", ctypes.c_int)]


def _ws_problems(problems):
    arr = (WsProblem * len(problems))()
    for i, (W, X, Y) in enumerate(problems):
        N, K = W.shape
        M, K2 = X.shape
        if K != K2 or tuple(Y.shape) != (M, N):
            raise ValueError(f"problem {i}: W [N,K], X [M,K] and Y [M,N] disagree")
        arr[i] = WsProblem(_ptr(W, "W", itemsize=2, dtypes=_BITS16), _ptr(X, "X", itemsize=2, dtypes=_BITS16),
                           _ptr(Y, "Y", dtypes=(torch.float16, torch.float32)),
                           1 if Y.dtype == torch.float32 else 0, M, N, K)
    return arr


def ws_matvec_grouped_workspace_bytes(problems) -> int:
    arr = _ws_problems(problems)
    return int(load_library().dspark_ws_matvec_grouped_workspace_bytes(ctypes.cast(arr, ctypes.c_void_p), len(arr)))


def ws_matvec_grouped(problems, *, workspace=None, stream=None):
    """Several independent Y = X W^T in one launch.  problems: list of (W [N,K] fp16,
    X [M,K] fp16, Y [M,N] fp16 or fp32) device tensors; Y is written in place."""
    lib = load_library()
    arr = _ws_problems(problems)
    if workspace is None:
        n = int(lib.dspark_ws_matvec_grouped_workspace_bytes(ctypes.cast(arr, ctypes.c_void_p), len(arr)))
        if n == 0:
            raise DsparkError(DSPARK_ERR_CUDA, "could not size the grouped ws_matvec workspace")
        workspace = torch.zeros(n, dtype=torch.uint8, device=problems[0][0].device)
    st = lib.dspark_ws_matvec_grouped(ctypes.cast(arr, ctypes.c_void_p), len(arr), _ptr(workspace, "workspace"),
                                      workspace.numel(), _stream(stream))
    _check(lib, st)
    return [Y for (_, _, Y) in problems]


def _ws_problems_host(problems):
    arr = (WsProblem * len(problems))()
    for i, (W, X_h, Y_h) in enumerate(problems):
        N, K = W.shape
        M, K2 = X_h.shape
        if K != K2 or tuple(Y_h.shape) != (M, N):
            raise ValueError(f"problem {i}: W [N,K], X [M,K] and Y [M,N] disagree")
        arr[i] = WsProblem(_ptr(W, "W", itemsize=2, dtypes=_BITS16), _host_ptr(X_h, "X_h", itemsize=2, dtypes=_BITS16),
                           _host_ptr(Y_h, "Y_h", dtypes=(torch.float16, torch.float32)),
                           1 if Y_h.dtype == torch.float32 else 0, M, N, K)
    return arr


def ws_matvec_grouped_host_scratch_bytes(problems) -> int:
    arr = _ws_problems_host(problems)
    return int(load_library().dspark_ws_matvec_grouped_host_scratch_bytes(ctypes.cast(arr, ctypes.c_void_p),
                                                                          len(arr)))


def ws_matvec_grouped_host(problems, scratch, *, inputs_copied=None, stream=None):
    """Grouped matvec from host buffers: problems = list of (W device [N,K], X_h host [M,K],
    Y_h host [M,N]); `scratch` zero-filled before first use."""
    lib = load_library()
    arr = _ws_problems_host(problems)
    st = lib.dspark_ws_matvec_grouped_host(ctypes.cast(arr, ctypes.c_void_p), len(arr), _ptr(scratch, "scratch"),
                                           scratch.numel() * scratch.element_size(), _event(inputs_copied),
                                           _stream(stream))
    _check(lib, st)
    return [Y for (_, _, Y) in problems]
