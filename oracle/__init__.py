"""CPU oracle for the DSpark draft step -- TEST INFRASTRUCTURE ONLY.

Plain single-threaded fp64 C (``oracle.c``) behind ctypes, plus an exact
rational brute force for tiny inputs (``brute.py``).  Only the tests, the smoke
check and the benchmark's CPU-baseline leg may import this package; the product
library never does, and this package imports nothing from the product except the
seeded input generator's output arrays passed in by the caller.

What each function follows:
  markov_draft  vllm.cpp issue #436 "SPEC-DSPARK W7", section "The fix"
  conf_probe    ds4 PR #772 "dspark: cut per-cycle CUDA overheads", section "Summary"
  ws_matvec     SharpInference issue #441, sections "Observation" / "Proposed work"
  ws_matvec_q8  SharpInference issue #441, "Proposed work" (quantized WS weights)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (gcc, -O2, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i = ctypes.c_int
        d = ctypes.c_double
        lib.oracle_markov_draft.argtypes = [P, P, P, P, P, i, i, i, i, P, P, P, P, P]
        lib.oracle_markov_draft.restype = i
        lib.oracle_conf_probe.argtypes = [P, P, i, i, d, d, P, P]
        lib.oracle_conf_probe.restype = i
        lib.oracle_ws_matvec.argtypes = [P, P, i, i, i, P, P]
        lib.oracle_ws_matvec.restype = i
        lib.oracle_ws_matvec_q8.argtypes = [P, P, i, i, i, P]
        lib.oracle_ws_matvec_q8.restype = i
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f64.restype = d
        lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_f64.restype = d
        lib.oracle_f64_to_f16_rne.argtypes = [d]
        lib.oracle_f64_to_f16_rne.restype = ctypes.c_uint16
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def markov_draft(base, w1, w2, d2t, prev0, *, forced_prev=None, want_logits=False,
                 want_bias=False):
    """Run the Markov block draft.

    base float32 [B,k,V]; w1, w2 uint16 bf16 bits [V,R]; d2t int32 [V] or None;
    prev0 int64 [B]; forced_prev int64 [B,k] or None (teacher forcing: the prev of
    position i+1 is forced_prev[:, i] instead of the oracle's own draft id).
    Returns dict(out_ids [B,k] int64 target ids, draft_ids [B,k] int64,
    logits [B,k,V] f64 | None, bias [B,k,V] f64 | None).
    """
    lib = _load()
    base = _c(base, np.float32)
    w1 = _c(w1, np.uint16)
    w2 = _c(w2, np.uint16)
    d2t = _c(d2t, np.int32)
    prev0 = _c(prev0, np.int64)
    forced_prev = _c(forced_prev, np.int64)
    B, k, V = base.shape
    R = w2.shape[1]
    assert w1.shape == (V, R) and w2.shape == (V, R) and prev0.shape == (B,)
    if forced_prev is not None:
        assert forced_prev.shape == (B, k)
    out = np.empty((B, k), np.int64)
    draft = np.empty((B, k), np.int64)
    logits = np.empty((B, k, V), np.float64) if want_logits else None
    bias = np.empty((B, k, V), np.float64) if want_bias else None
    rc = lib.oracle_markov_draft(_ptr(base), _ptr(w1), _ptr(w2), _ptr(d2t), _ptr(prev0),
                                 B, k, V, R, _ptr(forced_prev), _ptr(out), _ptr(draft),
                                 _ptr(logits), _ptr(bias))
    if rc != 0:
        raise ValueError("oracle_markov_draft rejected its arguments")
    return dict(out_ids=out, draft_ids=draft, logits=logits, bias=bias)


def conf_probe(wq, hidden, bias, threshold):
    """Run the confidence probe; returns (z float64 [n], gate int32 [n])."""
    lib = _load()
    wq = _c(wq, np.uint8)
    hidden = _c(hidden, np.float32)
    if hidden.ndim == 1:
        hidden = hidden[None, :]
    n, K = hidden.shape
    assert wq.size == (K // 32) * 34
    z = np.empty(n, np.float64)
    gate = np.empty(n, np.int32)
    rc = lib.oracle_conf_probe(_ptr(wq), _ptr(hidden), K, n, float(bias), float(threshold),
                               _ptr(z), _ptr(gate))
    if rc != 0:
        raise ValueError("oracle_conf_probe rejected its arguments")
    return z, gate


def ws_matvec(W, X):
    """Y = X W^T in fp64 from fp16 bits; returns (Y float64 [M,N], Y16 uint16 [M,N] RNE)."""
    lib = _load()
    W = _c(W, np.uint16)
    X = _c(X, np.uint16)
    N, K = W.shape
    M, K2 = X.shape
    assert K == K2
    Y = np.empty((M, N), np.float64)
    Y16 = np.empty((M, N), np.uint16)
    rc = lib.oracle_ws_matvec(_ptr(W), _ptr(X), M, N, K, _ptr(Y), _ptr(Y16))
    if rc != 0:
        raise ValueError("oracle_ws_matvec rejected its arguments")
    return Y, Y16


def ws_matvec_q8(Wq8, X):
    """Y = X dequant(W)^T in fp64; Wq8 uint8 [N * K/32 * 34] (Q8_0 blocks, row-major by row),
    X fp16 bits [M, K]; returns Y float64 [M, N]."""
    lib = _load()
    Wq8 = _c(Wq8, np.uint8).reshape(-1)
    X = _c(X, np.uint16)
    M, K = X.shape
    N = Wq8.size // ((K // 32) * 34)
    assert Wq8.size == N * (K // 32) * 34
    Y = np.empty((M, N), np.float64)
    rc = lib.oracle_ws_matvec_q8(_ptr(Wq8), _ptr(X), M, N, K, _ptr(Y))
    if rc != 0:
        raise ValueError("oracle_ws_matvec_q8 rejected its arguments")
    return Y


def bf16_to_f64(bits: int) -> float:
    return _load().oracle_bf16_to_f64(int(bits))


def f16_to_f64(bits: int) -> float:
    return _load().oracle_f16_to_f64(int(bits))


def f64_to_f16_rne(x: float) -> int:
    return int(_load().oracle_f64_to_f16_rne(float(x)))
