"""Exact brute force for tiny inputs -- TEST INFRASTRUCTURE ONLY.

Rational arithmetic (``fractions.Fraction``), independent of ``oracle.c``: the
Markov chain is evaluated through the full transition-bias matrix
P[v, u] = sum_j markov_w2[v, j] * markov_w1[u, j] rather than the gather + GEMV
order of the oracle, and number formats are decoded with ``struct`` / numpy.
Sized for vocab <= 64, rank <= 8 and K <= 256; pure-Python loops.
"""
from __future__ import annotations

import math
import struct
from fractions import Fraction

import numpy as np


def bf16_exact(bits: int) -> Fraction:
    (f,) = struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))
    return Fraction(f)


def f16_exact(bits: int) -> Fraction:
    return Fraction(float(np.array([bits], dtype=np.uint16).view(np.float16)[0]))


def markov_draft(base, w1, w2, d2t, prev0):
    """Exact draft ids (target space) and logits as Fractions.

    The bias added to step i is column ``prev`` of P = markov_w2 . markov_w1^T."""
    B, k, V = base.shape
    R = w2.shape[1]
    W1 = [[bf16_exact(w1[u, j]) for j in range(R)] for u in range(V)]
    W2 = [[bf16_exact(w2[v, j]) for j in range(R)] for v in range(V)]
    P = [[sum((W2[v][j] * W1[u][j] for j in range(R)), Fraction(0)) for u in range(V)]
         for v in range(V)]
    out = np.zeros((B, k), np.int64)
    draft = np.zeros((B, k), np.int64)
    logits = [[None] * k for _ in range(B)]
    for r in range(B):
        p = int(prev0[r])
        for i in range(k):
            row = [Fraction(float(base[r, i, v])) + P[v][p] for v in range(V)]
            m = max(row)
            ident = min(v for v in range(V) if row[v] == m)
            draft[r, i] = ident
            out[r, i] = ident if d2t is None else int(d2t[ident])
            logits[r][i] = row
            p = ident
    return out, draft, logits


def conf_probe(wq, hidden, bias, threshold):
    """Exact z (Fraction) and gate per probe.

    The gate is decided on sigmoid(z) >= t; away from exact equality, with
    t = a/b rational, sigmoid(z) >= t  <=>  exp(z) >= t/(1-t), evaluated here with
    math.exp only when |z - log(t/(1-t))| is comfortably large (the caller checks)."""
    n, K = hidden.shape
    nb = K // 32
    blocks = np.asarray(wq, dtype=np.uint8).reshape(nb, 34)
    zs, gates = [], []
    for p in range(n):
        z = Fraction(float(bias))
        for b in range(nb):
            d = f16_exact(int(blocks[b, 0]) | (int(blocks[b, 1]) << 8))
            q = blocks[b, 2:].view(np.int8)
            for j in range(32):
                z += d * int(q[j]) * Fraction(float(hidden[p, 32 * b + j]))
        zs.append(z)
        sig = 1.0 / (1.0 + math.exp(-float(z)))
        gates.append(1 if sig >= threshold else 0)
    return zs, gates


def ws_matvec(W, X):
    """Exact Y[m][n] = sum_k X[m,k] W[n,k] as Fractions."""
    N, K = W.shape
    M = X.shape[0]
    Wf = [[f16_exact(W[n, kk]) for kk in range(K)] for n in range(N)]
    Xf = [[f16_exact(X[m, kk]) for kk in range(K)] for m in range(M)]
    return [[sum((Xf[m][kk] * Wf[n][kk] for kk in range(K)), Fraction(0)) for n in range(N)]
            for m in range(M)]


def ws_matvec_q8(Wq8, X, N, K):
    """Exact Y[m][n] for Q8_0 weights (Fractions)."""
    nb = K // 32
    blocks = np.asarray(Wq8, dtype=np.uint8).reshape(N, nb, 34)
    M = X.shape[0]
    Xf = [[f16_exact(X[m, kk]) for kk in range(K)] for m in range(M)]
    out = [[Fraction(0)] * N for _ in range(M)]
    for n in range(N):
        for b in range(nb):
            d = f16_exact(int(blocks[n, b, 0]) | (int(blocks[n, b, 1]) << 8))
            q = blocks[n, b, 2:].view(np.int8)
            for m in range(M):
                s = sum((int(q[j]) * Xf[m][32 * b + j] for j in range(32)), Fraction(0))
                out[m][n] += d * s
    return out
