"""Seeded synthetic inputs for the DSpark draft step.

This module only draws random numbers and lays them out in the byte formats the
library takes (bf16 / fp16 bit patterns, Q8_0 blocks).  It contains none of the
draft step's arithmetic, so both the CPU oracle (test side) and the CUDA path
consume exactly the same arrays.

Workloads (shapes and value distributions of the pages' lanes):

* ``tiny``            num_reqs=1, k=4,  vocab=4096,   rank=64,  base N(0,1), w N(0,0.05)
* ``reduced_vocab``   num_reqs=1, k=9,  vocab=32000,  rank=256, base N(0,2), w N(0,0.02),
                      d2t = random injective map into a 151936-token target vocab,
                      0.5% of vocab rows in planted exact-tie pairs
* ``qwen3_8b``        num_reqs=1, k=7,  vocab=151936, rank=256 (markov_w2 ~78 MB bf16)
* ``full_vocab_27b``  num_reqs in {1,4,8}, k=15, vocab=248320, rank=256
* probe               hidden fp32 [7424] N(0,1), Q8_0 weights q~U{-127..127}, d=fp16(1e-3),
                      bias N(0,1), threshold 0.5, 2 probes per cycle x 1024 cycles
* ws matvec           M=7 fp16, W N(0,0.02) [N,K], X N(0,1) [M,K],
                      (K,N) in {(4096,4096), (4096,1024), (4096,12288), (12288,4096)}

Random streams: numpy PCG64 seeded with ``[seed, stream_id]`` so each tensor has its
own reproducible stream independent of generation order.
"""
from __future__ import annotations

import numpy as np

# stream ids: one per generated tensor
_S_BASE, _S_W1, _S_W2, _S_PREV, _S_D2T, _S_TIES = 1, 2, 3, 4, 5, 6
_S_QW, _S_QD, _S_HID, _S_BIAS = 11, 12, 13, 14
_S_WSW, _S_WSX = 21, 22
_S_Q8Q, _S_Q8D = 31, 32

TARGET_VOCAB = 151936
Q8_0_BLOCK = 32          # elements per Q8_0 block
Q8_0_BLOCK_BYTES = 34    # fp16 scale + 32 int8

MARKOV_CONFIGS = {
    "tiny": dict(num_reqs=1, k=4, vocab=4096, rank=64, base_sd=1.0, w_sd=0.05,
                 d2t="identity", tie_frac=0.0),
    "reduced_vocab": dict(num_reqs=1, k=9, vocab=32000, rank=256, base_sd=2.0, w_sd=0.02,
                          d2t="injective", tie_frac=0.005),
    "qwen3_8b": dict(num_reqs=1, k=7, vocab=151936, rank=256, base_sd=2.0, w_sd=0.02,
                     d2t="identity", tie_frac=0.0),
    "full_vocab_27b": dict(num_reqs=1, k=15, vocab=248320, rank=256, base_sd=2.0, w_sd=0.02,
                           d2t="identity", tie_frac=0.0),
}

WS_SHAPES = [(4096, 4096), (4096, 1024), (4096, 12288), (12288, 4096)]  # (K, N)
PROBE_K = 7424


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([seed, stream]))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest-even) and return the 16-bit patterns.

    Inputs must be finite (the generators never draw NaN/inf)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def f32_to_f16_bits(a: np.ndarray) -> np.ndarray:
    """Round to fp16 (numpy's nearest-even conversion) and return the bit patterns."""
    return np.ascontiguousarray(a, dtype=np.float32).astype(np.float16).view(np.uint16)


def _normal(seed, stream, shape, sd):
    x = _rng(seed, stream).standard_normal(size=shape, dtype=np.float32)
    if sd != 1.0:
        x *= np.float32(sd)
    return x


def markov_inputs(num_reqs: int, k: int, vocab: int, rank: int, *, base_sd: float = 2.0,
                  w_sd: float = 0.02, d2t: str = "identity", tie_frac: float = 0.0,
                  seed: int = 0, target_vocab: int = TARGET_VOCAB) -> dict:
    """Inputs of one Markov block draft.

    Returns a dict with
      base  float32 [num_reqs, k, vocab]   base logits, row i belongs to draft position i
      w1    uint16  [vocab, rank]          markov_w1 as bf16 bit patterns
      w2    uint16  [vocab, rank]          markov_w2 as bf16 bit patterns
      d2t   int32   [vocab] or None        draft->target id map (None = identity)
      prev0 int64   [num_reqs]             previous draft id per request
      ties  int64   [n_pairs, 2]           planted exact-tie pairs (v1 < v2)
      spiked_steps  list[int]              positions whose argmax is forced onto a tie pair

    Planted ties: the w2 row and every base entry of v2 are copies of v1's, so the two
    rows have bit-identical logits at every step.  On even positions one pair gets a
    +20 spike on both members, which makes that pair the maximum, so the lowest-index
    tie-break decides the draft id there.
    """
    if d2t not in ("identity", "injective"):
        raise ValueError("d2t must be 'identity' or 'injective'")
    base = markov_base(num_reqs, k, vocab, base_sd=base_sd, seed=seed)
    w1 = f32_to_bf16_bits(_normal(seed, _S_W1, (vocab, rank), w_sd))
    w2 = f32_to_bf16_bits(_normal(seed, _S_W2, (vocab, rank), w_sd))
    prev0 = _rng(seed, _S_PREV).integers(0, vocab, size=num_reqs, dtype=np.int64)
    d2t_arr = None
    if d2t == "injective":
        if target_vocab < vocab:
            raise ValueError("target vocab smaller than draft vocab")
        perm = _rng(seed, _S_D2T).permutation(target_vocab)
        d2t_arr = np.ascontiguousarray(perm[:vocab].astype(np.int32))
    n_pairs = int(round(tie_frac * vocab))
    ties = np.zeros((0, 2), dtype=np.int64)
    spiked = []
    if n_pairs > 0:
        rng = _rng(seed, _S_TIES)
        idx = rng.choice(vocab, size=2 * n_pairs, replace=False).reshape(n_pairs, 2)
        ties = np.sort(idx, axis=1).astype(np.int64)
        v1, v2 = ties[:, 0], ties[:, 1]
        w2[v2] = w2[v1]
        base[:, :, v2] = base[:, :, v1]
        for i in range(0, k, 2):
            p = ties[(i // 2) % n_pairs]
            base[:, i, p[0]] = np.float32(20.0)
            base[:, i, p[1]] = np.float32(20.0)
            spiked.append(i)
    return dict(base=base, w1=w1, w2=w2, d2t=d2t_arr, prev0=prev0, ties=ties,
                spiked_steps=spiked, num_reqs=num_reqs, k=k, vocab=vocab, rank=rank)


def markov_base(num_reqs: int, k: int, vocab: int, *, base_sd: float = 2.0, seed: int = 0) -> np.ndarray:
    """The base logits of markov_inputs alone (same stream, same values; request r's rows do
    not depend on num_reqs)."""
    return _normal(seed, _S_BASE, (num_reqs, k, vocab), base_sd)


def markov_config(name: str, *, num_reqs: int | None = None, seed: int = 0) -> dict:
    """Inputs of one of the named Markov lanes (see the module docstring)."""
    c = dict(MARKOV_CONFIGS[name])
    if num_reqs is not None:
        c["num_reqs"] = num_reqs
    return markov_inputs(c.pop("num_reqs"), c.pop("k"), c.pop("vocab"), c.pop("rank"),
                         seed=seed, **c)


def probe_inputs(n_probes: int, K: int = PROBE_K, *, seed: int = 0, scale: float = 1e-3,
                 threshold: float = 0.5, random_scales: bool = False) -> dict:
    """Inputs of a batch of confidence probes against one Q8_0 weight row.

    Returns
      wq        uint8 [K/32 * 34]   Q8_0 blocks: fp16 scale d (little endian) then 32 int8 q
      hidden    float32 [n_probes, K]
      bias      float (an fp32-representable value)
      threshold float in (0, 1)
    With ``random_scales`` every block gets its own fp16 scale drawn from
    |N(0, scale)| (used by edge-case tests); otherwise all scales are fp16(scale).
    """
    if K % Q8_0_BLOCK:
        raise ValueError("K must be a multiple of 32")
    nb = K // Q8_0_BLOCK
    q = _rng(seed, _S_QW).integers(-127, 128, size=(nb, Q8_0_BLOCK), dtype=np.int64).astype(np.int8)
    if random_scales:
        d = np.abs(_rng(seed, _S_QD).standard_normal(nb)).astype(np.float32) * np.float32(scale)
    else:
        d = np.full(nb, scale, dtype=np.float32)
    d_bits = f32_to_f16_bits(d)
    blocks = np.zeros((nb, Q8_0_BLOCK_BYTES), dtype=np.uint8)
    blocks[:, 0:2] = d_bits.astype("<u2").view(np.uint8).reshape(nb, 2)
    blocks[:, 2:] = q.view(np.uint8)
    hidden = _normal(seed, _S_HID, (n_probes, K), 1.0)
    bias = float(np.float32(_rng(seed, _S_BIAS).standard_normal()))
    return dict(wq=blocks.reshape(-1).copy(), hidden=hidden, bias=bias,
                threshold=float(threshold), K=K, n_probes=n_probes)


def ws_inputs(M: int, N: int, K: int, *, seed: int = 0, w_sd: float = 0.02,
              x_sd: float = 1.0) -> dict:
    """Inputs of one weight-stationary matvec: W fp16 bits [N, K], X fp16 bits [M, K]."""
    W = f32_to_f16_bits(_normal(seed, _S_WSW, (N, K), w_sd))
    X = f32_to_f16_bits(_normal(seed, _S_WSX, (M, K), x_sd))
    return dict(W=W, X=X, M=M, N=N, K=K)


def ws_exact_inputs(M: int, N: int, K: int, *, seed: int = 0) -> dict:
    """Weight-stationary matvec inputs whose products and partial sums are all exact in fp32:
    X integers in [-3, 3], W = k / 1024 with integer k in [-127, 127] (both exact in fp16).
    Every partial sum is a multiple of 2^-10 below K * 381 * 2^-10 in magnitude, exact in fp32
    while K * 381 < 2^24 (K <= 44034)."""
    if K * 381 >= (1 << 24):
        raise ValueError("K too large for exact fp32 partial sums")
    x = _rng(seed, _S_WSX).integers(-3, 4, size=(M, K)).astype(np.float32)
    w = (_rng(seed, _S_WSW).integers(-127, 128, size=(N, K), dtype=np.int16).astype(np.float32)
         * np.float32(1.0 / 1024.0))
    return dict(W=f32_to_f16_bits(w), X=f32_to_f16_bits(x), M=M, N=N, K=K)


def ws_q8_inputs(M: int, N: int, K: int, *, seed: int = 0, d_sd: float = 2e-4,
                 power_of_two_scales: bool = False) -> dict:
    """Inputs of a quantized weight-stationary matvec: W as Q8_0 blocks (row-major by weight
    row: N x K/32 blocks of 34 bytes, q ~ U{-127..127}, fp16 scales |N(0, d_sd)|), X fp16 bits
    [M, K] N(0,1).  With power_of_two_scales every scale is 2^-j (j in 8..12), so every
    dequantized weight d*q is exactly representable in fp16."""
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    nb = K // 32
    # drawn as int16 (exact for this range, a quarter of int64's memory at N ~ 2M rows)
    q = _rng(seed, _S_Q8Q).integers(-127, 128, size=(N, nb, 32), dtype=np.int16).astype(np.int8)
    if power_of_two_scales:
        j = _rng(seed, _S_Q8D).integers(8, 13, size=(N, nb))
        d = np.ldexp(1.0, -j).astype(np.float32)
    else:
        d = np.abs(_rng(seed, _S_Q8D).standard_normal((N, nb))).astype(np.float32) * np.float32(d_sd)
    blocks = np.zeros((N, nb, 34), dtype=np.uint8)
    blocks[:, :, 0:2] = f32_to_f16_bits(d).astype("<u2").view(np.uint8).reshape(N, nb, 2)
    blocks[:, :, 2:] = q.view(np.uint8)
    X = f32_to_f16_bits(_normal(seed, _S_WSX, (M, K), 1.0))
    return dict(Wq8=blocks.reshape(-1).copy(), X=X, M=M, N=N, K=K)
