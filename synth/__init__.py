"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module draws random numbers and rounds them to bf16; it holds none of the
Markov-head arithmetic.  Every generator uses numpy's PCG64 so that the host
bytes handed to the oracle and the bytes uploaded to the GPU are identical.

Recipe (the shape of the workloads on the DSpark pages; no dataset is used):

* base logits ``U[b, k, :]`` (the backbone output of DSpark's parallel pass,
  "Semi-autoregressive generation"): ``3 * N(0, 1)`` for every token, then 8
  distinct uniformly chosen tokens per (b, k) get ``+U(8, 12)`` (a handful of
  plausible continuations standing out of a broad tail);
* weights ``W1 [V, r]``, ``W2 [r, V]``, selector tables ``A, Bt [V, r]``, gate
  weight ``Wg [d, r]`` and confidence weight ``w [d (+ r)]``: ``N(0, 0.02)``
  rounded to bf16 (round to nearest even);
* hidden states ``h [B, K, d]``: ``N(0, 1)`` rounded to bf16;
* anchors: uniform in ``[0, V)``;
* target logits for verification (``target_logits``): the draft's base logits
  plus ``N(0, 1)`` per token for the K draft positions, and a bonus row of
  ``3 * N(0, 1)``.

bf16 tensors are returned as ``uint16`` bit patterns.
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

VOCAB_FULL = 151936  # 4B-class vocabulary: 2 * 151936 * 256 = 77.8M head parameters
RANK = 256


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return the uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    x = rng.standard_normal(int(np.prod(shape)), dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return bf16_bits(x).reshape(shape)


def base_logits(rng: np.random.Generator, B: int, K: int, V: int,
                spikes: int = 8, lo: float = 8.0, hi: float = 12.0) -> np.ndarray:
    """U [B, K, V] float32: 3*N(0,1) plus `spikes` distinct tokens per row raised by U(lo, hi)."""
    rows = B * K
    U = rng.standard_normal(rows * V, dtype=np.float32)
    U *= np.float32(3.0)
    U = U.reshape(rows, V)
    ns = min(spikes, V)
    if ns > 0:
        idx = rng.integers(0, V, size=(rows, ns))
        # redraw duplicates within a row until all spike tokens are distinct
        for rw in range(rows):
            row = idx[rw]
            while len(np.unique(row)) != ns:
                seen = set()
                for j in range(ns):
                    while int(row[j]) in seen:
                        row[j] = rng.integers(0, V)
                    seen.add(int(row[j]))
        add = rng.uniform(lo, hi, size=(rows, ns)).astype(np.float32)
        U[np.arange(rows)[:, None], idx] += add
    return U.reshape(B, K, V)


@dataclasses.dataclass
class DraftInputs:
    """Inputs of one Markov-head draft call (host arrays)."""
    B: int
    K: int
    V: int
    r: int
    U: np.ndarray            # float32 [B, K, V]
    W1: Optional[np.ndarray]  # uint16 (bf16) [V, r] (None for selector-only workloads)
    W2: Optional[np.ndarray]  # uint16 (bf16) [r, V]
    anchors: np.ndarray      # int32 [B]
    d: int = 0
    h: Optional[np.ndarray] = None     # uint16 (bf16) [B, K, d]
    Wg: Optional[np.ndarray] = None    # uint16 (bf16) [d, r] (gated head)
    w_conf: Optional[np.ndarray] = None  # uint16 (bf16) [d + r] (confidence head)
    A: Optional[np.ndarray] = None     # uint16 (bf16) [V, r] (selector)
    Bt: Optional[np.ndarray] = None    # uint16 (bf16) [V, r] (selector)
    Wa: Optional[np.ndarray] = None    # uint16 (bf16) [d, r] (RNN head's decay gate)


def make_inputs(seed: int, B: int, K: int, V: int, r: int = RANK, *, d: int = 0,
                gated: bool = False, confidence: bool = False, selector: bool = False,
                spikes: int = 8, weight_std: float = 0.02,
                selector_tables_only: bool = False, rnn: bool = False) -> DraftInputs:
    """Draw one synthetic workload from PCG64(seed) in a fixed order."""
    rng = np.random.default_rng(seed)
    U = base_logits(rng, B, K, V, spikes=spikes)
    if selector_tables_only:
        W1 = W2 = None
    else:
        W1 = _normal_bf16(rng, (V, r), weight_std)
        W2 = _normal_bf16(rng, (r, V), weight_std)
    anchors = rng.integers(0, V, size=B).astype(np.int32)
    inp = DraftInputs(B=B, K=K, V=V, r=r, U=U, W1=W1, W2=W2, anchors=anchors, d=d)
    if d > 0:
        inp.h = _normal_bf16(rng, (B, K, d), 1.0)
    if gated:
        assert d > 0
        inp.Wg = _normal_bf16(rng, (d, r), weight_std)
    if confidence:
        assert d > 0
        inp.w_conf = _normal_bf16(rng, (d + r,), weight_std)
    if selector:
        inp.A = _normal_bf16(rng, (V, r), weight_std)
        inp.Bt = _normal_bf16(rng, (V, r), weight_std)
    if rnn:  # drawn last, so the other arrays are those of the same call without it
        assert d > 0
        inp.Wa = _normal_bf16(rng, (d, r), weight_std)
    return inp


# The five workloads (sizes and distributions of the DSpark pages' setting).
CONFIGS = {
    0: dict(name="tiny-vanilla B=1 K=4 V=4096 r=256", B=1, K=4, V=4096, r=256,
            temperatures=(1.0, 0.0), seeds=(0,)),
    1: dict(name="single-request B=1 K=16 V=151936 r=256", B=1, K=16, V=VOCAB_FULL, r=256,
            temperatures=(0.0, 0.7, 1.0), seeds=tuple(range(10))),
    2: dict(name="serving+confidence B=128 K=16 V=151936 r=256 d=2048", B=128, K=16,
            V=VOCAB_FULL, r=256, d=2048, confidence=True, threshold=0.3, conf_bias=0.0,
            temperatures=(1.0, 0.0), seeds=tuple(range(10))),
    3: dict(name="gated B=64 K=16 V=151936 r=256 d=4096", B=64, K=16, V=VOCAB_FULL, r=256,
            d=4096, gated=True, temperatures=(1.0,), seeds=tuple(range(10))),
    4: dict(name="selector-top16 B=256 K=16 V=151936 r=256 d=4096", B=256, K=16,
            V=VOCAB_FULL, r=256, d=4096, gated=True, selector=True, topk=16,
            temperatures=(1.0,), seeds=tuple(range(4))),
    # the RNN head (no workload of the pages' own; the gated head's shapes, with both the
    # decay gate Wa and the input gate Wg drawn like Wg)
    5: dict(name="rnn B=64 K=16 V=151936 r=256 d=4096", B=64, K=16, V=VOCAB_FULL, r=256,
            d=4096, gated=True, rnn=True, temperatures=(1.0,), seeds=tuple(range(4))),
}


def target_logits(seed: int, U: np.ndarray, noise: float = 1.0, bonus_std: float = 3.0) -> np.ndarray:
    """Synthetic target logits P [B, K+1, V] for verification: the draft's base
    logits plus N(0, noise^2) per token (a target that mostly agrees with the
    draft), and a bonus row of N(0, bonus_std^2) after the block."""
    B, K, V = U.shape
    rng = np.random.default_rng(seed)
    P = np.empty((B, K + 1, V), np.float32)
    for b in range(B):
        P[b, :K] = U[b] + rng.standard_normal((K, V), dtype=np.float32) * np.float32(noise)
        P[b, K] = rng.standard_normal(V, dtype=np.float32) * np.float32(bonus_std)
    return P


def config_inputs(cfg: int) -> DraftInputs:
    """Inputs of workload `cfg`, drawn from PCG64(1000 + cfg)."""
    c = CONFIGS[cfg]
    return make_inputs(1000 + cfg, c["B"], c["K"], c["V"], c["r"], d=c.get("d", 0),
                       gated=c.get("gated", False), confidence=c.get("confidence", False),
                       selector=c.get("selector", False),
                       selector_tables_only=c.get("selector", False), rnn=c.get("rnn", False))


def schedule_inputs(seed: int, R: int, K: int):
    """Survival products a [R, K] (cumulative products of per-position confidences drawn
    from U(0.4, 0.995)) and a smooth saturating steps-per-second table SPS(B),
    B = 0 .. R (K + 1), as float32."""
    rng = np.random.default_rng(seed)
    a = np.cumprod(rng.uniform(0.4, 0.995, (R, K)), axis=1).astype(np.float32)
    B = np.arange(R * (K + 1) + 1, dtype=np.float64)
    sps = (3000.0 / (1.0 + (B / (0.6 * R * (K + 1))) ** 2)).astype(np.float32)
    return a, sps


def sts_inputs(seed: int, N: int, K: int, spread: float = 2.0, sharpness: float = 2.5):
    """Raw confidences [N, K] = sigmoid(z), z ~ N(0, spread^2), of a head that is too sharp by
    `sharpness`, and 0/1 acceptance outcomes drawn at sigmoid(z / sharpness), as float32."""
    rng = np.random.default_rng(seed)
    z = rng.normal(0.0, spread, (N, K))
    conf = (1.0 / (1.0 + np.exp(-z))).astype(np.float32)
    outcome = (rng.uniform(size=(N, K)) < 1.0 / (1.0 + np.exp(-z / sharpness))).astype(np.float32)
    return conf, outcome
