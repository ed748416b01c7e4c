"""fp64 CPU oracle of the DSpark Markov-head drafting hot path (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: the test-suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The product path never imports this
package.  The arithmetic lives in ``dspark_oracle.c`` (plain C, double
precision, optional OpenMP); this module only builds it with gcc, marshals
numpy arrays and reshapes outputs.  It shares no code with the CUDA path.

Every function cites the passage of the DSpark pages it follows in the C
source.  Every function here is pinned by ``tests/test_oracle_pins.py``
(printed values, known answers, closed forms through numpy/scipy, exhaustive
enumeration); ``tests/test_oracle_mutants.py`` compiles copies of the C source
with planted mistakes and checks that a pin catches each one.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dspark_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, no FP contraction); return the .so path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and \
            os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    P = ctypes.c_void_p
    i32, i64, f64, u64, u32 = (ctypes.c_int, ctypes.c_int64, ctypes.c_double,
                               ctypes.c_uint64, ctypes.c_uint32)
    lib.orc_set_threads.argtypes = [i32]
    lib.orc_max_threads.restype = i32
    lib.orc_philox4x32_10.argtypes = [P, P, P]
    lib.orc_uniform.argtypes = [u64, u32, u32, u32, u32]
    lib.orc_uniform.restype = f64
    lib.orc_uniform_ctr.argtypes = [u64, u32, u32, u32, u32, u32]
    lib.orc_uniform_ctr.restype = f64
    lib.orc_block_uniform.argtypes = [u64, u32, u32, u32]
    lib.orc_block_uniform.restype = f64
    lib.orc_within_uniform.argtypes = [u64, u32, u32, u32]
    lib.orc_within_uniform.restype = f64
    lib.orc_accept_uniform.argtypes = [u64, u32, u32]
    lib.orc_accept_uniform.restype = f64
    lib.orc_verify.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32, i32, f64, f64, u64, i32,
                               i32, P, P, P, P]
    lib.orc_verify.restype = i32
    lib.orc_schedule.argtypes = [P, i32, i32, P, P, P, P]
    lib.orc_schedule.restype = i32
    lib.orc_accept_label.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, f64, f64, P]
    lib.orc_accept_label.restype = i32
    lib.orc_gate.argtypes = [P, P, i64, i32, i32, P]
    lib.orc_markov_draft.argtypes = [P, P, P, P, P, i32, i32, i32, i32, f64, u64, i32, i32,
                                     P, P, P, P, P]
    lib.orc_markov_draft.restype = i32
    lib.orc_markov_logits.argtypes = [P, P, P, P, P, i32, i32, i32, i32, f64, i32, i32, P, P]
    lib.orc_markov_logits.restype = i32
    lib.orc_rnn_draft.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, f64, u64, i32, i32,
                                  P, P, P, P, P]
    lib.orc_rnn_draft.restype = i32
    lib.orc_rnn_logits.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, f64, i32, i32, P, P]
    lib.orc_rnn_logits.restype = i32
    lib.orc_confidence.argtypes = [P, P, P, P, P, f64, i32, i32, i32, i32, i32, i32, f64,
                                   P, P, P, P]
    lib.orc_confidence.restype = i32
    lib.orc_sts_fit.argtypes = [P, P, i32, i32, f64, f64, P, P]
    lib.orc_sts_fit.restype = i32
    lib.orc_topk.argtypes = [P, i32, i32, i32, i32, P, P, P]
    lib.orc_topk.restype = i32
    lib.orc_pair_scores.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, P]
    lib.orc_pair_scores.restype = i32
    lib.orc_walk.argtypes = [P, P, i32, i32, i32, f64, u64, i32, i32, P, P, P, P, P]
    lib.orc_walk.restype = i32
    return lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


class Oracle:
    """The oracle's functions bound to one compiled library (the default one, or a copy)."""

    def __init__(self, lib_path: str):
        self.lib_path = lib_path
        self._lib = _bind(ctypes.CDLL(lib_path))

    def set_threads(self, n: int) -> None:
        self._lib.orc_set_threads(int(n))

    def max_threads(self) -> int:
        return int(self._lib.orc_max_threads())

    def philox4x32_10(self, ctr, key) -> np.ndarray:
        """One Philox4x32-10 block: ctr (4 x uint32), key (2 x uint32) -> 4 x uint32."""
        c = np.ascontiguousarray(ctr, dtype=np.uint32)
        k = np.ascontiguousarray(key, dtype=np.uint32)
        out = np.zeros(4, np.uint32)
        self._lib.orc_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
        return out

    def uniform(self, seed: int, b: int, k: int, v: int, tag: int = 0) -> float:
        return float(self._lib.orc_uniform(seed, b, k, v, tag))

    def block_uniform(self, seed: int, b: int, k: int, blk: int) -> float:
        """Stage-1 uniform of 16-token block `blk` (request b, position k)."""
        return float(self._lib.orc_block_uniform(seed, b, k, blk))

    def within_uniform(self, seed: int, b: int, k: int, blk: int) -> float:
        """Stage-2 uniform of 16-token block `blk` (request b, position k)."""
        return float(self._lib.orc_within_uniform(seed, b, k, blk))

    def accept_uniform(self, seed: int, b: int, k: int) -> float:
        """The verifier's acceptance uniform of position k of request b."""
        return float(self._lib.orc_accept_uniform(seed, b, k))

    def verify(self, P, U, W1, W2, anchors, tokens, *, draft_temperature: float,
               target_temperature: float, seed: int, ell=None, H=None, b0: int = 0,
               nb: Optional[int] = None) -> dict:
        """Speculative verification of drafted tokens [B, K] against target logits
        P [B, K+1, V]: accepted prefix length and the next token per request."""
        P = _c(P, np.float32)
        U = _c(U, np.float32)
        B, K, V = U.shape
        assert P.shape == (B, K + 1, V)
        r = 0 if W1 is None else W1.shape[1]
        W1 = _c(W1, np.uint16) if r > 0 else np.zeros((V, 1), np.uint16)
        W2 = _c(W2, np.uint16) if r > 0 else np.zeros((1, V), np.uint16)
        anchors = _c(anchors, np.int32)
        tokens = _c(tokens, np.int32)
        ell = _c(ell, np.int32)
        H = _c(H, np.float64)
        nb = B - b0 if nb is None else nb
        n_acc = np.zeros(nb, np.int32)
        nxt = np.zeros(nb, np.int32)
        accept_prob = np.zeros((nb, K), np.float64)
        margins = np.zeros(nb, np.float64)
        rc = self._lib.orc_verify(_ptr(P), _ptr(U), _ptr(W1), _ptr(W2), _ptr(anchors), _ptr(H),
                                  _ptr(tokens), _ptr(ell), B, K, V, r, float(draft_temperature),
                                  float(target_temperature), seed, b0, nb, _ptr(n_acc), _ptr(nxt),
                                  _ptr(accept_prob), _ptr(margins))
        if rc != 0:
            raise ValueError("oracle verify rejected its arguments")
        return dict(n_acc=n_acc, next_token=nxt, accept_prob=accept_prob, margins=margins)

    def accept_label(self, P, U, W1, W2, anchors, tokens, *, draft_temperature: float,
                     target_temperature: float, H=None) -> np.ndarray:
        """c*_k = 1 - TV(p^d_k, p^t_k) of every drafted position [B, K]."""
        P = _c(P, np.float32)
        U = _c(U, np.float32)
        B, K, V = U.shape
        assert P.shape == (B, K + 1, V)
        r = 0 if W1 is None else W1.shape[1]
        W1 = _c(W1, np.uint16) if r > 0 else np.zeros((V, 1), np.uint16)
        W2 = _c(W2, np.uint16) if r > 0 else np.zeros((1, V), np.uint16)
        anchors = _c(anchors, np.int32)
        tokens = _c(tokens, np.int32)
        H = _c(H, np.float64)
        label = np.zeros((B, K), np.float64)
        rc = self._lib.orc_accept_label(_ptr(P), _ptr(U), _ptr(W1), _ptr(W2), _ptr(anchors),
                                        _ptr(H), _ptr(tokens), B, K, V, r,
                                        float(draft_temperature), float(target_temperature),
                                        _ptr(label))
        if rc != 0:
            raise ValueError("oracle accept_label rejected its arguments")
        return label

    def schedule(self, a, sps) -> dict:
        """Greedy load-aware prefix scheduler: survival a [R, K], SPS(B) table
        [R * (K + 1) + 1] -> verify lengths ell [R], Theta and the stopping margin."""
        a = _c(a, np.float64)
        R, K = a.shape
        sps = _c(sps, np.float64)
        assert sps.shape[0] >= R * (K + 1) + 1
        ell = np.zeros(R, np.int32)
        theta = np.zeros(1, np.float64)
        margin = np.zeros(1, np.float64)
        rc = self._lib.orc_schedule(_ptr(a), R, K, _ptr(sps), _ptr(ell), _ptr(theta), _ptr(margin))
        if rc != 0:
            raise ValueError("oracle schedule rejected its arguments")
        return dict(ell=ell, theta=float(theta[0]), margin=float(margin[0]))

    def gate(self, h: np.ndarray, Wg: np.ndarray) -> np.ndarray:
        """H = sigmoid(h . Wg) in fp64; h [..., d] bf16 bits, Wg [d, r] bf16 bits -> [..., r]."""
        h = _c(h, np.uint16)
        Wg = _c(Wg, np.uint16)
        d, r = Wg.shape
        M = h.size // d
        H = np.zeros(h.shape[:-1] + (r,), np.float64)
        self._lib.orc_gate(_ptr(h), _ptr(Wg), M, d, r, _ptr(H))
        return H

    def markov_draft(self, U, W1, W2, anchors, *, temperature: float, seed: int, H=None,
                     b0: int = 0, nb: Optional[int] = None, forced=None) -> dict:
        """Run the Markov-head draft for requests b0 .. b0+nb-1 (outputs compact [nb, K])."""
        U = _c(U, np.float32)
        B, K, V = U.shape
        r = 0 if W1 is None else W1.shape[1]
        W1 = _c(W1, np.uint16) if r > 0 else np.zeros((V, 1), np.uint16)
        W2 = _c(W2, np.uint16) if r > 0 else np.zeros((1, V), np.uint16)
        anchors = _c(anchors, np.int32)
        H = _c(H, np.float64)
        nb = B - b0 if nb is None else nb
        forced = _c(forced, np.int32)
        tokens = np.zeros((nb, K), np.int32)
        logprobs = np.zeros((nb, K), np.float64)
        margins = np.zeros((nb, K), np.float64)
        flp = np.zeros((nb, K), np.float64) if forced is not None else None
        rc = self._lib.orc_markov_draft(_ptr(U), _ptr(W1), _ptr(W2), _ptr(anchors), _ptr(H), B, K, V,
                                      r, float(temperature), int(seed), b0, nb, _ptr(forced),
                                      _ptr(tokens), _ptr(logprobs), _ptr(margins), _ptr(flp))
        if rc != 0:
            raise ValueError("oracle markov_draft rejected its arguments")
        out = dict(tokens=tokens, logprobs=logprobs, margins=margins)
        if forced is not None:
            out["forced_logprobs"] = flp
        return out

    def markov_logits(self, U, W1, W2, prev, *, temperature: float = 1.0, H=None, b0: int = 0,
                      nb: Optional[int] = None) -> dict:
        """Teacher-forced calibrated logits [nb, K, V] (fp64) and lse [nb, K]."""
        U = _c(U, np.float32)
        B, K, V = U.shape
        r = 0 if W1 is None else W1.shape[1]
        W1 = _c(W1, np.uint16) if r > 0 else np.zeros((V, 1), np.uint16)
        W2 = _c(W2, np.uint16) if r > 0 else np.zeros((1, V), np.uint16)
        prev = _c(prev, np.int32)
        H = _c(H, np.float64)
        nb = B - b0 if nb is None else nb
        logits = np.zeros((nb, K, V), np.float64)
        lse = np.zeros((nb, K), np.float64)
        rc = self._lib.orc_markov_logits(_ptr(U), _ptr(W1), _ptr(W2), _ptr(prev), _ptr(H), B, K, V, r,
                                       float(temperature), b0, nb, _ptr(logits), _ptr(lse))
        if rc != 0:
            raise ValueError("oracle markov_logits rejected its arguments")
        return dict(logits=logits, lse=lse)

    def rnn_draft(self, U, W1, W2, anchors, A, *, G=None, temperature: float, seed: int,
                  b0: int = 0, nb: Optional[int] = None, forced=None) -> dict:
        """The RNN head's draft: state s_k = A_k (.) s_{k-1} + G_k (.) W1[x_{k-1}] (G None:
        1), bias s_k W2.  A, G [B, K, r] gate values (fp64); outputs as markov_draft."""
        U = _c(U, np.float32)
        B, K, V = U.shape
        W1 = _c(W1, np.uint16)
        W2 = _c(W2, np.uint16)
        r = W1.shape[1]
        anchors = _c(anchors, np.int32)
        A = _c(A, np.float64)
        G = _c(G, np.float64)
        assert A.shape == (B, K, r)
        nb = B - b0 if nb is None else nb
        forced = _c(forced, np.int32)
        tokens = np.zeros((nb, K), np.int32)
        logprobs = np.zeros((nb, K), np.float64)
        margins = np.zeros((nb, K), np.float64)
        flp = np.zeros((nb, K), np.float64) if forced is not None else None
        rc = self._lib.orc_rnn_draft(_ptr(U), _ptr(W1), _ptr(W2), _ptr(anchors), _ptr(A), _ptr(G),
                                     B, K, V, r, float(temperature), int(seed), b0, nb,
                                     _ptr(forced), _ptr(tokens), _ptr(logprobs), _ptr(margins),
                                     _ptr(flp))
        if rc != 0:
            raise ValueError("oracle rnn_draft rejected its arguments")
        out = dict(tokens=tokens, logprobs=logprobs, margins=margins)
        if forced is not None:
            out["forced_logprobs"] = flp
        return out

    def rnn_logits(self, U, W1, W2, prev, A, *, G=None, temperature: float = 1.0, b0: int = 0,
                   nb: Optional[int] = None) -> dict:
        """Teacher-forced logits [nb, K, V] (fp64) and lse [nb, K] of the RNN head."""
        U = _c(U, np.float32)
        B, K, V = U.shape
        W1 = _c(W1, np.uint16)
        W2 = _c(W2, np.uint16)
        r = W1.shape[1]
        prev = _c(prev, np.int32)
        A = _c(A, np.float64)
        G = _c(G, np.float64)
        nb = B - b0 if nb is None else nb
        logits = np.zeros((nb, K, V), np.float64)
        lse = np.zeros((nb, K), np.float64)
        rc = self._lib.orc_rnn_logits(_ptr(U), _ptr(W1), _ptr(W2), _ptr(prev), _ptr(A), _ptr(G),
                                      B, K, V, r, float(temperature), b0, nb, _ptr(logits),
                                      _ptr(lse))
        if rc != 0:
            raise ValueError("oracle rnn_logits rejected its arguments")
        return dict(logits=logits, lse=lse)

    def confidence(self, h, W1, anchors, tokens, w, *, bias: float = 0.0, with_markov: bool = True,
                   threshold: float = 0.3, V: Optional[int] = None, tau=None) -> dict:
        """Confidence c_k (calibrated by per-position temperatures tau [K] when given),
        survival cumprod a_k and verify length per request."""
        h = _c(h, np.uint16)
        B, K, d = h.shape
        r = W1.shape[1] if (with_markov and W1 is not None) else 0
        V = (W1.shape[0] if W1 is not None else 1) if V is None else V
        W1c = _c(W1, np.uint16) if W1 is not None else np.zeros((1, 1), np.uint16)
        anchors = _c(anchors, np.int32)
        tokens = _c(tokens, np.int32)
        w = _c(w, np.uint16)
        conf = np.zeros((B, K), np.float64)
        cum = np.zeros((B, K), np.float64)
        vl = np.zeros(B, np.int32)
        tau = _c(tau, np.float64)
        rc = self._lib.orc_confidence(_ptr(h), _ptr(W1c), _ptr(anchors), _ptr(tokens), _ptr(w),
                                    float(bias), int(bool(with_markov)), B, K, d, r, V,
                                    float(threshold), _ptr(tau), _ptr(conf), _ptr(cum), _ptr(vl))
        if rc != 0:
            raise ValueError("oracle confidence rejected its arguments")
        return dict(conf=conf, cumprod=cum, verify_len=vl)

    def sts_fit(self, conf, label, *, lo: float = 1.0 / 64, hi: float = 64.0) -> dict:
        """Sequential temperature scaling: one temperature per position [K] from raw
        confidences and acceptance labels [N, K]."""
        conf = _c(conf, np.float32)
        label = _c(label, np.float32)
        N, K = conf.shape
        assert label.shape == (N, K)
        tau = np.zeros(K, np.float64)
        loss = np.zeros(K, np.float64)
        rc = self._lib.orc_sts_fit(_ptr(conf), _ptr(label), N, K, float(lo), float(hi), _ptr(tau),
                                   _ptr(loss))
        if rc != 0:
            raise ValueError("oracle sts_fit rejected its arguments")
        return dict(tau=tau, loss=loss)

    def topk(self, U, k: int = 16) -> dict:
        U = _c(U, np.float32)
        B, K, V = U.shape
        cand = np.zeros((B, K, k), np.int32)
        cval = np.zeros((B, K, k), np.float64)
        margin = np.zeros((B, K), np.float64)
        rc = self._lib.orc_topk(_ptr(U), B, K, V, k, _ptr(cand), _ptr(cval), _ptr(margin))
        if rc != 0:
            raise ValueError("oracle topk rejected its arguments")
        return dict(cand=cand, cval=cval, margin=margin)

    def pair_scores(self, cand, cval, A, Bt, anchors, *, V: int, H=None) -> np.ndarray:
        cand = _c(cand, np.int32)
        cval = _c(cval, np.float64)
        A = _c(A, np.uint16)
        Bt = _c(Bt, np.uint16)
        anchors = _c(anchors, np.int32)
        H = _c(H, np.float64)
        B, K, k = cand.shape
        r = A.shape[1]
        S = np.zeros((B, K, k, k), np.float64)
        rc = self._lib.orc_pair_scores(_ptr(cand), _ptr(cval), _ptr(A), _ptr(Bt), _ptr(anchors),
                                     _ptr(H), B, K, V, r, k, _ptr(S))
        if rc != 0:
            raise ValueError("oracle pair_scores rejected its arguments")
        return S

    def walk(self, cand, S, *, temperature: float, seed: int, b0: int = 0, nb: Optional[int] = None,
             forced=None) -> dict:
        cand = _c(cand, np.int32)
        S = _c(S, np.float64)
        B, K, k = cand.shape
        nb = B - b0 if nb is None else nb
        forced = _c(forced, np.int32)
        tokens = np.zeros((nb, K), np.int32)
        logprobs = np.zeros((nb, K), np.float64)
        margins = np.zeros((nb, K), np.float64)
        flp = np.zeros((nb, K), np.float64) if forced is not None else None
        rc = self._lib.orc_walk(_ptr(cand), _ptr(S), B, K, k, float(temperature), int(seed), b0, nb,
                              _ptr(forced), _ptr(tokens), _ptr(logprobs), _ptr(margins), _ptr(flp))
        if rc != 0:
            raise ValueError("oracle walk rejected its arguments")
        out = dict(tokens=tokens, logprobs=logprobs, margins=margins)
        if forced is not None:
            out["forced_logprobs"] = flp
        return out


def default() -> Oracle:
    """The oracle built from this directory's C source (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
        return _default


_default: Optional[Oracle] = None


def __getattr__(name):
    # module-level access (oracle.markov_draft, ...) goes to the default instance
    if name.startswith("_"):
        raise AttributeError(name)
    return getattr(default(), name)
