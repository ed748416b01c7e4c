"""ctypes binding of libdspark (include/dspark.h).

Argument marshalling only: every step of the hot path runs in the library's
CUDA kernels.  The low-level functions carry the C names (``dspark_*``) and
take torch tensors (device memory, caller-owned) plus an optional CUDA
stream; the convenience wrappers below them allocate the outputs.  There is no
CPU fallback: if the compiled library is missing, loading raises.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libdspark.so")
# the same library with the draft kernel's device-side offset checks compiled in
DEBUG_LIB_PATH = os.path.join(_HERE, "_build", "libdspark_debug.so")

STATUS = {
    0: "DSPARK_OK", 1: "DSPARK_ERR_INVALID_ARG", 2: "DSPARK_ERR_UNSUPPORTED",
    3: "DSPARK_ERR_CUDA", 4: "DSPARK_ERR_TIMEOUT", 5: "DSPARK_ERR_DEVICE_OOB",
    6: "DSPARK_ERR_NO_DEVICE", 7: "DSPARK_ERR_CTX_POISONED", 8: "DSPARK_ERR_CAPACITY",
}
OK, INVALID_ARG, UNSUPPORTED, CUDA, TIMEOUT, DEVICE_OOB, NO_DEVICE, POISONED, CAPACITY = range(9)

# Functions declared in include/dspark.h (checked against the header by the tests).
EXPORTS = (
    "dspark_ctx_create", "dspark_ctx_destroy", "dspark_ctx_reset", "dspark_get_status",
    "dspark_debug_set", "dspark_debug_refuse_next_launch", "dspark_debug_trace", "dspark_strerror",
    "dspark_abi_version", "dspark_last_launch_count",
    "dspark_markov_draft", "dspark_gated_draft", "dspark_gate", "dspark_selector_scores",
    "dspark_selector_walk", "dspark_confidence", "dspark_markov_logits",
    "dspark_markov_draft_noalloc", "dspark_verify", "dspark_schedule", "dspark_accept_label",
    "dspark_sts_fit", "dspark_rnn_draft", "dspark_rnn_logits",
)


class DSparkError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)} ({strerror(code)})")


class ConfArgs(ctypes.Structure):
    _fields_ = [
        ("h", ctypes.c_void_p), ("w", ctypes.c_void_p), ("bias", ctypes.c_float),
        ("d", ctypes.c_int), ("with_markov", ctypes.c_int), ("threshold", ctypes.c_float),
        ("conf", ctypes.c_void_p), ("cumprod", ctypes.c_void_p), ("verify_len", ctypes.c_void_p),
        ("tau", ctypes.c_void_p),
    ]


_libs = {}


def load(path: str = LIB_PATH):
    """Load libdspark.so (or its checked twin); raise if it has not been built."""
    if path in _libs:
        return _libs[path]
    if not os.path.exists(path):
        raise RuntimeError(f"{os.path.basename(path)} not found at {path}: build it first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    P, I, F, U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_uint64
    sig = {
        "dspark_ctx_create": [ctypes.POINTER(P), I, I, I, I],
        "dspark_ctx_destroy": [P],
        "dspark_ctx_reset": [P, P],
        "dspark_get_status": [P, ctypes.POINTER(I)],
        "dspark_debug_set": [P, I, I],
        "dspark_debug_refuse_next_launch": [P],
        "dspark_debug_trace": [P, P, ctypes.c_int64],
        "dspark_strerror": [I],
        "dspark_abi_version": [],
        "dspark_last_launch_count": [P],
        "dspark_markov_draft": [P, P, P, P, P, I, I, I, I, F, U64, P, P, P, P],
        "dspark_gated_draft": [P, P, P, P, P, P, P, I, I, I, I, I, F, U64, P, P, P, P],
        "dspark_gate": [P, P, P, I, I, I, P, P],
        "dspark_selector_scores": [P, P, P, P, P, P, P, I, I, I, I, I, I, P, P, P, P],
        "dspark_selector_walk": [P, P, P, P, P, I, I, I, I, I, F, U64, P, P, P, P],
        "dspark_confidence": [P, P, P, P, P, P, F, I, I, I, I, I, I, F, P, P, P, P, P],
        "dspark_markov_logits": [P, P, P, P, P, P, P, I, I, I, I, I, F, P, P, P],
        "dspark_markov_draft_noalloc": [P, P, P, P, I, I, I, I, F, U64, P, P, P, P],
        "dspark_verify": [P, P, P, P, P, P, P, P, I, P, P, P, I, I, I, I, F, F, U64, P, P, P, P],
        "dspark_schedule": [P, P, I, I, P, I, P, P, P],
        "dspark_accept_label": [P, P, P, P, P, P, P, P, I, P, P, I, I, I, I, F, F, P, P],
        "dspark_sts_fit": [P, P, P, I, I, F, F, P, P, P],
        "dspark_rnn_draft": [P, P, P, P, P, P, P, P, I, I, I, I, I, F, U64, P, P, P, P],
        "dspark_rnn_logits": [P, P, P, P, P, P, P, P, I, I, I, I, I, F, P, P, P],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_char_p if name == "dspark_strerror" else ctypes.c_int
    _libs[path] = lib
    return lib


def strerror(code: int) -> str:
    try:
        return load().dspark_strerror(int(code)).decode()
    except RuntimeError:
        return "library not loaded"


# ----------------------------------------------------------------- marshalling
_BF16 = (torch.bfloat16, torch.int16, torch.uint16)


def _ptr(t: Optional[torch.Tensor], dtypes=None, name: str = "tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if dtypes is not None and t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if t.device.type != "cuda":
        raise ValueError(f"{name}: must live in CUDA device memory")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(code: int, where: str):
    if code != OK:
        raise DSparkError(code, where)


class Context:
    """A dspark_ctx: per-device scratch for B_max requests, K_max positions, V_max tokens."""

    def __init__(self, device: int = 0, B_max: int = 128, V_max: int = 151936, K_max: int = 16,
                 checked: bool = False):
        # checked: run through libdspark_debug.so, whose draft kernel checks its on-chip
        # offsets (a failed check is reported as DSPARK_ERR_DEVICE_OOB)
        self.lib = load(DEBUG_LIB_PATH if checked else LIB_PATH)
        self.device = device
        self.B_max, self.V_max, self.K_max = B_max, V_max, K_max
        h = ctypes.c_void_p()
        _check(self.lib.dspark_ctx_create(ctypes.byref(h), device, B_max, V_max, K_max),
               "dspark_ctx_create")
        self.handle = h

    def close(self):
        if getattr(self, "handle", None):
            torch.cuda.synchronize(self.device)
            self.lib.dspark_ctx_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def reset(self, stream=None):
        _check(self.lib.dspark_ctx_reset(self.handle, _stream(stream, self.device)),
               "dspark_ctx_reset")

    def status(self) -> int:
        v = ctypes.c_int(0)
        _check(self.lib.dspark_get_status(self.handle, ctypes.byref(v)), "dspark_get_status")
        return v.value

    def debug_set(self, cta: int = -1, timeout_ms: int = 0):
        _check(self.lib.dspark_debug_set(self.handle, cta, timeout_ms), "dspark_debug_set")

    def refuse_next_launch(self):
        """The next draft-kernel launch is refused by the CUDA runtime (a test aid)."""
        _check(self.lib.dspark_debug_refuse_next_launch(self.handle),
               "dspark_debug_refuse_next_launch")

    def trace_next(self, buf: Optional[torch.Tensor]):
        """Record the next draft launch's phase stamps into buf (int64, >= grid * K * 8)."""
        if buf is None:
            _check(self.lib.dspark_debug_trace(self.handle, None, 0), "dspark_debug_trace")
            return
        _check(self.lib.dspark_debug_trace(self.handle, _ptr(buf, (torch.int64,), "trace"),
                                           buf.numel()), "dspark_debug_trace")

    @property
    def last_launches(self) -> int:
        return int(self.lib.dspark_last_launch_count(self.handle))


@dataclass
class Confidence:
    """Inputs and outputs of the confidence head (dspark_conf_args)."""
    h: torch.Tensor            # [B, K, d] bf16
    w: torch.Tensor            # [d + r] (with_markov) or [d] bf16
    bias: float = 0.0
    with_markov: bool = True
    threshold: float = 0.3
    conf: Optional[torch.Tensor] = None       # out [B, K] fp32
    cumprod: Optional[torch.Tensor] = None    # out [B, K] fp32
    verify_len: Optional[torch.Tensor] = None  # out [B] int32
    tau: Optional[torch.Tensor] = None         # [K] fp32 STS temperatures (None: all 1)

    def allocate(self, B: int, K: int):
        dev = self.h.device
        if self.conf is None:
            self.conf = torch.empty(B, K, dtype=torch.float32, device=dev)
        if self.cumprod is None:
            self.cumprod = torch.empty(B, K, dtype=torch.float32, device=dev)
        if self.verify_len is None:
            self.verify_len = torch.empty(B, dtype=torch.int32, device=dev)
        return self

    def struct(self) -> ConfArgs:
        return ConfArgs(_ptr(self.h, _BF16, "conf.h"), _ptr(self.w, _BF16, "conf.w"),
                        float(self.bias), int(self.h.shape[-1]), int(bool(self.with_markov)),
                        float(self.threshold), _ptr(self.conf, (torch.float32,), "conf.conf"),
                        _ptr(self.cumprod, (torch.float32,), "conf.cumprod"),
                        _ptr(self.verify_len, (torch.int32,), "conf.verify_len"),
                        _ptr(self.tau, (torch.float32,), "conf.tau"))


def _conf_ref(conf: Optional[Confidence]):
    return None if conf is None else ctypes.byref(conf.struct())


# ------------------------------------------------------- C-named entry points
def dspark_markov_draft(ctx: Context, U, W1, W2, anchors, B, K, V, r, temperature, seed,
                        tokens, logprobs, conf: Optional[Confidence] = None, stream=None):
    code = ctx.lib.dspark_markov_draft(
        ctx.handle, _ptr(U, (torch.float32,), "U"), _ptr(W1, _BF16, "W1"),
        _ptr(W2, _BF16, "W2"), _ptr(anchors, (torch.int32,), "anchors"), B, K, V, r,
        float(temperature), int(seed) & (2 ** 64 - 1), _ptr(tokens, (torch.int32,), "tokens"),
        _ptr(logprobs, (torch.float32,), "logprobs"), _conf_ref(conf), _stream(stream, ctx.device))
    _check(code, "dspark_markov_draft")


def dspark_gated_draft(ctx: Context, U, W1, W2, anchors, h, Wg, d, B, K, V, r, temperature,
                       seed, tokens, logprobs, conf: Optional[Confidence] = None, stream=None):
    code = ctx.lib.dspark_gated_draft(
        ctx.handle, _ptr(U, (torch.float32,), "U"), _ptr(W1, _BF16, "W1"),
        _ptr(W2, _BF16, "W2"), _ptr(anchors, (torch.int32,), "anchors"), _ptr(h, _BF16, "h"),
        _ptr(Wg, _BF16, "Wg"), d, B, K, V, r, float(temperature), int(seed) & (2 ** 64 - 1),
        _ptr(tokens, (torch.int32,), "tokens"), _ptr(logprobs, (torch.float32,), "logprobs"),
        _conf_ref(conf), _stream(stream, ctx.device))
    _check(code, "dspark_gated_draft")


def dspark_rnn_draft(ctx: Context, U, W1, W2, anchors, h, Wa, Wg, d, B, K, V, r, temperature,
                     seed, tokens, logprobs, conf: Optional[Confidence] = None, stream=None):
    code = ctx.lib.dspark_rnn_draft(
        ctx.handle, _ptr(U, (torch.float32,), "U"), _ptr(W1, _BF16, "W1"),
        _ptr(W2, _BF16, "W2"), _ptr(anchors, (torch.int32,), "anchors"), _ptr(h, _BF16, "h"),
        _ptr(Wa, _BF16, "Wa"), _ptr(Wg, _BF16, "Wg"), d, B, K, V, r, float(temperature),
        int(seed) & (2 ** 64 - 1), _ptr(tokens, (torch.int32,), "tokens"),
        _ptr(logprobs, (torch.float32,), "logprobs"), _conf_ref(conf), _stream(stream, ctx.device))
    _check(code, "dspark_rnn_draft")


def dspark_rnn_logits(ctx: Context, U, W1, W2, prev_tokens, h, Wa, Wg, d, B, K, V, r, temperature,
                      logits, lse, stream=None):
    code = ctx.lib.dspark_rnn_logits(
        ctx.handle, _ptr(U, (torch.float32,), "U"), _ptr(W1, _BF16, "W1"), _ptr(W2, _BF16, "W2"),
        _ptr(prev_tokens, (torch.int32,), "prev_tokens"), _ptr(h, _BF16, "h"),
        _ptr(Wa, _BF16, "Wa"), _ptr(Wg, _BF16, "Wg"), d, B, K, V, r, float(temperature),
        _ptr(logits, (torch.float32,), "logits"), _ptr(lse, (torch.float32,), "lse"),
        _stream(stream, ctx.device))
    _check(code, "dspark_rnn_logits")


def dspark_gate(ctx: Context, h, Wg, M, d, r, H, stream=None):
    code = ctx.lib.dspark_gate(ctx.handle, _ptr(h, _BF16, "h"), _ptr(Wg, _BF16, "Wg"), M, d, r,
                               _ptr(H, (torch.float32,), "H"), _stream(stream, ctx.device))
    _check(code, "dspark_gate")


def dspark_selector_scores(ctx: Context, U, A, Bt, anchors, h, Wg, d, B, K, V, r, topk, cand,
                           cand_U, scores, stream=None):
    code = ctx.lib.dspark_selector_scores(
        ctx.handle, _ptr(U, (torch.float32,), "U"), _ptr(A, _BF16, "A"), _ptr(Bt, _BF16, "Bt"),
        _ptr(anchors, (torch.int32,), "anchors"), _ptr(h, _BF16, "h"), _ptr(Wg, _BF16, "Wg"), d,
        B, K, V, r, topk, _ptr(cand, (torch.int32,), "cand"),
        _ptr(cand_U, (torch.float32,), "cand_U"), _ptr(scores, (torch.float32,), "scores"),
        _stream(stream, ctx.device))
    _check(code, "dspark_selector_scores")


def dspark_selector_walk(ctx: Context, cand, scores, anchors, A, B, K, V, r, topk, temperature,
                         seed, tokens, logprobs, conf: Optional[Confidence] = None, stream=None):
    code = ctx.lib.dspark_selector_walk(
        ctx.handle, _ptr(cand, (torch.int32,), "cand"), _ptr(scores, (torch.float32,), "scores"),
        _ptr(anchors, (torch.int32,), "anchors"), _ptr(A, _BF16, "A"), B, K, V, r, topk,
        float(temperature), int(seed) & (2 ** 64 - 1), _ptr(tokens, (torch.int32,), "tokens"),
        _ptr(logprobs, (torch.float32,), "logprobs"), _conf_ref(conf), _stream(stream, ctx.device))
    _check(code, "dspark_selector_walk")


def dspark_confidence(ctx: Context, h, W1, anchors, tokens, w, bias, with_markov, B, K, d, r, V,
                      threshold, tau, conf, cumprod, verify_len, stream=None):
    code = ctx.lib.dspark_confidence(
        ctx.handle, _ptr(h, _BF16, "h"), _ptr(W1, _BF16, "W1"),
        _ptr(anchors, (torch.int32,), "anchors"), _ptr(tokens, (torch.int32,), "tokens"),
        _ptr(w, _BF16, "w"), float(bias), int(bool(with_markov)), B, K, d, r, V, float(threshold),
        _ptr(tau, (torch.float32,), "tau"), _ptr(conf, (torch.float32,), "conf"), _ptr(cumprod, (torch.float32,), "cumprod"),
        _ptr(verify_len, (torch.int32,), "verify_len"), _stream(stream, ctx.device))
    _check(code, "dspark_confidence")


def dspark_markov_logits(ctx: Context, U, W1, W2, prev_tokens, h, Wg, d, B, K, V, r,
                         temperature, logits, lse, stream=None):
    code = ctx.lib.dspark_markov_logits(
        ctx.handle, _ptr(U, (torch.float32,), "U"), _ptr(W1, _BF16, "W1"), _ptr(W2, _BF16, "W2"),
        _ptr(prev_tokens, (torch.int32,), "prev_tokens"), _ptr(h, _BF16, "h"),
        _ptr(Wg, _BF16, "Wg"), d, B, K, V, r, float(temperature),
        _ptr(logits, (torch.float32,), "logits"), _ptr(lse, (torch.float32,), "lse"),
        _stream(stream, ctx.device))
    _check(code, "dspark_markov_logits")


def dspark_verify(ctx: Context, P, U, W1, W2, anchors, h, Wg, d, tokens, draft_logprobs, ell,
                  B, K, V, r, draft_temperature, target_temperature, seed, n_acc, next_token,
                  accept_prob, stream=None):
    code = ctx.lib.dspark_verify(
        ctx.handle, _ptr(P, (torch.float32,), "P"), _ptr(U, (torch.float32,), "U"),
        _ptr(W1, _BF16, "W1"), _ptr(W2, _BF16, "W2"), _ptr(anchors, (torch.int32,), "anchors"),
        _ptr(h, _BF16, "h"), _ptr(Wg, _BF16, "Wg"), d, _ptr(tokens, (torch.int32,), "tokens"),
        _ptr(draft_logprobs, (torch.float32,), "draft_logprobs"), _ptr(ell, (torch.int32,), "ell"),
        B, K, V, r, float(draft_temperature), float(target_temperature), int(seed) & (2 ** 64 - 1),
        _ptr(n_acc, (torch.int32,), "n_acc"), _ptr(next_token, (torch.int32,), "next_token"),
        _ptr(accept_prob, (torch.float32,), "accept_prob"), _stream(stream, ctx.device))
    _check(code, "dspark_verify")


def dspark_accept_label(ctx: Context, P, U, W1, W2, anchors, h, Wg, d, tokens, draft_logprobs,
                        B, K, V, r, draft_temperature, target_temperature, label, stream=None):
    code = ctx.lib.dspark_accept_label(
        ctx.handle, _ptr(P, (torch.float32,), "P"), _ptr(U, (torch.float32,), "U"),
        _ptr(W1, _BF16, "W1"), _ptr(W2, _BF16, "W2"), _ptr(anchors, (torch.int32,), "anchors"),
        _ptr(h, _BF16, "h"), _ptr(Wg, _BF16, "Wg"), d, _ptr(tokens, (torch.int32,), "tokens"),
        _ptr(draft_logprobs, (torch.float32,), "draft_logprobs"), B, K, V, r,
        float(draft_temperature), float(target_temperature), _ptr(label, (torch.float32,), "label"),
        _stream(stream, ctx.device))
    _check(code, "dspark_accept_label")


def dspark_sts_fit(ctx: Context, conf, label, N, K, tau_lo, tau_hi, tau, loss, stream=None):
    code = ctx.lib.dspark_sts_fit(
        ctx.handle, _ptr(conf, (torch.float32,), "conf"), _ptr(label, (torch.float32,), "label"),
        N, K, float(tau_lo), float(tau_hi), _ptr(tau, (torch.float32,), "tau"),
        _ptr(loss, (torch.float32,), "loss"), _stream(stream, ctx.device))
    _check(code, "dspark_sts_fit")


def dspark_schedule(ctx: Context, a, R, K, sps, ell, theta, stream=None):
    code = ctx.lib.dspark_schedule(
        ctx.handle, _ptr(a, (torch.float32,), "a"), R, K, _ptr(sps, (torch.float32,), "sps"),
        int(sps.numel()), _ptr(ell, (torch.int32,), "ell"), _ptr(theta, (torch.float32,), "theta"),
        _stream(stream, ctx.device))
    _check(code, "dspark_schedule")


def dspark_markov_draft_noalloc(U, W1, W2, anchors, B, K, V, r, temperature, seed, tokens,
                                logprobs, device_status=None, stream=None):
    """Context-free draft that allocates no device memory (scratch compiled into the library).

    For callers that may not allocate device memory themselves; the current CUDA
    device must hold every tensor.  Calls that overlap on the GPU race on the
    shared scratch.  device_status: optional int32 device tensor receiving the
    launch's device status.
    """
    lib = load()
    code = lib.dspark_markov_draft_noalloc(
        _ptr(U, (torch.float32,), "U"), _ptr(W1, _BF16, "W1"), _ptr(W2, _BF16, "W2"),
        _ptr(anchors, (torch.int32,), "anchors"), B, K, V, r, float(temperature),
        int(seed) & (2 ** 64 - 1), _ptr(tokens, (torch.int32,), "tokens"),
        _ptr(logprobs, (torch.float32,), "logprobs"),
        _ptr(device_status, (torch.int32,), "device_status"),
        _stream(stream, U.device))
    _check(code, "dspark_markov_draft_noalloc")


# ------------------------------------------------------ allocating wrappers
def _rank(W1) -> int:
    return 0 if W1 is None else int(W1.shape[1])


def markov_draft(ctx: Context, U, W1, W2, anchors, *, temperature=1.0, seed=0, h=None, Wg=None,
                 conf: Optional[Confidence] = None, stream=None) -> dict:
    """Vanilla (h, Wg None) or gated draft; returns tokens and logprobs [B, K]."""
    B, K, V = U.shape
    r = _rank(W1)
    tokens = torch.empty(B, K, dtype=torch.int32, device=U.device)
    logprobs = torch.empty(B, K, dtype=torch.float32, device=U.device)
    if conf is not None:
        conf.allocate(B, K)
    if h is None and Wg is None:
        dspark_markov_draft(ctx, U, W1, W2, anchors, B, K, V, r, temperature, seed, tokens,
                            logprobs, conf, stream)
    else:
        dspark_gated_draft(ctx, U, W1, W2, anchors, h, Wg, int(h.shape[-1]), B, K, V, r,
                           temperature, seed, tokens, logprobs, conf, stream)
    out = dict(tokens=tokens, logprobs=logprobs)
    if conf is not None:
        out.update(conf=conf.conf, cumprod=conf.cumprod, verify_len=conf.verify_len)
    return out


def gate(ctx: Context, h, Wg, stream=None) -> torch.Tensor:
    d, r = Wg.shape
    M = h.numel() // d
    H = torch.empty(*h.shape[:-1], r, dtype=torch.float32, device=h.device)
    dspark_gate(ctx, h, Wg, M, d, r, H, stream)
    return H


def selector_scores(ctx: Context, U, A, Bt, anchors, *, topk=16, h=None, Wg=None,
                    stream=None) -> dict:
    B, K, V = U.shape
    r = int(A.shape[1])
    cand = torch.empty(B, K, topk, dtype=torch.int32, device=U.device)
    cand_U = torch.empty(B, K, topk, dtype=torch.float32, device=U.device)
    scores = torch.empty(B, K, topk, topk, dtype=torch.float32, device=U.device)
    d = 0 if h is None else int(h.shape[-1])
    dspark_selector_scores(ctx, U, A, Bt, anchors, h, Wg, d, B, K, V, r, topk, cand, cand_U,
                           scores, stream)
    return dict(cand=cand, cand_U=cand_U, scores=scores)


def selector_walk(ctx: Context, cand, scores, anchors, *, V, A=None, temperature=1.0, seed=0,
                  conf: Optional[Confidence] = None, stream=None) -> dict:
    B, K, topk = cand.shape
    r = 0 if A is None else int(A.shape[1])
    tokens = torch.empty(B, K, dtype=torch.int32, device=cand.device)
    logprobs = torch.empty(B, K, dtype=torch.float32, device=cand.device)
    if conf is not None:
        conf.allocate(B, K)
    dspark_selector_walk(ctx, cand, scores, anchors, A, B, K, V, r, topk, temperature, seed,
                         tokens, logprobs, conf, stream)
    out = dict(tokens=tokens, logprobs=logprobs)
    if conf is not None:
        out.update(conf=conf.conf, cumprod=conf.cumprod, verify_len=conf.verify_len)
    return out


def confidence(ctx: Context, h, W1, anchors, tokens, w, *, V, bias=0.0, with_markov=True,
               threshold=0.3, tau=None, stream=None) -> dict:
    B, K, d = h.shape
    r = _rank(W1) if with_markov else 0
    conf = torch.empty(B, K, dtype=torch.float32, device=h.device)
    cum = torch.empty(B, K, dtype=torch.float32, device=h.device)
    vl = torch.empty(B, dtype=torch.int32, device=h.device)
    dspark_confidence(ctx, h, W1 if with_markov else None, anchors, tokens, w, bias, with_markov,
                      B, K, d, r, V, threshold, tau, conf, cum, vl, stream)
    return dict(conf=conf, cumprod=cum, verify_len=vl)


def verify(ctx: Context, P, U, W1, W2, anchors, tokens, draft_logprobs, *, draft_temperature,
           target_temperature, seed=0, ell=None, h=None, Wg=None, stream=None) -> dict:
    """Speculative verification of drafted tokens [B, K] against target logits P [B, K+1, V]."""
    B, K, V = U.shape
    r = _rank(W1)
    n_acc = torch.empty(B, dtype=torch.int32, device=U.device)
    next_token = torch.empty(B, dtype=torch.int32, device=U.device)
    accept_prob = torch.empty(B, K, dtype=torch.float32, device=U.device)
    d = 0 if h is None else int(h.shape[-1])
    dspark_verify(ctx, P, U, W1, W2, anchors, h, Wg, d, tokens, draft_logprobs, ell, B, K, V, r,
                  draft_temperature, target_temperature, seed, n_acc, next_token, accept_prob,
                  stream)
    return dict(n_acc=n_acc, next_token=next_token, accept_prob=accept_prob)


def accept_label(ctx: Context, P, U, W1, W2, anchors, tokens, draft_logprobs=None, *,
                 draft_temperature, target_temperature, h=None, Wg=None, stream=None):
    """Acceptance label 1 - TV(draft, target) [B, K] of drafted tokens [B, K]."""
    B, K, V = U.shape
    r = _rank(W1)
    label = torch.empty(B, K, dtype=torch.float32, device=U.device)
    d = 0 if h is None else int(h.shape[-1])
    dspark_accept_label(ctx, P, U, W1, W2, anchors, h, Wg, d, tokens, draft_logprobs, B, K, V, r,
                        draft_temperature, target_temperature, label, stream)
    return label


def sts_fit(ctx: Context, conf, label, *, tau_lo=1.0 / 64, tau_hi=64.0, stream=None) -> dict:
    """Sequential temperature scaling: temperatures [K] from raw confidences and labels [N, K]."""
    N, K = conf.shape
    tau = torch.empty(K, dtype=torch.float32, device=conf.device)
    loss = torch.empty(K, dtype=torch.float32, device=conf.device)
    dspark_sts_fit(ctx, conf, label, N, K, tau_lo, tau_hi, tau, loss, stream)
    return dict(tau=tau, loss=loss)


def schedule(ctx: Context, a, sps, stream=None) -> dict:
    """Greedy load-aware verify lengths: survival a [R, K], SPS(B) table [>= R (K+1) + 1]."""
    R, K = a.shape
    ell = torch.empty(R, dtype=torch.int32, device=a.device)
    theta = torch.empty(1, dtype=torch.float32, device=a.device)
    dspark_schedule(ctx, a, R, K, sps, ell, theta, stream)
    return dict(ell=ell, theta=theta)


def rnn_draft(ctx: Context, U, W1, W2, anchors, h, Wa, *, Wg=None, temperature=1.0, seed=0,
              conf: Optional[Confidence] = None, stream=None) -> dict:
    """The RNN head's draft (decay gate from Wa, input gate from Wg or 1); returns tokens and
    logprobs [B, K] (and the confidence head's outputs when conf is given)."""
    B, K, V = U.shape
    r = _rank(W1)
    tokens = torch.empty(B, K, dtype=torch.int32, device=U.device)
    logprobs = torch.empty(B, K, dtype=torch.float32, device=U.device)
    if conf is not None:
        conf.allocate(B, K)
    dspark_rnn_draft(ctx, U, W1, W2, anchors, h, Wa, Wg, int(h.shape[-1]), B, K, V, r,
                     temperature, seed, tokens, logprobs, conf, stream)
    out = dict(tokens=tokens, logprobs=logprobs)
    if conf is not None:
        out.update(conf=conf.conf, cumprod=conf.cumprod, verify_len=conf.verify_len)
    return out


def rnn_logits(ctx: Context, U, W1, W2, prev_tokens, h, Wa, *, Wg=None, temperature=1.0,
               stream=None) -> dict:
    """The RNN head's teacher-forced logits [B, K, V] and LSE [B, K]."""
    B, K, V = U.shape
    r = _rank(W1)
    logits = torch.empty(B, K, V, dtype=torch.float32, device=U.device)
    lse = torch.empty(B, K, dtype=torch.float32, device=U.device)
    dspark_rnn_logits(ctx, U, W1, W2, prev_tokens, h, Wa, Wg, int(h.shape[-1]), B, K, V, r,
                      temperature, logits, lse, stream)
    return dict(logits=logits, lse=lse)


def markov_logits(ctx: Context, U, W1, W2, prev_tokens, *, temperature=1.0, h=None, Wg=None,
                  stream=None) -> dict:
    B, K, V = U.shape
    r = _rank(W1)
    logits = torch.empty(B, K, V, dtype=torch.float32, device=U.device)
    lse = torch.empty(B, K, dtype=torch.float32, device=U.device)
    d = 0 if h is None else int(h.shape[-1])
    dspark_markov_logits(ctx, U, W1, W2, prev_tokens, h, Wg, d, B, K, V, r, temperature, logits,
                         lse, stream)
    return dict(logits=logits, lse=lse)
