"""C-ABI contract: the library loads, exports every function include/dspark.h
declares, and rejects bad arguments on the host before touching a GPU.

No compute call reaches a kernel here: every call below fails argument
validation, which the library performs before checking the context.
"""

import ctypes
import os
import re

import pytest

from rank_markov_draft_gb300 import binding, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "dspark.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dspark_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("dspark_markov_draft", "dspark_gated_draft", "dspark_selector_scores",
                     "dspark_selector_walk", "dspark_confidence", "dspark_markov_logits"):
        assert required in names
    assert set(names) == set(binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in dspark.h but not exported"


def test_checked_library_loads_and_exports_every_declared_symbol(lib):
    """libdspark_debug.so (the draft kernel with its on-chip offset checks) is built
    beside the release library and offers the same boundary."""
    checked = binding.load(binding.DEBUG_LIB_PATH)
    assert checked is not lib
    for name in declared_functions():
        assert hasattr(checked, name), f"{name} missing from the checked library"
    assert checked.dspark_abi_version() == lib.dspark_abi_version()


def test_refuse_next_launch_needs_a_context(lib):
    assert lib.dspark_debug_refuse_next_launch(None) == binding.INVALID_ARG


def test_abi_version_and_strerror(lib):
    assert lib.dspark_abi_version() == 2
    for code in range(9):
        assert lib.dspark_strerror(code).decode() != "unknown status"


P = ctypes.c_void_p
GOOD = P(0x1000)           # 16-byte aligned, never dereferenced by the host checks
ODD = P(0x1004)            # misaligned


def draft(lib, ctx=None, U=GOOD, W1=GOOD, W2=GOOD, anchors=GOOD, B=4, K=16, V=4096, r=256,
          T=1.0, tokens=GOOD, logprobs=GOOD, conf=None):
    return lib.dspark_markov_draft(ctx, U, W1, W2, anchors, B, K, V, r, T, 0, tokens, logprobs,
                                   conf, None)


def test_draft_argument_checks(lib):
    E = binding
    assert draft(lib) == E.INVALID_ARG                       # valid args, NULL context
    assert draft(lib, U=None) == E.INVALID_ARG
    assert draft(lib, tokens=None) == E.INVALID_ARG
    assert draft(lib, B=0) == E.INVALID_ARG
    assert draft(lib, K=0) == E.INVALID_ARG
    assert draft(lib, K=65) == E.UNSUPPORTED
    assert draft(lib, V=4100) == E.UNSUPPORTED                # V % 8 != 0
    assert draft(lib, V=(1 << 18) + 8) == E.UNSUPPORTED
    assert draft(lib, r=17) == E.UNSUPPORTED
    assert draft(lib, r=272) == E.UNSUPPORTED
    assert draft(lib, r=-16) == E.INVALID_ARG
    assert draft(lib, r=0, W1=None, W2=None) == E.INVALID_ARG  # valid rank-0 args, NULL ctx
    assert draft(lib, W2=None) == E.INVALID_ARG
    assert draft(lib, T=-1.0) == E.INVALID_ARG
    assert draft(lib, T=float("nan")) == E.INVALID_ARG
    assert draft(lib, U=ODD) == E.INVALID_ARG


def test_confidence_with_markov_needs_a_markov_head(lib):
    """vLLM guide: rank 0 must be paired with --no-confidence-head-with-markov."""
    conf = binding.ConfArgs(GOOD, GOOD, 0.0, 2048, 1, 0.3, GOOD, GOOD, GOOD)
    assert draft(lib, r=0, W1=None, W2=None, conf=ctypes.byref(conf)) == binding.INVALID_ARG
    conf.with_markov = 0
    assert draft(lib, r=0, W1=None, W2=None, conf=ctypes.byref(conf)) == binding.INVALID_ARG
    conf.d = 2047
    assert draft(lib, r=0, W1=None, W2=None, conf=ctypes.byref(conf)) == binding.INVALID_ARG


def test_gate_and_selector_argument_checks(lib):
    E = binding
    g = lambda M=8, d=128, r=64, H=GOOD: lib.dspark_gate(None, GOOD, GOOD, M, d, r, H, None)
    assert g() == E.INVALID_ARG
    assert g(d=100) == E.UNSUPPORTED
    assert g(r=48) == E.UNSUPPORTED
    assert g(H=None) == E.INVALID_ARG
    s = lambda topk=16, V=4096, r=256: lib.dspark_selector_scores(
        None, GOOD, GOOD, GOOD, GOOD, None, None, 0, 2, 4, V, r, topk, GOOD, GOOD, GOOD, None)
    assert s() == E.INVALID_ARG
    assert s(topk=33) == E.UNSUPPORTED
    assert s(topk=0) == E.INVALID_ARG
    assert s(V=4098) == E.UNSUPPORTED
    w = lambda topk=16, T=1.0: lib.dspark_selector_walk(
        None, GOOD, GOOD, GOOD, GOOD, 2, 4, 4096, 256, topk, T, 0, GOOD, GOOD, None, None)
    assert w() == E.INVALID_ARG
    assert w(topk=40) == E.UNSUPPORTED
    assert w(T=-0.5) == E.INVALID_ARG


def test_context_creation_without_a_device(lib):
    import torch
    h = P()
    code = lib.dspark_ctx_create(ctypes.byref(h), 0, 1, 4096, 4)
    if torch.cuda.is_available():
        assert code == binding.OK
        lib.dspark_ctx_destroy(h)
    else:
        assert code == binding.NO_DEVICE
    assert lib.dspark_ctx_create(ctypes.byref(h), 0, 0, 4096, 4) == binding.INVALID_ARG
    assert lib.dspark_ctx_create(ctypes.byref(h), 0, 1, 4096, 65) == binding.UNSUPPORTED
    assert lib.dspark_get_status(None, None) == binding.INVALID_ARG


def test_verify_label_schedule_sts_argument_checks(lib):
    """Size limits of the verification, label, scheduler and STS calls are enforced on the
    host before the context is looked at (with a NULL context every other valid call
    returns INVALID_ARG, so only the size codes below tell the checks apart)."""
    E = binding
    v = lambda B=4, K=16, V=4096, r=256, Td=1.0, Tt=1.0: lib.dspark_verify(
        None, GOOD, GOOD, GOOD, GOOD, GOOD, None, None, 0, GOOD, GOOD, None, B, K, V, r, Td, Tt,
        0, GOOD, GOOD, None, None)
    assert v() == E.INVALID_ARG
    assert v(K=65) == E.UNSUPPORTED
    assert v(r=17) == E.UNSUPPORTED
    assert v(V=4100) == E.UNSUPPORTED
    assert v(Tt=-1.0) == E.INVALID_ARG
    a = lambda B=4, K=16, V=4096, r=256: lib.dspark_accept_label(
        None, GOOD, GOOD, GOOD, GOOD, GOOD, None, None, 0, GOOD, GOOD, B, K, V, r, 1.0, 1.0, GOOD,
        None)
    assert a() == E.INVALID_ARG
    assert a(K=65) == E.UNSUPPORTED
    assert a(r=272) == E.UNSUPPORTED
    s = lambda R=128, K=16, sps_len=None, A=GOOD: lib.dspark_schedule(
        None, A, R, K, GOOD, R * (K + 1) + 1 if sps_len is None else sps_len, GOOD, None, None)
    assert s() == E.INVALID_ARG
    assert s(R=1025, K=16) == E.UNSUPPORTED            # more than 16384 candidates
    assert s(R=70000, K=0, A=None) == E.UNSUPPORTED    # R above 65535
    assert s(R=5, K=0, A=None) == E.INVALID_ARG        # nothing to admit: only the context
    assert s(sps_len=128 * 17) == E.INVALID_ARG        # SPS one entry short
    f = lambda N=8192, K=16, lo=1.0 / 64, hi=64.0: lib.dspark_sts_fit(
        None, GOOD, GOOD, N, K, lo, hi, GOOD, None, None)
    assert f() == E.INVALID_ARG
    assert f(K=65) == E.UNSUPPORTED
    assert f(lo=2.0, hi=1.0) == E.INVALID_ARG


def test_noalloc_host_limits(lib):
    """The allocation-free draft checks its fixed limits on the host, before any CUDA call:
    16 positions (its scratch holds 16 key rows) and 16383 chunks of 128 requests (one
    14-bit key epoch per chunk)."""
    E = binding
    na = lambda B=4, K=16, V=4096, r=256, T=1.0, U=GOOD: lib.dspark_markov_draft_noalloc(
        U, GOOD, GOOD, GOOD, B, K, V, r, T, 0, GOOD, GOOD, None, None)
    assert na(K=17) == E.CAPACITY
    assert na(B=16383 * 128 + 1) == E.CAPACITY
    assert na(B=0) == E.INVALID_ARG
    assert na(U=None) == E.INVALID_ARG
    assert na(V=4100) == E.UNSUPPORTED
    assert na(r=17) == E.UNSUPPORTED
    assert na(T=-1.0) == E.INVALID_ARG
    assert na(U=ODD) == E.INVALID_ARG
