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
