"""The context-free draft entry point that allocates no device memory.

Some callers may not allocate device memory themselves (a library running
inside a host framework that owns all device memory through its own pool, or
a serving loop that forbids cudaMalloc because it can synchronise the device);
dspark_markov_draft_noalloc serves them with scratch compiled into the
library.  These checks call it through the C ABI twice in a row and compare
each result with the context-based dspark_markov_draft on the same inputs, and
one call at the full vocabulary (one CTA per SM, the largest grid its fixed
scratch is sized for) with the context draft and the oracle.
This file is collected last so that a run stopping at the first failure has
already run every other test.
"""

import numpy as np
import pytest
import torch

import oracle
from rank_markov_draft_gb300 import binding, build
from synth import make_inputs
from tests.gpu_util import LOGPROB_TOL, bf, check_sequences, dev, host

pytestmark = pytest.mark.gpu


def test_noalloc_draft_matches_context_draft_on_two_calls_in_a_row():
    build.build()
    B, K, V, r = 130, 16, 4096, 256   # two request chunks, full block length
    inp = make_inputs(77, B, K, V, r)
    U, W1, W2, anchors = dev(inp.U), bf(inp.W1), bf(inp.W2), dev(inp.anchors)
    with binding.Context(0, B_max=B, V_max=V, K_max=K) as ctx:
        for call, (T, seed) in enumerate([(1.0, 11), (0.7, 12)]):
            ref = binding.markov_draft(ctx, U, W1, W2, anchors, temperature=T, seed=seed)
            tokens = torch.full((B, K), -1, dtype=torch.int32, device="cuda")
            logprobs = torch.zeros(B, K, dtype=torch.float32, device="cuda")
            status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
            binding.dspark_markov_draft_noalloc(U, W1, W2, anchors, B, K, V, r, T, seed, tokens,
                                                logprobs, device_status=status)
            torch.cuda.synchronize()
            assert ctx.status() == 0
            assert int(status.item()) == 0, f"call {call}: device status {int(status.item())}"
            assert torch.equal(tokens, ref["tokens"]), f"call {call}: tokens differ"
            err = (logprobs - ref["logprobs"]).abs().max().item()
            assert err <= LOGPROB_TOL, f"call {call}: max |dlogprob| {err:.3e}"


def _noalloc(U, W1, W2, anchors, B, K, V, r, T, seed):
    tokens = torch.full((B, K), -1, dtype=torch.int32, device="cuda")
    logprobs = torch.zeros(B, K, dtype=torch.float32, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    binding.dspark_markov_draft_noalloc(U, W1, W2, anchors, B, K, V, r, T, seed, tokens,
                                        logprobs, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    return tokens, logprobs


def test_noalloc_full_vocab_matches_context_draft_and_oracle():
    build.build()
    B, K, V, r = 1, 16, 151936, 256   # 2374 tiles: one CTA per SM
    inp = make_inputs(78, B, K, V, r)
    U, W1, W2, anchors = dev(inp.U), bf(inp.W1), bf(inp.W2), dev(inp.anchors)
    tokens, logprobs = _noalloc(U, W1, W2, anchors, B, K, V, r, 1.0, 5)
    with binding.Context(0, B_max=B, V_max=V, K_max=K) as ctx:
        ref = binding.markov_draft(ctx, U, W1, W2, anchors, temperature=1.0, seed=5)
        torch.cuda.synchronize()
        assert ctx.status() == 0
    assert torch.equal(tokens, ref["tokens"])
    assert (logprobs - ref["logprobs"]).abs().max().item() <= LOGPROB_TOL
    orc = oracle.markov_draft(inp.U, inp.W1, inp.W2, inp.anchors, temperature=1.0, seed=5)
    diverged, compared = check_sequences(host(tokens), host(logprobs), orc, what="noalloc")
    assert compared == K or diverged == 1


def test_noalloc_rejects_block_longer_than_its_scratch():
    lib = binding.load()
    g = torch.zeros(16, dtype=torch.int32, device="cuda")
    code = lib.dspark_markov_draft_noalloc(g.data_ptr(), g.data_ptr(), g.data_ptr(), g.data_ptr(),
                                           1, 17, 4096, 256, 1.0, 0, g.data_ptr(), g.data_ptr(),
                                           None, None)
    assert code == binding.CAPACITY
