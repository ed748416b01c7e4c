"""The context-free draft entry point that allocates no device memory.

Some callers may not allocate device memory themselves (a library running
inside a host framework that owns all device memory through its own pool, or
a serving loop that forbids cudaMalloc because it can synchronise the device);
dspark_markov_draft_noalloc serves them with scratch compiled into the
library.  These checks call it through the C ABI twice in a row and compare
each result with the context-based dspark_markov_draft on the same inputs.
This file is collected last so that a run stopping at the first failure has
already run every other test.
"""

import numpy as np
import pytest
import torch

from rank_markov_draft_gb300 import binding, build
from synth import make_inputs
from tests.gpu_util import LOGPROB_TOL, bf, dev

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


def test_noalloc_rejects_block_longer_than_its_scratch():
    lib = binding.load()
    g = torch.zeros(16, dtype=torch.int32, device="cuda")
    code = lib.dspark_markov_draft_noalloc(g.data_ptr(), g.data_ptr(), g.data_ptr(), g.data_ptr(),
                                           1, 17, 4096, 256, 1.0, 0, g.data_ptr(), g.data_ptr(),
                                           None, None)
    assert code == binding.CAPACITY
