"""Failure detection without a GPU fault.

The draft kernel bounds every wait.  A testing knob makes one CTA skip its
grid-barrier arrival at the first position, so every other CTA's (shortened)
wait runs out: the kernel must exit cleanly, report DSPARK_ERR_TIMEOUT through
the status word, poison the context, and leave the device usable; after
dspark_ctx_reset the same call must again agree with a clean context.
Nothing here traps, faults or hangs the GPU: the waits end after 200 ms.
"""

import pytest
import torch

from rank_markov_draft_gb300 import binding
from synth import make_inputs
from tests.gpu_util import bf, dev

pytestmark = pytest.mark.gpu


def test_barrier_timeout_is_reported_and_recoverable():
    B, K, V, r = 4, 3, 4096, 256
    inp = make_inputs(5, B, K, V, r)
    args = (dev(inp.U), bf(inp.W1), bf(inp.W2), dev(inp.anchors))
    with binding.Context(0, B_max=B, V_max=V, K_max=K) as ctx:
        clean = binding.markov_draft(ctx, *args, temperature=1.0, seed=3)
        torch.cuda.synchronize()
        assert ctx.status() == 0
        ctx.debug_set(cta=0, timeout_ms=200)
        binding.markov_draft(ctx, *args, temperature=1.0, seed=3)
        torch.cuda.synchronize()          # returns: the kernel exited on its own
        assert ctx.status() == binding.TIMEOUT
        with pytest.raises(binding.DSparkError) as err:
            binding.markov_draft(ctx, *args, temperature=1.0, seed=3)
        assert err.value.code == binding.POISONED
        ctx.reset()
        again = binding.markov_draft(ctx, *args, temperature=1.0, seed=3)
        torch.cuda.synchronize()
        assert ctx.status() == 0
        assert torch.equal(again["tokens"], clean["tokens"])
        assert torch.equal(again["logprobs"], clean["logprobs"])
