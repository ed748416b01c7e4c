"""Failure detection without a GPU fault.

The draft kernel bounds every wait.  A testing knob makes one CTA skip its
grid-barrier arrival at the first position, so every other CTA's (shortened)
wait runs out: the kernel must exit cleanly, report DSPARK_ERR_TIMEOUT through
the status word, poison the context, and leave the device usable; after
dspark_ctx_reset the same call must again agree with a clean context.
Nothing here traps, faults or hangs the GPU: the waits end after 200 ms.

Also here: a launch the CUDA runtime refuses on the host, and the debug library
(the draft kernel with its on-chip offset checks) on in-range work.
"""

import numpy as np
import pytest
import torch

from rank_markov_draft_gb300 import binding
from synth import make_inputs
from tests.gpu_util import bf, dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B", [4, 96])  # the batch-copies build; the build with noise warps
def test_barrier_timeout_is_reported_and_recoverable(B):
    K, V, r = 3, 4096, 256
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


def test_verify_draw_timeout_is_reported_and_recoverable():
    """The fault knob on the verification's draw (the residual-mode launch, whose row copies
    three warps issue): the draw's waits run out and it exits, the context reports the
    timeout, and after a reset the same call reproduces the clean result."""
    B, K, V, r = 8, 4, 4096, 64
    inp = make_inputs(7, B, K, V, r)
    rng = np.random.default_rng(8)
    P = np.empty((B, K + 1, V), np.float32)
    P[:, :K] = inp.U + rng.standard_normal((B, K, V)).astype(np.float32)
    P[:, K] = rng.standard_normal((B, V)).astype(np.float32)
    U, W1, W2, anchors = dev(inp.U), bf(inp.W1), bf(inp.W2), dev(inp.anchors)
    Pd = dev(P)
    with binding.Context(0, B_max=B, V_max=V, K_max=K) as ctx:
        d = binding.markov_draft(ctx, U, W1, W2, anchors, temperature=1.0, seed=3)
        kw = dict(draft_temperature=1.0, target_temperature=1.0, seed=5)
        clean = binding.verify(ctx, Pd, U, W1, W2, anchors, d["tokens"], d["logprobs"], **kw)
        torch.cuda.synchronize()
        assert ctx.status() == 0
        ctx.debug_set(cta=0, timeout_ms=200)
        binding.verify(ctx, Pd, U, W1, W2, anchors, d["tokens"], d["logprobs"], **kw)
        torch.cuda.synchronize()          # returns: the draw exited on its own
        assert ctx.status() == binding.TIMEOUT
        with pytest.raises(binding.DSparkError) as err:
            binding.verify(ctx, Pd, U, W1, W2, anchors, d["tokens"], d["logprobs"], **kw)
        assert err.value.code == binding.POISONED
        ctx.reset()
        again = binding.verify(ctx, Pd, U, W1, W2, anchors, d["tokens"], d["logprobs"], **kw)
        torch.cuda.synchronize()
        assert ctx.status() == 0
        for key in ("n_acc", "next_token", "accept_prob"):
            assert torch.equal(again[key], clean[key]), key


def test_refused_launch_returns_cuda_error_and_enqueues_nothing():
    """A launch configuration the CUDA runtime refuses (more dynamic shared memory than
    the kernel allows) comes back from the host call as DSPARK_ERR_CUDA: no kernel ran,
    the outputs are untouched, the runtime's last error is cleared, and the context
    drafts again without a reset."""
    B, K, V, r = 4, 3, 4096, 256
    inp = make_inputs(6, B, K, V, r)
    U, W1, W2, anchors = dev(inp.U), bf(inp.W1), bf(inp.W2), dev(inp.anchors)
    with binding.Context(0, B_max=B, V_max=V, K_max=K) as ctx:
        clean = binding.markov_draft(ctx, U, W1, W2, anchors, temperature=1.0, seed=3)
        tokens = torch.full((B, K), -7, dtype=torch.int32, device="cuda")
        logprobs = torch.full((B, K), float("nan"), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        ctx.refuse_next_launch()
        with pytest.raises(binding.DSparkError) as err:
            binding.dspark_markov_draft(ctx, U, W1, W2, anchors, B, K, V, r, 1.0, 3, tokens,
                                        logprobs)
        assert err.value.code == binding.CUDA
        assert ctx.last_launches == 0
        torch.cuda.synchronize()
        assert bool((tokens == -7).all()) and bool(torch.isnan(logprobs).all())
        assert ctx.status() == 0
        x = torch.full((8,), 2.0, device="cuda") * 3.0   # torch's own launch checks pass
        torch.cuda.synchronize()
        assert float(x.sum()) == 48.0
        again = binding.markov_draft(ctx, U, W1, W2, anchors, temperature=1.0, seed=3)
        torch.cuda.synchronize()
        assert ctx.status() == 0 and ctx.last_launches == 1
        assert torch.equal(again["tokens"], clean["tokens"])
        assert torch.equal(again["logprobs"], clean["logprobs"])


def _target(rng, U):
    B, K, V = U.shape
    P = np.empty((B, K + 1, V), np.float32)
    P[:, :K] = U + rng.standard_normal((B, K, V)).astype(np.float32) * np.float32(0.8)
    P[:, K] = rng.standard_normal((B, V)).astype(np.float32) * np.float32(3.0)
    return P


@pytest.mark.parametrize("B,K,V,r", [(5, 4, 1000, 256), (130, 3, 4096, 64)])
def test_checked_library_runs_clean_and_matches_release(dsp, B, K, V, r):
    """The debug library's draft kernel checks every TMEM address and shared-memory offset
    it computes (accumulators, operand, rings, merge records, best-block store) before the
    access.  On in-range work no check fires (status 0) and every mode's outputs equal the
    release library's bit for bit: sampled, greedy, teacher-forced, gated, RNN, the label
    pass and the verification draw, with batch copies (B = 5) and two request chunks
    (B = 130)."""
    inp = make_inputs(80 + B, B, K, V, r, d=64, gated=True, rnn=True, weight_std=0.05)
    U, W1, W2, anchors = dev(inp.U), bf(inp.W1), bf(inp.W2), dev(inp.anchors)
    h, Wg, Wa = bf(inp.h), bf(inp.Wg), bf(inp.Wa)
    P = dev(_target(np.random.default_rng(81), inp.U))

    def every_mode(ctx):
        out = {}
        for T in (1.0, 0.0):
            d = binding.markov_draft(ctx, U, W1, W2, anchors, temperature=T, seed=9)
            out[f"draft{T}"] = d
            out[f"gated{T}"] = binding.markov_draft(ctx, U, W1, W2, anchors, temperature=T,
                                                    seed=9, h=h, Wg=Wg)
            out[f"rnn{T}"] = binding.rnn_draft(ctx, U, W1, W2, anchors, h, Wa, Wg=Wg,
                                               temperature=T, seed=9)
        d = out["draft1.0"]
        out["logits"] = binding.markov_logits(ctx, U, W1, W2, d["tokens"], temperature=1.0)
        out["label"] = {"label": binding.accept_label(ctx, P, U, W1, W2, anchors, d["tokens"],
                                                      d["logprobs"], draft_temperature=1.0,
                                                      target_temperature=1.0)}
        out["verify"] = binding.verify(ctx, P, U, W1, W2, anchors, d["tokens"], d["logprobs"],
                                       draft_temperature=1.0, target_temperature=1.0, seed=4)
        torch.cuda.synchronize()
        assert ctx.status() == 0
        return out

    release = every_mode(dsp)
    with binding.Context(0, B_max=B, V_max=V, K_max=K, checked=True) as ctx:
        checked = every_mode(ctx)
    for name, res in release.items():
        for key, t in res.items():
            if isinstance(t, torch.Tensor):
                assert torch.equal(t, checked[name][key]), f"{name}.{key} differs"


def test_checked_library_at_full_vocabulary():
    """The offset checks over every tile of the full vocabulary (152 CTAs, one per SM): the
    serving batch and the gated head's batch-copies build, drafted and greedy, run clean
    (status 0) and equal the release library's outputs."""
    from synth import config_inputs
    for cfg in (2, 3):
        inp = config_inputs(cfg)
        B = inp.U.shape[0]
        U, W1, W2, anchors = dev(inp.U), bf(inp.W1), bf(inp.W2), dev(inp.anchors)
        gate = dict(h=bf(inp.h), Wg=bf(inp.Wg)) if cfg == 3 else {}
        outs = []
        for checked in (False, True):
            with binding.Context(0, B_max=B, V_max=inp.U.shape[2], K_max=inp.U.shape[1],
                                 checked=checked) as ctx:
                res = [binding.markov_draft(ctx, U, W1, W2, anchors, temperature=T, seed=5,
                                            **gate) for T in (1.0, 0.0)]
                torch.cuda.synchronize()
                assert ctx.status() == 0
                outs.append(res)
        for a, c in zip(*outs):
            assert torch.equal(a["tokens"], c["tokens"])
            assert torch.equal(a["logprobs"], c["logprobs"])
        del U
