"""GPU parity of the acceptance label (dspark_accept_label) against the fp64 oracle.

The drafted tokens and their log-probabilities come from the oracle's draft
and are handed to both sides, so the two label the same block and no oracle
input comes from the GPU.

Tolerance.  If every log q(v) and log p(v) is off by at most eps, each term
min(q, p) moves by a factor within exp(+-eps), so |label - label'| <= eps *
label + O(eps^2).  Ungated, the GPU's per-token log-probabilities carry fp32
accumulation of exact bf16 products, ex2.approx and fp32 normalisers: well
under 1e-4, so 2e-4 is asserted.  Gated, the GPU rounds the gated operand
W1[x] * g to bf16 for its MMA (the oracle keeps it in fp64), which is the
draft path's own logit tolerance (2e-3).
"""

import numpy as np
import pytest
import torch

import oracle
from rank_markov_draft_gb300 import binding
from synth import make_inputs
from tests.gpu_util import LOGPROB_TOL, bf, dev, host

pytestmark = pytest.mark.gpu

LABEL_TOL = 2e-4
LABEL_TOL_GATED = LOGPROB_TOL


def _target_logits(rng, U, noise=0.8):
    """Synthetic target: the draft's base logits plus independent noise (one more
    row, the bonus position, that the label does not read)."""
    B, K, V = U.shape
    P = np.empty((B, K + 1, V), np.float32)
    P[:, :K] = U + rng.standard_normal((B, K, V)).astype(np.float32) * np.float32(noise)
    P[:, K] = rng.standard_normal((B, V)).astype(np.float32)
    return P


def _both(ctx, inp, P, Td, Tt, *, gated=False, seed=5):
    H = oracle.gate(inp.h, inp.Wg) if gated else None
    dr = oracle.markov_draft(inp.U, inp.W1, inp.W2, inp.anchors, temperature=Td, seed=seed, H=H)
    ref = oracle.accept_label(P, inp.U, inp.W1, inp.W2, inp.anchors, dr["tokens"],
                              draft_temperature=Td, target_temperature=Tt, H=H)
    gate = dict(h=bf(inp.h), Wg=bf(inp.Wg)) if gated else {}
    W1 = bf(inp.W1) if inp.W1 is not None else None
    W2 = bf(inp.W2) if inp.W2 is not None else None
    lab = binding.accept_label(ctx, dev(P), dev(inp.U), W1, W2, dev(inp.anchors),
                               dev(dr["tokens"]), dev(dr["logprobs"].astype(np.float32)),
                               draft_temperature=Td, target_temperature=Tt, **gate)
    torch.cuda.synchronize()
    assert ctx.status() == 0
    return host(lab), ref


@pytest.mark.parametrize("Td,Tt", [(1.0, 1.0), (0.7, 1.3), (0.0, 1.0), (1.0, 0.0), (0.0, 0.0)])
def test_label_matches_oracle(dsp, Td, Tt):
    B, K, V, r = 12, 5, 1000, 64  # 16 tiles of 64 tokens, the last one ragged
    inp = make_inputs(71, B, K, V, r, weight_std=0.1)
    P = _target_logits(np.random.default_rng(72), inp.U)
    gpu, ref = _both(dsp, inp, P, Td, Tt)
    if Td == 0.0 and Tt == 0.0:
        assert np.array_equal(gpu, ref)  # an indicator: the argmax decides it exactly
    else:
        assert np.abs(gpu - ref).max() <= LABEL_TOL, np.abs(gpu - ref).max()
    assert np.all((gpu >= 0) & (gpu <= 1))


@pytest.mark.parametrize("B,r", [(3, 256), (40, 128), (130, 256), (9, 0)])
def test_label_batch_shapes(dsp, B, r):
    """Batch copies (B <= 64), two 128-request chunks, and the rank-0 head."""
    K, V = 4, 2056
    inp = make_inputs(73 + B, B, K, V, max(r, 16), weight_std=0.1)
    if r == 0:  # no Markov term: the calibrated logits are U
        inp.W1 = inp.W2 = None
    P = _target_logits(np.random.default_rng(74), inp.U, noise=1.5)
    gpu, ref = _both(dsp, inp, P, 1.0, 1.0)
    assert np.abs(gpu - ref).max() <= LABEL_TOL, np.abs(gpu - ref).max()


def test_label_gated(dsp):
    B, K, V, r, d = 16, 6, 2048, 64, 128
    inp = make_inputs(75, B, K, V, r, d=d, gated=True, weight_std=0.1)
    P = _target_logits(np.random.default_rng(76), inp.U)
    for Td, Tt in [(1.0, 1.0), (1.0, 0.0)]:
        gpu, ref = _both(dsp, inp, P, Td, Tt, gated=True)
        assert np.abs(gpu - ref).max() <= LABEL_TOL_GATED, (Td, Tt, np.abs(gpu - ref).max())


def test_label_of_a_target_equal_to_the_draft_is_one(dsp):
    """p^t = p^d at every position: no mass is rejected, the label is 1."""
    B, K, V, r = 6, 4, 1536, 64
    inp = make_inputs(77, B, K, V, r, weight_std=0.3)
    dr = oracle.markov_draft(inp.U, inp.W1, inp.W2, inp.anchors, temperature=1.0, seed=2)
    prev = np.concatenate([inp.anchors[:, None], dr["tokens"][:, :-1]], axis=1)
    lg = oracle.markov_logits(inp.U, inp.W1, inp.W2, prev)["logits"]
    P = np.concatenate([lg, np.zeros((B, 1, V))], axis=1).astype(np.float32)
    lab = binding.accept_label(dsp, dev(P), dev(inp.U), bf(inp.W1), bf(inp.W2), dev(inp.anchors),
                               dev(dr["tokens"]), dev(dr["logprobs"].astype(np.float32)),
                               draft_temperature=1.0, target_temperature=1.0)
    torch.cuda.synchronize()
    assert dsp.status() == 0
    assert np.abs(host(lab) - 1.0).max() <= LABEL_TOL


def test_label_full_size(dsp):
    """Serving shape (B=128, K=16, V=151936, r=256) in one call: the oracle drafts
    every request and labels every drafted position, and all B K labels are
    compared."""
    B, K, V, r = 128, 16, 151936, 256
    inp = make_inputs(78, B, K, V, r, weight_std=0.05)
    P = _target_logits(np.random.default_rng(79), inp.U, noise=1.0)
    dr = oracle.markov_draft(inp.U, inp.W1, inp.W2, inp.anchors, temperature=1.0, seed=4)
    ref = oracle.accept_label(P, inp.U, inp.W1, inp.W2, inp.anchors, dr["tokens"],
                              draft_temperature=1.0, target_temperature=1.0)
    lab = binding.accept_label(dsp, dev(P), dev(inp.U), bf(inp.W1), bf(inp.W2), dev(inp.anchors),
                               dev(dr["tokens"]), dev(dr["logprobs"].astype(np.float32)),
                               draft_temperature=1.0, target_temperature=1.0)
    torch.cuda.synchronize()
    assert dsp.status() == 0
    lab = host(lab)
    assert lab.shape == (B, K) and np.all((lab >= 0) & (lab <= 1))
    err = np.abs(lab - ref)
    print(f"labels compared: {err.size} of {B * K}, max |error| {err.max():.2e}")
    assert err.max() <= LABEL_TOL, (np.unravel_index(err.argmax(), err.shape), err.max())


def test_label_argument_errors(dsp):
    B, K, V, r = 2, 2, 512, 64
    inp = make_inputs(81, B, K, V, r)
    P = dev(np.zeros((B, K + 1, V), np.float32))
    args = (dev(inp.U), bf(inp.W1), bf(inp.W2), dev(inp.anchors), dev(np.zeros((B, K), np.int32)))
    with pytest.raises(binding.DSparkError) as err:  # sampled draft without its log-probabilities
        binding.accept_label(dsp, P, *args, None, draft_temperature=1.0, target_temperature=1.0)
    assert err.value.code == binding.INVALID_ARG
    buf = torch.zeros(B * (K + 1) * V + 2, dtype=torch.float32, device="cuda")
    P8 = buf[2:].view(B, K + 1, V)  # 8-byte but not 16-byte aligned
    with pytest.raises(binding.DSparkError) as err:
        binding.accept_label(dsp, P8, *args, dev(np.zeros((B, K), np.float32)),
                             draft_temperature=1.0, target_temperature=1.0)
    assert err.value.code == binding.INVALID_ARG


def test_label_token_out_of_range_is_reported():
    B, K, V, r = 2, 2, 512, 64
    inp = make_inputs(82, B, K, V, r)
    tokens = np.array([[1, 2], [3, V + 5]], np.int32)
    with binding.Context(0, B_max=B, V_max=V, K_max=K) as ctx:
        binding.accept_label(ctx, dev(np.zeros((B, K + 1, V), np.float32)), dev(inp.U),
                             bf(inp.W1), bf(inp.W2), dev(inp.anchors), dev(tokens),
                             dev(np.zeros((B, K), np.float32)), draft_temperature=1.0,
                             target_temperature=1.0)
        torch.cuda.synchronize()
        assert ctx.status() == binding.DEVICE_OOB
