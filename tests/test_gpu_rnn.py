"""GPU parity of the RNN head (dspark_rnn_draft, dspark_rnn_logits) with the oracle.

Reading of the head (DSpark explainer, "The RNN head"; "Repair the Joint, Meter
the Verify", "Fix 1"; vLLM guide, "Key Parameters"): s_k = a_k (.) s_{k-1} +
g_k (.) W1[x_{k-1}], s_{-1} = 0, a_k = sigmoid(h_k . Wa), g_k = sigmoid(h_k . Wg)
(or 1), logits_k = U_k + s_k W2.  The GPU carries the state as the bf16 MMA
operand; the oracle keeps it in fp64.  Tolerances are the draft's: 2e-3 on
logits and log-probabilities, tokens bit-exact wherever the oracle's decision
margin exceeds 1e-3.
"""

import numpy as np
import pytest
import torch

import oracle
from rank_markov_draft_gb300 import binding
from synth import CONFIGS, config_inputs, make_inputs
from tests.gpu_util import LOGPROB_TOL, assert_coverage, bf, check_sequences, dev, host

pytestmark = pytest.mark.gpu

CASES = [
    # B, K, V, r, d
    (5, 6, 1000, 256, 128),     # ragged last tile, two batch copies
    (130, 3, 520, 64, 64),      # two request chunks, rank 64
    (3, 16, 4096, 256, 64),     # full block length
]


def _gates(inp, input_gate):
    A = oracle.gate(inp.h, inp.Wa)
    G = oracle.gate(inp.h, inp.Wg) if input_gate else None
    return A, G


@pytest.mark.parametrize("B,K,V,r,d", CASES)
@pytest.mark.parametrize("input_gate", [True, False])
def test_rnn_teacher_forced_logits_match_oracle(dsp, B, K, V, r, d, input_gate):
    inp = make_inputs(40 + B + V, B, K, V, r, d=d, gated=True, rnn=True, weight_std=0.05)
    prev = np.random.default_rng(41).integers(0, V, size=(B, K)).astype(np.int32)
    for T in (1.0, 0.0):
        out = binding.rnn_logits(dsp, dev(inp.U), bf(inp.W1), bf(inp.W2), dev(prev), bf(inp.h),
                                 bf(inp.Wa), Wg=bf(inp.Wg) if input_gate else None,
                                 temperature=T)
        torch.cuda.synchronize()
        assert dsp.status() == 0
        A, G = _gates(inp, input_gate)
        ref = oracle.rnn_logits(inp.U, inp.W1, inp.W2, prev, A, G=G, temperature=T)
        err = np.abs(host(out["logits"]) - ref["logits"]).max()
        assert err <= LOGPROB_TOL, f"max |logit - oracle| = {err:.3e}"
        assert np.abs(host(out["lse"]) - ref["lse"]).max() <= LOGPROB_TOL


@pytest.mark.parametrize("B,K,V,r,d", CASES)
@pytest.mark.parametrize("T", [1.0, 0.7, 0.0])
def test_rnn_draft_matches_oracle(dsp, B, K, V, r, d, T):
    inp = make_inputs(50 + B + V, B, K, V, r, d=d, gated=True, rnn=True, weight_std=0.05)
    out = binding.rnn_draft(dsp, dev(inp.U), bf(inp.W1), bf(inp.W2), dev(inp.anchors),
                            bf(inp.h), bf(inp.Wa), Wg=bf(inp.Wg), temperature=T, seed=13)
    torch.cuda.synchronize()
    assert dsp.status() == 0
    A, G = _gates(inp, True)
    ref = oracle.rnn_draft(inp.U, inp.W1, inp.W2, inp.anchors, A, G=G, temperature=T, seed=13)
    d_, n_ = check_sequences(host(out["tokens"]), host(out["logprobs"]), ref, what="rnn draft")
    assert_coverage(f"rnn draft B={B} V={V} T={T}", d_, n_, B * K)


@pytest.mark.parametrize("input_gate", [False, True])
def test_rnn_with_zero_decay_equals_the_markov_head_bitwise(dsp, input_gate):
    """a = sigmoid(h . Wa) = 0 exactly (h = 1, Wa = -4: h . Wa = -4 d, whose sigmoid is 0
    in fp32): the RNN head is the gated head, or with no input gate the vanilla one."""
    B, K, V, r, d = 6, 8, 2048, 128, 64
    inp = make_inputs(60, B, K, V, r, d=d, gated=True, rnn=True, weight_std=0.05)
    ones = np.full((B, K, d), 0x3F80, np.uint16)       # 1.0
    Wa = np.full((d, r), 0xC080, np.uint16)             # -4.0
    for T in (1.0, 0.0):
        rnn = binding.rnn_draft(dsp, dev(inp.U), bf(inp.W1), bf(inp.W2), dev(inp.anchors),
                                bf(ones), bf(Wa), Wg=bf(inp.Wg) if input_gate else None,
                                temperature=T, seed=21)
        mk = binding.markov_draft(dsp, dev(inp.U), bf(inp.W1), bf(inp.W2), dev(inp.anchors),
                                  temperature=T, seed=21, h=bf(ones) if input_gate else None,
                                  Wg=bf(inp.Wg) if input_gate else None)
        torch.cuda.synchronize()
        assert dsp.status() == 0
        assert torch.equal(rnn["tokens"], mk["tokens"])
        assert torch.equal(rnn["logprobs"], mk["logprobs"])


def test_rnn_workload_full_size(dsp):
    """B = 64, K = 16, V = 151936, d = 4096 (the gated head's shapes, both gates): every
    request of seed 0 replayed by the oracle."""
    c = CONFIGS[5]
    inp = config_inputs(5)
    out = binding.rnn_draft(dsp, dev(inp.U), bf(inp.W1), bf(inp.W2), dev(inp.anchors),
                            bf(inp.h), bf(inp.Wa), Wg=bf(inp.Wg), temperature=1.0, seed=0)
    torch.cuda.synchronize()
    assert dsp.status() == 0
    A, G = _gates(inp, True)
    ref = oracle.rnn_draft(inp.U, inp.W1, inp.W2, inp.anchors, A, G=G, temperature=1.0, seed=0)
    d_, n_ = check_sequences(host(out["tokens"]), host(out["logprobs"]), ref, what="rnn full")
    assert_coverage("rnn workload (whole batch)", d_, n_, c["B"] * c["K"])
