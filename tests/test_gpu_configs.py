"""GPU parity at the five workloads' full sizes, in the launch configuration the
benchmark times, checked on sampled outputs the oracle computes one by one.

* tiny (B=1, K=4, V=4096): every output, T = 1 and greedy.
* single request (B=1, K=16, V=151936): every output, T in {0, 0.7, 1}, seeds 0-9.
* serving + confidence (B=128, K=16, V=151936, d=2048): the whole batch on the
  GPU, T = 1 (seeds 0-9) and greedy; the oracle drafts a rotating sample of
  requests on its own, with the confidence head of its drafts.
* gated (B=64, K=16, d=4096): T = 1, seeds 0-9, sampled requests.
* selector top-16 (B=256, K=16), gated and ungated: top-16 sets and score tables
  of every (request, position), walks of every request, seeds 0-3.

No GPU output enters the oracle: each side drafts from the same inputs and
noise, and sequences are compared up to the first near tie of the oracle's
decisions (later positions depend on the token taken there).
"""

import numpy as np
import pytest
import torch

import oracle
from rank_markov_draft_gb300 import binding
from synth import CONFIGS, config_inputs
from tests.gpu_util import LOGPROB_TOL, bf, check_sequences, dev, first_difference, host

pytestmark = pytest.mark.gpu


def _draft(dsp, inp, T, seed, conf=None, gated=False):
    out = binding.markov_draft(dsp, dev(inp.U), bf(inp.W1), bf(inp.W2), dev(inp.anchors),
                               temperature=T, seed=seed, conf=conf,
                               h=bf(inp.h) if gated else None, Wg=bf(inp.Wg) if gated else None)
    torch.cuda.synchronize()
    assert dsp.status() == 0
    return {k: host(v) for k, v in out.items()}


def _check_requests(inp, out, T, seed, requests, H=None):
    """The oracle drafts each listed request on its own (same inputs and noise);
    returns its drafts by request."""
    refs = {}
    for b in requests:
        ref = oracle.markov_draft(inp.U, inp.W1, inp.W2, inp.anchors, temperature=T, seed=seed,
                                  H=H, b0=b, nb=1)
        check_sequences(out["tokens"][b:b + 1], out["logprobs"][b:b + 1], ref)
        refs[b] = ref
    return refs


def test_tiny_workload(dsp):
    inp = config_inputs(0)
    for T in CONFIGS[0]["temperatures"]:
        out = _draft(dsp, inp, T, 0)
        _check_requests(inp, out, T, 0, [0])


def test_single_request_full_vocab(dsp):
    inp = config_inputs(1)
    c = CONFIGS[1]
    for T in c["temperatures"]:
        for seed in c["seeds"]:
            out = _draft(dsp, inp, T, seed)
            _check_requests(inp, out, T, seed, [0])


def test_serving_batch_with_confidence(dsp):
    inp = config_inputs(2)
    c = CONFIGS[2]
    dev_h, dev_w = bf(inp.h), bf(inp.w_conf)
    runs = [(1.0, s) for s in c["seeds"]] + [(0.0, 0)]
    for i, (T, seed) in enumerate(runs):
        conf = binding.Confidence(h=dev_h, w=dev_w, bias=c["conf_bias"], threshold=c["threshold"])
        out = _draft(dsp, inp, T, seed, conf=conf)
        tokens = out["tokens"]
        assert tokens.min() >= 0 and tokens.max() < c["V"]
        # two requests per run, rotating over the batch (22 of 128 replayed in all); the
        # oracle's confidence of its own draft, at positions whose predecessors agree
        refs = _check_requests(inp, out, T, seed, [(2 * i) % c["B"], (2 * i + 77) % c["B"]])
        for b, dr in refs.items():
            ref = oracle.confidence(inp.h[b:b + 1], inp.W1, inp.anchors[b:b + 1], dr["tokens"],
                                    inp.w_conf, bias=c["conf_bias"], threshold=c["threshold"])
            d = first_difference(tokens[b], dr["tokens"][0])
            n = min(d + 1, c["K"])
            assert np.abs(out["conf"][b, :n] - ref["conf"][0, :n]).max() < 1e-4
            assert np.abs(out["cumprod"][b, :n] - ref["cumprod"][0, :n]).max() < 1e-4
            if d == c["K"]:
                near = np.abs(ref["cumprod"][0] - c["threshold"]) < 1e-4
                assert out["verify_len"][b] == ref["verify_len"][0] or near.any()


def test_gated_head(dsp):
    inp = config_inputs(3)
    c = CONFIGS[3]
    H = oracle.gate(inp.h, inp.Wg)
    for i, seed in enumerate(c["seeds"]):
        out = _draft(dsp, inp, 1.0, seed, gated=True)
        _check_requests(inp, out, 1.0, seed, [(3 * i) % c["B"], (3 * i + 31) % c["B"]], H=H)


@pytest.mark.parametrize("gated", [False, True])
def test_selector_top16(dsp, gated):
    inp = config_inputs(4)
    c = CONFIGS[4]
    V = c["V"]
    sc = binding.selector_scores(dsp, dev(inp.U), bf(inp.A), bf(inp.Bt), dev(inp.anchors),
                                 topk=16, h=bf(inp.h) if gated else None,
                                 Wg=bf(inp.Wg) if gated else None)
    torch.cuda.synchronize()
    assert dsp.status() == 0
    top = oracle.topk(inp.U, 16)
    cand = host(sc["cand"])
    ties = top["margin"] == 0.0
    same = (cand == top["cand"]).all(axis=-1)
    assert (same | ties).all(), f"{int((~same & ~ties).sum())} candidate sets differ"
    assert np.array_equal(host(sc["cand_U"])[same], top["cval"].astype(np.float32)[same])
    H = oracle.gate(inp.h, inp.Wg) if gated else None
    S = oracle.pair_scores(top["cand"], top["cval"], inp.A, inp.Bt, inp.anchors, V=V, H=H)
    # scores of a position depend on its own and its predecessor's candidate set
    both = same.copy()
    both[:, 1:] &= same[:, :-1]
    assert np.abs(host(sc["scores"])[both] - S[both]).max() <= LOGPROB_TOL
    whole = both.all(axis=-1)  # requests whose every candidate set agrees
    assert whole.sum() >= c["B"] // 2
    for seed in c["seeds"]:
        wk = binding.selector_walk(dsp, sc["cand"], sc["scores"], dev(inp.anchors), V=V,
                                   temperature=1.0, seed=seed)
        torch.cuda.synchronize()
        ref = oracle.walk(top["cand"], S, temperature=1.0, seed=seed)
        sub = {k: v[whole] for k, v in ref.items()}
        check_sequences(host(wk["tokens"])[whole], host(wk["logprobs"])[whole], sub,
                        what="walk")
