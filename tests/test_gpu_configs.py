"""GPU parity at the five workloads' full sizes, in the launch configuration the
benchmark times, checked on sampled outputs the oracle computes one by one.

* tiny (B=1, K=4, V=4096): every output, T = 1 and greedy.
* single request (B=1, K=16, V=151936): every output, T in {0, 0.7, 1}, seeds 0-9.
* serving + confidence (B=128, K=16, V=151936, d=2048): the whole batch on the
  GPU, T = 1 (seeds 0-9) and greedy; the oracle replays a rotating sample of
  requests (forced on the GPU's tokens) and the confidence head on all of them.
* gated (B=64, K=16, d=4096): T = 1, seeds 0-9, sampled requests.
* selector top-16 (B=256, K=16), gated and ungated: top-16 sets and score tables
  of every (request, position), walks of every request, seeds 0-3.
"""

import numpy as np
import pytest
import torch

import oracle
from rank_markov_draft_gb300 import binding
from synth import CONFIGS, config_inputs
from tests.gpu_util import LOGPROB_TOL, bf, check_tokens, dev, host

pytestmark = pytest.mark.gpu


def _draft(dsp, inp, T, seed, conf=None, gated=False):
    out = binding.markov_draft(dsp, dev(inp.U), bf(inp.W1), bf(inp.W2), dev(inp.anchors),
                               temperature=T, seed=seed, conf=conf,
                               h=bf(inp.h) if gated else None, Wg=bf(inp.Wg) if gated else None)
    torch.cuda.synchronize()
    assert dsp.status() == 0
    return {k: host(v) for k, v in out.items()}


def _check_requests(inp, out, T, seed, requests, H=None):
    mism = near = 0
    for b in requests:
        ref = oracle.markov_draft(inp.U, inp.W1, inp.W2, inp.anchors, temperature=T, seed=seed,
                                  H=H, b0=b, nb=1, forced=out["tokens"][b:b + 1])
        m, n = check_tokens(out["tokens"][b:b + 1], out["logprobs"][b:b + 1], ref)
        mism += m
        near += n
    return mism, near


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
        # two requests per run, rotating over the batch (22 of 128 replayed in all)
        _check_requests(inp, out, T, seed, [(2 * i) % c["B"], (2 * i + 77) % c["B"]])
        ref = oracle.confidence(inp.h, inp.W1, inp.anchors, tokens, inp.w_conf,
                                bias=c["conf_bias"], threshold=c["threshold"])
        assert np.abs(out["conf"] - ref["conf"]).max() < 1e-4
        assert np.abs(out["cumprod"] - ref["cumprod"]).max() < 1e-4
        near = np.abs(ref["cumprod"] - c["threshold"]) < 1e-4
        ok = (out["verify_len"] == ref["verify_len"]) | near.any(axis=1)
        assert ok.all()


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
    S = oracle.pair_scores(cand, host(sc["cand_U"]).astype(np.float64), inp.A, inp.Bt,
                           inp.anchors, V=V, H=H)
    assert np.abs(host(sc["scores"]) - S).max() <= LOGPROB_TOL
    for seed in c["seeds"]:
        wk = binding.selector_walk(dsp, sc["cand"], sc["scores"], dev(inp.anchors), V=V,
                                   temperature=1.0, seed=seed)
        torch.cuda.synchronize()
        tok = host(wk["tokens"])
        ref = oracle.walk(cand, S, temperature=1.0, seed=seed, forced=tok)
        check_tokens(tok, host(wk["logprobs"]), ref, what="walk")
