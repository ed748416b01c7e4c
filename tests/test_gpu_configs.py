"""GPU parity at the five workloads' full sizes, in the launch configuration the
benchmark times, checked against the oracle's own drafts of whole batches (and
of rotating requests for the remaining seeds).

* tiny (B=1, K=4, V=4096): every output, T = 1 and greedy.
* single request (B=1, K=16, V=151936): every output, T in {0, 0.7, 1}, seeds 0-9.
* serving + confidence (B=128, K=16, V=151936, d=2048): the whole batch on the
  GPU, T = 1 (seeds 0-9) and greedy; the oracle drafts every request for seed 0
  and for the greedy run, and two rotating requests for each other seed, with
  the confidence head of its drafts.
* gated (B=64, K=16, d=4096): T = 1, seeds 0-9; every request for seed 0, two
  rotating requests for each other seed.
* selector top-16 (B=256, K=16), gated and ungated: top-16 sets and score tables
  of every (request, position), walks of every request, seeds 0-3.

No GPU output enters the oracle: each side drafts from the same inputs and
noise, and sequences are compared up to the first near tie of the oracle's
decisions (later positions depend on the token taken there).  Each test
prints how many positions it compared and how many requests stopped at a near
tie, and fails when fewer than 95% of the replayed positions were compared.
"""

import numpy as np
import pytest
import torch

import oracle
from rank_markov_draft_gb300 import binding
from synth import CONFIGS, config_inputs
from tests.gpu_util import (LOGPROB_TOL, assert_coverage, bf, check_sequences, dev,
                            first_difference, host)

pytestmark = pytest.mark.gpu


def _draft(dsp, inp, T, seed, conf=None, gated=False):
    out = binding.markov_draft(dsp, dev(inp.U), bf(inp.W1), bf(inp.W2), dev(inp.anchors),
                               temperature=T, seed=seed, conf=conf,
                               h=bf(inp.h) if gated else None, Wg=bf(inp.Wg) if gated else None)
    torch.cuda.synchronize()
    assert dsp.status() == 0
    return {k: host(v) for k, v in out.items()}


def _replay(inp, out, T, seed, requests=None, H=None, what="draft"):
    """The oracle drafts the listed requests (the whole batch when None) on its own,
    from the same inputs and noise, and each is compared with the GPU's draft of it.
    Returns the request indices, the oracle's drafts [n, K] and (requests that
    diverged at a near tie, positions compared)."""
    B = inp.U.shape[0]
    if requests is None:
        idx = np.arange(B)
        ref = oracle.markov_draft(inp.U, inp.W1, inp.W2, inp.anchors, temperature=T, seed=seed,
                                  H=H, b0=0, nb=B)
    else:
        idx = np.asarray(requests)
        parts = [oracle.markov_draft(inp.U, inp.W1, inp.W2, inp.anchors, temperature=T,
                                     seed=seed, H=H, b0=int(b), nb=1) for b in idx]
        ref = {k: np.concatenate([r[k] for r in parts]) for k in parts[0]}
    diverged, compared = check_sequences(out["tokens"][idx], out["logprobs"][idx], ref,
                                         what=what)
    return idx, ref, diverged, compared


def test_tiny_workload(dsp):
    inp = config_inputs(0)
    c = CONFIGS[0]
    div = comp = 0
    for T in c["temperatures"]:
        out = _draft(dsp, inp, T, 0)
        _, _, d, n = _replay(inp, out, T, 0)
        div, comp = div + d, comp + n
    assert_coverage("tiny", div, comp, len(c["temperatures"]) * c["K"])


def test_single_request_full_vocab(dsp):
    inp = config_inputs(1)
    c = CONFIGS[1]
    div = comp = runs = 0
    for T in c["temperatures"]:
        for seed in c["seeds"]:
            out = _draft(dsp, inp, T, seed)
            _, _, d, n = _replay(inp, out, T, seed)
            div, comp, runs = div + d, comp + n, runs + 1
    assert_coverage("single request", div, comp, runs * c["K"])


def test_serving_batch_with_confidence(dsp):
    """Every request of the batch replayed by the oracle for seed 0 at T = 1 and for the
    greedy run; two rotating requests for each other seed."""
    inp = config_inputs(2)
    c = CONFIGS[2]
    B, K = c["B"], c["K"]
    dev_h, dev_w = bf(inp.h), bf(inp.w_conf)
    runs = [(1.0, s) for s in c["seeds"]] + [(0.0, 0)]
    div = comp = total = 0
    for i, (T, seed) in enumerate(runs):
        conf = binding.Confidence(h=dev_h, w=dev_w, bias=c["conf_bias"], threshold=c["threshold"])
        out = _draft(dsp, inp, T, seed, conf=conf)
        tokens = out["tokens"]
        assert tokens.min() >= 0 and tokens.max() < c["V"]
        whole = seed == 0
        requests = None if whole else [(2 * i) % B, (2 * i + 77) % B]
        idx, dr, d, n = _replay(inp, out, T, seed, requests, what=f"serving T={T} seed={seed}")
        if whole:
            assert_coverage(f"serving T={T} seed={seed} (whole batch)", d, n, B * K)
        div, comp, total = div + d, comp + n, total + len(idx) * K
        # the oracle's confidence of its own drafts, at positions whose predecessors agree
        ref = oracle.confidence(inp.h[idx], inp.W1, inp.anchors[idx], dr["tokens"], inp.w_conf,
                                bias=c["conf_bias"], threshold=c["threshold"])
        for j, b in enumerate(idx):
            dd = first_difference(tokens[b], dr["tokens"][j])
            m = min(dd + 1, K)
            assert np.abs(out["conf"][b, :m] - ref["conf"][j, :m]).max() < 1e-4
            assert np.abs(out["cumprod"][b, :m] - ref["cumprod"][j, :m]).max() < 1e-4
            if dd == K:
                near = np.abs(ref["cumprod"][j] - c["threshold"]) < 1e-4
                assert out["verify_len"][b] == ref["verify_len"][j] or near.any()
    assert_coverage("serving, all runs", div, comp, total)


def test_gated_head(dsp):
    """Every request replayed for seed 0; two rotating requests for each other seed."""
    inp = config_inputs(3)
    c = CONFIGS[3]
    B, K = c["B"], c["K"]
    H = oracle.gate(inp.h, inp.Wg)
    div = comp = total = 0
    for i, seed in enumerate(c["seeds"]):
        out = _draft(dsp, inp, 1.0, seed, gated=True)
        requests = None if seed == 0 else [(3 * i) % B, (3 * i + 31) % B]
        idx, _, d, n = _replay(inp, out, 1.0, seed, requests, H=H, what=f"gated seed={seed}")
        if requests is None:
            assert_coverage("gated seed=0 (whole batch)", d, n, B * K)
        div, comp, total = div + d, comp + n, total + len(idx) * K
    assert_coverage("gated, all runs", div, comp, total)


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
    # candidate sets may differ only at an exact tie of the 16th and 17th values
    tied = ties.any(axis=-1)
    print(f"selector (gated={gated}): {int(tied.sum())} requests hold an exact top-16 tie, "
          f"{int((~same).sum())} candidate sets differ")
    assert whole.sum() >= c["B"] - int(tied.sum())
    for seed in c["seeds"]:
        wk = binding.selector_walk(dsp, sc["cand"], sc["scores"], dev(inp.anchors), V=V,
                                   temperature=1.0, seed=seed)
        torch.cuda.synchronize()
        ref = oracle.walk(top["cand"], S, temperature=1.0, seed=seed)
        sub = {k: v[whole] for k, v in ref.items()}
        d, n = check_sequences(host(wk["tokens"])[whole], host(wk["logprobs"])[whole], sub,
                               what="walk")
        assert_coverage(f"walk seed={seed}", d, n, int(whole.sum()) * c["K"])
