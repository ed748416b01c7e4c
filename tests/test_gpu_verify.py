"""GPU parity of speculative verification (dspark_verify) against the fp64 oracle.

The drafted tokens and their log-probabilities come from the oracle's draft and
are handed to both sides (no GPU output enters the oracle); the oracle
recomputes q from the draft head's inputs in fp64.  Accepted lengths
and next tokens must match wherever the oracle's smallest decision margin
(|u - min(1, p/q)| of every acceptance test, and the draw's block-race
margin) exceeds 1e-3.
"""

import numpy as np
import pytest
import torch
from scipy import special, stats

import oracle
from rank_markov_draft_gb300 import binding
from synth import bf16_bits, make_inputs
from tests.gpu_util import COVERAGE, MARGIN, bf, dev, host

pytestmark = pytest.mark.gpu


def _target_logits(rng, U, noise=0.8):
    """Synthetic target: the draft's base logits plus independent noise, and one
    more row for the bonus position."""
    B, K, V = U.shape
    P = np.empty((B, K + 1, V), np.float32)
    P[:, :K] = U + rng.standard_normal((B, K, V)).astype(np.float32) * np.float32(noise)
    P[:, K] = rng.standard_normal((B, V)).astype(np.float32) * np.float32(3.0)
    return P


def _run(dsp, inp, P, Td, Tt, seed, ell=None, gated=False):
    args = dict(h=bf(inp.h) if gated else None, Wg=bf(inp.Wg) if gated else None)
    H = oracle.gate(inp.h, inp.Wg) if gated else None
    dr = oracle.markov_draft(inp.U, inp.W1, inp.W2, inp.anchors, temperature=Td, seed=seed, H=H)
    out = binding.verify(dsp, dev(P), dev(inp.U), bf(inp.W1), bf(inp.W2), dev(inp.anchors),
                         dev(dr["tokens"]), dev(dr["logprobs"].astype(np.float32)),
                         draft_temperature=Td, target_temperature=Tt, seed=seed + 1,
                         ell=dev(ell) if ell is not None else None, **args)
    torch.cuda.synchronize()
    assert dsp.status() == 0
    return dr["tokens"], {k: host(v) for k, v in out.items()}


def _check(inp, P, tokens, out, Td, Tt, seed, ell=None, H=None, requests=None):
    B = P.shape[0]
    requests = range(B) if requests is None else requests
    hard = near = 0
    for b in requests:
        ref = oracle.verify(P, inp.U, inp.W1, inp.W2, inp.anchors, tokens,
                            draft_temperature=Td, target_temperature=Tt, seed=seed + 1,
                            ell=ell, H=H, b0=b, nb=1)
        same = (out["n_acc"][b] == ref["n_acc"][0]) and (out["next_token"][b] == ref["next_token"][0])
        if not same and ref["margins"][0] > MARGIN:
            hard += 1
        elif not same:
            near += 1
        if same:
            n = out["n_acc"][b]
            k = min(n + 1, P.shape[1] - 1, (ell[b] if ell is not None else P.shape[1] - 1))
            a_gpu, a_ref = out["accept_prob"][b, :k], ref["accept_prob"][0, :k]
            assert np.allclose(a_gpu, a_ref, rtol=2e-3, atol=2e-5), (b, a_gpu, a_ref)
    assert hard == 0, f"{hard} requests differ from the oracle with margin > {MARGIN}"
    n = len(requests)
    print(f"verify: {n - near} of {n} requests match the oracle; {near} differ at a near tie")
    assert near <= max(1, (1 - COVERAGE) * n), f"{near} of {n} requests stopped at a near tie"


def test_verify_repeated_calls_are_identical(dsp):
    """The scan keeps per-request counters and failure masks in the context, which each
    call's last CTA per request returns to zero: repeated calls on one context (with
    windows, so some CTAs only count) give identical results, equal to the oracle's."""
    B, K, V, r = 40, 6, 2048, 64
    inp = make_inputs(67, B, K, V, r, weight_std=0.1)
    P = _target_logits(np.random.default_rng(68), inp.U)
    ell = np.random.default_rng(69).integers(0, K + 1, B).astype(np.int32)
    runs = [_run(dsp, inp, P, 1.0, 1.0, seed=11, ell=ell) for _ in range(3)]
    tokens, first = runs[0]
    for _, out in runs[1:]:
        for key in ("n_acc", "next_token", "accept_prob"):
            assert np.array_equal(out[key], first[key]), key
    _check(inp, P, tokens, first, 1.0, 1.0, seed=11, ell=ell)


@pytest.mark.parametrize("Td,Tt", [(1.0, 1.0), (0.7, 1.3), (0.0, 1.0), (1.0, 0.0), (0.0, 0.0)])
def test_verify_matches_oracle(dsp, Td, Tt):
    B, K, V, r = 12, 5, 1000, 64
    inp = make_inputs(61, B, K, V, r, weight_std=0.1)
    P = _target_logits(np.random.default_rng(62), inp.U)
    tokens, out = _run(dsp, inp, P, Td, Tt, seed=7)
    assert np.all(out["n_acc"] >= 0) and np.all(out["n_acc"] <= K)
    assert np.all((out["next_token"] >= 0) & (out["next_token"] < V))
    _check(inp, P, tokens, out, Td, Tt, seed=7)


def test_verify_windows_and_gate(dsp):
    B, K, V, r, d = 16, 6, 2048, 64, 128
    inp = make_inputs(63, B, K, V, r, d=d, gated=True, weight_std=0.1)
    P = _target_logits(np.random.default_rng(64), inp.U)
    ell = np.random.default_rng(65).integers(0, K + 1, B).astype(np.int32)
    tokens, out = _run(dsp, inp, P, 1.0, 1.0, seed=9, ell=ell, gated=True)
    assert np.all(out["n_acc"] <= ell)
    beyond = np.arange(K)[None, :] >= ell[:, None]
    assert np.all(out["accept_prob"][beyond] == -1.0)
    _check(inp, P, tokens, out, 1.0, 1.0, seed=9, ell=ell, H=oracle.gate(inp.h, inp.Wg))


def test_verify_first_committed_token_is_the_target_distribution(dsp):
    """Losslessness on the GPU: the first committed token follows p_0 (chi-square)."""
    N, K, V, r = 2048, 2, 40, 16
    rng = np.random.default_rng(66)
    U1 = rng.standard_normal((1, K, V)).astype(np.float32)
    W1 = bf16_bits(rng.normal(0, 0.5, (V, r)).astype(np.float32))
    W2 = bf16_bits(rng.normal(0, 0.5, (r, V)).astype(np.float32))
    P1 = (rng.standard_normal((1, K + 1, V)) * 1.2).astype(np.float32)
    U = dev(np.ascontiguousarray(np.broadcast_to(U1, (N, K, V))))
    P = dev(np.ascontiguousarray(np.broadcast_to(P1, (N, K + 1, V))))
    anchors = dev(np.full(N, 3, np.int32))
    with binding.Context(0, B_max=N, V_max=V, K_max=K) as ctx:
        counts = np.zeros(V)
        acc = 0
        for rep in range(20):
            dr = binding.markov_draft(ctx, U, bf(W1), bf(W2), anchors, temperature=1.0, seed=rep)
            out = binding.verify(ctx, P, U, bf(W1), bf(W2), anchors, dr["tokens"], dr["logprobs"],
                                 draft_temperature=1.0, target_temperature=1.0, seed=1000 + rep)
            torch.cuda.synchronize()
            assert ctx.status() == 0
            n, y, x = host(out["n_acc"]), host(out["next_token"]), host(dr["tokens"])
            c0 = np.where(n >= 1, x[:, 0], y)
            counts += np.bincount(c0, minlength=V)
            acc += (n >= 1).sum()
    total = 20 * N
    p0 = special.softmax(P1[0, 0].astype(np.float64))
    exp = p0 * total
    small = exp < 5
    obs, ex = counts[~small], exp[~small]
    if small.any():
        obs = np.concatenate([obs, [counts[small].sum()]])
        ex = np.concatenate([ex, [exp[small].sum()]])
    assert stats.chisquare(obs, ex * obs.sum() / ex.sum()).pvalue > 0.01
    w1 = (W1.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    w2 = (W2.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    q0 = special.softmax(U1[0, 0].astype(np.float64) + w1[3] @ w2)
    a = 1.0 - 0.5 * np.abs(p0 - q0).sum()
    assert abs(acc / total - a) < 4 * np.sqrt(a * (1 - a) / total)


def test_verify_serving_size(dsp):
    """B=128, K=16, V=151936: the whole batch on the GPU, every request replayed by the
    oracle."""
    from synth import config_inputs
    inp = config_inputs(2)
    P = _target_logits(np.random.default_rng(67), inp.U, noise=1.0)
    tokens, out = _run(dsp, inp, P, 1.0, 1.0, seed=11)
    assert np.all(out["n_acc"] <= 16)
    _check(inp, P, tokens, out, 1.0, 1.0, seed=11)


@pytest.mark.parametrize("Td", [1.0, 0.0])
def test_verify_two_request_chunks(dsp, Td):
    """130 requests: the draw runs over two chunks of 128 rows (per-row constants, target
    rows and noise counters offset by the chunk)."""
    B, K, V, r = 130, 3, 1000, 64
    inp = make_inputs(68, B, K, V, r, weight_std=0.1)
    P = _target_logits(np.random.default_rng(69), inp.U)
    tokens, out = _run(dsp, inp, P, Td, 1.0, seed=13)
    assert np.all((out["next_token"] >= 0) & (out["next_token"] < V))
    _check(inp, P, tokens, out, Td, 1.0, seed=13)
