"""GPU parity: every kernel of the hot path against the fp64 oracle, through the C ABI.

Sizes span several vocabulary tiles, more than one 128-request chunk and
ragged tails; tolerances are the ones the task fixes (2e-3 absolute on
calibrated logits and log-probabilities; tokens bit-exact wherever the
oracle's top-2 perturbed-score margin exceeds 1e-3, near ties counted).
"""

import numpy as np
import pytest
import torch
from scipy import special, stats

import oracle
from rank_markov_draft_gb300 import binding
from synth import bf16_bits, make_inputs
from tests.gpu_util import (LOGPROB_TOL, assert_coverage, bf, check_sequences, dev,
                            first_difference, host)

pytestmark = pytest.mark.gpu


# ------------------------------------------------------------------- gate GEMM
@pytest.mark.parametrize("M,d,r", [(15, 128, 64), (300, 256, 256), (1024, 4096, 256)])
def test_gate_matches_oracle(dsp, M, d, r):
    rng = np.random.default_rng(M + d)
    h = bf16_bits(rng.standard_normal((M, d)).astype(np.float32))
    Wg = bf16_bits((rng.standard_normal((d, r)) * 0.02).astype(np.float32))
    H = host(binding.gate(dsp, bf(h), bf(Wg)))
    torch.cuda.synchronize()
    assert dsp.status() == 0
    ref = oracle.gate(h, Wg)
    assert np.abs(H - ref).max() < 2e-5


# -------------------------------------------------------- teacher-forced logits
TF_CASES = [
    # B, K, V, r, gated, d
    (1, 4, 4096, 256, False, 0),      # tiny workload shape
    (3, 5, 1000, 256, False, 0),      # ragged last tile (1000 = 15 * 64 + 40)
    (130, 2, 520, 64, False, 0),      # two request chunks, ragged B
    (4, 3, 8, 16, False, 0),          # one partial tile
    (5, 4, 1000, 128, True, 128),     # gated
    (2, 3, 4096, 256, True, 64),
]


@pytest.mark.parametrize("B,K,V,r,gated,d", TF_CASES)
@pytest.mark.parametrize("T", [1.0, 0.7, 0.0])
def test_teacher_forced_logits(dsp, B, K, V, r, gated, d, T):
    inp = make_inputs(7 + B + V, B, K, V, r, d=d, gated=gated)
    prev = np.random.default_rng(3).integers(0, V, size=(B, K)).astype(np.int32)
    out = binding.markov_logits(dsp, dev(inp.U), bf(inp.W1), bf(inp.W2), dev(prev),
                                temperature=T, h=bf(inp.h) if gated else None,
                                Wg=bf(inp.Wg) if gated else None)
    torch.cuda.synchronize()
    assert dsp.status() == 0
    H = oracle.gate(inp.h, inp.Wg) if gated else None
    ref = oracle.markov_logits(inp.U, inp.W1, inp.W2, prev, temperature=T, H=H)
    err = np.abs(host(out["logits"]) - ref["logits"]).max()
    assert err <= LOGPROB_TOL, f"max |logit - oracle| = {err:.3e}"
    lerr = np.abs(host(out["lse"]) - ref["lse"]).max()
    assert lerr <= LOGPROB_TOL, f"max |lse - oracle| = {lerr:.3e}"


def test_rank_zero_returns_base_logits_bitwise(dsp):
    """--markov-rank 0 disables the head: calibrated logits are U itself."""
    B, K, V = 3, 4, 1000
    inp = make_inputs(11, B, K, V, 16)
    prev = np.zeros((B, K), np.int32)
    out = binding.markov_logits(dsp, dev(inp.U), None, None, dev(prev), temperature=1.0)
    torch.cuda.synchronize()
    assert np.array_equal(host(out["logits"]), inp.U)


# ------------------------------------------------------------------ the draft
DRAFT_CASES = [
    # B, K, V, r
    (1, 4, 4096, 256),
    (5, 6, 1000, 256),
    (130, 3, 520, 32),
    (3, 5, 8, 16),
    (2, 16, 151936, 256),
    (96, 5, 40000, 64),     # one chunk above 64 requests, two or three tiles a CTA
]


@pytest.mark.parametrize("B,K,V,r", DRAFT_CASES)
@pytest.mark.parametrize("T,seed", [(1.0, 0), (0.7, 3), (0.0, 0)])
def test_draft_matches_oracle(dsp, B, K, V, r, T, seed):
    inp = make_inputs(100 + B + K, B, K, V, r)
    out = binding.markov_draft(dsp, dev(inp.U), bf(inp.W1), bf(inp.W2), dev(inp.anchors),
                               temperature=T, seed=seed)
    torch.cuda.synchronize()
    assert dsp.status() == 0
    tok, lp = host(out["tokens"]), host(out["logprobs"])
    assert tok.min() >= 0 and tok.max() < V
    ref = oracle.markov_draft(inp.U, inp.W1, inp.W2, inp.anchors, temperature=T, seed=seed)
    check_sequences(tok, lp, ref)


@pytest.mark.parametrize("B,K,V", [(3, 64, 4096), (2, 3, 1 << 18), (66, 2, 1 << 18)])
@pytest.mark.parametrize("T", [1.0, 0.0])
def test_draft_at_the_limits(B, K, V, T):
    """The largest block (K = 64: 64 key rows and partial planes) and the largest vocabulary
    (V = 2^18: token ids use every bit of the key's 18-bit token field, 2048 tiles), with and
    without batch copies; every position compared with the oracle."""
    r = 256
    inp = make_inputs(300 + K + B, B, K, V, r)
    with binding.Context(0, B_max=B, V_max=V, K_max=K) as ctx:
        out = binding.markov_draft(ctx, dev(inp.U), bf(inp.W1), bf(inp.W2), dev(inp.anchors),
                                   temperature=T, seed=17)
        torch.cuda.synchronize()
        assert ctx.status() == 0
        tok, lp = host(out["tokens"]), host(out["logprobs"])
    assert tok.min() >= 0 and tok.max() < V
    ref = oracle.markov_draft(inp.U, inp.W1, inp.W2, inp.anchors, temperature=T, seed=17)
    d_, n_ = check_sequences(tok, lp, ref)
    assert_coverage(f"limits B={B} K={K} V={V} T={T}", d_, n_, B * K)


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_gated_draft_matches_oracle(dsp, T):
    B, K, V, r, d = 6, 5, 1000, 256, 128
    inp = make_inputs(21, B, K, V, r, d=d, gated=True)
    out = binding.markov_draft(dsp, dev(inp.U), bf(inp.W1), bf(inp.W2), dev(inp.anchors),
                               temperature=T, seed=9, h=bf(inp.h), Wg=bf(inp.Wg))
    torch.cuda.synchronize()
    assert dsp.status() == 0
    tok = host(out["tokens"])
    ref = oracle.markov_draft(inp.U, inp.W1, inp.W2, inp.anchors, temperature=T, seed=9,
                              H=oracle.gate(inp.h, inp.Wg))
    check_sequences(tok, host(out["logprobs"]), ref)


def test_unit_gate_equals_vanilla_bitwise(dsp):
    """H = 1 makes the gated head the vanilla head (equivalence page): identical outputs."""
    B, K, V, r, d = 7, 5, 1000, 256, 64
    inp = make_inputs(22, B, K, V, r)
    h = np.full((B, K, d), 0x3F80, np.uint16)           # 1.0
    Wg = np.full((d, r), 0x4080, np.uint16)             # 4.0 -> h.Wg = 256, sigmoid = 1
    for T in (1.0, 0.0):
        a = binding.markov_draft(dsp, dev(inp.U), bf(inp.W1), bf(inp.W2), dev(inp.anchors),
                                 temperature=T, seed=5)
        g = binding.markov_draft(dsp, dev(inp.U), bf(inp.W1), bf(inp.W2), dev(inp.anchors),
                                 temperature=T, seed=5, h=bf(h), Wg=bf(Wg))
        torch.cuda.synchronize()
        assert torch.equal(a["tokens"], g["tokens"])
        assert torch.equal(a["logprobs"], g["logprobs"])


def test_rank_zero_draft_samples_the_base_logits(dsp):
    B, K, V = 4, 5, 1000
    inp = make_inputs(23, B, K, V, 16)
    out = binding.markov_draft(dsp, dev(inp.U), None, None, dev(inp.anchors), temperature=1.0,
                               seed=1)
    torch.cuda.synchronize()
    tok = host(out["tokens"])
    ref = oracle.markov_draft(inp.U, None, None, inp.anchors, temperature=1.0, seed=1)
    check_sequences(tok, host(out["logprobs"]), ref)


def test_fused_confidence_matches_oracle(dsp):
    B, K, V, r, d = 9, 6, 1000, 256, 256
    inp = make_inputs(24, B, K, V, r, d=d, confidence=True)
    conf = binding.Confidence(h=bf(inp.h), w=bf(inp.w_conf), bias=0.1, threshold=0.3)
    out = binding.markov_draft(dsp, dev(inp.U), bf(inp.W1), bf(inp.W2), dev(inp.anchors),
                               temperature=1.0, seed=2, conf=conf)
    torch.cuda.synchronize()
    dr = oracle.markov_draft(inp.U, inp.W1, inp.W2, inp.anchors, temperature=1.0, seed=2)
    ref = oracle.confidence(inp.h, inp.W1, inp.anchors, dr["tokens"], inp.w_conf, bias=0.1,
                            threshold=0.3)
    _check_confidence(host(out["tokens"]), dr["tokens"], out, ref, 0.3)


def _check_confidence(gpu_tokens, orc_tokens, out, ref, threshold, tol=1e-5):
    """Confidence of a GPU draft against the oracle's confidence of its own draft, at
    the positions whose predecessors agree (the first position where the drafts
    differ still has an agreed predecessor); verify lengths where whole drafts agree."""
    conf, cum, vl = host(out["conf"]), host(out["cumprod"]), host(out["verify_len"])
    K = gpu_tokens.shape[1]
    whole = 0
    for b in range(gpu_tokens.shape[0]):
        n = min(first_difference(gpu_tokens[b], orc_tokens[b]) + 1, K)
        assert np.abs(conf[b, :n] - ref["conf"][b, :n]).max() < tol, b
        assert np.abs(cum[b, :n] - ref["cumprod"][b, :n]).max() < tol, b
        if n == K and first_difference(gpu_tokens[b], orc_tokens[b]) == K:
            whole += 1
            near = np.abs(ref["cumprod"][b] - threshold) < tol
            assert vl[b] == ref["verify_len"][b] or near.any(), b
    assert whole >= gpu_tokens.shape[0] // 2  # divergences only at near ties


@pytest.mark.parametrize("with_markov", [True, False])
def test_standalone_confidence(dsp, with_markov):
    B, K, V, r, d = 11, 7, 500, 64, 96
    inp = make_inputs(25, B, K, V, r, d=d, confidence=True)
    w = inp.w_conf if with_markov else inp.w_conf[:d]
    tokens = np.random.default_rng(5).integers(0, V, size=(B, K)).astype(np.int32)
    out = binding.confidence(dsp, bf(inp.h), bf(inp.W1), dev(inp.anchors), dev(tokens), bf(w),
                             V=V, bias=-0.2, with_markov=with_markov, threshold=0.2)
    torch.cuda.synchronize()
    ref = oracle.confidence(inp.h, inp.W1, inp.anchors, tokens, w, bias=-0.2,
                            with_markov=with_markov, threshold=0.2, V=V)
    assert np.abs(host(out["conf"]) - ref["conf"]).max() < 1e-5
    assert np.array_equal(host(out["verify_len"]), ref["verify_len"])


def test_gpu_sampler_matches_exhaustive_joint(dsp):
    """10^6 GPU draws vs prod_k softmax(U_k + W1[x_{k-1}] W2) enumerated over all V^K paths."""
    V, K, r, N = 8, 3, 16, 1_000_000
    rng = np.random.default_rng(11)
    U1 = rng.standard_normal((1, K, V)).astype(np.float32)
    W1 = bf16_bits(rng.normal(0, 0.5, (V, r)).astype(np.float32))
    W2 = bf16_bits(rng.normal(0, 0.5, (r, V)).astype(np.float32))
    anchor = 5
    U = torch.from_numpy(U1).cuda().expand(N, K, V).contiguous()
    anchors = torch.full((N,), anchor, dtype=torch.int32, device="cuda")
    out = binding.markov_draft(dsp, U, bf(W1), bf(W2), anchors, temperature=1.0, seed=2024)
    torch.cuda.synchronize()
    paths = host(out["tokens"]).astype(np.int64)
    cell = (paths[:, 0] * V + paths[:, 1]) * V + paths[:, 2]
    counts = np.bincount(cell, minlength=V ** K).astype(np.float64)
    w1 = (W1.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    w2 = (W2.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    bias = w1 @ w2
    P = np.zeros((V,) * K)
    for x1 in range(V):
        p1 = special.softmax(U1[0, 0] + bias[anchor])[x1]
        for x2 in range(V):
            p2 = special.softmax(U1[0, 1] + bias[x1])[x2]
            P[x1, x2, :] = p1 * p2 * special.softmax(U1[0, 2] + bias[x2])
    exp = P.reshape(-1) * N
    small = exp < 5
    obs = np.concatenate([counts[~small], [counts[small].sum()]])
    ex = np.concatenate([exp[~small], [exp[small].sum()]])
    assert stats.chisquare(obs, ex).pvalue > 0.01
    lp = host(out["logprobs"])[:5000].sum(1)
    assert np.allclose(lp, np.log(P.reshape(-1)[cell[:5000]]), atol=3 * LOGPROB_TOL)


def test_gpu_block_race_over_several_blocks_matches_exhaustive_joint(dsp):
    """The draw's first stage (the exponential race between 16-token blocks) on the GPU:
    V = 56 spans four blocks (the last one ragged, 8 tokens) with unequal masses, K = 2,
    T = 0.8.  10^6 draws vs prod_k softmax((U_k + W1[x_{k-1}] W2) / T) enumerated over
    all V^2 paths, and the block frequencies at each position vs the blocks' masses."""
    V, K, r, N, T = 56, 2, 16, 1_000_000, 0.8
    rng = np.random.default_rng(12)
    offset = np.repeat([0.0, 1.5, -1.0, 0.8], 16)[:V]
    U1 = (rng.standard_normal((1, K, V)) + offset).astype(np.float32)
    W1 = bf16_bits(rng.normal(0, 0.3, (V, r)).astype(np.float32))
    W2 = bf16_bits(rng.normal(0, 0.3, (r, V)).astype(np.float32))
    anchor = 9
    U = torch.from_numpy(U1).cuda().expand(N, K, V).contiguous()
    anchors = torch.full((N,), anchor, dtype=torch.int32, device="cuda")
    out = binding.markov_draft(dsp, U, bf(W1), bf(W2), anchors, temperature=T, seed=77)
    torch.cuda.synchronize()
    assert dsp.status() == 0
    paths = host(out["tokens"]).astype(np.int64)
    w1 = (W1.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    w2 = (W2.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    bias = w1 @ w2
    p1 = special.softmax((U1[0, 0] + bias[anchor]) / T)
    P = np.stack([p1[x] * special.softmax((U1[0, 1] + bias[x]) / T) for x in range(V)])
    counts = np.bincount(paths[:, 0] * V + paths[:, 1], minlength=V * V).astype(np.float64)
    exp = P.reshape(-1) * N
    small = exp < 5
    obs = np.concatenate([counts[~small], [counts[small].sum()]])
    ex = np.concatenate([exp[~small], [exp[small].sum()]])
    assert stats.chisquare(obs, ex).pvalue > 0.01
    # the block marginal at each position (stage 1 alone)
    blocks0 = np.bincount(paths[:, 0] // 16, minlength=4)
    mass0 = np.add.reduceat(p1, [0, 16, 32, 48])
    assert stats.chisquare(blocks0, mass0 * N).pvalue > 0.01
    blocks1 = np.bincount(paths[:, 1] // 16, minlength=4)
    mass1 = np.add.reduceat(P.sum(axis=0), [0, 16, 32, 48])
    assert stats.chisquare(blocks1, mass1 * N).pvalue > 0.01
    assert mass0.max() / mass0.min() > 3  # the blocks' masses are far from equal
    lp = host(out["logprobs"])[:5000].sum(1)
    assert np.allclose(lp, np.log(P.reshape(-1)[paths[:5000, 0] * V + paths[:5000, 1]]),
                       atol=3 * LOGPROB_TOL)


# --------------------------------------------------------------------- selector
def _selector_inputs(seed, B, K, V, r, d=0, gated=False):
    return make_inputs(seed, B, K, V, r, d=d, gated=gated, selector=True)


@pytest.mark.parametrize("gated", [False, True])
def test_selector_scores_match_oracle(dsp, gated):
    B, K, V, r, d, k = 6, 5, 1000, 256, 128, 16
    inp = _selector_inputs(31, B, K, V, r, d=d, gated=gated)
    out = binding.selector_scores(dsp, dev(inp.U), bf(inp.A), bf(inp.Bt), dev(inp.anchors),
                                  topk=k, h=bf(inp.h) if gated else None,
                                  Wg=bf(inp.Wg) if gated else None)
    torch.cuda.synchronize()
    assert dsp.status() == 0
    top = oracle.topk(inp.U, k)
    assert np.array_equal(host(out["cand"]), top["cand"])
    assert np.array_equal(host(out["cand_U"]), top["cval"].astype(np.float32))
    H = oracle.gate(inp.h, inp.Wg) if gated else None
    S = oracle.pair_scores(top["cand"], top["cval"], inp.A, inp.Bt, inp.anchors, V=V, H=H)
    assert np.abs(host(out["scores"]) - S).max() <= LOGPROB_TOL


def test_topk_ties_and_ragged_rows(dsp):
    rng = np.random.default_rng(7)
    B, K, V = 3, 4, 1012
    U = np.round(rng.standard_normal((B, K, V)) * 2).astype(np.float32)   # heavy ties
    A = bf16_bits((rng.standard_normal((V, 16)) * 0.02).astype(np.float32))
    anchors = np.zeros(B, np.int32)
    for k in (1, 16, 32):
        out = binding.selector_scores(dsp, dev(U), bf(A), bf(A), dev(anchors), topk=k)
        torch.cuda.synchronize()
        ref = oracle.topk(U, k)
        assert np.array_equal(host(out["cand"]), ref["cand"])


@pytest.mark.parametrize("B,K,V", [(2, 3, 50012), (50, 20, 1012), (1, 2, 151936)])
def test_topk_streaming_shapes(dsp, B, K, V):
    """Rows split into pieces (few rows, long vocabulary) and CTAs scanning several
    rows in turn (many short rows); heavy ties across pieces and warp slices, plus an
    ascending row (every element enters a list) and a descending one."""
    rng = np.random.default_rng(B * 100003 + V)
    U = np.round(rng.standard_normal((B, K, V)) * 3).astype(np.float32)
    U[0, 0] = np.arange(V, dtype=np.float32)
    U[0, 1] = -np.arange(V, dtype=np.float32)
    A = bf16_bits((rng.standard_normal((V, 16)) * 0.02).astype(np.float32))
    anchors = np.zeros(B, np.int32)
    for k in (1, 16, 32):
        out = binding.selector_scores(dsp, dev(U), bf(A), bf(A), dev(anchors), topk=k)
        torch.cuda.synchronize()
        assert dsp.status() == 0
        ref = oracle.topk(U, k)
        assert np.array_equal(host(out["cand"]), ref["cand"]), k
        assert np.array_equal(host(out["cand_U"]), ref["cval"].astype(np.float32)), k


@pytest.mark.parametrize("r,gated", [(64, True), (48, False)])
def test_pair_scores_k_below_16_and_above(dsp, r, gated):
    """The 4 x 4 register-tiled path (k <= 16, here 5 and 16) and the one-thread-per-
    score path (k = 24) against the oracle; gated, and with a rank that is not a
    multiple of the 64-element split between the two half-warps."""
    B, K, V, d = 7, 5, 2000, 64
    inp = _selector_inputs(36, B, K, V, r, d=d, gated=gated)
    H = oracle.gate(inp.h, inp.Wg) if gated else None
    for k in (5, 16, 24):
        out = binding.selector_scores(dsp, dev(inp.U), bf(inp.A), bf(inp.Bt), dev(inp.anchors),
                                      topk=k, h=bf(inp.h) if gated else None,
                                      Wg=bf(inp.Wg) if gated else None)
        torch.cuda.synchronize()
        assert dsp.status() == 0
        top = oracle.topk(inp.U, k)
        assert np.array_equal(host(out["cand"]), top["cand"])
        S = oracle.pair_scores(top["cand"], top["cval"], inp.A, inp.Bt, inp.anchors, V=V, H=H)
        assert np.abs(host(out["scores"]) - S).max() <= LOGPROB_TOL, k


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_walk_matches_oracle(dsp, T):
    B, K, V, r, d, k = 40, 6, 1000, 256, 128, 16
    inp = _selector_inputs(32, B, K, V, r, d=d)
    sc = binding.selector_scores(dsp, dev(inp.U), bf(inp.A), bf(inp.Bt), dev(inp.anchors), topk=k)
    wk = binding.selector_walk(dsp, sc["cand"], sc["scores"], dev(inp.anchors), V=V,
                               temperature=T, seed=7)
    torch.cuda.synchronize()
    top = oracle.topk(inp.U, k)
    assert np.array_equal(host(sc["cand"]), top["cand"])
    S = oracle.pair_scores(top["cand"], top["cval"], inp.A, inp.Bt, inp.anchors, V=V)
    ref = oracle.walk(top["cand"], S, temperature=T, seed=7)
    check_sequences(host(wk["tokens"]), host(wk["logprobs"]), ref, what="walk")


def test_walk_with_fused_confidence(dsp):
    B, K, V, r, d, k = 10, 6, 1000, 64, 128, 16
    inp = make_inputs(33, B, K, V, r, d=d, selector=True, confidence=True)
    sc = binding.selector_scores(dsp, dev(inp.U), bf(inp.A), bf(inp.Bt), dev(inp.anchors), topk=k)
    conf = binding.Confidence(h=bf(inp.h), w=bf(inp.w_conf), bias=0.0, threshold=0.3)
    wk = binding.selector_walk(dsp, sc["cand"], sc["scores"], dev(inp.anchors), V=V,
                               A=bf(inp.A), temperature=1.0, seed=3, conf=conf)
    torch.cuda.synchronize()
    top = oracle.topk(inp.U, k)
    assert np.array_equal(host(sc["cand"]), top["cand"])
    S = oracle.pair_scores(top["cand"], top["cval"], inp.A, inp.Bt, inp.anchors, V=V)
    walked = oracle.walk(top["cand"], S, temperature=1.0, seed=3)
    ref = oracle.confidence(inp.h, inp.A, inp.anchors, walked["tokens"], inp.w_conf,
                            threshold=0.3)
    _check_confidence(host(wk["tokens"]), walked["tokens"], wk, ref, 0.3)


def test_walk_with_k_equal_V_is_the_full_head_on_gpu(dsp):
    """Top-k execution with k = V reproduces the Markov head's draws (equivalence page)."""
    B, K, V, r = 64, 6, 32, 16
    inp = make_inputs(34, B, K, V, r, weight_std=0.4)
    Bt = np.ascontiguousarray(inp.W2.T)
    sc = binding.selector_scores(dsp, dev(inp.U), bf(inp.W1), bf(Bt), dev(inp.anchors), topk=V)
    for T in (1.0, 0.0):
        wk = binding.selector_walk(dsp, sc["cand"], sc["scores"], dev(inp.anchors), V=V,
                                   temperature=T, seed=12)
        torch.cuda.synchronize()
        ref = oracle.markov_draft(inp.U, inp.W1, inp.W2, inp.anchors, temperature=T, seed=12)
        check_sequences(host(wk["tokens"]), host(wk["logprobs"]), ref,
                        what="walk k=V vs full head")


def test_walk_top16_is_the_masked_full_head_on_gpu(dsp):
    B, K, V, r, k = 64, 6, 200, 16, 16
    inp = make_inputs(35, B, K, V, r, weight_std=0.4)
    Bt = np.ascontiguousarray(inp.W2.T)
    sc = binding.selector_scores(dsp, dev(inp.U), bf(inp.W1), bf(Bt), dev(inp.anchors), topk=k)
    wk = binding.selector_walk(dsp, sc["cand"], sc["scores"], dev(inp.anchors), V=V,
                               temperature=1.0, seed=13)
    torch.cuda.synchronize()
    cand = oracle.topk(inp.U, k)["cand"]
    assert np.array_equal(host(sc["cand"]), cand)
    Um = np.full_like(inp.U, -np.inf)
    np.put_along_axis(Um, cand, np.take_along_axis(inp.U, cand, -1), -1)
    ref = oracle.markov_draft(Um, inp.W1, inp.W2, inp.anchors, temperature=1.0, seed=13)
    check_sequences(host(wk["tokens"]), host(wk["logprobs"]), ref,
                    what="walk k=16 vs masked head")
