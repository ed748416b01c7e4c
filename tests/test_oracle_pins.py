"""Pins of the fp64 oracle against what the DSpark pages and the mathematics fix.

None of these tests retypes the oracle's loops: each compares the oracle with
a printed value (tests/golden), a known-answer vector, a closed form evaluated
by an independent library routine (numpy/scipy), an exact special case the
pages state, or an exhaustive enumeration of the sampled distribution.
"""

import json
import os

import numpy as np
import pytest
from scipy import special, stats

from synth import bf16_bits, bf16_to_f32, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f64(bits):
    return bf16_to_f32(bits).astype(np.float64)


def small_inputs(seed, B, K, V, r, std=0.02, d=0, **kw):
    return make_inputs(seed, B, K, V, r, d=d, weight_std=std, **kw)


# --------------------------------------------------------------------------- RNG
def test_philox_known_answers(orc):
    kat = json.load(open(os.path.join(GOLDEN, "philox4x32_10_kat.json")))
    for vec in kat["vectors"]:
        ctr = [int(x, 16) for x in vec["ctr"]]
        key = [int(x, 16) for x in vec["key"]]
        out = [int(x, 16) for x in vec["out"]]
        assert list(orc.philox4x32_10(ctr, key)) == out


def test_uniform_grid_and_word_selection(orc):
    seed = 0x1234_5678_9ABC_DEF0
    for (b, k, v) in [(0, 0, 0), (3, 7, 5), (127, 15, 151935), (1, 2, 4)]:
        out = orc.philox4x32_10([v >> 2, k, b, 0], [seed & 0xFFFFFFFF, seed >> 32])
        u = orc.uniform(seed, b, k, v)
        # u = (2 * (word & 0x7FFFFF) + 1) * 2^-24: an odd multiple of 2^-24 inside (0, 1)
        assert u == ((int(out[v & 3]) & 0x7FFFFF) * 2 + 1) * 2.0 ** -24
        assert 0.0 < u < 1.0
        assert np.float32(u) == u  # exactly representable in fp32
        # the block-race streams: one call per two blocks of the same residue mod 4,
        # words (2h, 2h + 1) = (stage 1, stage 2) of the block with h = (blk >> 2) & 1
        blk = v >> 4
        key = [seed & 0xFFFFFFFF, seed >> 32]
        o = orc.philox4x32_10([blk >> 3, k, b, 1 + (blk & 3)], key)
        h = (blk >> 2) & 1
        assert orc.block_uniform(seed, b, k, blk) == \
            ((int(o[2 * h]) & 0x7FFFFF) * 2 + 1) * 2.0 ** -24
        assert orc.within_uniform(seed, b, k, blk) == \
            ((int(o[2 * h + 1]) & 0x7FFFFF) * 2 + 1) * 2.0 ** -24


def test_uniform_is_uniform(orc):
    us = np.array([orc.uniform(7, b, 3, v) for b in range(20) for v in range(2000)])
    counts, _ = np.histogram(us, bins=50, range=(0, 1))
    assert stats.chisquare(counts).pvalue > 1e-3
    # neighbouring words of one block and neighbouring requests are uncorrelated
    assert abs(np.corrcoef(us[:-1], us[1:])[0, 1]) < 0.02
    # the block-race streams: uniform, and stage 1 / stage 2 of a block independent
    u1 = np.array([orc.block_uniform(7, b, 3, blk) for b in range(20) for blk in range(1000)])
    u2 = np.array([orc.within_uniform(7, b, 3, blk) for b in range(20) for blk in range(1000)])
    for x in (u1, u2):
        assert stats.chisquare(np.histogram(x, bins=50, range=(0, 1))[0]).pvalue > 1e-3
    assert abs(np.corrcoef(u1, u2)[0, 1]) < 0.03
    assert abs(np.corrcoef(u1[:-1], u1[1:])[0, 1]) < 0.03


# ------------------------------------------------------------------- closed forms
def test_rank_zero_reproduces_base_logits_exactly(orc):
    """--markov-rank 0 disables the head, leaving the base logits (vLLM guide, "Markov Head")."""
    inp = small_inputs(1, 3, 4, 200, 16)
    prev = np.random.default_rng(0).integers(0, 200, size=(3, 4)).astype(np.int32)
    out = orc.markov_logits(inp.U, None, None, prev, temperature=1.0)
    assert np.array_equal(out["logits"], inp.U.astype(np.float64))
    assert np.allclose(out["lse"], special.logsumexp(inp.U.astype(np.float64), axis=-1),
                       rtol=0, atol=1e-12)


@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("T", [1.0, 0.7, 0.0])
def test_teacher_forced_logits_match_numpy(orc, gated, T):
    """logits_k = U_k + (W1[a] (.) H)^T W2 (equivalence page, Markov-head and gated rules)."""
    B, K, V, r, d = 3, 5, 96, 32, 24
    inp = small_inputs(2, B, K, V, r, std=0.3, d=d, gated=gated)
    prev = np.random.default_rng(1).integers(0, V, size=(B, K)).astype(np.int32)
    H = orc.gate(inp.h, inp.Wg) if gated else None
    out = orc.markov_logits(inp.U, inp.W1, inp.W2, prev, temperature=T, H=H)
    e = f64(inp.W1)[prev]  # [B, K, r]
    if gated:
        e = e * special.expit(np.einsum("bkd,dr->bkr", f64(inp.h), f64(inp.Wg)))
    ref = inp.U.astype(np.float64) + e @ f64(inp.W2)
    assert np.allclose(out["logits"], ref, rtol=1e-13, atol=1e-12)
    Tp = T if T > 0 else 1.0
    assert np.allclose(out["lse"], special.logsumexp(ref / Tp, axis=-1), rtol=0, atol=1e-12)
    # local normalisation: the per-position distribution sums to one
    p = np.exp(out["logits"] / Tp - out["lse"][..., None])
    assert np.allclose(p.sum(-1), 1.0, atol=1e-12)


def test_teacher_forced_subset_rows(orc):
    inp = small_inputs(3, 5, 3, 64, 16, std=0.3)
    prev = np.random.default_rng(2).integers(0, 64, size=(5, 3)).astype(np.int32)
    full = orc.markov_logits(inp.U, inp.W1, inp.W2, prev)
    part = orc.markov_logits(inp.U, inp.W1, inp.W2, prev, b0=2, nb=2)
    assert np.array_equal(part["logits"], full["logits"][2:4])
    assert np.array_equal(part["lse"], full["lse"][2:4])


def test_gate_matches_numpy(orc):
    inp = small_inputs(4, 2, 3, 16, 32, d=40, gated=True)
    H = orc.gate(inp.h, inp.Wg)
    ref = special.expit(np.einsum("bkd,dr->bkr", f64(inp.h), f64(inp.Wg)))
    assert np.allclose(H, ref, rtol=1e-14, atol=1e-15)


def test_gated_head_with_unit_gate_equals_vanilla(orc):
    """H = 1 turns the gated rule into the vanilla Markov head (equivalence page)."""
    B, K, V, r, d = 4, 5, 128, 32, 16
    inp = small_inputs(5, B, K, V, r, std=0.3)
    h = np.full((B, K, d), 0x3F80, np.uint16)        # 1.0
    Wg = np.full((d, r), 0x4080, np.uint16)          # 4.0 -> h.Wg = 64, sigmoid == 1.0 in fp64
    H = orc.gate(h, Wg)
    assert np.all(H == 1.0)
    for T in (1.0, 0.0):
        a = orc.markov_draft(inp.U, inp.W1, inp.W2, inp.anchors, temperature=T, seed=3)
        g = orc.markov_draft(inp.U, inp.W1, inp.W2, inp.anchors, temperature=T, seed=3, H=H)
        for key in ("tokens", "logprobs", "margins"):
            assert np.array_equal(a[key], g[key])


# ---------------------------------------------------------------------- RNN head
# Reading of the RNN head (DSpark explainer, "The RNN head"; "Repair the Joint",
# "Fix 1"): s_k = a_k (.) s_{k-1} + g_k (.) W1[x_{k-1}], s_{-1} = 0, bias_k = s_k W2.
def _rnn_unrolled(W1, prev, A, G):
    """The recurrence's solution in closed form: s_k = sum_{j<=k} (prod_{j<i<=k} a_i) g_j
    (.) W1[x_{j-1}], from cumulative products (no step-by-step update)."""
    B, K, r = A.shape
    E = f64(W1)[prev] * (1.0 if G is None else G)            # [B, K, r] inputs
    S = np.zeros((B, K, r))
    for k in range(K):
        # weight of input j at position k: prod of a over positions j+1..k
        w = np.ones((B, k + 1, r))
        if k > 0:
            rev = np.cumprod(A[:, k:0:-1], axis=1)[:, ::-1]  # [B, k, r]: prod_{i=j+1..k} a_i
            w[:, :k] = rev
        S[:, k] = (w * E[:, :k + 1]).sum(axis=1)
    return S


@pytest.mark.parametrize("gated", [False, True])
def test_rnn_with_zero_decay_is_the_markov_head(orc, gated):
    """a = 0 removes the state: the RNN head is then the gated head (input gate g = H)
    and, with g = 1, the vanilla Markov head -- bitwise, draft and teacher-forced."""
    B, K, V, r, d = 5, 6, 128, 32, 16
    inp = small_inputs(21, B, K, V, r, std=0.3, d=d, gated=True)
    H = orc.gate(inp.h, inp.Wg) if gated else None
    A = np.zeros((B, K, r))
    for T in (1.0, 0.7, 0.0):
        m = orc.markov_draft(inp.U, inp.W1, inp.W2, inp.anchors, temperature=T, seed=4, H=H)
        n = orc.rnn_draft(inp.U, inp.W1, inp.W2, inp.anchors, A, G=H, temperature=T, seed=4)
        for key in ("tokens", "logprobs", "margins"):
            assert np.array_equal(m[key], n[key])
    prev = np.random.default_rng(22).integers(0, V, size=(B, K)).astype(np.int32)
    ml = orc.markov_logits(inp.U, inp.W1, inp.W2, prev, H=H)
    nl = orc.rnn_logits(inp.U, inp.W1, inp.W2, prev, A, G=H)
    assert np.array_equal(ml["logits"], nl["logits"]) and np.array_equal(ml["lse"], nl["lse"])


@pytest.mark.parametrize("lam", [0.5, 0.75])
def test_rnn_state_is_a_geometric_series_under_constant_decay(orc, lam):
    """The same predecessor t at every position, a = lam, g = 1: the state is the partial
    geometric series s_k = (1 - lam^(k+1)) / (1 - lam) W1[t]."""
    B, K, V, r = 2, 7, 96, 32
    inp = small_inputs(23, B, K, V, r, std=0.3)
    prev = np.repeat(np.array([[5], [61]], np.int32), K, axis=1)
    A = np.full((B, K, r), lam)
    out = orc.rnn_logits(inp.U, inp.W1, inp.W2, prev, A)
    coef = (1.0 - lam ** np.arange(1, K + 1)) / (1.0 - lam)            # [K]
    bias_t = f64(inp.W1)[prev[:, 0]] @ f64(inp.W2)                       # [B, V]
    ref = inp.U.astype(np.float64) + coef[None, :, None] * bias_t[:, None, :]
    assert np.allclose(out["logits"], ref, rtol=1e-13, atol=1e-13)


def test_rnn_unrolled_state_matches_teacher_forced_logits(orc):
    """Random gates and predecessors: logits_k = U_k + s_k W2 with s_k from the unrolled
    (cumulative-product) solution of the recurrence."""
    B, K, V, r, d = 4, 6, 80, 32, 24
    inp = small_inputs(24, B, K, V, r, std=0.3, d=d, gated=True)
    rng = np.random.default_rng(25)
    prev = rng.integers(0, V, size=(B, K)).astype(np.int32)
    A = rng.uniform(0.0, 1.0, (B, K, r))
    G = orc.gate(inp.h, inp.Wg)
    for T in (1.0, 0.7):
        out = orc.rnn_logits(inp.U, inp.W1, inp.W2, prev, A, G=G, temperature=T)
        ref = inp.U.astype(np.float64) + _rnn_unrolled(inp.W1, prev, A, G) @ f64(inp.W2)
        assert np.allclose(out["logits"], ref, rtol=1e-12, atol=1e-12)
        assert np.allclose(out["lse"], special.logsumexp(ref / T, axis=-1), rtol=0, atol=1e-11)
    # the draft forced onto the same predecessors gives the same log-probabilities
    forced = np.concatenate([prev[:, 1:], prev[:, :1]], axis=1)
    anchors = prev[:, 0].copy()
    dr = orc.rnn_draft(inp.U, inp.W1, inp.W2, anchors, A, G=G, temperature=1.0, seed=5,
                       forced=forced)
    lp = ref - special.logsumexp(ref, axis=-1)[..., None]
    want = np.take_along_axis(lp, forced[..., None].astype(np.int64), axis=-1)[..., 0]
    assert np.allclose(dr["forced_logprobs"], want, atol=1e-11)


def test_rnn_sampler_matches_exhaustive_joint(orc):
    """2 * 10^5 draws of a V = 8, K = 3 RNN head vs the exhaustive joint
    prod_k softmax(U_k + s_k(x_{<k}) W2), s from the unrolled recurrence on each path."""
    V, K, r, N = 8, 3, 8, 200_000
    rng = np.random.default_rng(26)
    U1 = rng.standard_normal((1, K, V)).astype(np.float32)
    W1 = bf16_bits(rng.normal(0, 0.6, (V, r)).astype(np.float32))
    W2 = bf16_bits(rng.normal(0, 0.6, (r, V)).astype(np.float32))
    A1 = rng.uniform(0.3, 0.9, (1, K, r))
    G1 = rng.uniform(0.5, 1.0, (1, K, r))
    anchor = 3
    U = np.ascontiguousarray(np.broadcast_to(U1, (N, K, V)))
    A = np.ascontiguousarray(np.broadcast_to(A1, (N, K, r)))
    G = np.ascontiguousarray(np.broadcast_to(G1, (N, K, r)))
    out = orc.rnn_draft(U, W1, W2, np.full(N, anchor, np.int32), A, G=G, temperature=1.0, seed=7)
    paths = out["tokens"].astype(np.int64)
    cell = (paths[:, 0] * V + paths[:, 1]) * V + paths[:, 2]
    counts = np.bincount(cell, minlength=V ** K).astype(np.float64)
    P = np.zeros((V,) * K)
    for x1 in range(V):
        for x2 in range(V):
            prev = np.array([[anchor, x1, x2]], np.int32)
            S = _rnn_unrolled(W1, prev, A1, G1)[0]                    # [K, r]
            l = U1[0].astype(np.float64) + S @ f64(W2)
            p = special.softmax(l, axis=-1)
            P[x1, x2, :] = p[0, x1] * p[1, x2] * p[2]
    assert abs(P.sum() - 1) < 1e-12
    assert _chi2_pvalue(counts, P.reshape(-1) * N) > 0.01
    sel = slice(0, 2000)
    assert np.allclose(out["logprobs"][sel].sum(1), np.log(P.reshape(-1)[cell[sel]]), atol=1e-10)


# ----------------------------------------------------------------- sampling rule
def _replicate(inp, n):
    U = np.ascontiguousarray(np.broadcast_to(inp.U[:1], (n,) + inp.U.shape[1:]))
    anchors = np.full(n, inp.anchors[0], np.int32)
    return U, anchors


def _chi2_pvalue(counts, expected):
    small = expected < 5
    obs = np.concatenate([counts[~small], [counts[small].sum()]]) if small.any() else counts
    exp = np.concatenate([expected[~small], [expected[small].sum()]]) if small.any() else expected
    keep = exp > 0
    return stats.chisquare(obs[keep], exp[keep]).pvalue


def test_sampler_matches_exhaustive_joint(orc):
    """Empirical joint of 10^6 draws vs prod_k softmax(U_k + W1[x_{k-1}] W2) over all V^K paths."""
    V, K, r, N = 8, 3, 8, 1_000_000
    rng = np.random.default_rng(11)
    U1 = rng.standard_normal((1, K, V)).astype(np.float32)
    W1 = bf16_bits(rng.normal(0, 0.5, (V, r)).astype(np.float32))
    W2 = bf16_bits(rng.normal(0, 0.5, (r, V)).astype(np.float32))
    anchor = 5
    U = np.ascontiguousarray(np.broadcast_to(U1, (N, K, V)))
    anchors = np.full(N, anchor, np.int32)
    out = orc.markov_draft(U, W1, W2, anchors, temperature=1.0, seed=2024)
    paths = out["tokens"].astype(np.int64)
    cell = (paths[:, 0] * V + paths[:, 1]) * V + paths[:, 2]
    counts = np.bincount(cell, minlength=V ** K).astype(np.float64)
    # exhaustive joint, with numpy softmax rows per predecessor
    bias = f64(W1) @ f64(W2)                       # [V(prev), V]
    P = np.zeros((V,) * K)
    for x1 in range(V):
        p1 = special.softmax(U1[0, 0] + bias[anchor])[x1]
        for x2 in range(V):
            p2 = special.softmax(U1[0, 1] + bias[x1])[x2]
            p3 = special.softmax(U1[0, 2] + bias[x2])
            P[x1, x2, :] = p1 * p2 * p3
    assert abs(P.sum() - 1) < 1e-12
    assert _chi2_pvalue(counts, P.reshape(-1) * N) > 0.01
    # the log-probabilities returned with each draw are the exact conditionals
    sel = slice(0, 2000)
    joint_lp = out["logprobs"][sel].sum(1)
    assert np.allclose(joint_lp, np.log(P.reshape(-1)[cell[sel]]), atol=1e-10)


def test_temperature_scales_the_sampled_softmax(orc):
    """V = 40 spans three 16-token blocks (the last one ragged): the draw's token,
    block and within-block frequencies all follow softmax(U / T)."""
    V, N, T = 40, 300_000, 0.5
    rng = np.random.default_rng(12)
    U1 = (rng.standard_normal((1, 1, V)) * 0.8).astype(np.float32)
    U1[0, 0, 16:32] -= 0.6   # unequal block masses
    U = np.ascontiguousarray(np.broadcast_to(U1, (N, 1, V)))
    out = orc.markov_draft(U, None, None, np.zeros(N, np.int32), temperature=T, seed=99)
    tok = out["tokens"][:, 0]
    counts = np.bincount(tok, minlength=V).astype(np.float64)
    p = special.softmax(U1[0, 0].astype(np.float64) / T)
    assert _chi2_pvalue(counts, p * N) > 0.01
    pb = np.add.reduceat(p, [0, 16, 32])
    assert _chi2_pvalue(np.bincount(tok >> 4, minlength=3).astype(np.float64), pb * N) > 0.01
    assert np.allclose(out["logprobs"][:, 0], np.log(p[tok]), atol=1e-12)
    # margins are the smaller of the block gap and the in-block distance: in (0, ...)
    assert np.all(out["margins"] >= 0) and np.median(out["margins"]) > 1e-3


def test_greedy_is_argmax_of_calibrated_logits(orc):
    inp = small_inputs(6, 3, 6, 256, 32, std=0.3)
    out = orc.markov_draft(inp.U, inp.W1, inp.W2, inp.anchors, temperature=0.0, seed=0)
    prev = np.concatenate([inp.anchors[:, None], out["tokens"][:, :-1]], axis=1)
    logits = inp.U.astype(np.float64) + f64(inp.W1)[prev] @ f64(inp.W2)
    assert np.array_equal(out["tokens"], logits.argmax(-1))
    srt = np.sort(logits, axis=-1)
    assert np.allclose(out["margins"], srt[..., -1] - srt[..., -2], atol=1e-12)
    assert np.allclose(out["logprobs"], logits.max(-1) - special.logsumexp(logits, -1),
                       atol=1e-12)


def test_forced_continuation_on_own_tokens_is_identity(orc):
    inp = small_inputs(7, 4, 5, 128, 16, std=0.3)
    a = orc.markov_draft(inp.U, inp.W1, inp.W2, inp.anchors, temperature=1.0, seed=5)
    f = orc.markov_draft(inp.U, inp.W1, inp.W2, inp.anchors, temperature=1.0, seed=5,
                         forced=a["tokens"])
    assert np.array_equal(a["tokens"], f["tokens"])
    assert np.array_equal(a["logprobs"], f["forced_logprobs"])
    part = orc.markov_draft(inp.U, inp.W1, inp.W2, inp.anchors, temperature=1.0, seed=5,
                            b0=1, nb=2)
    assert np.array_equal(part["tokens"], a["tokens"][1:3])


def test_np_torch_worked_example(orc):
    """The np/torch tables: product of marginals without the head, the true joint with it."""
    gold = json.load(open(os.path.join(GOLDEN, "np_torch_tables.json")))
    NP, TORCH, ARRAY, TENSOR, PREFIX = 0, 1, 2, 3, 4
    V, K, N = 5, 2, 20000
    U1 = np.full((1, K, V), -30.0, np.float32)
    U1[0, 0, [NP, TORCH]] = 0.0
    U1[0, 1, [ARRAY, TENSOR]] = 0.0
    U = np.ascontiguousarray(np.broadcast_to(U1, (N, K, V)))
    anchors = np.full(N, PREFIX, np.int32)

    def table(out):
        t = np.zeros((2, 2))
        for x1, x2 in out["tokens"]:
            t[int(x1) - NP, int(x2) - ARRAY] += 1
        return t / N

    # mean-field (rank 0): every cell is the product of the two marginals
    mf = orc.markov_draft(U, None, None, anchors, temperature=1.0, seed=1)
    assert np.all(np.abs(table(mf) - np.array(gold["product_of_marginals"])) < 0.015)
    lp = mf["logprobs"].sum(1)
    assert np.allclose(np.exp(lp), gold["product_of_marginals"][0][0], atol=1e-9)

    # Markov head with a rank-2 coupling: np -> .array, torch -> .tensor
    r = 2
    W1 = np.zeros((V, r), np.float32)
    W1[NP] = (1, 0)
    W1[TORCH] = (0, 1)
    W2 = np.zeros((r, V), np.float32)
    W2[:, ARRAY] = (0, -30)
    W2[:, TENSOR] = (-30, 0)
    mk = orc.markov_draft(U, bf16_bits(W1), bf16_bits(W2), anchors, temperature=1.0, seed=1)
    t = table(mk)
    joint = np.array(gold["true_joint"])
    assert np.all(t[joint == 0] == 0)
    assert np.all(np.abs(t - joint) < 0.015)
    assert np.allclose(t.sum(1), gold["true_margins_rows"], atol=0.015)
    assert np.allclose(t.sum(0), gold["true_margins_cols"], atol=0.015)
    assert np.allclose(np.exp(mk["logprobs"].sum(1)), 0.5, atol=1e-9)


# ----------------------------------------------------------------------- selector
def test_topk_matches_lexsort(orc):
    rng = np.random.default_rng(8)
    U = np.round(rng.standard_normal((3, 4, 300)) * 2).astype(np.float32)  # many exact ties
    for k in (1, 16, 32):
        out = orc.topk(U, k)
        for b in range(3):
            for t in range(4):
                order = np.lexsort((np.arange(300), -U[b, t].astype(np.float64)))
                assert np.array_equal(out["cand"][b, t], order[:k])
                assert np.array_equal(out["cval"][b, t], U[b, t, order[:k]])
                assert out["margin"][b, t] == U[b, t, order[k - 1]] - U[b, t, order[k]]


@pytest.mark.parametrize("gated", [False, True])
def test_pair_scores_match_numpy(orc, gated):
    B, K, V, r, d, k = 2, 4, 300, 32, 24, 16
    inp = small_inputs(9, B, K, V, r, std=0.3, d=d, gated=gated, selector=True)
    top = orc.topk(inp.U, k)
    H = orc.gate(inp.h, inp.Wg) if gated else None
    S = orc.pair_scores(top["cand"], top["cval"], inp.A, inp.Bt, inp.anchors, V=V, H=H)
    prev = np.concatenate([np.repeat(inp.anchors[:, None, None], k, axis=2),
                           top["cand"][:, :-1]], axis=1)        # [B, K, k]
    Ap = f64(inp.A)[prev]                                        # [B, K, k, r]
    if gated:
        Ap = Ap * H[:, :, None, :]
    Bc = f64(inp.Bt)[top["cand"]]                                # [B, K, k, r]
    ref = top["cval"][:, :, None, :] + np.einsum("btiq,btjq->btij", Ap, Bc)
    assert np.allclose(S, ref, rtol=1e-13, atol=1e-12)


def test_walk_with_k_equal_V_is_the_full_head(orc):
    """Top-k execution with k = V recovers the Markov head exactly (equivalence page)."""
    B, K, V, r = 64, 6, 32, 16
    inp = small_inputs(10, B, K, V, r, std=0.4)
    A, Bt = inp.W1, np.ascontiguousarray(inp.W2.T)
    top = orc.topk(inp.U, V)
    S = orc.pair_scores(top["cand"], top["cval"], A, Bt, inp.anchors, V=V)
    for T in (1.0, 0.7, 0.0):
        full = orc.markov_draft(inp.U, inp.W1, inp.W2, inp.anchors, temperature=T, seed=21)
        wk = orc.walk(top["cand"], S, temperature=T, seed=21)
        assert np.array_equal(full["tokens"], wk["tokens"])
        assert np.allclose(full["logprobs"], wk["logprobs"], atol=1e-12)


def test_walk_top16_is_the_masked_full_head(orc):
    """k = 16: the walk equals the full head with logits -inf outside each candidate set."""
    B, K, V, r, k = 64, 6, 200, 16, 16
    inp = small_inputs(12, B, K, V, r, std=0.4)
    top = orc.topk(inp.U, k)
    S = orc.pair_scores(top["cand"], top["cval"], inp.W1, np.ascontiguousarray(inp.W2.T),
                        inp.anchors, V=V)
    Um = np.full_like(inp.U, -np.inf)
    np.put_along_axis(Um, top["cand"], np.take_along_axis(inp.U, top["cand"], -1), -1)
    for T in (1.0, 0.0):
        full = orc.markov_draft(Um, inp.W1, inp.W2, inp.anchors, temperature=T, seed=4)
        wk = orc.walk(top["cand"], S, temperature=T, seed=4)
        assert np.array_equal(full["tokens"], wk["tokens"])
        assert np.allclose(full["logprobs"], wk["logprobs"], atol=1e-12)
        assert np.all(np.isin(wk["tokens"], top["cand"].reshape(B, -1)))


def test_walk_forced_continuation(orc):
    B, K, V, r, k = 8, 5, 200, 16, 16
    inp = small_inputs(13, B, K, V, r, std=0.4, selector=True)
    top = orc.topk(inp.U, k)
    S = orc.pair_scores(top["cand"], top["cval"], inp.A, inp.Bt, inp.anchors, V=V)
    a = orc.walk(top["cand"], S, temperature=1.0, seed=8)
    f = orc.walk(top["cand"], S, temperature=1.0, seed=8, forced=a["tokens"])
    assert np.array_equal(a["tokens"], f["tokens"])
    assert np.array_equal(a["logprobs"], f["forced_logprobs"])


# --------------------------------------------------------------------- confidence
@pytest.mark.parametrize("with_markov", [True, False])
def test_confidence_closed_form(orc, with_markov):
    B, K, V, r, d = 5, 7, 64, 16, 32
    inp = small_inputs(14, B, K, V, r, d=d, confidence=True)
    w = inp.w_conf if with_markov else inp.w_conf[:d]
    tokens = np.random.default_rng(3).integers(0, V, size=(B, K)).astype(np.int32)
    out = orc.confidence(inp.h, inp.W1, inp.anchors, tokens, w, bias=0.25,
                         with_markov=with_markov, threshold=0.3, V=V)
    prev = np.concatenate([inp.anchors[:, None], tokens[:, :-1]], axis=1)
    z = np.einsum("bkd,d->bk", f64(inp.h), f64(w[:d])) + 0.25
    if with_markov:
        z = z + f64(inp.W1)[prev] @ f64(inp.w_conf[d:])
    c = special.expit(z)
    assert np.allclose(out["conf"], c, rtol=1e-13, atol=1e-15)
    assert np.allclose(out["cumprod"], np.cumprod(c, axis=1), rtol=1e-13)
    assert np.all(np.diff(out["cumprod"], axis=1) <= 0)        # survival never grows
    assert np.array_equal(out["verify_len"], (np.cumprod(c, axis=1) >= 0.3).sum(1))


def test_confidence_threshold_extremes_and_monotonicity(orc):
    B, K, V, r, d = 6, 9, 64, 16, 32
    inp = small_inputs(15, B, K, V, r, d=d, confidence=True)
    tokens = np.random.default_rng(4).integers(0, V, size=(B, K)).astype(np.int32)
    lens = []
    for th in (0.0, 0.05, 0.1, 0.3, 0.6, 0.9, 1.0 + 1e-9):
        out = orc.confidence(inp.h, inp.W1, inp.anchors, tokens, inp.w_conf, threshold=th, V=V)
        lens.append(out["verify_len"])
    assert np.all(lens[0] == K)          # threshold 0: verify the whole block
    assert np.all(lens[-1] == 0)         # threshold above 1: verify nothing
    assert np.all(np.diff(np.stack(lens), axis=0) <= 0)


def test_head_parameter_count():
    """2 * V * r = 77.8M parameters for a 151936-token vocabulary at rank 256 (explainer's ablation)."""
    assert 2 * 151936 * 256 == 77_791_232


# ------------------------------------------------------------------ verification
def _verify_case(orc, N, V, K, r, seed, Td=1.0, Tt=1.0, std=0.5, ell=None):
    """N requests sharing one draft head and one target table; the drafted tokens
    are the oracle draft's own draws (tokens must be draws from q for the
    acceptance rule to be lossless)."""
    rng = np.random.default_rng(seed)
    U1 = rng.standard_normal((1, K, V)).astype(np.float32)
    W1 = bf16_bits(rng.normal(0, std, (V, r)).astype(np.float32))
    W2 = bf16_bits(rng.normal(0, std, (r, V)).astype(np.float32))
    P1 = (rng.standard_normal((1, K + 1, V)) * 1.2).astype(np.float32)
    U = np.ascontiguousarray(np.broadcast_to(U1, (N, K, V)))
    P = np.ascontiguousarray(np.broadcast_to(P1, (N, K + 1, V)))
    anchors = np.full(N, 3, np.int32)
    drafted = orc.markov_draft(U, W1, W2, anchors, temperature=Td, seed=seed + 1)
    out = orc.verify(P, U, W1, W2, anchors, drafted["tokens"], draft_temperature=Td,
                     target_temperature=Tt, seed=seed + 2, ell=ell)
    return U1, W1, W2, P1, drafted, out


def _softmax_rows(x, T):
    return special.softmax(x.astype(np.float64) / T, axis=-1)


def test_verify_commits_the_target_distribution(orc):
    """Lossless acceptance: the first committed token is distributed as p_0, and, once
    position 1 is reached, the second as p_1; the acceptance rate at position 0 is
    1 - TV(p_0, q_0) (the confidence label's definition)."""
    N, V, K, r = 200_000, 40, 2, 8
    U1, W1, W2, P1, drafted, out = _verify_case(orc, N, V, K, r, seed=41)
    x, n, y = drafted["tokens"], out["n_acc"], out["next_token"]
    c0 = np.where(n >= 1, x[:, 0], y)
    p0 = _softmax_rows(P1[0, 0], 1.0)
    assert _chi2_pvalue(np.bincount(c0, minlength=V).astype(np.float64), p0 * N) > 0.01
    reached = n >= 1
    c1 = np.where(n[reached] >= 2, x[reached, 1], y[reached])
    p1 = _softmax_rows(P1[0, 1], 1.0)
    assert _chi2_pvalue(np.bincount(c1, minlength=V).astype(np.float64), p1 * reached.sum()) > 0.01
    # q_0: the draft's softmax after the anchor
    q0 = _softmax_rows(U1[0, 0] + f64(W1)[3] @ f64(W2), 1.0)
    acc = 1.0 - 0.5 * np.abs(p0 - q0).sum()
    rate = reached.mean()
    assert abs(rate - acc) < 4 * np.sqrt(acc * (1 - acc) / N)
    # the reported acceptance probabilities are min(1, p/q) of the drafted tokens
    assert np.allclose(out["accept_prob"][:, 0], np.minimum(1.0, p0[x[:, 0]] / q0[x[:, 0]]),
                       atol=1e-12)


def test_verify_greedy_target_is_the_argmax_rule(orc):
    N, V, K, r = 300, 64, 4, 8
    U1, W1, W2, P1, drafted, out = _verify_case(orc, N, V, K, r, seed=42, Tt=0.0)
    am = P1[0].argmax(-1)                               # [K+1]
    x = drafted["tokens"]
    match = x == am[None, :K]
    n_ref = np.where(match.all(1), K, np.argmin(match, axis=1))
    assert np.array_equal(out["n_acc"], n_ref)
    assert np.array_equal(out["next_token"], am[n_ref])


def test_verify_target_equal_to_draft_accepts_every_token(orc):
    """p == q: every min(1, p/q) is one, so the whole window is accepted and the bonus
    comes from the target's row after it."""
    N, V, K, r = 20_000, 48, 3, 8
    rng = np.random.default_rng(43)
    inp = make_inputs(44, N, K, V, r, weight_std=0.5)
    drafted = orc.markov_draft(inp.U, inp.W1, inp.W2, inp.anchors, temperature=0.8, seed=5)
    prev = np.concatenate([inp.anchors[:, None], drafted["tokens"][:, :-1]], axis=1)
    lg = orc.markov_logits(inp.U, inp.W1, inp.W2, prev)["logits"]
    bonus = np.broadcast_to(rng.standard_normal((1, 1, V)), (N, 1, V))
    P = np.concatenate([lg, bonus], axis=1).astype(np.float32)
    # the fp32 rounding of P makes p and q differ by ~1e-7: use P's own rounding on both sides
    U32 = (P[:, :K] - (lg - inp.U)).astype(np.float32)
    out = orc.verify(P, U32, inp.W1, inp.W2, inp.anchors, drafted["tokens"], draft_temperature=0.8,
                     target_temperature=0.8, seed=6)
    assert (out["n_acc"] == K).mean() > 0.995
    full = out["n_acc"] == K
    pb = _softmax_rows(P[0, K], 0.8)
    cnt = np.bincount(out["next_token"][full], minlength=V).astype(np.float64)
    assert _chi2_pvalue(cnt, pb * full.sum()) > 0.01


def test_verify_window_zero_draws_the_bonus_at_position_zero(orc):
    N, V, K, r = 100_000, 40, 3, 8
    U1, W1, W2, P1, drafted, out = _verify_case(orc, N, V, K, r, seed=45,
                                                ell=np.zeros(100_000, np.int32))
    assert np.all(out["n_acc"] == 0)
    p0 = _softmax_rows(P1[0, 0], 1.0)
    assert _chi2_pvalue(np.bincount(out["next_token"], minlength=V).astype(np.float64), p0 * N) > 0.01
    assert np.all(out["accept_prob"] == -1.0)


def test_verify_greedy_draft_accepts_with_the_target_probability(orc):
    """Td = 0: q is one-hot at the drafted token, so it survives with probability p(x)."""
    N, V, K, r = 100_000, 40, 1, 8
    U1, W1, W2, P1, drafted, out = _verify_case(orc, N, V, K, r, seed=46, Td=0.0)
    x = drafted["tokens"][0, 0]
    assert np.all(drafted["tokens"][:, 0] == x)        # greedy draft: one token
    p = _softmax_rows(P1[0, 0], 1.0)[x]
    rate = (out["n_acc"] >= 1).mean()
    assert abs(rate - p) < 4 * np.sqrt(p * (1 - p) / N)
    # the rejections resample from p with x removed
    rej = out["n_acc"] == 0
    pr = _softmax_rows(P1[0, 0], 1.0)
    pr[x] = 0.0
    pr /= pr.sum()
    cnt = np.bincount(out["next_token"][rej], minlength=V).astype(np.float64)
    assert cnt[x] == 0
    keep = np.arange(V) != x
    assert _chi2_pvalue(cnt[keep], pr[keep] * rej.sum()) > 0.01


# ------------------------------------------------------------------ scheduler
def _survival(rng, R, K, lo=0.55, hi=0.98):
    return np.cumprod(rng.uniform(lo, hi, (R, K)), axis=1)


def test_schedule_constant_throughput_admits_everything(orc):
    a = _survival(np.random.default_rng(70), 6, 5)
    out = orc.schedule(a, np.full(6 * 6 + 1, 3.0))
    assert np.all(out["ell"] == 5)
    assert np.isclose(out["theta"], (6 + a.sum()) * 3.0)


def test_schedule_fixed_token_budget_admits_nothing(orc):
    """SPS(B) = s / B: Theta is s times the mean survival per verified token, and every
    extension survives with probability below the baseline token's 1."""
    R, K = 5, 4
    a = _survival(np.random.default_rng(71), R, K)
    sps = np.array([0.0] + [7.0 / B for B in range(1, R * (K + 1) + 1)])
    out = orc.schedule(a, sps)
    assert np.all(out["ell"] == 0)
    assert np.isclose(out["theta"], 7.0)


def test_schedule_matches_exhaustive_search_when_theta_is_unimodal(orc):
    """For a fixed number of admitted tokens the best set is the top survivors, so with a
    smooth, saturating SPS the greedy's Theta is the optimum over every set of prefixes
    (checked by enumerating all (K+1)^R verify-length vectors)."""
    import itertools
    rng = np.random.default_rng(72)
    R, K = 3, 4
    for trial in range(20):
        a = _survival(rng, R, K, 0.3, 0.99)
        B0 = rng.uniform(3.0, 12.0)
        sps = np.array([1000.0 / (1.0 + (B / B0) ** 2) for B in range(R * (K + 1) + 1)])
        out = orc.schedule(a, sps)
        best = -1.0
        for ell in itertools.product(range(K + 1), repeat=R):
            n = sum(ell)
            th = (R + sum(a[r, :ell[r]].sum() for r in range(R))) * sps[R + n]
            best = max(best, th)
        assert np.isclose(out["theta"], best, rtol=1e-12), trial
        # the reported Theta is the objective of the reported lengths
        th = (R + sum(a[r, :out["ell"][r]].sum() for r in range(R))) * sps[R + out["ell"].sum()]
        assert np.isclose(out["theta"], th, rtol=1e-12)


def test_schedule_stops_at_the_first_dip_of_a_jagged_curve(orc):
    """The greedy stops when the next admission would lower Theta, even if a larger batch
    further on would be better (a jagged SPS, as profiled engines have)."""
    R, K = 4, 4
    a = np.full((R, K), 0.9) ** np.arange(1, K + 1)[None, :]
    sps = np.full(R * (K + 1) + 1, 100.0)
    sps[R + 2] = 60.0                                     # a dip at B = R + 2
    out = orc.schedule(a, sps)
    assert out["ell"].sum() == 1                          # admits one, refuses the second
    assert out["ell"][0] == 1                             # ties go to the first request
    assert 0.0 < out["margin"] < 1.0


# ------------------------------------------------------------------ acceptance label
def test_accept_label_is_the_verifier_acceptance_rate(orc):
    """c*_k is the per-step acceptance probability: across requests sharing one head and
    one target table, the verifier accepts position 0 at rate c*_0, and position 1 (given
    position 0 survived, with its own predecessor) at the mean of c*_1 over those requests."""
    N, V, K, r = 100_000, 40, 2, 8
    U1, W1, W2, P1, drafted, out = _verify_case(orc, N, V, K, r, seed=91)
    U = np.ascontiguousarray(np.broadcast_to(U1, (N, K, V)))
    P = np.ascontiguousarray(np.broadcast_to(P1, (N, K + 1, V)))
    anchors = np.full(N, 3, np.int32)
    lab = orc.accept_label(P, U, W1, W2, anchors, drafted["tokens"], draft_temperature=1.0,
                           target_temperature=1.0)
    c0 = lab[0, 0]
    assert np.allclose(lab[:, 0], c0)                      # same predecessor for everyone
    rate0 = (out["n_acc"] >= 1).mean()
    assert abs(rate0 - c0) < 4 * np.sqrt(c0 * (1 - c0) / N)
    reached = out["n_acc"] >= 1
    c1 = lab[reached, 1].mean()
    rate1 = (out["n_acc"][reached] >= 2).mean()
    assert abs(rate1 - c1) < 4 * np.sqrt(c1 * (1 - c1) / reached.sum())


def test_accept_label_special_cases(orc):
    V, K, r = 48, 3, 8
    inp = make_inputs(92, 5, K, V, r, weight_std=0.5)
    drafted = orc.markov_draft(inp.U, inp.W1, inp.W2, inp.anchors, temperature=1.0, seed=3)
    prev = np.concatenate([inp.anchors[:, None], drafted["tokens"][:, :-1]], axis=1)
    lg = orc.markov_logits(inp.U, inp.W1, inp.W2, prev)["logits"]
    # the target equal to the draft: label 1
    P = np.concatenate([lg, np.zeros((5, 1, V))], axis=1).astype(np.float32)
    U32 = (P[:, :K] - (lg - inp.U)).astype(np.float32)
    lab = orc.accept_label(P, U32, inp.W1, inp.W2, inp.anchors, drafted["tokens"],
                           draft_temperature=1.0, target_temperature=1.0)
    assert np.allclose(lab, 1.0, atol=1e-6)
    # greedy draft: the label is the target probability of the drafted token
    Pr = np.random.default_rng(93).standard_normal((5, K + 1, V)).astype(np.float32)
    lab = orc.accept_label(Pr, inp.U, inp.W1, inp.W2, inp.anchors, drafted["tokens"],
                           draft_temperature=0.0, target_temperature=1.0)
    pt = special.softmax(Pr[:, :K].astype(np.float64), axis=-1)
    assert np.allclose(lab, np.take_along_axis(pt, drafted["tokens"][..., None], -1)[..., 0],
                       atol=1e-12)
    # both greedy: 1 where the drafted token is the target's argmax, else 0
    lab = orc.accept_label(Pr, inp.U, inp.W1, inp.W2, inp.anchors, drafted["tokens"],
                           draft_temperature=0.0, target_temperature=0.0)
    assert np.array_equal(lab, (drafted["tokens"] == Pr[:, :K].argmax(-1)).astype(np.float64))
    assert np.all((lab >= 0) & (lab <= 1))


# ------------------------------------------------------------------ sequential temperature scaling
def _raw_confidences(rng, N, K, spread=2.0):
    z = rng.normal(0.0, spread, (N, K))
    conf = special.expit(z).astype(np.float32)
    c = np.clip(conf.astype(np.float64), 2.0 ** -24, 1 - 2.0 ** -24)
    return conf, np.log(c / (1 - c))  # the logit the fit sees


def test_sts_recovers_the_generating_temperatures(orc):
    """Labels drawn as sigmoid(z_k / tau_k): the cross-entropy of the cumulative survival is
    minimised exactly there, position after position."""
    rng = np.random.default_rng(101)
    N, K = 4000, 5
    conf, z = _raw_confidences(rng, N, K)
    tau_true = np.array([0.5, 1.7, 1.0, 3.0, 0.8])
    label = special.expit(z / tau_true).astype(np.float32)
    out = orc.sts_fit(conf, label)
    assert np.abs(np.log(out["tau"]) - np.log(tau_true)).max() < 1e-4, out["tau"]


def test_sts_leaves_calibrated_confidences_alone(orc):
    rng = np.random.default_rng(102)
    conf, _ = _raw_confidences(rng, 3000, 4)
    out = orc.sts_fit(conf, conf)
    assert np.abs(np.log(out["tau"])).max() < 1e-4, out["tau"]


def test_sts_matches_a_dense_scan(orc):
    """Each temperature is the minimiser of its position's loss over a fine scan of ln tau
    (earlier temperatures fixed at the fitted ones)."""
    rng = np.random.default_rng(103)
    N, K = 300, 3
    conf, z = _raw_confidences(rng, N, K, spread=1.5)
    label = rng.uniform(0.2, 1.0, (N, K)).astype(np.float32)
    out = orc.sts_fit(conf, label)
    xs = np.linspace(np.log(1 / 64), np.log(64), 200001)
    a = np.ones(N)
    y = np.ones(N)
    for k in range(K):
        y = y * label[:, k].astype(np.float64)
        q = np.clip(a[None, :] * special.expit(z[None, :, k] * np.exp(-xs)[:, None]), 1e-7, 1 - 1e-7)
        L = -(y * np.log(q) + (1 - y) * np.log1p(-q)).sum(axis=1)
        assert abs(np.log(out["tau"][k]) - xs[np.argmin(L)]) < 2e-4, k
        assert out["loss"][k] <= L.min() / N + 1e-12
        a = a * special.expit(z[:, k] / out["tau"][k])


def test_sts_calibrates_and_keeps_the_ranking(orc):
    """A head that is overconfident at every position: after STS the predicted survival
    matches the realised one (expected calibration error drops) and the order of
    confidences within a position is unchanged."""
    rng = np.random.default_rng(104)
    N, K = 20000, 4
    conf, z = _raw_confidences(rng, N, K, spread=3.0)
    true_p = special.expit(z / 2.5)                    # the head is too sharp by 2.5x
    acc = (rng.uniform(size=(N, K)) < true_p).astype(np.float32)  # 0/1 outcomes
    out = orc.sts_fit(conf, acc)
    assert np.all(np.abs(out["tau"] - 2.5) < 0.25), out["tau"]
    cal = special.expit(z / out["tau"])
    surv_true = np.cumprod(acc, axis=1)
    def ece(p, y, bins=10):
        idx = np.minimum((p * bins).astype(int), bins - 1)
        return sum(abs(p[idx == i].mean() - y[idx == i].mean()) * (idx == i).mean()
                   for i in range(bins) if (idx == i).any())
    before = ece(np.cumprod(conf, axis=1).ravel(), surv_true.ravel())
    after = ece(np.cumprod(cal, axis=1).ravel(), surv_true.ravel())
    assert after < 0.5 * before and after < 0.02, (before, after)
    for k in range(K):
        assert np.array_equal(np.argsort(conf[:, k], kind="stable"), np.argsort(cal[:, k], kind="stable"))


def test_confidence_applies_per_position_temperatures(orc):
    V, K, r, d = 64, 3, 16, 32
    inp = make_inputs(105, 4, K, V, r, d=d, confidence=True, weight_std=0.3)
    toks = np.random.default_rng(106).integers(0, V, (4, K)).astype(np.int32)
    tau = np.array([0.5, 2.0, 1.0])
    raw = orc.confidence(inp.h, inp.W1, inp.anchors, toks, inp.w_conf, bias=0.3)
    cal = orc.confidence(inp.h, inp.W1, inp.anchors, toks, inp.w_conf, bias=0.3, tau=tau)
    z = special.logit(raw["conf"])
    assert np.allclose(cal["conf"], special.expit(z / tau), atol=1e-12)
    assert np.allclose(cal["cumprod"], np.cumprod(cal["conf"], axis=1), atol=1e-12)
