"""GPU parity of the load-aware prefix scheduler (dspark_schedule) with the oracle,
and the draft -> schedule -> verify chain on one stream."""

import numpy as np
import pytest
import torch

import oracle
from rank_markov_draft_gb300 import binding
from synth import make_inputs
from tests.gpu_util import bf, dev, host

pytestmark = pytest.mark.gpu


def _tables(rng, R, K, kind):
    lo = 0.9 if kind == "cliff" else 0.4
    a = np.cumprod(rng.uniform(lo, 0.995, (R, K)), axis=1).astype(np.float32)
    Bmax = R * (K + 1)
    B = np.arange(Bmax + 1, dtype=np.float64)
    if kind == "cliff":
        # flat up to two thirds of the candidates, then half the rate: every admission
        # before the cliff raises Theta by a relative a / (R + sum a) >= 0.9^K / (R (K + 1)),
        # and the one at the cliff would halve it, so every test clears the 1e-5 margin
        sps = np.where(B <= R + (2 * R * K) // 3, 1000.0, 500.0)
    elif kind == "smooth":
        sps = 2000.0 / (1.0 + (B / (0.6 * Bmax)) ** 2)
    elif kind == "flat":
        sps = np.full(Bmax + 1, 50.0)
    else:  # jagged: a saturating curve with steps (CUDA-graph batch buckets)
        sps = 2000.0 / (1.0 + (B / (0.7 * Bmax)) ** 1.5) * (1.0 - 0.08 * ((B // 37) % 3))
    return a, sps.astype(np.float32)


# candidate counts padded to 32, 2048, 4096, 8192 and 16384: one, two, four, eight and sixteen
# keys a thread; K = 0 admits nothing
@pytest.mark.parametrize("R,K", [(1, 1), (7, 3), (128, 16), (200, 16), (500, 16), (300, 40),
                                 (5, 0)])
@pytest.mark.parametrize("kind", ["smooth", "flat", "jagged", "cliff"])
def test_schedule_matches_oracle(dsp, R, K, kind):
    rng = np.random.default_rng(R * 1000 + K)
    a, sps = _tables(rng, R, K, kind)
    out = binding.schedule(dsp, dev(a), dev(sps))
    torch.cuda.synchronize()
    assert dsp.status() == 0
    ref = oracle.schedule(a.astype(np.float64), sps.astype(np.float64))
    ell = host(out["ell"])
    exact = ref["margin"] > 1e-5
    print(f"schedule R={R} K={K} {kind}: margin {ref['margin']:.2e}, "
          f"{'exact' if exact else 'bounds-only'} comparison")
    if kind == "cliff" and R * K >= 2048:
        assert exact, "the cliff tables are built so that the exact comparison runs"
    if exact:
        assert np.array_equal(ell, ref["ell"])
        assert np.isclose(host(out["theta"])[0], ref["theta"], rtol=1e-5)
    # prefixes are whole and within bounds in any case
    assert np.all((ell >= 0) & (ell <= K))


def test_schedule_bench_workload(dsp):
    """The scheduler line the bench times: R = 128 requests x K = 16, its own seeded inputs."""
    import bench
    from synth import schedule_inputs
    c = bench.SMALL["schedule"]
    a, sps = schedule_inputs(c["seed"], c["R"], c["K"])
    out = binding.schedule(dsp, dev(a), dev(sps))
    torch.cuda.synchronize()
    assert dsp.status() == 0
    ref = oracle.schedule(a.astype(np.float64), sps.astype(np.float64))
    ell = host(out["ell"])
    if ref["margin"] > 1e-5:
        assert np.array_equal(ell, ref["ell"])
    else:  # a near-tie at the cut (this input has one): one admission either way
        assert abs(int(ell.sum()) - int(ref["ell"].sum())) <= 1
        assert np.all(np.abs(ell - ref["ell"]) <= 1)
    assert np.isclose(host(out["theta"])[0], ref["theta"], rtol=1e-5)


@pytest.mark.parametrize("R,K", [(64, 16), (200, 16)])
def test_schedule_equal_survivals(dsp, R, K):
    """Survivals on a grid of 1/20: many candidates share a value, so the order among equals
    (position ascending, then request ascending) decides who is admitted at the cut."""
    rng = np.random.default_rng(R + 7)
    a = np.cumprod(rng.choice([0.5, 0.75, 0.9, 1.0], (R, K)), axis=1)
    a = (np.round(a * 20.0) / 20.0).astype(np.float32)
    a = np.minimum.accumulate(a, axis=1)  # still non-increasing along each request
    Bmax = R * (K + 1)
    sps = (2000.0 / (1.0 + (np.arange(Bmax + 1) / (0.4 * Bmax)) ** 2)).astype(np.float32)
    out = binding.schedule(dsp, dev(a), dev(sps))
    torch.cuda.synchronize()
    assert dsp.status() == 0
    ref = oracle.schedule(a.astype(np.float64), sps.astype(np.float64))
    ell = host(out["ell"])
    if ref["margin"] > 1e-5:
        assert np.array_equal(ell, ref["ell"])
    else:  # the same number admitted, all prefixes whole
        assert ell.sum() == ref["ell"].sum()
    assert np.all((ell >= 0) & (ell <= K))


def test_draft_schedule_verify_chain(dsp):
    """The confidence head's survival feeds the scheduler, whose lengths feed the
    verifier: every step on the GPU, in stream order."""
    B, K, V, r, d = 32, 8, 4096, 64, 128
    inp = make_inputs(81, B, K, V, r, d=d, confidence=True, weight_std=0.1)
    conf = binding.Confidence(h=bf(inp.h), w=bf(inp.w_conf), bias=1.5, threshold=0.3)
    dr = binding.markov_draft(dsp, dev(inp.U), bf(inp.W1), bf(inp.W2), dev(inp.anchors),
                              temperature=1.0, seed=3, conf=conf)
    Bmax = B * (K + 1)
    sps = dev((3000.0 / (1.0 + (np.arange(Bmax + 1) / 150.0) ** 2)).astype(np.float32))
    sc = binding.schedule(dsp, dr["cumprod"], sps)
    rng = np.random.default_rng(82)
    P = np.concatenate([inp.U + rng.standard_normal(inp.U.shape).astype(np.float32),
                        rng.standard_normal((B, 1, V)).astype(np.float32)], axis=1)
    out = binding.verify(dsp, dev(P), dev(inp.U), bf(inp.W1), bf(inp.W2), dev(inp.anchors),
                         dr["tokens"], dr["logprobs"], draft_temperature=1.0,
                         target_temperature=1.0, seed=4, ell=sc["ell"])
    torch.cuda.synchronize()
    assert dsp.status() == 0
    ell, n = host(sc["ell"]), host(out["n_acc"])
    # the oracle's own chain: its draft, its confidence, its schedule
    od = oracle.markov_draft(inp.U, inp.W1, inp.W2, inp.anchors, temperature=1.0, seed=3)
    oc = oracle.confidence(inp.h, inp.W1, inp.anchors, od["tokens"], inp.w_conf, bias=1.5,
                           threshold=0.3)
    ref = oracle.schedule(oc["cumprod"], host(sps).astype(np.float64))
    if np.array_equal(host(dr["tokens"]), od["tokens"]) and ref["margin"] > 1e-5:
        assert np.array_equal(ell, ref["ell"])
    assert np.all(n <= ell)
    assert np.all(host(out["accept_prob"])[np.arange(K)[None, :] >= ell[:, None]] == -1.0)
