"""Helpers shared by the GPU parity tests (upload, compare with tolerances)."""

import numpy as np
import torch

LOGPROB_TOL = 2e-3     # teacher-forced logits / log-probabilities, absolute
MARGIN = 1e-3          # tokens must match wherever the oracle's top-2 margin exceeds this
COVERAGE = 0.95        # share of the replayed (request, position) pairs that must be compared


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bf(a):
    """Upload bf16 bit patterns (uint16) as an int16 device tensor."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def host(t):
    return t.detach().cpu().numpy()


def check_sequences(gpu_tokens, gpu_logprobs, ref, margin=MARGIN, tol=LOGPROB_TOL, what="draft"):
    """Compare a GPU draft with the oracle's own run on the same inputs and noise
    (no GPU output enters the oracle).  Per request, positions are compared in
    order: the tokens must agree up to the first position where the oracle's
    decision was a near tie (its decision margin <= margin), and a request that
    disagrees there is not compared further, since every later position depends on
    the token taken.  Log-probabilities must agree within tol wherever the tokens
    do.  Returns (requests that diverged at a near tie, positions compared)."""
    gt, rt = np.asarray(gpu_tokens), ref["tokens"]
    B, K = gt.shape
    diverged = compared = 0
    for b in range(B):
        n = first_difference(gt[b], rt[b])
        if n < K:
            assert ref["margins"][b, n] <= margin, (
                f"{what}: request {b} position {n}: gpu {gt[b, n]} vs oracle {rt[b, n]}, "
                f"oracle margin {ref['margins'][b, n]:.3e} > {margin}")
            diverged += 1
        if n > 0:
            err = np.abs(gpu_logprobs[b, :n] - ref["logprobs"][b, :n]).max()
            assert err <= tol, f"{what}: request {b}: max |logprob - oracle| = {err:.3e}"
        compared += n
    assert np.all(gpu_logprobs <= 1e-6)
    return diverged, compared


def assert_coverage(what, diverged, compared, total, min_share=COVERAGE):
    """Print how many replayed positions were compared and how many requests stopped at a
    near tie, and fail when fewer than min_share of the replayed positions were compared
    (a run in which most positions went uncompared would otherwise pass)."""
    share = compared / total if total else 1.0
    print(f"{what}: compared {compared} of {total} positions ({share:.4f}); "
          f"{diverged} requests diverged at a near tie")
    assert share >= min_share, (
        f"{what}: only {compared} of {total} positions compared ({share:.3f} < {min_share})")


def first_difference(a, b):
    """Index of the first position where two token rows differ (len when equal)."""
    d = np.flatnonzero(np.asarray(a) != np.asarray(b))
    return int(d[0]) if d.size else len(a)
