"""Helpers shared by the GPU parity tests (upload, compare with tolerances)."""

import numpy as np
import torch

LOGPROB_TOL = 2e-3     # teacher-forced logits / log-probabilities, absolute
MARGIN = 1e-3          # tokens must match wherever the oracle's top-2 margin exceeds this


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bf(a):
    """Upload bf16 bit patterns (uint16) as an int16 device tensor."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def host(t):
    return t.detach().cpu().numpy()


def check_tokens(gpu_tokens, gpu_logprobs, ref, margin=MARGIN, tol=LOGPROB_TOL, what="draft"):
    """ref: oracle run forced on the GPU's tokens.  Returns (near-tie mismatches, near ties)."""
    mism = gpu_tokens != ref["tokens"]
    near = ref["margins"] <= margin
    hard = mism & ~near
    assert not hard.any(), (
        f"{what}: {int(hard.sum())} tokens differ from the oracle with margin > {margin}: "
        f"first at {np.argwhere(hard)[:5].tolist()}, gpu {gpu_tokens[hard][:5]}, "
        f"oracle {ref['tokens'][hard][:5]}, margins {ref['margins'][hard][:5]}")
    err = np.abs(gpu_logprobs - ref["forced_logprobs"])
    assert err.max() <= tol, f"{what}: max |logprob - oracle| = {err.max():.3e}"
    assert np.all(gpu_logprobs <= 1e-6)
    return int(mism.sum()), int(near.sum())
