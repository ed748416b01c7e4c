"""Phase trace of one draft-kernel launch (dspark_debug_trace), printed per position.

    python -m rank_markov_draft_gb300.trace [--mode sample|greedy|label] [--B 128] [--gated]

Runs the serving-size workload (K = 16, V = 151936, r = 256) on cuda:0 with
synthetic inputs: U ~ 3 N(0, 1) with eight boosted tokens per row, weights
N(0, 0.02) in bf16; for the label mode, target logits = U + N(0, 1).  --gated
adds the gate H = sigmoid(h . Wg), h ~ N(0, 1) [B, K, 4096] and Wg ~ N(0, 0.02)
[4096, 256] (the trace covers the draft kernel, after the gate's kernels).  After
three untraced calls it arms the trace for one call and prints, per position,
the median and the largest across CTAs of each phase, then each CTA's spread.

Timestamp slots written by the kernel for CTA c at position k:
  0 position start (before the embedding gather)
  1 operand in TMEM, MMAs released
  2 first tile of the position taken by the epilogue
  3 last tile done
  7 merge records written (the CTA's arrival at the grid barrier)
  4 speculative gather for the next position issued
  5 grid barrier passed (teacher-forced modes: last position only)
  6 end of the launch (last position only)
"""

from __future__ import annotations

import argparse

import numpy as np
import torch

from rank_markov_draft_gb300 import binding

K, V, R = 16, 151936, 256
SLOTS = 8
PHASES = [(0, 1, "gather+copy"), (1, 2, "to first tile"), (2, 3, "tiles"), (3, 7, "merge"),
          (7, 4, "spec gather"), (4, 5, "barrier")]


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--mode", choices=["sample", "greedy", "label"], default="sample")
    ap.add_argument("--B", type=int, default=128)
    ap.add_argument("--gated", action="store_true")
    args = ap.parse_args()
    B = args.B
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev).manual_seed(0)
    U = torch.randn(B, K, V, device=dev, generator=g) * 3
    idx = torch.randint(0, V, (B * K, 8), device=dev, generator=g)
    U.view(B * K, V).scatter_add_(1, idx, 8 + 4 * torch.rand(B * K, 8, device=dev, generator=g))
    W1 = (torch.randn(V, R, device=dev, generator=g) * 0.02).to(torch.bfloat16)
    W2 = (torch.randn(R, V, device=dev, generator=g) * 0.02).to(torch.bfloat16)
    anc = torch.randint(0, V, (B,), device=dev, dtype=torch.int32, generator=g)
    T = 0.0 if args.mode == "greedy" else 1.0
    grid = min(torch.cuda.get_device_properties(dev).multi_processor_count, (V + 127) // 128)
    buf = torch.zeros(grid * K * SLOTS, dtype=torch.int64, device=dev)
    with binding.Context(0, B_max=B, V_max=V, K_max=K) as ctx:
        if args.mode == "label":
            P = torch.cat([U + torch.randn(B, K, V, device=dev, generator=g),
                           torch.randn(B, 1, V, device=dev, generator=g)], dim=1).contiguous()
            dr = binding.markov_draft(ctx, U, W1, W2, anc, temperature=1.0, seed=1)
            call = lambda: binding.accept_label(ctx, P, U, W1, W2, anc, dr["tokens"],
                                                dr["logprobs"], draft_temperature=1.0,
                                                target_temperature=1.0)
        elif args.gated:
            h = torch.randn(B, K, 4096, device=dev, generator=g).to(torch.bfloat16)
            Wg = (torch.randn(4096, R, device=dev, generator=g) * 0.02).to(torch.bfloat16)
            call = lambda: binding.markov_draft(ctx, U, W1, W2, anc, temperature=T, seed=7,
                                                h=h, Wg=Wg)
        else:
            call = lambda: binding.markov_draft(ctx, U, W1, W2, anc, temperature=T, seed=7)
        for _ in range(3):
            call()
        torch.cuda.synchronize(dev)
        ctx.trace_next(buf)
        call()
        torch.cuda.synchronize(dev)
        status = ctx.status()
    tr = buf.cpu().numpy().reshape(grid, K, SLOTS).astype(np.float64)
    t0 = tr[:, 0, 0][tr[:, 0, 0] > 0].min()
    tr = np.where(tr > 0, (tr - t0) / 1000.0, np.nan)  # microseconds from the first stamp
    print(f"mode {args.mode}{' gated' if args.gated else ''}, B = {B}, {grid} CTAs, "
          f"device status {status}")
    print(f"launch span {np.nanmax(tr):.1f} us (median / largest across CTAs per phase, us)")
    for k in range(K):
        row = tr[:, k, :]
        parts = []
        for a, b, name in PHASES:
            d = row[:, b] - row[:, a]
            if not np.all(np.isnan(d)):
                parts.append(f"{name} {np.nanmedian(d):6.2f}/{np.nanmax(d):6.2f}")
        print(f" k={k:2d} start {np.nanmedian(row[:, 0]):7.1f}  " + "  ".join(parts))
    dur = tr[:, 1:, 0] - tr[:, :-1, 0]
    per_cta = np.nanmean(dur, axis=1)
    half = (K - 1) // 2
    corr = np.corrcoef(np.nanmean(dur[:, :half], 1), np.nanmean(dur[:, half:], 1))[0, 1]
    end = tr[:, K - 1, 4]
    print(f"per-position time per CTA: median {np.nanmedian(dur):.2f}, CTA means "
          f"{np.nanmin(per_cta):.2f} .. {np.nanmax(per_cta):.2f} us; correlation of a CTA's "
          f"first and second half {corr:.3f}")
    print(f"last position done: fastest CTA {np.nanmin(end):.1f}, median {np.nanmedian(end):.1f}, "
          f"slowest {np.nanmax(end):.1f} us")


if __name__ == "__main__":
    main()
