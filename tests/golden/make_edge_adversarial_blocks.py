"""Writes edge_adversarial_blocks.npz: the adversarial 16-output blocks of
the edge-case workload (16384 rows, I = 4096, 10% adversarial blocks), found
with the oracle only.

    python tests/golden/make_edge_adversarial_blocks.py

The blocks aim at the rounding boundaries of the NVFP4 step as the pages fix
them ("2026-05-28 Status", the E4M3 cast with round-to-nearest-even and
carry; "NVFP4-1.1 Approach, Part 2", the round-half-even half steps):

  fused     [N, 32] BF16 bits, [gate x8, up x8] x 2: (gate, up) pairs whose
            oracle SwiGLU (L = 7) lands as close as BF16 pairs allow to a
            target: the block amax on 6 x an E4M3 value or on 6 x the
            midpoint of two neighbouring codes (FP8 RNE ties, subnormal
            scales m * 2^-9 included), the other 15 outputs on the half-step
            ties (2k+1)/4 * d of the block's scale d. Each target is hit by
            its nearest BF16 pair, a few fp32 ulps away, inside the kernel's
            decision window. Exact hits are all but absent: evaluating every
            BF16 pair (10.7 M with |y| >= 2^-12) finds the SwiGLU value on a
            half-step tie for a single pair; the last N_EXACT blocks carry
            it (15 outputs exactly on that tie under their scale, the amax
            on 6 x the scale). `fused_exact_pairs` lists the pairs found.
  quantize  [M, 16] BF16 bits for quantize-only: amax on 6 x E4M3 values and
            midpoints, elements on half-step ties and their BF16 neighbours,
            subnormal scales, the underflow tie, saturation (amax = 448 x 6
            and beyond) and signed zeros. These reach the scale's saturation,
            which the clamp keeps out of the fused path.

Deterministic: a fixed seed, and only the oracle (plus the seeded input
helpers) is called. The workload generator places these blocks at seeded
positions; it never evaluates them.
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))                   # tests/ (parity)
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))  # repo root (oracle, workloads)

import oracle  # noqa: E402
import parity  # noqa: E402

OUT = os.path.join(HERE, "edge_adversarial_blocks.npz")
SEED = 20260528
N_FUSED = 4096
N_EXACT = 256
N_QUANT = 8192
L = 7.0


def build_table():
    """(fused blocks, quantize blocks, near-tie search stats, exact pairs)."""
    oracle.build()
    rng = np.random.default_rng(SEED)
    near, stats = parity.fused_near_tie_blocks(rng, N_FUSED, L, gate_lo=-16.0)
    pairs = parity.exact_tie_pairs(L)
    exact = parity.fused_exact_tie_blocks(rng, N_EXACT if pairs else 0, L, pairs, gate_lo=-16.0)
    fused = np.concatenate([near, exact])
    quant = parity.quantize_edge_blocks(rng, N_QUANT)
    return fused, quant, stats, pairs, exact


def main():
    fused, quant, stats, pairs, exact = build_table()
    near = fused[:fused.shape[0] - exact.shape[0]]
    y = oracle.swiglu_values(fused, L)
    np.savez_compressed(OUT, fused=fused.astype(np.uint16), quantize=quant.astype(np.uint16),
                        fused_clamp_L=np.float32(L), seed=np.int64(SEED),
                        fused_exact_blocks=np.int64(exact.shape[0]),
                        fused_exact_pairs=np.asarray([p[:3] + (p[3], p[4]) for p in pairs], np.float64).reshape(-1, 5),
                        fused_near_targets=np.int64(stats["targets"]),
                        fused_near_median_rel_distance=np.float64(stats["median_rel_distance"]))
    print(f"wrote {OUT}: {near.shape[0]} near-tie fused blocks ({stats}), {exact.shape[0]} exact-tie "
          f"blocks from {len(pairs)} exact pair(s) {pairs}, {N_QUANT} quantize blocks; "
          f"|y| range {np.abs(y).min():.3g} .. {np.abs(y).max():.3g}")


if __name__ == "__main__":
    main()
