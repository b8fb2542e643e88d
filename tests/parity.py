"""Test helpers: comparing kernel outputs with the oracle, and building
adversarial inputs by searching the oracle. Uses only the oracle, numpy and
the seeded workload generators -- never the CUDA path."""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

import oracle
from moe_swiglu_epilogue_gb300 import workloads as W

# Fused-path tolerance: scale bytes exact; a nibble may differ by one E2M1
# step, on at most 1e-5 of the elements, and only where a fp32 SwiGLU value
# within 2 ulp of the oracle's would have produced the kernel's nibble.
MAX_NIBBLE_MISMATCH_FRACTION = 1e-5
MAX_ULPS = 2


def unpack_nibbles(packed: np.ndarray) -> np.ndarray:
    """[..., n/2] bytes -> [..., n] nibbles (even element = low nibble)."""
    p = np.asarray(packed, np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = p & 0x0F
    out[..., 1::2] = p >> 4
    return out


def signed_index(nib: np.ndarray) -> np.ndarray:
    idx = (nib & 7).astype(np.int32)
    return np.where(nib & 8, -idx, idx)


@dataclass
class FusedReport:
    elements: int
    sf_mismatches: int
    nibble_mismatches: int
    outside_tolerance: int

    @property
    def exact(self) -> bool:
        return self.sf_mismatches == 0 and self.nibble_mismatches == 0

    def assert_within_tolerance(self):
        assert self.sf_mismatches == 0, self
        assert self.nibble_mismatches <= MAX_NIBBLE_MISMATCH_FRACTION * self.elements, self
        assert self.outside_tolerance == 0, self


def _ulp_neighbours(y: float, k: int):
    v = np.float32(y)
    out = []
    up, dn = v, v
    for _ in range(k):
        up = np.nextafter(up, np.float32(np.inf))
        dn = np.nextafter(dn, np.float32(-np.inf))
        out += [up, dn]
    return out


def compare_fused(gpu_packed, gpu_sf, ref_packed, ref_sf, y_oracle_at) -> FusedReport:
    """gpu_* / ref_*: packed [n, I/2] and sf [n, I/16] for the same n rows or
    blocks. y_oracle_at(row, col) gives the oracle's fp32 SwiGLU value there
    (only called for mismatching nibbles)."""
    gpu_sf = np.asarray(gpu_sf); ref_sf = np.asarray(ref_sf)
    sf_bad = int(np.count_nonzero(gpu_sf != ref_sf))
    gn = unpack_nibbles(gpu_packed); rn = unpack_nibbles(ref_packed)
    bad = np.argwhere(gn != rn)
    outside = 0
    for r, c in bad:
        g, o = int(gn[r, c]), int(rn[r, c])
        if abs(int(signed_index(np.uint8(g))) - int(signed_index(np.uint8(o)))) > 1:
            outside += 1
            continue
        y = y_oracle_at(int(r), int(c))
        code = int(ref_sf[r, c // 16])
        if not any(oracle.quantize_element_with_scale(float(v), code) == g
                   for v in _ulp_neighbours(y, MAX_ULPS)):
            outside += 1
    return FusedReport(int(gn.size), sf_bad, int(bad.shape[0]), outside)


# ---------------------------------------------------------------------------
# Adversarial blocks
# ---------------------------------------------------------------------------

def e4m3_value(code: int) -> float:
    return oracle.fp8_e4m3_to_float32(code)


def quantize_edge_blocks(rng, n_blocks: int) -> np.ndarray:
    """BF16 quantize-only blocks [n, 16] (uint16) built around exact
    boundaries: the block amax on 6 x E4M3 values and on 6 x the midpoints
    between neighbours (scale ties, including the subnormal ones and the
    underflow tie 6 * 2^-10), elements on half-step ties (2k+1)/4 * d and
    their BF16 neighbours, +-0, and saturating blocks (amax 6 * 448 and far
    beyond). Values that BF16 cannot hold exactly round to a neighbour."""
    blocks = []
    codes = list(range(1, 0x7f))
    for n in range(n_blocks):
        kind = n % 6
        c = codes[rng.integers(len(codes))]
        d = e4m3_value(c)
        y = np.zeros(16, np.float64)
        if kind in (0, 1):                      # half-step ties under scale d
            y[0] = 6 * d
            k = rng.integers(0, 12, 15)
            y[1:] = (2 * k + 1) / 4 * d
        elif kind == 2:                         # scale tie: amax = 6 * midpoint
            c2 = min(c + 1, 0x7e)
            y[0] = 3 * (d + e4m3_value(c2))
            y[1:] = rng.uniform(-1, 1, 15) * y[0]
        elif kind == 3:                         # subnormal scales and their ties
            m = rng.integers(1, 9)
            y[0] = 6 * (m + (0.5 if rng.integers(2) else 0.0)) * 2.0 ** -9
            y[1:] = rng.uniform(-1, 1, 15) * y[0]
        elif kind == 4:                         # saturation
            y[0] = [6 * 448.0, 6 * 464.0, 6 * 480.0, 1e5, 3e38][rng.integers(5)]
            y[1:] = rng.uniform(-1, 1, 15) * y[0]
        else:                                   # signed zeros and tiny values
            y[:] = rng.choice([0.0, -0.0, 1e-40, -1e-40, 6 * 2.0 ** -10, -6 * 2.0 ** -11], 16)
        y *= np.where(rng.integers(0, 2, 16) == 1, -1.0, 1.0)
        perm = rng.permutation(16)
        bits = W.bf16_bits(y.astype(np.float32))
        # keep exact ties exact: when the fp32 -> bf16 rounding moved a value,
        # also try the truncated neighbour at random
        trunc = (y.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        pick = rng.integers(0, 2, 16) == 1
        bits = np.where(pick, trunc, bits)
        blocks.append(bits[perm])
    return np.stack(blocks)


def _gate_table(L: float, gate_lo: float):
    """Every BF16 gate in [gate_lo, L + 1] whose oracle silu is >= 2^-6 in
    magnitude, with that silu value (float64)."""
    allg = np.arange(0x10000, dtype=np.uint32).astype(np.uint16)
    gf = W.bf16_to_f32(allg)
    sel = np.isfinite(gf) & (gf >= gate_lo) & (gf <= L + 1.0)
    gf = gf[sel]
    sig = oracle.swiglu_clamped_array(gf, np.ones_like(gf), L).astype(np.float64)
    keep = np.abs(sig) >= 2.0 ** -6
    return gf[keep], sig[keep]


def nearest_pairs(targets, L: float, gate_lo: float = -6.0):
    """For every target value, the BF16 (gate, up) pair whose oracle SwiGLU
    lies nearest to it: every BF16 gate in [gate_lo, L + 1] is paired with
    the two BF16 ups around target / silu(gate). Returns (gates, ups,
    distances), float32 / float32 / float64 arrays shaped like targets."""
    gf, sig = _gate_table(L, gate_lo)
    flat = np.asarray(targets, np.float64).ravel()
    best_g = np.zeros(flat.size, np.float32)
    best_u = np.zeros(flat.size, np.float32)
    best_all = np.full(flat.size, np.inf)
    for c0 in range(0, flat.size, 256):
        t = flat[c0:c0 + 256]
        ustar = t[:, None] / sig[None, :]
        ok = np.abs(ustar) <= L
        ub = (np.where(ok, ustar, 0.0).astype(np.float32).view(np.uint32) >> 16)
        G = np.broadcast_to(gf[None, :], ustar.shape)
        best_d = np.full(t.size, np.inf)
        for delta in (0, 1):
            U = W.bf16_to_f32((ub + delta).astype(np.uint16))
            y = oracle.swiglu_clamped_array(G, U, L).reshape(ustar.shape).astype(np.float64)
            dist = np.where(ok, np.abs(y - t[:, None]), np.inf)
            j = np.argmin(dist, axis=1)
            dj = dist[np.arange(t.size), j]
            better = dj < best_d
            best_d = np.where(better, dj, best_d)
            rows = np.nonzero(better)[0]
            best_g[c0 + rows] = gf[j[rows]]
            best_u[c0 + rows] = U[rows, j[rows]]
        best_all[c0:c0 + t.size] = best_d
    shape = np.shape(targets)
    return best_g.reshape(shape), best_u.reshape(shape), best_all.reshape(shape)


def _blocks_from_pairs(rng, g, u):
    """[n, 16] gate / up values -> interleaved BF16 blocks [n, 32], the 16
    outputs of each block in a random order."""
    n = g.shape[0]
    out = np.zeros((n, 32), np.uint16)
    for k in range(n):
        perm = rng.permutation(16)
        out[k] = W.interleave_gate_up(W.bf16_bits(g[k][perm])[None, :], W.bf16_bits(u[k][perm])[None, :])[0]
    return out


def fused_near_tie_blocks(rng, n_blocks: int, L: float, gate_lo: float = -6.0):
    """Interleaved BF16 blocks [n, 32] whose oracle SwiGLU values land as
    close as BF16 (gate, up) pairs allow to rounding boundaries: the block
    amax on 6 x an E4M3 value, or on 6 x the midpoint between two (a scale
    tie, subnormal scales included), the other 15 outputs on half-step ties
    (2k+1)/4 * d. Exact hits are rare (exact_tie_pairs: an exhaustive count);
    most values end a few ulps from their boundary, inside the fused
    kernel's decision window.
    Returns (blocks, {"exact_hits", "median_rel_distance", "targets"})."""
    targets = np.zeros((n_blocks, 16))
    for n in range(n_blocks):
        code = int(rng.integers(1, 0x48))         # scales up to 3.75: |y| <= L silu(L)
        d = e4m3_value(code)
        amax = 3 * (d + e4m3_value(code + 1)) if n % 3 == 0 else 6 * d
        targets[n, 0] = amax
        targets[n, 1:] = (2 * rng.integers(0, 12, 15) + 1) / 4 * d
    targets *= np.where(rng.integers(0, 2, targets.shape) == 1, -1.0, 1.0)
    g, u, dist = nearest_pairs(targets, L, gate_lo)
    out = _blocks_from_pairs(rng, g, u)
    return out, {"exact_hits": int(np.count_nonzero(dist == 0)),
                 "median_rel_distance": float(np.median(dist / np.abs(targets))),
                 "targets": int(targets.size)}


def exact_tie_pairs(L: float, min_abs: float = 2.0 ** -12):
    """Every BF16 pair (gate in [-16, L + 1] with |gate| >= 2^-14, up in
    [2^-16, L]) whose oracle SwiGLU y (|y| >= min_abs) sits exactly on a
    half-step tie (2k+1)/4 * d of an E4M3 scale d (k = 0..11), found by
    evaluating all of them. Returns a list of (gate, up, y, code, k); ups of
    the other sign give -y (the clamp is symmetric)."""
    allb = np.arange(0x10000, dtype=np.uint32).astype(np.uint16)
    f = W.bf16_to_f32(allb)
    g = f[np.isfinite(f) & (f >= -16) & (f <= L + 1) & (np.abs(f) >= 2.0 ** -14)]
    u = f[np.isfinite(f) & (f > 0) & (f <= L) & (f >= 2.0 ** -16)]
    G = np.repeat(g, u.size)
    U = np.tile(u, g.size)
    y = oracle.swiglu_clamped_array(G, U, L)
    # a tie value has at most 9 significant bits: (2k+1) <= 23 times a 4-bit d
    short = ((y.view(np.uint32) & 0x7FFF) == 0) & (np.abs(y) >= min_abs)
    d = {c: e4m3_value(c) for c in range(1, 0x7f)}
    found = []
    for gi, ui, yi in zip(G[short], U[short], y[short]):
        for k in range(12):
            want = abs(float(yi)) * 4 / (2 * k + 1)
            for c, dc in d.items():
                if dc == want:
                    found.append((float(gi), float(ui), float(yi), c, k))
    return found


def fused_exact_tie_blocks(rng, n_blocks: int, L: float, pairs, gate_lo: float = -6.0):
    """Blocks around the exact tie pairs (exact_tie_pairs): the amax on
    6 x the pair's scale d (nearest pair), and the other 15 outputs the pair
    itself with random signs, each exactly on its half-step tie under d."""
    if not pairs:
        return np.zeros((0, 32), np.uint16)
    g = np.zeros((n_blocks, 16), np.float32)
    u = np.zeros((n_blocks, 16), np.float32)
    amax_t = np.zeros(n_blocks)
    for n in range(n_blocks):
        pg, pu, _, code, _ = pairs[n % len(pairs)]
        amax_t[n] = 6 * e4m3_value(code)
        g[n, 1:] = pg
        u[n, 1:] = np.where(rng.integers(0, 2, 15) == 1, -pu, pu)
    ag, au, _ = nearest_pairs(amax_t, L, gate_lo)
    g[:, 0], u[:, 0] = ag, au
    return _blocks_from_pairs(rng, g, u)


def near_bf16_midpoint_blocks(rng, n_blocks: int, L: float, max_ulps: int = 8,
                              candidates: int = 1 << 22, gate_range=None):
    """Interleaved BF16 blocks [n, 32] whose oracle fp32 SwiGLU values lie
    within `max_ulps` fp32 ulps of a BF16 rounding midpoint (low 16 bits
    0x8000), where a fast evaluation may round to the other BF16
    neighbour. Drawn by searching random (gate, up) pairs with the oracle;
    gates ~ N(0, 3^2) (or uniform in gate_range), ups ~ N(0, 1). Returns
    (blocks, the distances in ulps)."""
    picked_g, picked_u, dist = [], [], []
    need = 16 * n_blocks
    while len(picked_g) < need:
        if gate_range is None:
            g = W.bf16_to_f32(W.bf16_bits(rng.standard_normal(candidates, dtype=np.float32) * 3))
        else:
            g = W.bf16_to_f32(W.bf16_bits(rng.uniform(*gate_range, candidates).astype(np.float32)))
        u = W.bf16_to_f32(W.bf16_bits(rng.standard_normal(candidates, dtype=np.float32)))
        y = oracle.swiglu_clamped_array(g, u, L).astype(np.float32)
        d = np.abs((y.view(np.uint32) & 0xFFFF).astype(np.int64) - 0x8000)
        sel = np.nonzero((d <= max_ulps) & (np.abs(y) >= 2.0 ** -100))[0]
        picked_g += list(g[sel]); picked_u += list(u[sel]); dist += list(d[sel])
    g = np.array(picked_g[:need], np.float32).reshape(n_blocks, 16)
    u = np.array(picked_u[:need], np.float32).reshape(n_blocks, 16)
    blocks = W.interleave_gate_up(W.bf16_bits(g), W.bf16_bits(u))
    return blocks, np.array(dist[:need])


# ---------------------------------------------------------------------------
# The L1 GEMM with the step in its epilogue
# ---------------------------------------------------------------------------

# The epilogue evaluates SwiGLU in fast fp32 on fp32 accumulators; its value
# is within this relative distance of the oracle's (the fast path's bound on
# BF16 gates is 1.72e-6; fp32 gates get the same argument rounding, plus
# margin).
GEMM_Y_REL_TOL = 4e-6
GEMM_MAX_MISMATCH_FRACTION = 1e-4


def compare_gemm_fused(gpu_packed, gpu_sf, y_ref, rel=GEMM_Y_REL_TOL):
    """Kernel outputs vs the oracle's fp32 SwiGLU values y_ref [n, I] of the
    same accumulators. A scale code may differ only where amax * (1 +- rel)
    / 6 round to different codes; a nibble only where y * (1 +- rel) under
    the kernel's scale quantizes to the kernel's nibble. Returns (sf
    mismatches, nibble mismatches, elements); raises on any outside that."""
    y_ref = np.ascontiguousarray(y_ref, np.float32)
    n, I = y_ref.shape
    ref_p, ref_s = oracle.quantize_nvfp4_f32(y_ref)
    gpu_sf = np.asarray(gpu_sf)
    amax = np.abs(y_ref.astype(np.float64)).reshape(n, I // 16, 16).max(-1)
    lo = oracle.fp8_e4m3_from_float32_array((amax * (1 - rel) / 6).astype(np.float32)).reshape(n, -1)
    hi = oracle.fp8_e4m3_from_float32_array((amax * (1 + rel) / 6).astype(np.float32)).reshape(n, -1)
    sf_bad = np.argwhere(gpu_sf != ref_s)
    for r, b in sf_bad:
        assert lo[r, b] != hi[r, b] and gpu_sf[r, b] in (lo[r, b], hi[r, b]), \
            ("scale outside tolerance", r, b, gpu_sf[r, b], ref_s[r, b], amax[r, b])
    gn = unpack_nibbles(gpu_packed)
    rn = unpack_nibbles(ref_p)
    bad = np.argwhere(gn != rn)
    for r, c in bad:
        code = int(gpu_sf[r, c // 16])
        y = float(y_ref[r, c])
        allowed = {oracle.quantize_element_with_scale(v, code)
                   for v in (y, np.float32(y * (1 - rel)), np.float32(y * (1 + rel)))}
        assert int(gn[r, c]) in allowed, ("nibble outside tolerance", r, c, y, code, gn[r, c], rn[r, c])
    nib_mismatch_in_matching_blocks = sum(1 for r, c in bad if gpu_sf[r, c // 16] == ref_s[r, c // 16])
    assert nib_mismatch_in_matching_blocks <= GEMM_MAX_MISMATCH_FRACTION * gn.size, \
        (nib_mismatch_in_matching_blocks, gn.size)
    return len(sf_bad), len(bad), gn.size
