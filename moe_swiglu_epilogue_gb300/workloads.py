"""Seeded synthetic inputs for the five workloads.

This module only draws random numbers and lays them out: BF16 rounding of the
draws, the [gate x8, up x8, ...] interleaved column layout, and top-8 expert
routing turned into per-expert row offsets. It holds none of the SwiGLU or
NVFP4 arithmetic, so the CUDA path and the oracle can both consume its output
without sharing any of the computation under test.

Workloads (rows x width, distribution, clamp L):
  quantize   x [128, 2048] ~ N(0, 1), seed 0                 (quantize-only)
  fused      gu [512, 2*2048], gate ~ N(0, 2^2), up ~ N(0, 1), L = 7
  ragged     4096 tokens x top-8 of 256 experts -> 32768 rows in per-expert
             segments, gu [32768, 2*2048] ~ N(0, 1.5^2), L = 7
  prefill    gu [65536, 2*3072] ~ 0.5 * Student-t(3), 0.1% of values x100,
             5% of output 16-blocks zeroed (all 32 inputs), L = 10
  edge       gu [16384, 2*4096], 90% of output blocks ~ N(0, 1), 10% of
             blocks adversarial (signed zeros, saturated gates with tiny ups
             reaching subnormal scales, clamp-boundary values, huge
             magnitudes, and blocks whose SwiGLU values sit on, or within a
             few ulps of, FP8 scale ties and E2M1 half-step ties), L = 7
  edge_quantize
             x [16384, 4096] ~ N(0, 1) with 10% of the 16-blocks adversarial
             (ties, subnormal scales, saturation at amax = 448 * 6, zeros):
             the edge cases the clamp keeps out of the fused path
The tie blocks come from a table (tests/golden/edge_adversarial_blocks.npz)
written by a committed script with the oracle; this module only places its
rows at seeded positions.
Every generator takes a row count (and width) so tests can draw the same
distributions at sizes the oracle finishes in seconds.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
from dataclasses import dataclass, field

import numpy as np

ROW_CHUNK = 2048          # rows per independently seeded chunk


def bf16_bits(x) -> np.ndarray:
    """fp32 values -> BF16 bit patterns (uint16), round to nearest even."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    b = b + (np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1)))
    return (b >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def interleave_gate_up(gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    """gate, up [rows, I] -> [rows, 2I] laid out as column groups
    [gate x8, up x8, gate x8, up x8, ...]."""
    rows, width = gate.shape
    assert up.shape == gate.shape and width % 8 == 0
    return np.stack([gate.reshape(rows, width // 8, 8), up.reshape(rows, width // 8, 8)],
                    axis=2).reshape(rows, 2 * width)


def gate_column_mask(width: int) -> np.ndarray:
    """True for the gate columns of an interleaved row of 2*width values."""
    return ((np.arange(2 * width) // 8) % 2) == 0


def routing_offsets(tokens: int, experts: int, topk: int, seed: int) -> np.ndarray:
    """Each token picks `topk` distinct experts uniformly at random; rows are
    grouped by expert. Returns int32 offsets [experts + 1], offsets[-1] =
    tokens * topk."""
    rng = np.random.default_rng([seed, 0xE0])
    keys = rng.random((tokens, experts))
    picks = np.argsort(keys, axis=1)[:, :topk]
    counts = np.bincount(picks.ravel(), minlength=experts)
    off = np.zeros(experts + 1, np.int64)
    np.cumsum(counts, out=off[1:])
    return off.astype(np.int32)


def _chunked(rows: int, width: int, seed: int, tag: int, fill) -> np.ndarray:
    """Build a [rows, width] uint16 array chunk by chunk; chunk c draws from
    its own generator seeded by (seed, tag, c), so the result does not depend
    on how many threads run."""
    out = np.empty((rows, width), np.uint16)
    starts = list(range(0, rows, ROW_CHUNK))

    def work(c_start):
        c = c_start // ROW_CHUNK
        rng = np.random.default_rng([seed, tag, c])
        n = min(ROW_CHUNK, rows - c_start)
        out[c_start:c_start + n] = fill(rng, n, c_start)

    threads = min(len(starts), os.cpu_count() or 1, 32)
    if threads <= 1:
        for s in starts:
            work(s)
    else:
        with cf.ThreadPoolExecutor(threads) as ex:
            list(ex.map(work, starts))
    return out


@dataclass
class Workload:
    name: str
    kind: str                       # "quantize" or "fused"
    rows: int
    width: int                      # K (quantize) or I (fused)
    data: np.ndarray                # uint16 BF16 bits: x [rows, K] or gu [rows, 2I]
    clamp_L: float = 0.0
    offsets: np.ndarray | None = None          # int32 [E+1] or None
    meta: dict = field(default_factory=dict)

    @property
    def active_rows(self) -> int:
        if self.offsets is None:
            return self.rows
        return int(self.offsets[-1]) - int(self.offsets[0])

    def algorithmic_bytes(self) -> int:
        """BF16 read + packed FP4 write + E4M3 scale write, for active rows."""
        w = self.width
        per_row = (2 * w if self.kind == "quantize" else 4 * w) + w // 2 + w // 16
        return per_row * self.active_rows


def quantize_normal(rows=128, K=2048, seed=0) -> Workload:
    x = _chunked(rows, K, seed, 1,
                 lambda rng, n, _: bf16_bits(rng.standard_normal((n, K), dtype=np.float32)))
    return Workload("quantize", "quantize", rows, K, x)


def fused_normal(rows=512, I=2048, seed=1, gate_sigma=2.0, up_sigma=1.0, L=7.0) -> Workload:
    sig = np.where(gate_column_mask(I), np.float32(gate_sigma), np.float32(up_sigma))
    gu = _chunked(rows, 2 * I, seed, 2,
                  lambda rng, n, _: bf16_bits(rng.standard_normal((n, 2 * I), dtype=np.float32)
                                              * sig))
    return Workload("fused", "fused", rows, I, gu, clamp_L=L)


def ragged_routing(tokens=4096, experts=256, topk=8, I=2048, seed=2, sigma=1.5, L=7.0,
                   pad_rows=0) -> Workload:
    """Per-expert contiguous segments; `pad_rows` extra rows after the last
    segment belong to no expert (they must be left untouched)."""
    offsets = routing_offsets(tokens, experts, topk, seed)
    rows = int(offsets[-1]) + pad_rows
    gu = _chunked(rows, 2 * I, seed, 3,
                  lambda rng, n, _: bf16_bits(rng.standard_normal((n, 2 * I), dtype=np.float32)
                                              * np.float32(sigma)))
    return Workload("ragged", "fused", rows, I, gu, clamp_L=L, offsets=offsets,
                    meta={"tokens": tokens, "experts": experts, "topk": topk})


def _heavy_tail_fill(width_vals: int, outlier_frac: float, zero_block_frac: float,
                     block_vals: int):
    """0.5 * t(3) values, a fraction of them x100, and a fraction of
    `block_vals`-wide groups set to +0."""
    def fill(rng, n, _):
        v = (0.5 * rng.standard_t(3, (n, width_vals))).astype(np.float32)
        out = rng.random((n, width_vals)) < outlier_frac
        v[out] *= np.float32(100.0)
        zb = rng.random((n, width_vals // block_vals)) < zero_block_frac
        v.reshape(n, width_vals // block_vals, block_vals)[zb] = 0.0
        return bf16_bits(v)
    return fill


def prefill_heavy_tail(rows=65536, I=3072, seed=3, L=10.0) -> Workload:
    # one output 16-block reads 32 consecutive interleaved values
    gu = _chunked(rows, 2 * I, seed, 4, _heavy_tail_fill(2 * I, 1e-3, 0.05, 32))
    return Workload("prefill", "fused", rows, I, gu, clamp_L=L)


def prefill_heavy_tail_quantize(rows=65536, K=3072, seed=3) -> Workload:
    """The prefill distribution as quantize-only input: there the E4M3 scale
    reaches its 448 saturation, which the clamp keeps out of the fused path."""
    x = _chunked(rows, K, seed, 5, _heavy_tail_fill(K, 1e-3, 0.05, 16))
    return Workload("prefill_quantize", "quantize", rows, K, x)


EDGE_KINDS = ("signed_zero", "saturated_gate_tiny_up", "clamp_boundary", "huge", "structured")
EDGE_TABLE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "tests", "golden",
                          "edge_adversarial_blocks.npz")
_edge_table = None


def edge_table() -> dict:
    """The adversarial blocks: "fused" [n, 32] interleaved BF16 bits (for
    L = 7) and "quantize" [m, 16] BF16 bits. Raises if the table is missing:
    the edge workloads are not built without it."""
    global _edge_table
    if _edge_table is None:
        if not os.path.exists(EDGE_TABLE):
            raise FileNotFoundError(f"{EDGE_TABLE} is missing (tests/golden/make_edge_adversarial_blocks.py)")
        with np.load(EDGE_TABLE) as z:
            _edge_table = {"fused": z["fused"].astype(np.uint16), "quantize": z["quantize"].astype(np.uint16),
                           "fused_clamp_L": float(z["fused_clamp_L"])}
    return _edge_table


def edge_structured(rows=16384, I=4096, seed=4, L=7.0, adversarial_frac=0.10) -> Workload:
    """90% N(0,1) blocks; the rest one of EDGE_KINDS per output block. The
    "structured" blocks are rows of the adversarial table (for L = 7; at
    another L they stay N(0,1)): SwiGLU values on or next to scale ties and
    half-step ties. meta["kinds"][r, b] is the kind index + 1 (0 = plain)."""
    Lf = np.float32(L)
    nb = I // 16
    tab = edge_table()
    tie_blocks = bf16_to_f32(tab["fused"]) if L == tab["fused_clamp_L"] else None

    def fill(rng, n, r0):
        v = rng.standard_normal((n, 2 * I), dtype=np.float32)
        blocks = v.reshape(n, nb, 2, 2, 8)        # [row, block, group, gate/up, 8]
        kind = np.where(rng.random((n, nb)) < adversarial_frac,
                        rng.integers(1, len(EDGE_KINDS) + 1, (n, nb)), 0)
        sel = kind == 1                          # ups exactly +-0
        ups = blocks[sel][:, :, 1, :]
        signs = np.where(rng.random(ups.shape) < 0.5, np.float32(-0.0), np.float32(0.0))
        tmp = blocks[sel]; tmp[:, :, 1, :] = signs; blocks[sel] = tmp
        sel = kind == 2                          # gates above L, ups tiny
        tmp = blocks[sel]
        m = tmp.shape[0]
        tmp[:, :, 0, :] = Lf * (1.0 + np.abs(rng.standard_normal((m, 2, 8), dtype=np.float32)))
        umax = np.exp(rng.uniform(np.log(6 * 2.0 ** -12 / L), np.log(6 * 2.0 ** -5 / L),
                                  (m, 1, 1))).astype(np.float32)
        tmp[:, :, 1, :] = umax * rng.uniform(-1, 1, (m, 2, 8)).astype(np.float32)
        blocks[sel] = tmp
        sel = kind == 3                          # values on and next to +-L
        tmp = blocks[sel]
        choices = np.array([L, -L, L * (1 + 2 ** -7), L * (1 - 2 ** -8), -L * (1 + 2 ** -7),
                            -L * (1 - 2 ** -8), 2 * L, -2 * L], np.float32)
        tmp[...] = rng.choice(choices, tmp.shape)
        blocks[sel] = tmp
        sel = kind == 4                          # huge magnitudes both ways
        tmp = blocks[sel]
        tmp[...] = (rng.choice(np.array([-1, 1], np.float32), tmp.shape)
                    * np.exp(rng.uniform(np.log(30.0), np.log(3e38), tmp.shape))).astype(np.float32)
        blocks[sel] = tmp
        sel = kind == 5                          # table rows: ties and near-ties
        if tie_blocks is not None and np.any(sel):
            v.reshape(n, nb, 32)[sel] = tie_blocks[rng.integers(0, tie_blocks.shape[0], int(np.count_nonzero(sel)))]
        kinds_out[r0:r0 + n] = kind
        return bf16_bits(v)

    kinds_out = np.zeros((rows, nb), np.uint8)
    gu = _chunked(rows, 2 * I, seed, 6, fill)
    return Workload("edge", "fused", rows, I, gu, clamp_L=L, meta={"kinds": kinds_out})


def edge_quantize(rows=16384, K=4096, seed=4, adversarial_frac=0.10) -> Workload:
    """x ~ N(0, 1) with a fraction of the 16-blocks replaced by rows of
    the adversarial quantize table. meta["adversarial"][r, b] marks them."""
    tab = edge_table()["quantize"]
    nb = K // 16

    def fill(rng, n, r0):
        v = bf16_bits(rng.standard_normal((n, K), dtype=np.float32)).reshape(n, nb, 16)
        sel = rng.random((n, nb)) < adversarial_frac
        v[sel] = tab[rng.integers(0, tab.shape[0], int(np.count_nonzero(sel)))]
        marks[r0:r0 + n] = sel
        return v.reshape(n, K)

    marks = np.zeros((rows, nb), bool)
    x = _chunked(rows, K, seed, 9, fill)
    return Workload("edge_quantize", "quantize", rows, K, x, meta={"adversarial": marks})


@dataclass
class GemmWorkload:
    """Inputs of the L1 GEMM with the step in its epilogue."""
    name: str
    rows: int
    H: int
    I: int
    x: np.ndarray                   # uint16 BF16 bits [rows, H]
    w1: np.ndarray                  # uint16 BF16 bits [experts, 2I, H]
    offsets: np.ndarray             # int32 [experts + 1]
    clamp_L: float
    meta: dict = field(default_factory=dict)

    @property
    def active_rows(self) -> int:
        return int(self.offsets[-1]) - int(self.offsets[0])

    def active_experts(self) -> int:
        return int(np.count_nonzero(np.diff(self.offsets.astype(np.int64)) > 0))

    def algorithmic_bytes(self) -> int:
        """x rows read once, every used expert's weights read once, NVFP4 out."""
        return (self.active_rows * (2 * self.H + self.I // 2 + self.I // 16)
                + self.active_experts() * 2 * self.I * self.H * 2)

    def flops(self) -> int:
        return 2 * self.active_rows * self.H * 2 * self.I


def gemm_weights(experts=256, H=7168, I=2048, seed=6, sigma=1.5) -> np.ndarray:
    """w1 [experts, 2I, H] BF16 ~ N(0, sigma^2 / H): the accumulators of x ~
    N(0, 1) rows are then ~N(0, sigma^2), like the ragged workload's gate/up
    values. Rows come in [gate x8, up x8] groups only by name: every row is
    drawn alike."""
    ws = np.float32(sigma / np.sqrt(H))
    w1 = _chunked(experts * 2 * I, H, seed, 8,
                  lambda rng, n, _: bf16_bits(rng.standard_normal((n, H), dtype=np.float32) * ws))
    return w1.reshape(experts, 2 * I, H)


def gemm_rows(tokens=4096, experts=256, topk=8, H=7168, seed=6, pad_rows=0):
    """(x [rows, H] BF16 ~ N(0, 1), offsets) with routing as ragged_routing."""
    offsets = routing_offsets(tokens, experts, topk, seed)
    rows = int(offsets[-1]) + pad_rows
    x = _chunked(rows, H, seed, 7,
                 lambda rng, n, _: bf16_bits(rng.standard_normal((n, H), dtype=np.float32)))
    return x, offsets


def gemm_ragged(tokens=4096, experts=256, topk=8, H=7168, I=2048, seed=6, sigma=1.5, L=7.0,
                pad_rows=0, w1=None) -> GemmWorkload:
    """The L1 GEMM's inputs: gemm_rows and gemm_weights (w1 may be passed
    in to share it between row sets)."""
    x, offsets = gemm_rows(tokens, experts, topk, H, seed, pad_rows)
    if w1 is None:
        w1 = gemm_weights(experts, H, I, seed, sigma)
    return GemmWorkload("gemm_ragged", x.shape[0], H, I, x, w1, offsets, L,
                        meta={"tokens": tokens, "experts": experts, "topk": topk})


def make(name: str, **kw) -> Workload:
    """Workload by name, at full size unless sizes are given."""
    table = {
        "quantize": quantize_normal,
        "fused": fused_normal,
        "ragged": ragged_routing,
        "prefill": prefill_heavy_tail,
        "prefill_quantize": prefill_heavy_tail_quantize,
        "edge": edge_structured,
        "edge_quantize": edge_quantize,
    }
    return table[name](**kw)
