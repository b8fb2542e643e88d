"""Pins for the oracle: every check compares it with something that is not
its own code -- the pages' printed values, torch's float8_e4m3fn cast (the
routine the pages' own Python reference used), brute-force nearest-even
searches over the format's value sets, exact rational arithmetic, and a
50-digit decimal evaluation of SwiGLU.

Each test is chosen so that a plausible slip in the oracle (a wrong bias, a
missing carry, round-half-up instead of half-even, a dropped sign, a
transposed gate/up operand, a wrong nibble order) fails at least one of them.
"""
import math
import os
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

# ---------------------------------------------------------------------------
# Value sets written from the format definitions, used by brute-force search.
#   E4M3: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent field 0
#   is subnormal (m / 512); exp 15 / mant 7 is NaN, so codes 0x00..0x7e are
#   the finite non-negative values.  (Cross-checked against torch below.)
#   E2M1: magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6} for indices 0..7.
# ---------------------------------------------------------------------------
E4M3_VALUES = [Fraction(c & 7, 512) if (c >> 3) == 0
               else Fraction(8 + (c & 7), 8) * Fraction(2) ** ((c >> 3) - 7)
               for c in range(0x7f)]
E2M1_GRID = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2),
             Fraction(2), Fraction(3), Fraction(4), Fraction(6)]


def nearest_even_code(q: Fraction, values) -> int:
    """Index of the value nearest to q; on a tie the even index (mantissa 0)."""
    best_d, best_c = None, None
    for c, v in enumerate(values):
        d = abs(q - v)
        if best_d is None or d < best_d or (d == best_d and c % 2 == 0):
            best_d, best_c = d, c
    return best_c


def round_half_even(x: Fraction) -> int:
    f = math.floor(x)
    r = x - f
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and f % 2 == 1):
        return f + 1
    return f


def exact_nibble(s: float) -> int:
    """E2M1 nibble of s in exact arithmetic: half-step h = nearest-even
    integer to 2 min(|s|, 6), then the E2M1 magnitude nearest h/2."""
    h = round_half_even(2 * min(abs(Fraction(s)), Fraction(6)))
    idx = nearest_even_code(Fraction(h, 2), E2M1_GRID)
    return idx | (8 if math.copysign(1.0, s) < 0 else 0)


def exact_block(y32):
    """One NVFP4 block in exact rational arithmetic (no fp32 division)."""
    ys = [Fraction(float(v)) for v in y32]
    amax = max(abs(v) for v in ys)
    sf = nearest_even_code(amax / 6, E4M3_VALUES)
    d = E4M3_VALUES[sf]
    nibs = []
    for v, raw in zip(ys, y32):
        neg = math.copysign(1.0, float(raw)) < 0
        mag = Fraction(0) if d == 0 else abs(v) / d
        h = round_half_even(2 * min(mag, Fraction(6)))
        nibs.append(nearest_even_code(Fraction(h, 2), E2M1_GRID) | (8 if neg else 0))
    packed = [nibs[2 * j] | (nibs[2 * j + 1] << 4) for j in range(8)]
    return np.array(packed, np.uint8), sf


def f32_from_bits(bits):
    return np.asarray(bits, dtype=np.uint32).view(np.float32)


# ---------------------------------------------------------------------------
# 1. The pages' printed values
# ---------------------------------------------------------------------------

def _golden_rows():
    rows = []
    with open(os.path.join(GOLDEN, "pages_printed_values.txt")) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            kind, inp, exp, where = [p.strip() for p in line.split("|")]
            rows.append((kind, inp, exp, where))
    return rows


@pytest.mark.parametrize("kind,inp,exp,where", _golden_rows())
def test_pages_printed_values(oracle_mod, kind, inp, exp, where):
    o = oracle_mod
    if kind == "e4m3_encode":
        assert o.fp8_e4m3_from_float32(float(inp)) == int(exp, 16), where
    elif kind == "e4m3_decode":
        digits = len(exp.split(".")[1]) if "." in exp else 0
        assert round(o.fp8_e4m3_to_float32(int(inp, 16)), digits) == float(exp), where
    elif kind == "e4m3_is_nan":
        assert math.isnan(o.fp8_e4m3_to_float32(int(inp, 16))) == bool(int(exp)), where
    elif kind == "e2m1_nibble":
        assert o.quantize_e2m1_nibble(float(inp)) == int(exp), where
    elif kind == "step_to_idx":
        assert o.half_step_to_e2m1_idx(int(inp)) == int(exp), where
    else:
        raise AssertionError(f"unknown fixture kind {kind}")


# ---------------------------------------------------------------------------
# 2. FP8 E4M3
# ---------------------------------------------------------------------------

def test_e4m3_decode_all_256_codes_match_torch(oracle_mod):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).float().numpy()
    for c in range(256):
        got = oracle_mod.fp8_e4m3_to_float32(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), hex(c)
        else:
            assert got == ref[c] and math.copysign(1, got) == math.copysign(1, ref[c]), hex(c)
    nan_codes = [c for c in range(256) if math.isnan(oracle_mod.fp8_e4m3_to_float32(c))]
    assert nan_codes == [0x7f, 0xff]


def test_e4m3_value_table_matches_torch():
    # the brute-force value set used below is the format itself
    ref = torch.arange(0x7f, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    assert [float(v) for v in E4M3_VALUES] == ref.tolist()


def test_e4m3_roundtrip_all_finite_codes(oracle_mod):
    for c in range(256):
        if c & 0x7f == 0x7f:
            continue
        v = oracle_mod.fp8_e4m3_to_float32(c)
        assert oracle_mod.fp8_e4m3_from_float32(v) == c, hex(c)


def _dense_fp32_below(limit_bits: int) -> np.ndarray:
    """Every fp32 whose bits 8..30 take each value below limit_bits >> 8, each
    with low byte 0x00, 0x01, 0x7f, 0x80, 0x81 and 0xff: covers every E4M3
    rounding tie (the bits under the kept mantissa exactly 100..0) and both
    neighbours of each, across all binades including fp32 subnormals."""
    hi = np.arange(0, limit_bits >> 8, dtype=np.uint32) << 8
    lows = np.array([0x00, 0x01, 0x7f, 0x80, 0x81, 0xff], dtype=np.uint32)
    return f32_from_bits((hi[:, None] | lows[None, :]).ravel())


def test_e4m3_encode_matches_torch_cast_below_464(oracle_mod):
    v = _dense_fp32_below(0x43E80000)       # every |v| < 464
    got = oracle_mod.fp8_e4m3_from_float32_array(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(v[i]), hex(got[i]), hex(ref[i])) for i in bad[:10]]
    neg = oracle_mod.fp8_e4m3_from_float32_array(-v[::97])
    assert np.array_equal(neg, got[::97] | 0x80)


def test_e4m3_encode_saturates_at_448(oracle_mod):
    # READING: the pages clamp to 448 where torch's cast gives NaN
    for v in [448.0, 455.99, 464.0, 464.01, 479.9, 480.0, 1000.0, 3.0e38, float("inf")]:
        assert oracle_mod.fp8_e4m3_from_float32(v) == 0x7e, v
        assert oracle_mod.fp8_e4m3_from_float32(-v) == 0xfe, v


def test_e4m3_encode_brute_force_nearest_even(oracle_mod):
    rng = np.random.default_rng(1234)
    mids = [(E4M3_VALUES[i] + E4M3_VALUES[i + 1]) / 2 for i in range(len(E4M3_VALUES) - 1)]
    vals = []
    for m in mids:                          # every rounding tie and its neighbours
        t = np.float32(float(m))
        assert Fraction(float(t)) == m
        vals += [t, np.nextafter(t, np.float32(0)), np.nextafter(t, np.float32(1e9))]
    vals += list(np.float32(np.exp(rng.uniform(np.log(1e-5), np.log(600), 4000))))
    vals += [np.float32(2.0 ** -10), np.float32(1.5 * 2.0 ** -10), np.float32(2.0 ** -6)]
    vals = np.array(vals, np.float32)
    got = oracle_mod.fp8_e4m3_from_float32_array(vals)
    for v, g in zip(vals, got):
        assert g == nearest_even_code(Fraction(float(v)), E4M3_VALUES), (float(v), hex(g))
    # the two subnormal ties: 2^-10 is half of the smallest subnormal -> 0
    assert oracle_mod.fp8_e4m3_from_float32(2.0 ** -10) == 0x00
    assert oracle_mod.fp8_e4m3_from_float32(1.5 * 2.0 ** -10) == 0x01


# ---------------------------------------------------------------------------
# 3. E2M1 nibbles
# ---------------------------------------------------------------------------

def test_step_to_idx_is_nearest_even_on_the_e2m1_grid(oracle_mod):
    for h in range(13):
        assert oracle_mod.half_step_to_e2m1_idx(h) == nearest_even_code(Fraction(h, 2), E2M1_GRID)


def test_e2m1_all_16_codes_roundtrip(oracle_mod):
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for nib in range(16):
        v = oracle_mod.e2m1_nibble_to_float32(nib)
        assert abs(v) == grid[nib & 7]
        assert oracle_mod.quantize_e2m1_nibble(v if nib != 8 else -0.0) == nib


def test_nibble_brute_force_on_a_fine_grid(oracle_mod):
    ks = np.arange(-7 * 256, 7 * 256 + 1)
    s = (ks / 256.0).astype(np.float32)             # every multiple of 2^-8 in [-7, 7]
    s = np.concatenate([s, np.nextafter(s, np.float32(-1e9)), np.nextafter(s, np.float32(1e9)),
                        np.array([-0.0, 0.0], np.float32)])
    got = oracle_mod.quantize_e2m1_nibble_array(s)
    for v, g in zip(s, got):
        assert g == exact_nibble(float(v)), (float(v), g)


def test_nibble_two_stage_rounding_is_not_direct_rne(oracle_mod):
    # The pages' 5.25 case: RNE(10.5) = 10 -> idx 6 (value 4), whereas rounding
    # 5.25 straight onto the E2M1 grid gives 6.0 (idx 7). The two rules differ
    # on (2.5, 2.75), (3.25, 3.5) and (5.0, 5.25].
    for s, nib in [(5.25, 6), (5.1, 6), (5.26, 7), (2.6, 4), (2.75, 5), (3.4, 6), (3.25, 5)]:
        assert oracle_mod.quantize_e2m1_nibble(s) == nib, s
        assert oracle_mod.quantize_e2m1_nibble(-s) == nib | 8, s
    direct = [nearest_even_code(Fraction(s), E2M1_GRID) for s in (5.25, 5.1, 2.6, 3.4)]
    assert direct == [7, 7, 5, 5]


def test_nibble_error_bound(oracle_mod):
    rng = np.random.default_rng(7)
    s = rng.uniform(-8, 8, 200000).astype(np.float32)
    nib = oracle_mod.quantize_e2m1_nibble_array(s)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)
    deq = grid[nib & 7] * np.where(nib & 8, -1.0, 1.0)
    m = np.minimum(np.abs(s.astype(np.float64)), 6.0)
    err = np.abs(np.abs(deq) - m)
    assert np.all(np.sign(deq[deq != 0]) == np.sign(s[deq != 0]))
    assert err[m <= 2.0].max() <= 0.25          # half-step error only
    assert err.max() <= 1.25                    # worst case s = 5.25 -> 4
    assert err.max() > 1.2


# ---------------------------------------------------------------------------
# 4. One NVFP4 block, against exact rational arithmetic
# ---------------------------------------------------------------------------

def _adversarial_blocks(rng):
    blocks = []
    # amax / 6 on every E4M3 rounding tie (and its fp32 neighbours)
    for i in range(len(E4M3_VALUES) - 1):
        m = (E4M3_VALUES[i] + E4M3_VALUES[i + 1]) / 2
        amax = np.float32(float(6 * m))
        assert Fraction(float(amax)) == 6 * m
        for a in (amax, np.nextafter(amax, np.float32(0)), np.nextafter(amax, np.float32(1e9))):
            y = rng.uniform(-1, 1, 16).astype(np.float32) * a
            y[rng.integers(16)] = -a if rng.integers(2) else a
            blocks.append(y)
    # elements on every half-step tie of a scale, and their neighbours
    for code in list(range(1, 0x7f, 3)):
        d = float(E4M3_VALUES[code])
        ties = [(2 * k + 1) / 4 * d for k in range(12)]
        cand = []
        for t in ties:
            t32 = np.float32(t)
            cand += [t32, np.nextafter(t32, np.float32(0)), np.nextafter(t32, np.float32(1e9))]
        cand = np.array(cand, np.float32)
        for j in range(0, len(cand), 15):
            y = np.zeros(16, np.float32)
            part = cand[j:j + 15]
            y[:len(part)] = part * np.where(rng.integers(0, 2, len(part)) == 1, -1, 1)
            y[15] = np.float32(6 * d)               # fixes sf = code exactly
            blocks.append(y)
    # subnormal scales, the underflow tie, saturation, signed zeros
    for m in range(1, 9):
        for amax in (6 * m * 2.0 ** -9, 6 * (m + 0.5) * 2.0 ** -9):
            y = (rng.uniform(-1, 1, 16) * amax).astype(np.float32)
            y[0] = np.float32(amax)
            blocks.append(y)
    for amax in (6 * 2.0 ** -10, 6 * 2.0 ** -11, 6 * 448.0, 6 * 464.0, 6 * 470.0, 1e30):
        y = (rng.uniform(-1, 1, 16) * amax).astype(np.float32)
        y[3] = np.float32(-amax)
        blocks.append(y)
    blocks.append(np.array([0.0, -0.0] * 8, np.float32))
    blocks.append(np.array([1e-30, -1e-30, 0.0, -0.0] * 4, np.float32))
    return blocks


def test_block_quantization_against_exact_arithmetic(oracle_mod):
    rng = np.random.default_rng(2024)
    blocks = _adversarial_blocks(rng)
    for scale in (1e-4, 1e-2, 1.0, 30.0, 1e3, 1e5):
        for _ in range(60):
            blocks.append((rng.standard_normal(16) * scale).astype(np.float32))
    for _ in range(100):   # BF16-valued blocks, the quantize-only domain
        x = (rng.standard_normal(16) * 4).astype(np.float32)
        blocks.append((x.view(np.uint32) & 0xFFFF0000).view(np.float32))
    for y in blocks:
        packed, sf = oracle_mod.quantize_nvfp4_block(y)
        e_packed, e_sf = exact_block(y)
        assert sf == e_sf, (y, hex(sf), hex(e_sf))
        assert np.array_equal(packed, e_packed), (y, packed, e_packed)


def test_block_invariants(oracle_mod):
    rng = np.random.default_rng(99)
    for _ in range(2000):
        y = (rng.standard_normal(16) * 10.0 ** rng.uniform(-4, 4)).astype(np.float32)
        packed, sf = oracle_mod.quantize_nvfp4_block(y)
        assert sf <= 0x7e and sf != 0x7f
        nib = np.stack([packed & 15, packed >> 4], 1).ravel()
        i = int(np.argmax(np.abs(y)))
        # the amax element scales to s = amax/d with d within the scale's
        # rounding of amax/6: for a normal scale s is in [6/(1+1/16),
        # 6/(1-1/16)] -> index 7; a subnormal scale m * 2^-9 rounds amax/6 by
        # up to half a step, so s >= 6(m-1/2)/m: >= 3 for m = 1 (index >= 5),
        # >= 4.5 for m >= 2 (index >= 6)
        if 8 <= sf < 0x7e:
            assert nib[i] & 7 == 7
        elif sf == 1:
            assert nib[i] & 7 >= 5
        elif 2 <= sf < 8:
            assert nib[i] & 7 >= 6


def test_packing_order_low_nibble_is_even_element(oracle_mod):
    y = np.array([0.0, 6.0] * 8, np.float32)       # amax 6 -> sf = E4M3(1.0)
    packed, sf = oracle_mod.quantize_nvfp4_block(y)
    assert sf == 0x38
    assert packed.tolist() == [0x70] * 8
    y = np.array([-3.0, 0.5] + [0.0] * 13 + [6.0], np.float32)
    packed, sf = oracle_mod.quantize_nvfp4_block(y)
    assert packed[0] == (0x8 | 5) | (1 << 4)
    assert packed[7] == 0 | (7 << 4)


# ---------------------------------------------------------------------------
# 5. Clamped SwiGLU, against a 50-digit decimal evaluation
# ---------------------------------------------------------------------------

def _nearest_f32_of_decimal(y: Decimal):
    """(nearest fp32 to y, the runner-up, undecidable) where undecidable
    means y lies so close to the midpoint of the two that a double-precision
    evaluation (relative error ~2^-50) cannot tell which side it is on."""
    c = np.float32(float(y))
    cands = [np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))]
    dist = sorted((abs(Decimal(float(v)) - y), int(np.float32(v).view(np.uint32)) & 1, v)
                  for v in cands if np.isfinite(v))
    undecidable = dist[1][0] - dist[0][0] <= abs(y) * Decimal(2) ** -45
    return dist[0][2], dist[1][2], undecidable


def test_swiglu_against_decimal(oracle_mod):
    getcontext().prec = 50
    rng = np.random.default_rng(5)

    def bf16(a):
        return ((np.asarray(a, np.float32).view(np.uint32) & 0xFFFF0000).view(np.float32))

    L = 7.0
    g = np.concatenate([bf16(rng.standard_normal(3000) * 4),
                        np.array([0.0, 7.0, 6.96875, 7.0625, 20.0, -15.0, -40.0, -87.5,
                                  -100.0, -300.0, 1e-20, -1e-20, 1e30], np.float32)])
    u = bf16(rng.standard_normal(g.size) * 2)
    skipped = 0
    for gi, ui in zip(g, u):
        a = min(float(gi), L)
        b = min(max(float(ui), -L), L)
        A, B = Decimal(a), Decimal(b)
        exact = A / (1 + (-A).exp()) * B
        want, runner_up, undecidable = _nearest_f32_of_decimal(exact)
        got = oracle_mod.swiglu_clamped(float(gi), float(ui), L)
        if undecidable:
            # e.g. a tiny gate: y = a*b/2 + a^2*b/4 with a*b/2 on an fp32
            # midpoint and the a^2 term below double precision
            skipped += 1
            assert got in (float(want), float(runner_up))
            continue
        if want == 0:
            assert got == 0
        else:
            assert got == float(want), (float(gi), float(ui), got, float(want))
    assert skipped <= 2


def test_swiglu_closed_forms(oracle_mod):
    o = oracle_mod
    L = 7.0
    for u in (-9.0, -1.0, -0.0, 0.0, 2.5, 9.0):
        y = o.swiglu_clamped(0.0, u, L)                  # silu(0) = 0
        assert y == 0.0 and math.copysign(1, y) == math.copysign(1, u)
    for u in (-3.0, 0.5, 6.0):
        assert o.swiglu_clamped(7.0, u, L) == o.swiglu_clamped(50.0, u, L) == \
            o.swiglu_clamped(1e30, u, L)                 # gate clamped at L
    for g in (-2.0, 0.75, 3.0, 9.0):
        assert o.swiglu_clamped(g, 100.0, L) == o.swiglu_clamped(g, 7.0, L)
        assert o.swiglu_clamped(g, -100.0, L) == o.swiglu_clamped(g, -7.0, L)
        assert o.swiglu_clamped(g, -3.0, L) == -o.swiglu_clamped(g, 3.0, L)
    rng = np.random.default_rng(3)
    for g, u in rng.standard_normal((500, 2)) * 3:
        y = o.swiglu_clamped(g, u, L)
        assert np.sign(y) == np.sign(np.float32(g)) * np.sign(np.float32(u)) or y == 0
    # |y| <= L * silu(L): the largest value reachable through the clamp
    assert abs(o.swiglu_clamped(30.0, 30.0, L)) == pytest.approx(7 * 7 / (1 + math.exp(-7)))


# ---------------------------------------------------------------------------
# 6. Tensor level: the interleaved layout, the ragged rows, the output layout
# ---------------------------------------------------------------------------

def _interleave(gate, up):
    """[rows, I] gate and up -> [rows, 2I] as groups [gate x8, up x8, ...]."""
    rows, I = gate.shape
    return np.stack([gate.reshape(rows, I // 8, 8), up.reshape(rows, I // 8, 8)],
                    axis=2).reshape(rows, 2 * I)


def _bf16_bits(a):
    return (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_deinterleave_pairs_each_output_with_its_own_gate_and_up(oracle_mod):
    rng = np.random.default_rng(11)
    rows, I, L = 3, 64, 7.0
    gate = _bf16_bits(rng.standard_normal((rows, I)) * 3)
    up = _bf16_bits(rng.standard_normal((rows, I)) * 3)
    gu = _interleave(gate, up)
    y = oracle_mod.swiglu_values(gu, L)
    gf = (gate.astype(np.uint32) << 16).view(np.float32)
    uf = (up.astype(np.uint32) << 16).view(np.float32)
    want = oracle_mod.swiglu_clamped_array(gf, uf, L).reshape(rows, I)
    assert np.array_equal(y, want)
    swapped = oracle_mod.swiglu_clamped_array(uf, gf, L).reshape(rows, I)
    assert not np.array_equal(y, swapped)


def test_quantize_tensor_layout(oracle_mod):
    rng = np.random.default_rng(12)
    x = _bf16_bits(rng.standard_normal((5, 48)))
    packed, sf = oracle_mod.quantize_nvfp4(x)
    assert packed.shape == (5, 24) and sf.shape == (5, 3)
    xf = (x.astype(np.uint32) << 16).view(np.float32)
    for r in range(5):
        for b in range(3):
            p, s = oracle_mod.quantize_nvfp4_block(xf[r, 16 * b:16 * b + 16])
            assert s == sf[r, b] and np.array_equal(p, packed[r, 8 * b:8 * b + 8])


def test_ragged_rows_outside_segments_untouched(oracle_mod):
    rng = np.random.default_rng(13)
    rows, I, L = 40, 32, 7.0
    gu = _bf16_bits(rng.standard_normal((rows, 2 * I)) * 2)
    full_p, full_s = oracle_mod.swiglu_quantize_nvfp4(gu, L)
    offsets = np.array([3, 3, 10, 25], np.int32)       # one empty segment
    packed = np.full((rows, I // 2), 0xA5, np.uint8)
    sf = np.full((rows, I // 16), 0x5A, np.uint8)
    oracle_mod.swiglu_quantize_nvfp4(gu, L, offsets, packed=packed, sf=sf)
    assert np.all(packed[:3] == 0xA5) and np.all(packed[25:] == 0xA5)
    assert np.all(sf[:3] == 0x5A) and np.all(sf[25:] == 0x5A)
    assert np.array_equal(packed[3:25], full_p[3:25]) and np.array_equal(sf[3:25], full_s[3:25])


def test_sampled_blocks_match_full_evaluation(oracle_mod):
    rng = np.random.default_rng(14)
    rows, I, L = 6, 64, 7.0
    gu = _bf16_bits(rng.standard_normal((rows, 2 * I)) * 2)
    full_p, full_s = oracle_mod.swiglu_quantize_nvfp4(gu, L)
    r = np.array([0, 5, 2, 3]); b = np.array([3, 0, 1, 2])
    p, s = oracle_mod.swiglu_quantize_nvfp4_blocks(gu, L, r, b)
    for k in range(4):
        assert s[k] == full_s[r[k], b[k]]
        assert np.array_equal(p[k], full_p[r[k], 8 * b[k]:8 * b[k] + 8])
