"""The numeric constants of the CUDA kernels' double-float exponential,
recomputed here to 80 digits from their definitions (read from the source
text; nothing is executed on a GPU)."""
import os
import re
from decimal import Decimal, getcontext

import numpy as np

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "moe_swiglu_epilogue_gb300", "csrc", "moe_nvfp4.cu")
getcontext().prec = 80


def _hexfloat(tok: str) -> Decimal:
    tok = tok.strip().rstrip("f")
    if tok in ("0.0", "0"):
        return Decimal(0)
    return Decimal(float.fromhex(tok))


def _const(name: str) -> Decimal:
    m = re.search(rf"constexpr float {name} = ([-0-9a-fx.p+]+f);", open(SRC).read())
    assert m, name
    return _hexfloat(m.group(1))


def test_ln2_over_64_split():
    c = Decimal(2).ln() / 64
    hi, mid, lo = _const("kLn2x64Hi"), _const("kLn2x64Mid"), _const("kLn2x64Lo")
    assert abs(hi + mid + lo - c) < Decimal(2) ** -66
    # the head has at most 9 significant bits, so n * head is exact for |n| < 2^15
    m, e = np.frexp(float(hi))
    assert float(m * 2 ** 9).is_integer()
    assert abs(_const("kInvLn2x64") - 64 / Decimal(2).ln()) < Decimal(2) ** -17


def test_exp2_table_is_two_to_the_j_over_64():
    text = open(SRC).read()
    body = text[text.index("kExp2Table[64] = {"):]
    body = body[:body.index("};")]
    pairs = re.findall(r"\{([-0-9a-fx.p+]+f), ([-0-9a-fx.p+]+f)\}", body)
    assert len(pairs) == 64
    for j, (hi, lo) in enumerate(pairs):
        exact = Decimal(2) ** (Decimal(j) / 64)
        h, l = _hexfloat(hi), _hexfloat(lo)
        assert Decimal(float(np.float32(float(exact)))) == h, j       # hi = RN(2^(j/64))
        assert abs(h + l - exact) <= exact * Decimal(2) ** -47, j
