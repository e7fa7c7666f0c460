"""The GPU quantizer's shortcut, restated on the CPU and checked against the
oracle: codes come from rounding d * lo and d * hi, where d = fp32(x - bias)
and lo <= 1/scale <= hi are fp32(rs * (1 -+ 2^-21)), rs = fp32(1 / scale);
where the two roundings agree the code is taken, elsewhere the exact rule
decides ("Fused int4 Attention for Gemma 4 31B", Background: per-group scale
and bias; codes rounded half to even).  The claim: wherever they agree, the
code equals rint(fp32(d / scale)).  Each rounding here is round-half-even of
the exact product (the product of two binary32 values is exact in binary64),
which is what one fused multiply-add with 1.5 * 2^23 computes.  Random and
crafted near-tie groups, int4 and int8; the near-tie groups must send their
words to the exact rule, random data almost none."""
import numpy as np
import pytest

import oracle
from tests.near_ties import near_tie_groups
from tests.test_quant_op_order import random_groups, unpack


def bracket_codes(groups: np.ndarray, bits: int):
    """(codes where the bracket decides, mask of words it leaves to the exact rule)."""
    _, scale, bias = oracle.quantize_rows(groups, 64, bits)
    s = scale.reshape(-1).view(np.float16).astype(np.float32)[:, None]
    b = bias.reshape(-1).view(np.float16).astype(np.float32)[:, None]
    x = groups.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        rs = (np.float32(1.0) / s).astype(np.float32)
    lo = (rs * np.float32(1.0 - 2.0 ** -21)).astype(np.float32)
    hi = (rs * np.float32(1.0 + 2.0 ** -21)).astype(np.float32)
    d = (x - b).astype(np.float32)
    with np.errstate(invalid="ignore"):
        ra = np.rint(d.astype(np.float64) * lo.astype(np.float64))
        rb = np.rint(d.astype(np.float64) * hi.astype(np.float64))
    normal = s >= np.float32(2.0 ** -14)
    agree = (ra == rb).reshape(len(groups), 8, 8).all(axis=2)  # per 8-element word
    exact_words = ~(agree & normal)
    return ra, exact_words, s[:, 0] == 0, normal[:, 0]


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("kind", ["random", "near_ties"])
def test_bracket_agrees_with_division(bits, kind):
    groups = random_groups(4096, 71 + bits) if kind == "random" else near_tie_groups(600, bits, seed=9 + bits)
    codes, _, _ = oracle.quantize_rows(groups, 64, bits)
    want = unpack(codes, bits).astype(np.float64)
    ra, exact_words, zero_scale, normal = bracket_codes(groups, bits)
    fast = ~np.repeat(exact_words, 8, axis=1) & ~zero_scale[:, None]
    assert np.array_equal(ra[fast], want[fast])
    share = exact_words[normal].mean()  # subnormal scales always take the exact rule
    if kind == "near_ties":
        assert share > 0.5  # the crafted elements sit where the two roundings can differ
    else:
        # exact ties included (the fp16 grid of the 1e-3-scaled groups lands on
        # half-integers of t now and then); int8 scales of those groups are
        # subnormal and always take the exact rule
        assert fast[normal].mean() > 0.98 and share < 1e-2
