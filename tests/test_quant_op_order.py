"""The quantizer's operation order, pinned against an independent numpy
restatement of the rule ("Fused int4 Attention for Gemma 4 31B", Background:
per-group scale and bias; the affine rule scale = (max - min) / L, bias = min,
codes rounded half to even), in numpy's IEEE binary32 arithmetic:

    r = f32(max - min);  s32 = f32(r / L);  scale = f16(s32);  bias = f16(min)
    (a zero minimum stored as +0);  code = clip(rint(f32(f32(x - bias) / scale)), 0, L)
    (all codes 0 when scale rounds to 0).

The grid, tie and round-trip pins hold for several evaluation orders; this
one fixes it: over random groups and over crafted groups whose elements sit
on or within two ulps of a code boundary, the oracle must agree with the
restatement bit for bit, and the crafted groups must contain elements on
which a multiplication by a rounded reciprocal rounds to another code (so a
quantizer that took that shortcut would fail here)."""
import numpy as np
import pytest

import oracle
from tests.near_ties import near_tie_groups


def restated(groups: np.ndarray, bits: int):
    """numpy float32 restatement: groups [n, 64] fp16 -> (codes [n, 64], scale u16, bias u16)."""
    levels = np.float32((1 << bits) - 1)
    x = groups.astype(np.float32)
    mn = x.min(axis=1)
    mn = np.where(mn == 0, np.float32(0.0), mn)            # +0 for a zero minimum
    mx = x.max(axis=1)
    r = (mx - mn).astype(np.float32)
    s32 = (r / levels).astype(np.float32)
    scale = s32.astype(np.float16)
    bias = mn.astype(np.float16)
    s = scale.astype(np.float32)[:, None]
    b = bias.astype(np.float32)[:, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        t = ((x - b).astype(np.float32) / s).astype(np.float32)
    codes = np.clip(np.rint(t), 0, levels)
    codes = np.where(s == 0, 0, codes).astype(np.uint8)
    return codes, scale.view(np.uint16), bias.view(np.uint16)


def unpack(packed: np.ndarray, bits: int) -> np.ndarray:
    """Oracle codes [n, 64 * bits / 8] -> one code per element (low nibble first)."""
    if bits == 8:
        return packed
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out


def random_groups(n: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    g = rng.standard_normal((n, 64)).astype(np.float32)
    g[: n // 4] *= np.float32(20.0)                      # outlier-scaled groups
    g[n // 4: n // 2] *= np.float32(1e-3)                # tiny ranges
    g[n // 2: n // 2 + 8] = np.float32(0.5)              # degenerate: max == min
    g[n // 2 + 8: n // 2 + 16] = rng.standard_normal((8, 1)).astype(np.float32) * np.float32(6e-8)  # subnormal
    g[n // 2 + 16: n // 2 + 24, 0] = np.float32(-0.0)    # signed-zero minimum
    g[n // 2 + 16: n // 2 + 24, 1:] = np.abs(g[n // 2 + 16: n // 2 + 24, 1:])
    return g.astype(np.float16)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("kind", ["random", "near_ties"])
def test_oracle_matches_float32_restatement(bits, kind):
    groups = random_groups(4096, 31 + bits) if kind == "random" else near_tie_groups(600, bits, seed=bits)
    want_codes, want_scale, want_bias = restated(groups, bits)
    codes, scale, bias = oracle.quantize_rows(groups, 64, bits)
    assert np.array_equal(scale.reshape(-1), want_scale)
    assert np.array_equal(bias.reshape(-1), want_bias)
    assert np.array_equal(unpack(codes, bits), want_codes)


@pytest.mark.parametrize("bits", [4, 8])
def test_near_tie_groups_separate_division_from_reciprocal(bits):
    """The crafted groups have elements whose code under a multiplication by
    the rounded reciprocal 1/scale differs from the division's."""
    groups = near_tie_groups(600, bits, seed=bits)
    codes, scale, bias = restated(groups, bits)
    s = scale.view(np.float16).astype(np.float32)[:, None]
    b = bias.view(np.float16).astype(np.float32)[:, None]
    inv = (np.float32(1.0) / s).astype(np.float32)
    t_mul = ((groups.astype(np.float32) - b).astype(np.float32) * inv).astype(np.float32)
    alt = np.clip(np.rint(t_mul), 0, (1 << bits) - 1).astype(np.uint8)
    differ = int((alt != codes).sum())
    assert differ > 0
    # and exact ties are present (rounded to the even code)
    t = ((groups.astype(np.float32) - b) / s).astype(np.float32)
    ties = (t - np.floor(t)) == np.float32(0.5)
    assert ties.any()
    assert np.all(codes[ties] % 2 == 0)
