"""Pins for the CPU oracle: checks that do not reuse the oracle's own arithmetic.

Each test ties an oracle function to something fixed outside it: the IEEE
binary16 definition as implemented by numpy, values the pages print, closed
forms of softmax attention, invariances, and an independent library routine
(torch's scaled_dot_product_attention in float64).  A plausible slip in the
oracle (dropped bias, wrong nibble, wrong GQA head, sign error, transposed
operand, wrong rounding rule, wrong chunk merge) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# binary16 codec vs numpy (an independent implementation of IEEE 754)
# --------------------------------------------------------------------------

def test_f16_decode_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.f16_to_f64(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_f16_encode_random_and_ties():
    rng = np.random.default_rng(11)
    # random bit patterns over the whole binary32 range
    u = rng.integers(0, 2**32, size=400000, dtype=np.uint64).astype(np.uint32)
    x = u.view(np.float32)
    # values around the binary16 range, including subnormals and overflow
    y = (rng.standard_normal(200000) * np.exp2(rng.uniform(-30, 18, 200000))).astype(np.float32)
    # exact ties: midpoints between neighbouring binary16 values (representable in binary32)
    h = np.arange(0, 0x7bff, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    mid = ((lo + hi) / 2).astype(np.float32)
    assert np.array_equal(mid.astype(np.float64), (lo + hi) / 2)
    z = np.concatenate([x, y, mid, -mid, np.array([65504, 65520, 65519.99, 2**-25, 2**-24,
                                                   3 * 2**-26, 0.0, -0.0, np.inf, -np.inf],
                                                  dtype=np.float32)])
    ours = oracle.f32_to_f16(z)
    with np.errstate(over="ignore"):
        ref = z.astype(np.float16).view(np.uint16)
    nan = np.isnan(z)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.all((ours[nan] & 0x7c00) == 0x7c00) and np.all((ours[nan] & 0x3ff) != 0)


# --------------------------------------------------------------------------
# affine int4 quantisation (one group of 64)
# --------------------------------------------------------------------------

def _grid_group(bias=-1.0, step=0.125, order=None):
    ks = np.tile(np.arange(16), 4) if order is None else np.asarray(order)
    x = (bias + step * ks).astype(np.float16)
    assert np.array_equal(x.astype(np.float64), bias + step * ks)  # exact in fp16
    return x, ks


def test_quantize_grid_values_exact():
    x, ks = _grid_group()
    codes, s, b = oracle.quantize_group(x)
    assert np.frombuffer(np.uint16(s).tobytes(), np.float16)[0] == np.float16(0.125)
    assert np.frombuffer(np.uint16(b).tobytes(), np.float16)[0] == np.float16(-1.0)
    assert np.array_equal(codes, ks)
    codes_p, sc, bi = oracle.quantize_rows(x.reshape(1, 64))
    xh = oracle.dequantize_rows(codes_p, sc, bi)
    assert np.array_equal(xh.ravel(), x.astype(np.float64))


def test_quantize_ties_round_half_even():
    # group holds both ends of the grid (-1 .. 0.875, scale 0.125) plus crafted
    # midpoints k + 0.5 that must round to the even neighbour
    base = list(range(16)) * 3
    halves = [0.5, 1.5, 2.5, 3.5, 6.5, 9.5, 13.5, 14.5]
    ks = np.array(base + halves + [0, 15, 7, 8, 0, 15, 7, 8][: 64 - len(base) - len(halves)],
                  dtype=np.float64)
    assert ks.size == 64
    x = (-1.0 + 0.125 * ks).astype(np.float16)
    assert np.array_equal(x.astype(np.float64), -1.0 + 0.125 * ks)
    codes, s, b = oracle.quantize_group(x)
    want = np.array([int(k) if k == int(k) else (int(k) if int(k) % 2 == 0 else int(k) + 1)
                     for k in ks])
    assert np.array_equal(codes, want)
    # spot values: 2.5 -> 2, 3.5 -> 4, 0.5 -> 0, 14.5 -> 14
    tail = dict(zip(halves, codes[48:56]))
    assert tail[2.5] == 2 and tail[3.5] == 4 and tail[0.5] == 0 and tail[14.5] == 14


def _random_groups(rng, n):
    out = []
    for i in range(n):
        kind = i % 5
        g = rng.standard_normal(64).astype(np.float32)
        if kind == 1:
            g[rng.integers(64)] *= 20          # one outlier channel
        elif kind == 2:
            g *= 1e-4                          # small range, subnormal scale
        elif kind == 3:
            g = g * 3000 + 10000               # large magnitudes
        elif kind == 4:
            g = np.round(g * 4) / 4            # many repeated values
        out.append(g.astype(np.float16))
    return np.stack(out)


def test_quantize_round_trip_bound_and_ends():
    rng = np.random.default_rng(5)
    xs = _random_groups(rng, 3000)
    codes_p, sc, bi = oracle.quantize_rows(xs)
    xh = oracle.dequantize_rows(codes_p, sc, bi)
    x = xs.astype(np.float64)
    s = sc.view(np.float16).astype(np.float64)[:, 0]
    b = bi.view(np.float16).astype(np.float64)[:, 0]
    mn, mx = x.min(axis=1), x.max(axis=1)
    assert np.array_equal(b, mn)                                  # bias = group minimum
    # scale is within half an fp16 ulp of (max - min) / 15 (relative 2^-11 for
    # normal fp16, absolute 2^-25 in the subnormal range)
    exact = (mx - mn) / 15.0
    assert np.all(np.abs(s - exact) <= np.maximum(exact * 2.0**-11, 2.0**-25) * (1 + 1e-9))
    err = np.abs(x - xh)
    assert np.all(err <= s[:, None] * (0.5 + 1e-5))               # |x - xhat| <= scale / 2
    codes = np.stack([(codes_p & 0xF), (codes_p >> 4)], axis=-1).reshape(xs.shape)
    assert codes.max() <= 15
    rows = np.arange(xs.shape[0])
    assert np.all(codes[rows, x.argmin(axis=1)] == 0)             # minimum -> code 0
    assert np.all(codes[rows, x.argmax(axis=1)] == 15)            # maximum -> code 15
    assert np.all(xh[rows, x.argmin(axis=1)] == mn)               # minimum reproduced exactly
    # codes are monotone in x within each group
    order = np.argsort(x, axis=1, kind="stable")
    assert np.all(np.diff(np.take_along_axis(codes.astype(int), order, axis=1), axis=1) >= 0)


def _ulp16(v):
    """Spacing of binary16 numbers at |v| (2^-24 in the subnormal range)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0**-14)))
    return 2.0 ** (e - 10)


def test_dequantize_f16_pins():
    """fp16 dequantisation (the float cache of the dequantize-then-attend
    baseline): grid values exact, code 0 gives the bias bits, within half an
    fp16 ulp (plus the fp32 step) of the exact fp64 value, monotone in the code."""
    x, ks = _grid_group()
    codes_p, sc, bi = oracle.quantize_rows(x.reshape(1, 64))
    assert np.array_equal(oracle.dequantize_rows_f16(codes_p, sc, bi).view(np.float16).ravel(), x)

    rng = np.random.default_rng(9)
    xs = _random_groups(rng, 2000)
    codes_p, sc, bi = oracle.quantize_rows(xs)
    h = oracle.dequantize_rows_f16(codes_p, sc, bi)
    got = h.view(np.float16).astype(np.float64)
    exact = oracle.dequantize_rows(codes_p, sc, bi)          # fp64, exact
    err = np.abs(got - exact)
    assert np.all(err <= 0.5 * _ulp16(np.maximum(np.abs(got), np.abs(exact))) + np.abs(exact) * 2.0**-24)
    codes = np.stack([(codes_p & 0xF), (codes_p >> 4)], axis=-1).reshape(xs.shape)
    zero = codes == 0
    assert np.array_equal(h[zero], np.broadcast_to(bi[:, :1], codes.shape)[zero])  # code 0 -> bias bits
    # every code of every group: monotone non-decreasing in the code (scale >= 0)
    all_codes = np.tile(np.arange(16, dtype=np.uint8), 4)
    packed = (all_codes[0::2] | (all_codes[1::2] << 4)).astype(np.uint8)
    grid = oracle.dequantize_rows_f16(np.broadcast_to(packed, (sc.shape[0], 32)), sc, bi)
    g = grid.view(np.float16).astype(np.float64)[:, :16]
    assert np.all(np.diff(g, axis=1) >= 0)


def test_quantize_degenerate_groups():
    for v in (0.0, 1.5, -7.25, 65504.0, -2.0**-24):
        x = np.full(64, v, dtype=np.float16)
        codes, s, b = oracle.quantize_group(x)
        assert s == 0 and np.all(codes == 0)
        assert np.float16(np.frombuffer(np.uint16(b).tobytes(), np.float16)[0]) == np.float16(v)
    # range so small that (max - min)/15 rounds to a zero fp16 scale: every code 0,
    # reconstruction is the minimum, error at most the range
    x = np.zeros(64, dtype=np.float16)
    x[3] = np.float16(2.0**-24)
    codes, s, b = oracle.quantize_group(x)
    assert s == 0 and np.all(codes == 0) and b == 0


def test_quantize_group_of_zeros_scale_follows_first_element():
    """All 64 elements are ±0: the rule's maximum is the first element holding
    the largest value (a plain scan), so r = first - (+0) and the stored scale
    is -0 exactly when the group opens with -0; codes 0 and bias +0 always.
    The cases are written out by hand: which zero a scan keeps is the point."""
    neg, pos = np.float16(-0.0), np.float16(0.0)
    cases = [
        (np.full(64, neg), 0x8000),                                  # all -0
        (np.full(64, pos), 0x0000),                                  # all +0
        (np.array([neg] + [pos] * 63, np.float16), 0x8000),          # -0 first
        (np.array([pos] + [neg] * 63, np.float16), 0x0000),          # +0 first
        (np.array([neg, pos] * 32, np.float16), 0x8000),
        (np.array([pos, neg] * 32, np.float16), 0x0000),
    ]
    for x, want_scale in cases:
        for bits in (4, 8):
            codes, s, b = oracle.quantize_rows(x.reshape(1, 64), 64, bits)
            assert int(s.reshape(-1)[0]) == want_scale, (x[:2], bits)
            assert int(b.reshape(-1)[0]) == 0x0000
            assert not codes.any()
    # one nonzero element: the range is positive whatever the zeros' signs
    x = np.array([neg] * 63 + [np.float16(-1.0)], np.float16)
    _, s, _ = oracle.quantize_rows(x.reshape(1, 64), 64, 4)
    assert int(s.reshape(-1)[0]) == int(np.float16(1.0 / 15).view(np.uint16))


def test_quantize_signed_zero_minimum_is_positive_zero():
    # -0 and +0 both present at the minimum: the bias is +0 whichever comes first
    for first in (-0.0, 0.0):
        x = np.linspace(0, 3, 64).astype(np.float16)
        x[0] = np.float16(first)
        x[9] = np.float16(-first)
        codes, s, b = oracle.quantize_group(x)
        assert b == 0x0000 and codes[0] == 0 and codes[9] == 0


def test_nibble_order_fixture():
    lines = [l.split() for l in open(os.path.join(GOLDEN, "nibble_order.txt"))
             if l.strip() and not l.startswith("#")]
    pairs = [(lines[i], lines[i + 1]) for i in range(0, len(lines), 2)]
    for codes_line, bytes_line in pairs:
        assert codes_line[0] == "codes" and bytes_line[0] == "bytes"
        want_codes = [int(c) for c in codes_line[1:]]
        want_bytes = [int(b, 16) for b in bytes_line[1:]]
        n = len(want_codes)
        # build a group of 64 on the -1 + 0.125 k grid whose first n elements carry the
        # fixture codes; both ends of the grid are present so the codes are k exactly
        ks = np.array(want_codes + [0, 15] + [7] * (64 - n - 2))
        x = (-1.0 + 0.125 * ks).astype(np.float16)
        codes_p, _, _ = oracle.quantize_rows(x.reshape(1, 64))
        assert list(codes_p[0, : n // 2]) == want_bytes


# --------------------------------------------------------------------------
# decode attention
# --------------------------------------------------------------------------

def _small_problem(seed, B=2, Hq=8, Hkv=2, D=128, S=37):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, Hq, D)).astype(np.float16)
    k = rng.standard_normal((B, Hkv, S, D)).astype(np.float16)
    v = rng.standard_normal((B, Hkv, S, D)).astype(np.float16)
    return q, k, v


def _dequant(cache):
    kh = oracle.dequantize_rows(cache.kc, cache.ks, cache.kb, cache.group, cache.bits)
    vh = oracle.dequantize_rows(cache.vc, cache.vs, cache.vb, cache.group, cache.bits)
    return kh, vh


def test_attention_single_token_returns_value():
    q, k, v = _small_problem(1, S=1)
    cache = oracle.Cache.from_fp16(k, v)
    out = oracle.attention(q, cache, np.array([1, 1]), 1 / math.sqrt(128))
    _, vh = _dequant(cache)
    G = 4
    for h in range(8):
        assert np.array_equal(out[:, h], vh[:, h // G, 0])


def test_attention_identical_keys_give_mean_of_values():
    q, k, v = _small_problem(2, S=29)
    k[:] = k[:, :, :1]
    cache = oracle.Cache.from_fp16(k, v)
    out = oracle.attention(q, cache, np.array([29, 17]), 0.3)
    _, vh = _dequant(cache)
    for b, n in ((0, 29), (1, 17)):
        for h in range(8):
            np.testing.assert_allclose(out[b, h], vh[b, h // 4, :n].mean(axis=0), rtol=0, atol=1e-12)


def test_attention_zero_scale_gives_mean():
    q, k, v = _small_problem(3, S=23)
    cache = oracle.Cache.from_fp16(k, v)
    out = oracle.attention(q, cache, np.array([23, 5]), 0.0)
    _, vh = _dequant(cache)
    np.testing.assert_allclose(out[1, 6], vh[1, 1, :5].mean(axis=0), atol=1e-12)


def test_attention_two_tokens_closed_form():
    q, k, v = _small_problem(4, S=2, B=1)
    cache = oracle.Cache.from_fp16(k, v)
    a = 0.7
    out = oracle.attention(q, cache, np.array([2]), a)
    kh, vh = _dequant(cache)
    qd = q.astype(np.float64)
    for h in range(8):
        s0 = a * qd[0, h] @ kh[0, h // 4, 0]
        s1 = a * qd[0, h] @ kh[0, h // 4, 1]
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        w1 = 1.0 / (1.0 + math.exp(s0 - s1))
        np.testing.assert_allclose(out[0, h], w0 * vh[0, h // 4, 0] + w1 * vh[0, h // 4, 1],
                                   rtol=1e-13, atol=1e-13)


def test_attention_matches_torch_sdpa_float64():
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F

    for seed, (B, Hq, Hkv, D, S, a) in enumerate([(2, 8, 2, 128, 61, 1 / math.sqrt(128)),
                                                   (1, 32, 16, 256, 33, 1.0),
                                                   (3, 4, 4, 64, 10, 0.125),
                                                   (1, 64, 8, 128, 300, 1 / math.sqrt(128))]):
        q, k, v = _small_problem(100 + seed, B, Hq, Hkv, D, S)
        cache = oracle.Cache.from_fp16(k, v)
        lens = np.full(B, S, np.int32)
        out = oracle.attention(q, cache, lens, a)
        kh, vh = _dequant(cache)
        G = Hq // Hkv
        tq = torch.from_numpy(q.astype(np.float64)).unsqueeze(2)            # [B,Hq,1,D]
        tk = torch.from_numpy(kh).repeat_interleave(G, dim=1)               # [B,Hq,S,D]
        tv = torch.from_numpy(vh).repeat_interleave(G, dim=1)
        ref = F.scaled_dot_product_attention(tq, tk, tv, scale=a).squeeze(2).numpy()
        np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)


def test_attention_needle():
    # one key aligned with q: its score exceeds the others by >= 30, so the output is
    # that key's value up to e^-30 * S * max|v|
    rng = np.random.default_rng(7)
    B, Hq, Hkv, D, S = 1, 4, 1, 128, 1000
    q = np.zeros((B, Hq, D), np.float16)
    q[0, :, :] = 1.0
    k = (rng.standard_normal((B, Hkv, S, D)) * 0.05).astype(np.float16)
    v = rng.standard_normal((B, Hkv, S, D)).astype(np.float16)
    for pos in (0, 511, 512, S - 1):
        kk = k.copy()
        kk[0, 0, pos] = 1.0
        cache = oracle.Cache.from_fp16(kk, v)
        out = oracle.attention(q, cache, np.array([S]), 1.0)
        _, vh = _dequant(cache)
        assert np.abs(out[0] - vh[0, 0, pos]).max() <= math.exp(-30) * S * 5


def test_attention_token_permutation_invariant():
    q, k, v = _small_problem(8, S=50)
    perm = np.random.default_rng(9).permutation(50)
    c1 = oracle.Cache.from_fp16(k, v)
    c2 = oracle.Cache.from_fp16(k[:, :, perm], v[:, :, perm])
    lens = np.array([50, 50])
    np.testing.assert_allclose(oracle.attention(q, c1, lens, 0.2),
                               oracle.attention(q, c2, lens, 0.2), rtol=1e-12, atol=1e-13)


def test_attention_ragged_lengths_and_empty():
    q, k, v = _small_problem(10, B=3, S=40)
    cache = oracle.Cache.from_fp16(k, v)
    lens = np.array([40, 0, 13], np.int32)
    out = oracle.attention(q, cache, lens, 0.1)
    assert np.all(out[1] == 0.0)
    # sequence 2 over 13 tokens equals a cache truncated to 13 tokens
    c13 = oracle.Cache.from_fp16(k[2:3, :, :13].copy(), v[2:3, :, :13].copy())
    ref = oracle.attention(q[2:3].copy(), c13, np.array([13]), 0.1)
    np.testing.assert_array_equal(out[2], ref[0])
    # pairs restrict the work and leave other rows untouched (NaN)
    part = oracle.attention(q, cache, lens, 0.1, pairs=[(0, 3), (2, 7)])
    np.testing.assert_array_equal(part[0, 3], out[0, 3])
    np.testing.assert_array_equal(part[2, 7], out[2, 7])
    assert np.isnan(part[1, 0]).all()


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("chunk", [1, 7, 64, 512, 1000])
def test_split_k_equals_unsplit(chunk, bits):
    q, k, v = _small_problem(12, B=2, S=1000)
    cache = oracle.Cache.from_fp16(k, v, bits=bits)
    lens = np.array([1000, 517], np.int32)
    ref = oracle.attention(q, cache, lens, 1 / math.sqrt(128))
    m, l, acc = oracle.attention_partials(q, cache, lens, 1 / math.sqrt(128), chunk)
    out = oracle.merge_partials(m, l, acc)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)
    # empty chunks (beyond the second sequence's length) are marked empty
    nc = m.shape[-1]
    first_empty = -(-517 // chunk)
    if first_empty < nc:
        assert np.all(l[1, :, first_empty:] == 0) and np.all(np.isneginf(m[1, :, first_empty:]))


@pytest.mark.parametrize("bits", [4, 8])
def test_partial_state_definition(bits):
    # one chunk covering the sequence: m = max score, l = sum exp(s - m),
    # acc / l = attention output (int4 and int8 caches)
    q, k, v = _small_problem(13, B=1, S=20)
    cache = oracle.Cache.from_fp16(k, v, bits=bits)
    a = 0.25
    m, l, acc = oracle.attention_partials(q, cache, np.array([20]), a, chunk=64)
    kh, vh = _dequant(cache)
    for h in range(8):
        s = a * (kh[0, h // 4] @ q[0, h].astype(np.float64))
        np.testing.assert_allclose(m[0, h, 0], s.max(), rtol=1e-14)
        np.testing.assert_allclose(l[0, h, 0], np.exp(s - s.max()).sum(), rtol=1e-13)
        np.testing.assert_allclose(acc[0, h, 0], np.exp(s - s.max()) @ vh[0, h // 4], rtol=1e-12,
                                   atol=1e-13)


# --------------------------------------------------------------------------
# Hadamard rotation ("Running and Evaluating TurboQuant optimized Gemma 4")
# --------------------------------------------------------------------------

def _hadamard_fixture():
    rows = {l.split()[0]: np.array([float(v) for v in l.split()[1:]])
            for l in open(os.path.join(GOLDEN, "hadamard_worked_example.txt")) if l.strip() and not l.startswith("#")}
    return rows["input"], rows["rotated"]


def test_hadamard_worked_example():
    x, want = _hadamard_fixture()
    for dt in (np.float64, np.float32):
        y = oracle.hadamard(x.astype(dt))
        assert np.allclose(y, want, atol=5e-4, rtol=0)           # the page prints three decimals
        assert np.allclose(oracle.hadamard(y), x, atol=1e-6, rtol=0)  # its own inverse
    assert np.allclose(oracle.hadamard(x), want, atol=1e-15, rtol=0)  # the printed values are exact here


def test_hadamard_matches_sylvester_matrix():
    scipy_linalg = pytest.importorskip("scipy.linalg")
    rng = np.random.default_rng(21)
    for n in (2, 4, 64, 128, 256):
        H = scipy_linalg.hadamard(n) / math.sqrt(n)
        x = rng.standard_normal((5, n))
        x[:, 3 % n] *= 20.0                                          # an outlier channel
        ref = x @ H.T
        assert np.allclose(oracle.hadamard(x), ref, atol=1e-12, rtol=0)
        # fp32 fast transform: log2(n) rounded adds and one rounded scale
        y32 = oracle.hadamard(x.astype(np.float32)).astype(np.float64)
        ref32 = x.astype(np.float32).astype(np.float64) @ H.T
        bound = (math.log2(n) + 2) * 2.0**-24 * np.abs(x).sum(axis=1, keepdims=True)
        assert np.all(np.abs(y32 - ref32) <= bound)


def test_hadamard_norm_inverse_and_spreading():
    rng = np.random.default_rng(22)
    x = rng.standard_normal((20, 128))
    y = oracle.hadamard(x)
    assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    assert np.allclose(oracle.hadamard(y), x, atol=1e-13)
    q = rng.standard_normal(128)
    assert np.allclose(oracle.hadamard(q) @ y.T, q @ x.T, atol=1e-11)  # dot products kept
    spike = np.zeros(128)
    spike[17] = 1.0
    assert np.allclose(np.abs(oracle.hadamard(spike)), 1 / math.sqrt(128), atol=1e-15)  # an outlier spread evenly


def test_rotate_rows_f16_is_rounded_fp32_transform():
    rng = np.random.default_rng(23)
    x = (rng.standard_normal((50, 128)) * 3).astype(np.float16)
    got = oracle.rotate_rows_f16(x).astype(np.float64)
    exact = oracle.hadamard(x.astype(np.float64))
    # fp32 transform error (bound above) plus one fp16 rounding
    bound = 0.5 * _ulp16(np.maximum(np.abs(got), np.abs(exact))) + 9 * 2.0**-24 * np.abs(x.astype(np.float64)).sum(
        axis=1, keepdims=True)
    assert np.all(np.abs(got - exact) <= bound)
    # exactly representable results come back exactly: +-1 entries of a scaled Hadamard column
    e = np.zeros((1, 64), np.float16)
    e[0, 5] = 8.0                                                    # 8 / sqrt(64) = 1
    assert np.array_equal(np.abs(oracle.rotate_rows_f16(e).astype(np.float64)), np.ones((1, 64)))


# --------------------------------------------------------------------------
# int8 codes ("Running and Evaluating TurboQuant optimized Gemma 4", driver
# flags --kv-bits {4,8}): the same affine rule with 255 levels
# --------------------------------------------------------------------------

def test_int8_grid_values_and_ties():
    # four groups of 64 cover codes 0..255 on the grid -1 + k/128 (exact in fp16),
    # each holding both ends so that scale = (max - min)/255 = 1/128 exactly
    ks = np.arange(256)
    for part in range(4):
        k = np.concatenate([[0, 255], ks[part * 62:(part + 1) * 62]])[:64]
        if k.size < 64:
            k = np.concatenate([k, np.full(64 - k.size, 7)])
        x = (-1.0 + k / 128.0).astype(np.float16)
        assert np.array_equal(x.astype(np.float64), -1.0 + k / 128.0)
        codes, s, b = oracle.quantize_group(x, bits=8)
        assert np.uint16(s).view(np.float16) == np.float16(1 / 128) and np.uint16(b).view(np.float16) == -1
        assert np.array_equal(codes, k)
    # exact midpoints k + 0.5 round to the even neighbour
    half = np.array([0.5, 1.5, 2.5, 100.5, 101.5, 253.5, 254.5])
    k = np.concatenate([[0, 255], half, np.full(64 - 2 - half.size, 9)])
    x = (-1.0 + k / 128.0).astype(np.float16)
    assert np.array_equal(x.astype(np.float64), -1.0 + k / 128.0)
    codes, _, _ = oracle.quantize_group(x, bits=8)
    assert list(codes[2:2 + half.size]) == [0, 2, 2, 100, 102, 254, 254]


def test_int8_round_trip_bound_and_ends():
    rng = np.random.default_rng(31)
    xs = _random_groups(rng, 2000)
    codes, sc, bi = oracle.quantize_rows(xs, bits=8)
    assert codes.shape == xs.shape                                   # one byte per code
    xh = oracle.dequantize_rows(codes, sc, bi, bits=8)
    x = xs.astype(np.float64)
    s = sc.view(np.float16).astype(np.float64)[:, 0]
    mn, mx = x.min(axis=1), x.max(axis=1)
    exact = (mx - mn) / 255.0
    assert np.all(np.abs(s - exact) <= np.maximum(exact * 2.0**-11, 2.0**-25) * (1 + 1e-9))
    # half a step, plus what the scale's own rounding costs the top codes
    # (255 |s - (max - min)/255|: large only for subnormal fp16 scales, where
    # codes past 255 clamp)
    assert np.all(np.abs(x - xh) <= (s * (0.5 + 1e-5) + 255 * np.abs(s - exact))[:, None] * (1 + 1e-9))
    assert np.all(np.abs(x - xh)[s >= 2.0**-14] <= s[s >= 2.0**-14, None] * 0.63)
    rows = np.arange(xs.shape[0])
    assert np.all(codes[rows, x.argmin(axis=1)] == 0)
    normal = s >= 2.0**-14                                            # subnormal scales may clamp below 255
    assert np.all(codes[rows, x.argmax(axis=1)][normal] == 255)
    # int8 error is about 17x below int4 on the same groups
    c4, s4, b4 = oracle.quantize_rows(xs)
    e4 = np.abs(x - oracle.dequantize_rows(c4, s4, b4)).mean()
    assert np.abs(x - xh).mean() < e4 / 10


def test_int8_attention_closed_forms():
    rng = np.random.default_rng(32)
    q = rng.standard_normal((1, 4, 64)).astype(np.float16)
    k = rng.standard_normal((1, 2, 5, 64)).astype(np.float16)
    v = rng.standard_normal((1, 2, 5, 64)).astype(np.float16)
    c = oracle.Cache.from_fp16(k, v, bits=8)
    vh = oracle.dequantize_rows(c.vc, c.vs, c.vb, bits=8)
    out = oracle.attention(q, c, np.array([1], np.int32), 0.3)      # one token: the value itself
    assert np.allclose(out[0, :2], vh[0, 0, 0], atol=1e-12) and np.allclose(out[0, 2:], vh[0, 1, 0], atol=1e-12)
    out0 = oracle.attention(q, c, np.array([5], np.int32), 0.0)     # attn_scale 0: the mean value
    assert np.allclose(out0[0, 0], vh[0, 0].mean(axis=0), atol=1e-12)


def test_dequantize_f16_int8_pins():
    """The fp16 expansion of int8 codes: grid values exact, half an fp16 ulp of
    the exact value otherwise."""
    k = np.concatenate([[0, 255], np.arange(1, 63)])
    x = (-1.0 + k / 128.0).astype(np.float16)
    c, sc, bi = oracle.quantize_rows(x.reshape(1, 64), bits=8)
    assert np.array_equal(oracle.dequantize_rows_f16(c, sc, bi, bits=8).view(np.float16).ravel(), x)
    rng = np.random.default_rng(33)
    xs = _random_groups(rng, 500)
    c, sc, bi = oracle.quantize_rows(xs, bits=8)
    got = oracle.dequantize_rows_f16(c, sc, bi, bits=8).view(np.float16).astype(np.float64)
    exact = oracle.dequantize_rows(c, sc, bi, bits=8)
    assert np.all(np.abs(got - exact) <= 0.5 * _ulp16(np.maximum(np.abs(got), np.abs(exact))) +
                  np.abs(exact) * 2.0**-24)
