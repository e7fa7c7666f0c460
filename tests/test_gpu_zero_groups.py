"""Groups whose elements are all zero, on every store path.  The rule takes the
group maximum as the first element holding the largest value, so when every
element is a zero the range max - min is that first element minus +0: the
stored scale is -0 when the group opens with -0 and +0 otherwise ("Fused int4
Attention for Gemma 4 31B", Background: per-group scale (max - min) / L and
bias min; the oracle's rule).  Rows of all -0 keep the case alive through the
rotation (H x of a -0 row opens with -0).  Codes, scales and biases must be
the oracle's bit for bit."""
import math

import numpy as np
import pytest

import oracle
from tests.gpu_helpers import cache_arrays, need_gpu, workspace_for

pytestmark = pytest.mark.gpu

HKV = 8


def _zero_rows(n_rows, D, seed):
    """fp16 [n_rows, D]: a mix of all -0 rows, rows of all-zero groups with the
    first element -0 or +0 and the other signs random, and random rows with
    some groups zeroed."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n_rows, D)).astype(np.float16)
    kind = rng.integers(0, 4, n_rows)
    neg0 = np.float16(-0.0)
    for r in range(n_rows):
        if kind[r] == 0:
            x[r] = neg0
        elif kind[r] == 1:
            x[r] = np.where(rng.random(D) < 0.5, neg0, np.float16(0.0))
            x[r, ::64] = neg0 if rng.random() < 0.5 else np.float16(0.0)
        elif kind[r] == 2:
            g = rng.integers(0, D // 64)
            x[r, 64 * g: 64 * g + 64] = np.where(rng.random(64) < 0.5, neg0, np.float16(0.0))
    return x


def _rows(B, n, D, seed):
    k = _zero_rows(B * HKV * n, D, seed).reshape(B, HKV, n, D)
    v = _zero_rows(B * HKV * n, D, seed + 1).reshape(B, HKV, n, D)
    return k, v


def _check(cache, rows_k, rows_v, pos, bits, flags):
    n, D = rows_k.shape[2], rows_k.shape[3]
    got = cache_arrays(cache)
    for which, rows in ((0, rows_k), (1, rows_v)):
        src = oracle.rotate_rows_f16(rows) if flags & (1 << which) else rows
        wc, ws, wb = oracle.quantize_rows(src, 64, bits)
        gc, gs, gb = got[3 * which: 3 * which + 3]
        for b in range(rows.shape[0]):
            sl = slice(int(pos[b]), int(pos[b]) + n)
            assert np.array_equal(gs[b, :, sl], ws[b]), (which, b, "scale")
            assert np.array_equal(gb[b, :, sl], wb[b]), (which, b, "bias")
            assert np.array_equal(gc[b, :, sl], wc[b]), (which, b, "codes")


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("flags", [0, 1, 3])
@pytest.mark.parametrize("n", [8, 600])  # one-thread kernel; persistent TMA kernel
@pytest.mark.parametrize("D", [64, 128, 256])
def test_append_zero_groups(D, n, flags, bits):
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    if bits == 8 and flags == 1:
        pytest.skip("one rotated tensor is exercised on the int4 cache")
    B = 2
    k, v = _rows(B, n, D, seed=7 * n + D + bits + flags)
    cap = -(-(n + 40) // 16) * 16
    cache = tq.KVCache(B, HKV, D, cap, bits=bits)
    pos = np.array([5, 33], np.int32)
    tq.tq_quantize_kv_append(cache, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                             torch.from_numpy(pos).cuda(), flags=flags)
    torch.cuda.synchronize()
    _check(cache, k, v, pos, bits, flags)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("B,S", [(2, 4096), (1, 40000)])  # several CTAs per SM; one 12-warp CTA per SM
@pytest.mark.parametrize("flags", [0, 3])
def test_fused_step_zero_groups(bits, B, S, flags):
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    D, n = 128, 16
    k, v = _rows(B, n, D, seed=S + bits + flags)
    cache = tq.KVCache(B, HKV, D, S, bits=bits)
    pos = np.array([S - n, S // 2 + 5][:B], np.int32)
    rng = np.random.default_rng(5)
    q = torch.from_numpy(rng.standard_normal((B, 64, D)).astype(np.float16)).cuda()
    lens = torch.from_numpy(pos + n).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tq.tq_decode_step(cache, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), torch.from_numpy(pos).cuda(),
                      q, lens, S, 1 / math.sqrt(D), workspace_for(B, 64, HKV, D, S), status=st, flags=flags)
    torch.cuda.synchronize()
    assert st.item() == 0
    _check(cache, k, v, pos, bits, flags)
