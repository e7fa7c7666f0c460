"""Quantizer near-ties on the GPU: rows made of groups whose elements sit on or
within two binary32 ulps of a code boundary (tests/near_ties.py), stored by
every append path, must be the oracle's codes, scales and biases bit for bit
("Fused int4 Attention for Gemma 4 31B", Background: per-group scale + bias;
rounding half to even).  Paths: the one-thread append kernel, the persistent
TMA append kernel (8,192 groups or more), the decode step's own append in
phase 1 (in both SM layouts of the decode kernel), the rotated appends
(keys and values stored as quantize(H x)), int4 and int8."""
import math

import numpy as np
import pytest

import oracle
from tests.gpu_helpers import cache_arrays, need_gpu, workspace_for
from tests.near_ties import tie_rows

pytestmark = pytest.mark.gpu

HKV, D = 8, 128


def _rows(B, n, bits, seed):
    k = tie_rows(B * HKV * n, D, bits, seed).reshape(B, HKV, n, D)
    v = tie_rows(B * HKV * n, D, bits, seed + 7).reshape(B, HKV, n, D)
    return k, v


def _check(cache, rows_k, rows_v, pos, bits, flags=0):
    n = rows_k.shape[2]
    got = cache_arrays(cache)
    for which, rows in ((0, rows_k), (1, rows_v)):
        src = oracle.rotate_rows_f16(rows) if flags & (1 << which) else rows
        wc, ws, wb = oracle.quantize_rows(src, 64, bits)
        gc, gs, gb = got[3 * which: 3 * which + 3]
        for b in range(rows.shape[0]):
            sl = slice(int(pos[b]), int(pos[b]) + n)
            assert np.array_equal(gc[b, :, sl], wc[b]), (which, b)
            assert np.array_equal(gs[b, :, sl], ws[b]), (which, b)
            assert np.array_equal(gb[b, :, sl], wb[b]), (which, b)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("flags", [0, 3])
@pytest.mark.parametrize("n", [8, 600])  # one-thread kernel; persistent TMA kernel
def test_append_kernels_near_ties(bits, flags, n):
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    if bits == 8 and flags:
        pytest.skip("rotation is exercised on the int4 cache")
    B = 2
    k, v = _rows(B, n, bits, seed=11 * n + bits)
    cap = -(-(n + 40) // 16) * 16
    cache = tq.KVCache(B, HKV, D, cap, bits=bits)
    pos = np.array([3, 40], np.int32)
    tq.tq_quantize_kv_append(cache, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                             torch.from_numpy(pos).cuda(), flags=flags)
    torch.cuda.synchronize()
    _check(cache, k, v, pos, bits, flags)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("B,S", [(2, 4096), (1, 40000)])  # several CTAs per SM; one 12-warp CTA per SM
@pytest.mark.parametrize("flags", [0, 3])
def test_fused_step_near_ties(bits, B, S, flags):
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    if bits == 8 and flags:
        pytest.skip("rotation is exercised on the int4 cache")
    n = 16  # the most rows a step appends inside phase 1
    k, v = _rows(B, n, bits, seed=101 + S + bits)
    cache = tq.KVCache(B, HKV, D, S, bits=bits)
    pos = np.array([S - n, S // 2 + 5][:B], np.int32)
    rng = np.random.default_rng(3)
    q = torch.from_numpy(rng.standard_normal((B, 64, D)).astype(np.float16)).cuda()
    lens = torch.from_numpy(pos + n).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tq.tq_decode_step(cache, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), torch.from_numpy(pos).cuda(),
                      q, lens, S, 1 / math.sqrt(D), workspace_for(B, 64, HKV, D, S), status=st, flags=flags)
    torch.cuda.synchronize()
    assert st.item() == 0
    _check(cache, k, v, pos, bits, flags)
