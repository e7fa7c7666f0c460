"""Caches past 2^31 and 2^32 bytes.  A long context fills a large cache (the
"turboquant-llama3.170B" README's memory table: 80 layers x 8 KV heads at up
to 128K tokens, and longer contexts beyond it), and every kernel addresses a
row as (sequence x kv heads + head) x capacity + token, or through a page
index, so the byte offsets of the later sequences, heads and pages pass 2^31,
and those of the V arrays 2^32.  The caches here are sized so that
the rows a test writes and reads sit there: sequence 1 starts at code byte
2^31 of K, and V's codes start past 2^32.  Only short prefixes and the last
rows of the capacity are written (the rest of the allocation is never
touched), so the oracle stays cheap.  Codes, scales and biases must equal the
oracle's bit for bit; decodes match the oracle within the bar."""
import math

import numpy as np
import pytest

import oracle
from int4_kv_cache_gb300 import synth
from tests.gpu_helpers import assert_close, need_gpu, workspace_for

pytestmark = pytest.mark.gpu

HQ, HKV, D = 64, 8, 128
ATTN = 1 / math.sqrt(D)


def _rows(cache, b, lo, hi):
    """Codes, scale bits and bias bits of rows [lo, hi) of sequence b (all kv
    heads) of a contiguous cache, read from the device slice by slice."""
    out = []
    for t in (cache.k_codes, cache.k_scale, cache.k_bias, cache.v_codes, cache.v_scale, cache.v_bias):
        a = t[b, :, lo:hi].cpu().numpy()
        out.append(a.view(np.uint16) if a.dtype == np.float16 else a)
    return out


def _check_rows(got, k, v, bits):
    """got: _rows() of one sequence; k, v: that sequence's fp16 rows [Hkv, n, D]."""
    for which, x in ((0, k), (1, v)):
        wc, ws, wb = oracle.quantize_rows(x, 64, bits)
        gc, gs, gb = got[3 * which: 3 * which + 3]
        assert np.array_equal(gs, ws), ("scale", which)
        assert np.array_equal(gb, wb), ("bias", which)
        assert np.array_equal(gc, wc), ("codes", which)


@pytest.mark.parametrize("bits,cap", [(4, 1 << 22), (8, 1 << 21)])
def test_contiguous_cache_past_4gib(bits, cap):
    """Two sequences of 2^22 (int4) or 2^21 (int8) tokens x 8 kv heads: about
    9 GB, sequence 1 from K code byte 2^31 on.  The prefill append (TMA path)
    of both prefixes and of the last rows of the capacity, the decode, the
    fused one-row step and the dequantisation, all against the oracle."""
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    B, S = 2, 3000
    cw = D * bits // 8
    assert HKV * cap * cw == 1 << 31  # sequence 1's first K code byte
    x = synth.decode_inputs(811 + bits, B, HQ, HKV, D, S, lens=np.array([S, S - 500], np.int32), outliers=True)
    cache = tq.KVCache(B, HKV, D, cap, bits=bits)
    assert cache.nbytes > 1 << 33
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")

    # prefixes [0, S) of both sequences, then the last n_end rows of the capacity
    tq.tq_quantize_kv_append(cache, dev(x.k), dev(x.v), torch.zeros(B, dtype=torch.int32, device="cuda"), status=st)
    n_end = 700
    ke, ve = synth.append_tokens(812 + bits, 5, B, HKV, D, n_end, outliers=x.outlier_channels)
    tq.tq_quantize_kv_append(cache, dev(ke), dev(ve), torch.full((B,), cap - n_end, dtype=torch.int32, device="cuda"),
                             status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    for b in range(B):
        _check_rows(_rows(cache, b, 0, S), x.k[b], x.v[b], bits)
        _check_rows(_rows(cache, b, cap - n_end, cap), ke[b], ve[b], bits)

    # decode over the prefixes (ragged), against the oracle's own cache
    oc = oracle.Cache.from_fp16(x.k, x.v, bits=bits)
    q, lt = dev(x.q), dev(x.lens)
    out = tq.tq_sdpa_int4_decode(cache, q, lt, S, ATTN, workspace_for(B, HQ, HKV, D, S), status=st)
    got = out.float().cpu().numpy().astype(np.float64)
    assert st.item() == 0
    assert_close(got, oracle.attention(x.q, oc, x.lens, ATTN), what=f"decode int{bits}")

    # dequantisation of the prefixes (before the step below rewrites a row of sequence 1)
    k16, v16 = tq.tq_dequantize_kv(cache, S)
    assert np.array_equal(k16.cpu().numpy().view(np.uint16),
                          oracle.dequantize_rows_f16(oc.kc, oc.ks, oc.kb, bits=bits))
    assert np.array_equal(v16.cpu().numpy().view(np.uint16),
                          oracle.dequantize_rows_f16(oc.vc, oc.vs, oc.vb, bits=bits))

    # the fused step: one new row per sequence at its length, then the decode
    kn, vn = synth.append_tokens(813 + bits, 6, B, HKV, D, 1, outliers=x.outlier_channels)
    pos = x.lens.copy()
    lens = pos + 1
    got = tq.tq_decode_step(cache, dev(kn), dev(vn), dev(pos), q, dev(lens), S + 1, ATTN,
                            workspace_for(B, HQ, HKV, D, S + 1), status=st).float().cpu().numpy()
    assert st.item() == 0
    kk = np.concatenate([x.k, np.zeros((B, HKV, 1, D), np.float16)], axis=2)
    vv = np.concatenate([x.v, np.zeros((B, HKV, 1, D), np.float16)], axis=2)
    for b in range(B):
        kk[b, :, pos[b]] = kn[b, :, 0]
        vv[b, :, pos[b]] = vn[b, :, 0]
        _check_rows(_rows(cache, b, pos[b], pos[b] + 1), kn[b], vn[b], bits)
    assert_close(got.astype(np.float64), oracle.attention(x.q, oracle.Cache.from_fp16(kk, vv, bits=bits), lens, ATTN),
                 what=f"fused step int{bits}")

    del cache
    torch.cuda.empty_cache()


def test_paged_pool_past_4gib():
    """A page pool of 33,024 pages of 128 tokens (about 4.9 GB): the two
    sequences' pages are taken from page 32,768 on, where K codes start at
    byte 2^31 and V codes lie past 2^32.  Append (small and prefill paths),
    the fused step and the decode against the oracle."""
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    B, S, P = 2, 3000, 128
    num_pages, per = 33024, 32
    assert 32768 * HKV * P * (D // 2) == 1 << 31
    paged = tq.PagedKVCache(B, HKV, D, P, num_pages, per)
    assert paged.buffer.numel() > 1 << 32
    rng = np.random.default_rng(77)
    table = (32768 + rng.permutation(num_pages - 32768)[: B * per]).reshape(B, per).astype(np.int32)
    paged.block_table.copy_(torch.from_numpy(table))
    x = synth.decode_inputs(815, B, HQ, HKV, D, S, lens=np.array([S - 1, 1700], np.int32), outliers=True)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    zero = torch.zeros(B, dtype=torch.int32, device="cuda")
    tq.tq_quantize_kv_append(paged, dev(x.k[:, :, :S - 8]), dev(x.v[:, :, :S - 8]), zero, status=st)  # prefill
    tq.tq_quantize_kv_append(paged, dev(x.k[:, :, S - 8:]), dev(x.v[:, :, S - 8:]),
                             torch.full((B,), S - 8, dtype=torch.int32, device="cuda"), status=st)  # a short append
    torch.cuda.synchronize()
    assert st.item() == 0
    # sampled rows (both append paths), read through the block table
    want = (oracle.quantize_rows(x.k, 64, 4), oracle.quantize_rows(x.v, 64, 4))
    for b in range(B):
        for t in (0, 129, 1700, S - 9, S - 8, S - 1):
            pg, r = int(table[b, t // P]), t % P
            for which, arrays in ((0, (paged.k_codes, paged.k_scale, paged.k_bias)),
                                  (1, (paged.v_codes, paged.v_scale, paged.v_bias))):
                for a, w in zip(arrays, want[which]):
                    g = a[pg, :, r].cpu().numpy()
                    assert np.array_equal(g.view(np.uint16) if g.dtype == np.float16 else g, w[b, :, t]), (b, t)

    kn, vn = synth.append_tokens(816, 7, B, HKV, D, 1, outliers=x.outlier_channels)
    pos = x.lens.copy()
    lens = pos + 1
    got = tq.tq_decode_step(paged, dev(kn), dev(vn), dev(pos), dev(x.q), dev(lens), S, ATTN,
                            workspace_for(B, HQ, HKV, D, S), status=st).float().cpu().numpy()
    assert st.item() == 0
    kk, vv = x.k.copy(), x.v.copy()
    for b in range(B):
        kk[b, :, pos[b]] = kn[b, :, 0]
        vv[b, :, pos[b]] = vn[b, :, 0]
    assert_close(got.astype(np.float64), oracle.attention(x.q, oracle.Cache.from_fp16(kk, vv), lens, ATTN),
                 what="paged step")
    del paged
    torch.cuda.empty_cache()
