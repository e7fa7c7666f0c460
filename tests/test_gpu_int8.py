"""GPU int8 cache ("Running and Evaluating TurboQuant optimized Gemma 4",
driver flags --kv-bits {4,8}) against the oracle: quantize-on-store bit for
bit (edge groups included), decode within the output tolerance, the fused and
separate appends, the paged layout and the fp16 expansion."""
import math

import numpy as np
import pytest

import oracle
from int4_kv_cache_gb300 import synth
from tests.gpu_helpers import assert_close, cache_arrays, need_gpu, workspace_for

pytestmark = pytest.mark.gpu


def _cache8(tq, torch, k, v, capacity=None):
    B, Hkv, S, D = k.shape
    c = tq.KVCache(B, Hkv, D, capacity or -(-max(S, 16) // 16) * 16, bits=8)
    c.buffer.zero_()  # rows past S are never written: keep whole-buffer comparisons meaningful
    tq.tq_quantize_kv_append(c, torch.from_numpy(np.ascontiguousarray(k)).cuda(),
                             torch.from_numpy(np.ascontiguousarray(v)).cuda(),
                             torch.zeros(B, dtype=torch.int32, device="cuda"))
    return c


@pytest.mark.parametrize("D", [64, 128, 256])
def test_int8_quantize_bit_exact_with_edge_groups(D):
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    rng = np.random.default_rng(200 + D)
    k = rng.standard_normal((2, 3, 48, D)).astype(np.float32)
    v = rng.standard_normal((2, 3, 48, D)).astype(np.float32)
    flat = k.reshape(-1, D)
    flat[0] = 1.5                                                           # degenerate
    flat[1, :] = np.tile(-1 + np.arange(64) / 128.0, D // 64)               # grid
    flat[2, :] = np.tile(-1 + np.array([0, 255, 2.5, 3.5, 100.5, 254.5] * 10 + [0, 255, 1, 2]) / 128.0, D // 64)
    flat[3] *= 1e-4                                                         # subnormal scale
    flat[4] = flat[4] * 3000 + 10000                                        # large magnitudes
    flat[5, 3] *= 20                                                        # outlier
    flat[6, :] = 0.0
    flat[6, ::3] = 301 * 2.0**-24                                           # codes past 255, clamped
    kh, vh = k.astype(np.float16), v.astype(np.float16)
    c = _cache8(tq, torch, kh, vh)
    torch.cuda.synchronize()
    got = cache_arrays(c)
    for arrs, x in ((got[:3], kh), (got[3:], vh)):
        codes, sc, bi = oracle.quantize_rows(x, bits=8)
        assert np.array_equal(arrs[0][:, :, :48], codes)
        assert np.array_equal(arrs[1][:, :, :48], sc)
        assert np.array_equal(arrs[2][:, :, :48], bi)


@pytest.mark.parametrize("name", ["llama70b_1k", "llama70b_16k"])
def test_int8_decode_matches_oracle(name):
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    w = synth.WORKLOADS[name]
    x = w.draw()
    c = _cache8(tq, torch, x.k, x.v)
    ws = workspace_for(x.q.shape[0], x.q.shape[1], x.k.shape[1], x.k.shape[3], w.seq_len)
    out = tq.tq_sdpa_int4_decode(c, torch.from_numpy(x.q).cuda(), torch.from_numpy(x.lens).cuda(), w.seq_len,
                                 w.attn_scale, ws).float().cpu().numpy()
    ref = oracle.attention(x.q, oracle.Cache.from_fp16(x.k, x.v, bits=8), x.lens, w.attn_scale)
    assert_close(out, ref, what=f"int8 {name}")


@pytest.mark.parametrize("D,Hq,Hkv", [(128, 8, 2), (64, 8, 8), (128, 8, 1), (256, 16, 2)])
def test_int8_ragged_lengths_and_chunks(D, Hq, Hkv):
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    lens = np.array([0, 1, 17, 511, 513, 1000, 1024, 1040], dtype=np.int32)
    x = synth.decode_inputs(210 + D, len(lens), Hq, Hkv, D, 1040, lens=lens)
    c = _cache8(tq, torch, x.k, x.v)
    a = 1 / math.sqrt(D)
    ref = oracle.attention(x.q, oracle.Cache.from_fp16(x.k, x.v, bits=8), lens, a)
    for chunk in (16, 512):
        ws = workspace_for(len(lens), Hq, Hkv, D, 1040, chunk)
        out = tq.tq_sdpa_int4_decode(c, torch.from_numpy(x.q).cuda(), torch.from_numpy(lens).cuda(), 1040, a, ws,
                                     chunk=chunk).float().cpu().numpy()
        assert np.all(out[0] == 0.0)
        assert_close(out, ref, what=f"int8 D{D} chunk {chunk}")


@pytest.mark.parametrize("n_new", [1, 20])
def test_int8_step_equals_append_then_decode(n_new):
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    B, Hq, Hkv, D, S = 3, 64, 8, 128, 3000
    x = synth.decode_inputs(220 + n_new, B, Hq, Hkv, D, S, outliers=True)
    kn, vn = synth.append_tokens(220, n_new, B, Hkv, D, n_new, outliers=x.outlier_channels)
    pos = np.array([0, 1500, S - n_new], np.int32)
    lens = pos + n_new
    q, wp, lt = (torch.from_numpy(a).cuda() for a in (x.q, pos, lens))
    knt, vnt = torch.from_numpy(kn).cuda(), torch.from_numpy(vn).cuda()
    ws = workspace_for(B, Hq, Hkv, D, S)
    c1 = _cache8(tq, torch, x.k, x.v, capacity=3008)
    tq.tq_quantize_kv_append(c1, knt, vnt, wp)
    ref = tq.tq_sdpa_int4_decode(c1, q, lt, S, 0.088, ws).float().cpu().numpy()
    c2 = _cache8(tq, torch, x.k, x.v, capacity=3008)
    got = tq.tq_decode_step(c2, knt, vnt, wp, q, lt, S, 0.088, ws).float().cpu().numpy()
    assert torch.equal(c1.buffer, c2.buffer)
    assert np.array_equal(got, ref)
    kk, vv = x.k.copy(), x.v.copy()
    for b in range(B):
        kk[b, :, pos[b]:pos[b] + n_new] = kn[b]
        vv[b, :, pos[b]:pos[b] + n_new] = vn[b]
    assert_close(got, oracle.attention(x.q, oracle.Cache.from_fp16(kk, vv, bits=8), lens, 0.088), what="int8 step")


def test_int8_paged_equals_contiguous():
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    B, Hq, Hkv, D, S, P = 3, 16, 2, 128, 1500, 128
    lens = np.array([1500, 129, 777], np.int32)
    x = synth.decode_inputs(230, B, Hq, Hkv, D, S, lens=lens, outliers=True)
    cont = _cache8(tq, torch, x.k, x.v, capacity=1536)
    per = -(-S // P)
    paged = tq.PagedKVCache(B, Hkv, D, P, B * per + 2, per, bits=8)
    paged.buffer.zero_()
    perm = np.random.default_rng(230).permutation(B * per + 2)[: B * per].reshape(B, per).astype(np.int32)
    paged.block_table.copy_(torch.from_numpy(perm))
    tq.tq_quantize_kv_append(paged, torch.from_numpy(x.k).cuda(), torch.from_numpy(x.v).cuda(),
                             torch.zeros(B, dtype=torch.int32, device="cuda"))
    q, lt = torch.from_numpy(x.q).cuda(), torch.from_numpy(lens).cuda()
    ws = workspace_for(B, Hq, Hkv, D, S)
    o_c = tq.tq_sdpa_int4_decode(cont, q, lt, S, 0.088, ws).float().cpu().numpy()
    o_p = tq.tq_sdpa_int4_decode(paged, q, lt, S, 0.088, ws).float().cpu().numpy()
    assert np.array_equal(o_p, o_c)
    kc = paged.k_codes.cpu().numpy()[perm].transpose(0, 2, 1, 3, 4).reshape(B, Hkv, -1, D)[:, :, :S]
    assert np.array_equal(kc, cont.k_codes[:, :, :S].cpu().numpy())


def test_int8_dequantize_bit_exact():
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    x = synth.decode_inputs(240, 2, 4, 2, 128, 700, outliers=True)
    c = _cache8(tq, torch, x.k, x.v)
    k16, v16 = tq.tq_dequantize_kv(c, 650)
    torch.cuda.synchronize()
    oc = oracle.Cache.from_fp16(x.k, x.v, bits=8)  # the oracle's own codes (the GPU's are checked equal elsewhere)
    assert np.array_equal(k16.cpu().numpy().view(np.uint16),
                          oracle.dequantize_rows_f16(oc.kc[:, :, :650], oc.ks[:, :, :650], oc.kb[:, :, :650], bits=8))
    assert np.array_equal(v16.cpu().numpy().view(np.uint16),
                          oracle.dequantize_rows_f16(oc.vc[:, :, :650], oc.vs[:, :, :650], oc.vb[:, :, :650], bits=8))


@pytest.mark.parametrize("name", ["gemma_33", "gemma_423", "gemma_786", "gemma_950"])
def test_int8_gemma_shape_matches_oracle(name):
    """int8 at head_dim 256 (two 128-byte column blocks per 256-byte row) on the
    Gemma-style unscaled-attention configs."""
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    w = synth.WORKLOADS[name]
    x = w.draw()
    c = _cache8(tq, torch, x.k, x.v)
    ws = workspace_for(x.q.shape[0], x.q.shape[1], x.k.shape[1], x.k.shape[3], w.seq_len)
    out = tq.tq_sdpa_int4_decode(c, torch.from_numpy(x.q).cuda(), torch.from_numpy(x.lens).cuda(), w.seq_len,
                                 w.attn_scale, ws).float().cpu().numpy()
    ref = oracle.attention(x.q, oracle.Cache.from_fp16(x.k, x.v, bits=8), x.lens, w.attn_scale)
    assert_close(out, ref, what=f"int8 {name}")


@pytest.mark.parametrize("paged", [False, True])
def test_int8_d256_step_stores_oracle_rows(paged):
    """The decode step with int8 head_dim 256 rows: fused append bit-exact
    with the oracle's quantiser, output within tolerance; paged too."""
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    B, Hq, Hkv, D, S, P = 2, 16, 2, 256, 1024, 128
    x = synth.decode_inputs(260 + int(paged), B, Hq, Hkv, D, S, outliers=True)
    kn, vn = synth.append_tokens(261, 0, B, Hkv, D, 2, outliers=x.outlier_channels)
    pos = np.array([S - 2, 500], np.int32)
    lens = pos + 2
    if paged:
        per = S // P
        c = tq.PagedKVCache(B, Hkv, D, P, B * per, per, bits=8)
        perm = np.random.default_rng(3).permutation(B * per).astype(np.int32).reshape(B, per)
        c.block_table.copy_(torch.from_numpy(perm))
    else:
        c = tq.KVCache(B, Hkv, D, S, bits=8)
    kh, vh = x.k.copy(), x.v.copy()
    for b in range(B):
        kh[b, :, pos[b]:] = 0
        vh[b, :, pos[b]:] = 0
    tq.tq_quantize_kv_append(c, torch.from_numpy(kh).cuda(), torch.from_numpy(vh).cuda(),
                             torch.zeros(B, dtype=torch.int32, device="cuda"))
    ws = workspace_for(B, Hq, Hkv, D, S)
    out = tq.tq_decode_step(c, torch.from_numpy(kn).cuda(), torch.from_numpy(vn).cuda(), torch.from_numpy(pos).cuda(),
                            torch.from_numpy(x.q).cuda(), torch.from_numpy(lens).cuda(), S, 1.0, ws)
    torch.cuda.synchronize()
    for b in range(B):
        kh[b, :, pos[b]:pos[b] + 2] = kn[b]
        vh[b, :, pos[b]:pos[b] + 2] = vn[b]
    want = oracle.Cache.from_fp16(kh, vh, bits=8)
    arrays = cache_arrays(c)
    if paged:
        arrays = [a[perm].transpose(0, 2, 1, 3, 4).reshape(B, Hkv, -1, a.shape[3]) for a in arrays]
    for b in range(B):
        n = lens[b]
        for g_, w_ in zip(arrays, (want.kc, want.ks, want.kb, want.vc, want.vs, want.vb)):
            assert np.array_equal(g_[b, :, :n], w_[b, :, :n])
    ref = oracle.attention(x.q, want, lens, 1.0)
    assert_close(out.float().cpu().numpy(), ref, what=f"int8 D256 step paged={paged}")


@pytest.mark.parametrize("D,Hq,Hkv", [(128, 16, 2), (256, 32, 16), (64, 8, 4)])
def test_int8_partials_match_oracle_chunks(D, Hq, Hkv):
    """Phase 1 alone on an int8 cache, one partial state per chunk ("Running and
    Evaluating TurboQuant optimized Gemma 4", --kv-bits 8; "turboquant-
    llama3.170B" README, split-K paragraph), against the oracle's per-chunk
    states (m, l, acc) with an empty chunk beyond the shorter sequence."""
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    lens = np.array([700, 1100], dtype=np.int32)
    x = synth.decode_inputs(43 + D, 2, Hq, Hkv, D, 1100, lens=lens, outliers=True)
    cache = tq.KVCache(2, Hkv, D, 1104, bits=8)
    tq.tq_quantize_kv_append(cache, torch.from_numpy(x.k).cuda(), torch.from_numpy(x.v).cuda(),
                             torch.zeros(2, dtype=torch.int32, device="cuda"))
    oc = oracle.Cache.from_fp16(x.k, x.v, bits=8)
    a = 1 / math.sqrt(D)
    for chunk in (64, 512):
        om, ol, oa = oracle.attention_partials(x.q, oc, lens, a, chunk)
        m, l, acc = tq.tq_sdpa_int4_partial(cache, torch.from_numpy(x.q).cuda(), torch.from_numpy(lens).cuda(),
                                            1100, a, chunk=chunk, chunks_per_split=1)
        torch.cuda.synchronize()
        m, l, acc = m.cpu().numpy(), l.cpu().numpy(), acc.cpu().numpy()
        empty = ol == 0
        assert empty.any()
        assert np.array_equal(l == 0, empty)
        assert np.all(np.isneginf(m[empty]))
        ne = ~empty
        np.testing.assert_allclose(m[ne], om[ne], rtol=1e-5, atol=1e-5)
        np.testing.assert_allclose(l[ne], ol[ne], rtol=1e-3)
        assert_close(acc[ne] / l[ne][:, None], oa[ne] / ol[ne][:, None], what=f"int8 D{D} chunk{chunk}")
