"""GPU quantize-on-store vs the CPU oracle: codes, scales and biases bit-exact."""
import numpy as np
import pytest

import oracle
from int4_kv_cache_gb300 import synth
from tests.gpu_helpers import cache_arrays, gpu_cache_from_fp16, need_gpu

pytestmark = pytest.mark.gpu


def _compare(cache, k, v):
    kc, ks, kb, vc, vs, vb = cache_arrays(cache)
    S = k.shape[2]
    okc, oks, okb = oracle.quantize_rows(k)
    ovc, ovs, ovb = oracle.quantize_rows(v)
    for got, want in ((kc, okc), (ks, oks), (kb, okb), (vc, ovc), (vs, ovs), (vb, ovb)):
        np.testing.assert_array_equal(got[:, :, :S], want)


@pytest.mark.parametrize("name", ["tiny", "llama70b_1k", "gemma_950", "gemma_33"])
def test_prefill_quantize_bit_exact(name):
    need_gpu()
    x = synth.WORKLOADS[name].draw()
    _compare(gpu_cache_from_fp16(x.k, x.v), x.k, x.v)


@pytest.mark.parametrize("D", [64, 128, 256])
def test_quantize_edge_groups_bit_exact(D):
    need_gpu()
    rng = np.random.default_rng(D)
    S = 48
    k = rng.standard_normal((2, 3, S, D)).astype(np.float32)
    v = rng.standard_normal((2, 3, S, D)).astype(np.float32)
    flat = k.reshape(-1, D)
    flat[0] = 1.5                                                       # degenerate groups
    flat[1, :] = np.tile(-1 + 0.125 * np.arange(16), D // 16)           # exact grid
    flat[2, :] = np.tile(-1 + 0.125 * np.array([0, 15, 2.5, 3.5, 0.5, 14.5, 7, 8] * 2), D // 16)  # ties
    flat[3] = 0.0
    flat[3, 1::7] = -0.0                                                # signed zeros at the minimum
    flat[3, 2::5] = 2.0
    flat[4] *= 1e-4                                                     # subnormal scale
    flat[5] = flat[5] * 3000 + 10000                                    # large magnitudes
    flat[6, 3] *= 20                                                    # outlier channel
    flat[7] = np.round(flat[7] * 4) / 4                                 # repeated values
    flat[8, :] = 0.0
    flat[8, 5] = 2.0**-24                                               # scale rounds to zero
    flat[9, :] = 0.0
    flat[9, ::3] = 21 * 2.0**-24                  # scale 1.4 * 2^-24 rounds to 2^-24: codes up to 21, clamped
    kh, vh = k.astype(np.float16), v.astype(np.float16)
    _compare(gpu_cache_from_fp16(kh, vh), kh, vh)


def test_append_ragged_positions_and_untouched_rows():
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    B, Hkv, D, cap = 3, 2, 128, 64
    cache = tq.KVCache(B, Hkv, D, cap)
    cache.buffer.fill_(0xA5)
    expect = [a.copy() for a in cache_arrays(cache)]
    for n_new, pos in ((1, [0, 17, 63]), (5, [3, 40, 59])):
        k, v = synth.append_tokens(9, n_new, B, Hkv, D, n_new)
        wp = torch.tensor(pos, dtype=torch.int32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        tq.tq_quantize_kv_append(cache, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), wp, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        okc, oks, okb = oracle.quantize_rows(k)
        ovc, ovs, ovb = oracle.quantize_rows(v)
        for old, ref in zip(expect, (okc, oks, okb, ovc, ovs, ovb)):
            for b in range(B):
                old[b, :, pos[b]:pos[b] + n_new] = ref[b]
        for got, want in zip(cache_arrays(cache), expect):
            np.testing.assert_array_equal(got, want)  # written rows match, nothing else changed


def test_append_out_of_range_position_sets_status_and_skips():
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    B, Hkv, D, cap = 2, 2, 64, 32
    cache = tq.KVCache(B, Hkv, D, cap)
    cache.buffer.fill_(0x5A)
    before = [a.copy() for a in cache_arrays(cache)]
    k, v = synth.append_tokens(3, 0, B, Hkv, D, 4)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    wp = torch.tensor([30, -1], dtype=torch.int32, device="cuda")  # 30 + 4 > 32, and negative
    tq.tq_quantize_kv_append(cache, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), wp, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & tq.TQ_DEV_WRITE_POS
    for arr, old in zip(cache_arrays(cache), before):
        np.testing.assert_array_equal(arr, old)


def test_prefill_full_128k_layer_bit_exact_sampled():
    """Full 128K Llama-70B-shape layer quantized on the GPU; the oracle checks a
    seeded sample of rows (every KV head, a spread of token positions)."""
    need_gpu()
    w = synth.WORKLOADS["llama70b_128k"]
    q, k, v, _ = synth.torch_decode_inputs(w.seed, w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                           w.seq_len, outliers=True)
    cache = gpu_cache_from_fp16(k, v)
    rng = np.random.default_rng(77)
    toks = np.unique(np.concatenate([rng.integers(0, w.seq_len, 2000), [0, 511, 512, w.seq_len - 1]]))
    kh = np.ascontiguousarray(k[0][:, toks].cpu().numpy())
    vh = np.ascontiguousarray(v[0][:, toks].cpu().numpy())
    okc, oks, okb = oracle.quantize_rows(kh)
    ovc, ovs, ovb = oracle.quantize_rows(vh)
    got = [a[0][:, toks] for a in cache_arrays(cache)]
    for g, want in zip(got, (okc, oks, okb, ovc, ovs, ovb)):
        np.testing.assert_array_equal(g, want)


@pytest.mark.parametrize("flags,bits,D", [(0, 4, 128), (3, 4, 128), (0, 8, 128), (1, 4, 64), (0, 4, 256),
                                          (2, 4, 256), (3, 8, 256), (3, 8, 128)])
def test_large_append_tma_path_bit_exact(flags, bits, D):
    """Appends of >= 8192 groups stream through the persistent TMA kernels:
    bit-exact against the oracle with a ragged last tile (the group count is
    not a multiple of the 256-row tile), with the rotation fused in (one or
    both tensors), and for int8."""
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    B, Hkv, S = 2, 3, 2731
    x = synth.decode_inputs(260 + D + flags, B, 2 * Hkv, Hkv, D, S, outliers=True)
    assert (B * Hkv * S * (D // 64)) % 256 != 0 and B * Hkv * S * (D // 64) >= 8192
    c = tq.KVCache(B, Hkv, D, 2736, bits=bits)
    tq.tq_quantize_kv_append(c, torch.from_numpy(x.k).cuda(), torch.from_numpy(x.v).cuda(),
                             torch.zeros(B, dtype=torch.int32, device="cuda"), flags=flags)
    torch.cuda.synchronize()
    kk = oracle.rotate_rows_f16(x.k) if flags & 1 else x.k
    vv = oracle.rotate_rows_f16(x.v) if flags & 2 else x.v
    got = cache_arrays(c)
    for arrs, src in ((got[:3], kk), (got[3:], vv)):
        codes, sc, bi = oracle.quantize_rows(src, bits=bits)
        assert np.array_equal(arrs[0][:, :, :S], codes)
        assert np.array_equal(arrs[1][:, :, :S], sc)
        assert np.array_equal(arrs[2][:, :, :S], bi)
