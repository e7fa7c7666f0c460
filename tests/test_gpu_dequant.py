"""GPU fp16 dequantisation of the int4 cache (the dequantize-then-attend
comparison path, "Fused int4 Attention for Gemma 4 31B on Apple Silicon",
What I Built Instead) against the oracle: bit-exact fp16 K/V, and attention
over them by torch's SDPA within the output tolerance of the oracle."""
import math

import numpy as np
import pytest

import oracle
from int4_kv_cache_gb300 import synth
from tests.gpu_helpers import assert_close, gpu_cache_from_fp16, need_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D,Hkv,S,n_rows", [(128, 8, 1040, 1040), (128, 2, 1040, 517), (64, 4, 96, 33),
                                            (256, 2, 512, 500)])
def test_dequantize_bit_exact(D, Hkv, S, n_rows):
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    x = synth.decode_inputs(81 + D, 2, 2 * Hkv, Hkv, D, S, outliers=True)
    cache = gpu_cache_from_fp16(x.k, x.v)
    k16, v16 = tq.tq_dequantize_kv(cache, n_rows)
    torch.cuda.synchronize()
    oc = oracle.Cache.from_fp16(x.k, x.v)  # the oracle's own codes (the GPU's are checked equal elsewhere)
    want_k = oracle.dequantize_rows_f16(oc.kc[:, :, :n_rows], oc.ks[:, :, :n_rows], oc.kb[:, :, :n_rows])
    want_v = oracle.dequantize_rows_f16(oc.vc[:, :, :n_rows], oc.vs[:, :, :n_rows], oc.vb[:, :, :n_rows])
    assert np.array_equal(k16.cpu().numpy().view(np.uint16), want_k)
    assert np.array_equal(v16.cpu().numpy().view(np.uint16), want_v)


def test_dequantize_then_sdpa_matches_oracle():
    """The comparison path end to end: dequantize, then torch SDPA with GQA,
    against fp64 attention over the same int4 cache.  Its error is that of fp16
    K/V storage (2^-12 relative per element) plus the library's fp16 softmax
    weights, so it is held to 4e-3 max-abs / 2e-3 rel-L2 -- twice the fused
    path's bar -- and the fused decode on the same inputs must stay within
    its own bar (2e-3 / 1e-3)."""
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq
    from tests.gpu_helpers import decode

    w = synth.WORKLOADS["llama70b_16k"]
    x = w.draw()
    cache = gpu_cache_from_fp16(x.k, x.v)
    k16, v16 = tq.tq_dequantize_kv(cache, w.seq_len)
    q = torch.from_numpy(x.q).cuda()
    G = q.shape[1] // k16.shape[1]
    out = torch.nn.functional.scaled_dot_product_attention(
        q.unsqueeze(2), k16.repeat_interleave(G, dim=1), v16.repeat_interleave(G, dim=1), scale=w.attn_scale)
    torch.cuda.synchronize()
    ref = oracle.attention(x.q, oracle.Cache.from_fp16(x.k, x.v), x.lens, w.attn_scale)
    base_err = assert_close(out.squeeze(2).float().cpu().numpy(), ref, atol=4e-3, rtol_l2=2e-3,
                            what="dequantize + SDPA")
    fused_err = assert_close(decode(cache, x.q, x.lens, w.seq_len, w.attn_scale), ref, what="fused decode")
    print(f"max-abs / rel-L2 vs fp64 over the int4 cache: dequantize+SDPA {base_err}, fused {fused_err}")


def test_dequantize_then_sdpa_128k_as_benchmarked():
    """The comparison leg the bench times, at its size: the 128K Llama cache
    expanded to fp16 (every element bit for bit against the oracle's
    expansion), then torch SDPA with GQA (enable_gqa, as the bench calls it)
    against fp64 attention over the int4 cache, at the comparison path's own
    bar (4e-3 / 2e-3)."""
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    S, Hq, Hkv, D = 131072, 64, 8, 128
    q, k, v, _ = synth.torch_decode_inputs(11, 1, Hq, Hkv, D, S, outliers=True)
    cache = tq.KVCache(1, Hkv, D, S)
    tq.tq_quantize_kv_append(cache, k, v, torch.zeros(1, dtype=torch.int32, device="cuda"))
    oc = oracle.Cache.from_fp16(k.cpu().numpy(), v.cpu().numpy())  # the oracle's own cache
    del k, v
    k16, v16 = tq.tq_dequantize_kv(cache, S)
    out = torch.nn.functional.scaled_dot_product_attention(q.unsqueeze(2), k16, v16, scale=1 / np.sqrt(D),
                                                           enable_gqa=True)
    torch.cuda.synchronize()
    assert np.array_equal(k16.cpu().numpy().view(np.uint16), oracle.dequantize_rows_f16(oc.kc, oc.ks, oc.kb))
    assert np.array_equal(v16.cpu().numpy().view(np.uint16), oracle.dequantize_rows_f16(oc.vc, oc.vs, oc.vb))
    ref = oracle.attention(q.cpu().numpy(), oc, np.array([S], np.int32), 1 / np.sqrt(D))
    assert_close(out.squeeze(2).float().cpu().numpy(), ref, atol=4e-3, rtol_l2=2e-3, what="dequantize + SDPA 128K")
