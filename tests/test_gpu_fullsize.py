"""Full-size parity for exactly what the benchmark times.

* The decode step at the Llama-3.1-70B single-layer shape ("turboquant-
  llama3.170B" README, kernel latency table: 64 q / 8 kv heads, head_dim 128)
  at 64K and 128K tokens, called as the benchmark calls it: tq_decode_step
  appending the new token at row S - 1 and decoding over S rows, eagerly and
  replayed from a CUDA graph.  Every query head against the oracle, and the
  appended row bit for bit.
* The 80-layer model at 128K (the same README, memory table: 80 layers x 8
  kv heads): the 80 caches built as the benchmark builds them and one model
  step of 80 tq_decode_step calls.  Layers 0, 79 and one seeded layer are
  compared in full (every code, scale and bias bit for bit, every head of the
  output within the bar); every layer has seeded rows and its appended row
  compared bit for bit.
* The Hadamard-rotated and the int8 legs at 128K: each prefill checked in
  full and each timed step against the oracle.
* The ragged batch of 32 sequences (1K-32K tokens), contiguous and paged:
  one step as the bench's graph runs it, every head against the oracle.
"""
import math

import numpy as np
import pytest

import oracle
from int4_kv_cache_gb300 import synth
from tests.gpu_helpers import assert_close, cache_arrays, need_gpu, workspace_for

pytestmark = pytest.mark.gpu

B, HQ, HKV, D = 1, 64, 8, 128
ATTN = 1.0 / math.sqrt(128.0)
STEP_SEED = 2  # the benchmark's first layer cache and its new token


def _host(t):
    return np.ascontiguousarray(t.cpu().numpy())


def _with_row(x, row, new):
    """fp16 host copy of x [B, Hkv, S, D] with row `row` replaced by new [B, Hkv, 1, D]."""
    y = x.copy()
    y[:, :, row] = new[:, :, 0]
    return y


@pytest.mark.parametrize("S", [65536, 131072])
def test_timed_step_all_heads(S):
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    q, k, v, chans = synth.torch_decode_inputs(STEP_SEED, B, HQ, HKV, D, S, outliers=True)
    cache = tq.KVCache(B, HKV, D, S)
    tq.tq_quantize_kv_append(cache, k, v, torch.zeros(B, dtype=torch.int32, device="cuda"))
    kn, vn = synth.append_tokens(STEP_SEED, 0, B, HKV, D, 1, outliers=chans)
    knt, vnt = torch.from_numpy(kn).cuda(), torch.from_numpy(vn).cuda()
    wp = torch.full((B,), S - 1, dtype=torch.int32, device="cuda")
    lens = torch.full((B,), S, dtype=torch.int32, device="cuda")
    ws = workspace_for(B, HQ, HKV, D, S)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty((B, HQ, D), dtype=torch.float16, device="cuda")

    def step():
        tq.tq_decode_step(cache, knt, vnt, wp, q, lens, S, ATTN, ws, out=out, chunk=512, status=st)

    step()
    torch.cuda.synchronize()
    eager = _host(out).copy()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert st.item() == 0
    assert np.array_equal(_host(out).view(np.uint16), eager.view(np.uint16))
    # the appended row, bit for bit
    for new, codes, scale, bias in ((kn, cache.k_codes, cache.k_scale, cache.k_bias),
                                    (vn, cache.v_codes, cache.v_scale, cache.v_bias)):
        wc, ws_, wb = oracle.quantize_rows(new)
        assert np.array_equal(_host(codes[:, :, S - 1:S]), wc)
        assert np.array_equal(_host(scale[:, :, S - 1:S]).view(np.uint16), ws_)
        assert np.array_equal(_host(bias[:, :, S - 1:S]).view(np.uint16), wb)
    # every head against the oracle over the cache that now holds the new row
    kk, vv = _with_row(_host(k), S - 1, kn), _with_row(_host(v), S - 1, vn)
    del k, v
    ref = oracle.attention(_host(q), oracle.Cache.from_fp16(kk, vv), np.array([S], np.int32), ATTN)
    assert_close(eager.astype(np.float64), ref, what=f"timed step S={S}")


def test_full_model_80_layers():
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    L, S = synth.FULL_MODEL_LAYERS, synth.WORKLOADS["llama70b_128k"].seq_len
    check = sorted({0, L - 1, int(np.random.default_rng(80).integers(1, L - 1))})
    rng = np.random.default_rng(81)
    samples = {}  # layer -> (kv heads, tokens, fp16 K rows, fp16 V rows)
    full = {}     # checked layer -> host (q, k, v)
    caches, qs = [], []
    zero = torch.zeros(B, dtype=torch.int32, device="cuda")
    chans0 = None
    for layer in range(L):
        q, k, v, chans = synth.full_model_layer(layer)
        if layer == 0:
            chans0 = chans
        c = tq.KVCache(B, HKV, D, S)
        tq.tq_quantize_kv_append(c, k, v, zero)
        h = rng.integers(0, HKV, 16)
        t = rng.integers(0, S - 1, 16)
        hi, ti = torch.from_numpy(h).cuda(), torch.from_numpy(t).cuda()
        samples[layer] = (h, t, _host(k[0, hi, ti]), _host(v[0, hi, ti]))
        if layer in check:
            full[layer] = (_host(q), _host(k), _host(v))
        caches.append(c)
        qs.append(q)
        del k, v
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    kn, vn = synth.append_tokens(synth.FULL_MODEL_SEED0, 0, B, HKV, D, 1, outliers=chans0)
    knt, vnt = torch.from_numpy(kn).cuda(), torch.from_numpy(vn).cuda()
    wp = torch.full((B,), S - 1, dtype=torch.int32, device="cuda")
    lens = torch.full((B,), S, dtype=torch.int32, device="cuda")
    ws = workspace_for(B, HQ, HKV, D, S)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = [torch.empty((B, HQ, D), dtype=torch.float16, device="cuda") for _ in range(L)]

    def model_step():
        for layer in range(L):
            tq.tq_decode_step(caches[layer], knt, vnt, wp, qs[layer], lens, S, ATTN, ws, out=outs[layer], chunk=512,
                              status=st)

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        model_step()
    g.replay()
    torch.cuda.synchronize()
    assert st.item() == 0
    # every layer: seeded rows and the appended row, bit for bit
    new_k = oracle.quantize_rows(kn)
    new_v = oracle.quantize_rows(vn)
    for layer in range(L):
        c = caches[layer]
        h, t, kr, vr = samples[layer]
        for rows, want_new, codes, scale, bias in ((kr, new_k, c.k_codes, c.k_scale, c.k_bias),
                                                   (vr, new_v, c.v_codes, c.v_scale, c.v_bias)):
            wc, wsc, wb = oracle.quantize_rows(rows)
            idx_h, idx_t = torch.from_numpy(h).cuda(), torch.from_numpy(t).cuda()
            assert np.array_equal(_host(codes[0, idx_h, idx_t]), wc), layer
            assert np.array_equal(_host(scale[0, idx_h, idx_t]).view(np.uint16), wsc), layer
            assert np.array_equal(_host(bias[0, idx_h, idx_t]).view(np.uint16), wb), layer
            assert np.array_equal(_host(codes[:, :, S - 1:S]), want_new[0]), layer
            assert np.array_equal(_host(scale[:, :, S - 1:S]).view(np.uint16), want_new[1]), layer
            assert np.array_equal(_host(bias[:, :, S - 1:S]).view(np.uint16), want_new[2]), layer
    # the checked layers in full
    for layer in check:
        qh, kh, vh = full[layer]
        oc = oracle.Cache.from_fp16(_with_row(kh, S - 1, kn), _with_row(vh, S - 1, vn))
        got = cache_arrays(caches[layer])
        for g_, w_ in zip(got, (oc.kc, oc.ks, oc.kb, oc.vc, oc.vs, oc.vb)):
            assert np.array_equal(g_, w_), layer
        ref = oracle.attention(qh, oc, np.array([S], np.int32), ATTN)
        assert_close(_host(outs[layer]).astype(np.float64), ref, what=f"80-layer model, layer {layer}")


def test_rotated_timed_step_128k():
    """The bench's Hadamard-rotated leg at full size ("Running and Evaluating
    TurboQuant optimized Gemma 4", TurboQuant section: K and V stored as
    quantize(H x / sqrt(D))): the 128K prefill through the rotated TMA
    kernel, every code, scale and bias bit for bit against the oracle's
    rotate-then-quantize; then the step the bench times (flags K | V: the
    query rotated in phase 1, the new row rotated before it is quantized, the
    output rotated back by the reduce), every head against the oracle."""
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    S, flags = 131072, tq.TQ_ROTATE_K | tq.TQ_ROTATE_V
    q, k, v, chans = synth.torch_decode_inputs(STEP_SEED + 77, B, HQ, HKV, D, S, outliers=True)
    cache = tq.KVCache(B, HKV, D, S)
    tq.tq_quantize_kv_append(cache, k, v, torch.zeros(B, dtype=torch.int32, device="cuda"), flags=flags)
    torch.cuda.synchronize()
    kh, vh = _host(k), _host(v)
    del k, v
    got = cache_arrays(cache)
    for rows, arrs in ((kh, got[:3]), (vh, got[3:])):
        wc, ws_, wb = oracle.quantize_rows(oracle.rotate_rows_f16(rows))
        assert np.array_equal(arrs[0], wc)
        assert np.array_equal(arrs[1], ws_)
        assert np.array_equal(arrs[2], wb)
    kn, vn = synth.append_tokens(STEP_SEED + 77, 0, B, HKV, D, 1, outliers=chans)
    wp = torch.full((B,), S - 1, dtype=torch.int32, device="cuda")
    lens = torch.full((B,), S, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = tq.tq_decode_step(cache, torch.from_numpy(kn).cuda(), torch.from_numpy(vn).cuda(), wp, q, lens, S, ATTN,
                            workspace_for(B, HQ, HKV, D, S), chunk=512, status=st, flags=flags)
    torch.cuda.synchronize()
    assert st.item() == 0
    kk = oracle.rotate_rows_f16(_with_row(kh, S - 1, kn))
    vv = oracle.rotate_rows_f16(_with_row(vh, S - 1, vn))
    for new, codes, scale, bias in ((kk, cache.k_codes, cache.k_scale, cache.k_bias),
                                    (vv, cache.v_codes, cache.v_scale, cache.v_bias)):
        wc, ws_, wb = oracle.quantize_rows(new[:, :, S - 1:S])
        assert np.array_equal(_host(codes[:, :, S - 1:S]), wc)
        assert np.array_equal(_host(scale[:, :, S - 1:S]).view(np.uint16), ws_)
        assert np.array_equal(_host(bias[:, :, S - 1:S]).view(np.uint16), wb)
    ref = oracle.attention(oracle.rotate_rows_f16(_host(q)), oracle.Cache.from_fp16(kk, vv), np.array([S], np.int32),
                           ATTN)
    assert_close(_host(out).astype(np.float64), oracle.hadamard(ref), what="rotated timed step S=131072")


def test_int8_timed_step_128k():
    """The bench's int8 leg at full size ("Running and Evaluating TurboQuant
    optimized Gemma 4", driver flag --kv-bits 8): the 128K int8 prefill
    through the TMA kernel checked in full, then the timed step (the fused
    one-row append at S - 1 and the decode) over every head."""
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    S = 131072
    q, k, v, chans = synth.torch_decode_inputs(STEP_SEED + 90, B, HQ, HKV, D, S, outliers=True)
    cache = tq.KVCache(B, HKV, D, S, bits=8)
    tq.tq_quantize_kv_append(cache, k, v, torch.zeros(B, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    kh, vh = _host(k), _host(v)
    del k, v
    got = cache_arrays(cache)
    for rows, arrs in ((kh, got[:3]), (vh, got[3:])):
        wc, ws_, wb = oracle.quantize_rows(rows, 64, 8)
        assert np.array_equal(arrs[0], wc)
        assert np.array_equal(arrs[1], ws_)
        assert np.array_equal(arrs[2], wb)
    kn, vn = synth.append_tokens(STEP_SEED + 90, 0, B, HKV, D, 1, outliers=chans)
    wp = torch.full((B,), S - 1, dtype=torch.int32, device="cuda")
    lens = torch.full((B,), S, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = tq.tq_decode_step(cache, torch.from_numpy(kn).cuda(), torch.from_numpy(vn).cuda(), wp, q, lens, S, ATTN,
                            workspace_for(B, HQ, HKV, D, S), chunk=512, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    kk, vv = _with_row(kh, S - 1, kn), _with_row(vh, S - 1, vn)
    ref = oracle.attention(_host(q), oracle.Cache.from_fp16(kk, vv, bits=8), np.array([S], np.int32), ATTN)
    assert_close(_host(out).astype(np.float64), ref, what="int8 timed step S=131072")


@pytest.mark.parametrize("paged", [False, True])
def test_ragged_batch_step_all_heads(paged):
    """The bench's ragged leg: 32 sequences with lengths uniform in [1K, 32K]
    (Llama heads), one step as the bench's graph runs it (append one token per
    sequence at write_pos = len, decode over len + 1, lengths advanced on the
    device, the longest-first run order of a multi-wave grid), on the
    contiguous cache and on 256-token pages from a shuffled pool; every head
    of every sequence against the oracle."""
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    Bt, P, smax = 32, 256, 32768
    lens = synth.ragged_lengths(4, Bt, 1024, smax)
    cap = smax + P
    q, k, v, chans = synth.torch_decode_inputs(4, Bt, HQ, HKV, D, smax, outliers=True)
    kn, vn = synth.append_tokens(4, 0, Bt, HKV, D, 1, outliers=chans)
    zero = torch.zeros(Bt, dtype=torch.int32, device="cuda")
    if paged:
        per = [-(-(int(n) + 2) // P) for n in lens]
        pages = sum(per) + 1
        cache = tq.PagedKVCache(Bt, HKV, D, P, pages, cap // P)
        bt = np.full((Bt, cap // P), pages - 1, np.int32)  # logical pages past a sequence: one scratch page
        perm = np.random.default_rng(4).permutation(pages - 1)
        nxt = 0
        for b in range(Bt):
            bt[b, :per[b]] = perm[nxt:nxt + per[b]]
            nxt += per[b]
        cache.block_table.copy_(torch.from_numpy(bt))
    else:
        cache = tq.KVCache(Bt, HKV, D, cap)
    tq.tq_quantize_kv_append(cache, k, v, zero)
    kh, vh = _host(k), _host(v)
    del k, v
    wp = torch.from_numpy(lens.copy()).cuda()
    lt = torch.from_numpy(lens + 1).cuda()
    max_len = int(lens.max()) + 2
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = tq.tq_decode_step(cache, torch.from_numpy(kn).cuda(), torch.from_numpy(vn).cuda(), wp, q, lt, max_len, ATTN,
                            workspace_for(Bt, HQ, HKV, D, max_len), chunk=512, status=st, flags=tq.TQ_STEP_ADVANCE)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert np.array_equal(_host(wp), lens + 1) and np.array_equal(_host(lt), lens + 2)
    for b in range(Bt):  # the appended token replaces row len of each sequence
        kh[b, :, lens[b]] = kn[b, :, 0]
        vh[b, :, lens[b]] = vn[b, :, 0]
    ref = oracle.attention(_host(q), oracle.Cache.from_fp16(kh, vh), lens + 1, ATTN)
    assert_close(_host(out).astype(np.float64), ref, what=f"ragged step paged={paged}")
