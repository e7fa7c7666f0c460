"""GPU paged int4 cache (block table over a page pool) against the contiguous
cache and the oracle: same bytes in the pages, a decode bit-identical to the
same rows with the pages in order (and to the contiguous cache wherever both
run the same kernel layout), fused and separate appends, a bad block-table
entry, and a CUDA-graph decode loop whose lengths advance on the device."""
import math

import numpy as np
import pytest

import oracle
from int4_kv_cache_gb300 import synth
from tests.gpu_helpers import (assert_close, gpu_cache_from_fp16, identity_paged, need_gpu, same_layout,
                               workspace_for)

pytestmark = pytest.mark.gpu


def _paged_like(tq, torch, B, Hkv, D, S, P, seed, spare=3):
    """A paged cache with ceil(S / P) pages per sequence taken from a shuffled pool."""
    per = -(-S // P)
    pages = B * per + spare
    c = tq.PagedKVCache(B, Hkv, D, P, pages, per)
    c.buffer.zero_()  # spare pages are never written: keep whole-buffer comparisons meaningful
    perm = np.random.default_rng(seed).permutation(pages)[: B * per].reshape(B, per).astype(np.int32)
    c.block_table.copy_(torch.from_numpy(perm))
    return c, perm


def _gather(paged, perm, S):
    """Paged arrays back in contiguous [B, Hkv, S, ...] order (host)."""
    out = []
    for arr in (paged.k_codes, paged.k_scale, paged.k_bias, paged.v_codes, paged.v_scale, paged.v_bias):
        a = arr.cpu().numpy()                                  # [pages, Hkv, P, w]
        g = a[perm]                                            # [B, per, Hkv, P, w]
        g = g.transpose(0, 2, 1, 3, 4).reshape(perm.shape[0], a.shape[1], -1, a.shape[3])
        out.append(g[:, :, :S])
    return out


@pytest.mark.parametrize("D,Hq,Hkv,P", [(128, 64, 8, 128), (128, 16, 2, 256), (256, 8, 2, 128), (64, 8, 4, 256),
                                        (128, 16, 2, 384), (128, 64, 8, 640), (256, 32, 16, 1152)])
def test_paged_equals_contiguous_and_oracle(D, Hq, Hkv, P):
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    B, S = 3, 2000
    lens = np.array([2000, 129, 1377], np.int32)
    x = synth.decode_inputs(140 + D, B, Hq, Hkv, D, S, lens=lens, outliers=True)
    cont = gpu_cache_from_fp16(x.k, x.v, capacity=2048)
    paged, perm = _paged_like(tq, torch, B, Hkv, D, S, P, seed=D)
    tq.tq_quantize_kv_append(paged, torch.from_numpy(x.k).cuda(), torch.from_numpy(x.v).cuda(),
                             torch.zeros(B, dtype=torch.int32, device="cuda"))
    for got, want in zip(_gather(paged, perm, S), (cont.k_codes, cont.k_scale, cont.k_bias, cont.v_codes,
                                                   cont.v_scale, cont.v_bias)):
        assert np.array_equal(got.view(np.uint8), want[:, :, :S].cpu().numpy().view(np.uint8))
    q, lt = torch.from_numpy(x.q).cuda(), torch.from_numpy(lens).cuda()
    ws = workspace_for(B, Hq, Hkv, D, S)
    a = 1 / math.sqrt(D)
    out_c = tq.tq_sdpa_int4_decode(cont, q, lt, S, a, ws).float().cpu().numpy()
    out_p = tq.tq_sdpa_int4_decode(paged, q, lt, S, a, ws).float().cpu().numpy()
    out_i = tq.tq_sdpa_int4_decode(identity_paged(tq, torch, paged, P), q, lt, S, a, ws).float().cpu().numpy()
    assert np.array_equal(out_p, out_i)
    if same_layout(D):
        assert np.array_equal(out_p, out_c)
    else:
        assert_close(out_p, out_c, what="paged vs contiguous")
    assert_close(out_p, oracle.attention(x.q, oracle.Cache.from_fp16(x.k, x.v), lens, a), what="paged decode")


@pytest.mark.parametrize("n_new", [1, 20])
def test_paged_step_equals_contiguous_step(n_new):
    """Fused (1 row) and separate (20 rows) appends land in the right pages."""
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    B, Hq, Hkv, D, S, P = 2, 64, 8, 128, 1500, 128
    x = synth.decode_inputs(150 + n_new, B, Hq, Hkv, D, S, outliers=True)
    kn, vn = synth.append_tokens(150, n_new, B, Hkv, D, n_new, outliers=x.outlier_channels)
    pos = np.array([1000, 127], np.int32)  # sequence 1 crosses a page boundary when n_new > 1
    lens = pos + n_new
    cont = gpu_cache_from_fp16(x.k, x.v, capacity=1536)
    paged, perm = _paged_like(tq, torch, B, Hkv, D, S, P, seed=n_new)
    zero = torch.zeros(B, dtype=torch.int32, device="cuda")
    tq.tq_quantize_kv_append(paged, torch.from_numpy(x.k).cuda(), torch.from_numpy(x.v).cuda(), zero)
    q, wp, lt = (torch.from_numpy(a).cuda() for a in (x.q, pos, lens))
    knt, vnt = torch.from_numpy(kn).cuda(), torch.from_numpy(vn).cuda()
    ws = workspace_for(B, Hq, Hkv, D, S)
    o_c = tq.tq_decode_step(cont, knt, vnt, wp, q, lt, S, 0.088, ws).float().cpu().numpy()
    o_p = tq.tq_decode_step(paged, knt, vnt, wp, q, lt, S, 0.088, ws).float().cpu().numpy()
    # the rows now in the pool, pages in order: the same decode bit for bit
    o_i = tq.tq_sdpa_int4_decode(identity_paged(tq, torch, paged, P), q, lt, S, 0.088, ws).float().cpu().numpy()
    assert np.array_equal(o_p, o_i)
    assert_close(o_p, o_c, what="paged step vs contiguous step")
    for got, want in zip(_gather(paged, perm, S), (cont.k_codes, cont.k_scale, cont.k_bias, cont.v_codes,
                                                   cont.v_scale, cont.v_bias)):
        assert np.array_equal(got.view(np.uint8), want[:, :, :S].cpu().numpy().view(np.uint8))


def test_bad_block_table_entry_sets_status():
    """An entry outside [0, num_pages) is reported and replaced by page 0: the
    kernels stay in bounds and finish."""
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    B, Hq, Hkv, D, S, P = 2, 8, 2, 128, 512, 128
    x = synth.decode_inputs(160, B, Hq, Hkv, D, S)
    paged, perm = _paged_like(tq, torch, B, Hkv, D, S, P, seed=160)
    zero = torch.zeros(B, dtype=torch.int32, device="cuda")
    tq.tq_quantize_kv_append(paged, torch.from_numpy(x.k).cuda(), torch.from_numpy(x.v).cuda(), zero)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    paged.block_table[1, 2] = paged.num_pages + 7
    out = tq.tq_sdpa_int4_decode(paged, torch.from_numpy(x.q).cuda(),
                                 torch.full((B,), S, dtype=torch.int32, device="cuda"), S, 0.088,
                                 workspace_for(B, Hq, Hkv, D, S), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & tq.TQ_DEV_PAGE
    assert torch.isfinite(out.float()).all()
    # sequence 0 does not touch the bad entry: its rows are exact
    lens = np.array([S, S], np.int32)
    ref = oracle.attention(x.q[:1], oracle.Cache.from_fp16(x.k[:1], x.v[:1]), lens[:1], 0.088)
    assert_close(out[:1].float().cpu().numpy(), ref, what="sequence without the bad entry")


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv", [(2, 64, 8), (160, 16, 2)])
def test_graph_captured_steps_advance_on_device(paged, B, Hq, Hkv):
    """One tq_decode_step captured in a CUDA graph with TQ_STEP_ADVANCE and
    replayed token after token (new K/V copied into the captured buffers
    between replays) gives the outputs and the cache of eager steps with
    host-advanced lengths.  The 160-sequence batch spans several waves, so
    each replay also runs the kernel that orders the runs from the lengths
    the previous replay advanced."""
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    D, S0, steps, cap = 128, 700, 6, 1024
    x = synth.decode_inputs(170 + B, B, Hq, Hkv, D, cap, outliers=True)
    toks = [synth.append_tokens(170, i, B, Hkv, D, 1, outliers=x.outlier_channels) for i in range(steps)]
    start = (np.array([S0, S0 - 300], np.int32) if B == 2
             else np.random.default_rng(B).integers(100, 1000 - steps, B).astype(np.int32))

    def make():
        if paged:
            c, _ = _paged_like(tq, torch, B, Hkv, D, cap, 128, seed=171)
        else:
            c = tq.KVCache(B, Hkv, D, cap)
        tq.tq_quantize_kv_append(c, torch.from_numpy(x.k).cuda(), torch.from_numpy(x.v).cuda(),
                                 torch.zeros(B, dtype=torch.int32, device="cuda"))
        return c

    q = torch.from_numpy(x.q).cuda()
    ws = workspace_for(B, Hq, Hkv, D, cap)
    # eager reference
    c1 = make()
    ref = []
    for i, (kn, vn) in enumerate(toks):
        wp = torch.from_numpy(start + i).cuda()
        lt = torch.from_numpy(start + i + 1).cuda()
        ref.append(tq.tq_decode_step(c1, torch.from_numpy(kn).cuda(), torch.from_numpy(vn).cuda(), wp, q, lt, cap,
                                     0.088, ws).clone())
    # graph with device-side advance
    c2 = make()
    kbuf = torch.from_numpy(toks[0][0]).cuda()
    vbuf = torch.from_numpy(toks[0][1]).cuda()
    wp = torch.from_numpy(start.copy()).cuda()
    lt = torch.from_numpy(start + 1).cuda()
    out = torch.empty_like(q)
    flags = tq.TQ_STEP_ADVANCE
    tq.tq_decode_step(c2, kbuf, vbuf, wp, q, lt, cap, 0.088, ws, out=out, flags=flags)  # step 0, eager (warm-up)
    got = [out.clone()]
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        tq.tq_decode_step(c2, kbuf, vbuf, wp, q, lt, cap, 0.088, ws, out=out, flags=flags)
    for i in range(1, steps):
        kbuf.copy_(torch.from_numpy(toks[i][0]))
        vbuf.copy_(torch.from_numpy(toks[i][1]))
        g.replay()
        got.append(out.clone())
    torch.cuda.synchronize()
    assert np.array_equal(wp.cpu().numpy(), start + steps)
    assert np.array_equal(lt.cpu().numpy(), start + steps + 1)
    for i in range(steps):
        assert torch.equal(got[i], ref[i]), i
    assert torch.equal(c1.buffer, c2.buffer)


@pytest.mark.parametrize("paged", [False, True])
def test_advance_after_separate_append(paged):
    """TQ_STEP_ADVANCE with an append long enough to run as its own kernel:
    same output as the step without the flag, lengths advanced by n_new."""
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    B, Hq, Hkv, D, S, n_new = 2, 16, 2, 128, 1024, 20
    x = synth.decode_inputs(180, B, Hq, Hkv, D, S)
    kn, vn = synth.append_tokens(180, 1, B, Hkv, D, n_new)
    pos = np.array([600, 900], np.int32)
    outs = []
    for flags in (0, tq.TQ_STEP_ADVANCE):
        if paged:
            c, _ = _paged_like(tq, torch, B, Hkv, D, S, 128, seed=181)
        else:
            c = tq.KVCache(B, Hkv, D, S)
        tq.tq_quantize_kv_append(c, torch.from_numpy(x.k).cuda(), torch.from_numpy(x.v).cuda(),
                                 torch.zeros(B, dtype=torch.int32, device="cuda"))
        wp, lt = torch.from_numpy(pos.copy()).cuda(), torch.from_numpy(pos + n_new).cuda()
        o = tq.tq_decode_step(c, torch.from_numpy(kn).cuda(), torch.from_numpy(vn).cuda(), wp,
                              torch.from_numpy(x.q).cuda(), lt, S, 0.088, workspace_for(B, Hq, Hkv, D, S),
                              flags=flags)
        outs.append(o.float().cpu().numpy())
        torch.cuda.synchronize()
        want = 1 if flags else 0
        assert np.array_equal(wp.cpu().numpy(), pos + want * n_new)
        assert np.array_equal(lt.cpu().numpy(), pos + n_new + want * n_new)
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("n_new", [1, 20])  # the append fused into phase 1; its own kernel
def test_advance_with_rotation(paged, n_new):
    """TQ_STEP_ADVANCE on a rotated cache (TQ_ROTATE_K | TQ_ROTATE_V): the
    reduce both rotates the merged output and advances the lengths.  Same
    output as the step without the flag (both plan without merging), the
    rows stored the same, lengths advanced by n_new."""
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    B, Hq, Hkv, D, S = 2, 16, 2, 128, 1024
    rot = tq.TQ_ROTATE_K | tq.TQ_ROTATE_V
    x = synth.decode_inputs(185 + n_new, B, Hq, Hkv, D, S, outliers=True)
    kn, vn = synth.append_tokens(185, 2, B, Hkv, D, n_new, outliers=x.outlier_channels)
    pos = np.array([600, 1000 - n_new], np.int32)
    outs, caches = [], []
    for flags in (rot, rot | tq.TQ_STEP_ADVANCE):
        if paged:
            c, _ = _paged_like(tq, torch, B, Hkv, D, S, 128, seed=186)
        else:
            c = tq.KVCache(B, Hkv, D, S)
        tq.tq_quantize_kv_append(c, torch.from_numpy(x.k).cuda(), torch.from_numpy(x.v).cuda(),
                                 torch.zeros(B, dtype=torch.int32, device="cuda"), flags=rot)
        wp, lt = torch.from_numpy(pos.copy()).cuda(), torch.from_numpy(pos + n_new).cuda()
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        o = tq.tq_decode_step(c, torch.from_numpy(kn).cuda(), torch.from_numpy(vn).cuda(), wp,
                              torch.from_numpy(x.q).cuda(), lt, S, 0.088, workspace_for(B, Hq, Hkv, D, S),
                              status=st, flags=flags)
        outs.append(o.float().cpu().numpy())
        caches.append(c)
        torch.cuda.synchronize()
        assert st.item() == 0
        want = n_new if flags & tq.TQ_STEP_ADVANCE else 0
        assert np.array_equal(wp.cpu().numpy(), pos + want)
        assert np.array_equal(lt.cpu().numpy(), pos + n_new + want)
    assert np.array_equal(outs[0], outs[1])
    assert torch.equal(caches[0].buffer, caches[1].buffer)


@pytest.mark.parametrize("flags,D,bits", [(3, 128, 4), (1, 64, 4), (2, 256, 8)])
def test_paged_rotated_prefill_equals_oracle(flags, D, bits):
    """A rotated prefill large enough for the persistent TMA kernels, into a
    paged cache from a shuffled pool: the pages hold the oracle's codes,
    scales and biases of the rotated rows, bit for bit."""
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    B, Hkv, S, P = 2, 4, 1500, 256
    assert B * Hkv * S * (D // 64) >= 8192
    x = synth.decode_inputs(170 + D + flags, B, 2 * Hkv, Hkv, D, S, outliers=True)
    per = -(-S // P)
    pages = B * per + 3
    paged = tq.PagedKVCache(B, Hkv, D, P, pages, per, bits=bits)
    paged.buffer.zero_()
    perm = np.random.default_rng(D + flags).permutation(pages)[: B * per].reshape(B, per).astype(np.int32)
    paged.block_table.copy_(torch.from_numpy(perm))
    tq.tq_quantize_kv_append(paged, torch.from_numpy(x.k).cuda(), torch.from_numpy(x.v).cuda(),
                             torch.zeros(B, dtype=torch.int32, device="cuda"), flags=flags)
    torch.cuda.synchronize()
    kk = oracle.rotate_rows_f16(x.k) if flags & 1 else x.k
    vv = oracle.rotate_rows_f16(x.v) if flags & 2 else x.v
    got = _gather(paged, perm, S)
    for arrs, src in ((got[:3], kk), (got[3:], vv)):
        codes, sc, bi = oracle.quantize_rows(src, bits=bits)
        assert np.array_equal(arrs[0].view(np.uint8), codes)
        assert np.array_equal(arrs[1].view(np.uint16), sc)
        assert np.array_equal(arrs[2].view(np.uint16), bi)
