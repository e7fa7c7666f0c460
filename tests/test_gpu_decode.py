"""GPU fused int4 decode attention vs the fp64 CPU oracle.

Bar: output within 2e-3 max-abs and 1e-3 relative L2 of fp64 attention over
the dequantised cache (fp32 accumulation on the GPU, fp16 output).  The GPU
side quantizes with its own kernel; the oracle quantizes the same fp16 inputs
itself.
"""
import math

import numpy as np
import pytest

import oracle
from int4_kv_cache_gb300 import synth
from tests.gpu_helpers import (ATOL, assert_close, decode, gpu_cache_from_fp16, gpu_cache_from_oracle, identity_paged,
                               need_gpu, workspace_for)

pytestmark = pytest.mark.gpu

IMPLS = [1, 2]  # TQ_IMPL_MMA, TQ_IMPL_SIMT


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("name", ["tiny", "llama70b_1k", "gemma_33", "gemma_423", "gemma_786", "gemma_950"])
def test_decode_matches_oracle(name, impl):
    need_gpu()
    w = synth.WORKLOADS[name]
    x = w.draw()
    cache = gpu_cache_from_fp16(x.k, x.v)
    out = decode(cache, x.q, x.lens, int(x.lens.max()), w.attn_scale, impl=impl)
    ref = oracle.attention(x.q, oracle.Cache.from_fp16(x.k, x.v), x.lens, w.attn_scale)
    assert_close(out, ref, what=f"{name}/impl{impl}")


@pytest.mark.parametrize("impl", IMPLS)
def test_decode_llama_16k_all_heads(impl):
    need_gpu()
    w = synth.WORKLOADS["llama70b_16k"]
    x = w.draw()
    cache = gpu_cache_from_fp16(x.k, x.v)
    out = decode(cache, x.q, x.lens, w.seq_len, w.attn_scale, impl=impl)
    ref = oracle.attention(x.q, oracle.Cache.from_fp16(x.k, x.v), x.lens, w.attn_scale)
    assert_close(out, ref, what=f"llama16k/impl{impl}")


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("D,Hq,Hkv", [(128, 8, 2), (64, 8, 8), (256, 16, 2), (128, 8, 1)])
def test_ragged_lengths_and_tails(D, Hq, Hkv, impl):
    """Lengths that are not multiples of 16 / 64 / 512, a zero-length
    sequence, a single-token sequence, and the capacity itself, at several
    chunk sizes (split-K invariance)."""
    need_gpu()
    lens = np.array([0, 1, 17, 511, 513, 1000, 1024, 1040], dtype=np.int32)
    x = synth.decode_inputs(31 + D, len(lens), Hq, Hkv, D, 1040, lens=lens)
    cache = gpu_cache_from_fp16(x.k, x.v)
    a = 1 / math.sqrt(D)
    ref = oracle.attention(x.q, oracle.Cache.from_fp16(x.k, x.v), lens, a)
    for chunk in (16, 64, 512, 2048):
        out = decode(cache, x.q, lens, int(lens.max()), a, chunk=chunk, impl=impl)
        assert np.all(out[0] == 0.0)  # empty sequence -> zero row
        assert_close(out, ref, what=f"D{D} chunk{chunk} impl{impl}")


@pytest.mark.parametrize("B,pattern", [(2, "equal"), (64, "ties"), (128, "ties"), (129, "random"),
                                       (200, "random"), (37, "zeros"), (1500, "random")])
def test_batch_order_and_empty_runs(B, pattern):
    """Batches whose grid spans several waves (here B >= 128) are dispatched
    longest run first in an order the device computes from the lengths: every
    run still lands in its own sequence's output, for equal lengths, many ties
    and empty sequences; smaller batches keep the grid order."""
    need_gpu()
    S = 300
    rng = np.random.default_rng(B)
    if pattern == "equal":
        lens = np.full(B, S, np.int32)
    elif pattern == "ties":
        lens = rng.choice(np.array([0, 1, 129, S], np.int32), size=B)
    elif pattern == "zeros":
        lens = np.where(rng.random(B) < 0.5, 0, rng.integers(1, S + 1, B)).astype(np.int32)
    else:
        lens = rng.integers(0, S + 1, B).astype(np.int32)
    lens[rng.integers(0, B)] = S
    x = synth.decode_inputs(500 + B, B, 8, 2, 64, S, lens=lens)
    cache = gpu_cache_from_fp16(x.k, x.v)
    a = 1 / math.sqrt(64)
    out = decode(cache, x.q, lens, S, a, chunk=64)
    assert np.all(out[lens == 0] == 0.0)
    assert_close(out, oracle.attention(x.q, oracle.Cache.from_fp16(x.k, x.v), lens, a), what=f"B{B} {pattern}")


def test_batch_order_paged_equals_contiguous():
    """The dispatch order with a paged cache: the same output as the same rows
    with the pages in order bit for bit, the contiguous cache's and the
    oracle's within the tolerance."""
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    B, Hq, Hkv, D, S, P = 160, 8, 2, 128, 384, 128
    rng = np.random.default_rng(11)
    lens = rng.integers(0, S + 1, B).astype(np.int32)
    lens[3] = S
    x = synth.decode_inputs(611, B, Hq, Hkv, D, S, lens=lens)
    cont = gpu_cache_from_fp16(x.k, x.v)
    per = S // P
    paged = tq.PagedKVCache(B, Hkv, D, P, B * per, per)
    perm = rng.permutation(B * per).astype(np.int32).reshape(B, per)
    paged.block_table.copy_(torch.from_numpy(perm))
    tq.tq_quantize_kv_append(paged, torch.from_numpy(x.k).cuda(), torch.from_numpy(x.v).cuda(),
                             torch.zeros(B, dtype=torch.int32, device="cuda"))
    q, lt = torch.from_numpy(x.q).cuda(), torch.from_numpy(lens).cuda()
    ws = workspace_for(B, Hq, Hkv, D, S)
    a = 1 / math.sqrt(D)
    out_c = tq.tq_sdpa_int4_decode(cont, q, lt, S, a, ws).float().cpu().numpy()
    out_p = tq.tq_sdpa_int4_decode(paged, q, lt, S, a, ws).float().cpu().numpy()
    out_i = tq.tq_sdpa_int4_decode(identity_paged(tq, torch, paged, P), q, lt, S, a, ws).float().cpu().numpy()
    assert np.array_equal(out_p, out_i)
    assert_close(out_p, out_c, what="ordered paged vs contiguous")
    assert_close(out_c, oracle.attention(x.q, oracle.Cache.from_fp16(x.k, x.v), lens, a), what="ordered paged")


@pytest.mark.parametrize("impl", IMPLS)
def test_oracle_quantised_cache_decode(impl):
    """Decode over a cache the oracle quantized (isolates attention from the
    quantize kernel)."""
    need_gpu()
    w = synth.WORKLOADS["llama70b_1k"]
    x = w.draw()
    oc = oracle.Cache.from_fp16(x.k, x.v)
    cache = gpu_cache_from_oracle(oc)
    out = decode(cache, x.q, x.lens, int(x.lens.max()), w.attn_scale, impl=impl)
    assert_close(out, oracle.attention(x.q, oc, x.lens, w.attn_scale), what="oracle cache")


@pytest.mark.parametrize("impl", IMPLS)
def test_single_token_gives_value(impl):
    need_gpu()
    x = synth.decode_inputs(5, 2, 16, 2, 128, 1)
    cache = gpu_cache_from_fp16(x.k, x.v)
    out = decode(cache, x.q, x.lens, 1, 0.3, impl=impl)
    oc = oracle.Cache.from_fp16(x.k, x.v)
    vh = oracle.dequantize_rows(oc.vc, oc.vs, oc.vb)
    for h in range(16):
        np.testing.assert_allclose(out[:, h], vh[:, h // 8, 0], atol=ATOL, rtol=0)


@pytest.mark.parametrize("impl", IMPLS)
def test_needles_at_chunk_edges(impl):
    """One key per KV head aligned with its group's first query (score margin
    >= 30): that head's output is the needle's value.  Placed at 0, 15/16,
    511/512 and S-1."""
    need_gpu()
    B, Hq, Hkv, D, S = 1, 8, 2, 128, 1536
    rng = np.random.default_rng(21)
    q = rng.choice([-1.0, 1.0], size=(B, Hq, D)).astype(np.float16)
    k = (rng.standard_normal((B, Hkv, S, D)) * 0.02).astype(np.float16)
    v = rng.standard_normal((B, Hkv, S, D)).astype(np.float16)
    for pos in (0, 15, 16, 511, 512, S - 1):
        kk = k.copy()
        for h in range(Hkv):
            kk[0, h, pos] = q[0, h * (Hq // Hkv)]
        cache = gpu_cache_from_fp16(kk, v)
        out = decode(cache, q, [S], S, 1.0, impl=impl)
        oc = oracle.Cache.from_fp16(kk, v)
        ref = oracle.attention(q, oc, np.array([S]), 1.0)
        assert_close(out, ref, what=f"needle@{pos}")
        vh = oracle.dequantize_rows(oc.vc, oc.vs, oc.vb)
        for h in range(Hkv):
            np.testing.assert_allclose(out[0, h * (Hq // Hkv)], vh[0, h, pos], atol=ATOL)


def test_partials_match_oracle_chunks():
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    lens = np.array([700, 1100], dtype=np.int32)
    x = synth.decode_inputs(41, 2, 16, 2, 128, 1100, lens=lens, outliers=True)
    cache = gpu_cache_from_fp16(x.k, x.v)
    oc = oracle.Cache.from_fp16(x.k, x.v)
    a = 1 / math.sqrt(128)
    for chunk in (64, 512):
        om, ol, oa = oracle.attention_partials(x.q, oc, lens, a, chunk)
        for impl in IMPLS:
            m, l, acc = tq.tq_sdpa_int4_partial(cache, torch.from_numpy(x.q).cuda(), torch.from_numpy(lens).cuda(),
                                                1100, a, chunk=chunk, chunks_per_split=1, impl=impl)
            torch.cuda.synchronize()
            m, l, acc = m.cpu().numpy(), l.cpu().numpy(), acc.cpu().numpy()
            empty = ol == 0
            assert np.array_equal(l == 0, empty)
            assert np.all(np.isneginf(m[empty]))
            ne = ~empty
            np.testing.assert_allclose(m[ne], om[ne], rtol=1e-5, atol=1e-5)
            np.testing.assert_allclose(l[ne], ol[ne], rtol=1e-3)
            # acc / l is the attention output over that chunk
            assert_close(acc[ne] / l[ne][:, None], oa[ne] / ol[ne][:, None], what=f"chunk{chunk} impl{impl}")


@pytest.mark.parametrize("name", ["llama70b_16k", "gemma_33", "tiny"])
def test_decode_equals_partial_plan_plus_reduce(name):
    """tq_sdpa_int4_decode == phase 1 with the decode's own plan + phase 2,
    bit for bit: with the reduce (llama70b_16k: 43 runs), with one run per
    sequence (gemma_33: phase 1 writes the output itself with the reduce's
    arithmetic), and with runs merged inside a thread-block cluster (tiny: 2
    runs, the reduce's operations in the reduce's order)."""
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    w = synth.WORKLOADS[name]
    x = w.draw()
    cache = gpu_cache_from_fp16(x.k, x.v)
    q = torch.from_numpy(x.q).cuda()
    lens = torch.from_numpy(x.lens).cuda()
    full = decode(cache, x.q, x.lens, w.seq_len, w.attn_scale)
    m, l, acc = tq.tq_sdpa_int4_partial(cache, q, lens, w.seq_len, w.attn_scale, chunks_per_split=0)
    two = tq.tq_sdpa_int4_reduce(m, l, acc).float().cpu().numpy()
    assert np.array_equal(full, two.astype(np.float64))


@pytest.mark.parametrize("D,Hq,Hkv,S,bits", [(128, 64, 8, 1024, 4), (128, 16, 2, 700, 4), (256, 32, 16, 423, 4),
                                             (64, 8, 4, 900, 4), (128, 64, 8, 500, 8), (256, 32, 16, 786, 8)])
def test_cluster_merged_decode_matches_oracle(D, Hq, Hkv, S, bits):
    """Two to eight runs per (sequence, kv head) in a grid of one wave: the
    runs form one thread-block cluster and merge their states in shared
    memory, with no reduce launch.  Against the oracle, with ragged lengths
    (runs past a sequence's end are empty) and a sequence of length 0."""
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    B = 3
    lens = np.array([S, S // 3 + 5, 0], np.int32)
    x = synth.decode_inputs(400 + D + bits, B, Hq, Hkv, D, S, lens=lens, outliers=True)
    k, v = torch.from_numpy(x.k).cuda(), torch.from_numpy(x.v).cuda()
    cap = -(-S // 16) * 16
    cache = tq.KVCache(B, Hkv, D, cap, bits=bits)
    tq.tq_quantize_kv_append(cache, k, v, torch.zeros(B, dtype=torch.int32, device="cuda"))
    n_splits = tq.tq_sdpa_plan(cache, Hq, S)[0]
    assert 2 <= n_splits <= 8, n_splits
    a = 1 / math.sqrt(D)
    got = decode(cache, x.q, lens, S, a)
    oc = oracle.Cache.from_fp16(x.k, x.v, bits=bits)
    ref = oracle.attention(x.q, oc, lens, a)
    assert np.all(got[2] == 0)
    assert_close(got, ref, what=f"cluster D{D} bits{bits}")
    # the same bits as phase 1 with partial states plus the reduce
    lt = torch.from_numpy(lens).cuda()
    m, l, acc = tq.tq_sdpa_int4_partial(cache, torch.from_numpy(x.q).cuda(), lt, S, a, chunks_per_split=0)
    two = tq.tq_sdpa_int4_reduce(m, l, acc).float().cpu().numpy().astype(np.float64)
    assert np.array_equal(got, two)


def test_reduce_matches_oracle_merge():
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    rng = np.random.default_rng(8)
    B, Hq, n, D = 2, 4, 37, 128
    m = rng.normal(0, 3, (B, Hq, n)).astype(np.float32)
    l = rng.uniform(0.5, 50, (B, Hq, n)).astype(np.float32)
    acc = rng.normal(0, 5, (B, Hq, n, D)).astype(np.float32)
    l[0, 1, 5:] = 0.0
    m[0, 1, 5:] = -np.inf
    l[1, 3, :] = 0.0  # every part empty -> zero row
    m[1, 3, :] = -np.inf
    out = tq.tq_sdpa_int4_reduce(torch.from_numpy(m).cuda(), torch.from_numpy(l).cuda(), torch.from_numpy(acc).cuda())
    torch.cuda.synchronize()
    ref = oracle.merge_partials(m.astype(np.float64), l.astype(np.float64), acc.astype(np.float64))
    got = out.float().cpu().numpy()
    assert np.all(got[1, 3] == 0)
    assert np.all(np.abs(got - ref) <= 1e-3 + 1e-3 * np.abs(ref))  # fp16 output rounding


def test_determinism_and_impl_agreement():
    need_gpu()
    w = synth.WORKLOADS["llama70b_1k"]
    x = w.draw()
    cache = gpu_cache_from_fp16(x.k, x.v)
    o1 = decode(cache, x.q, x.lens, 1024, w.attn_scale, impl=1)
    o2 = decode(cache, x.q, x.lens, 1024, w.attn_scale, impl=1)
    assert np.array_equal(o1, o2)
    o3 = decode(cache, x.q, x.lens, 1024, w.attn_scale, impl=2)
    assert np.abs(o1 - o3).max() <= 2 * ATOL


def test_seq_len_beyond_bound_sets_status_and_clamps():
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    x = synth.decode_inputs(12, 2, 8, 2, 128, 64)
    cache = gpu_cache_from_fp16(x.k, x.v)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = decode(cache, x.q, [64, 64], 48, 0.1, status=st)  # lens above max_seq_len = 48
    assert int(st.item()) & tq.TQ_DEV_SEQ_LEN
    oc = oracle.Cache.from_fp16(x.k, x.v)
    assert_close(out, oracle.attention(x.q, oc, np.array([48, 48]), 0.1), what="clamped")


def test_llama_128k_full_size_sampled():
    """The headline shape at full size (one layer, 128K tokens, 64 q / 8 kv
    heads) in the launch configuration the benchmark times; the oracle
    computes a seeded sample of heads one by one."""
    need_gpu()
    w = synth.WORKLOADS["llama70b_128k"]
    q, k, v, _ = synth.torch_decode_inputs(w.seed, 1, 64, 8, 128, w.seq_len, outliers=True)
    cache = gpu_cache_from_fp16(k, v)
    lens = np.array([w.seq_len], np.int32)
    out = decode(cache, q, lens, w.seq_len, w.attn_scale)
    qh = q.cpu().numpy()
    for h in (0, 13, 27, 38, 45, 63):
        kvh = h // 8
        oc = oracle.Cache.from_fp16(np.ascontiguousarray(k[:, kvh:kvh + 1].cpu().numpy()),
                                    np.ascontiguousarray(v[:, kvh:kvh + 1].cpu().numpy()))
        ref = oracle.attention(np.ascontiguousarray(qh[:, h:h + 1]), oc, lens, w.attn_scale)
        assert_close(out[:, h:h + 1], ref, what=f"128k head {h}")


def test_ragged32_decode_step_full_size_sampled():
    """32 sequences with lengths uniform in [1K, 32K]: append one token per
    sequence at position len[b], then decode over len[b] + 1.  Sampled rows are
    checked against the oracle, which quantizes the same fp16 inputs."""
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    w = synth.WORKLOADS["ragged32"]
    lens = synth.ragged_lengths(w.seed, 32, 1024, 32768)
    q, k, v, chans = synth.torch_decode_inputs(w.seed, 32, 64, 8, 128, 32768, outliers=True)
    cache = gpu_cache_from_fp16(k, v, capacity=32768 + 16)
    kn, vn = synth.append_tokens(w.seed, 0, 32, 8, 128, 1, outliers=chans)
    tq.tq_quantize_kv_append(cache, torch.from_numpy(kn).cuda(), torch.from_numpy(vn).cuda(),
                             torch.from_numpy(lens).cuda())
    new_lens = lens + 1
    out = decode(cache, q, new_lens, int(new_lens.max()), w.attn_scale)
    qh = q.cpu().numpy()
    rng = np.random.default_rng(5)
    for b, h in zip(rng.choice(32, 6, replace=False), rng.integers(0, 64, 6)):
        kvh, L = h // 8, int(lens[b])
        kk = np.concatenate([k[b:b + 1, kvh:kvh + 1, :L].cpu().numpy(), kn[b:b + 1, kvh:kvh + 1]], axis=2)
        vv = np.concatenate([v[b:b + 1, kvh:kvh + 1, :L].cpu().numpy(), vn[b:b + 1, kvh:kvh + 1]], axis=2)
        oc = oracle.Cache.from_fp16(kk, vv)
        ref = oracle.attention(np.ascontiguousarray(qh[b:b + 1, h:h + 1]), oc, np.array([L + 1]), w.attn_scale)
        assert_close(out[b:b + 1, h:h + 1], ref, what=f"ragged b{b} h{h}")


def test_fused_step_equals_append_then_decode():
    """tq_decode_step (append, then a decode launched before the append ends)
    gives what the two calls give in order, with the appended rows at the
    start, in the middle and at the end of a CTA's run, and in a ragged batch."""
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    B, Hq, Hkv, D, S = 3, 64, 8, 128, 20000
    x = synth.decode_inputs(61, B, Hq, Hkv, D, S, outliers=True)
    pos = np.array([0, 9001, S - 2], np.int32)  # the new tokens go to rows pos[b], pos[b] + 1
    kn, vn = synth.append_tokens(61, 3, B, Hkv, D, 2, outliers=x.outlier_channels)
    lens = pos + 2
    q = torch.from_numpy(x.q).cuda()
    wp = torch.from_numpy(pos).cuda()
    lt = torch.from_numpy(lens).cuda()
    knt, vnt = torch.from_numpy(kn).cuda(), torch.from_numpy(vn).cuda()
    ws = workspace_for(B, Hq, Hkv, D, S)
    c1 = gpu_cache_from_fp16(x.k, x.v)
    tq.tq_quantize_kv_append(c1, knt, vnt, wp)
    ref = tq.tq_sdpa_int4_decode(c1, q, lt, S, 0.088, ws).float().cpu().numpy()
    c2 = gpu_cache_from_fp16(x.k, x.v)
    for _ in range(2):  # a second step rewrites the same rows: same result
        got = tq.tq_decode_step(c2, knt, vnt, wp, q, lt, S, 0.088, ws).float().cpu().numpy()
        assert np.array_equal(got, ref)
    assert torch.equal(c1.buffer, c2.buffer)
    # and against the oracle on the appended cache
    kk, vv = x.k.copy(), x.v.copy()
    for b in range(B):
        kk[b, :, pos[b]:pos[b] + 2] = kn[b]
        vv[b, :, pos[b]:pos[b] + 2] = vn[b]
    oref = oracle.attention(x.q, oracle.Cache.from_fp16(kk, vv), lens, 0.088)
    assert_close(got, oref, what="fused step")


def _run_begins(n_splits, max_len, unit=128):
    units = -(-max_len // unit)
    return [(s * units // n_splits) * unit for s in range(n_splits + 1)]


def _plan_runs(n_splits, max_run, max_len):
    """Run boundaries of a plan: its unit is the kernel's tile (384 tokens in
    the one-CTA-per-SM layout, 128 otherwise), the one whose longest run is the
    plan's."""
    for unit in (384, 128, 64):
        rb = _run_begins(n_splits, max_len, unit)
        if max(b - a for a, b in zip(rb, rb[1:])) == max_run:
            return rb
    raise AssertionError("no tile size reproduces the plan's runs")


@pytest.mark.parametrize("n_new", [1, 16, 17, 40])
def test_fused_step_rows_across_run_boundaries(n_new):
    """Up to 16 new rows per sequence are quantized by the decode kernel (each
    CTA writes the rows its run owns, then reads them); longer appends run the
    append kernel first.  Rows straddling a run boundary, at the start of the
    cache and at its end give the same cache bytes and the same output as the
    append kernel followed by the decode."""
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    B, Hq, Hkv, D, S = 3, 64, 8, 128, 20000
    x = synth.decode_inputs(71, B, Hq, Hkv, D, S, outliers=True)
    c1 = gpu_cache_from_fp16(x.k, x.v)
    ns, run = tq.tq_sdpa_plan(c1, Hq, S)
    rb = _plan_runs(ns, run, S)  # the boundaries the kernel uses
    pos = np.array([0, rb[ns // 2] - n_new // 2, S - n_new], np.int32)
    kn, vn = synth.append_tokens(71, n_new, B, Hkv, D, n_new, outliers=x.outlier_channels)
    lens = pos + n_new
    q = torch.from_numpy(x.q).cuda()
    wp, lt = torch.from_numpy(pos).cuda(), torch.from_numpy(lens).cuda()
    knt, vnt = torch.from_numpy(kn).cuda(), torch.from_numpy(vn).cuda()
    ws = workspace_for(B, Hq, Hkv, D, S)
    tq.tq_quantize_kv_append(c1, knt, vnt, wp)
    ref = tq.tq_sdpa_int4_decode(c1, q, lt, S, 0.088, ws).float().cpu().numpy()
    c2 = gpu_cache_from_fp16(x.k, x.v)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = tq.tq_decode_step(c2, knt, vnt, wp, q, lt, S, 0.088, ws, status=st).float().cpu().numpy()
    assert int(st.item()) == 0
    assert torch.equal(c1.buffer, c2.buffer)
    assert np.array_equal(got, ref)


def test_fused_step_write_pos_out_of_range():
    """A fused append whose rows would pass the capacity writes nothing and sets
    TQ_DEV_WRITE_POS; the decode over the unchanged cache still runs."""
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    B, Hq, Hkv, D, S = 2, 16, 2, 128, 1024
    x = synth.decode_inputs(73, B, Hq, Hkv, D, S)
    c = gpu_cache_from_fp16(x.k, x.v)
    before = c.buffer.clone()
    kn, vn = synth.append_tokens(73, 0, B, Hkv, D, 2)
    pos = np.array([S - 1, 5], np.int32)  # b = 0 overflows, b = 1 is in range
    lens = np.array([S, S], np.int32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = workspace_for(B, Hq, Hkv, D, S)
    got = tq.tq_decode_step(c, torch.from_numpy(kn).cuda(), torch.from_numpy(vn).cuda(),
                            torch.from_numpy(pos).cuda(), torch.from_numpy(x.q).cuda(), torch.from_numpy(lens).cuda(),
                            S, 0.088, ws, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & tq.TQ_DEV_WRITE_POS
    after = c.buffer
    # sequence 0's rows are untouched; sequence 1's rows 5, 6 were written
    ref_c = gpu_cache_from_fp16(x.k, x.v)
    kk, vv = x.k.copy(), x.v.copy()
    kk[1, :, 5:7] = kn[1]
    vv[1, :, 5:7] = vn[1]
    ref_c2 = gpu_cache_from_fp16(kk, vv)
    assert not torch.equal(before, after)
    assert torch.equal(after, ref_c2.buffer)
    oref = oracle.attention(x.q, oracle.Cache.from_fp16(kk, vv), lens, 0.088)
    assert_close(got.float().cpu().numpy(), oref, what="fused step, one row out of range")


def test_host_buffer_step_equals_device_step():
    """tq_decode_step_host (copies in, step, copy out, one call) gives the
    device-buffer step's output and cache."""
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    B, Hq, Hkv, D, S = 2, 64, 8, 128, 4096
    x = synth.decode_inputs(250, B, Hq, Hkv, D, S, outliers=True)
    kn, vn = synth.append_tokens(250, 0, B, Hkv, D, 1, outliers=x.outlier_channels)
    pos = np.array([S - 1, 1000], np.int32)
    wp, lt = torch.from_numpy(pos).cuda(), torch.from_numpy(pos + 1).cuda()
    ws = workspace_for(B, Hq, Hkv, D, S)
    c1 = gpu_cache_from_fp16(x.k, x.v)
    ref = tq.tq_decode_step(c1, torch.from_numpy(kn).cuda(), torch.from_numpy(vn).cuda(), wp,
                            torch.from_numpy(x.q).cuda(), lt, S, 0.088, ws).cpu()
    staging = torch.empty(tq.tq_host_staging_bytes(B, Hq, Hkv, D, 1), dtype=torch.uint8, device="cuda")
    for pinned in (True, False):  # mapped host memory read in place; pageable memory through the staging copies
        c2 = gpu_cache_from_fp16(x.k, x.v)
        hq, hk, hv = (torch.from_numpy(a.copy()) for a in (x.q, kn, vn))
        h_out = torch.empty((B, Hq, D), dtype=torch.float16)
        if pinned:
            hq, hk, hv, h_out = hq.pin_memory(), hk.pin_memory(), hv.pin_memory(), h_out.pin_memory()
        tq.tq_decode_step_host(c2, hk, hv, wp.clone(), hq, lt, S, 0.088, ws, staging, h_out)
        torch.cuda.synchronize()
        assert torch.equal(h_out, ref), pinned
        assert torch.equal(c1.buffer, c2.buffer), pinned
