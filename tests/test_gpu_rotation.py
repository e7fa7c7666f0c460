"""GPU Hadamard-rotated int4 ("Running and Evaluating TurboQuant optimized
Gemma 4", TurboQuant section) against the oracle: the rotation kernel and the
rotated append bit for bit, the rotated decode within the output tolerance."""
import math
import types

import numpy as np
import pytest

import oracle
from int4_kv_cache_gb300 import synth
from tests.fwht_f32 import sequential_transform_f32
from tests.gpu_helpers import assert_close, cache_arrays, gpu_cache_from_fp16, need_gpu, workspace_for

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D", [64, 128, 256])
def test_rotate_rows_bit_exact(D):
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    rng = np.random.default_rng(100 + D)
    x = (rng.standard_normal((37, 3, D)) * 2).astype(np.float16)
    x[:, :, 5] *= 20
    xt = torch.from_numpy(x).cuda()
    got = tq.tq_hadamard_rotate(xt).cpu().numpy()
    assert np.array_equal(got.view(np.uint16), oracle.rotate_rows_f16(x).view(np.uint16))
    tq.tq_hadamard_rotate(xt, out=xt)  # in place
    assert np.array_equal(xt.cpu().numpy().view(np.uint16), got.view(np.uint16))


@pytest.mark.parametrize("D,flags", [(128, 1), (128, 3), (64, 3), (256, 2)])
def test_rotated_append_bit_exact(D, flags):
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    x = synth.decode_inputs(110 + D, 2, 2, 2, D, 300, outliers=True)
    cache = tq.KVCache(2, 2, D, 304)
    wp = torch.zeros(2, dtype=torch.int32, device="cuda")
    tq.tq_quantize_kv_append(cache, torch.from_numpy(x.k).cuda(), torch.from_numpy(x.v).cuda(), wp, flags=flags)
    torch.cuda.synchronize()
    kk = oracle.rotate_rows_f16(x.k) if flags & tq.TQ_ROTATE_K else x.k
    vv = oracle.rotate_rows_f16(x.v) if flags & tq.TQ_ROTATE_V else x.v
    oc = oracle.Cache.from_fp16(kk, vv)
    kc, ks, kb, vc, vs, vb = cache_arrays(cache)
    S = 300
    for got, want in ((kc, oc.kc), (ks, oc.ks), (kb, oc.kb), (vc, oc.vc), (vs, oc.vs), (vb, oc.vb)):
        assert np.array_equal(got[:, :, :S], want)


def _rotated_reference(x, lens, scale, flags, bits=4):
    kk = oracle.rotate_rows_f16(x.k) if flags & 1 else x.k
    vv = oracle.rotate_rows_f16(x.v) if flags & 2 else x.v
    qq = oracle.rotate_rows_f16(x.q) if flags & 1 else x.q
    out = oracle.attention(qq, oracle.Cache.from_fp16(kk, vv, bits=bits), lens, scale)
    return oracle.hadamard(out) if flags & 2 else out


@pytest.mark.parametrize("flags,D,bits", [(1, 128, 4), (2, 128, 4), (3, 128, 4), (3, 64, 4), (1, 256, 4),
                                          (3, 128, 8)])
def test_rotated_decode_matches_oracle(flags, D, bits):
    # the tensor-core kernel rotates each query head as it loads it
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    B, Hq, Hkv, S = 3, 16, 2, 3000
    lens = np.array([3000, 1, 1377], np.int32)
    x = synth.decode_inputs(120 + flags + D + bits, B, Hq, Hkv, D, S, lens=lens, outliers=True)
    cache = tq.KVCache(B, Hkv, D, S + 8, bits=bits)
    wp = torch.zeros(B, dtype=torch.int32, device="cuda")
    tq.tq_quantize_kv_append(cache, torch.from_numpy(x.k).cuda(), torch.from_numpy(x.v).cuda(), wp, flags=flags)
    ws = workspace_for(B, Hq, Hkv, D, S)
    out = tq.tq_sdpa_int4_decode(cache, torch.from_numpy(x.q).cuda(), torch.from_numpy(lens).cuda(), S,
                                 1 / math.sqrt(D), ws, flags=flags)
    torch.cuda.synchronize()
    assert_close(out.float().cpu().numpy(), _rotated_reference(x, lens, 1 / math.sqrt(D), flags, bits),
                 what=f"rotated decode flags={flags} D={D} bits={bits}")


def test_rotated_step_equals_append_then_decode():
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    B, Hq, Hkv, D, S, flags = 2, 64, 8, 128, 4992, 3
    x = synth.decode_inputs(131, B, Hq, Hkv, D, S, outliers=True)
    kn, vn = synth.append_tokens(131, 0, B, Hkv, D, 1, outliers=x.outlier_channels)
    pos = np.array([S - 1, 2500], np.int32)
    lens = pos + 1
    q, wp, lt = (torch.from_numpy(a).cuda() for a in (x.q, pos, lens))
    knt, vnt = torch.from_numpy(kn).cuda(), torch.from_numpy(vn).cuda()
    ws = workspace_for(B, Hq, Hkv, D, S)
    zero = torch.zeros(B, dtype=torch.int32, device="cuda")
    caches = []
    for _ in range(2):
        c = tq.KVCache(B, Hkv, D, S)
        tq.tq_quantize_kv_append(c, torch.from_numpy(x.k).cuda(), torch.from_numpy(x.v).cuda(), zero, flags=flags)
        caches.append(c)
    tq.tq_quantize_kv_append(caches[0], knt, vnt, wp, flags=flags)
    ref = tq.tq_sdpa_int4_decode(caches[0], q, lt, S, 0.088, ws, flags=flags).float().cpu().numpy()
    got = tq.tq_decode_step(caches[1], knt, vnt, wp, q, lt, S, 0.088, ws, flags=flags).float().cpu().numpy()
    assert torch.equal(caches[0].buffer, caches[1].buffer)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("D,bits,flags,n_new,paged", [
    (128, 4, 3, 1, False), (128, 4, 1, 3, False), (128, 4, 2, 1, False), (64, 4, 3, 2, False),
    (128, 8, 3, 1, False), (64, 8, 1, 1, False), (256, 4, 3, 1, False), (128, 4, 3, 2, True),
    (256, 8, 3, 2, False), (256, 4, 1, 3, True), (256, 4, 2, 16, False), (128, 4, 3, 17, False)])
def test_rotated_step_stores_oracle_rows(D, bits, flags, n_new, paged):
    # A rotated step of up to 16 rows appends them inside the decode kernel
    # (each tensor's row rotated across the warp lanes that hold it; at
    # head_dim 256 a whole warp), longer ones through the append kernel:
    # either way the stored rows are the oracle's quantised fp16(H x /
    # sqrt(D)) bit for bit, and the output is the rotated attention within the
    # output tolerance.
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    B, Hq, Hkv, S = 2, 16, 2, 1504
    x = synth.decode_inputs(140 + D + bits + flags + n_new, B, Hq, Hkv, D, S, outliers=True)
    kn, vn = synth.append_tokens(141 + D, 0, B, Hkv, D, n_new, outliers=x.outlier_channels)
    pos = np.array([S - n_new, 767 - n_new // 2], np.int32)  # the last run; a run boundary (768)
    lens = pos + n_new
    if paged:
        per = -(-S // 256)
        cache = tq.PagedKVCache(B, Hkv, D, 256, B * per + 1, per, bits=bits)
        perm = np.random.default_rng(7).permutation(B * per + 1)[:B * per].astype(np.int32).reshape(B, per)
        cache.block_table.copy_(torch.from_numpy(perm))
    else:
        cache = tq.KVCache(B, Hkv, D, S, bits=bits)
    zero = torch.zeros(B, dtype=torch.int32, device="cuda")
    # history: rows [0, pos[b]) of each sequence
    kh, vh = x.k.copy(), x.v.copy()
    for b in range(B):
        kh[b, :, pos[b]:] = 0
        vh[b, :, pos[b]:] = 0
    tq.tq_quantize_kv_append(cache, torch.from_numpy(kh).cuda(), torch.from_numpy(vh).cuda(), zero, flags=flags)
    ws = workspace_for(B, Hq, Hkv, D, S)
    wp = torch.from_numpy(pos).cuda()
    out = tq.tq_decode_step(cache, torch.from_numpy(kn).cuda(), torch.from_numpy(vn).cuda(), wp,
                            torch.from_numpy(x.q).cuda(), torch.from_numpy(lens).cuda(), S, 1 / math.sqrt(D), ws,
                            flags=flags)
    torch.cuda.synchronize()
    # the fp16 rows the cache now holds, in sequence order
    k_all, v_all = kh.copy(), vh.copy()
    for b in range(B):
        k_all[b, :, pos[b]:pos[b] + n_new] = kn[b]
        v_all[b, :, pos[b]:pos[b] + n_new] = vn[b]
    kk = oracle.rotate_rows_f16(k_all) if flags & 1 else k_all
    vv = oracle.rotate_rows_f16(v_all) if flags & 2 else v_all
    want = oracle.Cache.from_fp16(kk, vv, bits=bits)
    arrays = cache_arrays(cache)
    if paged:  # pages back in sequence order: [pages, Hkv, P, w] -> [B, Hkv, per * P, w]
        arrays = [a[perm].transpose(0, 2, 1, 3, 4).reshape(B, Hkv, -1, a.shape[3]) for a in arrays]
    for b in range(B):
        n = lens[b]
        for g_, w_ in zip(arrays, (want.kc, want.ks, want.kb, want.vc, want.vs, want.vb)):
            assert np.array_equal(g_[b, :, :n], w_[b, :, :n])
    full = types.SimpleNamespace(q=x.q, k=k_all, v=v_all)
    assert_close(out.float().cpu().numpy(), _rotated_reference(full, lens, 1 / math.sqrt(D), flags, bits),
                 what=f"rotated step D={D} bits={bits} flags={flags} n_new={n_new} paged={paged}")


@pytest.mark.parametrize("D", [64, 128, 256])
def test_reduce_rotates_the_merged_output_bit_for_bit(D):
    """TQ_ROTATE_V: the decode applies H to the merged fp32 output, then the
    scale fp32(1 / sqrt(D)) and one fp16 rounding (tq.h, rotation flags).  With
    one run per sequence the merged output is fp32(acc / l) of phase 1's own
    state (the weight is expf(0) = 1; the sum starts from +0), so the same
    transform restated in numpy float32 from that state must give the decode's
    output bit for bit, whichever threads, lanes and warps the reduce spreads
    the stages over.  A consistency check of the rotation step; parity with
    the oracle is test_rotated_decode_matches_oracle."""
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    B, Hq, Hkv, S = 3, 16, 2, 60  # within one tile at every head_dim: one run
    lens = np.array([60, 37, 0], np.int32)
    x = synth.decode_inputs(140 + D, B, Hq, Hkv, D, S, lens=lens, outliers=True)
    cache = tq.KVCache(B, Hkv, D, 64)
    tq.tq_quantize_kv_append(cache, torch.from_numpy(x.k).cuda(), torch.from_numpy(x.v).cuda(),
                             torch.zeros(B, dtype=torch.int32, device="cuda"), flags=tq.TQ_ROTATE_V)
    q, lt = torch.from_numpy(x.q).cuda(), torch.from_numpy(lens).cuda()
    a = 1 / math.sqrt(D)
    assert tq.tq_sdpa_plan(cache, Hq, S)[0] == 1
    out = tq.tq_sdpa_int4_decode(cache, q, lt, S, a, workspace_for(B, Hq, Hkv, D, S), flags=tq.TQ_ROTATE_V)
    _, l, acc = tq.tq_sdpa_int4_partial(cache, q, lt, S, a, chunks_per_split=0)
    l = l.cpu().numpy()[:, :, 0]
    acc = acc.cpu().numpy()[:, :, 0, :]
    z = np.float32(0.0)
    t = (acc + z) + z  # the reduce's t = 0 + fmaf(1, acc, 0)
    with np.errstate(divide="ignore", invalid="ignore"):
        o = np.where(l[..., None] > 0, t / l[..., None], z).astype(np.float32)
    rs = np.float32(1.0 / np.sqrt(np.float64(D)))
    want = (sequential_transform_f32(o) * rs).astype(np.float16)
    assert np.array_equal(out.cpu().numpy().view(np.uint16), want.view(np.uint16))
    assert np.all(want[2] == 0)
