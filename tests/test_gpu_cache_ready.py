"""TQ_CACHE_READY: the decode kernel may stream the cache before the kernel
ahead of it on the stream has finished, and reads the query and the new K/V
rows only after waiting for it.  A chain of steps over several layer caches,
where each step's query is computed by torch kernels from the previous
step's output (so a query read too early would be stale), must give the same
bits with and without the flag, eagerly and replayed from a CUDA graph, for
the fused one-row append, the append-kernel path (more than 16 rows) and a
rotated cache; one step is also checked against the oracle."""
import math

import numpy as np
import pytest

import oracle
from int4_kv_cache_gb300 import synth
from tests.gpu_helpers import assert_close, gpu_cache_from_fp16, need_gpu, workspace_for

pytestmark = pytest.mark.gpu

B, HQ, HKV, D, S, LAYERS = 2, 64, 8, 128, 6016, 3


def _layers(torch, tq, n_new, flags):
    xs, caches, news = [], [], []
    for layer in range(LAYERS):
        x = synth.decode_inputs(700 + layer, B, HQ, HKV, D, S, outliers=True)
        kn, vn = synth.append_tokens(700 + layer, 5, B, HKV, D, n_new, outliers=x.outlier_channels)
        if flags & (tq.TQ_ROTATE_K | tq.TQ_ROTATE_V):
            cache = tq.KVCache(B, HKV, D, S)
            tq.tq_quantize_kv_append(cache, torch.from_numpy(x.k).cuda(), torch.from_numpy(x.v).cuda(),
                                     torch.zeros(B, dtype=torch.int32, device="cuda"), flags=flags)
        else:
            cache = gpu_cache_from_fp16(x.k, x.v, capacity=S)
        xs.append(x)
        caches.append(cache)
        news.append((torch.from_numpy(kn).cuda(), torch.from_numpy(vn).cuda()))
    return xs, caches, news


@pytest.mark.parametrize("n_new,rot", [(1, 0), (20, 0), (1, 3)])
def test_cache_ready_chain_matches_plain_chain(n_new, rot):
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    flags_rot = rot  # TQ_ROTATE_K | TQ_ROTATE_V when 3
    a = 1 / math.sqrt(D)
    pos = np.array([S - n_new, S // 2], np.int32)
    wp = torch.from_numpy(pos).cuda()
    lt = torch.from_numpy(pos + n_new).cuda()
    q0 = torch.from_numpy(synth.decode_inputs(799, B, HQ, HKV, D, 16).q).cuda()

    def chain(extra_flags, graph):
        xs, caches, news = _layers(torch, tq, n_new, flags_rot)
        ws = workspace_for(B, HQ, HKV, D, S)
        outs = [torch.empty((B, HQ, D), dtype=torch.float16, device="cuda") for _ in range(2 * LAYERS)]
        qs = [torch.empty_like(q0) for _ in range(2 * LAYERS)]

        def run():
            q = q0
            for i in range(2 * LAYERS):
                layer = i % LAYERS
                tq.tq_decode_step(caches[layer], news[layer][0], news[layer][1], wp, q, lt, S, a, ws, out=outs[i],
                                  flags=flags_rot | extra_flags)
                # the next layer's query depends on this output
                torch.add(q0, outs[i], alpha=0.5, out=qs[i])
                q = qs[i]

        if graph:
            run()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                run()
            g.replay()
        else:
            run()
        torch.cuda.synchronize()
        return [o.cpu().numpy() for o in outs], xs, news

    plain, xs, news = chain(0, False)
    for graph in (False, True):
        ready, _, _ = chain(tq.TQ_CACHE_READY, graph)
        for i, (p, r) in enumerate(zip(plain, ready)):
            assert np.array_equal(p.view(np.uint16), r.view(np.uint16)), (i, graph)
    if rot == 0:
        # the first step against the oracle (layer 0's cache with its new rows)
        x = xs[0]
        kn, vn = news[0][0].cpu().numpy(), news[0][1].cpu().numpy()
        kk, vv = x.k.copy(), x.v.copy()
        for b in range(B):
            kk[b, :, pos[b]:pos[b] + n_new] = kn[b]
            vv[b, :, pos[b]:pos[b] + n_new] = vn[b]
        ref = oracle.attention(q0.cpu().numpy(), oracle.Cache.from_fp16(kk, vv), pos + n_new, a)
        assert_close(plain[0].astype(np.float64), ref, what=f"ready chain n_new={n_new}")


def test_cache_ready_decode_only():
    """tq_sdpa_int4_decode_ex with TQ_CACHE_READY after a torch kernel that
    writes the query: the same bits as without the flag."""
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    x = synth.decode_inputs(811, B, HQ, HKV, D, S, outliers=True)
    cache = gpu_cache_from_fp16(x.k, x.v, capacity=S)
    ws = workspace_for(B, HQ, HKV, D, S)
    lt = torch.from_numpy(x.lens).cuda()
    q0 = torch.from_numpy(x.q).cuda()
    res = []
    for flags in (0, tq.TQ_CACHE_READY):
        q = torch.empty_like(q0)
        torch.mul(q0, 2.0, out=q)  # written by the kernel just ahead of the decode (exact in fp16)
        res.append(tq.tq_sdpa_int4_decode(cache, q, lt, S, 0.088, ws, flags=flags).cpu().numpy())
    assert np.array_equal(res[0].view(np.uint16), res[1].view(np.uint16))
    ref = oracle.attention((x.q.astype(np.float32) * 2.0).astype(np.float16), oracle.Cache.from_fp16(x.k, x.v),
                           x.lens, 0.088)
    assert_close(res[1].astype(np.float64), ref, what="ready decode")
