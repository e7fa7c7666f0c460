"""The allocation-free decode entry point, checked against the regular one.

tq_sdpa_int4_decode_noalloc exists for callers that cannot hand the library a
workspace (no allocator at hand, or allocation not allowed where they run); it
keeps the split-K partial states in a fixed device array inside the library.
This file is collected last so that a run stopping at its first failure has
already run every other test; it passes alone in a fresh process too.
"""
import ctypes

import numpy as np
import pytest

import oracle
from int4_kv_cache_gb300 import synth
from tests.gpu_helpers import assert_close, gpu_cache_from_fp16, need_gpu, workspace_for

pytestmark = pytest.mark.gpu


def _noalloc(L, cache, q, lens, max_len, attn, out):
    import torch

    st = L.tq_sdpa_int4_decode_noalloc(cache.ref(), ctypes.c_void_p(q.data_ptr()), q.shape[1],
                                       ctypes.c_void_p(lens.data_ptr()), max_len, ctypes.c_float(attn), 512,
                                       ctypes.c_void_p(out.data_ptr()), None,
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return st


def test_noalloc_decode_matches_workspace_decode_on_two_calls():
    """Four calls in a row on different problems (a stale array from one call
    would show in the next), covering both ways the call merges the runs:
    the reduce over partial states in the array (16K tokens, batch 2: more
    than 8 runs; the same with ragged lengths) and the merge inside phase 1
    (1K tokens: at most 8 runs in thread-block clusters; Gemma shape at 33
    tokens: one run).  Each output must equal the workspace decode's bit for
    bit (same plan, same kernels) and the oracle's within the bar."""
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    L = tq.lib()
    llama = synth.WORKLOADS["llama70b_16k"]
    gemma = synth.WORKLOADS["gemma_33"]
    problems = [
        (synth.decode_inputs(llama.seed, 2, 64, 8, 128, 16384, outliers=True), llama.attn_scale, "reduce"),
        (synth.decode_inputs(llama.seed + 1, 2, 64, 8, 128, 16384, outliers=True,
                             lens=np.array([3001, 129], np.int32)), llama.attn_scale, "reduce"),
        (synth.decode_inputs(llama.seed + 2, 1, 64, 8, 128, 1024, outliers=True), llama.attn_scale, "merged"),
        (gemma.draw(), gemma.attn_scale, "merged"),
    ]
    for x, attn, branch in problems:
        B, Hq, D = x.q.shape
        Hkv = x.k.shape[1]
        cache = gpu_cache_from_fp16(x.k, x.v)
        q = torch.from_numpy(x.q).cuda()
        lens = torch.from_numpy(x.lens).cuda()
        max_len = int(x.lens.max())
        n_splits = tq.tq_sdpa_plan(cache, Hq, max_len)[0]
        assert (n_splits > 8) if branch == "reduce" else (n_splits <= 8), (branch, n_splits)
        ref = tq.tq_sdpa_int4_decode(cache, q, lens, max_len, attn, workspace_for(B, Hq, Hkv, D, max_len), chunk=512)
        out = torch.full_like(q, float("nan"))
        assert _noalloc(L, cache, q, lens, max_len, attn, out) == 0
        got = out.cpu().numpy()
        assert np.array_equal(got.view(np.uint16), ref.cpu().numpy().view(np.uint16)), branch
        want = oracle.attention(x.q, oracle.Cache.from_fp16(x.k, x.v), x.lens, attn)
        assert_close(got.astype(np.float64), want, what=f"noalloc {branch} {x.k.shape}")


def test_noalloc_rejects_requests_beyond_its_array():
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    L = tq.lib()
    # 128 sequences x 64 heads: even one split per (sequence, kv head) needs
    # 128 * 64 * 130 * 4 bytes > 4 MiB of partial states
    B, Hq, Hkv, D, cap = 128, 64, 8, 128, 16
    cache = tq.KVCache(B, Hkv, D, cap)
    q = torch.zeros((B, Hq, D), dtype=torch.float16, device="cuda")
    lens = torch.full((B,), cap, dtype=torch.int32, device="cuda")
    out = torch.zeros_like(q)
    assert B * Hq * (D + 2) * 4 > tq.NOALLOC_SCRATCH_BYTES
    assert _noalloc(L, cache, q, lens, cap, 0.1, out) == 4  # TQ_ERR_WORKSPACE, nothing launched
    assert torch.count_nonzero(out).item() == 0
