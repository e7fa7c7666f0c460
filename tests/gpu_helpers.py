"""Shared helpers for the GPU parity tests (marshalling and comparison only)."""
import numpy as np
import pytest

ATOL = 2e-3      # max-abs bound on the fp16 output vs fp64 attention
RTOL_L2 = 1e-3   # relative L2 bound over the compared output rows


def need_gpu():
    import torch

    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU required for tests marked gpu")
    from int4_kv_cache_gb300 import build

    build.build()
    return torch


def gpu_cache_from_fp16(k, v, capacity=None):
    """Quantize fp16 K/V [B, Hkv, S, D] (numpy or torch) into a fresh GPU cache via the ABI."""
    import torch

    import int4_kv_cache_gb300 as tq

    kt = k if isinstance(k, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(k)).cuda()
    vt = v if isinstance(v, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(v)).cuda()
    B, Hkv, S, D = kt.shape
    cap = capacity or max(16, -(-S // 16) * 16)
    cache = tq.KVCache(B, Hkv, D, cap)
    if S:
        wp = torch.zeros(B, dtype=torch.int32, device="cuda")
        tq.tq_quantize_kv_append(cache, kt.contiguous(), vt.contiguous(), wp)
    return cache


def gpu_cache_from_oracle(oc, capacity=None):
    """Load an oracle-quantised cache (host arrays) into a GPU cache."""
    import torch

    import int4_kv_cache_gb300 as tq

    cap = capacity or max(16, -(-oc.cap // 16) * 16)
    cache = tq.KVCache(oc.B, oc.Hkv, oc.D, cap)
    S = oc.cap
    cache.k_codes[:, :, :S].copy_(torch.from_numpy(oc.kc))
    cache.v_codes[:, :, :S].copy_(torch.from_numpy(oc.vc))
    cache.k_scale[:, :, :S].copy_(torch.from_numpy(oc.ks.view(np.float16)))
    cache.k_bias[:, :, :S].copy_(torch.from_numpy(oc.kb.view(np.float16)))
    cache.v_scale[:, :, :S].copy_(torch.from_numpy(oc.vs.view(np.float16)))
    cache.v_bias[:, :, :S].copy_(torch.from_numpy(oc.vb.view(np.float16)))
    return cache


def same_layout(head_dim, bits=4):
    """Whether contiguous and paged caches of this width decode with the same
    kernel layout (then their outputs agree bit for bit; the contiguous int4
    cache at head_dim 128 runs twelve warps per CTA, the paged one four, so
    there the two sum in different orders and agree within the tolerance)."""
    return not (head_dim == 128 and bits == 4)


def identity_paged(tq, torch, src, page_tokens):
    """A paged cache holding the rows of the paged cache `src` with each
    sequence's pages in order (block_table[b, i] = b * per + i): decoding it
    runs the same kernel over the same rows as `src`, so any difference from
    `src`'s output is the block-table translation."""
    B, per = src.block_table.shape
    ident = tq.PagedKVCache(B, src.num_kv_heads, src.head_dim, page_tokens, B * per, per, bits=src.bits)
    ident.block_table.copy_(torch.arange(B * per, dtype=torch.int32, device="cuda").reshape(B, per))
    tab = src.block_table.long()
    for f in ("k_codes", "v_codes", "k_scale", "k_bias", "v_scale", "v_bias"):
        getattr(ident, f).copy_(getattr(src, f)[tab.reshape(-1)])
    return ident


def workspace_for(B, Hq, Hkv, D, max_len, chunk=512):
    import torch

    import int4_kv_cache_gb300 as tq

    return tq.workspace(B, Hq, Hkv, D, max_len, chunk)


def decode(cache, q, lens, max_len, attn_scale, chunk=512, impl=0, status=None):
    """Run tq_sdpa_int4_decode and return the output as float64 numpy."""
    import torch

    import int4_kv_cache_gb300 as tq

    qt = q if isinstance(q, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(q)).cuda()
    lt = torch.from_numpy(np.asarray(lens, dtype=np.int32)).cuda()
    ws = workspace_for(cache.batch, qt.shape[1], cache.num_kv_heads, cache.head_dim, max_len, chunk)
    out = tq.tq_sdpa_int4_decode(cache, qt, lt, max_len, attn_scale, ws, chunk=chunk, impl=impl, status=status)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64)


def assert_close(out, ref, atol=ATOL, rtol_l2=RTOL_L2, what=""):
    """max-abs <= atol and relative L2 (||o - r|| / ||r||) <= rtol_l2."""
    o = np.asarray(out, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert o.shape == r.shape, (o.shape, r.shape)
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    err = np.abs(o - r)
    mx = float(err.max(initial=0.0))
    nrm = float(np.linalg.norm(r))
    rel = float(np.linalg.norm(o - r) / nrm) if nrm > 0 else float(np.linalg.norm(o - r))
    assert mx <= atol, f"{what}: max abs err {mx:.3e} > {atol}"
    assert rel <= rtol_l2, f"{what}: rel L2 err {rel:.3e} > {rtol_l2}"
    return mx, rel


def cache_arrays(cache):
    """GPU cache contents as host numpy arrays (codes, scale/bias bits)."""
    return (cache.k_codes.cpu().numpy(), cache.k_scale.cpu().numpy().view(np.uint16),
            cache.k_bias.cpu().numpy().view(np.uint16), cache.v_codes.cpu().numpy(),
            cache.v_scale.cpu().numpy().view(np.uint16), cache.v_bias.cpu().numpy().view(np.uint16))
