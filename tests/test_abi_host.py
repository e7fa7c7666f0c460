"""C-ABI checks that need no GPU: the library loads, exports every entry point
include/tq.h declares, its host-only size helpers are right, and argument
errors are reported before anything is launched."""
import ctypes
import math
import os
import re

import pytest

import int4_kv_cache_gb300 as tq
from int4_kv_cache_gb300 import build as tqbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def L():
    tqbuild.build()
    return tq.lib()


def declared_functions():
    names = set()
    for fname in os.listdir(os.path.join(ROOT, "include")):
        text = open(os.path.join(ROOT, "include", fname)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(tq_[a-z0-9_]+)\s*\(", text,
                                flags=re.M))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("tq_quantize_kv_append", "tq_sdpa_int4_decode", "tq_sdpa_int4_partial", "tq_sdpa_int4_reduce",
                 "tq_sdpa_workspace_bytes", "tq_kv_cache_bytes", "tq_status_string", "tq_sdpa_plan"):
        assert must in names


def test_library_exports_every_declared_symbol(L):
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing
    assert tq.tq_abi_version() == 2


def test_status_strings(L):
    for s in range(8):
        assert isinstance(tq.tq_status_string(s), str) and tq.tq_status_string(s)


def test_cache_bytes_closed_form(L):
    # rows * (D/2 codes + 2 fp16 scale/bias per group) for K and V, each array 256-aligned
    B, Hkv, D, cap = 1, 8, 128, 131072
    rows = B * Hkv * cap
    assert tq.tq_kv_cache_bytes(B, Hkv, D, 64, cap) == 2 * rows * (D // 2) + 4 * rows * (D // 64) * 2
    assert tq.tq_kv_cache_bytes(0, 8, 128, 64, 16) == 0
    assert tq.tq_kv_cache_bytes(1, 8, 100, 64, 16) == 0


def test_memory_table_of_the_llama_page(L):
    # FP16 column of the memory table: 80 layers x 8 kv heads x ctx x 128 x 2 B x 2 (K+V), in GiB
    rows = [l.split() for l in open(os.path.join(GOLDEN, "llama70b_kv_memory_table.txt"))
            if l.strip() and not l.startswith("#")]
    for ctx, fp16_gib, _int4_printed in rows:
        ctx = int(ctx)
        fp16 = 80 * 8 * ctx * 128 * 2 * 2
        assert round(fp16 / 2**30, 1) == float(fp16_gib)
        # int4 at group 64 with fp16 scale+bias: (64 + 8) bytes per 128-element row vs 256
        int4 = 80 * tq.tq_kv_cache_bytes(1, 8, 128, 64, ctx)
        assert int4 * 128 == fp16 * 36
    assert 80 * tq.tq_kv_cache_bytes(1, 8, 128, 64, 131072) == 12_079_595_520


def test_workspace_bytes(L):
    # runs per (sequence, kv head) are bounded by 2048 CTAs / (B * Hkv) and by
    # the sequence length in 16-token units
    def want(B, Hq, Hkv, D, S):
        ns = min(math.ceil(S / 16), max(1, 2048 // (B * Hkv)))
        parts = B * Hq * ns
        a256 = lambda n: -(-n // 256) * 256
        # m, l, acc per part, room for the rotated query (B * Hq * D fp16), then
        # the dispatch order of the runs (B * ns int32)
        return 2 * a256(parts * 4) + a256(parts * D * 4) + a256(B * Hq * D * 2) + a256(B * ns * 8)

    assert tq.tq_sdpa_workspace_bytes(1, 64, 8, 128, 131072, 512) == want(1, 64, 8, 128, 131072)
    assert tq.tq_sdpa_workspace_bytes(32, 64, 8, 128, 32768, 512) == want(32, 64, 8, 128, 32768)
    assert tq.tq_sdpa_workspace_bytes(1, 8, 2, 128, 40, 512) == want(1, 8, 2, 128, 40)
    assert tq.tq_sdpa_workspace_bytes(1, 64, 8, 128, 0, 512) == 0


def _fake_cache(B=1, Hkv=2, D=128, cap=256):
    c = tq.tq_kv_cache()
    base = 1 << 20
    for i, f in enumerate(("k_codes", "v_codes", "k_scale", "k_bias", "v_scale", "v_bias")):
        setattr(c, f, base + i * (1 << 20))
    c.batch, c.num_kv_heads, c.head_dim, c.group_size, c.capacity = B, Hkv, D, 64, cap
    c.bits = 4
    return c


def _decode(L, c, q=0x100000, hq=8, lens=0x200000, max_len=256, chunk=512, ws=0x300000, ws_bytes=1 << 30,
            out=0x400000, impl=0):
    return L.tq_sdpa_int4_decode_impl(ctypes.byref(c) if c is not None else None, q, hq, lens, max_len,
                                      ctypes.c_float(0.1), chunk, ws, ws_bytes, out, None, impl, None)


def test_decode_argument_errors_launch_nothing(L):
    # Host-side checks fire before any CUDA call, so they work without a GPU.
    c = _fake_cache()
    assert _decode(L, None) == 1                                  # TQ_ERR_NULL
    assert _decode(L, c, q=0) == 1
    assert _decode(L, c, hq=7) == 2                               # Hq % Hkv != 0
    assert _decode(L, c, hq=2 * 16) == 6                          # GQA ratio 16 > 8
    assert _decode(L, c, max_len=0) == 2
    assert _decode(L, c, max_len=257) == 3                        # beyond capacity
    assert _decode(L, c, chunk=24) == 2                           # not a multiple of 16
    assert _decode(L, c, ws_bytes=16) == 4                        # workspace too small
    assert _decode(L, c, ws=0) == 4
    assert _decode(L, c, ws=0x300010) == 7                        # workspace not 256-aligned
    assert _decode(L, c, q=0x100002) == 7                         # misaligned q
    assert _decode(L, c, impl=9) == 6
    assert _decode(L, _fake_cache(D=96)) == 6
    assert _decode(L, _fake_cache(cap=250), max_len=200) == 2
    bad = _fake_cache()
    bad.group_size = 32
    assert _decode(L, bad) == 6
    bad = _fake_cache()
    bad.v_bias = 0
    assert _decode(L, bad) == 1
    bad = _fake_cache()
    bad.k_scale += 2
    assert _decode(L, bad) == 7


def test_append_argument_errors_launch_nothing(L):
    c = _fake_cache()
    f = L.tq_quantize_kv_append
    assert f(ctypes.byref(c), 0, 0x1000, 1, 0x2000, None, None) == 1
    assert f(ctypes.byref(c), 0x1000, 0x1000, -1, 0x2000, None, None) == 2
    assert f(ctypes.byref(c), 0x1000, 0x1000, 257, 0x2000, None, None) == 3
    assert f(ctypes.byref(c), 0x1008, 0x1000, 1, 0x2000, None, None) == 7
    assert f(ctypes.byref(c), 0x1000, 0x1000, 0, 0x2000, None, None) == 0  # nothing to do


def test_reduce_partial_and_plan_argument_errors(L):
    assert L.tq_sdpa_int4_reduce(0, 0x10, 0x10, 1, 1, 128, 1, 0x10, None) == 1
    assert L.tq_sdpa_int4_reduce(0x10, 0x10, 0x10, 1, 1, 128, 0, 0x10, None) == 2
    assert L.tq_sdpa_int4_reduce(0x10, 0x10, 0x10, 1, 1, 128, 20000, 0x10, None) == 2
    assert L.tq_sdpa_int4_reduce(0x10, 0x10, 0x10, 1, 1, 96, 1, 0x10, None) == 6
    c = _fake_cache()
    f = L.tq_sdpa_int4_partial
    assert f(ctypes.byref(c), 0x1000, 8, 0x2000, 256, ctypes.c_float(1.0), 512, 1, 0x3000, 0, 0x4000, None, 0,
             None) == 1
    assert f(ctypes.byref(c), 0x1000, 8, 0x2000, 256, ctypes.c_float(1.0), 512, -1, 0x3000, 0x3000, 0x4000, None,
             0, None) == 2
    ns, run = ctypes.c_int32(), ctypes.c_int32()
    assert L.tq_sdpa_plan(ctypes.byref(c), 8, 256, 500, 0, ctypes.byref(ns), ctypes.byref(run)) == 2
    assert L.tq_sdpa_plan(ctypes.byref(c), 8, 256, 512, 0, None, ctypes.byref(run)) == 1
    assert L.tq_sdpa_plan(ctypes.byref(c), 8, 256, 512, 7, ctypes.byref(ns), ctypes.byref(run)) == 6


def test_carve_layout(L):
    c = tq.tq_kv_cache()
    assert L.tq_kv_cache_carve(ctypes.byref(c), 0x10000, 2, 8, 128, 64, 64) == 0
    rows = 2 * 8 * 64
    assert c.v_codes - c.k_codes == rows * 64
    assert c.k_scale - c.k_codes == 2 * rows * 64
    assert c.k_bias - c.k_scale == rows * 2 * 2
    assert (c.capacity, c.head_dim, c.num_kv_heads, c.batch) == (64, 128, 8, 2)
    assert L.tq_kv_cache_carve(ctypes.byref(c), 0x10010, 2, 8, 128, 64, 64) == 7


def test_dequantize_argument_errors_launch_nothing(L):
    c = _fake_cache()
    f = L.tq_dequantize_kv
    assert f(None, 16, 0x1000, 0x2000, None) == 1
    assert f(ctypes.byref(c), 16, 0, 0x2000, None) == 1
    assert f(ctypes.byref(c), -1, 0x1000, 0x2000, None) == 2
    assert f(ctypes.byref(c), 257, 0x1000, 0x2000, None) == 3
    assert f(ctypes.byref(c), 16, 0x1008, 0x2000, None) == 7
    assert f(ctypes.byref(c), 0, 0x1000, 0x2000, None) == 0  # nothing to do


def test_rotation_argument_errors_launch_nothing(L):
    c = _fake_cache()
    assert L.tq_hadamard_rotate(None, 4, 128, 0x2000, None) == 1
    assert L.tq_hadamard_rotate(0x1000, -1, 128, 0x2000, None) == 2
    assert L.tq_hadamard_rotate(0x1000, 4, 96, 0x2000, None) == 6
    assert L.tq_hadamard_rotate(0x1008, 4, 128, 0x2000, None) == 7
    assert L.tq_hadamard_rotate(0x1000, 0, 128, 0x2000, None) == 0  # nothing to do
    f = L.tq_quantize_kv_append_ex
    assert f(ctypes.byref(c), 0x1000, 0x1000, 1, 0x2000, 4, None, None) == 6   # unknown flag bit
    assert f(ctypes.byref(c), 0x1000, 0x1000, 0, 0x2000, 3, None, None) == 0
    d = L.tq_sdpa_int4_decode_ex
    assert d(ctypes.byref(c), 0x100000, 8, 0x200000, 256, ctypes.c_float(0.1), 512, 8, 0x300000, 1 << 30,
             0x400000, None, None) == 6
    assert d(ctypes.byref(c), 0x100000, 8, 0x200000, 256, ctypes.c_float(0.1), 512, 1, 0x300000, 16, 0x400000,
             None, None) == 4


def _fake_paged(B=2, Hkv=2, D=128, P=128, pages=8, maxp=4):
    c = tq.tq_paged_kv_cache()
    base = 1 << 20
    for i, f in enumerate(("k_codes", "v_codes", "k_scale", "k_bias", "v_scale", "v_bias", "block_table")):
        setattr(c, f, base + i * (1 << 20))
    c.batch, c.num_kv_heads, c.head_dim, c.group_size = B, Hkv, D, 64
    c.page_tokens, c.num_pages, c.max_pages_per_seq = P, pages, maxp
    c.bits = 4
    return c


def test_paged_pool_bytes_and_carve(L):
    # a page is one [Hkv][page_tokens] block of the six arrays
    assert tq.lib().tq_paged_kv_cache_bytes(10, 8, 128, 64, 4, 256) == tq.tq_kv_cache_bytes(10, 8, 128, 64, 256)
    c = tq.tq_paged_kv_cache()
    assert L.tq_paged_kv_cache_carve(ctypes.byref(c), 0x100000, 0x2000, 3, 8, 128, 64, 4, 256, 10, 5) == 0
    rows = 10 * 8 * 256
    assert c.v_codes - c.k_codes == rows * 64 and c.block_table == 0x2000
    assert (c.batch, c.page_tokens, c.num_pages, c.max_pages_per_seq) == (3, 256, 10, 5)
    assert L.tq_paged_kv_cache_carve(ctypes.byref(c), 0x100000, 0x2000, 3, 8, 128, 64, 4, 200, 10, 5) == 2
    assert L.tq_paged_kv_cache_carve(ctypes.byref(c), 0x100000, None, 3, 8, 128, 64, 4, 256, 10, 5) == 1


def test_paged_argument_errors_launch_nothing(L):
    d = L.tq_paged_sdpa_int4_decode
    args = lambda c, max_len=256, flags=0: (ctypes.byref(c), 0x100000, 8, 0x200000, max_len, ctypes.c_float(0.1),
                                            512, flags, 0x300000, 1 << 30, 0x400000, None, None)
    bad = _fake_paged()
    bad.block_table = 0
    assert d(*args(bad)) == 1
    assert d(*args(_fake_paged(P=192))) == 2                 # pages hold whole 128-token tiles
    assert d(*args(_fake_paged(), max_len=513)) == 3         # beyond max_pages * page_tokens
    assert d(*args(_fake_paged(), flags=0x100)) == 6         # no advance on a decode without append
    s = L.tq_paged_decode_step
    c = _fake_paged()
    assert s(ctypes.byref(c), 0x1000, 0x1000, 1, 0x200000, 0x100000, 8, 0x200000, 256, ctypes.c_float(0.1), 512,
             0x100, 0x300000, 1 << 30, 0x400000, None, None) == 2   # advance with write_pos == seq_lens
    a = L.tq_paged_quantize_kv_append
    assert a(ctypes.byref(c), 0x1000, 0x1000, 513, 0x2000, 0, None, None) == 3
    assert a(ctypes.byref(c), 0x1000, 0x1000, 1, 0x2000, 8, None, None) == 6


def test_int8_sizes_and_validation(L):
    # int8: D bytes of codes per row instead of D/2
    B, Hkv, D, cap = 1, 8, 128, 4096
    rows = B * Hkv * cap
    assert L.tq_kv_cache_bytes_ex(B, Hkv, D, 64, 8, cap) == 2 * rows * D + 4 * rows * (D // 64) * 2
    assert L.tq_kv_cache_bytes_ex(B, Hkv, D, 64, 4, cap) == tq.tq_kv_cache_bytes(B, Hkv, D, 64, cap)
    assert L.tq_kv_cache_bytes_ex(B, Hkv, D, 64, 5, cap) == 0
    c = tq.tq_kv_cache()
    assert L.tq_kv_cache_carve_ex(ctypes.byref(c), 0x100000, 2, 8, 128, 64, 8, 64) == 0
    assert c.bits == 8 and c.v_codes - c.k_codes == 2 * 8 * 64 * 128
    assert _decode(L, _fake_cache()) != 6
    wide = _fake_cache(D=256)
    wide.bits = 8  # int8 rows of 256 bytes: two 128-byte column blocks per tile
    assert _decode(L, wide) != 6
    bad = _fake_cache()
    bad.bits = 0
    assert _decode(L, bad) == 6


def test_wait_timeout_selftest_argument_errors(L):
    f = L.tq_wait_timeout_selftest
    assert f(None, 0x1000, 100, 0x2000, None) == 1
    assert f(0x1000, None, 100, 0x2000, None) == 1
    assert f(0x1000, 0x2000, 100, None, None) == 1
    assert f(0x1008, 0x2000, 100, 0x3000, None) == 7   # src not 16-byte aligned
    assert f(0x1000, 0x2000, 0, 0x3000, None) == 2     # limit out of range
    assert f(0x1000, 0x2000, 100001, 0x3000, None) == 2
