"""int4 KV-cache quantize-on-store and fused decode attention for GB300.

Thin Python binding over the C-ABI library ``libtq.so`` (see include/tq.h):
argument marshalling only.  Every step of the path runs in the library's CUDA
kernels; PyTorch supplies device memory and the current stream.  There is no
fallback: if the compiled library is missing, every entry point raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

__all__ = [
    "TQ_OK", "TQ_IMPL_AUTO", "TQ_IMPL_MMA", "TQ_IMPL_SIMT", "TQ_DEV_WRITE_POS", "TQ_DEV_SEQ_LEN",
    "TQ_DEV_TIMEOUT", "TQError", "lib", "lib_path", "tq_kv_cache", "KVCache",
    "tq_abi_version", "tq_status_string", "tq_kv_cache_bytes", "tq_sdpa_workspace_bytes", "workspace",
    "tq_quantize_kv_append", "tq_sdpa_int4_decode", "tq_sdpa_int4_partial", "tq_sdpa_int4_reduce",
    "tq_sdpa_plan", "tq_split_plan", "tq_sdpa_int4_decode_noalloc", "NOALLOC_SCRATCH_BYTES", "tq_decode_step",
    "tq_dequantize_kv", "tq_hadamard_rotate", "TQ_ROTATE_K", "TQ_ROTATE_V", "TQ_STEP_ADVANCE", "TQ_DEV_PAGE",
    "tq_paged_kv_cache", "PagedKVCache", "tq_decode_step_host", "tq_host_staging_bytes",
]

TQ_OK = 0
TQ_IMPL_AUTO, TQ_IMPL_MMA, TQ_IMPL_SIMT = 0, 1, 2
TQ_DEV_WRITE_POS, TQ_DEV_SEQ_LEN, TQ_DEV_TIMEOUT = 0x1, 0x2, 0x4
TQ_ROTATE_K, TQ_ROTATE_V = 0x1, 0x2
TQ_STEP_ADVANCE = 0x100
TQ_DEV_PAGE = 0x8
GROUP_SIZE = 64
DEFAULT_CHUNK = 512
NOALLOC_SCRATCH_BYTES = 4 << 20

_HERE = os.path.dirname(os.path.abspath(__file__))


def lib_path() -> str:
    return os.path.join(_HERE, "_build", "libtq.so")


class TQError(RuntimeError):
    def __init__(self, fn: str, status: int):
        msg = lib().tq_status_string(status).decode()
        if status == 5:
            msg += f" (cudaError {lib().tq_last_cuda_error()})"
        super().__init__(f"{fn}: {msg} [status {status}]")
        self.status = status


class tq_kv_cache(ctypes.Structure):
    _fields_ = [
        ("k_codes", ctypes.c_void_p), ("v_codes", ctypes.c_void_p),
        ("k_scale", ctypes.c_void_p), ("k_bias", ctypes.c_void_p),
        ("v_scale", ctypes.c_void_p), ("v_bias", ctypes.c_void_p),
        ("batch", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("group_size", ctypes.c_int32),
        ("capacity", ctypes.c_int32), ("bits", ctypes.c_int32),
    ]


class tq_paged_kv_cache(ctypes.Structure):
    _fields_ = [
        ("k_codes", ctypes.c_void_p), ("v_codes", ctypes.c_void_p),
        ("k_scale", ctypes.c_void_p), ("k_bias", ctypes.c_void_p),
        ("v_scale", ctypes.c_void_p), ("v_bias", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p),
        ("batch", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("group_size", ctypes.c_int32),
        ("page_tokens", ctypes.c_int32), ("num_pages", ctypes.c_int32),
        ("max_pages_per_seq", ctypes.c_int32), ("bits", ctypes.c_int32),
    ]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libtq.so (built by ``build.build()``); raises if it is not there."""
    global _lib
    if _lib is None:
        path = lib_path()
        if not os.path.exists(path):
            raise ImportError(f"libtq.so not built ({path}); run int4_kv_cache_gb300.build.build()")
        L = ctypes.CDLL(path)
        P, i32, sz, f32, u32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float, ctypes.c_uint32
        C = ctypes.POINTER(tq_kv_cache)
        PC = ctypes.POINTER(tq_paged_kv_cache)
        sig = {
            "tq_abi_version": ([], i32),
            "tq_status_string": ([i32], ctypes.c_char_p),
            "tq_last_cuda_error": ([], i32),
            "tq_wait_timeout_selftest": ([P, P, u32, P, P], i32),
            "tq_kv_cache_bytes": ([i32] * 5, sz),
            "tq_kv_cache_carve": ([C, P, i32, i32, i32, i32, i32], i32),
            "tq_quantize_kv_append": ([C, P, P, i32, P, P, P], i32),
            "tq_sdpa_workspace_bytes": ([i32] * 6, sz),
            "tq_sdpa_int4_decode": ([C, P, i32, P, i32, f32, i32, P, sz, P, P, P], i32),
            "tq_sdpa_int4_decode_impl": ([C, P, i32, P, i32, f32, i32, P, sz, P, P, i32, P], i32),
            "tq_sdpa_plan": ([C, i32, i32, i32, i32, P, P], i32),
            "tq_split_plan": ([i32, i32, i32, i32, i32, i32, i32, P, P], i32),
            "tq_sdpa_int4_partial": ([C, P, i32, P, i32, f32, i32, i32, P, P, P, P, i32, P], i32),
            "tq_sdpa_int4_reduce": ([P, P, P, i32, i32, i32, i32, P, P], i32),
            "tq_sdpa_int4_decode_noalloc": ([C, P, i32, P, i32, f32, i32, P, P, P], i32),
            "tq_decode_step": ([C, P, P, i32, P, P, i32, P, i32, f32, i32, P, sz, P, P, P], i32),
            "tq_dequantize_kv": ([C, i32, P, P, P], i32),
            "tq_quantize_kv_append_ex": ([C, P, P, i32, P, u32, P, P], i32),
            "tq_hadamard_rotate": ([P, ctypes.c_int64, i32, P, P], i32),
            "tq_sdpa_int4_decode_ex": ([C, P, i32, P, i32, f32, i32, u32, P, sz, P, P, P], i32),
            "tq_decode_step_ex": ([C, P, P, i32, P, P, i32, P, i32, f32, i32, u32, P, sz, P, P, P], i32),
            "tq_paged_kv_cache_bytes": ([i32] * 6, sz),
            "tq_paged_kv_cache_carve": ([PC, P, P] + [i32] * 8, i32),
            "tq_kv_cache_bytes_ex": ([i32] * 6, sz),
            "tq_host_staging_bytes": ([i32] * 5, sz),
            "tq_decode_step_host": ([C, P, P, i32, P, P, i32, P, i32, f32, i32, u32, P, sz, P, sz, P, P, P], i32),
            "tq_kv_cache_carve_ex": ([C, P] + [i32] * 6, i32),
            "tq_paged_quantize_kv_append": ([PC, P, P, i32, P, u32, P, P], i32),
            "tq_paged_sdpa_int4_decode": ([PC, P, i32, P, i32, f32, i32, u32, P, sz, P, P, P], i32),
            "tq_paged_decode_step": ([PC, P, P, i32, P, P, i32, P, i32, f32, i32, u32, P, sz, P, P, P], i32),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        if L.tq_abi_version() != 2:
            raise ImportError("libtq.so ABI version mismatch")
        _lib = L
    return _lib


def _check(fn: str, status: int) -> None:
    if status != TQ_OK:
        raise TQError(fn, status)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream: Optional[torch.cuda.Stream]):
    if stream is not None:
        return ctypes.c_void_p(stream.cuda_stream)
    if _raw_stream is not None:  # the current stream's handle without building a Stream object
        return ctypes.c_void_p(_raw_stream(torch.cuda.current_device()))
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _need(t: torch.Tensor, dtype, name: str) -> None:
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous CUDA {dtype} tensor, got {t.dtype} on {t.device}")


# ------------------------------------------------------------------ host-only
def tq_abi_version() -> int:
    return int(lib().tq_abi_version())


def tq_wait_timeout_selftest(src: torch.Tensor, status: torch.Tensor, limit_us: int, copied: torch.Tensor,
                             stream=None) -> None:
    """The bounded-wait diagnostic: a 1 KB copy from ``src`` (uint8, >= 1024
    bytes), then a wait nothing ends, given up after ``limit_us``."""
    _need(src, torch.uint8, "src")
    _need(status, torch.int32, "status")
    _need(copied, torch.int32, "copied")
    if src.numel() < 1024:
        raise ValueError("src must hold at least 1024 bytes")
    _check("tq_wait_timeout_selftest", lib().tq_wait_timeout_selftest(_ptr(src), _ptr(status), int(limit_us),
                                                                      _ptr(copied), _stream(stream)))


def tq_status_string(status: int) -> str:
    return lib().tq_status_string(status).decode()


def tq_kv_cache_bytes(batch: int, num_kv_heads: int, head_dim: int, group_size: int, capacity: int) -> int:
    return int(lib().tq_kv_cache_bytes(batch, num_kv_heads, head_dim, group_size, capacity))


def tq_sdpa_workspace_bytes(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int, max_seq_len: int,
                            chunk: int = DEFAULT_CHUNK) -> int:
    return int(lib().tq_sdpa_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, max_seq_len, chunk))


def workspace(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int, max_seq_len: int,
              chunk: int = DEFAULT_CHUNK, device="cuda") -> torch.Tensor:
    """A decode workspace of tq_sdpa_workspace_bytes bytes (zero-filled)."""
    return torch.zeros(tq_sdpa_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, max_seq_len, chunk),
                       dtype=torch.uint8, device=device)


# ------------------------------------------------------------------ the cache
class KVCache:
    """One layer's int4 cache in a single device allocation (torch uint8).

    Views: k_codes/v_codes uint8 [B, Hkv, cap, D/2]; k_scale/k_bias/v_scale/v_bias
    fp16 [B, Hkv, cap, D/64].  ``struct`` is the tq_kv_cache handed to the ABI.
    """

    def __init__(self, batch: int, num_kv_heads: int, head_dim: int, capacity: int,
                 device=None, group_size: int = GROUP_SIZE, bits: int = 4):
        nbytes = int(lib().tq_kv_cache_bytes_ex(batch, num_kv_heads, head_dim, group_size, bits, capacity))
        if nbytes == 0:
            raise ValueError("invalid cache sizes")
        self.buffer = torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")
        self.struct = tq_kv_cache()
        _check("tq_kv_cache_carve_ex", lib().tq_kv_cache_carve_ex(ctypes.byref(self.struct), _ptr(self.buffer),
                                                                   batch, num_kv_heads, head_dim, group_size, bits,
                                                                   capacity))
        self.batch, self.num_kv_heads, self.head_dim, self.capacity = batch, num_kv_heads, head_dim, capacity
        self.group_size, self.bits = group_size, bits
        base = self.buffer.data_ptr()
        rows = batch * num_kv_heads * capacity
        ng = head_dim // group_size

        def view(addr, n, dtype, shape):
            off = addr - base
            nb = n * torch.empty((), dtype=dtype).element_size()
            return self.buffer[off: off + nb].view(dtype).view(shape)

        cw = head_dim * bits // 8
        cs = (batch, num_kv_heads, capacity, cw)
        ss = (batch, num_kv_heads, capacity, ng)
        s = self.struct
        self.k_codes = view(s.k_codes, rows * cw, torch.uint8, cs)
        self.v_codes = view(s.v_codes, rows * cw, torch.uint8, cs)
        self.k_scale = view(s.k_scale, rows * ng, torch.float16, ss)
        self.k_bias = view(s.k_bias, rows * ng, torch.float16, ss)
        self.v_scale = view(s.v_scale, rows * ng, torch.float16, ss)
        self.v_bias = view(s.v_bias, rows * ng, torch.float16, ss)

    @property
    def nbytes(self) -> int:
        return self.buffer.numel()

    def ref(self):
        return ctypes.byref(self.struct)


class PagedKVCache:
    """A page pool (one device allocation) plus a device block table.

    Views: k_codes/v_codes uint8 [num_pages, Hkv, page_tokens, D/2];
    k_scale/k_bias/v_scale/v_bias fp16 [num_pages, Hkv, page_tokens, D/64];
    block_table int32 [B, max_pages_per_seq] (the caller fills it: page of
    logical page j of sequence b).  Every call of this binding that takes a
    ``KVCache`` takes a ``PagedKVCache`` as well.
    """

    paged = True

    def __init__(self, batch: int, num_kv_heads: int, head_dim: int, page_tokens: int, num_pages: int,
                 max_pages_per_seq: int, device=None, group_size: int = GROUP_SIZE, bits: int = 4):
        nbytes = int(lib().tq_paged_kv_cache_bytes(num_pages, num_kv_heads, head_dim, group_size, bits, page_tokens))
        if nbytes == 0:
            raise ValueError("invalid page pool sizes")
        dev = device or "cuda"
        self.buffer = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.block_table = torch.zeros((batch, max_pages_per_seq), dtype=torch.int32, device=dev)
        self.struct = tq_paged_kv_cache()
        _check("tq_paged_kv_cache_carve", lib().tq_paged_kv_cache_carve(
            ctypes.byref(self.struct), _ptr(self.buffer), _ptr(self.block_table), batch, num_kv_heads, head_dim,
            group_size, bits, page_tokens, num_pages, max_pages_per_seq))
        self.batch, self.num_kv_heads, self.head_dim = batch, num_kv_heads, head_dim
        self.page_tokens, self.num_pages, self.max_pages_per_seq = page_tokens, num_pages, max_pages_per_seq
        self.capacity = page_tokens * max_pages_per_seq
        self.group_size, self.bits = group_size, bits
        base = self.buffer.data_ptr()
        rows = num_pages * num_kv_heads * page_tokens
        ng = head_dim // group_size

        def view(addr, n, dtype, shape):
            off = addr - base
            nb = n * torch.empty((), dtype=dtype).element_size()
            return self.buffer[off: off + nb].view(dtype).view(shape)

        cw = head_dim * bits // 8
        cs = (num_pages, num_kv_heads, page_tokens, cw)
        ss = (num_pages, num_kv_heads, page_tokens, ng)
        st = self.struct
        self.k_codes = view(st.k_codes, rows * cw, torch.uint8, cs)
        self.v_codes = view(st.v_codes, rows * cw, torch.uint8, cs)
        self.k_scale = view(st.k_scale, rows * ng, torch.float16, ss)
        self.k_bias = view(st.k_bias, rows * ng, torch.float16, ss)
        self.v_scale = view(st.v_scale, rows * ng, torch.float16, ss)
        self.v_bias = view(st.v_bias, rows * ng, torch.float16, ss)

    def ref(self):
        return ctypes.byref(self.struct)


# ------------------------------------------------------------------ device ops
def tq_quantize_kv_append(cache: KVCache, k_new: torch.Tensor, v_new: torch.Tensor, write_pos: torch.Tensor,
                          status: Optional[torch.Tensor] = None, stream=None, flags: int = 0) -> None:
    """Quantize k_new/v_new [B, Hkv, n_new, D] fp16 into cache rows write_pos[b] + i
    (flags TQ_ROTATE_K / TQ_ROTATE_V: Hadamard-rotate the rows first)."""
    _need(k_new, torch.float16, "k_new")
    _need(v_new, torch.float16, "v_new")
    _need(write_pos, torch.int32, "write_pos")
    if status is not None:
        _need(status, torch.int32, "status")
    n_new = k_new.shape[2] if k_new.dim() == 4 else 0
    if tuple(k_new.shape) != (cache.batch, cache.num_kv_heads, n_new, cache.head_dim) or v_new.shape != k_new.shape:
        raise ValueError(f"k_new/v_new must be [B, Hkv, n_new, D]; got {tuple(k_new.shape)}")
    if getattr(cache, "paged", False):
        _check("tq_paged_quantize_kv_append", lib().tq_paged_quantize_kv_append(
            cache.ref(), _ptr(k_new), _ptr(v_new), n_new, _ptr(write_pos), int(flags), _ptr(status), _stream(stream)))
        return
    if flags:
        _check("tq_quantize_kv_append_ex", lib().tq_quantize_kv_append_ex(
            cache.ref(), _ptr(k_new), _ptr(v_new), n_new, _ptr(write_pos), int(flags), _ptr(status), _stream(stream)))
        return
    _check("tq_quantize_kv_append", lib().tq_quantize_kv_append(cache.ref(), _ptr(k_new), _ptr(v_new), n_new,
                                                                _ptr(write_pos), _ptr(status), _stream(stream)))


def tq_sdpa_int4_decode(cache: KVCache, q: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                        attn_scale: float, workspace: torch.Tensor, out: Optional[torch.Tensor] = None,
                        chunk: int = DEFAULT_CHUNK, status: Optional[torch.Tensor] = None,
                        impl: int = TQ_IMPL_AUTO, stream=None, flags: int = 0) -> torch.Tensor:
    """Fused int4 decode attention; q [B, Hq, D] fp16 -> out [B, Hq, D] fp16
    (flags: the rotation flags the cache was written with)."""
    _need(q, torch.float16, "q")
    _need(seq_lens, torch.int32, "seq_lens")
    _need(workspace, torch.uint8, "workspace")
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.float16, "out")
    if status is not None:
        _need(status, torch.int32, "status")
    if q.dim() != 3 or q.shape[0] != cache.batch or q.shape[2] != cache.head_dim or out.shape != q.shape:
        raise ValueError(f"q must be [B, Hq, D]; got {tuple(q.shape)}")
    if getattr(cache, "paged", False):
        if impl == TQ_IMPL_SIMT:
            raise ValueError("a paged cache takes the tensor-core implementation")
        _check("tq_paged_sdpa_int4_decode", lib().tq_paged_sdpa_int4_decode(
            cache.ref(), _ptr(q), q.shape[1], _ptr(seq_lens), int(max_seq_len), float(attn_scale), int(chunk),
            int(flags), _ptr(workspace), workspace.numel(), _ptr(out), _ptr(status), _stream(stream)))
        return out
    if flags:
        if impl != TQ_IMPL_AUTO:
            raise ValueError("rotation flags take the default implementation")
        _check("tq_sdpa_int4_decode_ex", lib().tq_sdpa_int4_decode_ex(
            cache.ref(), _ptr(q), q.shape[1], _ptr(seq_lens), int(max_seq_len), float(attn_scale), int(chunk),
            int(flags), _ptr(workspace), workspace.numel(), _ptr(out), _ptr(status), _stream(stream)))
        return out
    _check("tq_sdpa_int4_decode", lib().tq_sdpa_int4_decode_impl(
        cache.ref(), _ptr(q), q.shape[1], _ptr(seq_lens), int(max_seq_len), float(attn_scale), int(chunk),
        _ptr(workspace), workspace.numel(), _ptr(out), _ptr(status), int(impl), _stream(stream)))
    return out


def tq_decode_step(cache: KVCache, k_new: torch.Tensor, v_new: torch.Tensor, write_pos: torch.Tensor,
                   q: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int, attn_scale: float,
                   workspace: torch.Tensor, out: Optional[torch.Tensor] = None, chunk: int = DEFAULT_CHUNK,
                   status: Optional[torch.Tensor] = None, stream=None, flags: int = 0) -> torch.Tensor:
    """Append k_new/v_new [B, Hkv, n_new, D] at write_pos, then decode q [B, Hq, D]
    over seq_lens (which must already count the new tokens); flags: rotation."""
    for t, n, dt in ((k_new, "k_new", torch.float16), (v_new, "v_new", torch.float16), (q, "q", torch.float16),
                     (write_pos, "write_pos", torch.int32), (seq_lens, "seq_lens", torch.int32),
                     (workspace, "workspace", torch.uint8)):
        _need(t, dt, n)
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.float16, "out")
    if status is not None:
        _need(status, torch.int32, "status")
    n_new = k_new.shape[2] if k_new.dim() == 4 else 0
    if tuple(k_new.shape) != (cache.batch, cache.num_kv_heads, n_new, cache.head_dim) or v_new.shape != k_new.shape:
        raise ValueError(f"k_new/v_new must be [B, Hkv, n_new, D]; got {tuple(k_new.shape)}")
    if q.dim() != 3 or q.shape[0] != cache.batch or q.shape[2] != cache.head_dim or out.shape != q.shape:
        raise ValueError(f"q must be [B, Hq, D]; got {tuple(q.shape)}")
    if getattr(cache, "paged", False):
        _check("tq_paged_decode_step", lib().tq_paged_decode_step(
            cache.ref(), _ptr(k_new), _ptr(v_new), n_new, _ptr(write_pos), _ptr(q), q.shape[1], _ptr(seq_lens),
            int(max_seq_len), float(attn_scale), int(chunk), int(flags), _ptr(workspace), workspace.numel(),
            _ptr(out), _ptr(status), _stream(stream)))
        return out
    if flags:
        _check("tq_decode_step_ex", lib().tq_decode_step_ex(
            cache.ref(), _ptr(k_new), _ptr(v_new), n_new, _ptr(write_pos), _ptr(q), q.shape[1], _ptr(seq_lens),
            int(max_seq_len), float(attn_scale), int(chunk), int(flags), _ptr(workspace), workspace.numel(),
            _ptr(out), _ptr(status), _stream(stream)))
        return out
    _check("tq_decode_step", lib().tq_decode_step(
        cache.ref(), _ptr(k_new), _ptr(v_new), n_new, _ptr(write_pos), _ptr(q), q.shape[1], _ptr(seq_lens),
        int(max_seq_len), float(attn_scale), int(chunk), _ptr(workspace), workspace.numel(), _ptr(out),
        _ptr(status), _stream(stream)))
    return out


def tq_sdpa_plan(cache: KVCache, num_q_heads: int, max_seq_len: int, chunk: int = DEFAULT_CHUNK,
                 impl: int = TQ_IMPL_AUTO):
    """(n_splits, max_run_tokens) of the runs tq_sdpa_int4_decode uses on this device."""
    ns, run = ctypes.c_int32(0), ctypes.c_int32(0)
    _check("tq_sdpa_plan", lib().tq_sdpa_plan(cache.ref(), num_q_heads, int(max_seq_len), int(chunk), int(impl),
                                              ctypes.byref(ns), ctypes.byref(run)))
    return ns.value, run.value


def tq_split_plan(batch: int, num_kv_heads: int, max_seq_len: int, chunk: int, tile_tokens: int,
                  resident_ctas: int, merge: bool = True):
    """(n_splits, max_run_tokens) of the split rule for a device holding
    ``resident_ctas`` phase-1 CTAs at once (host arithmetic, no device);
    ``merge``: the decode may merge its runs itself (no reduce)."""
    ns, run = ctypes.c_int32(0), ctypes.c_int32(0)
    _check("tq_split_plan", lib().tq_split_plan(int(batch), int(num_kv_heads), int(max_seq_len), int(chunk),
                                                int(tile_tokens), int(resident_ctas), int(bool(merge)),
                                                ctypes.byref(ns), ctypes.byref(run)))
    return ns.value, run.value


def tq_sdpa_int4_partial(cache: KVCache, q: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                         attn_scale: float, chunk: int = DEFAULT_CHUNK, chunks_per_split: int = 1,
                         status: Optional[torch.Tensor] = None, impl: int = TQ_IMPL_AUTO, stream=None,
                         out=None):
    """Phase 1 alone: (m, l, acc) fp32 per part of ``chunks_per_split`` chunks
    (1 = per chunk; 0 = the runs tq_sdpa_int4_decode uses), m in natural-log units."""
    _need(q, torch.float16, "q")
    _need(seq_lens, torch.int32, "seq_lens")
    B, Hq, D = q.shape
    nc = max(1, math.ceil(max_seq_len / chunk))
    if chunks_per_split > 0:
        n_parts = math.ceil(nc / chunks_per_split)
    else:
        n_parts = tq_sdpa_plan(cache, Hq, max_seq_len, chunk, impl)[0]
    if out is None:
        m = torch.empty((B, Hq, n_parts), dtype=torch.float32, device=q.device)
        l = torch.empty_like(m)
        acc = torch.empty((B, Hq, n_parts, D), dtype=torch.float32, device=q.device)
    else:
        m, l, acc = out
        if m.numel() < B * Hq * n_parts or acc.numel() < B * Hq * n_parts * D:
            raise ValueError("partial output buffers too small")
    _check("tq_sdpa_int4_partial", lib().tq_sdpa_int4_partial(
        cache.ref(), _ptr(q), Hq, _ptr(seq_lens), int(max_seq_len), float(attn_scale), int(chunk),
        int(chunks_per_split),
        _ptr(m), _ptr(l), _ptr(acc), _ptr(status), int(impl), _stream(stream)))
    return m, l, acc


def tq_sdpa_int4_reduce(m: torch.Tensor, l: torch.Tensor, acc: torch.Tensor, out: Optional[torch.Tensor] = None,
                        stream=None) -> torch.Tensor:
    """Phase 2 alone: LSE merge of [B, Hq, n] partials -> fp16 [B, Hq, D]."""
    for t, n in ((m, "m"), (l, "l"), (acc, "acc")):
        _need(t, torch.float32, n)
    B, Hq, n, D = acc.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float16, device=acc.device)
    _need(out, torch.float16, "out")
    _check("tq_sdpa_int4_reduce", lib().tq_sdpa_int4_reduce(_ptr(m), _ptr(l), _ptr(acc), B, Hq, D, n, _ptr(out),
                                                            _stream(stream)))
    return out


def tq_sdpa_int4_decode_noalloc(cache: KVCache, q: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                                attn_scale: float, out: Optional[torch.Tensor] = None, chunk: int = DEFAULT_CHUNK,
                                status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """tq_sdpa_int4_decode without a workspace: the partial states live in a
    fixed 4 MiB device array owned by the library (for callers that cannot
    allocate).  Calls that overlap on the GPU share that array and race."""
    _need(q, torch.float16, "q")
    _need(seq_lens, torch.int32, "seq_lens")
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.float16, "out")
    if status is not None:
        _need(status, torch.int32, "status")
    if q.dim() != 3 or q.shape[0] != cache.batch or q.shape[2] != cache.head_dim or out.shape != q.shape:
        raise ValueError(f"q must be [B, Hq, D]; got {tuple(q.shape)}")
    _check("tq_sdpa_int4_decode_noalloc", lib().tq_sdpa_int4_decode_noalloc(
        cache.ref(), _ptr(q), q.shape[1], _ptr(seq_lens), int(max_seq_len), float(attn_scale), int(chunk),
        _ptr(out), _ptr(status), _stream(stream)))
    return out


def tq_dequantize_kv(cache: KVCache, n_rows: int, out=None, stream=None):
    """fp16 K and V [B, Hkv, n_rows, D] of rows [0, n_rows) of the cache:
    fp16_rne(fp32(scale * code + bias)).  The float cache of the
    dequantize-then-attend comparison path; the fused decode never uses it."""
    shape = (cache.batch, cache.num_kv_heads, int(n_rows), cache.head_dim)
    if out is None:
        dev = cache.buffer.device
        out = (torch.empty(shape, dtype=torch.float16, device=dev), torch.empty(shape, dtype=torch.float16, device=dev))
    k, v = out
    for t, n in ((k, "k_out"), (v, "v_out")):
        _need(t, torch.float16, n)
        if tuple(t.shape) != shape:
            raise ValueError(f"{n} must be {shape}; got {tuple(t.shape)}")
    _check("tq_dequantize_kv", lib().tq_dequantize_kv(cache.ref(), int(n_rows), _ptr(k), _ptr(v), _stream(stream)))
    return k, v


def tq_hadamard_rotate(x: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """fp16 rows [..., D] (D = 64, 128, 256) -> fp16_rne(H x) per row, H the
    normalised Sylvester Hadamard matrix (out may be x)."""
    _need(x, torch.float16, "x")
    if out is None:
        out = torch.empty_like(x)
    _need(out, torch.float16, "out")
    if out.shape != x.shape:
        raise ValueError("out must have the shape of x")
    dim = x.shape[-1]
    _check("tq_hadamard_rotate", lib().tq_hadamard_rotate(_ptr(x), x.numel() // dim, dim, _ptr(out),
                                                          _stream(stream)))
    return out


def tq_host_staging_bytes(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int, n_new: int) -> int:
    return int(lib().tq_host_staging_bytes(batch, num_q_heads, num_kv_heads, head_dim, n_new))


def _need_host(t: torch.Tensor, name: str) -> None:
    if t.is_cuda or t.dtype != torch.float16 or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous host float16 tensor (pinned for asynchronous copies)")


def tq_decode_step_host(cache: KVCache, h_k_new: torch.Tensor, h_v_new: torch.Tensor, write_pos: torch.Tensor,
                        h_q: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int, attn_scale: float,
                        workspace: torch.Tensor, staging: torch.Tensor, h_out: torch.Tensor,
                        chunk: int = DEFAULT_CHUNK, flags: int = 0, status: Optional[torch.Tensor] = None,
                        stream=None) -> torch.Tensor:
    """tq_decode_step with q / k_new / v_new / out in host memory: the copies and
    the step are queued by one library call; h_out is valid once the stream
    has reached it."""
    for t, n in ((h_k_new, "h_k_new"), (h_v_new, "h_v_new"), (h_q, "h_q"), (h_out, "h_out")):
        _need_host(t, n)
    for t, n, dt in ((write_pos, "write_pos", torch.int32), (seq_lens, "seq_lens", torch.int32),
                     (workspace, "workspace", torch.uint8), (staging, "staging", torch.uint8)):
        _need(t, dt, n)
    n_new = h_k_new.shape[2] if h_k_new.dim() == 4 else 0
    _check("tq_decode_step_host", lib().tq_decode_step_host(
        cache.ref(), _ptr(h_k_new), _ptr(h_v_new), n_new, _ptr(write_pos), _ptr(h_q), h_q.shape[1], _ptr(seq_lens),
        int(max_seq_len), float(attn_scale), int(chunk), int(flags), _ptr(workspace), workspace.numel(),
        _ptr(staging), staging.numel(), _ptr(h_out), _ptr(status), _stream(stream)))
    return h_out
