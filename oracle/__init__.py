"""CPU oracle for int4 KV-cache quantize-on-store and fused decode attention.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product library never
imports this package, and this package never imports the product.

Thin ctypes marshalling over ``tq_oracle.c`` (plain C, fp64 accumulation);
every arithmetic step lives in the C file, which cites the pages it restates.
"""
from __future__ import annotations

import ctypes
import math
from typing import Optional, Sequence, Tuple

import numpy as np

_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        from . import build as _build

        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i64, i32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        L.tqo_f32_to_f16.argtypes = [ctypes.c_float]
        L.tqo_f32_to_f16.restype = ctypes.c_uint16
        L.tqo_f16_to_f64.argtypes = [ctypes.c_uint16]
        L.tqo_f16_to_f64.restype = f64
        L.tqo_f32_to_f16_array.argtypes = [P, i64, P]
        L.tqo_f16_to_f64_array.argtypes = [P, i64, P]
        L.tqo_quantize_group.argtypes = [P, i32, P, P, P]
        L.tqo_quantize_rows.argtypes = [P, i64, i32, i32, P, P, P]
        L.tqo_dequantize_rows.argtypes = [P, P, P, i64, i32, i32, P]
        L.tqo_dequantize_rows_f16.argtypes = [P, P, P, i64, i32, i32, P]
        L.tqo_hadamard_f64.argtypes = [P, i32]
        L.tqo_quantize_group_b.argtypes = [P, i32, i32, P, P, P]
        L.tqo_quantize_rows_b.argtypes = [P, i64, i32, i32, i32, P, P, P]
        L.tqo_dequantize_rows_b.argtypes = [P, P, P, i64, i32, i32, i32, P]
        L.tqo_dequantize_rows_f16_b.argtypes = [P, P, P, i64, i32, i32, i32, P]
        L.tqo_attention_b.argtypes = [P, i32, i32, i32, i32, i32, i64, P, P, P, P, P, P, P, f64, P, i64, i32, P]
        L.tqo_hadamard_f32.argtypes = [P, i32]
        L.tqo_rotate_rows_f16.argtypes = [P, i64, i32, P]
        L.tqo_attention.argtypes = [P, i32, i32, i32, i32, i32, i64, P, P, P, P, P, P, P, f64,
                                    P, i64, P]
        L.tqo_attention_partials.argtypes = [P, i32, i32, i32, i32, i32, i64, P, P, P, P, P, P,
                                             P, f64, i32, i32, P, P, P]
        L.tqo_attention_partials_b.argtypes = [P, i32, i32, i32, i32, i32, i64, P, P, P, P, P, P,
                                               P, f64, i32, i32, i32, P, P, P]
        L.tqo_merge_partials.argtypes = [P, P, P, i32, i32, i32, i32, P]
        L.tqo_num_threads.restype = i32
        _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def _bits16(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    assert a.dtype == np.uint16, a.dtype
    return a


def num_threads() -> int:
    return int(lib().tqo_num_threads())


def f32_to_f16(x: np.ndarray) -> np.ndarray:
    """IEEE binary32 -> binary16 bits (RNE), oracle codec."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().tqo_f32_to_f16_array(_ptr(x), x.size, _ptr(out))
    return out


def f16_to_f64(h: np.ndarray) -> np.ndarray:
    """binary16 bits -> float64, oracle codec."""
    h = _bits16(h)
    out = np.empty(h.shape, dtype=np.float64)
    lib().tqo_f16_to_f64_array(_ptr(h), h.size, _ptr(out))
    return out


def quantize_group(x: np.ndarray, bits: int = 4) -> Tuple[np.ndarray, int, int]:
    """One group -> (unpacked codes uint8[n], scale bits, bias bits); bits 4 or 8."""
    x = _bits16(x).ravel()
    codes = np.empty(x.size, dtype=np.uint8)
    s = np.zeros(1, dtype=np.uint16)
    b = np.zeros(1, dtype=np.uint16)
    lib().tqo_quantize_group_b(_ptr(x), x.size, int(bits), _ptr(codes), _ptr(s), _ptr(b))
    return codes, int(s[0]), int(b[0])


def quantize_rows(x: np.ndarray, group: int = 64, bits: int = 4):
    """x[..., D] fp16 -> (codes uint8[..., D*bits/8], scale u16[..., D/g], bias u16[..., D/g])."""
    x = _bits16(x)
    D = x.shape[-1]
    assert D % group == 0 and D % 2 == 0 and D <= 1024 and bits in (4, 8)
    rows = x.size // D
    codes = np.empty(x.shape[:-1] + (D * bits // 8,), dtype=np.uint8)
    scale = np.empty(x.shape[:-1] + (D // group,), dtype=np.uint16)
    bias = np.empty_like(scale)
    lib().tqo_quantize_rows_b(_ptr(x), rows, D, group, int(bits), _ptr(codes), _ptr(scale), _ptr(bias))
    return codes, scale, bias


def dequantize_rows(codes: np.ndarray, scale: np.ndarray, bias: np.ndarray, group: int = 64, bits: int = 4):
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scale, bias = _bits16(scale), _bits16(bias)
    D = codes.shape[-1] * 8 // bits
    rows = codes.size // (D * bits // 8)
    out = np.empty(codes.shape[:-1] + (D,), dtype=np.float64)
    lib().tqo_dequantize_rows_b(_ptr(codes), _ptr(scale), _ptr(bias), rows, D, group, int(bits), _ptr(out))
    return out


def dequantize_rows_f16(codes: np.ndarray, scale: np.ndarray, bias: np.ndarray, group: int = 64, bits: int = 4):
    """fp16 bits [.., D] of fp16_rne(fp32(scale * code + bias)) per element."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scale, bias = _bits16(scale), _bits16(bias)
    D = codes.shape[-1] * 8 // bits
    rows = codes.size // (D * bits // 8)
    out = np.empty(codes.shape[:-1] + (D,), dtype=np.uint16)
    lib().tqo_dequantize_rows_f16_b(_ptr(codes), _ptr(scale), _ptr(bias), rows, D, group, int(bits), _ptr(out))
    return out


def hadamard(x: np.ndarray) -> np.ndarray:
    """(1/sqrt(n)) H_n x along the last axis: float64 in, float64 out; float32 in,
    the fp32 fast transform out."""
    x = np.array(x, copy=True, order="C")
    n = x.shape[-1]
    fn = lib().tqo_hadamard_f32 if x.dtype == np.float32 else lib().tqo_hadamard_f64
    if x.dtype not in (np.float32, np.float64):
        x = x.astype(np.float64)
        fn = lib().tqo_hadamard_f64
    flat = x.reshape(-1, n)
    for r in range(flat.shape[0]):
        fn(flat[r].ctypes.data_as(ctypes.c_void_p), n)
    return x


def rotate_rows_f16(x: np.ndarray) -> np.ndarray:
    """fp16 rows rotated by the fp32 transform, rounded to fp16 (same shape, float16)."""
    xb = _bits16(np.asarray(x))
    n = xb.shape[-1]
    out = np.empty_like(xb)
    lib().tqo_rotate_rows_f16(_ptr(xb), xb.size // n, n, _ptr(out))
    return out.view(np.float16)


class Cache:
    """A quantised cache as plain host arrays (oracle side).

    codes: [B, Hkv, cap, D * bits / 8] uint8 (bits 4: two codes per byte; 8: one);
    scale/bias: [B, Hkv, cap, D/group] u16.
    """

    def __init__(self, kc, ks, kb, vc, vs, vb, group: int = 64, bits: int = 4):
        self.kc = np.ascontiguousarray(kc, dtype=np.uint8)
        self.vc = np.ascontiguousarray(vc, dtype=np.uint8)
        self.ks, self.kb = _bits16(ks), _bits16(kb)
        self.vs, self.vb = _bits16(vs), _bits16(vb)
        self.group, self.bits = group, bits
        self.B, self.Hkv, self.cap = self.kc.shape[:3]
        self.D = self.kc.shape[3] * 8 // bits

    @classmethod
    def from_fp16(cls, k: np.ndarray, v: np.ndarray, group: int = 64, bits: int = 4) -> "Cache":
        kc, ks, kb = quantize_rows(k, group, bits)
        vc, vs, vb = quantize_rows(v, group, bits)
        return cls(kc, ks, kb, vc, vs, vb, group, bits)

    def _args(self):
        return (_ptr(self.kc), _ptr(self.ks), _ptr(self.kb), _ptr(self.vc), _ptr(self.vs),
                _ptr(self.vb))


def attention(q: np.ndarray, cache: Cache, lens: np.ndarray, attn_scale: float,
              pairs: Optional[Sequence[Tuple[int, int]]] = None) -> np.ndarray:
    """fp64 decode attention, out[B, Hq, D] (rows not in ``pairs`` are NaN)."""
    q = _bits16(q)
    B, Hq, D = q.shape
    assert B == cache.B and D == cache.D and Hq % cache.Hkv == 0
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    assert lens.shape == (B,) and int(lens.max(initial=0)) <= cache.cap and int(lens.min(initial=0)) >= 0
    out = np.full((B, Hq, D), np.nan, dtype=np.float64)
    if pairs is None:
        pp, n = None, 0
    else:
        arr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
        pp, n = _ptr(arr), arr.shape[0]
    lib().tqo_attention_b(_ptr(q), B, Hq, cache.Hkv, D, cache.group, cache.cap, *cache._args(),
                          _ptr(lens), float(attn_scale), pp, n, int(cache.bits), _ptr(out))
    return out


def attention_partials(q: np.ndarray, cache: Cache, lens: np.ndarray, attn_scale: float,
                       chunk: int, n_chunks: Optional[int] = None):
    """Per-chunk (m, l, acc): m[B,Hq,nc], l[B,Hq,nc], acc[B,Hq,nc,D]."""
    q = _bits16(q)
    B, Hq, D = q.shape
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    if n_chunks is None:
        n_chunks = max(1, math.ceil(int(lens.max(initial=0)) / chunk))
    m = np.empty((B, Hq, n_chunks))
    l = np.empty((B, Hq, n_chunks))
    acc = np.empty((B, Hq, n_chunks, D))
    a = cache._args()
    lib().tqo_attention_partials_b(_ptr(q), B, Hq, cache.Hkv, D, cache.group, cache.cap, *a,
                                   _ptr(lens), float(attn_scale), chunk, n_chunks, int(cache.bits), _ptr(m),
                                   _ptr(l), _ptr(acc))
    return m, l, acc


def merge_partials(m: np.ndarray, l: np.ndarray, acc: np.ndarray) -> np.ndarray:
    m = np.ascontiguousarray(m, dtype=np.float64)
    l = np.ascontiguousarray(l, dtype=np.float64)
    acc = np.ascontiguousarray(acc, dtype=np.float64)
    B, Hq, nc, D = acc.shape
    out = np.empty((B, Hq, D))
    lib().tqo_merge_partials(_ptr(m), _ptr(l), _ptr(acc), B, Hq, D, nc, _ptr(out))
    return out
