"""Seeded synthetic inputs for the int4 KV-cache decode path.

This module holds no quantisation and no attention arithmetic.  It only draws
random numbers and shapes them the way the workloads on the pages look:

* Llama-3.1-70B single-layer decode shape (64 query heads, 8 KV heads,
  head_dim 128) -- "Llama 3.1 70B" page, kernel latency table;
* Gemma-style unscaled attention (attn_scale = 1.0, Q/K normalised per head)
  -- "Fused int4 Attention for Gemma 4 31B", Background and Performance;
* a batch of ragged sequences that append one token per step.

Both the CUDA path (tests, bench) and the CPU oracle are fed from here, so the
two sides always see the same fp16 bytes.

Recipe (one place, so that tests and bench agree):
  * every array is drawn as float32 N(0, 1) from ``numpy.random.default_rng``
    (PCG64) seeded with the workload seed, then rounded to fp16 (RNE);
  * order of draws: Q, then K, then V, each in C order of its shape;
  * "outliers": round(0.01 * D) head_dim channels per KV head (1 at D = 128),
    chosen with ``rng.choice`` (no replacement) after V is drawn, multiplied
    by 20 in float32 before the fp16 rounding, for every token of that head;
  * "rms_qk": Q and K rows are divided by sqrt(mean(x^2)) in float32 before
    the fp16 rounding (unit RMS per head vector, eps 0);
  * ragged lengths: ``rng.integers(lo, hi + 1)`` from a generator seeded
    with the workload seed + 1000003.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

__all__ = [
    "DecodeInputs",
    "decode_inputs",
    "ragged_lengths",
    "append_tokens",
    "WORKLOADS",
    "Workload",
    "FULL_MODEL_LAYERS",
    "FULL_MODEL_SEED0",
    "full_model_layer",
]


@dataclasses.dataclass
class DecodeInputs:
    """fp16 tensors (numpy float16) of one synthetic decode problem.

    q: [B, Hq, D] query of the single decode token (Sq = 1)
    k, v: [B, Hkv, S, D] keys / values of the cached tokens
    lens: [B] int32 per-sequence KV lengths (<= S)
    outlier_channels: [Hkv] channel index scaled x20 in K, or None
    """

    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    lens: np.ndarray
    outlier_channels: Optional[np.ndarray]


def _rms_rows(x: np.ndarray) -> np.ndarray:
    # unit RMS per last-axis vector, float32, eps 0 (workload shaping only)
    x = x.astype(np.float32, copy=False)
    r = np.sqrt(np.mean(x * x, axis=-1, keepdims=True, dtype=np.float32))
    return x / r


def decode_inputs(
    seed: int,
    batch: int,
    num_q_heads: int,
    num_kv_heads: int,
    head_dim: int,
    seq_len: int,
    *,
    outliers: bool = False,
    rms_qk: bool = False,
    lens: Optional[np.ndarray] = None,
) -> DecodeInputs:
    """Draw Q, K, V for one decode problem (see the module recipe)."""
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((batch, num_q_heads, head_dim), dtype=np.float32)
    k = rng.standard_normal((batch, num_kv_heads, seq_len, head_dim), dtype=np.float32)
    v = rng.standard_normal((batch, num_kv_heads, seq_len, head_dim), dtype=np.float32)
    chans = None
    if outliers:
        n_out = max(1, int(round(0.01 * head_dim)))
        chans = np.stack([rng.choice(head_dim, size=n_out, replace=False) for _ in range(num_kv_heads)])
        for h in range(num_kv_heads):
            for c in chans[h]:
                k[:, h, :, c] *= np.float32(20.0)
        chans = chans[:, 0].astype(np.int64) if n_out == 1 else chans
    if rms_qk:
        q = _rms_rows(q)
        k = _rms_rows(k)
    if lens is None:
        lens = np.full((batch,), seq_len, dtype=np.int32)
    return DecodeInputs(
        q=q.astype(np.float16),
        k=k.astype(np.float16),
        v=v.astype(np.float16),
        lens=np.asarray(lens, dtype=np.int32),
        outlier_channels=chans,
    )


def ragged_lengths(seed: int, n: int, lo: int, hi: int) -> np.ndarray:
    """Per-sequence lengths uniform in [lo, hi] (inclusive), int32."""
    rng = np.random.default_rng(seed + 1000003)
    return rng.integers(lo, hi + 1, size=n).astype(np.int32)


def append_tokens(seed: int, step: int, batch: int, num_kv_heads: int, head_dim: int,
                  n_new: int = 1, *, outliers: Optional[np.ndarray] = None):
    """K/V of ``n_new`` new tokens per sequence for decode step ``step``.

    Returns (k_new, v_new) fp16 of shape [B, Hkv, n_new, D].  ``outliers`` (one
    channel per KV head) reuses the channels of the cached K so that appended
    keys look like the cached ones.
    """
    rng = np.random.default_rng([seed, 7919, step])
    k = rng.standard_normal((batch, num_kv_heads, n_new, head_dim), dtype=np.float32)
    v = rng.standard_normal((batch, num_kv_heads, n_new, head_dim), dtype=np.float32)
    if outliers is not None:
        for h in range(num_kv_heads):
            k[:, h, :, int(np.atleast_1d(outliers[h])[0])] *= np.float32(20.0)
    return k.astype(np.float16), v.astype(np.float16)


@dataclasses.dataclass(frozen=True)
class Workload:
    """A named synthetic workload (shapes + input recipe)."""

    name: str
    seed: int
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    seq_len: int
    attn_scale: float
    outliers: bool = False
    rms_qk: bool = False
    chunk: int = 512

    def draw(self, lens: Optional[np.ndarray] = None) -> DecodeInputs:
        return decode_inputs(self.seed, self.batch, self.num_q_heads, self.num_kv_heads,
                             self.head_dim, self.seq_len, outliers=self.outliers,
                             rms_qk=self.rms_qk, lens=lens)


_LLAMA_SCALE = 1.0 / float(np.sqrt(128.0))

WORKLOADS = {
    # tiny decode: one 512-token chunk holds the whole sequence
    "tiny": Workload("tiny", 1, 1, 8, 2, 128, 256, _LLAMA_SCALE),
    # Llama-3.1-70B single layer: 64 q heads / 8 kv heads, head_dim 128
    **{f"llama70b_{n // 1024}k": Workload(f"llama70b_{n // 1024}k", 2, 1, 64, 8, 128, n,
                                          _LLAMA_SCALE, outliers=True)
       for n in (1024, 16384, 65536, 131072)},
    # Gemma-style: attn_scale 1.0, Q/K unit RMS, head_dim 256, 32 q / 16 kv heads
    **{f"gemma_{n}": Workload(f"gemma_{n}", 3, 1, 32, 16, 256, n, 1.0, rms_qk=True)
       for n in (33, 423, 786, 950)},
    # ragged batch of 32 sequences, lengths uniform in [1K, 32K]
    "ragged32": Workload("ragged32", 4, 32, 64, 8, 128, 32768, _LLAMA_SCALE, outliers=True),
}

# The full model at 128K: FULL_MODEL_LAYERS caches of the Llama-70B layer,
# layer l drawn by torch_decode_inputs with seed FULL_MODEL_SEED0 + l; one
# decode step appends the same new token (append_tokens(FULL_MODEL_SEED0, 0),
# outlier channels of layer 0) at row 131071 of every layer, then decodes it.
FULL_MODEL_LAYERS = 80
FULL_MODEL_SEED0 = 5


def full_model_layer(layer: int, device="cuda"):
    """(q, k, v, outlier_channels) of one layer of the full-model workload."""
    w = WORKLOADS["llama70b_128k"]
    return torch_decode_inputs(FULL_MODEL_SEED0 + layer, w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim,
                               w.seq_len, outliers=True, device=device)


def torch_decode_inputs(seed: int, batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                        seq_len: int, *, outliers: bool = False, rms_qk: bool = False, device="cuda"):
    """Same recipe as ``decode_inputs`` drawn on the device with torch's
    seeded generator (different numbers than numpy, same distributions).

    Used where the host generator would be too slow (hundreds of millions of
    elements); a test that needs the oracle copies the fp16 tensors to the host.
    Returns (q, k, v, outlier_channels) with fp16 tensors on ``device``.
    """
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed)
    q = torch.randn((batch, num_q_heads, head_dim), generator=g, device=device, dtype=torch.float32)
    k = torch.randn((batch, num_kv_heads, seq_len, head_dim), generator=g, device=device, dtype=torch.float32)
    v = torch.randn((batch, num_kv_heads, seq_len, head_dim), generator=g, device=device, dtype=torch.float32)
    chans = None
    if outliers:
        chans = np.random.default_rng(seed).integers(0, head_dim, size=num_kv_heads)
        for h in range(num_kv_heads):
            k[:, h, :, int(chans[h])] *= 20.0
    if rms_qk:
        q = q / torch.sqrt(torch.mean(q * q, dim=-1, keepdim=True))
        k = k / torch.sqrt(torch.mean(k * k, dim=-1, keepdim=True))
    return q.half(), k.half(), v.half(), chans
