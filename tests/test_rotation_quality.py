"""What the rotation is for ("Running and Evaluating TurboQuant optimized
Gemma 4", TurboQuant section: the Hadamard rotation spreads extreme outliers so
that quantisation loses less).  CPU only, oracle arithmetic: with one K channel
x20 per kv head, int4 attention over rotated keys (and the rotated query) is
closer to fp64 attention over the unquantized cache than int4 attention over
the keys as they are."""
import numpy as np

import oracle
from int4_kv_cache_gb300 import synth


def _exact_attention(q, k, v, scale):
    """fp64 softmax attention over float K/V (GQA by consecutive heads)."""
    B, Hq, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    out = np.empty((B, Hq, D))
    for b in range(B):
        for h in range(Hq):
            s = scale * (k[b, h // G] @ q[b, h])
            p = np.exp(s - s.max())
            out[b, h] = (p / p.sum()) @ v[b, h // G]
    return out


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def test_rotation_reduces_error_with_outlier_channels():
    x = synth.decode_inputs(91, 1, 16, 2, 128, 2048, outliers=True)
    scale = 1.0 / np.sqrt(128)
    q64, k64, v64 = (a.astype(np.float64) for a in (x.q, x.k, x.v))
    exact = _exact_attention(q64, k64, v64, scale)
    plain = oracle.attention(x.q, oracle.Cache.from_fp16(x.k, x.v), x.lens, scale)
    kr = oracle.rotate_rows_f16(x.k)
    qr = oracle.rotate_rows_f16(x.q)
    rotated = oracle.attention(qr, oracle.Cache.from_fp16(kr, x.v), x.lens, scale)
    e_plain, e_rot = _rel(plain, exact), _rel(rotated, exact)
    assert e_rot < 0.5 * e_plain, (e_plain, e_rot)
    # rotating V as well and rotating the output back keeps the gain
    vr = oracle.rotate_rows_f16(x.v)
    both = oracle.hadamard(oracle.attention(qr, oracle.Cache.from_fp16(kr, vr), x.lens, scale))
    assert _rel(both, exact) < 0.5 * e_plain
