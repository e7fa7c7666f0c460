"""The Hadamard rotation's fp32 arithmetic restated in numpy for the tests: H_n
x (unnormalised Sylvester order) with the stages in increasing order
h = 1, 2, ..., n/2, each butterfly (a, b) -> (a + b, a - b) one
round-to-nearest float32 operation ("Running and Evaluating TurboQuant
optimized Gemma 4", TurboQuant section: x -> H x / sqrt(n)).  Pinned in
tests/test_fwht_restatement.py."""
import numpy as np


def sequential_transform_f32(x: np.ndarray) -> np.ndarray:
    v = x.astype(np.float32).copy()
    n = v.shape[-1]
    h = 1
    while h < n:
        w = v.reshape(v.shape[:-1] + (n // (2 * h), 2, h))
        a, b = w[..., 0, :].copy(), w[..., 1, :].copy()
        w[..., 0, :] = a + b
        w[..., 1, :] = a - b
        v = w.reshape(v.shape)
        h *= 2
    return v
