"""Crafted quantizer inputs for the tests (no quantizer arithmetic of the
product or the oracle): fp16 groups of 64 values whose interior elements sit
on, or within two binary32 ulps of, a half-integer of
t = (x - bias) / scale, the points where rounding t to the nearest code
depends on how t is computed (an IEEE division and a multiplication by a
rounded reciprocal can land on different sides of k + 0.5)."""
import numpy as np

GROUP = 64

# every finite fp16 value, ascending (the candidates a group can draw from)
_ALL = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16)
_ALL = np.unique(_ALL[np.isfinite(_ALL)].astype(np.float32))


def _rule_scale(mn: np.float32, mx: np.float32, levels: int) -> np.float32:
    """The group's stored scale as the library defines it (max - min and the
    division by the level count in binary32, then rounded to fp16)."""
    r = np.float32(mx - mn)
    return np.float32(np.float16(np.float32(r / np.float32(levels))))


def near_tie_groups(n_groups: int, bits: int = 4, seed: int = 0) -> np.ndarray:
    """[n_groups, 64] fp16: element 0 is the group minimum, element 1 its
    maximum, the other 62 are drawn from the values of [min, max] whose t lies
    within 2 ulps of a half-integer (exact ties included), topped up with
    random values of the range when there are fewer."""
    rng = np.random.default_rng(seed)
    levels = (1 << bits) - 1
    out = np.empty((n_groups, GROUP), np.float16)
    g = 0
    while g < n_groups:
        mn = np.float32(np.float16(rng.normal(0.0, 1.5)))
        span = np.float32(rng.choice([0.01, 0.1, 0.7, 3.0, 15.0, 60.0]) * rng.uniform(0.5, 2.0))
        mx = np.float32(np.float16(mn + span))
        if not np.isfinite(mx) or mx <= mn:
            continue
        s = _rule_scale(mn, mx, levels)
        if s == 0:
            continue
        cand = _ALL[(_ALL >= mn) & (_ALL <= mx)]
        t = np.float32(cand - mn) / s
        dist = np.abs((t - np.floor(t)).astype(np.float32) - np.float32(0.5))
        near = cand[dist <= 2 * np.spacing(np.abs(t).astype(np.float32))]
        if near.size == 0:
            continue
        pick = rng.choice(near, size=GROUP - 2, replace=near.size < GROUP - 2)
        row = np.concatenate([[mn, mx], pick]).astype(np.float16)
        out[g] = row
        g += 1
    return out


def tie_rows(n_rows: int, head_dim: int, bits: int = 4, seed: int = 0, pool: int = 512) -> np.ndarray:
    """[n_rows, head_dim] fp16 rows made of near-tie groups (at most `pool`
    distinct ones, repeated in a seeded order), each group's elements
    shuffled."""
    per = head_dim // GROUP
    n = n_rows * per
    base = near_tie_groups(min(n, pool), bits, seed)
    rng = np.random.default_rng(seed + 1)
    groups = base[rng.integers(0, base.shape[0], n)] if n > base.shape[0] else base.copy()
    idx = np.argsort(rng.random(groups.shape), axis=1)
    groups = np.take_along_axis(groups, idx, axis=1)
    return groups.reshape(n_rows, head_dim)
