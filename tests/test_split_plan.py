"""The split-K plan rule, as host arithmetic (tq_split_plan, no device).

Decode cuts each (sequence, kv head) into n balanced runs of whole units; the
rule picks n to minimise waves x (longest run + two tiles) + the reduce (one
tile, none when the decode merges its runs itself: one run, or up to eight in
a grid of one wave), waves = ceil(CTAs / resident CTA slots).  The library
searches a few candidates (the largest run count of each wave count, the
largest it can merge, one run); these tests check that shortcut against a
brute force over every n, and the picks on the shapes whose run counts were
timed on a GB300 (456 resident slots: 152 SMs x 3 CTAs of the int4
head_dim-128 kernel)."""
import math

import pytest

import int4_kv_cache_gb300 as tq
from int4_kv_cache_gb300 import build as tqbuild

MAX_CTAS = 2048  # most CTAs one decode plan launches
MAX_CLUSTER = 8  # most runs a decode merges itself


@pytest.fixture(scope="module", autouse=True)
def _built():
    tqbuild.build()


def brute(batch, hkv, max_len, chunk, tile, slots, merge):
    unit = min(chunk, tile)
    units = math.ceil(max_len / unit)
    heads = batch * hkv
    cap = max(1, min(units, MAX_CTAS // heads))
    best = None
    for n in range(1, cap + 1):
        waves = math.ceil(heads * n / slots)
        cost = waves * (math.ceil(units / n) * unit + 2 * tile)
        if not (merge and (n == 1 or (n <= MAX_CLUSTER and waves == 1))):
            cost += tile  # the reduce
        if best is None or cost < best[0]:
            best = (cost, n)
    n = best[1]
    return n, math.ceil(units / n) * unit


@pytest.mark.parametrize("merge", [False, True])
@pytest.mark.parametrize("batch", [1, 2, 3, 4, 7, 8, 16, 32, 57, 64, 128, 256])
@pytest.mark.parametrize("hkv", [1, 2, 8, 16])
@pytest.mark.parametrize("max_len", [1, 33, 100, 423, 950, 2048, 4096, 8192, 32768, 131072])
def test_candidates_equal_brute_force(batch, hkv, max_len, merge):
    for chunk, tile, slots in ((512, 128, 456), (512, 64, 304), (32, 128, 456), (16, 64, 7)):
        assert tq.tq_split_plan(batch, hkv, max_len, chunk, tile, slots, merge) == brute(
            batch, hkv, max_len, chunk, tile, slots, merge)


# (sequences, tokens each) -> runs the GB300 timed fastest for int4 head_dim 128, 8 kv heads
# (phase 1 + reduce, CUDA graph; so merge = False): the plan's pick and the measured best agree.
MEASURED_BEST = {
    (1, 131072): 57,   # one wave of 456 CTAs
    (2, 131072): 28,
    (4, 131072): 14,
    (4, 32768): 14,
    (8, 32768): 7,
    (8, 8192): 7,
    (16, 8192): 3,     # 3 (40.6 us) and 7 (41.9 us) tie in the model; 4 runs: 45.8 us
    (16, 32768): 7,    # 896 CTAs: 110.0 us; 4 runs (512 CTAs): 140.6 us
    (32, 8192): 5,     # 72.2 us
    (32, 32768): 7,    # 210.7 us; 4 runs: 223.3 us
}


@pytest.mark.parametrize("shape,runs", sorted(MEASURED_BEST.items()))
def test_measured_best_run_counts(shape, runs):
    batch, tokens = shape
    assert tq.tq_split_plan(batch, 8, tokens, 512, 128, 456, merge=False)[0] == runs
    if runs > MAX_CLUSTER:  # too many runs to merge in phase 1: the same pick either way
        assert tq.tq_split_plan(batch, 8, tokens, 512, 128, 456, merge=True)[0] == runs


# shapes whose decode merges its runs in phase 1 (no reduce launch)
@pytest.mark.parametrize("batch,hkv,tokens,tile,slots,runs", [
    (1, 8, 1024, 128, 456, 8),     # Llama 1K: 8 runs of one tile, one cluster per kv head
    (1, 8, 2048, 128, 456, 8),     # Llama 2K: 8 runs of two tiles (ties 16 runs + reduce: fewer runs)
    (1, 16, 950, 64, 304, 8),      # Gemma shape, 950 tokens: 8 runs of two tiles (7.3 us; 15 + reduce 7.5)
    (1, 16, 2048, 64, 304, 16),    # Gemma shape, 2,048 tokens: 16 runs + reduce (8.8 us; 8 merged 9.6)
    (1, 16, 33, 64, 304, 1),       # Gemma shape, 33 tokens: one run
])
def test_merge_picks(batch, hkv, tokens, tile, slots, runs):
    assert tq.tq_split_plan(batch, hkv, tokens, 512, tile, slots, merge=True)[0] == runs


def test_plan_properties():
    # runs cover the sequence; never more CTAs than the cap; never more runs than units
    for batch, hkv, max_len in ((1, 8, 131072), (64, 8, 8192), (1, 1, 100000), (300, 8, 2000), (1, 8, 16)):
        ns, run = tq.tq_split_plan(batch, hkv, max_len, 512, 128, 456)
        assert ns * run >= max_len and (ns - 1) * run < max_len + run
        assert 1 <= ns and (ns == 1 or batch * hkv * ns <= MAX_CTAS)
        assert ns <= math.ceil(max_len / 128)


def test_argument_errors():
    with pytest.raises(tq.TQError):
        tq.tq_split_plan(0, 8, 100, 512, 128, 456)
    with pytest.raises(tq.TQError):
        tq.tq_split_plan(1, 8, 100, 500, 128, 456)
    with pytest.raises(tq.TQError):
        tq.tq_split_plan(1, 8, 100, 512, 128, 0)
