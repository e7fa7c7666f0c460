"""The device-side failure path without a GPU fault: a pipeline wait that
runs out.  The decode kernels wait on their stages with a time limit and,
when it runs out, record TQ_DEV_TIMEOUT and leave instead of hanging.  The
diagnostic entry point runs that wait on one CTA with a short limit, on a
barrier nothing arrives at, after a bulk copy it has waited for (nothing is
in flight when it leaves).  The status bit must be set, the kernel must have
waited at least the limit, its copy must have landed, and the context must
stay usable: a decode right after it matches the oracle."""
import numpy as np
import pytest

import oracle
from int4_kv_cache_gb300 import synth
from tests.gpu_helpers import assert_close, decode, gpu_cache_from_fp16, need_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_us", [200, 5000])
def test_bounded_wait_runs_out_and_reports(limit_us):
    torch = need_gpu()
    import int4_kv_cache_gb300 as tq

    src = torch.randint(0, 256, (1024,), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    copied = torch.zeros(1, dtype=torch.int32, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    tq.tq_wait_timeout_selftest(src, status, limit_us, copied)
    e1.record()
    torch.cuda.synchronize()
    assert status.item() & tq.TQ_DEV_TIMEOUT
    assert e0.elapsed_time(e1) * 1e3 >= limit_us  # it waited out its limit
    want = int(src.cpu().numpy().view(np.uint32).astype(np.uint64).sum() % (1 << 32))
    assert int(copied.item()) & 0xFFFFFFFF == want  # the copy landed before the CTA left
    # the context is fine: a decode right after it
    w = synth.WORKLOADS["tiny"]
    x = w.draw()
    out = decode(gpu_cache_from_fp16(x.k, x.v), x.q, x.lens, w.seq_len, w.attn_scale)
    assert_close(out, oracle.attention(x.q, oracle.Cache.from_fp16(x.k, x.v), x.lens, w.attn_scale),
                 what="decode after a timed-out wait")
