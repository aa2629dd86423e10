"""Bounded waits on the GPU: a wait that can never complete gives up, the
host reads the timeout from the device status word, and the context stays
usable. Nothing here faults, traps or hangs the GPU: the waits are bounded
(0.2 s) and the kernel exits normally after giving up."""
import os
import sys
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def test_wait_gives_up_reports_timeout_and_releases_the_other_warp():
    import attention_fa_fwd_03_gb300 as fa
    import fa_inputs
    fa.fa_device_status(clear=True)                     # start from a clean word
    t0 = time.perf_counter()
    fa.fa_selftest_wait_timeout(200)
    bits = fa.fa_device_status(clear=True)              # synchronises the stream
    took = time.perf_counter() - t0
    assert bits & 1, f"timeout bit not set: {bits:#x}"
    # warp 1's own limit is 4 x 200 ms: leaving well before it means the abort
    # flag raised by warp 0 released it
    assert took < 0.6, f"self-test took {took:.3f} s"
    assert fa.fa_device_status(clear=True) == 0         # cleared

    # the context is still usable: a normal forward runs and reports no timeout
    w = fa_inputs.WORKLOADS["c1_b1_h2x1_t64_d64_fp16_causal"]
    x = fa_inputs.make_inputs(w)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    fa.fa_fwd(q, k, v, o, lse, w.scale, w.causal, w.window)
    assert fa.fa_device_status(clear=True) == 0
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


def test_selftest_rejects_out_of_range_limits():
    import attention_fa_fwd_03_gb300 as fa
    with pytest.raises(fa.FaError):
        fa.fa_selftest_wait_timeout(0)
    with pytest.raises(fa.FaError):
        fa.fa_selftest_wait_timeout(20000)
