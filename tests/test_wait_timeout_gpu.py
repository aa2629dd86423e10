"""Bounded waits on the GPU: a wait that can never complete gives up, the
host reads the timeout from the device status word, and the context stays
usable. Nothing here faults, traps or hangs the GPU: every wait is bounded
(0.2 s in the self-test kernel; a few cycles, set through
fa_set_wait_limit_cycles, in the production kernels) and the kernels exit
normally after giving up."""
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


# Shapes whose kernels run on a few CTAs each: the tile kernels (forward,
# dK/dV, dQ) at D = 64, the D = 256 two-CTA dK/dV and dQ, the split-key
# forward and dQ of a single query row.
GIVE_UP_CASES = [
    ("tile_d64", 1, 2, 1, 64, 64, 64, "fp16", True, 0),
    ("pair_d256", 1, 2, 1, 200, 200, 256, "bf16", True, 0),
    # enough keys that each CTA of the split-key kernels walks several stages
    # (a stage load that has landed before its first wait never gives up)
    ("split_key_tq1", 1, 2, 1, 1, 5000, 128, "fp16", False, 0),
]


@pytest.mark.parametrize("name,B,Hq,Hkv,Tq,Tkv,D,dt,causal,window", GIVE_UP_CASES)
def test_production_kernels_give_up_cleanly(name, B, Hq, Hkv, Tq, Tkv, D, dt, causal, window):
    """With every ordinary wait bounded to a few cycles, the production
    kernels give up at their first wait, report the timeout in the status word
    and return (their waits at exit keep the default bound, so copies and MMAs
    in flight finish before TMEM is freed and the CTAs leave). The same calls
    afterwards, with the default bound, are clean and match the oracle."""
    import numpy as np
    import attention_fa_fwd_03_gb300 as fa
    import fa_inputs
    import oracle
    w = fa_inputs.Workload(f"give_up_{name}", B, Hq, Hkv, Tq, Tkv, D, dt, causal, window, seed=31)
    x = fa_inputs.make_inputs(w)
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))

    def run():
        o = torch.full_like(q, float("nan"))
        lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device=dev)
        grads = [torch.full_like(q, float("nan")), torch.full_like(k, float("nan")),
                 torch.full_like(v, float("nan"))]
        ws = torch.empty(fa.fa_bwd_workspace_size(B, Hq, Tq), dtype=torch.uint8, device=dev)
        fa.fa_fwd(q, k, v, o, lse, w.scale, causal, window)
        fa.fa_bwd(q, k, v, o, do, lse, *grads, w.scale, causal, window, workspace=ws)
        return o, lse, grads

    torch.cuda.synchronize()
    fa.fa_device_status(clear=True)
    t0 = time.perf_counter()
    try:
        fa.fa_set_wait_limit_cycles(8)
        run()
        bits = fa.fa_device_status(clear=True)   # synchronises the stream
    finally:
        fa.fa_set_wait_limit_cycles(0)
    took = time.perf_counter() - t0
    assert bits & 1, f"{name}: no wait gave up (status {bits:#x})"
    assert took < 2.0, f"{name}: the calls took {took:.2f} s to give up"

    o, lse, (dq, dk, dv) = run()
    assert fa.fa_device_status(clear=True) == 0, f"{name}: a wait gave up with the default bound"
    ref = oracle.attn_bwd(*(x[n].double().numpy() for n in ("q", "k", "v", "do")),
                          w.scale, causal, window)
    got_o = o.double().cpu().numpy()
    assert np.abs(got_o - ref["o"]).max() <= 2e-2
    fin = np.isfinite(ref["lse"])
    assert np.abs(lse.double().cpu().numpy()[fin] - ref["lse"][fin]).max() <= 1e-3
    for n, g in (("dq", dq), ("dk", dk), ("dv", dv)):
        a = g.double().cpu().numpy()
        rel = np.linalg.norm(a - ref[n]) / np.linalg.norm(ref[n])
        assert rel <= 1e-2, f"{name}: {n} rel-Frobenius {rel:.3e}"
