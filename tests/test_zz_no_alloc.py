"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device
memory (a plug-in inside a host program that owns every device allocation, or
a loop that may not call the allocator once it runs). It keeps the D-vector
in a fixed array inside the library instead of a caller workspace.

The GPU test calls it through the C ABI twice in a row, on different inputs
and sizes, and requires each result to equal bit for bit what fa_bwd (which
takes a caller workspace) gives on the same inputs: both run the same kernels
in the same summation order. This file is collected last and needs nothing
from the others, so it passes alone in a fresh process as well as after them.
"""
import ctypes

import pytest
import torch

import attention_fa_fwd_03_gb300 as fa
import fa_inputs
from attention_fa_fwd_03_gb300 import build_lib


def noalloc_fn():
    lib = fa.library()
    fn = lib.fa_bwd_noalloc
    vp, i = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, ctypes.c_float, i, i, i,
                   vp]
    fn.restype = i
    lib.fa_bwd_noalloc_max_rows.argtypes = []
    lib.fa_bwd_noalloc_max_rows.restype = ctypes.c_size_t
    return fn, int(lib.fa_bwd_noalloc_max_rows())


def test_noalloc_rejects_sizes_beyond_its_array():
    """Host-side: too many D-vector rows is refused before any launch."""
    build_lib.build()
    fn, max_rows = noalloc_fn()
    assert max_rows == 1 << 20
    base, gap = 1 << 40, 1 << 36
    p = [base + j * gap for j in range(9)]
    Tq = max_rows // 8 + 1                  # B * Hq * Tq = max_rows + 8
    assert fn(*p, 1, 8, 2, Tq, 64, 128, 0.1, 0, 0, 1, None) == 1   # FA_ERR_INVALID_ARG
    assert fn(*p, 1, 8, 2, 64, 64, 80, 0.1, 0, 0, 1, None) == 2    # head dim still checked


def run_fa_bwd(x, w):
    """Forward, then fa_bwd with a caller-owned workspace: the reference."""
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    fa.fa_fwd(q, k, v, o, lse, w.scale, w.causal, w.window)
    ws = torch.empty(fa.fa_bwd_workspace_size(w.B, w.Hq, w.Tq), dtype=torch.uint8, device=dev)
    ref = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
    fa.fa_bwd(q, k, v, o, do, lse, *ref, w.scale, w.causal, w.window, workspace=ws)
    return (q, k, v, o, do, lse), ref


@pytest.mark.gpu
def test_noalloc_matches_fa_bwd_on_two_calls_in_a_row():
    """Two calls in a row through the C ABI, each compared bit for bit with
    fa_bwd on the same inputs (same kernels, same summation order). The second
    call has other inputs and a smaller D-vector than the first, so a call
    that read the array's previous contents instead of rewriting them would
    give other gradients."""
    fn, _ = noalloc_fn()
    calls = [
        fa_inputs.Workload("noalloc1", 2, 8, 2, 333, 333, 128, "bf16", True, window=0, seed=4242),
        fa_inputs.Workload("noalloc2", 1, 4, 2, 200, 260, 128, "bf16", True, window=0, seed=777),
    ]
    stream = torch.cuda.current_stream().cuda_stream
    for call, w in enumerate(calls):
        x = fa_inputs.make_inputs(w)
        (q, k, v, o, do, lse), ref = run_fa_bwd(x, w)
        got = [torch.full_like(q, float("nan")), torch.full_like(k, float("nan")),
               torch.full_like(v, float("nan"))]
        st = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                lse.data_ptr(), got[0].data_ptr(), got[1].data_ptr(), got[2].data_ptr(),
                w.B, w.Hq, w.Hkv, w.Tq, w.Tkv, w.D, w.scale, int(w.causal), w.window, 1, stream)
        assert st == 0, f"call {call}: status {st}"
        torch.cuda.synchronize()
        assert fa.fa_device_status() == 0
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            assert not torch.isnan(g).any(), f"call {call}: NaN in {name}"
            assert torch.equal(g, r), f"call {call}: {name} differs from fa_bwd"
