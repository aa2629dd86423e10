"""The differentiable wrapper (torch.autograd.Function over the C ABI)
against the oracle, and against direct C-ABI calls bit for bit.

Gradients are taken of the scalar sum(O * dO), so q.grad, k.grad and v.grad
are the VJP the oracle computes for cotangent dO.
"""
import math

import numpy as np
import pytest
import torch

import fa_inputs
import oracle

GRAD_TOL, O_TOL, LSE_TOL = 1e-2, 2e-2, 1e-3


def _wrapper():
    from attention_fa_fwd_03_gb300.autograd import flash_attention
    return flash_attention


def _rel_fro(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def _run(x, w, **kw):
    flash_attention = _wrapper()
    dev = torch.device("cuda")
    q, k, v = (x[n].to(dev).requires_grad_() for n in ("q", "k", "v"))
    do = x["do"].to(dev)
    o, lse = flash_attention(q, k, v, w.scale, w.causal, w.window, return_lse=True, **kw)
    (o.float() * do.float()).sum().backward()
    torch.cuda.synchronize()
    return {"o": o.detach(), "lse": lse, "dq": q.grad, "dk": k.grad, "dv": v.grad}


CASES = [
    ("c1_b1_h2x1_t64_d64_fp16_causal", None),
    (None, fa_inputs.Workload("ag_gqa_window", 1, 4, 2, 300, 300, 128, "bf16", True, 64, seed=41)),
    (None, fa_inputs.Workload("ag_cross", 2, 4, 1, 90, 200, 96, "fp16", False, 0, seed=42)),
    # decode-shaped: split-key forward and dQ, folded dK/dV
    (None, fa_inputs.Workload("ag_short", 2, 8, 2, 4, 600, 128, "bf16", False, 0, seed=45)),
]


@pytest.mark.gpu
@pytest.mark.parametrize("name,w", CASES)
def test_autograd_matches_oracle(name, w):
    w = w or fa_inputs.WORKLOADS[name]
    x = fa_inputs.make_inputs(w)
    got = {n: t.double().cpu().numpy() for n, t in _run(x, w).items()}
    ref = oracle.attn_bwd(*(x[n].double().numpy() for n in ("q", "k", "v", "do")),
                          w.scale, w.causal, w.window)
    assert np.abs(got["o"] - ref["o"]).max() <= O_TOL
    fin = np.isfinite(ref["lse"])
    assert np.array_equal(fin, np.isfinite(got["lse"]))
    assert np.abs(got["lse"][fin] - ref["lse"][fin]).max() <= LSE_TOL
    for n in ("dq", "dk", "dv"):
        assert _rel_fro(got[n], ref[n]) <= GRAD_TOL, n


@pytest.mark.gpu
def test_autograd_equals_direct_abi_calls():
    """Same kernels, same inputs: the wrapper adds no arithmetic of its own."""
    import attention_fa_fwd_03_gb300 as fa
    w = fa_inputs.Workload("ag_direct", 1, 4, 2, 257, 257, 128, "bf16", True, seed=43)
    x = fa_inputs.make_inputs(w)
    got = _run(x, w)
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_bwd_workspace_size(*q.shape[:3]), dtype=torch.uint8, device=dev)
    fa.fa_fwd(q, k, v, o, lse, w.scale, w.causal, w.window)
    # the wrapper's cotangent of sum(O * dO) taken in fp32 is dO cast back to O's dtype
    fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, w.scale, w.causal, w.window, workspace=ws)
    torch.cuda.synchronize()
    for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
        assert torch.equal(got[n], t), n


@pytest.mark.gpu
def test_autograd_default_scale_and_noncontiguous_inputs():
    flash_attention = _wrapper()
    w = fa_inputs.Workload("ag_layout", 1, 2, 1, 130, 130, 64, "fp16", True, seed=44)
    x = fa_inputs.make_inputs(w)
    dev = torch.device("cuda")
    # [B, T, H, D] storage viewed as [B, H, T, D]: not contiguous
    q, k, v = (x[n].transpose(1, 2).contiguous().to(dev).transpose(1, 2) for n in ("q", "k", "v"))
    assert not q.is_contiguous()
    for t in (q, k, v):
        t.requires_grad_()
    o = flash_attention(q, k, v, causal=True)   # scale defaults to 1/sqrt(D)
    o.backward(x["do"].to(dev))
    torch.cuda.synchronize()
    ref = oracle.attn_bwd(*(x[n].double().numpy() for n in ("q", "k", "v", "do")),
                          1.0 / math.sqrt(w.D), True, 0)
    assert np.abs(o.detach().double().cpu().numpy() - ref["o"]).max() <= O_TOL
    for n, t in (("dq", q), ("dk", k), ("dv", v)):
        assert _rel_fro(t.grad.double().cpu().numpy(), ref[n]) <= GRAD_TOL, n


def test_autograd_has_no_cpu_path():
    """CPU tensors are refused (or the missing library is reported), never computed."""
    flash_attention = _wrapper()
    q = torch.zeros(1, 2, 8, 64, dtype=torch.float16, requires_grad=True)
    k = torch.zeros(1, 1, 8, 64, dtype=torch.float16)
    with pytest.raises((ValueError, RuntimeError)):
        flash_attention(q, k, k)
