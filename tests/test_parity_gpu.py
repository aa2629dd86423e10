"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs, element by element.

Tolerances (the headline requirement for fp16/bf16 inputs): O max-abs error
<= 2e-2; dQ, dK, dV relative Frobenius error <= 1e-2; LSE absolute error
<= 1e-3 on finite entries, with -inf exactly where the oracle has -inf.

Small workloads are compared in full (or on whole (batch, KV group) slices,
which are independent problems). The two large workloads run at full size in
the same launch configuration the benchmark times, and whole (batch, KV
group) slices of their outputs are compared with the oracle on every row:
four of the 32 groups of the causal B4 Hq32 Hkv8 T4096 workload (first,
middle and last of the grid), and both groups (the whole output) of the
sliding-window B1 Hq16 Hkv2 T16384 workload. Their gradients are checked per
128-row block as well. Properties that hold at any size (no NaN, each dK
column sums to zero over keys, dV sums to the group's dO) cover every group.
"""
import math

import numpy as np
import pytest
import torch

import fa_inputs
import oracle

pytestmark = pytest.mark.gpu

O_TOL, LSE_TOL, GRAD_TOL = 2e-2, 1e-3, 1e-2


def fa():
    import attention_fa_fwd_03_gb300 as m
    return m


def run_gpu(x, w, window=None):
    """fwd + bwd on the GPU; returns CPU float64 numpy arrays."""
    m = fa()
    window = w.window if window is None else window
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    # poison outputs so that a row the kernels forget to write shows up
    for t in (o, dq, dk, dv):
        t.fill_(float("nan"))
    lse.fill_(float("nan"))
    ws = torch.empty(m.fa_bwd_workspace_size(*q.shape[:3]), dtype=torch.uint8, device=dev)
    m.fa_fwd(q, k, v, o, lse, w.scale, w.causal, window)
    m.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, w.scale, w.causal, window, workspace=ws)
    torch.cuda.synchronize()
    assert m.fa_device_status() == 0, "a bounded device wait gave up"
    out = {n: t.double().cpu().numpy() for n, t in
           (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}
    return out


def rel_fro(a, b):
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / nb) if nb > 0 else float(np.linalg.norm(a))


def check_fwd(o, lse, ro, rlse, what=""):
    assert not np.isnan(o).any(), f"{what}: NaN in O"
    err = np.abs(o - ro).max()
    assert err <= O_TOL, f"{what}: O max-abs {err:.3e}"
    assert np.array_equal(np.isneginf(lse), np.isneginf(rlse)), f"{what}: -inf LSE pattern"
    fin = np.isfinite(rlse)
    lerr = np.abs(lse[fin] - rlse[fin]).max() if fin.any() else 0.0
    assert lerr <= LSE_TOL, f"{what}: LSE max-abs {lerr:.3e}"
    return err, lerr


def check_grads(g, r, what="", names=("dq", "dk", "dv")):
    errs = {}
    for n in names:
        assert not np.isnan(g[n]).any(), f"{what}: NaN in {n}"
        errs[n] = rel_fro(g[n], r[n])
        assert errs[n] <= GRAD_TOL, f"{what}: {n} rel-Frobenius {errs[n]:.3e}"
    return errs


def as64(x, names=("q", "k", "v", "do")):
    return [x[n].double().numpy() for n in names]


def group_views(x, b, g, reps):
    h0, h1 = g * reps, (g + 1) * reps
    return {"q": x["q"][b:b + 1, h0:h1], "k": x["k"][b:b + 1, g:g + 1],
            "v": x["v"][b:b + 1, g:g + 1], "do": x["do"][b:b + 1, h0:h1]}


def compare_full(w, x=None, window=None):
    x = x or fa_inputs.make_inputs(w)
    window = w.window if window is None else window
    got = run_gpu(x, w, window)
    ref = oracle.attn_bwd(*as64(x), w.scale, w.causal, window)
    check_fwd(got["o"], got["lse"], ref["o"], ref["lse"], w.name)
    return check_grads(got, ref, w.name)


def compare_groups(w, groups):
    """Full GPU run; oracle on whole (batch, KV group) slices."""
    x = fa_inputs.make_inputs(w)
    got = run_gpu(x, w)
    reps = w.Hq // w.Hkv
    for (b, g) in groups:
        xs = group_views(x, b, g, reps)
        ref = oracle.attn_bwd(*as64(xs), w.scale, w.causal, w.window)
        h0, h1 = g * reps, (g + 1) * reps
        sl = {"o": got["o"][b:b + 1, h0:h1], "lse": got["lse"][b:b + 1, h0:h1],
              "dq": got["dq"][b:b + 1, h0:h1], "dk": got["dk"][b:b + 1, g:g + 1],
              "dv": got["dv"][b:b + 1, g:g + 1]}
        check_fwd(sl["o"], sl["lse"], ref["o"], ref["lse"], f"{w.name} b{b} g{g}")
        check_grads(sl, ref, f"{w.name} b{b} g{g}")
    return got, x


# ---------------------------------------------------------------- workloads
def test_c1_smoke_shape_full():
    compare_full(fa_inputs.WORKLOADS["c1_b1_h2x1_t64_d64_fp16_causal"])


def test_c2_mha_noncausal_full():
    compare_full(fa_inputs.WORKLOADS["c2_b2_h8x8_t1024_d128_bf16"])


@pytest.mark.parametrize("name", ["c5a_b2_h8x2_t2048_d64_fp16_causal",
                                  "c5b_b2_h8x2_t2048_d96_fp16_causal",
                                  "c5c_b2_h8x2_t2048_d256_fp16_causal",
                                  "c5d_b2_h8x2_tq512_tkv2048_d128_fp16"])
def test_c5_shape_sweep_group_slices(name):
    w = fa_inputs.WORKLOADS[name]
    compare_groups(w, [(0, 0), (1, w.Hkv - 1)])


@pytest.mark.parametrize("name", ["c5e1_b2_h8x2_tq1_tkv1024_d128_fp16",
                                  "c5e4_b2_h8x2_tq4_tkv1024_d128_fp16",
                                  "c5e8_b2_h8x2_tq8_tkv1024_d128_fp16"])
def test_c5e_short_queries_full(name):
    compare_full(fa_inputs.WORKLOADS[name])


def run_gpu_device(x, w):
    """fwd + bwd on the GPU at full size; outputs stay on the device."""
    m = fa()
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    out = {"o": torch.empty_like(q), "lse": torch.empty(q.shape[:3], dtype=torch.float32, device=dev),
           "dq": torch.empty_like(q), "dk": torch.empty_like(k), "dv": torch.empty_like(v)}
    for t in out.values():
        t.fill_(float("nan"))
    ws = torch.empty(m.fa_bwd_workspace_size(*q.shape[:3]), dtype=torch.uint8, device=dev)
    m.fa_fwd(q, k, v, out["o"], out["lse"], w.scale, w.causal, w.window)
    m.fa_bwd(q, k, v, out["o"], do, out["lse"], out["dq"], out["dk"], out["dv"], w.scale,
             w.causal, w.window, workspace=ws)
    torch.cuda.synchronize()
    assert m.fa_device_status() == 0, "a bounded device wait gave up"
    return out


def check_row_blocks(got, ref, what, rows=128):
    """Relative Frobenius error of every block of `rows` rows (the last axis
    but one): a wrong block cannot hide behind the norm of a whole slice."""
    T = ref.shape[-2]
    worst = 0.0
    for r0 in range(0, T, rows):
        e = rel_fro(got[..., r0:r0 + rows, :], ref[..., r0:r0 + rows, :])
        assert e <= GRAD_TOL, f"{what}: rows [{r0}, {min(T, r0 + rows)}) rel-Frobenius {e:.3e}"
        worst = max(worst, e)
    return worst


def check_large_groups(w, groups):
    """Full-size run in the benchmark's launch configuration; whole (batch,
    KV group) slices compared with the oracle on every row of every output:
    O, LSE and dQ of the group's query heads, dK and dV of its KV head. The
    gradients are also checked block by block (128 rows), and properties that
    hold at any size cover the groups not compared."""
    x = fa_inputs.make_inputs(w)
    got = run_gpu_device(x, w)
    for name, t in got.items():
        nf = ~torch.isfinite(t)
        if name == "lse":
            nf &= ~torch.isneginf(t)
        assert not bool(nf.any()), f"{w.name}: {int(nf.sum())} non-finite values in {name}"
    reps = w.Hq // w.Hkv
    for (b, g) in groups:
        xs = group_views(x, b, g, reps)
        ref = oracle.attn_bwd(*as64(xs), w.scale, w.causal, w.window)
        h0, h1 = g * reps, (g + 1) * reps
        sl = {"o": got["o"][b:b + 1, h0:h1], "lse": got["lse"][b:b + 1, h0:h1],
              "dq": got["dq"][b:b + 1, h0:h1], "dk": got["dk"][b:b + 1, g:g + 1],
              "dv": got["dv"][b:b + 1, g:g + 1]}
        sl = {n: t.double().cpu().numpy() for n, t in sl.items()}
        what = f"{w.name} b{b} g{g}"
        o_err, lse_err = check_fwd(sl["o"], sl["lse"], ref["o"], ref["lse"], what)
        errs = check_grads(sl, ref, what)
        blk = {n: check_row_blocks(sl[n], ref[n], f"{what} {n}") for n in ("dq", "dk", "dv")}
        print(f"{what}: O max-abs {o_err:.2e}, LSE {lse_err:.2e}, rel-Frobenius "
              + ", ".join(f"{n} {errs[n]:.2e} (worst block {blk[n]:.2e})" for n in errs))
    # any-size properties over every group: the rows of dS sum to zero, so each
    # dK column sums to zero over the keys; the rows of P sum to one, so dV
    # summed over the keys is the group's dO summed over its rows
    dk = got["dk"].double()
    dk_sum = dk.sum(dim=2)
    assert float(dk_sum.abs().max()) <= 1e-2 * float(dk.abs().sum(dim=2).max()) + 1e-3
    want_dv = x["do"].double().reshape(w.B, w.Hkv, reps, w.Tq, w.D).sum(dim=(2, 3))
    got_dv = got["dv"].double().sum(dim=2).cpu()
    assert rel_fro(got_dv.numpy(), want_dv.numpy()) <= 1e-2


def test_c3_headline_full_size_whole_groups():
    """B4 Hq32 Hkv8 T4096 D128 bf16 causal: four whole (batch, KV group)
    slices, at the start, in the middle and at the end of the grid."""
    check_large_groups(fa_inputs.WORKLOADS["c3_b4_h32x8_t4096_d128_bf16_causal"],
                       groups=((0, 0), (1, 3), (2, 5), (3, 7)))


def test_c4_sliding_window_full_size_every_group():
    """B1 Hq16 Hkv2 T16384 D128 bf16 causal, window 4096: both KV groups,
    i.e. the whole output, compared with the oracle."""
    check_large_groups(fa_inputs.WORKLOADS["c4_b1_h16x2_t16384_d128_bf16_causal_w4096"],
                       groups=((0, 0), (0, 1)))


# --------------------------------------------------------------- edge cases
EDGE = [
    # (B, Hq, Hkv, Tq, Tkv, D, dtype, causal, window)
    (1, 2, 1, 200, 200, 128, "bf16", True, 0),       # ragged tail, several tiles
    (2, 4, 4, 333, 333, 64, "fp16", False, 0),
    (1, 4, 2, 129, 129, 96, "bf16", True, 0),
    (1, 2, 1, 257, 257, 256, "bf16", True, 0),
    (1, 2, 2, 300, 300, 256, "fp16", False, 0),
    (1, 16, 1, 150, 150, 64, "bf16", True, 0),       # GQA 16:1
    (1, 8, 1, 140, 140, 128, "fp16", True, 0),       # GQA 8:1
    (1, 4, 1, 500, 500, 128, "bf16", True, 100),     # causal window
    (1, 4, 2, 400, 400, 64, "fp16", False, 77),      # window without causal (future visible)
    (1, 2, 1, 300, 100, 128, "bf16", True, 40),      # fully masked rows (Tq > Tkv + window)
    (1, 2, 1, 77, 300, 128, "bf16", True, 0),        # Tq < Tkv causal (top-left)
    (1, 2, 1, 300, 77, 64, "fp16", True, 0),         # Tq > Tkv causal
    (2, 4, 2, 1, 257, 128, "bf16", False, 0),        # single query row
    (1, 2, 1, 1, 1, 64, "fp16", False, 0),           # single key and query
    (1, 2, 2, 5, 700, 256, "bf16", False, 0),        # short queries, D=256
    (3, 6, 3, 256, 384, 96, "fp16", False, 0),       # exact tile multiples, cross-attention
    # grids large enough for two 128-row query tiles per forward CTA, ragged tails
    (4, 40, 8, 300, 300, 128, "bf16", True, 0),
    (2, 80, 10, 200, 260, 64, "fp16", False, 70),
    # small grids: each KV block's tiles split over a two-CTA cluster
    (1, 4, 1, 700, 700, 64, "fp16", True, 200),      # causal window, 4 heads per group
    (2, 6, 2, 333, 500, 128, "bf16", False, 0),      # 3 heads per group, Tq != Tkv
    (1, 2, 2, 500, 500, 96, "fp16", True, 0),        # one head per group: split by query tiles
    # small causal / windowed grids with a heavy first block: four-CTA clusters
    (1, 4, 1, 1024, 1024, 64, "fp16", True, 0),      # 8 blocks of 4-32 tiles
    (1, 8, 2, 700, 700, 128, "bf16", True, 256),     # causal window
    (2, 6, 2, 900, 900, 96, "fp16", True, 0),        # 3 heads per group, ragged tail
    # head dim 256: two-CTA dK/dV clusters, dQ with Q in TMEM
    (1, 2, 1, 300, 100, 256, "bf16", True, 40),      # fully masked rows
    (1, 8, 2, 260, 300, 256, "fp16", False, 50),     # window without causal, 4 heads per group
    # short query blocks (Tq <= 8): the split-key forward
    (1, 4, 2, 6, 300, 128, "bf16", True, 0),         # causal, top-left: row i sees i + 1 keys
    (1, 4, 2, 8, 500, 64, "fp16", False, 3),         # window without causal
    (1, 2, 1, 8, 1000, 96, "bf16", True, 4),         # causal window
    (3, 6, 3, 4, 5000, 128, "fp16", False, 0),       # long keys: 8-CTA clusters
    (1, 2, 1, 2, 33, 256, "fp16", False, 0),         # ragged key block, D=256
    (1, 16, 1, 3, 2000, 64, "bf16", False, 0),       # GQA 16:1
    (1, 8, 1, 1, 20000, 128, "bf16", False, 0),      # decode over a long key range
    (1, 4, 2, 8, 9000, 96, "fp16", False, 1000),     # long keys, window 1000 (past only)
    # short query blocks: the vector dK/dV (rows of all the group's heads, any mask)
    (2, 16, 2, 8, 100, 256, "bf16", True, 0),        # 64 rows per group (two chunks), D=256
    (1, 12, 4, 5, 3, 64, "fp16", True, 0),           # fewer keys than query rows, causal
    (1, 8, 2, 7, 1500, 128, "bf16", True, 3),        # causal window of 3
    (2, 32, 2, 8, 64, 96, "fp16", False, 5),         # 128 rows per group, window without causal
    # mask-free GQA below one tile: the heads' rows share tiles
    (2, 8, 2, 40, 300, 128, "bf16", False, 0),       # 4 x 40 rows per group
    (1, 6, 2, 100, 200, 64, "fp16", False, 0),       # 3 x 100 rows, ragged tiles
    (1, 32, 1, 9, 129, 96, "bf16", False, 0),        # 32 x 9 rows, just past the split-key path
]


@pytest.mark.parametrize("B,Hq,Hkv,Tq,Tkv,D,dt,causal,window", EDGE)
def test_edge_cases(B, Hq, Hkv, Tq, Tkv, D, dt, causal, window):
    w = fa_inputs.Workload(f"edge_{B}_{Hq}_{Hkv}_{Tq}_{Tkv}_{D}_{dt}_{int(causal)}_{window}",
                           B, Hq, Hkv, Tq, Tkv, D, dt, causal, window,
                           seed=1000 + Tq + 7 * Tkv + D)
    compare_full(w)


def test_large_values_stay_finite():
    """Sharp softmax (Q, K scaled by 8) exercises the lazy rescale path."""
    w = fa_inputs.Workload("sharp", 1, 2, 1, 700, 700, 128, "bf16", True, qk_mult=8.0, seed=77)
    compare_full(w)


def test_repeat_calls_are_deterministic():
    w = fa_inputs.Workload("det", 1, 4, 2, 300, 300, 128, "bf16", True, seed=5)
    x = fa_inputs.make_inputs(w)
    a = run_gpu(x, w)
    b = run_gpu(x, w)
    for n in a:
        assert np.array_equal(np.nan_to_num(a[n], neginf=-1e300), np.nan_to_num(b[n], neginf=-1e300)), n


def test_full_size_runs_repeat_bit_for_bit():
    """Races between warps show up as runs that differ: repeat the full-size
    sliding-window workload (where a barrier-phase race once gave NaN rows in
    about one run in 30) with NaN-poisoned outputs and require every run to be
    finite and bitwise equal to the first."""
    m = fa()
    w = fa_inputs.WORKLOADS["c4_b1_h16x2_t16384_d128_bf16_causal_w4096"]
    x = fa_inputs.make_inputs(w)
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    outs = {"o": torch.empty_like(q), "lse": torch.empty(q.shape[:3], dtype=torch.float32, device=dev),
            "dq": torch.empty_like(q), "dk": torch.empty_like(k), "dv": torch.empty_like(v)}
    ws = torch.empty(m.fa_bwd_workspace_size(*q.shape[:3]), dtype=torch.uint8, device=dev)
    first = None
    for run in range(24):
        for t in outs.values():
            t.fill_(float("nan"))
        m.fa_fwd(q, k, v, outs["o"], outs["lse"], w.scale, w.causal, w.window)
        m.fa_bwd(q, k, v, outs["o"], do, outs["lse"], outs["dq"], outs["dk"], outs["dv"], w.scale,
                 w.causal, w.window, workspace=ws)
        assert m.fa_device_status() == 0, "a bounded device wait gave up"
        for n, t in outs.items():
            assert bool(torch.isfinite(t).all()), f"run {run}: non-finite values in {n}"
        if first is None:
            first = {n: t.clone() for n, t in outs.items()}
        else:
            for n, t in outs.items():
                assert torch.equal(t, first[n]), f"run {run}: {n} differs from the first run"


@pytest.mark.parametrize("B,Hq,Hkv,Tq,Tkv,D,dt,causal,window", [
    (1, 4, 2, 300, 300, 128, "bf16", True, 0),       # tile kernels, dQ beside dK/dV
    (2, 4, 2, 260, 260, 64, "fp16", False, 0),       # tile kernels, dQ after dK/dV
    (2, 8, 2, 4, 700, 128, "fp16", False, 0),        # short queries: vector dK/dV, split-key dQ
    (1, 2, 1, 200, 200, 256, "bf16", True, 64),      # D = 256 kernels
    (1, 6, 2, 400, 400, 96, "bf16", False, 150),     # window without causal: dQ beside dK/dV
    (2, 8, 2, 6, 900, 64, "fp16", True, 0),          # causal short queries: vector dK/dV
])
def test_phase_calls_equal_fa_bwd(B, Hq, Hkv, Tq, Tkv, D, dt, causal, window):
    """fa_bwd_preprocess + fa_bwd_dkv + fa_bwd_dq (the phases the benchmark
    times one by one, each waiting for the one before) give exactly what one
    fa_bwd call gives, where dQ may run beside dK/dV."""
    m = fa()
    w = fa_inputs.Workload("phases", B, Hq, Hkv, Tq, Tkv, D, dt, causal, window, seed=55)
    x = fa_inputs.make_inputs(w)
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    m.fa_fwd(q, k, v, o, lse, w.scale, causal, window)
    ws = torch.empty(m.fa_bwd_workspace_size(B, Hq, Tq), dtype=torch.uint8, device=dev)
    one = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
    m.fa_bwd(q, k, v, o, do, lse, *one, w.scale, causal, window, workspace=ws)
    ws2 = torch.empty_like(ws)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    m.fa_bwd_preprocess(o, do, ws2)
    m.fa_bwd_dkv(q, k, v, do, lse, ws2, dk, dv, w.scale, causal, window)
    m.fa_bwd_dq(q, k, v, do, lse, ws2, dq, w.scale, causal, window)
    torch.cuda.synchronize()
    assert m.fa_device_status() == 0
    for name, a, b in (("dq", one[0], dq), ("dk", one[1], dk), ("dv", one[2], dv)):
        assert torch.equal(a, b), name


@pytest.mark.parametrize("B,Hq,Hkv,T,D,dt,causal,window", [
    (2, 8, 2, 2048, 64, "fp16", True, 0),    # dQ starts beside dK/dV
    (1, 8, 2, 8, 128, "bf16", False, 0),     # short queries: vector dK/dV beside split-key dQ
    (2, 8, 8, 1024, 128, "bf16", False, 0),  # dQ after dK/dV
])
def test_stream_order_after_backward(B, Hq, Hkv, T, D, dt, causal, window):
    """Kernels start while the previous one in the stream finishes, and dQ may
    run beside dK/dV; work queued after fa_bwd on the same stream must still
    see the whole backward done. Right after fa_bwd (no synchronisation) a
    forward on other inputs overwrites O and the LSE the backward reads, and
    stream-ordered copies take dQ, dK and dV: all must equal a backward run
    alone."""
    m = fa()
    Tq, Tkv = T, (T if T > 8 else 1500)  # short queries read a longer key range
    w = fa_inputs.Workload("order", B, Hq, Hkv, Tq, Tkv, D, dt, causal, window, seed=77)
    x = fa_inputs.make_inputs(w)
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    q2 = torch.flip(q, dims=[2]).contiguous()
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    ws = torch.empty(m.fa_bwd_workspace_size(B, Hq, Tq), dtype=torch.uint8, device=dev)
    m.fa_fwd(q, k, v, o, lse, w.scale, causal, window)
    o_keep, lse_keep = o.clone(), lse.clone()
    ref = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
    m.fa_bwd(q, k, v, o, do, lse, *ref, w.scale, causal, window, workspace=ws)
    torch.cuda.synchronize()
    for _ in range(5):
        o.copy_(o_keep)
        lse.copy_(lse_keep)
        got = [torch.full_like(t, float("nan")) for t in ref]
        m.fa_bwd(q, k, v, o, do, lse, *got, w.scale, causal, window, workspace=ws)
        m.fa_fwd(q2, k, v, o, lse, w.scale, causal, window)
        copies = [t.clone() for t in got]
        torch.cuda.synchronize()
        assert m.fa_device_status() == 0
        for name, a, b, c in zip(("dq", "dk", "dv"), ref, got, copies):
            assert torch.equal(a, b), name
            assert torch.equal(a, c), name + " (stream-ordered copy)"


@pytest.mark.parametrize("B,Hq,Hkv,T,D,dt,causal", [
    (2, 8, 2, 2048, 64, "fp16", True),      # one query tile per CTA, two score buffers
    (2, 8, 8, 1024, 128, "bf16", False),    # the same at D = 128
    (2, 8, 2, 2048, 256, "fp16", True),     # D = 256: 64-key tiles, two score buffers
])
def test_two_buffer_forward_repeats_bitwise(B, Hq, Hkv, T, D, dt, causal):
    """Forward configurations with two score buffers per query tile, run
    back to back many times with each kernel launched while the previous one
    finishes: every run bitwise equal to the first and no bounded wait gives
    up. (A late softmax warp once found the forward's single O-ready barrier
    two phases past its wait, which then never ended.)"""
    m = fa()
    w = fa_inputs.Workload("rep", B, Hq, Hkv, T, T, D, dt, causal, 0, seed=91)
    x = fa_inputs.make_inputs(w)
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(m.fa_bwd_workspace_size(B, Hq, T), dtype=torch.uint8, device=dev)
    m.fa_device_status(clear=True)
    runs = []
    for r in range(100):
        m.fa_fwd(q, k, v, o, lse, w.scale, causal, 0)
        m.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, w.scale, causal, 0, workspace=ws)
        if r % 25 == 0 or r == 99:  # copies on the stream; the runs between chain directly
            runs.append([t.clone() for t in (o, lse, dq, dk, dv)])
    torch.cuda.synchronize()
    assert m.fa_device_status() == 0, "a bounded device wait gave up"
    for got in runs[1:]:
        for name, a, b in zip(("o", "lse", "dq", "dk", "dv"), runs[0], got):
            assert torch.equal(a, b), name
    assert bool(torch.isfinite(runs[0][0]).all())


@pytest.mark.parametrize("B,Hq,Hkv,Tq,Tkv,D,dt,causal,window", [
    (2, 8, 2, 1024, 1024, 128, "bf16", True, 0),     # tile kernels, dQ beside dK/dV
    (2, 4, 4, 640, 640, 64, "fp16", False, 0),       # tile kernels, dQ after dK/dV
    (2, 8, 2, 4, 1000, 128, "fp16", False, 0),       # short queries
    (1, 4, 2, 300, 300, 256, "bf16", True, 0),       # D = 256
])
def test_cuda_graph_capture_and_replay(B, Hq, Hkv, Tq, Tkv, D, dt, causal, window):
    """fa_fwd + fa_bwd captured into a CUDA graph (consecutive kernels become
    programmatic edges) and replayed on new inputs copied into the captured
    buffers: bitwise what the same calls give outside the graph."""
    m = fa()
    w = fa_inputs.Workload("graph", B, Hq, Hkv, Tq, Tkv, D, dt, causal, window, seed=61)
    x = fa_inputs.make_inputs(w)
    x2 = fa_inputs.make_inputs(fa_inputs.Workload("graph2", B, Hq, Hkv, Tq, Tkv, D, dt, causal,
                                                  window, seed=62))
    dev = torch.device("cuda")
    bufs = {n: x[n].to(dev) for n in ("q", "k", "v", "do")}
    q, k, v, do = (bufs[n] for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(m.fa_bwd_workspace_size(B, Hq, Tq), dtype=torch.uint8, device=dev)

    def step(stream=None):
        m.fa_fwd(q, k, v, o, lse, w.scale, causal, window, stream=stream)
        m.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, w.scale, causal, window, workspace=ws,
                 stream=stream)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):   # warm-up (tensor maps, kernel attributes) off the capture
        step(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(torch.cuda.current_stream())
    for inputs in (x2, x):
        for n in ("q", "k", "v", "do"):
            bufs[n].copy_(inputs[n].to(dev))
        g.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in (o, lse, dq, dk, dv)]
        step()
        torch.cuda.synchronize()
        assert m.fa_device_status() == 0
        for name, a, b in zip(("o", "lse", "dq", "dk", "dv"), got, (o, lse, dq, dk, dv)):
            assert torch.equal(a, b), name
