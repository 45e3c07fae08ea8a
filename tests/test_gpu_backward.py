"""GPU parity of the backward: dq, dk, dv and the per-head parameter gradients
of the CUDA path (through the C ABI) against the fp64 oracle's backward on the
same seeded inputs and the same dout.

Tolerance (bf16 inputs, fp32 accumulation; the weights W and the score
gradients C enter the tensor cores as bf16, each rounded to 2^-9 relative,
and the outputs are stored as bf16): every element of dq, dk and dv within
2e-2 of that tensor's largest oracle magnitude, the same normwise bound the
forward's output meets (2e-2 max|v|); each head's parameter gradient (a sum
over all of its pairs) within 2e-2 of the largest over the heads.
"""
import numpy as np
import pytest
import torch

import oracle
import parity_utils as pu
from softmax_free_attention_gb300 import attention, workloads

pytestmark = pytest.mark.gpu

VARIANTS = ["yat", "softmax", "stau"]
GRAD_TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    from softmax_free_attention_gb300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _wl(B, h, hkv, Tq, Tk, d, causal, seed, qk=1.0, name="bwd"):
    return workloads.Workload(name, B=B, h=h, hkv=hkv, Tq=Tq, Tk=Tk, dk=d, dv=d, dtype="bf16",
                              causal=causal, qk_factor=qk, yat_param="softplus_uniform", seed=seed)


def _params(variant, inp):
    return pu.params_for(variant, inp)


def run_gpu_backward(variant, inp, dout, *, causal, scale, yat_m=1):
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    do = dout.cuda()
    kw = _params(variant, inp)
    out, mass, _ = attention.forward(variant, q, k, v, causal=causal, scale=scale, yat_m=yat_m,
                                     **kw)
    res = attention.backward(variant, q, k, v, out, do, mass, causal=causal, scale=scale,
                             yat_m=yat_m, **kw)
    torch.cuda.synchronize()
    assert attention.check_status() == 0
    return res


def compare_grads(gpu, ora, where, tol=GRAD_TOL):
    dq, dk, dv, gp = gpu
    odq, odk, odv, op = ora
    for name, g, o in (("dq", dq, odq), ("dk", dk, odk), ("dv", dv, odv)):
        g = pu.to_np(g)
        assert np.isfinite(g).all(), f"{where}: non-finite {name}"
        scale = float(np.abs(o).max()) if o.size else 0.0
        err = float(np.abs(g - o).max()) if o.size else 0.0
        assert err <= tol * scale + 1e-6, f"{where}: {name} max err {err:.3e} vs max {scale:.3e}"
    assert sorted(gp) == sorted(op), where
    for name in op:
        g = pu.to_np(gp[name])
        o = op[name]
        err = float(np.abs(g - o).max())
        lim = tol * float(np.abs(o).max()) + 1e-6
        assert err <= lim, f"{where}: d{name} err {err:.3e} > {lim:.3e} ({g} vs {o})"


BWD_SHAPES = [
    # B, h, hkv, Tq, Tk, d, causal
    (1, 1, 1, 1, 1, 64, True),
    (1, 2, 2, 2, 2, 64, True),
    (2, 2, 1, 127, 127, 64, True),
    (1, 2, 2, 128, 128, 128, True),
    (1, 2, 2, 129, 129, 128, True),
    (1, 2, 1, 384, 384, 128, True),
    (2, 2, 2, 640, 640, 64, True),
    (1, 2, 2, 300, 300, 128, False),
    (1, 4, 2, 200, 700, 128, False),
    (1, 1, 1, 1, 129, 64, False),
    (1, 2, 1, 65, 1000, 64, False),
    (1, 8, 2, 200, 200, 64, True),      # four query heads per kv head
    (2, 4, 1, 150, 400, 128, False),
]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", BWD_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_backward_matches_oracle(variant, shape):
    B, h, hkv, Tq, Tk, d, causal = shape
    w = _wl(B, h, hkv, Tq, Tk, d, causal, seed=3 * Tq + Tk)
    inp = workloads.generate(w)
    dout = workloads.grad_output(w)
    gpu = run_gpu_backward(variant, inp, dout, causal=causal, scale=w.scale)
    ora = oracle.backward(variant, inp["q"], inp["k"], inp["v"], dout, causal=causal,
                          scale=w.scale, **_params(variant, inp))
    compare_grads(gpu, ora, f"{variant} {shape}")


DKV_SHAPES = [
    # B, h, hkv, Tq, Tk, dk, dv, causal: q/k rows wider than v rows
    (1, 2, 1, 200, 200, 128, 64, True),
    (2, 2, 2, 129, 129, 128, 64, True),
    (1, 4, 2, 130, 700, 128, 64, False),
]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", DKV_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_backward_dk_wider_than_dv(variant, shape):
    B, h, hkv, Tq, Tk, dk, dv, causal = shape
    w = workloads.Workload("bwd_dkv", B=B, h=h, hkv=hkv, Tq=Tq, Tk=Tk, dk=dk, dv=dv,
                           dtype="bf16", causal=causal, yat_param="softplus_uniform",
                           seed=5 * Tq + Tk)
    inp = workloads.generate(w)
    dout = workloads.grad_output(w)
    gpu = run_gpu_backward(variant, inp, dout, causal=causal, scale=w.scale)
    ora = oracle.backward(variant, inp["q"], inp["k"], inp["v"], dout, causal=causal,
                          scale=w.scale, **_params(variant, inp))
    compare_grads(gpu, ora, f"{variant} {shape}")


F32_SHAPES = [
    # B, h, hkv, Tq, Tk, dk, dv, causal
    (1, 4, 4, 256, 256, 32, 32, True),     # the fp32 workload's shape
    (1, 2, 1, 77, 77, 64, 64, True),
    (2, 2, 2, 100, 150, 128, 64, False),
    (1, 1, 1, 65, 65, 128, 128, True),
]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", F32_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_backward_fp32(variant, shape):
    """The CUDA-core fp32 backward, held to the fp32 bound 1e-4 of each
    tensor's largest magnitude."""
    B, h, hkv, Tq, Tk, dk, dv, causal = shape
    w = workloads.Workload("bwd32", B=B, h=h, hkv=hkv, Tq=Tq, Tk=Tk, dk=dk, dv=dv, dtype="f32",
                           causal=causal, yat_param="ln2", seed=Tq + 11)
    inp = workloads.generate(w)
    dout = workloads.grad_output(w)
    gpu = run_gpu_backward(variant, inp, dout, causal=causal, scale=w.scale)
    ora = oracle.backward(variant, inp["q"], inp["k"], inp["v"], dout, causal=causal,
                          scale=w.scale, **_params(variant, inp))
    compare_grads(gpu, ora, f"f32 {variant} {shape}", tol=1e-4)


@pytest.mark.parametrize("m", [2, 3])
@pytest.mark.parametrize("shape", [(1, 2, 1, 200, 200, 128, True), (1, 2, 2, 130, 300, 64, False)],
                         ids=lambda s: "x".join(map(str, s)))
def test_backward_yat_power(m, shape):
    B, h, hkv, Tq, Tk, d, causal = shape
    w = _wl(B, h, hkv, Tq, Tk, d, causal, seed=Tq + 17 * m)
    inp = workloads.generate(w)
    dout = workloads.grad_output(w)
    gpu = run_gpu_backward("yat", inp, dout, causal=causal, scale=w.scale, yat_m=m)
    ora = oracle.backward("yat", inp["q"], inp["k"], inp["v"], dout, causal=causal,
                          yat_m=m, **_params("yat", inp))
    compare_grads(gpu, ora, f"yat m={m} {shape}")


@pytest.mark.parametrize("variant", VARIANTS)
def test_backward_large_scores(variant):
    """q and k scaled by 4 (char-level GPT shapes, the q/k x4 recipe): sharper
    rows and, for Yat, a wide range of kappa."""
    w = _wl(2, 4, 4, 256, 256, 64, True, seed=5, qk=4.0)
    inp = workloads.generate(w)
    dout = workloads.grad_output(w)
    gpu = run_gpu_backward(variant, inp, dout, causal=True, scale=w.scale)
    ora = oracle.backward(variant, inp["q"], inp["k"], inp["v"], dout, causal=True,
                          scale=w.scale, **_params(variant, inp))
    compare_grads(gpu, ora, f"{variant} qk x4")


def test_backward_deterministic_and_empty():
    w = _wl(1, 4, 2, 300, 300, 128, True, seed=9)
    inp = workloads.generate(w)
    dout = workloads.grad_output(w)
    a = run_gpu_backward("yat", inp, dout, causal=True, scale=w.scale)
    b = run_gpu_backward("yat", inp, dout, causal=True, scale=w.scale)
    for x, y in zip(a[:3], b[:3]):
        assert torch.equal(x, y)
    # no query rows: zero gradients for k and v
    q = torch.zeros(1, 2, 0, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.randn(1, 2, 5, 64, device="cuda").bfloat16()
    v = torch.randn(1, 2, 5, 64, device="cuda").bfloat16()
    out = torch.zeros(1, 2, 0, 64, dtype=torch.bfloat16, device="cuda")
    mass = torch.zeros(1, 2, 0, device="cuda")
    dq, dk, dv, gp = attention.backward("softmax", q, k, v, out, out, mass)
    torch.cuda.synchronize()
    assert dk.abs().max().item() == 0 and dv.abs().max().item() == 0 and dq.numel() == 0


def test_backward_rejects_unsupported():
    q = torch.zeros(1, 1, 4, 96, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16, device="cuda")
    mass = torch.zeros(1, 1, 4, device="cuda")
    with pytest.raises(ValueError):
        attention.backward("softmax", q, q, v, out, out, mass)  # dk = 96
    f = torch.zeros(1, 1, 4, 48, device="cuda")
    with pytest.raises(ValueError):
        attention.backward("softmax", f, f, f, f, f, mass)  # fp32 width 48


# ---------------------------------------------------------------- full size

@pytest.fixture(scope="module")
def cfg3_bwd():
    w = workloads.WORKLOADS["cfg3"]
    return w, workloads.generate(w), workloads.grad_output(w)


@pytest.mark.parametrize("variant", VARIANTS)
def test_backward_cfg3_full_size_slices(variant, cfg3_bwd):
    """B=16 h=16 T=4096 d=128 causal on the GPU; the oracle on two whole
    (batch, head) slices (with h == hkv every slice is independent)."""
    w, inp, dout = cfg3_bwd
    dq, dk, dv, gp = run_gpu_backward(variant, inp, dout, causal=True, scale=w.scale)
    kw = _params(variant, inp)
    for bi, hd in ((0, 0), (w.B - 1, w.h - 1)):
        sub = {n: x[hd:hd + 1] for n, x in kw.items()}
        ora = oracle.backward(variant, inp["q"][bi:bi + 1, hd:hd + 1],
                              inp["k"][bi:bi + 1, hd:hd + 1], inp["v"][bi:bi + 1, hd:hd + 1],
                              dout[bi:bi + 1, hd:hd + 1], causal=True, scale=w.scale, **sub)
        gpu = (dq[bi:bi + 1, hd:hd + 1], dk[bi:bi + 1, hd:hd + 1], dv[bi:bi + 1, hd:hd + 1], {})
        compare_grads(gpu, ora[:3] + ({},), f"cfg3 {variant} slice ({bi}, {hd})")
    for name, g in gp.items():
        assert torch.isfinite(g).all(), name


def test_backward_cfg4_gqa_slice():
    """B=4 h=16 hkv=8 T=8192 causal, s^tau (the workload's own map): the
    oracle on one kv head and the two query heads that share it."""
    w = workloads.WORKLOADS["cfg4_gqa"]
    inp = workloads.generate(w)
    dout = workloads.grad_output(w)
    dq, dk, dv, _ = run_gpu_backward("stau", inp, dout, causal=True, scale=w.scale)
    bi, g = 1, 5
    heads = slice(2 * g, 2 * g + 2)
    kw = {n: x[heads] for n, x in _params("stau", inp).items()}
    ora = oracle.backward("stau", inp["q"][bi:bi + 1, heads], inp["k"][bi:bi + 1, g:g + 1],
                          inp["v"][bi:bi + 1, g:g + 1], dout[bi:bi + 1, heads], causal=True,
                          scale=w.scale, **kw)
    gpu = (dq[bi:bi + 1, heads], dk[bi:bi + 1, g:g + 1], dv[bi:bi + 1, g:g + 1], {})
    compare_grads(gpu, ora[:3] + ({},), "cfg4 stau kv head 5")


@pytest.mark.parametrize("causal", [True, False])
def test_yat_b_zero_ablation_forward_and_backward(causal):
    """The Yat page's b = 0 ablation (kappa = (q.k)^2 / (|q - k|^2 + eps)):
    the same kernels with every b_h = 0, forward and backward against the
    oracle with b = 0."""
    w = _wl(1, 4, 2, 257, 257 if causal else 400, 128, causal, seed=41)
    inp = workloads.generate(w)
    inp = dict(inp, yat_b=np.zeros_like(inp["yat_b"]))
    dout = workloads.grad_output(w)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    out, mass, mx = attention.forward("yat", q, k, v, b=inp["yat_b"], eps=inp["yat_eps"],
                                      causal=causal)
    torch.cuda.synchronize()
    ora_f = oracle.forward("yat", inp["q"], inp["k"], inp["v"], b=inp["yat_b"], eps=inp["yat_eps"],
                           causal=causal)
    pu.compare("yat", tuple(pu.to_np(t) for t in (out, mass, mx)), ora_f,
               float(inp["v"].abs().max()), inp["q"].dtype, where=f"yat b=0 causal={causal}")
    gpu = run_gpu_backward("yat", inp, dout, causal=causal, scale=w.scale)
    ora = oracle.backward("yat", inp["q"], inp["k"], inp["v"], dout, causal=causal,
                          **_params("yat", inp))
    compare_grads(gpu, ora, f"yat b=0 causal={causal}")


def test_backward_cfg5_cross_slice():
    """Non-causal cross-attention Tq=2048 Tk=32768 dk=128 dv=64 with q, k x8
    (B=1 h=32), Yat: the whole problem on the GPU, the oracle on two heads."""
    w = workloads.WORKLOADS["cfg5_cross"]
    inp = workloads.generate(w)
    dout = workloads.grad_output(w)
    dq, dk, dv, gp = run_gpu_backward("yat", inp, dout, causal=False, scale=w.scale)
    kw = _params("yat", inp)
    for hd in (0, w.h - 1):
        sub = {n: x[hd:hd + 1] for n, x in kw.items()}
        ora = oracle.backward("yat", inp["q"][:, hd:hd + 1], inp["k"][:, hd:hd + 1],
                              inp["v"][:, hd:hd + 1], dout[:, hd:hd + 1], causal=False, **sub)
        gpu = (dq[:, hd:hd + 1], dk[:, hd:hd + 1], dv[:, hd:hd + 1],
               {n: g[hd:hd + 1] for n, g in gp.items()})
        compare_grads(gpu, ora, f"cfg5 yat head {hd}")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_backward_yat_cancelling_numerator(dtype):
    """Edge case: the first (one-key) row of a causal head whose numerator
    q.k + b nearly cancels, so kappa is tiny and the gradient's factor
    2 / (q.k + b) is large; the row's weight is kappa / (kappa + 1e-9)."""
    w = workloads.Workload("bwd_cancel", B=1, h=2, hkv=2, Tq=130, Tk=130, dk=64, dv=64,
                           dtype=dtype, causal=True, yat_param="ln2", seed=23)
    inp = workloads.generate(w)
    q = inp["q"].double()
    k = inp["k"].double().clone()
    b = float(inp["yat_b"][0])
    for target in (0.02, -0.005):  # head 0 and head 1
        hd = 0 if target > 0 else 1
        q0, k0 = q[0, hd, 0], k[0, hd, 0]
        k[0, hd, 0] = k0 - ((q0 @ k0 + b - target) / (q0 @ q0)) * q0
    inp = dict(inp, k=k.to(inp["k"].dtype))
    dout = workloads.grad_output(w)
    gpu = run_gpu_backward("yat", inp, dout, causal=True, scale=w.scale)
    ora = oracle.backward("yat", inp["q"], inp["k"], inp["v"], dout, causal=True,
                          **_params("yat", inp))
    num = float(inp["q"][0, 0, 0].double() @ inp["k"][0, 0, 0].double()) + b
    compare_grads(gpu, ora, f"yat cancelling numerator {dtype} (q.k + b = {num:.3g})",
                  tol=GRAD_TOL if dtype == "bf16" else 1e-4)


WIDTH_SHAPES = [  # dtype, B, h, hkv, Tq, Tk, dk, dv, causal
    ("bf16", 1, 2, 1, 100, 100, 32, 32, True),
    ("bf16", 1, 2, 2, 70, 140, 64, 128, False),
    ("bf16", 1, 2, 2, 90, 90, 128, 32, True),
    ("f32", 1, 2, 2, 80, 80, 64, 32, True),
    ("f32", 1, 2, 1, 50, 120, 32, 128, False),
]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", WIDTH_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_backward_cuda_core_widths(variant, shape):
    """Width pairs without tensor-core tiles: the CUDA-core backward for bf16
    (gradients rounded to bf16: the bf16 bound) and fp32 (the fp32 bound)."""
    dtype, B, h, hkv, Tq, Tk, dk, dv, causal = shape
    w = workloads.Workload("bwd_widths", B=B, h=h, hkv=hkv, Tq=Tq, Tk=Tk, dk=dk, dv=dv,
                           dtype=dtype, causal=causal, yat_param="softplus_uniform",
                           seed=Tq + dk + 3 * dv)
    inp = workloads.generate(w)
    dout = workloads.grad_output(w)
    gpu = run_gpu_backward(variant, inp, dout, causal=causal, scale=w.scale)
    ora = oracle.backward(variant, inp["q"], inp["k"], inp["v"], dout, causal=causal,
                          scale=w.scale, **_params(variant, inp))
    compare_grads(gpu, ora, f"{variant} {shape}", tol=GRAD_TOL if dtype == "bf16" else 1e-4)
