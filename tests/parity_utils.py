"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
and the fp64 oracle on the same seeded inputs, and compare.

Tolerances (stated by the target for this path):
  out            max|gpu - oracle| <= 1e-4 * max|v| (fp32 inputs)
                                   <= 2e-2 * max|v| (bf16 inputs, fp32 accumulation)
  Yat telemetry  row mass and max kappa within 1e-3 relative
  softmax/s^tau  log-domain row mass and max score within 1e-3 * max(1, |value|)
"""
import numpy as np
import torch

import oracle
from softmax_free_attention_gb300 import attention

OUT_TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}
TEL_TOL = 1e-3


def params_for(variant, inputs):
    if variant == "yat":
        return dict(b=inputs["yat_b"], eps=inputs["yat_eps"])
    if variant == "stau":
        return dict(eps=inputs["stau_eps"], tau=inputs["tau"])
    return {}


def run_gpu(variant, inputs, *, causal, scale, two_step=False):
    """The forward through the C ABI on cuda:0; returns device tensors."""
    q, k, v = (inputs[n].cuda() for n in ("q", "k", "v"))
    kw = params_for(variant, inputs)
    if two_step and variant == "yat" and q.dtype == torch.bfloat16:
        # the launch sequence the benchmark times: norm prologue, then the
        # forward told that the norms are ready
        prob = attention.make_problem(q, k, v, causal=causal, scale=scale)
        ws = torch.empty(attention.workspace_bytes("yat", prob), dtype=torch.uint8, device="cuda")
        attention.key_norms(q, k, v, ws, causal=causal, scale=scale)
        res = attention.forward(variant, q, k, v, causal=causal, scale=scale, workspace=ws,
                                norms_ready=True, **kw)
    else:
        res = attention.forward(variant, q, k, v, causal=causal, scale=scale, **kw)
    torch.cuda.synchronize()
    assert attention.check_status() == 0
    return res


def run_oracle(variant, inputs, *, causal, scale, rows=None):
    kw = params_for(variant, inputs)
    return oracle.forward(variant, inputs["q"], inputs["k"], inputs["v"], causal=causal,
                          scale=scale, rows=rows, **kw)


def compare(variant, gpu, ora, vmax, dtype, where=""):
    """gpu, ora: (out, row_mass, row_max) as float64 numpy arrays of equal shape."""
    out_g, mass_g, max_g = gpu
    out_o, mass_o, max_o = ora
    assert np.isfinite(out_g).all(), f"{where}: non-finite output"
    err = np.abs(out_g - out_o).max() if out_o.size else 0.0
    tol = OUT_TOL[dtype] * vmax
    assert err <= tol, f"{where}: out max err {err:.3e} > {tol:.3e}"
    if variant == "yat":
        rel = np.abs(mass_g - mass_o) / np.maximum(np.abs(mass_o), 1e-30)
        assert rel.max() <= TEL_TOL, f"{where}: row mass rel err {rel.max():.3e}"
        rel = np.abs(max_g - max_o) / np.maximum(np.abs(max_o), 1e-30)
        assert rel.max() <= TEL_TOL, f"{where}: max kappa rel err {rel.max():.3e}"
    else:
        lim = TEL_TOL * np.maximum(1.0, np.abs(mass_o))
        assert (np.abs(mass_g - mass_o) <= lim).all(), \
            f"{where}: log mass err {np.abs(mass_g - mass_o).max():.3e}"
        lim = TEL_TOL * np.maximum(1.0, np.abs(max_o))
        assert (np.abs(max_g - max_o) <= lim).all(), \
            f"{where}: max score err {np.abs(max_g - max_o).max():.3e}"
    return err


def to_np(t):
    return t.detach().to("cpu", torch.float64).numpy()


def full_parity(variant, inputs, *, causal, scale, two_step=False, where=""):
    gpu = run_gpu(variant, inputs, causal=causal, scale=scale, two_step=two_step)
    ora = run_oracle(variant, inputs, causal=causal, scale=scale)
    vmax = float(inputs["v"].abs().max())
    return compare(variant, tuple(to_np(t) for t in gpu), ora, vmax, inputs["q"].dtype,
                   where=where)


def sampled_parity(variant, inputs, *, causal, scale, pairs, rows_per_pair, two_step=False,
                   where=""):
    """Full-size GPU run; oracle only on the given (batch, head) pairs and rows.

    Each pair becomes a one-head oracle problem (its query head, its kv head
    and its per-head parameters), so the oracle never widens the whole tensor.
    """
    out, mass, mx = run_gpu(variant, inputs, causal=causal, scale=scale, two_step=two_step)
    q, k, v = inputs["q"], inputs["k"], inputs["v"]
    h, hkv = q.shape[1], k.shape[1]
    vmax = float(v.abs().max())
    kw_all = params_for(variant, inputs)
    worst = 0.0
    for (bi, head) in pairs:
        g = head // (h // hkv)
        rows = np.asarray(rows_per_pair(bi, head), dtype=np.int64)
        sub = {n: (x[head:head + 1] if x is not None else None) for n, x in kw_all.items()}
        ora = oracle.forward(variant, q[bi:bi + 1, head:head + 1], k[bi:bi + 1, g:g + 1],
                             v[bi:bi + 1, g:g + 1], causal=causal, scale=scale, rows=rows, **sub)
        idx = torch.as_tensor(rows, device=out.device)
        gpu = (to_np(out[bi, head].index_select(0, idx)), to_np(mass[bi, head].index_select(0, idx)),
               to_np(mx[bi, head].index_select(0, idx)))
        worst = max(worst, compare(variant, gpu, ora, vmax, q.dtype,
                                   where=f"{where} b={bi} h={head}"))
    return worst
