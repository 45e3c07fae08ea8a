"""cattn_forward_noalloc: the forward for callers that cannot allocate device
memory on the call path (for example a plug-in whose host engine plans all
device memory at start-up and forbids later allocations).

The GPU test calls the entry point through the C ABI on several problems in a
row (causal ones, then non-causal ones whose keys are split, so that their
partial outputs share the array), and checks each result against
cattn_forward run with an ordinary caller-supplied workspace.  This file is
collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from softmax_free_attention_gb300 import attention, native, workloads

OUT_TOL = 2e-2   # x max|v|, bf16 inputs with fp32 accumulation
TEL_TOL = 1e-3   # relative, Yat row mass and max kappa


@pytest.fixture(scope="module")
def lib():
    from softmax_free_attention_gb300 import build
    build.build()
    return native.load()


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def test_noalloc_rejects_oversized_problem_on_the_host(lib):
    # bf16 Yat workspace for these sizes is far above the fixed 16 MiB array;
    # the call must fail before it touches any pointer or the GPU
    p = native.Problem(B=64, h=32, hkv=32, Tq=4096, Tk=4096, dk=128, dv=128, dtype=native.BF16,
                       causal=1, scale=0.088, flags=0)
    fake = ctypes.c_void_p(1 << 20)
    rc = lib.cattn_forward_noalloc(native.YAT, ctypes.byref(p), fake, fake, fake, fake, fake, None,
                                   fake, None, None, None)
    assert rc == native.ERR_SCRATCH_LIMIT
    assert b"noalloc" in lib.cattn_error_string(rc)
    p.B, p.flags = 1, native.FLAG_NORMS_READY  # norms can never be supplied here
    rc = lib.cattn_forward_noalloc(native.YAT, ctypes.byref(p), fake, fake, fake, fake, fake, None,
                                   fake, None, None, None)
    assert rc == native.ERR_INVALID_ARG


def _problem_inputs(name, B, h, hkv, Tq, Tk, d, causal, seed):
    w = workloads.Workload(name, B=B, h=h, hkv=hkv, Tq=Tq, Tk=Tk, dk=d, dv=d, dtype="bf16",
                           causal=causal, qk_factor=2.0, yat_param="softplus_uniform", seed=seed)
    return w, workloads.generate(w, device="cuda")


@pytest.mark.gpu
def test_noalloc_matches_forward_on_two_calls_in_a_row(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # different problems back to back: each call finds the previous one's
    # norms (and, for the last, key-split partials) in the shared scratch and
    # must not be affected by them; the last is non-causal with few query
    # rows, so its keys are split in two and the partials of both splits sit
    # in the shared array before the combine
    for (B, h, hkv, Tq, Tk, d, causal, seed) in [(2, 4, 2, 640, 640, 128, True, 11),
                                                 (1, 2, 2, 300, 300, 64, True, 12),
                                                 (1, 2, 2, 128, 2048, 64, False, 13),
                                                 (1, 2, 2, 128, 2048, 64, False, 14)]:
        w, inp = _problem_inputs("noalloc", B, h, hkv, Tq, Tk, d, causal, seed)
        q, k, v = inp["q"], inp["k"], inp["v"]
        b = torch.as_tensor(inp["yat_b"], device="cuda")
        eps = torch.as_tensor(inp["yat_eps"], device="cuda")
        ref_out, ref_mass, ref_max = attention.forward("yat", q, k, v, b=b, eps=eps, causal=causal,
                                                       scale=w.scale)
        prob = attention.make_problem(q, k, v, causal=causal, scale=w.scale)
        out = torch.empty_like(ref_out)
        mass = torch.empty_like(ref_mass)
        mx = torch.empty_like(ref_max)
        rc = lib.cattn_forward_noalloc(native.YAT, ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v),
                                       _ptr(b), _ptr(eps), None, _ptr(out), _ptr(mass), _ptr(mx),
                                       stream)
        assert rc == native.OK, native.error_string(rc)
        torch.cuda.synchronize()
        assert attention.check_status() == 0
        vmax = float(v.abs().max())
        err = (out.float() - ref_out.float()).abs().max().item()
        assert err <= OUT_TOL * vmax, f"out differs by {err}"
        for got, ref in ((mass, ref_mass), (mx, ref_max)):
            rel = ((got - ref).abs() / ref.abs().clamp_min(1e-30)).max().item()
            assert rel <= TEL_TOL, f"telemetry differs by {rel}"
    # a map that needs no scratch goes straight through
    out = torch.empty_like(ref_out)
    rc = lib.cattn_forward_noalloc(native.SOFTMAX, ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v),
                                   None, None, None, _ptr(out), None, None, stream)
    assert rc == native.OK
    ref = attention.forward("softmax", q, k, v, causal=causal, scale=w.scale, telemetry=False)[0]
    torch.cuda.synchronize()
    assert (out.float() - ref.float()).abs().max().item() <= OUT_TOL * float(v.abs().max())
