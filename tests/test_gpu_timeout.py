"""The forward kernel's bounded waits, driven to expiry on purpose.

CATTN_FLAG_TEST_STALL makes the tensor-core forward's MMA warp start with a
wait on a barrier that nothing completes.  The wait gives up after its short
limit, every role leaves its loop (copies already started land first, tensor
memory is released) and the kernel returns; cattn_check_status then reports
CATTN_ERR_TIMEOUT.  No fault and no hang: the limit ends the wait.  The next
ordinary call on the same context must succeed and match the oracle.
"""
import ctypes

import numpy as np
import pytest
import torch

import parity_utils as pu
from softmax_free_attention_gb300 import attention, native, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from softmax_free_attention_gb300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("variant", ["yat", "softmax", "stau"])
def test_stalled_wait_reports_timeout_then_recovers(variant):
    w = workloads.Workload("stall", B=2, h=4, hkv=2, Tq=300, Tk=300, dk=128, dv=128,
                           dtype="bf16", causal=True, qk_factor=1.0,
                           yat_param="softplus_uniform", seed=11)
    inp = workloads.generate(w)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    kw = pu.params_for(variant, inp)
    vid = attention.variant_id(variant)
    prob = attention.make_problem(q, k, v, causal=True, scale=w.scale)
    prob.flags = native.FLAG_TEST_STALL
    lib = native.load()
    need = int(lib.cattn_workspace_bytes(vid, ctypes.byref(prob)))
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    out = torch.empty((w.B, w.h, w.Tq, w.dv), dtype=q.dtype, device="cuda")
    mass = torch.empty((w.B, w.h, w.Tq), dtype=torch.float32, device="cuda")
    mx = torch.empty_like(mass)
    per_head = {n: torch.as_tensor(kw[n], dtype=torch.float32).cuda() if n in kw else None
                for n in ("b", "eps", "tau")}
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert attention.check_status() == native.OK
    status = lib.cattn_forward(vid, ctypes.byref(prob), ptr(q), ptr(k), ptr(v), ptr(per_head["b"]),
                               ptr(per_head["eps"]), ptr(per_head["tau"]), ptr(out), ptr(mass),
                               ptr(mx), ptr(ws), need, stream)
    assert status == native.OK  # the launch itself is fine
    assert lib.cattn_check_status(stream) == native.ERR_TIMEOUT
    # the status word was cleared by that check, and the context still works
    assert lib.cattn_check_status(stream) == native.OK
    pu.full_parity(variant, inp, causal=True, scale=w.scale, where=f"after stall {variant}")

