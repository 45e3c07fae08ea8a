"""The C-ABI library without a GPU: it loads, exports what include/cattn.h
declares, and rejects bad arguments on the host before touching CUDA.

Every call here fails validation on purpose (or never reaches CUDA), so the
same tests are safe on a machine with a GPU: no kernel is ever launched with
the placeholder pointers used below.
"""
import ctypes
import os
import re

import pytest

from softmax_free_attention_gb300 import native, workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from softmax_free_attention_gb300 import build
    build.build()
    return native.load()


def _declared_symbols():
    with open(os.path.join(ROOT, "include", "cattn.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"\b(cattn_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    declared = _declared_symbols()
    assert set(declared) == set(native.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name
    assert lib.cattn_version() == 100


def test_error_strings(lib):
    for code in range(7):
        assert lib.cattn_error_string(code)
    assert lib.cattn_error_string(99) == b"unknown status"


FAKE = ctypes.c_void_p(1 << 20)          # 16-byte aligned, never dereferenced
MISALIGNED = ctypes.c_void_p((1 << 20) + 8)


def prob(**kw):
    base = dict(B=1, h=4, hkv=4, Tq=256, Tk=256, dk=128, dv=128, dtype=native.BF16, causal=1,
                scale=0.088, flags=0)
    base.update(kw)
    return native.Problem(**base)


def validate(lib, variant, p, q=FAKE, k=FAKE, v=FAKE, b=FAKE, eps=FAKE, tau=FAKE, out=FAKE,
             ws=None, ws_bytes=0):
    return lib.cattn_validate(variant, ctypes.byref(p), q, k, v, b, eps, tau, out, ws, ws_bytes)


@pytest.mark.parametrize("kw,code", [
    (dict(h=3, hkv=2), native.ERR_SHAPE),               # h % hkv != 0
    (dict(Tq=256, Tk=128), native.ERR_SHAPE),           # causal needs Tq == Tk
    (dict(Tk=0, causal=0), native.ERR_SHAPE),
    (dict(B=-1), native.ERR_INVALID_ARG),
    (dict(hkv=0), native.ERR_INVALID_ARG),
    (dict(dtype=7), native.ERR_INVALID_ARG),
    (dict(scale=0.0), native.ERR_INVALID_ARG),
    (dict(scale=-1.0), native.ERR_INVALID_ARG),
    (dict(flags=4), native.ERR_INVALID_ARG),            # no such flag
    (dict(dk=96, dv=96), native.ERR_UNSUPPORTED),
    (dict(dk=64, dv=256), native.ERR_UNSUPPORTED),
    (dict(dk=48, dv=32), native.ERR_UNSUPPORTED),       # widths are 32, 64 or 128
])
def test_problem_rejections(lib, kw, code):
    assert validate(lib, native.SOFTMAX, prob(**kw)) == code
    assert lib.cattn_workspace_bytes(native.SOFTMAX, ctypes.byref(prob(**kw))) == 0


@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 128), (32, 64), (128, 32)])
def test_cuda_core_widths_need_no_workspace(lib, dk, dv):
    # bf16 widths without tensor-core tiles run on the CUDA-core kernel, which
    # needs no workspace; the tensor-core-only passes over q and k (tau*, row
    # statistics) take a key width of 64 or 128 whatever dv is
    p = prob(dk=dk, dv=dv)
    for variant in (native.SOFTMAX, native.YAT, native.STAU):
        assert lib.cattn_workspace_bytes(variant, ctypes.byref(p)) == 0
        assert validate(lib, variant, p) == native.OK
    tc_keys = dk in (64, 128)
    assert (lib.cattn_tau_star_workspace_bytes(ctypes.byref(p)) > 0) == tc_keys
    assert (lib.cattn_row_stats_workspace_bytes(native.YAT, ctypes.byref(p)) > 0) == tc_keys
    assert lib.cattn_backward_workspace_bytes(native.YAT, ctypes.byref(p)) > 0


def test_pointer_rejections(lib):
    p = prob()
    assert validate(lib, 9, p) == native.ERR_INVALID_ARG                       # unknown variant
    assert validate(lib, native.SOFTMAX, p, q=None) == native.ERR_INVALID_ARG
    assert validate(lib, native.SOFTMAX, p, out=None) == native.ERR_INVALID_ARG
    assert validate(lib, native.SOFTMAX, p, k=MISALIGNED) == native.ERR_UNSUPPORTED
    assert validate(lib, native.STAU, p, tau=None) == native.ERR_INVALID_ARG
    assert validate(lib, native.YAT, p, b=None) == native.ERR_INVALID_ARG
    # Yat bf16 needs a workspace of the advertised size, 256-byte aligned
    need = lib.cattn_workspace_bytes(native.YAT, ctypes.byref(p))
    assert need > 0
    assert validate(lib, native.YAT, p) == native.ERR_INVALID_ARG
    assert validate(lib, native.YAT, p, ws=FAKE, ws_bytes=need - 1) == native.ERR_SHAPE
    assert validate(lib, native.YAT, p, ws=ctypes.c_void_p((1 << 20) + 16),
                    ws_bytes=need) == native.ERR_UNSUPPORTED
    assert validate(lib, native.YAT, p, ws=FAKE, ws_bytes=need) == native.OK
    # every bf16 map needs at least the 256-byte work-unit ticket
    assert validate(lib, native.SOFTMAX, p) == native.ERR_INVALID_ARG
    assert validate(lib, native.SOFTMAX, p, ws=FAKE, ws_bytes=255) == native.ERR_SHAPE
    assert validate(lib, native.SOFTMAX, p, ws=FAKE, ws_bytes=256) == native.OK
    # the forward itself returns the same codes without touching the GPU
    assert lib.cattn_forward(native.SOFTMAX, ctypes.byref(prob(h=3, hkv=2)), FAKE, FAKE, FAKE,
                             None, None, None, FAKE, None, None, None, 0, None) == native.ERR_SHAPE
    assert lib.cattn_forward(native.YAT, ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, None,
                             FAKE, None, None, FAKE, need - 1, None) == native.ERR_SHAPE


def test_workspace_layout(lib):
    # 256-byte control block, then (Yat) nk [B*hkv, ceil(Tk/128)*128] fp32 and
    # the near-key list (one 8-byte entry per row and key split), each rounded
    # to 256 B
    p = prob(B=2, h=4, hkv=2, Tq=300, Tk=300, dk=64, dv=64)
    nk = (2 * 2 * 384 * 4 + 255) // 256 * 256
    near = (2 * 4 * 300 * 8 + 255) // 256 * 256
    assert lib.cattn_workspace_bytes(native.YAT, ctypes.byref(p)) == 256 + nk + near
    assert lib.cattn_workspace_bytes(native.SOFTMAX, ctypes.byref(p)) == 256
    assert lib.cattn_workspace_bytes(native.STAU, ctypes.byref(p)) == 256
    # fp32 (three-pass tf32 on the tensor cores): the control block, hi / lo
    # of q and k, hi / lo of v transposed with its keys padded to a multiple of
    # 128, then (Yat) |k|^2 and the near-key list; each part rounded to 256 B
    p32 = prob(dtype=native.F32, dk=32, dv=32)
    r256 = lambda x: (x + 255) // 256 * 256
    qk = r256(1 * 4 * 256 * 32 * 4)
    vt = r256(1 * 4 * 32 * 256 * 4)
    base32 = 256 + 4 * qk + 2 * vt
    assert lib.cattn_workspace_bytes(native.SOFTMAX, ctypes.byref(p32)) == base32
    assert lib.cattn_workspace_bytes(native.YAT, ctypes.byref(p32)) == \
        base32 + r256(1 * 4 * 256 * 4) + r256(1 * 4 * 256 * 8)
    # non-causal with two 256-row units and 17 key tiles: two key splits of 9
    # and 8 tiles, each leaving fp32 partials [2, B*h, Tq, dv] and [2, B*h, Tq, 4]
    ps = prob(B=1, h=2, hkv=2, Tq=200, Tk=2100, causal=0)
    part = 2 * 2 * 200 * 128 * 4 + 2 * 2 * 200 * 16
    assert lib.cattn_workspace_bytes(native.SOFTMAX, ctypes.byref(ps)) == 256 + part
    # causal problems are never split
    pc = prob(B=1, h=2, hkv=2, Tq=2100, Tk=2100)
    assert lib.cattn_workspace_bytes(native.SOFTMAX, ctypes.byref(pc)) == 256


def test_test_stall_flag_is_accepted(lib):
    # the timeout-path test flag (alone or with the norms flag) passes the checks
    for f in (native.FLAG_TEST_STALL, native.FLAG_TEST_STALL | native.FLAG_NORMS_READY):
        p = prob(flags=f)
        need = lib.cattn_workspace_bytes(native.YAT, ctypes.byref(p))
        assert need > 0
        assert validate(lib, native.YAT, p, ws=FAKE, ws_bytes=need) == native.OK


def test_yat_power_range(lib):
    for m, code in ((0, native.OK), (1, native.OK), (3, native.OK), (4, native.ERR_INVALID_ARG),
                    (-1, native.ERR_INVALID_ARG)):
        p = prob(yat_m=m)
        need = lib.cattn_workspace_bytes(native.YAT, ctypes.byref(p))
        assert validate(lib, native.YAT, p, ws=FAKE, ws_bytes=need) == code


def test_tau_star_workspace_and_argument_checks(lib):
    # 256-byte ticket, then the per-head moments [h][6] fp64 rounded to 256 B
    p = prob(B=2, h=5, hkv=5, Tq=300, Tk=300, dk=128, dv=64)
    assert lib.cattn_tau_star_workspace_bytes(ctypes.byref(p)) == 256 + 256
    assert lib.cattn_tau_star_workspace_bytes(ctypes.byref(prob(h=40, hkv=40))) == 256 + 2048
    # bf16 only, key widths the tensor-core path has
    assert lib.cattn_tau_star_workspace_bytes(ctypes.byref(prob(dtype=native.F32))) == 0
    assert lib.cattn_tau_star_workspace_bytes(ctypes.byref(prob(dk=32, dv=32))) == 0
    need = lib.cattn_tau_star_workspace_bytes(ctypes.byref(p))
    f = lib.cattn_tau_star
    # argument errors come back before any CUDA call
    assert f(None, FAKE, FAKE, FAKE, FAKE, None, FAKE, need, None) == native.ERR_INVALID_ARG
    assert f(ctypes.byref(p), FAKE, FAKE, None, FAKE, None, FAKE, need, None) == native.ERR_INVALID_ARG
    assert f(ctypes.byref(p), FAKE, FAKE, FAKE, None, None, FAKE, need, None) == native.ERR_INVALID_ARG
    assert f(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, None, FAKE, need - 1, None) == native.ERR_SHAPE
    assert f(ctypes.byref(prob(dtype=native.F32, dk=32, dv=32)), FAKE, FAKE, FAKE, FAKE, None,
             FAKE, need, None) == native.ERR_UNSUPPORTED
    assert f(ctypes.byref(prob(h=3, hkv=2)), FAKE, FAKE, FAKE, FAKE, None, FAKE, need,
             None) == native.ERR_SHAPE


def test_empty_problem_is_a_noop_on_the_host(lib):
    # B = 0: nothing to compute, accepted without pointers and without CUDA
    p = prob(B=0)
    assert validate(lib, native.SOFTMAX, p, q=None, k=None, v=None, out=None) == native.OK
    assert lib.cattn_forward(native.SOFTMAX, ctypes.byref(p), None, None, None, None, None, None,
                             None, None, None, None, 0, None) == native.OK


def test_python_problem_marshalling():
    import torch
    from softmax_free_attention_gb300 import attention
    q = torch.zeros(2, 4, 10, 64, dtype=torch.bfloat16)
    k = torch.zeros(2, 2, 12, 64, dtype=torch.bfloat16)
    v = torch.zeros(2, 2, 12, 64, dtype=torch.bfloat16)
    p = attention.make_problem(q, k, v, causal=False)
    assert (p.B, p.h, p.hkv, p.Tq, p.Tk, p.dk, p.dv, p.dtype) == (2, 4, 2, 10, 12, 64, 64, 1)
    assert p.scale == pytest.approx(1 / 8)
    with pytest.raises(ValueError):
        attention.make_problem(q, k, v[:, :, :5])
    with pytest.raises(ValueError):
        attention.make_problem(q, k.float(), v)
    with pytest.raises(ValueError):
        attention.variant_id("relu")


def test_workload_table_matches_stated_shapes():
    w = workloads.WORKLOADS
    assert (w["cfg3"].B, w["cfg3"].h, w["cfg3"].Tq, w["cfg3"].dk) == (16, 16, 4096, 128)
    assert w["cfg3"].flops() == pytest.approx(2 ** 40)
    assert (w["cfg4_gqa"].h, w["cfg4_gqa"].hkv, w["cfg4_gqa"].Tq) == (16, 8, 8192)
    assert (w["cfg5_cross"].Tq, w["cfg5_cross"].Tk, w["cfg5_cross"].dv) == (2048, 32768, 64)
    assert not w["cfg5_cross"].causal
    rows = workloads.sample_rows(w["cfg2_s1"])
    assert rows.min() >= 0 and rows.max() < 32 * 4 * 256


def _bwd(lib, variant, p, *, q=FAKE, k=FAKE, v=FAKE, out=FAKE, dout=FAKE, b=FAKE, eps=FAKE,
         tau=FAKE, mass=FAKE, dq=FAKE, dk=FAKE, dv=FAKE, ws=FAKE, ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = lib.cattn_backward_workspace_bytes(variant, ctypes.byref(p))
    return lib.cattn_backward(variant, ctypes.byref(p), q, k, v, out, dout, b, eps, tau, mass,
                              dq, dk, dv, None, None, None, ws, ws_bytes, None)


def test_backward_workspace_sizes(lib):
    # tensor cores: [h][2] fp64 parameter sums + key-norm maximum (256-byte
    # block), the [B*h, ceil(Tq/128)*128] float4 row scalars, and (Yat) the
    # key norms [B*hkv, ceil(Tk/128)*128] fp32
    p = prob(B=2, h=4, hkv=2, Tq=200, Tk=200)
    sm = lib.cattn_backward_workspace_bytes(native.SOFTMAX, ctypes.byref(p))
    ya = lib.cattn_backward_workspace_bytes(native.YAT, ctypes.byref(p))
    assert sm == 256 + 2 * 4 * 256 * 16
    assert ya == sm + 2 * 2 * 256 * 4
    # CUDA cores (fp32, or bf16 widths without tensor-core tiles): the rows' D and Z
    for q in (prob(dtype=native.F32, dk=32, dv=32, Tq=100, Tk=100), prob(dk=32, dv=64)):
        need = 256 + ((2 * q.B * q.h * q.Tq * 4 + 255) // 256) * 256
        assert lib.cattn_backward_workspace_bytes(native.YAT, ctypes.byref(q)) == need
    # unsupported widths and bad problems: 0
    assert lib.cattn_backward_workspace_bytes(native.YAT, ctypes.byref(prob(dk=96, dv=96))) == 0
    assert lib.cattn_backward_workspace_bytes(native.YAT, ctypes.byref(prob(h=3, hkv=2))) == 0
    assert lib.cattn_backward_workspace_bytes(9, ctypes.byref(prob())) == 0


def test_backward_argument_errors(lib):
    # every error below is reported before any CUDA call
    p = prob()
    assert lib.cattn_backward(native.SOFTMAX, None, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None,
                              FAKE, FAKE, FAKE, FAKE, None, None, None, FAKE, 1 << 20,
                              None) == native.ERR_INVALID_ARG
    assert _bwd(lib, 9, p, ws_bytes=1 << 20) == native.ERR_INVALID_ARG          # unknown map
    assert _bwd(lib, native.SOFTMAX, prob(dk=96, dv=96), ws_bytes=1 << 20) == native.ERR_UNSUPPORTED
    assert _bwd(lib, native.SOFTMAX, prob(h=3, hkv=2), ws_bytes=1 << 20) == native.ERR_SHAPE
    for name in ("q", "k", "v", "out", "dout", "mass", "dq", "dk", "dv", "ws"):
        assert _bwd(lib, native.SOFTMAX, p, **{name: None}) == native.ERR_INVALID_ARG, name
    for name in ("q", "k", "v", "out", "dout", "dq", "dk", "dv"):
        assert _bwd(lib, native.SOFTMAX, p, **{name: MISALIGNED}) == native.ERR_UNSUPPORTED, name
    assert _bwd(lib, native.SOFTMAX, p, ws=ctypes.c_void_p((1 << 20) + 16)) == native.ERR_UNSUPPORTED
    need = lib.cattn_backward_workspace_bytes(native.YAT, ctypes.byref(p))
    assert _bwd(lib, native.YAT, p, ws_bytes=need - 1) == native.ERR_SHAPE
    assert _bwd(lib, native.YAT, p, b=None) == native.ERR_INVALID_ARG
    assert _bwd(lib, native.YAT, p, eps=None) == native.ERR_INVALID_ARG
    assert _bwd(lib, native.STAU, p, tau=None) == native.ERR_INVALID_ARG
    assert _bwd(lib, native.STAU, p, eps=None) == native.ERR_INVALID_ARG
    assert _bwd(lib, native.SOFTMAX, prob(yat_m=4)) == native.ERR_INVALID_ARG


def test_host_forward_workspace_and_argument_checks(lib):
    """cattn_forward_host sizes its workspace for the largest chunk and
    rejects bad arguments on the host, before any CUDA call."""
    ws = lambda v, p: lib.cattn_workspace_bytes(v, ctypes.byref(p))
    hws = lambda v, p, n: lib.cattn_forward_host_workspace_bytes(v, ctypes.byref(p), n)
    p = prob(B=16, h=4, hkv=2, Tq=300, Tk=300, dk=64, dv=64)
    assert hws(native.YAT, p, 8) == ws(native.YAT, prob(B=2, h=4, hkv=2, Tq=300, Tk=300, dk=64,
                                                        dv=64))
    assert hws(native.YAT, p, 1) == ws(native.YAT, p)
    # 16 entries in 3 chunks: sizes 5 and 6; the larger one's workspace
    assert hws(native.YAT, p, 3) == ws(native.YAT, prob(B=6, h=4, hkv=2, Tq=300, Tk=300, dk=64,
                                                        dv=64))
    # more chunks than batch entries: one entry per chunk
    assert hws(native.SOFTMAX, p, 100) == ws(native.SOFTMAX, prob(B=1, h=4, hkv=2, Tq=300,
                                                                  Tk=300, dk=64, dv=64))
    # split problems need more room per entry when there are fewer units:
    # the size is the larger of the two chunk sizes' workspaces
    ps = prob(B=3, h=2, hkv=2, Tq=200, Tk=2100, causal=0)
    assert hws(native.SOFTMAX, ps, 2) == max(ws(native.SOFTMAX, prob(B=1, h=2, hkv=2, Tq=200,
                                                                     Tk=2100, causal=0)),
                                             ws(native.SOFTMAX, prob(B=2, h=2, hkv=2, Tq=200,
                                                                     Tk=2100, causal=0)))
    assert hws(native.SOFTMAX, p, 0) == 0 and hws(native.SOFTMAX, prob(B=0), 4) == 0

    need = hws(native.YAT, p, 4)

    def call(prob_=p, chunks=4, qh=FAKE, mass_h=None, mass_d=None, ws_ptr=FAKE, ws_bytes=need):
        return lib.cattn_forward_host(native.YAT, ctypes.byref(prob_), qh, FAKE, FAKE, FAKE,
                                      FAKE, None, FAKE, mass_h, None, FAKE, FAKE, FAKE, FAKE,
                                      mass_d, None, ws_ptr, ws_bytes, chunks, None, None, None)
    assert call(chunks=0) == native.ERR_INVALID_ARG
    assert call(qh=None) == native.ERR_INVALID_ARG
    assert call(mass_h=FAKE) == native.ERR_INVALID_ARG          # host telemetry, no device one
    assert call(mass_d=FAKE) == native.ERR_INVALID_ARG
    assert call(prob_=prob(B=16, h=4, hkv=2, Tq=300, Tk=300, dk=64, dv=64,
                           flags=native.FLAG_NORMS_READY)) == native.ERR_INVALID_ARG
    assert call(ws_bytes=need - 1) == native.ERR_SHAPE           # the chunk's workspace
    assert call(prob_=prob(B=16, h=3, hkv=2)) == native.ERR_SHAPE
    assert call(prob_=prob(B=0, h=4, hkv=2)) == native.OK        # empty: nothing enqueued


def test_log1p_polynomial_coefficients():
    """The s^tau map's log1p(e) = e P(e) on [0, 1] (csrc/maps.cuh): the
    coefficients as written, evaluated in fp32 Horner form like the kernels,
    stay within the stated 1e-5 relative error against numpy's log1p, tiny
    arguments included, and are the degree-5 Chebyshev interpolant they are
    said to be."""
    import numpy as np
    from numpy.polynomial import chebyshev, polynomial
    with open(os.path.join(ROOT, "softmax_free_attention_gb300", "csrc", "maps.cuh")) as f:
        text = f.read()
    coef = {int(i): float(c) for i, c in re.findall(r"kL1p(\d) = (-?[0-9.]+)f", text)}
    assert sorted(coef) == list(range(6))
    c32 = [np.float32(coef[i]) for i in range(6)]
    x = np.concatenate([np.geomspace(1e-30, 1e-3, 2000), np.linspace(1e-3, 1.0, 200001)])
    x = x.astype(np.float32)
    p = np.full_like(x, c32[5])
    for c in c32[4::-1]:
        p = (p * x + c).astype(np.float32)
    approx = (x * p).astype(np.float64)
    exact = np.log1p(x.astype(np.float64))
    assert (np.abs(approx - exact) / exact).max() < 1e-5
    # interpolation at the Chebyshev points, which exclude the end points
    ref = chebyshev.Chebyshev.interpolate(lambda t: np.log1p(t) / t, 5, domain=[0, 1])
    want = ref.convert(kind=polynomial.Polynomial).coef
    assert np.allclose(np.float32(want), c32, rtol=0, atol=2e-7)
