"""Python entry points over the C ABI (torch tensors in, torch tensors out).

PyTorch supplies device memory and the current stream; the library's CUDA
kernels do every step of the forward.  Host (CPU) tensors are accepted too:
they are copied to the GPU, the forward runs there, and the results are copied
back; this is the end-to-end form of the same call.
"""
from __future__ import annotations

import ctypes
import math

import torch

from . import native

_VARIANTS = {"softmax": native.SOFTMAX, "yat": native.YAT, "stau": native.STAU,
             native.SOFTMAX: native.SOFTMAX, native.YAT: native.YAT, native.STAU: native.STAU}
_DTYPES = {torch.float32: native.F32, torch.bfloat16: native.BF16}


def variant_id(variant) -> int:
    try:
        return _VARIANTS[variant]
    except KeyError:
        raise ValueError(f"unknown variant {variant!r}; use 'yat', 'softmax' or 'stau'") from None


def make_problem(q, k, v, *, causal=False, scale=None, norms_ready=False,
                 yat_m=1) -> native.Problem:
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D: [B, h, Tq, dk], [B, hkv, Tk, dk], [B, hkv, Tk, dv]")
    B, h, Tq, dk = q.shape
    Bk, hkv, Tk, dk2 = k.shape
    Bv, hkv2, Tk2, dv = v.shape
    if (Bk, dk2) != (B, dk) or (Bv, hkv2, Tk2) != (B, hkv, Tk):
        raise ValueError(f"inconsistent shapes q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    if not (q.dtype == k.dtype == v.dtype) or q.dtype not in _DTYPES:
        raise ValueError("q, k, v must share one dtype: torch.bfloat16 or torch.float32")
    if scale is None:
        scale = 1.0 / math.sqrt(dk)
    if int(yat_m) != yat_m or not 1 <= yat_m <= 3:
        raise ValueError("yat_m must be 1, 2 or 3")
    return native.Problem(B, h, hkv, Tq, Tk, dk, dv, _DTYPES[q.dtype], int(bool(causal)),
                          float(scale), native.FLAG_NORMS_READY if norms_ready else 0,
                          int(yat_m))


def workspace_bytes(variant, problem: native.Problem) -> int:
    return int(native.load().cattn_workspace_bytes(variant_id(variant), ctypes.byref(problem)))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _per_head(x, h, device, name):
    if x is None:
        return None
    t = torch.as_tensor(x, dtype=torch.float32)
    if t.numel() == 1:
        t = t.reshape(1).expand(h)
    t = t.reshape(-1).contiguous()
    if t.numel() != h:
        raise ValueError(f"{name} needs one value per query head ({h}), got {t.numel()}")
    return t.to(device)


def _stream_handle(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def key_norms(q, k, v, workspace, *, causal=False, scale=None):
    """Fill a Yat workspace with the squared k row norms (bf16 inputs).

    A later ``forward('yat', ..., workspace=workspace, norms_ready=True)`` on the
    same q, k, v skips this prologue.
    """
    prob = make_problem(q, k, v, causal=causal, scale=scale)
    lib = native.load()
    native.check(lib.cattn_key_norms(ctypes.byref(prob), _ptr(k), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(),
                                     _stream_handle(q.device)), "cattn_key_norms")


def forward(variant, q, k, v, *, b=None, eps=None, tau=None, causal=False, scale=None,
            out=None, row_mass=None, row_max=None, telemetry=True, workspace=None,
            norms_ready=False, yat_m=1):
    """Attention forward with a pluggable score-to-weight map.

    variant: 'yat' | 'softmax' | 'stau'.  q [B,h,Tq,dk], k [B,hkv,Tk,dk],
    v [B,hkv,Tk,dv], all torch.bfloat16 or all torch.float32, contiguous.
    b, eps (Yat) and eps, tau (s^tau): one value per query head (or a scalar).
    scale: softmax / s^tau score scale (default 1/sqrt(dk)); Yat ignores it.
    yat_m: Yat numerator (q.k + b)^{2 yat_m}, yat_m in {1, 2, 3}.

    Returns (out [B,h,Tq,dv], row_mass [B,h,Tq] or None, row_max [B,h,Tq] or None).
    CUDA tensors: runs asynchronously on the current stream.  CPU tensors: copied
    to the current CUDA device, computed there, and copied back into pinned host
    tensors (or into the host tensors passed as out / row_mass / row_max),
    pipelined over HOST_CHUNKS chunks of the batch (synchronous; one library
    call per chunk, so Yat's key-norm bound and the key split are those of the
    chunk).
    """
    vid = variant_id(variant)
    if q.device.type == "cpu":
        return _forward_from_host(vid, q, k, v, b=b, eps=eps, tau=tau, causal=causal,
                                  scale=scale, telemetry=telemetry, yat_m=yat_m, out=out,
                                  row_mass=row_mass, row_max=row_max)
    if q.device.type != "cuda":
        raise ValueError("tensors must live on a CUDA device or on the host")
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
        if t.device != q.device:
            raise ValueError("q, k, v must be on one device")
    prob = make_problem(q, k, v, causal=causal, scale=scale, norms_ready=norms_ready,
                        yat_m=yat_m)
    dev = q.device
    B, h, Tq, _ = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((B, h, Tq, dv), dtype=q.dtype, device=dev)
    if telemetry:
        if row_mass is None:
            row_mass = torch.empty((B, h, Tq), dtype=torch.float32, device=dev)
        if row_max is None:
            row_max = torch.empty((B, h, Tq), dtype=torch.float32, device=dev)
    bt = _per_head(b, h, dev, "b") if vid == native.YAT else None
    et = _per_head(eps, h, dev, "eps") if vid in (native.YAT, native.STAU) else None
    tt = _per_head(tau, h, dev, "tau") if vid == native.STAU else None
    lib = native.load()
    need = int(lib.cattn_workspace_bytes(vid, ctypes.byref(prob)))
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    status = lib.cattn_forward(vid, ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(bt),
                               _ptr(et), _ptr(tt), _ptr(out), _ptr(row_mass), _ptr(row_max),
                               _ptr(workspace), ws_bytes, _stream_handle(dev))
    native.check(status, "cattn_forward")
    return out, row_mass, row_max


def forward_entropy(variant, q, k, v, *, b=None, eps=None, tau=None, causal=False, scale=None,
                    workspace=None, norms_ready=False):
    """forward() on CUDA bf16 tensors, plus each row's normalised entropy of the
    map's weights accumulated in the same pass (cattn_forward_entropy).

    Returns (out, row_mass, row_max, row_entropy), the last [B, h, Tq] fp32.
    """
    vid = variant_id(variant)
    prob = make_problem(q, k, v, causal=causal, scale=scale, norms_ready=norms_ready)
    dev = q.device
    B, h, Tq, _ = q.shape
    out = torch.empty((B, h, Tq, v.shape[-1]), dtype=q.dtype, device=dev)
    row_mass = torch.empty((B, h, Tq), dtype=torch.float32, device=dev)
    row_max = torch.empty_like(row_mass)
    row_ent = torch.empty_like(row_mass)
    bt = _per_head(b, h, dev, "b") if vid == native.YAT else None
    et = _per_head(eps, h, dev, "eps") if vid in (native.YAT, native.STAU) else None
    tt = _per_head(tau, h, dev, "tau") if vid == native.STAU else None
    lib = native.load()
    need = int(lib.cattn_workspace_bytes(vid, ctypes.byref(prob)))
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    status = lib.cattn_forward_entropy(vid, ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v),
                                       _ptr(bt), _ptr(et), _ptr(tt), _ptr(out), _ptr(row_mass),
                                       _ptr(row_max), _ptr(row_ent), _ptr(workspace), ws_bytes,
                                       _stream_handle(dev))
    native.check(status, "cattn_forward_entropy")
    return out, row_mass, row_max, row_ent


HOST_CHUNKS = 8  # batch chunks of the host-buffer forward (copy / compute overlap)


def _forward_from_host(vid, q, k, v, *, b, eps, tau, causal, scale, telemetry, yat_m,
                       out=None, row_mass=None, row_max=None, chunks=None):
    """Host tensors in, host tensors out, through cattn_forward_host: the
    library pipelines the copies in, the forward and the copies out over
    chunks of the batch on three streams (the current stream computes).  The
    outputs go to the caller's host tensors, else to new pinned ones.
    Returns once they are on the host."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        if t.device.type != "cpu":
            raise ValueError("q, k, v must all be on the host or all on one CUDA device")
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    prob = make_problem(q, k, v, causal=causal, scale=scale, yat_m=yat_m)
    dev = torch.device("cuda", torch.cuda.current_device())
    B, h, Tq, _ = q.shape
    dv = v.shape[-1]

    def host_out(t, shape, dtype, name):
        if t is None:
            return torch.empty(shape, dtype=dtype, pin_memory=True)
        if t.device.type != "cpu" or tuple(t.shape) != shape or t.dtype != dtype or \
                not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous host tensor of shape {shape}, {dtype}")
        return t

    out = host_out(out, (B, h, Tq, dv), q.dtype, "out")
    mass = host_out(row_mass, (B, h, Tq), torch.float32, "row_mass") if telemetry else None
    mx = host_out(row_max, (B, h, Tq), torch.float32, "row_max") if telemetry else None
    qd, kd, vd = (torch.empty(t.shape, dtype=t.dtype, device=dev) for t in (q, k, v))
    od = torch.empty(out.shape, dtype=out.dtype, device=dev)
    massd = torch.empty(mass.shape, dtype=torch.float32, device=dev) if telemetry else None
    mxd = torch.empty(mx.shape, dtype=torch.float32, device=dev) if telemetry else None
    bt = _per_head(b, h, dev, "b") if vid == native.YAT else None
    et = _per_head(eps, h, dev, "eps") if vid in (native.YAT, native.STAU) else None
    tt = _per_head(tau, h, dev, "tau") if vid == native.STAU else None
    n = HOST_CHUNKS if chunks is None else int(chunks)
    lib = native.load()
    need = int(lib.cattn_forward_host_workspace_bytes(vid, ctypes.byref(prob), n))
    ws = torch.empty(need, dtype=torch.uint8, device=dev) if need else None
    compute = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    status = lib.cattn_forward_host(
        vid, ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(bt), _ptr(et), _ptr(tt),
        _ptr(out), _ptr(mass), _ptr(mx), _ptr(qd), _ptr(kd), _ptr(vd), _ptr(od), _ptr(massd),
        _ptr(mxd), _ptr(ws), need, n, ctypes.c_void_p(compute.cuda_stream),
        ctypes.c_void_p(s_in.cuda_stream), ctypes.c_void_p(s_out.cuda_stream))
    native.check(status, "cattn_forward_host")
    compute.synchronize()  # it waits for the last copy out
    return out, mass, mx


def tau_star(q, k, eps, *, causal=False, scale=None, return_moments=False, workspace=None):
    """tau* of the s^tau map per query head from one pass over the softmax
    scores ("s^tau: a focal-length knob for attention", closed form):
    Cov(s, ln phi(s)) / Var(ln phi(s)) over the allowed scores s = scale q.k of
    each head, pooled over the batch, phi = softplus + eps.

    q [B,h,Tq,dk], k [B,hkv,Tk,dk]: torch.bfloat16 CUDA tensors, dk 64 or 128.
    eps: one value per query head.  scale defaults to 1/sqrt(dk).
    Returns tau [h] (float32) and, with ``return_moments``, the per-head
    moments [h, 6] (float64: n, sum s, sum g, sum s g, sum g^2, g0).
    """
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q, k must be 4-D: [B, h, Tq, dk], [B, hkv, Tk, dk]")
    if q.device.type != "cuda" or k.device != q.device:
        raise ValueError("q and k must be CUDA tensors on one device")
    if not (q.is_contiguous() and k.is_contiguous()):
        raise ValueError("q and k must be contiguous")
    B, h, Tq, dk = q.shape
    # v is not read: a view of k stands in for its shape
    prob = make_problem(q, k, k, causal=causal, scale=scale)
    dev = q.device
    et = _per_head(eps, h, dev, "eps")
    lib = native.load()
    need = int(lib.cattn_tau_star_workspace_bytes(ctypes.byref(prob)))
    if need == 0:
        raise ValueError("unsupported problem for tau* (bf16, dk 64 or 128)")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    tau = torch.empty(h, dtype=torch.float32, device=dev)
    mom = torch.empty((h, 6), dtype=torch.float64, device=dev) if return_moments else None
    status = lib.cattn_tau_star(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(et), _ptr(tau),
                                _ptr(mom), _ptr(workspace),
                                workspace.numel() * workspace.element_size(),
                                _stream_handle(dev))
    native.check(status, "cattn_tau_star")
    return (tau, mom) if return_moments else tau


def row_stats(variant, q, k, row_mass, *, b=None, eps=None, tau=None, causal=False, scale=None):
    """Per-row statistics of the attention map (a second pass over the scores):
    normalised entropy, fraction of allowed keys with weight below 1e-6, and
    the sum of the ten largest weights; each [B, h, Tq] float32.

    row_mass: the ``row_mass`` the forward returned for the same inputs and map.
    bf16 CUDA tensors, dk 64 or 128.
    """
    vid = variant_id(variant)
    if q.dim() != 4 or k.dim() != 4 or q.device.type != "cuda":
        raise ValueError("q, k must be 4-D CUDA tensors")
    prob = make_problem(q, k, k, causal=causal, scale=scale)
    dev = q.device
    B, h, Tq, _ = q.shape
    bt = _per_head(b, h, dev, "b") if vid == native.YAT else None
    et = _per_head(eps, h, dev, "eps") if vid in (native.YAT, native.STAU) else None
    tt = _per_head(tau, h, dev, "tau") if vid == native.STAU else None
    lib = native.load()
    need = int(lib.cattn_row_stats_workspace_bytes(vid, ctypes.byref(prob)))
    if need == 0:
        raise ValueError("unsupported problem for row statistics (bf16, dk 64 or 128)")
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    ent, small, top = (torch.empty((B, h, Tq), dtype=torch.float32, device=dev) for _ in range(3))
    status = lib.cattn_row_stats(vid, ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(bt), _ptr(et),
                                 _ptr(tt), _ptr(row_mass.contiguous()), _ptr(ent), _ptr(small),
                                 _ptr(top), _ptr(ws), need, _stream_handle(dev))
    native.check(status, "cattn_row_stats")
    return ent, small, top


def backward(variant, q, k, v, out, dout, row_mass, *, b=None, eps=None, tau=None,
             causal=False, scale=None, yat_m=1, workspace=None):
    """Gradients of sum(dout * out) for the forward that produced ``out`` and
    ``row_mass`` from the same inputs and map.

    CUDA tensors, bf16 or fp32, widths as for the forward.  Returns
    (dq, dk, dv, dparams):
    dq, dk, dv shaped and typed like q, k, v (GQA: dk, dv summed over the query
    heads sharing a kv head); dparams a dict of fp32 [h] tensors -- Yat:
    'b', 'eps'; s^tau: 'eps', 'tau'; softmax: empty.  Runs asynchronously on
    the current stream.
    """
    vid = variant_id(variant)
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout")):
        if t.device.type != "cuda" or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous CUDA tensor")
    prob = make_problem(q, k, v, causal=causal, scale=scale, yat_m=yat_m)
    if tuple(out.shape) != (q.shape[0], q.shape[1], q.shape[2], v.shape[3]) or \
            dout.shape != out.shape or out.dtype != q.dtype or dout.dtype != q.dtype:
        raise ValueError("out and dout must be [B, h, Tq, dv] in the dtype of q")
    dev = q.device
    h = q.shape[1]
    lib = native.load()
    need = int(lib.cattn_backward_workspace_bytes(vid, ctypes.byref(prob)))
    if need == 0:
        raise ValueError("unsupported problem for the backward (widths 32, 64 or 128)")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    bt = _per_head(b, h, dev, "b") if vid == native.YAT else None
    et = _per_head(eps, h, dev, "eps") if vid in (native.YAT, native.STAU) else None
    tt = _per_head(tau, h, dev, "tau") if vid == native.STAU else None
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    names = {native.YAT: ("b", "eps"), native.STAU: ("eps", "tau")}.get(vid, ())
    grads = {n: torch.empty(h, dtype=torch.float32, device=dev) for n in names}
    status = lib.cattn_backward(vid, ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(out),
                                _ptr(dout), _ptr(bt), _ptr(et), _ptr(tt),
                                _ptr(row_mass.contiguous()), _ptr(dq), _ptr(dk), _ptr(dv),
                                _ptr(grads.get("b")), _ptr(grads.get("eps")),
                                _ptr(grads.get("tau")), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream_handle(dev))
    native.check(status, "cattn_backward")
    return dq, dk, dv, grads


def check_status(stream=None) -> int:
    """Synchronise `stream` (default: current) and return the kernels' wait status."""
    handle = ctypes.c_void_p(stream.cuda_stream if stream is not None
                             else torch.cuda.current_stream().cuda_stream)
    return int(native.load().cattn_check_status(handle))
