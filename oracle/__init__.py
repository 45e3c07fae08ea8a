"""fp64 CPU oracle for the pluggable-map attention forward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(``softmax_free_attention_gb300``) never imports it, and this package imports
nothing from the product path.

The arithmetic lives in ``cattn_oracle.c`` (plain C, double precision, one
query row at a time); this module only compiles it with ``gcc`` when needed
and marshals numpy arrays through ``ctypes``.  The definitions it follows are
cited in the C file's header:

* softmax and Yat branches -- "Softmax-Free Attention in JAX/Flax NNX",
  section "One module, two compatibility functions";
* the Yat kernel and its row mass -- "The Kernel Between the Roles";
* shapes, key-axis softmax, masks -- "NNX Scaled Dot-Product Attention";
* s^tau -- "s^tau: a focal-length knob for attention" (forum.trae.cn), core
  formula a_i = phi(s_i)^tau / sum_j phi(s_j)^tau, phi = softplus(s) + eps.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

SOFTMAX, YAT, STAU = 0, 1, 2
VARIANTS = {"softmax": SOFTMAX, "yat": YAT, "stau": STAU}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cattn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libcattn_oracle.so")
_lock = threading.Lock()
_lib = None


class _Problem(ctypes.Structure):
    _fields_ = [
        ("variant", ctypes.c_int),
        ("B", ctypes.c_int), ("h", ctypes.c_int), ("hkv", ctypes.c_int),
        ("Tq", ctypes.c_int), ("Tk", ctypes.c_int), ("dk", ctypes.c_int), ("dv", ctypes.c_int),
        ("causal", ctypes.c_int),
        ("scale", ctypes.c_double),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("b", ctypes.c_void_p), ("eps", ctypes.c_void_p), ("tau", ctypes.c_void_p),
        ("rows", ctypes.c_void_p), ("nrows", ctypes.c_int64),
        ("out", ctypes.c_void_p), ("row_mass", ctypes.c_void_p), ("row_max", ctypes.c_void_p),
        ("weights", ctypes.c_void_p),
        ("yat_m", ctypes.c_int),
    ]


def build(force: bool = False) -> str:
    """Compile cattn_oracle.c into libcattn_oracle.so next to it (gcc, -O2)."""
    with _lock:
        stale = (not os.path.exists(_LIB_PATH)
                 or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
        if force or stale:
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread",
                   "-o", tmp, _SRC, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        lib.oracle_forward.argtypes = [ctypes.POINTER(_Problem), ctypes.c_int]
        lib.oracle_forward.restype = ctypes.c_int
        lib.oracle_tau_star_scores.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_double]
        lib.oracle_tau_star_scores.restype = ctypes.c_double
        lib.oracle_tau_star.argtypes = [ctypes.POINTER(_Problem), ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_tau_star.restype = ctypes.c_int
        _lib = lib
    return _lib


def _as_f64(x, name):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: widen exactly on the host
        import torch
        x = x.detach().to(device="cpu", dtype=torch.float64).numpy()
    arr = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    return arr


def _per_head(x, h, name):
    if x is None:
        return None
    arr = _as_f64(x, name).reshape(-1)
    if arr.size == 1:
        arr = np.full(h, arr[0], dtype=np.float64)
    if arr.size != h:
        raise ValueError(f"{name} must have one value per query head ({h}), got {arr.size}")
    return arr


def forward(variant, q, k, v, *, b=None, eps=None, tau=None, causal=False, scale=None,
            rows=None, nthreads=None, return_weights=False, yat_m=1):
    """Attention forward in fp64.

    q: [B, h, Tq, dk]; k: [B, hkv, Tk, dk]; v: [B, hkv, Tk, dv] (numpy arrays or
    torch tensors of any float dtype; widened exactly to fp64).  b / eps / tau:
    one value per query head (or a scalar).  ``scale`` multiplies q.k for
    softmax and s^tau (default 1/sqrt(dk)); Yat uses the raw q.k.

    rows: optional flat indices into [B, h, Tq]; only those rows are computed
    and the outputs are returned in that order with a leading ``len(rows)``
    axis.  Without ``rows`` the outputs have the full [B, h, Tq(, dv)] shape.

    yat_m: the Yat numerator exponent is 2 * yat_m (an integer >= 1).

    Returns (out, row_mass, row_max) and, with ``return_weights``, the weight
    matrix [.., Tk] as a fourth element.
    """
    if int(yat_m) != yat_m or yat_m < 1:
        raise ValueError("yat_m must be an integer >= 1")
    variant = VARIANTS.get(variant, variant)
    q = _as_f64(q, "q")
    k = _as_f64(k, "k")
    v = _as_f64(v, "v")
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be 4-D [B, heads, T, d]")
    B, h, Tq, dk = q.shape
    Bk, hkv, Tk, dk2 = k.shape
    Bv, hkv2, Tk2, dv = v.shape
    if (Bk, dk2) != (B, dk) or (Bv, hkv2, Tk2) != (B, hkv, Tk):
        raise ValueError("inconsistent q/k/v shapes")
    if scale is None:
        scale = 1.0 / np.sqrt(dk)
    b = _per_head(b, h, "b")
    eps = _per_head(eps, h, "eps")
    tau = _per_head(tau, h, "tau")

    if rows is None:
        rows_arr = None
        nrows = B * h * Tq
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
        nrows = rows_arr.size
    out = np.zeros((nrows, dv), dtype=np.float64)
    row_mass = np.zeros(nrows, dtype=np.float64)
    row_max = np.zeros(nrows, dtype=np.float64)
    weights = np.zeros((nrows, Tk), dtype=np.float64) if return_weights else None

    def ptr(a):
        return None if a is None else a.ctypes.data

    prob = _Problem(variant, B, h, hkv, Tq, Tk, dk, dv, int(bool(causal)), float(scale),
                    ptr(q), ptr(k), ptr(v), ptr(b), ptr(eps), ptr(tau),
                    ptr(rows_arr), nrows, ptr(out), ptr(row_mass), ptr(row_max), ptr(weights),
                    int(yat_m))
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    rc = _load().oracle_forward(ctypes.byref(prob), int(nthreads))
    if rc == -2:
        raise FloatingPointError("oracle: phi^tau is not finite in fp64 for this input")
    if rc != 0:
        raise ValueError(f"oracle_forward failed with code {rc}")
    if rows_arr is None:
        out = out.reshape(B, h, Tq, dv)
        row_mass = row_mass.reshape(B, h, Tq)
        row_max = row_max.reshape(B, h, Tq)
        if weights is not None:
            weights = weights.reshape(B, h, Tq, Tk)
    if return_weights:
        return out, row_mass, row_max, weights
    return out, row_mass, row_max


def tau_star_scores(s, eps):
    """tau* = Cov(s, ln phi(s)) / Var(ln phi(s)) over a vector of scores, phi =
    softplus + eps ("s^tau: a focal-length knob for attention", the closed-form
    paragraph).  fp64; NaN for fewer than two scores."""
    arr = np.ascontiguousarray(np.asarray(s, dtype=np.float64).reshape(-1))
    return float(_load().oracle_tau_star_scores(arr.ctypes.data, arr.size, float(eps)))


def tau_star(q, k, eps, *, causal=False, scale=None):
    """tau* of every query head from the softmax scores s = scale * q.k of all
    allowed (row, key) pairs of that head, pooled over the batch.

    q: [B, h, Tq, dk]; k: [B, hkv, Tk, dk]; eps: one value per query head.
    Returns (tau [h], n [h]) in fp64, n = the number of allowed pairs.
    """
    q = _as_f64(q, "q")
    k = _as_f64(k, "k")
    if q.ndim != 4 or k.ndim != 4:
        raise ValueError("q, k must be 4-D [B, heads, T, d]")
    B, h, Tq, dk = q.shape
    Bk, hkv, Tk, dk2 = k.shape
    if (Bk, dk2) != (B, dk):
        raise ValueError("inconsistent q/k shapes")
    if scale is None:
        scale = 1.0 / np.sqrt(dk)
    eps = _per_head(eps, h, "eps")
    tau = np.zeros(h, dtype=np.float64)
    n = np.zeros(h, dtype=np.float64)
    prob = _Problem(STAU, B, h, hkv, Tq, Tk, dk, 1, int(bool(causal)), float(scale),
                    q.ctypes.data, k.ctypes.data, None, None, eps.ctypes.data, None,
                    None, 0, None, None, None, None, 1)
    rc = _load().oracle_tau_star(ctypes.byref(prob), tau.ctypes.data, n.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle_tau_star failed with code {rc}")
    return tau, n


def row_stats(variant, q, k, v, *, b=None, eps=None, tau=None, causal=False, scale=None,
              yat_m=1, rows=None):
    """Per-row statistics of the attention map, from the oracle's own weights:

    * normalised entropy  -sum_j w_j ln w_j / ln n  over the n allowed keys
      (0 for a row on one key, 1 for a row spread evenly; 0 when n = 1) --
      "The Kernel Between the Roles", section "The run";
    * the fraction of allowed keys whose weight is below 1e-6 (the s^tau page's
      attention sparsity);
    * the top-10 mass: the sum of the row's ten largest weights (the s^tau
      page's top-10 concentration).

    Returns three arrays shaped like row_mass ([B, h, Tq], or [len(rows)]).
    """
    out, _, _, w = forward(variant, q, k, v, b=b, eps=eps, tau=tau, causal=causal, scale=scale,
                           rows=rows, return_weights=True, yat_m=yat_m)
    B, h, Tq, _ = np.shape(q)
    Tk = np.shape(k)[2]
    w = w.reshape(-1, Tk)
    flat = np.arange(B * h * Tq) if rows is None else np.asarray(rows, dtype=np.int64).reshape(-1)
    t = flat % Tq
    n = np.minimum(t + 1, Tk) if causal else np.full(flat.shape, Tk)
    ent = np.zeros(len(flat))
    small = np.zeros(len(flat))
    top = np.zeros(len(flat))
    for r in range(len(flat)):
        wr = w[r, :n[r]]
        pos = wr[wr > 0]
        hsum = -np.sum(pos * np.log(pos))
        ent[r] = hsum / np.log(n[r]) if n[r] > 1 else 0.0
        small[r] = np.count_nonzero(wr < 1e-6) / n[r]
        top[r] = np.sum(np.sort(wr)[::-1][:10])
    shape = (B, h, Tq) if rows is None else (len(flat),)
    return ent.reshape(shape), small.reshape(shape), top.reshape(shape)


def backward(variant, q, k, v, dout, *, b=None, eps=None, tau=None, causal=False, scale=None,
             yat_m=1):
    """Gradients of L = sum(dout * out) through the attention forward, in fp64.

    Per (batch, query head) with the full score matrix: f_tj the map's
    unnormalised weight (softmax exp(s), s^tau phi(s)^tau, Yat kappa), Z_t =
    sum_j f_tj (plus the forward's 1e-9 for Yat), w = f / Z, dW = dout V^T and
    D_t = dout_t . out_t.  The chain rule through the normalisation gives
    dL/df_tj = (dW_tj - D_t) / Z_t, then
      softmax  dS = w (dW - D),                       ds/dq = scale k
      s^tau    dS = w (dW - D) tau sigma(s) / phi,    ds/dq = scale k,
               d tau = sum w (dW - D) ln phi,  d eps = sum w (dW - D) tau / phi
      Yat      g = (dW - D) / Z,  A = g 2m (q.k + b)^{2m-1} / den,
               E = -g kappa / den  (the gradient on den = max(d2, 0) + eps),
               d2 = |q|^2 + |k|^2 - 2 q.k with d d2/dq = 2 (q - k), zero where
               the clamp is active (d2 <= 0):
               dq_t = sum_j A_tj k_j + 2 sum_j E'_tj (q_t - k_j)
               dk_j = sum_t A_tj q_t + 2 sum_t E'_tj (k_j - q_t),  E' = E [d2 > 0]
               d b = sum A,  d eps = sum E
    and dv = w^T dout.  Masked pairs have f = 0 and no gradient.  GQA: the
    gradients of a kv head are summed over the query heads that share it.

    Returns (dq, dk, dv, dparams) with dparams a dict of per-head arrays
    ('b', 'eps' for Yat; 'eps', 'tau' for s^tau; empty for softmax).
    """
    variant = VARIANTS.get(variant, variant)
    q = _as_f64(q, "q")
    k = _as_f64(k, "k")
    v = _as_f64(v, "v")
    do = _as_f64(dout, "dout")
    B, h, Tq, dk = q.shape
    _, hkv, Tk, _ = k.shape
    if scale is None:
        scale = 1.0 / np.sqrt(dk)
    group = h // hkv
    bb = _per_head(b, h, "b")
    ee = _per_head(eps, h, "eps")
    tt = _per_head(tau, h, "tau")
    m = int(yat_m)
    dq = np.zeros_like(q)
    dkk = np.zeros_like(k)
    dvv = np.zeros_like(v)
    dpar = {}
    if variant == YAT:
        dpar = {"b": np.zeros(h), "eps": np.zeros(h)}
    elif variant == STAU:
        dpar = {"eps": np.zeros(h), "tau": np.zeros(h)}
    allowed = np.ones((Tq, Tk), dtype=bool)
    if causal:
        allowed = np.arange(Tk)[None, :] <= np.arange(Tq)[:, None]
    for bi in range(B):
        for i in range(h):
            g_ = i // group
            Q, K, V, dO = q[bi, i], k[bi, g_], v[bi, g_], do[bi, i]
            dots = Q @ K.T
            if variant == SOFTMAX:
                s_ = np.where(allowed, scale * dots, -np.inf)
                f = np.exp(s_ - s_.max(axis=1, keepdims=True))
                Z = f.sum(axis=1, keepdims=True)
            elif variant == STAU:
                s_ = scale * dots
                phi = np.logaddexp(0.0, s_) + ee[i]
                lf = np.where(allowed, tt[i] * np.log(phi), -np.inf)
                f = np.exp(lf - lf.max(axis=1, keepdims=True))
                Z = f.sum(axis=1, keepdims=True)
            else:
                num = dots + bb[i]
                d2 = (Q * Q).sum(axis=1)[:, None] + (K * K).sum(axis=1)[None, :] - 2.0 * dots
                den = np.maximum(d2, 0.0) + ee[i]
                f = np.where(allowed, num ** (2 * m) / den, 0.0)
                Z = f.sum(axis=1, keepdims=True) + 1e-9
            w = f / Z
            out = w @ V
            dW = dO @ V.T
            D = (dO * out).sum(axis=1, keepdims=True)
            dvv[bi, g_] += w.T @ dO
            if variant == SOFTMAX:
                dS = w * (dW - D)
                dq[bi, i] += scale * (dS @ K)
                dkk[bi, g_] += scale * (dS.T @ Q)
            elif variant == STAU:
                base = w * (dW - D)
                sig = 1.0 / (1.0 + np.exp(-s_))
                dS = base * tt[i] * sig / phi
                dq[bi, i] += scale * (dS @ K)
                dkk[bi, g_] += scale * (dS.T @ Q)
                dpar["tau"][i] += float(np.sum(base * np.log(phi)))
                dpar["eps"][i] += float(np.sum(base * tt[i] / phi))
            else:
                G = np.where(allowed, (dW - D) / Z, 0.0)
                A = G * 2 * m * num ** (2 * m - 1) / den
                E = -G * f / den
                Ea = np.where(d2 > 0.0, E, 0.0)
                dq[bi, i] += A @ K + 2.0 * (Ea.sum(axis=1)[:, None] * Q - Ea @ K)
                dkk[bi, g_] += A.T @ Q + 2.0 * (Ea.sum(axis=0)[:, None] * K - Ea.T @ Q)
                dpar["b"][i] += float(np.sum(A))
                dpar["eps"][i] += float(np.sum(E))
    return dq, dkk, dvv, dpar
