"""Pins for the fp64 oracle, against facts the pages and the mathematics fix.

Each test checks the oracle against something other than its own code: a
worked example printed on a page (fixtures under tests/golden/, each with its
citation), a hand derivation in exact rationals, a closed form, an invariant,
or a special case that reduces to a library routine (scipy's softmax).  The
cases are chosen so that a plausible slip in the oracle (a dropped bias, a
wrong sign in the distance, an unsquared distance, a scale applied to Yat,
the wrong key axis, a wrong GQA head map, a mask that leaks) fails one of
them.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.special

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def _arr(x):
    return np.asarray(x, dtype=np.float64)


# --------------------------------------------------------------------------
# softmax: the SDPA page's worked example and its quoted weights
# --------------------------------------------------------------------------

def test_sdpa_worked_example(golden_dir):
    g = _load(golden_dir, "sdpa_worked_example.json")
    q = _arr(g["q"])[None, None]
    k = _arr(g["k"])[None, None]
    v = _arr(g["v"])[None, None]
    out, lse, mx, w = oracle.forward("softmax", q, k, v, scale=1.0, return_weights=True)
    np.testing.assert_allclose(out[0, 0], _arr(g["out"]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(w[0, 0, 0], _arr(g["weights_row0"]), atol=1e-15)
    np.testing.assert_allclose(w[0, 0, 1], _arr(g["weights_row1"]), atol=1e-15)
    # default scale is 1/sqrt(d_k) = 1 for d_k = 1
    out2, _, _ = oracle.forward("softmax", q, k, v)
    np.testing.assert_array_equal(out2, out)
    # telemetry: max scaled score and log-sum-exp of the row
    assert mx[0, 0, 0] == pytest.approx(math.log(2.0), abs=1e-15)
    assert lse[0, 0, 0] == pytest.approx(math.log(3.0), abs=1e-15)  # log(2 + 1)
    assert lse[0, 0, 1] == pytest.approx(math.log(2.0), abs=1e-15)  # log(1 + 1)


def test_sdpa_quoted_weights(golden_dir):
    g = _load(golden_dir, "sdpa_score_examples.json")
    # scores [0.5, 0, 0, 0]: one query, d_k = 1, q = 1, keys carry the scores
    s = _arr(g["scores_a"])
    q = np.ones((1, 1, 1, 1))
    k = s.reshape(1, 1, -1, 1)
    v = np.eye(s.size).reshape(1, 1, s.size, s.size)  # out row = weight row
    out, _, _ = oracle.forward("softmax", q, k, v, scale=1.0)
    w = out[0, 0, 0]
    tol = g["page_rounding"]
    assert abs(w[0] - g["weight_first_a"]) <= tol
    for j in range(1, s.size):
        assert abs(w[j] - g["weight_other_a"]) <= tol
    # weights [1/4, 3/4] on scalar values [2, 6] give 5
    sb = _arr(g["scores_b"])
    out_b, _, _, wb = oracle.forward("softmax", q, sb.reshape(1, 1, -1, 1),
                                     _arr(g["values_b"]).reshape(1, 1, -1, 1), scale=1.0,
                                     return_weights=True)
    np.testing.assert_allclose(wb[0, 0, 0], _arr(g["weights_b"]), atol=1e-15)
    assert out_b[0, 0, 0, 0] == pytest.approx(g["out_b"], abs=1e-14)


def test_softmax_matches_scipy_and_key_axis():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((2, 3, 7, 5))
    k = rng.standard_normal((2, 3, 9, 5))
    v = rng.standard_normal((2, 3, 9, 4))
    scale = 0.37
    out, lse, mx, w = oracle.forward("softmax", q, k, v, scale=scale, return_weights=True)
    scores = scale * np.einsum("bhtd,bhjd->bhtj", q, k)
    ref_w = scipy.special.softmax(scores, axis=-1)  # key axis, not the query axis
    np.testing.assert_allclose(w, ref_w, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(out, ref_w @ v, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, scipy.special.logsumexp(scores, axis=-1), rtol=1e-13)
    np.testing.assert_allclose(mx, scores.max(-1), rtol=1e-15)
    # normalising over the query axis instead would give different weights
    assert not np.allclose(w, scipy.special.softmax(scores, axis=-2))


# --------------------------------------------------------------------------
# Yat: exact rational hand example, closed forms and kernel invariants
# --------------------------------------------------------------------------

def test_yat_hand_example_exact(golden_dir):
    g = _load(golden_dir, "yat_hand_example.json")
    k = _arr(g["k"])[None, None]
    v = _arr(g["v"])[None, None]
    q = np.stack([_arr(hd["q"]) for hd in g["heads"]])[None, :, None, :]  # [1, 2, 1, 2]
    b = [float(Fraction(hd["b"])) for hd in g["heads"]]
    eps = [float(Fraction(hd["eps"])) for hd in g["heads"]]
    # a score scale must not touch Yat: pass a deliberately odd one
    out, mass, mx, w = oracle.forward("yat", q, k, v, b=b, eps=eps, scale=0.123,
                                      return_weights=True)
    for i, hd in enumerate(g["heads"]):
        kap = [Fraction(x) for x in hd["kappa"]]
        m = Fraction(hd["mass"])
        assert sum(kap) == m  # the fixture is self-consistent
        assert mass[0, i, 0] == pytest.approx(float(m), rel=1e-15)
        assert mx[0, i, 0] == pytest.approx(float(Fraction(hd["row_max"])), rel=1e-15)
        denom = float(m) + 1e-9
        np.testing.assert_allclose(w[0, i, 0], [float(x) / denom for x in kap], rtol=1e-14)
        exp_out = [float(Fraction(x)) / denom for x in hd["weighted_value_sum"]]
        np.testing.assert_allclose(out[0, i, 0], exp_out, rtol=1e-14)


def _yat_kappa_matrix(x, b, eps):
    """Gram matrix kappa(x_i, x_j) recovered from the oracle's weights and mass."""
    n, d = x.shape
    q = x[None, None]
    _, mass, _, w = oracle.forward("yat", q, q, np.zeros((1, 1, n, 1)), b=[b], eps=[eps],
                                   return_weights=True)
    return w[0, 0] * (mass[0, 0][:, None] + 1e-9)


def test_yat_self_similarity_closed_form_and_symmetry():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((16, 6)) * 1.5
    b, eps = 0.8, 0.3
    kap = _yat_kappa_matrix(x, b, eps)
    # kappa(q, q) = (|q|^2 + b)^2 / eps  ("The Kernel Between the Roles")
    diag = (np.sum(x * x, axis=1) + b) ** 2 / eps
    np.testing.assert_allclose(np.diag(kap), diag, rtol=1e-12)
    # symmetric, nonnegative, and positive semidefinite (Schur product of a
    # polynomial kernel and an inverse-distance kernel)
    np.testing.assert_allclose(kap, kap.T, rtol=1e-12)
    assert (kap >= 0).all()
    evals = np.linalg.eigvalsh(0.5 * (kap + kap.T))
    assert evals.min() >= -1e-10 * np.trace(kap)


@pytest.mark.parametrize("m", [2, 3])
def test_yat_numerator_power_exact(m):
    # kappa_m = (q.k + b)^{2m} / (max(|q-k|^2, 0) + eps) ("The Kernel Between the
    # Roles", section "The run"), checked on small integers in exact rationals:
    # q = (1, 2); keys (3, 0), (1, 1), (-2, 1); b = 1/2, eps = 1/4
    q = np.array([[[[1.0, 2.0]]]])
    keys = [(3, 0), (1, 1), (-2, 1)]
    k = np.array([[[list(map(float, kk)) for kk in keys]]])
    v = np.array([[[[1.0], [10.0], [100.0]]]])
    b, eps = Fraction(1, 2), Fraction(1, 4)
    kap = []
    for kx, ky in keys:
        dotp = 1 * kx + 2 * ky
        d2 = (1 - kx) ** 2 + (2 - ky) ** 2
        kap.append((dotp + b) ** (2 * m) / (d2 + eps))
    mass_x = sum(kap)
    out, mass, mx = oracle.forward("yat", q, k, v, b=[float(b)], eps=[float(eps)], yat_m=m)
    assert mass[0, 0, 0] == pytest.approx(float(mass_x), rel=1e-14)
    assert mx[0, 0, 0] == pytest.approx(float(max(kap)), rel=1e-14)
    want = sum(kk * vv for kk, vv in zip(kap, (1, 10, 100))) / mass_x
    assert out[0, 0, 0, 0] == pytest.approx(float(want), rel=1e-9)
    # m = 1 is the base kernel, and the diagonal is (|q|^2 + b)^{2m} / eps
    base = oracle.forward("yat", q, k, v, b=[0.5], eps=[0.25])
    np.testing.assert_array_equal(oracle.forward("yat", q, k, v, b=[0.5], eps=[0.25],
                                                 yat_m=1)[1], base[1])
    x = np.random.default_rng(8).standard_normal((5, 4))
    _, mq, _, wq = oracle.forward("yat", x[None, None], x[None, None], np.zeros((1, 1, 5, 1)),
                                  b=[0.5], eps=[0.25], yat_m=m, return_weights=True)
    kq = wq[0, 0] * (mq[0, 0][:, None] + 1e-9)
    np.testing.assert_allclose(np.diag(kq), (np.sum(x * x, axis=1) + 0.5) ** (2 * m) / 0.25,
                               rtol=1e-12)
    np.testing.assert_allclose(kq, kq.T, rtol=1e-12)
    with pytest.raises(ValueError):
        oracle.forward("yat", q, k, v, b=[0.5], eps=[0.25], yat_m=0)


def test_yat_b0_orthogonal_scores_zero():
    # b = 0 and q orthogonal to k gives kappa = 0 whatever the distance
    q = np.array([[[[1.0, 0.0]]]])
    k = np.array([[[[0.0, 0.001], [0.0, 50.0], [3.0, 0.0]]]])
    v = np.array([[[[1.0], [2.0], [4.0]]]])
    _, mass, _, w = oracle.forward("yat", q, k, v, b=[0.0], eps=[0.5], return_weights=True)
    assert w[0, 0, 0, 0] == 0.0 and w[0, 0, 0, 1] == 0.0
    assert mass[0, 0, 0] == pytest.approx(9.0 / (4.0 + 0.5), rel=1e-15)  # only k3


def test_yat_rows_sum_to_mass_ratio_and_large_scores_finite():
    rng = np.random.default_rng(11)
    q = rng.standard_normal((1, 2, 8, 16)) * 16
    k = rng.standard_normal((1, 2, 8, 16)) * 16
    v = rng.standard_normal((1, 2, 8, 3))
    out, mass, mx, w = oracle.forward("yat", q, k, v, b=[0.5, 2.0], eps=[0.1, 3.0],
                                      causal=True, return_weights=True)
    np.testing.assert_allclose(w.sum(-1), mass / (mass + 1e-9), rtol=1e-14)
    assert np.isfinite(out).all() and (mx > 0).all()


# --------------------------------------------------------------------------
# s^tau: the page's focal example and the softmax equivalence
# --------------------------------------------------------------------------

def test_stau_focal_example(golden_dir):
    g = _load(golden_dir, "stau_focal_example.json")
    eps = g["eps"]
    phi = _arr(g["phi"])
    s = np.log(np.expm1(phi - eps))  # inverse of softplus, independent of the oracle
    q = np.ones((1, 1, 1, 1))
    k = s.reshape(1, 1, -1, 1)
    v = np.eye(3).reshape(1, 1, 3, 3)
    for case in g["cases"]:
        tau = case["tau"]
        out, lz, mx = oracle.forward("stau", q, k, v, eps=[eps], tau=[tau], scale=1.0)
        expect = phi ** tau / np.sum(phi ** tau)
        if "weights" in case:
            np.testing.assert_allclose(expect, case["weights"], rtol=1e-15)
        np.testing.assert_allclose(out[0, 0, 0], expect, rtol=1e-10, atol=1e-300)
        assert lz[0, 0, 0] == pytest.approx(math.log(np.sum(phi ** tau)), rel=1e-12)
        assert mx[0, 0, 0] == pytest.approx(s.max(), rel=1e-15)
    # tau = 20: only the largest survives
    out, _, _ = oracle.forward("stau", q, k, v, eps=[eps], tau=[20.0], scale=1.0)
    assert out[0, 0, 0, 0] >= 1 - 1e-15 and out[0, 0, 0, 2] < 1e-39


def test_stau_equals_softmax_of_tau_log_phi():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((2, 4, 6, 8))
    k = rng.standard_normal((2, 2, 10, 8))
    v = rng.standard_normal((2, 2, 10, 5))
    tau = np.array([1.0, 1.7, 3.2, 6.0])
    eps = np.array([1e-6, 1e-3, 0.2, 1e-6])
    scale = 1 / math.sqrt(8)
    out, lz, mx, w = oracle.forward("stau", q, k, v, eps=eps, tau=tau, scale=scale,
                                    return_weights=True)
    kk = np.repeat(k, 2, axis=1)  # GQA: query head i reads kv head i // 2
    vv = np.repeat(v, 2, axis=1)
    s = scale * np.einsum("bhtd,bhjd->bhtj", q, kk)
    sigma = tau[None, :, None, None] * np.log(np.logaddexp(0.0, s) + eps[None, :, None, None])
    ref_w = scipy.special.softmax(sigma, axis=-1)
    np.testing.assert_allclose(w, ref_w, rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(out, ref_w @ vv, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(lz, scipy.special.logsumexp(sigma, axis=-1), rtol=1e-12)
    np.testing.assert_allclose(mx, s.max(-1), rtol=1e-15)


def test_stau_tau_one_is_phi_proportional():
    rng = np.random.default_rng(4)
    s = rng.standard_normal(9) * 3
    q = np.ones((1, 1, 1, 1))
    _, _, _, w = oracle.forward("stau", q, s.reshape(1, 1, -1, 1), np.zeros((1, 1, 9, 1)),
                                eps=[0.05], tau=[1.0], scale=1.0, return_weights=True)
    phi = np.log1p(np.exp(s)) + 0.05
    np.testing.assert_allclose(w[0, 0, 0], phi / phi.sum(), rtol=1e-13)


# --------------------------------------------------------------------------
# every variant: masks, prefixes, GQA, permutations, constant values
# --------------------------------------------------------------------------

VARIANT_KW = {
    "softmax": {},
    "yat": {"b": [0.7, 1.1, 0.3, 2.0], "eps": [0.69, 0.2, 1.5, 0.05]},
    "stau": {"eps": [1e-6, 1e-6, 0.1, 0.01], "tau": [2.31, 1.0, 4.0, 1.5]},
}


@pytest.mark.parametrize("variant", ["softmax", "yat", "stau"])
def test_causal_row_equals_prefix_and_mask_is_exact_zero(variant):
    rng = np.random.default_rng(21)
    T = 12
    q = rng.standard_normal((1, 4, T, 6))
    k = rng.standard_normal((1, 4, T, 6))
    v = rng.standard_normal((1, 4, T, 3))
    kw = VARIANT_KW[variant]
    out, mass, mx, w = oracle.forward(variant, q, k, v, causal=True, return_weights=True, **kw)
    for t in range(T):
        assert (w[0, :, t, t + 1:] == 0.0).all()  # future keys get exactly zero weight
        o2, m2, x2 = oracle.forward(variant, q[:, :, t:t + 1], k[:, :, :t + 1], v[:, :, :t + 1],
                                    causal=False, **kw)
        np.testing.assert_allclose(out[:, :, t], o2[:, :, 0], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(mass[:, :, t], m2[:, :, 0], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(mx[:, :, t], x2[:, :, 0], rtol=1e-14)
    # row 0 attends only to key 0: its output is v[0] (scaled by mass/(mass+1e-9) for Yat)
    if variant != "yat":
        np.testing.assert_allclose(out[0, :, 0], v[0, :, 0], rtol=1e-14)


@pytest.mark.parametrize("variant", ["softmax", "yat", "stau"])
def test_gqa_equals_repeated_heads(variant):
    rng = np.random.default_rng(8)
    q = rng.standard_normal((2, 4, 5, 6))
    k = rng.standard_normal((2, 2, 7, 6))
    v = rng.standard_normal((2, 2, 7, 3))
    kw = VARIANT_KW[variant]
    a = oracle.forward(variant, q, k, v, **kw)
    r = oracle.forward(variant, q, np.repeat(k, 2, axis=1), np.repeat(v, 2, axis=1), **kw)
    for x, y in zip(a, r):
        np.testing.assert_array_equal(x, y)
    # a wrong group map (interleaved heads) would differ
    bad = oracle.forward(variant, q, np.tile(k, (1, 2, 1, 1)), np.tile(v, (1, 2, 1, 1)), **kw)
    assert not np.allclose(a[0], bad[0])


@pytest.mark.parametrize("variant", ["softmax", "yat", "stau"])
def test_key_permutation_and_constant_values(variant):
    rng = np.random.default_rng(9)
    q = rng.standard_normal((1, 4, 3, 4))
    k = rng.standard_normal((1, 4, 8, 4))
    v = rng.standard_normal((1, 4, 8, 2))
    kw = VARIANT_KW[variant]
    perm = rng.permutation(8)
    a = oracle.forward(variant, q, k, v, **kw)
    p = oracle.forward(variant, q, k[:, :, perm], v[:, :, perm], **kw)
    for x, y in zip(a, p):
        np.testing.assert_allclose(x, y, rtol=1e-13, atol=1e-14)
    const = np.broadcast_to(np.array([1.5, -2.0]), v.shape).copy()
    out, mass, _ = oracle.forward(variant, q, k, const, **kw)
    expect = np.broadcast_to(np.array([1.5, -2.0]), out.shape)
    if variant == "yat":
        expect = expect * (mass / (mass + 1e-9))[..., None]
    np.testing.assert_allclose(out, expect, rtol=1e-13)


def test_row_subset_matches_full():
    rng = np.random.default_rng(10)
    q = rng.standard_normal((2, 2, 9, 4))
    k = rng.standard_normal((2, 2, 9, 4))
    v = rng.standard_normal((2, 2, 9, 3))
    full = oracle.forward("yat", q, k, v, b=[1, 2], eps=[0.5, 0.25], causal=True)
    rows = np.array([0, 5, 17, 35])
    sub = oracle.forward("yat", q, k, v, b=[1, 2], eps=[0.5, 0.25], causal=True, rows=rows)
    np.testing.assert_array_equal(sub[0], full[0].reshape(-1, 3)[rows])
    np.testing.assert_array_equal(sub[1], full[1].reshape(-1)[rows])


def test_bad_arguments_rejected():
    q = np.zeros((1, 3, 2, 2))
    k = np.zeros((1, 2, 2, 2))
    with pytest.raises(ValueError):
        oracle.forward("softmax", q, k, np.zeros((1, 2, 2, 1)))  # 3 % 2 != 0
    with pytest.raises(ValueError):
        oracle.forward("yat", np.zeros((1, 1, 2, 2)), np.zeros((1, 1, 2, 2)),
                       np.zeros((1, 1, 2, 1)))  # Yat needs b and eps


# --------------------------------------------------------------------------
# the input generator's parametrisations (not oracle arithmetic)
# --------------------------------------------------------------------------

def test_generator_parametrisations():
    from softmax_free_attention_gb300 import workloads as wl
    # raw 0 through softplus gives log 2 ("One module, two compatibility functions")
    assert float(wl._softplus64(0.0)) == pytest.approx(math.log(2.0), rel=1e-15)
    # tau = softplus(1) + 1 = 2.3133, the "2.31" initial value on the s^tau page
    assert float(wl._softplus64(1.0)) + 1.0 == pytest.approx(2.3133, abs=5e-5)
    g1 = wl.generate(wl.WORKLOADS["cfg1_f32"])
    g2 = wl.generate(wl.WORKLOADS["cfg1_f32"])
    for key in ("q", "k", "v"):
        assert (g1[key] == g2[key]).all()  # seeded
    assert np.all(g1["yat_b"] == np.float32(math.log(2.0)))


# --------------------------------------------------------------------------
# tau* ("s^tau: a focal-length knob for attention", closed-form paragraph:
# tau* = Cov(s, log phi(s)) / Var(log phi(s)), per head, from the scores of
# one forward pass)
# --------------------------------------------------------------------------

def _ln_phi(s, eps):
    # softplus by its definition log(1 + e^s), in exact-enough fp64 for |s| < 30
    return math.log(math.log1p(math.exp(s)) + eps)


@pytest.mark.parametrize("s1,s2,eps", [(0.3, -1.2, 0.1), (2.5, 0.0, 1e-6), (-3.0, -2.0, 0.7)])
def test_tau_star_two_scores_closed_form(s1, s2, eps):
    # with two scores the least-squares slope is the secant slope: a wrong
    # log base, eps inside the softplus or a variance in the numerator fail it
    want = (s1 - s2) / (_ln_phi(s1, eps) - _ln_phi(s2, eps))
    assert oracle.tau_star_scores([s1, s2], eps) == pytest.approx(want, rel=1e-12)


def test_tau_star_matches_polyfit_and_invariances():
    rng = np.random.default_rng(5)
    s = rng.standard_normal(3001) * 1.7 + 0.4
    eps = 1e-6
    g = np.log(np.logaddexp(0.0, s) + eps)
    slope = np.polyfit(g, s, 1)[0]  # least squares s ~ tau g + C, a library routine
    t = oracle.tau_star_scores(s, eps)
    assert t == pytest.approx(slope, rel=1e-9)
    assert oracle.tau_star_scores(s[::-1], eps) == pytest.approx(t, rel=1e-12)
    assert oracle.tau_star_scores(np.concatenate([s, s]), eps) == pytest.approx(t, rel=1e-12)
    assert math.isnan(oracle.tau_star_scores([1.0], eps))


def test_tau_star_heads_gather_allowed_scores():
    # brute force on a tiny GQA problem: enumerate the allowed (row, key) scores
    # of each query head over the batch, then the score-level estimator
    rng = np.random.default_rng(6)
    B, h, hkv, T, d = 2, 4, 2, 7, 5
    q = rng.standard_normal((B, h, T, d))
    k = rng.standard_normal((B, hkv, T, d))
    eps = np.array([1e-6, 0.3, 1e-3, 2.0])
    scale = 0.45
    for causal in (True, False):
        tau, n = oracle.tau_star(q, k, eps, causal=causal, scale=scale)
        for i in range(h):
            sc = [scale * float(np.dot(q[b, i, t], k[b, i // (h // hkv), j]))
                  for b in range(B) for t in range(T) for j in range(T)
                  if not (causal and j > t)]
            assert n[i] == len(sc) == (B * T * (T + 1) // 2 if causal else B * T * T)
            assert tau[i] == pytest.approx(oracle.tau_star_scores(sc, eps[i]), rel=1e-12)


# --------------------------------------------------------------------------
# row statistics of the map (normalised entropy: "The Kernel Between the
# Roles", section "The run"; sparsity below 1e-6 and top-10 concentration:
# the s^tau page's fine-tuning comparison)
# --------------------------------------------------------------------------

def test_row_stats_uniform_onehot_and_two_keys():
    # equal scores give equal weights: entropy 1, top-10 mass 10/n, nothing small
    n = 16
    q = np.zeros((1, 1, 1, 4))
    k = np.zeros((1, 1, n, 4))
    v = np.zeros((1, 1, n, 1))
    ent, small, top = oracle.row_stats("softmax", q, k, v, scale=1.0)
    assert ent[0, 0, 0] == pytest.approx(1.0, rel=1e-12)
    assert small[0, 0, 0] == 0.0
    assert top[0, 0, 0] == pytest.approx(10 / n, rel=1e-12)
    # one key 60 logits ahead: one weight ~1, the rest e^-60 < 1e-6
    k2 = k.copy()
    k2[0, 0, 3, 0] = 60.0
    q2 = np.zeros((1, 1, 1, 4))
    q2[..., 0] = 1.0
    ent, small, top = oracle.row_stats("softmax", q2, k2, v, scale=1.0)
    assert ent[0, 0, 0] == pytest.approx(0.0, abs=1e-20)
    assert small[0, 0, 0] == pytest.approx((n - 1) / n, rel=1e-15)
    assert top[0, 0, 0] == pytest.approx(1.0, rel=1e-12)
    # two keys with weights p, 1-p: entropy -(p ln p + (1-p) ln(1-p)) / ln 2
    k3 = np.zeros((1, 1, 2, 4))
    k3[0, 0, 0, 0] = 1.0
    ent, small, top = oracle.row_stats("softmax", q2, k3, np.zeros((1, 1, 2, 1)), scale=1.0)
    p = math.e / (math.e + 1.0)
    assert ent[0, 0, 0] == pytest.approx(-(p * math.log(p) + (1 - p) * math.log(1 - p))
                                         / math.log(2), rel=1e-12)
    assert top[0, 0, 0] == pytest.approx(1.0, rel=1e-15)


def test_row_stats_causal_counts_allowed_keys_only():
    # causal row t has t + 1 keys; row 0 (one key) has entropy 0 and top-10 mass 1
    rng = np.random.default_rng(9)
    q = rng.standard_normal((1, 2, 12, 8))
    k = rng.standard_normal((1, 2, 12, 8))
    v = rng.standard_normal((1, 2, 12, 3))
    ent, small, top = oracle.row_stats("yat", q, k, v, b=[0.5, 1.0], eps=[0.3, 1e-3], causal=True)
    _, mass, _, w = oracle.forward("yat", q, k, v, b=[0.5, 1.0], eps=[0.3, 1e-3], causal=True,
                                   return_weights=True)
    wsum = mass / (mass + 1e-9)  # a Yat row's weights sum to M / (M + 1e-9)
    assert (ent[:, :, 0] == 0.0).all()
    # rows with at most ten keys put all their weight in the top ten
    np.testing.assert_allclose(top[:, :, :10], wsum[:, :, :10], rtol=1e-12)
    assert (ent >= 0).all() and (ent <= 1 + 1e-12).all()
    # a brute-force recount of one row from the weights
    wr = w[0, 1, 11]
    assert small[0, 1, 11] == np.count_nonzero(wr < 1e-6) / 12
    assert top[0, 1, 11] == pytest.approx(sum(sorted(wr, reverse=True)[:10]), rel=1e-12)


# --------------------------------------------------------------------------
# backward: gradients of sum(dout * out) against central differences of the
# (pinned) oracle forward, and softmax against torch autograd of the
# library's scaled_dot_product_attention
# --------------------------------------------------------------------------

def _fd_grads(variant, q, k, v, do, names, kw, h=1e-6):
    def loss(**over):
        a = dict(q=q, k=k, v=v)
        kk = dict(kw)
        for n_, x in over.items():
            (a if n_ in a else kk)[n_] = x
        out, _, _ = oracle.forward(variant, a["q"], a["k"], a["v"], **kk)
        return float(np.sum(out * do))

    grads = {}
    for n_ in names:
        base = dict(q=q, k=k, v=v, **kw)[n_]
        base = np.asarray(base, dtype=np.float64)
        g = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            x = base.copy()
            x[idx] += h
            lp = loss(**{n_: x})
            x[idx] -= 2 * h
            lm = loss(**{n_: x})
            g[idx] = (lp - lm) / (2 * h)
        grads[n_] = g
    return grads


@pytest.mark.parametrize("variant,kw", [
    ("softmax", dict(scale=0.7)),
    ("stau", dict(scale=0.7, eps=np.array([0.3, 0.1]), tau=np.array([1.7, 2.5]))),
    ("yat", dict(b=np.array([0.4, 0.9]), eps=np.array([0.5, 0.2]))),
    ("yat", dict(b=np.array([0.4, -0.6]), eps=np.array([0.5, 0.2]), yat_m=2)),
])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_central_differences(variant, kw, causal):
    # GQA (two query heads on one key/value head), dk != dv, and for the
    # non-causal case Tq != Tk, so a transposed operand or a wrong head map fails
    rng = np.random.default_rng(11)
    Tq, Tk = (5, 5) if causal else (4, 6)
    q = rng.standard_normal((1, 2, Tq, 3))
    k = rng.standard_normal((1, 1, Tk, 3))
    v = rng.standard_normal((1, 1, Tk, 2))
    do = rng.standard_normal((1, 2, Tq, 2))
    kw = dict(kw, causal=causal)
    dq, dk, dv, dpar = oracle.backward(variant, q, k, v, do, **kw)
    names = ["q", "k", "v"] + sorted(dpar)
    fd = _fd_grads(variant, q, k, v, do, names, kw)
    got = dict(q=dq, k=dk, v=dv, **dpar)
    for n_ in names:
        np.testing.assert_allclose(got[n_], fd[n_], rtol=1e-6, atol=1e-7, err_msg=n_)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_softmax_matches_torch_autograd(causal):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(12)
    q = rng.standard_normal((2, 4, 9, 8))
    k = rng.standard_normal((2, 2, 9, 8))
    v = rng.standard_normal((2, 2, 9, 5))
    do = rng.standard_normal((2, 4, 9, 5))
    dq, dk, dv, dpar = oracle.backward("softmax", q, k, v, do, causal=causal)
    assert dpar == {}
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    rep = lambda x: x.repeat_interleave(2, dim=1)
    out = torch.nn.functional.scaled_dot_product_attention(tq, rep(tk), rep(tv), is_causal=causal)
    out.backward(torch.tensor(do))
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_backward_invariants():
    # every row's weights sum to one (softmax, s^tau) or to M / (M + 1e-9)
    # (Yat), so the dv rows of one head sum to the weighted dout rows; softmax
    # is unchanged by adding one vector to every key, so its dk rows sum to 0
    rng = np.random.default_rng(13)
    q = rng.standard_normal((1, 1, 7, 4))
    k = rng.standard_normal((1, 1, 7, 4))
    v = rng.standard_normal((1, 1, 7, 3))
    do = rng.standard_normal((1, 1, 7, 3))
    for variant, kw in [("softmax", {}), ("stau", dict(eps=0.2, tau=3.0))]:
        dq, dk, dv, _ = oracle.backward(variant, q, k, v, do, causal=True, **kw)
        np.testing.assert_allclose(dv.sum(axis=2), do.sum(axis=2), atol=1e-12)
    _, dk, _, _ = oracle.backward("softmax", q, k, v, do, causal=True)
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12)
    _, mass, _ = oracle.forward("yat", q, k, v, b=0.3, eps=0.1, causal=True)
    _, _, dv, _ = oracle.backward("yat", q, k, v, do, b=0.3, eps=0.1, causal=True)
    ratio = mass / (mass + 1e-9)
    np.testing.assert_allclose(dv.sum(axis=2), (do * ratio[..., None]).sum(axis=2), atol=1e-12)
    # dout = 0 gives zero gradients; a one-key row gives w = 1 (softmax) and no dq
    z = oracle.backward("yat", q, k, v, np.zeros_like(do), b=0.3, eps=0.1)
    assert all(np.all(x == 0) for x in z[:3])
    dq, _, _, _ = oracle.backward("softmax", q[:, :, :1], k[:, :, :1], v[:, :, :1], do[:, :, :1])
    np.testing.assert_array_equal(dq, 0.0)


def test_yat_b_zero_is_squared_cosine_over_distance():
    # b = 0 (the Yat page's ablation): kappa = (q.k)^2 / (|q - k|^2 + eps), so
    # a key orthogonal to q gets zero weight and flipping a key's sign changes
    # only the distance term
    q = _arr([[[[1.0, 0.0]]]])
    k = _arr([[[[0.0, 2.0], [3.0, 0.0], [-3.0, 0.0]]]])
    v = _arr([[[[1.0], [2.0], [4.0]]]])
    out, mass, _, w = oracle.forward("yat", q, k, v, b=0.0, eps=1.0, return_weights=True)
    k1 = 9.0 / (4.0 + 1.0)    # q.k = 3, |q - k|^2 = 4
    k2 = 9.0 / (16.0 + 1.0)   # q.k = -3, |q - k|^2 = 16
    assert w[0, 0, 0, 0] == 0.0
    assert mass[0, 0, 0] == pytest.approx(k1 + k2, rel=1e-15)
    assert out[0, 0, 0, 0] == pytest.approx((2.0 * k1 + 4.0 * k2) / (k1 + k2 + 1e-9), rel=1e-14)
