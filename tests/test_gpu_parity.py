"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs, element by element.

Small problems are compared on every output; the full-size workloads are run
in the same launch sequence the benchmark times and compared on sampled rows
the oracle computes one by one.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import parity_utils as pu
from softmax_free_attention_gb300 import attention, workloads

pytestmark = pytest.mark.gpu

VARIANTS = ["yat", "softmax", "stau"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from softmax_free_attention_gb300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _wl(name, B, h, hkv, Tq, Tk, dk, dv, dtype="bf16", causal=True, qk=1.0, seed=0):
    return workloads.Workload(name, B=B, h=h, hkv=hkv, Tq=Tq, Tk=Tk, dk=dk, dv=dv, dtype=dtype,
                              causal=causal, qk_factor=qk, yat_param="softplus_uniform", seed=seed)


# ---------------------------------------------------------------- worked example

def test_sdpa_worked_example_on_gpu(golden_dir):
    """The SDPA page's example, zero-padded to a supported head width (which
    leaves every dot product and every output column unchanged)."""
    with open(os.path.join(golden_dir, "sdpa_worked_example.json")) as f:
        g = json.load(f)
    q = torch.zeros(1, 1, 2, 32)
    k = torch.zeros(1, 1, 2, 32)
    v = torch.zeros(1, 1, 2, 32)
    q[0, 0, :, :1] = torch.tensor(g["q"])
    k[0, 0, :, :1] = torch.tensor(g["k"])
    v[0, 0, :, :2] = torch.tensor(g["v"])
    out, lse, mx = attention.forward("softmax", q.cuda(), k.cuda(), v.cuda(), scale=1.0)
    torch.cuda.synchronize()
    np.testing.assert_allclose(out[0, 0, :, :2].cpu().numpy(), g["out"], atol=1e-6)
    assert out[0, 0, :, 2:].abs().max().item() == 0.0
    np.testing.assert_allclose(lse[0, 0].cpu().numpy(), [math.log(3), math.log(2)], atol=1e-6)
    # the tensor-core path on the same example (bf16 rounds ln 2 to 0.69140625)
    qb, kb, vb = (t.new_zeros(1, 1, 2, 64) for t in (q, k, v))
    qb[..., :32], kb[..., :32], vb[..., :32] = q, k, v
    ob, _, _ = attention.forward("softmax", qb.bfloat16().cuda(), kb.bfloat16().cuda(),
                                 vb.bfloat16().cuda(), scale=1.0)
    torch.cuda.synchronize()
    assert np.abs(ob[0, 0, :, :2].float().cpu().numpy() - np.array(g["out"])).max() <= 2e-2 * 6


# ---------------------------------------------------------------- ragged / edge shapes

SHAPES = [
    # B, h, hkv, Tq, Tk, dk, dv, causal
    (1, 2, 2, 1, 1, 64, 64, True),
    (1, 2, 2, 2, 2, 64, 64, True),
    (2, 2, 1, 127, 127, 64, 64, True),
    (1, 2, 2, 128, 128, 128, 128, True),
    (1, 2, 2, 129, 129, 128, 128, True),
    (1, 2, 2, 255, 255, 128, 64, True),
    (1, 2, 2, 300, 300, 128, 128, False),
    (1, 4, 2, 200, 700, 128, 64, False),
    (2, 2, 2, 640, 640, 64, 64, True),
    (1, 1, 1, 1, 129, 64, 64, False),
    (1, 2, 1, 384, 384, 128, 128, True),
    # more units than SMs: later units come from the work ticket; odd tile count
    (8, 8, 4, 1100, 1100, 64, 64, True),
    # non-causal with few units: the keys are split and the partials combined
    (1, 2, 2, 200, 2100, 128, 128, False),   # 2 splits of 9 and 8 key tiles
    (1, 1, 1, 130, 4100, 128, 64, False),    # 4 splits, the last one ragged
    (2, 2, 1, 64, 2048, 64, 64, False),      # 2 splits, GQA
    # causal with few query pairs and long rows: one wave, the heaviest unit
    # (the last pair) 17 key tiles, the last one ragged; GQA with 8 key tiles
    (1, 2, 2, 2100, 2100, 128, 128, True),
    (2, 2, 1, 1024, 1024, 64, 64, True),
]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_tensor_core_ragged(variant, shape):
    B, h, hkv, Tq, Tk, dk, dv, causal = shape
    w = _wl("ragged", B, h, hkv, Tq, Tk, dk, dv, causal=causal, seed=Tq * 7 + Tk)
    inp = workloads.generate(w)
    pu.full_parity(variant, inp, causal=causal, scale=w.scale, where=f"{variant} {shape}")


F32_SHAPES = [
    (1, 2, 2, 1, 1, 32, 32, True),
    (1, 2, 1, 77, 77, 64, 64, True),
    (2, 2, 2, 100, 150, 128, 64, False),
    (1, 1, 1, 65, 65, 128, 128, True),
]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", F32_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_fp32_ragged(variant, shape):
    B, h, hkv, Tq, Tk, dk, dv, causal = shape
    w = _wl("ragged32", B, h, hkv, Tq, Tk, dk, dv, dtype="f32", causal=causal, seed=Tq + 3)
    inp = workloads.generate(w)
    pu.full_parity(variant, inp, causal=causal, scale=w.scale, where=f"f32 {variant} {shape}")


# ---------------------------------------------------------------- the small workloads

@pytest.mark.parametrize("variant", VARIANTS)
def test_cfg1_fp32(variant):
    w = workloads.WORKLOADS["cfg1_f32"]
    pu.full_parity(variant, workloads.generate(w), causal=w.causal, scale=w.scale,
                   where=f"cfg1 {variant}")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("name", ["cfg2_s1", "cfg2_s4", "cfg2_s16"])
def test_cfg2_char_gpt(variant, name):
    w = workloads.WORKLOADS[name]
    pu.full_parity(variant, workloads.generate(w), causal=w.causal, scale=w.scale,
                   two_step=True, where=f"{name} {variant}")


# ---------------------------------------------------------------- full-size workloads

def _rows(T, seed):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 127, 128, 129, 255, 256, T // 2, T - 2, T - 1]
    return sorted(set([r for r in fixed if 0 <= r < T] + rng.integers(0, T, 12).tolist()))


@pytest.fixture(scope="module")
def cfg3_inputs():
    return workloads.generate(workloads.WORKLOADS["cfg3"])


@pytest.mark.parametrize("variant", VARIANTS)
def test_cfg3_full_size_sampled(variant, cfg3_inputs):
    w = workloads.WORKLOADS["cfg3"]
    pairs = [(0, 0), (15, 15), (7, 3)]
    pu.sampled_parity(variant, cfg3_inputs, causal=True, scale=w.scale, pairs=pairs,
                      rows_per_pair=lambda b, hh: _rows(w.Tq, b * 31 + hh), two_step=True,
                      where=f"cfg3 {variant}")


@pytest.mark.parametrize("variant", VARIANTS)
def test_cfg4_gqa_full_size_sampled(variant):
    w = workloads.WORKLOADS["cfg4_gqa"]
    inp = workloads.generate(w)
    pairs = [(0, 0), (0, 1), (3, 14), (2, 7)]  # heads 0 and 1 share kv head 0
    pu.sampled_parity(variant, inp, causal=True, scale=w.scale, pairs=pairs,
                      rows_per_pair=lambda b, hh: _rows(w.Tq, b * 17 + hh), two_step=True,
                      where=f"cfg4 {variant}")


@pytest.mark.parametrize("variant", VARIANTS)
def test_cfg5_cross_full_size_sampled(variant):
    w = workloads.WORKLOADS["cfg5_cross"]
    inp = workloads.generate(w)
    pairs = [(0, 0), (0, 31)]
    pu.sampled_parity(variant, inp, causal=False, scale=w.scale, pairs=pairs,
                      rows_per_pair=lambda b, hh: _rows(w.Tq, hh)[:10], two_step=True,
                      where=f"cfg5 {variant}")


# ---------------------------------------------------------------- properties and API paths

def test_deterministic_and_telemetry_optional():
    w = _wl("det", 2, 4, 2, 333, 333, 128, 128, causal=True, seed=5)
    inp = workloads.generate(w, device="cuda")
    kw = dict(b=inp["yat_b"], eps=inp["yat_eps"], causal=True)
    a = attention.forward("yat", inp["q"], inp["k"], inp["v"], **kw)
    b = attention.forward("yat", inp["q"], inp["k"], inp["v"], **kw)
    c = attention.forward("yat", inp["q"], inp["k"], inp["v"], telemetry=False, **kw)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    assert c[1] is None and c[2] is None and torch.equal(a[0], c[0])


def test_host_tensors_round_trip():
    w = _wl("host", 1, 2, 2, 256, 256, 64, 64, causal=True, seed=9)
    inp = workloads.generate(w)
    pinned = {n: inp[n].pin_memory() for n in ("q", "k", "v")}
    host = attention.forward("softmax", pinned["q"], pinned["k"], pinned["v"], causal=True)
    dev = attention.forward("softmax", inp["q"].cuda(), inp["k"].cuda(), inp["v"].cuda(),
                            causal=True)
    torch.cuda.synchronize()
    assert host[0].device.type == "cpu"
    assert torch.equal(host[0], dev[0].cpu()) and torch.equal(host[1], dev[1].cpu())


@pytest.mark.parametrize("variant,causal,hkv,dtype", [("yat", True, 4, "bf16"),
                                                       ("stau", False, 2, "bf16"),
                                                       ("softmax", False, 4, "bf16"),
                                                       ("yat", True, 2, "f32")])
def test_host_tensors_pipelined_chunks(variant, causal, hkv, dtype):
    """The host-buffer forward (cattn_forward_host) runs one forward per batch
    chunk, with the copies on their own streams; each chunk must equal the
    same call made on device tensors, bit for bit, outputs and telemetry
    alike."""
    w = _wl("host_chunks", 6, 4, hkv, 200, 200 if causal else 330, 64, 64, dtype=dtype,
            causal=causal, qk=2.0, seed=11)
    inp = workloads.generate(w)
    kw = {"yat": dict(b=inp["yat_b"], eps=inp["yat_eps"]), "softmax": {},
          "stau": dict(eps=inp["stau_eps"], tau=inp["tau"])}[variant]
    pinned = {n: inp[n].pin_memory() for n in ("q", "k", "v")}
    host = attention.forward(variant, pinned["q"], pinned["k"], pinned["v"], causal=causal,
                             scale=w.scale, **kw)
    assert all(t.device.type == "cpu" for t in host)
    n = min(w.B, attention.HOST_CHUNKS)
    edges = [w.B * i // n for i in range(n + 1)]
    for a, z in zip(edges[:-1], edges[1:]):
        dev = attention.forward(variant, *(inp[x][a:z].contiguous().cuda() for x in ("q", "k", "v")),
                                causal=causal, scale=w.scale, **kw)
        torch.cuda.synchronize()
        for got, want in zip(host, dev):
            assert torch.equal(got[a:z], want.cpu())
    # the caller's own (pageable) host outputs get the same values
    mine = (torch.empty_like(host[0]), torch.empty_like(host[1]), torch.empty_like(host[2]))
    attention.forward(variant, pinned["q"], pinned["k"], pinned["v"], causal=causal,
                      scale=w.scale, out=mine[0], row_mass=mine[1], row_max=mine[2], **kw)
    assert all(torch.equal(a, b) for a, b in zip(mine, host))
    # one chunk gives the same answer within the tolerance (Yat's fast-path
    # bound and the key split depend on the whole call)
    one = attention._forward_from_host(attention.variant_id(variant), pinned["q"], pinned["k"],
                                       pinned["v"], b=kw.get("b"), eps=kw.get("eps"),
                                       tau=kw.get("tau"), causal=causal, scale=w.scale,
                                       telemetry=True, yat_m=1, chunks=1)
    vmax = float(inp["v"].abs().max())
    assert float((one[0].float() - host[0].float()).abs().max()) <= 2e-2 * vmax


def test_host_entry_on_one_stream_and_empty():
    """cattn_forward_host with one stream for all three roles (nothing
    overlaps) gives the same bits; an empty batch is a no-op."""
    import ctypes
    from softmax_free_attention_gb300 import native
    # causal: never split over keys, so the chunking cannot change a bit
    w = _wl("host_one_stream", 5, 2, 2, 130, 130, 128, 64, causal=True, seed=12)
    inp = workloads.generate(w)
    q, k, v = (inp[n].contiguous() for n in ("q", "k", "v"))
    ref = attention.forward("softmax", q, k, v, causal=True, scale=w.scale)
    prob = attention.make_problem(q, k, v, causal=True, scale=w.scale)
    lib = native.load()
    need = int(lib.cattn_forward_host_workspace_bytes(native.SOFTMAX, ctypes.byref(prob), 3))
    dev = [torch.empty(t.shape, dtype=t.dtype, device="cuda") for t in (q, k, v, ref[0])]
    tel = [torch.empty(ref[1].shape, device="cuda") for _ in range(2)]
    out = [torch.empty_like(ref[0]), torch.empty_like(ref[1]), torch.empty_like(ref[2])]
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = lib.cattn_forward_host(native.SOFTMAX, ctypes.byref(prob), p(q), p(k), p(v), None, None,
                                None, p(out[0]), p(out[1]), p(out[2]), *(p(t) for t in dev),
                                p(tel[0]), p(tel[1]), p(ws), need, 3, s, s, s)
    assert st == native.OK
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(out, ref))
    e = attention.forward("softmax", q[:0], k[:0], v[:0], causal=True)
    assert e[0].shape == (0, 2, 130, 64)


def test_empty_problems():
    q = torch.zeros(0, 2, 16, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(0, 2, 16, 64, dtype=torch.bfloat16, device="cuda")
    out, m, x = attention.forward("softmax", q, k, k, causal=True)
    assert out.shape == (0, 2, 16, 64)
    q = torch.zeros(1, 2, 0, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 2, 5, 64, dtype=torch.bfloat16, device="cuda")
    out, m, x = attention.forward("yat", q, k, k, b=1.0, eps=1.0)
    torch.cuda.synchronize()
    assert out.shape == (1, 2, 0, 64)


def test_constant_values_give_constant_output():
    # weights sum to one (Yat: mass / (mass + 1e-9)) so a constant v comes back
    w = _wl("const", 1, 2, 2, 300, 300, 128, 128, causal=True, seed=4)
    inp = workloads.generate(w, device="cuda")
    v = torch.full_like(inp["v"], 0.75)
    for variant in VARIANTS:
        kw = pu.params_for(variant, inp)
        out, _, _ = attention.forward(variant, inp["q"], inp["k"], v, causal=True, **kw)
        torch.cuda.synchronize()
        assert (out.float() - 0.75).abs().max().item() <= 2e-2 * 0.75, variant


# ---------------------------------------------------------------- both Yat map paths

def test_yat_workspace_contents_do_not_matter():
    """The forward needs no zeroed workspace: the key-norm kernel zeroes the
    control words it reads and keeps the largest key norm in a word tagged
    with the call's generation, replacing a word of any other generation.  A
    workspace full of 0xFF bytes, or one whose maximum word carries a
    generation no call has drawn yet, must give the same bits as a zeroed
    one (with eps large enough that the map takes its fast path, which a
    stale maximum would switch off).  2100 keys: more than the one-launch
    path takes, so the key-norm kernel and its maximum word are used."""
    w = _wl("ws", 1, 2, 2, 2100, 2100, 128, 128, causal=True, qk=1.0, seed=21)
    inp = workloads.generate(w, device="cuda")
    b = torch.full((2,), 0.5, device="cuda")
    eps = torch.full((2,), 0.5, device="cuda")
    prob = attention.make_problem(inp["q"], inp["k"], inp["v"], causal=True, scale=w.scale)
    need = attention.workspace_bytes("yat", prob)
    zero = torch.zeros(need, dtype=torch.uint8, device="cuda")
    full = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
    future = torch.zeros(need, dtype=torch.uint8, device="cuda")
    # bytes 8-15: the largest key norm (0.0) under generation 0xFFFFFFF0
    future[8:16] = torch.tensor([0, 0, 0, 0, 0xF0, 0xFF, 0xFF, 0xFF], dtype=torch.uint8)
    outs = [attention.forward("yat", inp["q"], inp["k"], inp["v"], b=b, eps=eps, causal=True,
                              workspace=ws) for ws in (zero, full, future, zero)]
    torch.cuda.synchronize()
    assert attention.check_status() == 0
    for o in outs[1:]:
        for x, y in zip(outs[0], o):
            assert torch.equal(x, y)


@pytest.mark.parametrize("eps,qk,where", [
    (0.5, 1.0, "fast path: eps well above the rounding of |q|^2 + |k|^2"),
    (1e-3, 4.0, "exact path: eps below (|q|^2 + max |k|^2) 2^-16"),
    (1e-20, 1.0, "exact path: eps below 2^-60"),
])
def test_yat_fast_and_exact_map_paths(eps, qk, where):
    """The Yat map has a fast path (one reciprocal per key pair, no clamp)
    taken only when the norms bound its rounding, and the plain path
    otherwise; both must match the oracle."""
    w = _wl("paths", 1, 2, 2, 300, 300, 128, 128, causal=True, qk=qk, seed=77)
    inp = workloads.generate(w)
    inp["yat_b"] = np.full(2, 0.5, dtype=np.float32)
    inp["yat_eps"] = np.full(2, eps, dtype=np.float32)
    pu.full_parity("yat", inp, causal=True, scale=w.scale, where=where)


@pytest.mark.parametrize("b,qk,where", [
    (1.0, 0.01, "b far above |q|^2 + eps: every row recomputed by the plain definition"),
    (1.0, 0.06, "b a few times |q|^2: the scores carry b, no row flagged"),
    (-3.0, 0.3, "negative b"),
    (40.0, 1.0, "b a third of |q|^2"),
])
def test_yat_bias_against_the_norms(b, qk, where):
    """b from far above |q|^2 + eps to a third of |q|^2, and negative, with a
    small eps: the numerator (q.k + b)^2 and the assembled distance must
    match the oracle whichever term dominates."""
    w = _wl("bias", 1, 2, 2, 300, 300, 128, 128, causal=True, qk=qk, seed=31)
    inp = workloads.generate(w)
    inp["yat_b"] = np.full(2, b, dtype=np.float32)
    inp["yat_eps"] = np.full(2, 1e-3, dtype=np.float32)
    pu.full_parity("yat", inp, causal=True, scale=w.scale, where=where)


def test_yat_zero_query_rows():
    """Query rows of zeros have kappa = b^2 / (|k|^2 + eps) exactly, eps far
    below b (both Yat paths: the one-launch form at 256 keys, the key-norm
    kernel path at 1100)."""
    for T in (256, 1100):
        w = _wl("zrows", 1, 2, 2, T, T, 128, 128, causal=True, seed=32)
        inp = workloads.generate(w)
        inp["q"][:, :, ::5, :] = 0
        inp["yat_b"] = np.full(2, 0.75, dtype=np.float32)
        inp["yat_eps"] = np.full(2, 1e-4, dtype=np.float32)
        pu.full_parity("yat", inp, causal=True, scale=w.scale, where=f"zero rows T={T}")


# ---------------------------------------------------------------- Yat with q close to k

# (name, d, q/k factor, eps): the char-level norms x16 at d = 64 and the
# cross-attention norms x8 at d = 128; eps = 1 takes the map's fast path at
# these norms, eps = 0.05 its clamped path
NEAR_CASES = [
    ("s16_d64_fast", 64, 16.0, 1.0),
    ("s16_d64_exact", 64, 16.0, 0.05),
    ("x8_d128_fast", 128, 8.0, 1.0),
    ("x8_d128_exact", 128, 8.0, 0.05),
]


def _closed_form_self(q, b, eps):
    """kappa(q, q) = (|q|^2 + b)^2 / eps per row ("The Kernel Between the
    Roles", section "Two of our beliefs, measured"), in fp64 from the stored
    bf16 values: [B, h, T]."""
    qq = q.to(torch.float64)
    n = (qq * qq).sum(-1)
    return ((n + torch.as_tensor(b, dtype=torch.float64)[None, :, None]) ** 2
            / torch.as_tensor(eps, dtype=torch.float64)[None, :, None]).numpy()


@pytest.mark.parametrize("case", NEAR_CASES, ids=lambda c: c[0])
def test_yat_keys_equal_to_queries(case):
    """k = q (tied, causal): every row's own key sits at distance zero, where
    |q|^2 + |k|^2 - 2 q.k cancels completely.  out, the row mass and max
    kappa must match the oracle, and max kappa must equal the closed form
    (|q|^2 + b)^2 / eps of the diagonal."""
    name, d, s, eps = case
    w = _wl("tied", 2, 2, 2, 300, 300, d, d, causal=True, qk=s, seed=31)
    inp = workloads.generate(w)
    inp["k"] = inp["q"].clone()
    inp["yat_b"] = np.array([0.3, 2.0], dtype=np.float32)
    inp["yat_eps"] = np.full(2, eps, dtype=np.float32)
    # the key-norm kernel with the separate near-key pass, and the one call
    # whose units all run in one wave (its rows recomputed inside the kernel)
    pu.full_parity("yat", inp, causal=True, scale=w.scale, two_step=True, where=f"tied {name}")
    pu.full_parity("yat", inp, causal=True, scale=w.scale, where=f"tied {name} one launch")
    _, _, mx = pu.run_gpu("yat", inp, causal=True, scale=w.scale)
    ref = _closed_form_self(inp["q"], inp["yat_b"], inp["yat_eps"])
    rel = np.abs(pu.to_np(mx) - ref) / ref
    assert rel.max() <= pu.TEL_TOL, f"tied {name}: max kappa vs closed form {rel.max():.3e}"


@pytest.mark.parametrize("case", NEAR_CASES, ids=lambda c: c[0])
def test_yat_some_keys_copied_from_queries(case):
    """Random keys with a few rows replaced by query rows (exact copies and
    copies with one element nudged by one bf16 step), non-causal with a
    ragged key tail, and causal: the near-coincident keys must not lose the
    row mass or max kappa to the cancellation of the assembled distance."""
    name, d, s, eps = case
    for causal, Tk in ((False, 700), (True, 300)):
        w = _wl("copied", 1, 2, 2, 300, Tk, d, d, causal=causal, qk=s, seed=57)
        inp = workloads.generate(w)
        k = inp["k"].clone()
        q = inp["q"]
        pairs = [(5, 3), (100, 140), (299, 299), (128, 130)] if causal else \
                [(5, 3), (100, 400), (299, 699), (128, 130), (17, 255)]
        for n_pair, (t, j) in enumerate(pairs):
            k[0, :, j] = q[0, :, t]
            if n_pair % 2:
                # one element moved by a bf16 step or two: a tiny, nonzero distance
                k[0, :, j, 7] = (k[0, :, j, 7].float() * (1.0 + 2.0 ** -7)).to(torch.bfloat16)
        inp["k"] = k
        inp["yat_b"] = np.array([0.3, 2.0], dtype=np.float32)
        inp["yat_eps"] = np.full(2, eps, dtype=np.float32)
        pu.full_parity("yat", inp, causal=causal, scale=w.scale, two_step=True,
                       where=f"copied {name} causal={causal}")
        pu.full_parity("yat", inp, causal=causal, scale=w.scale,
                       where=f"copied {name} causal={causal} one call")


# ---------------------------------------------------------------- tau*

TAU_SHAPES = [  # B, h, hkv, T_q, T_k, d, causal
    (2, 4, 2, 300, 300, 128, True),    # several query tiles, ragged tail, GQA
    (1, 2, 1, 130, 130, 64, True),     # one pair, dk 64
    (1, 2, 2, 200, 2100, 64, False),   # non-causal with key splits
    (3, 1, 1, 129, 129, 128, False),   # a query tile of one row
]


@pytest.mark.parametrize("shape", TAU_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_tau_star_matches_oracle(shape):
    """tau* per head against the fp64 oracle on the same bf16 inputs.

    Tolerance 2e-3 relative: the kernel's scores are fp32 sums of exact bf16
    products (relative error ~1e-7), ln phi goes through the SFU's log2 and
    exp2 (~1e-6), and each thread's sums over a unit (at most a few thousand
    scores) are fp32 before they are added in fp64 (relative error below
    ~3e-4 for these sizes); the ratio of two such centred sums stays within
    a few 1e-4 unless the variance nearly cancels, which these inputs avoid.
    """
    import oracle
    B, h, hkv, Tq, Tk, d, causal = shape
    g = torch.Generator().manual_seed(11)
    q = (torch.randn(B, h, Tq, d, generator=g) * 1.5).to(torch.bfloat16)
    k = torch.randn(B, hkv, Tk, d, generator=g).to(torch.bfloat16)
    eps = torch.tensor([1e-6, 0.5, 1e-3, 2.0][:h], dtype=torch.float32)
    scale = 1.0 / math.sqrt(d)
    tau, mom = attention.tau_star(q.cuda(), k.cuda(), eps.cuda(), causal=causal, scale=scale,
                                  return_moments=True)
    torch.cuda.synchronize()
    assert attention.check_status() == 0
    want, n = oracle.tau_star(q, k, eps, causal=causal, scale=scale)
    got = tau.cpu().double().numpy()
    mom = mom.cpu().numpy()
    np.testing.assert_array_equal(mom[:, 0], n)  # every allowed pair counted once
    np.testing.assert_allclose(mom[:, 5], np.log(np.log(2.0) + eps.double().numpy()), rtol=1e-6)
    np.testing.assert_allclose(got, want, rtol=2e-3)


def test_tau_star_cfg4_gqa():
    """The GQA s^tau workload (B=4, 16 query heads on 8 KV heads, T=8192):
    tau* of every head on the GPU; the oracle checks the same data cut to its
    first 2048 rows and keys, one batch, heads 0 and 1 (sharing KV head 0),
    since tau* pools each head's whole score set."""
    import oracle
    w = workloads.WORKLOADS["cfg4_gqa"]
    inp = workloads.generate(w, device="cuda")
    eps = torch.from_numpy(inp["stau_eps"])
    tau = attention.tau_star(inp["q"], inp["k"], eps, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert attention.check_status() == 0
    assert torch.isfinite(tau).all()
    q1 = inp["q"][:1, :2, :2048].contiguous()
    k1 = inp["k"][:1, :1, :2048].contiguous()
    got = attention.tau_star(q1, k1, eps[:2], causal=True, scale=w.scale).cpu().double().numpy()
    want, _ = oracle.tau_star(q1.cpu(), k1.cpu(), eps[:2], causal=True, scale=w.scale)
    np.testing.assert_allclose(got, want, rtol=2e-3)


# ---------------------------------------------------------------- Yat numerator power

YAT_M_SHAPES = [  # B, h, hkv, Tq, Tk, dk, dv, causal, dtype
    (2, 4, 2, 300, 300, 128, 128, True, "bf16"),
    (1, 2, 1, 130, 130, 64, 64, True, "bf16"),
    (1, 2, 2, 200, 2100, 128, 64, False, "bf16"),   # key splits
    (1, 2, 1, 77, 77, 64, 64, True, "f32"),
]


@pytest.mark.parametrize("m", [2, 3])
@pytest.mark.parametrize("shape", YAT_M_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_yat_numerator_power(m, shape):
    """kappa = (q.k + b)^{2m} / (max(|q-k|^2, 0) + eps) against the oracle, with
    the same tolerances as the m = 1 map (the power only sharpens the rows)."""
    B, h, hkv, Tq, Tk, dk, dv, causal, dtype = shape
    w = _wl("yat_m", B, h, hkv, Tq, Tk, dk, dv, dtype=dtype, causal=causal, seed=Tq + 31 * m)
    inp = workloads.generate(w)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    res = attention.forward("yat", q, k, v, b=inp["yat_b"], eps=inp["yat_eps"], causal=causal,
                            yat_m=m)
    torch.cuda.synchronize()
    assert attention.check_status() == 0
    ora = oracle_forward_m(inp, causal, m)
    pu.compare("yat", tuple(pu.to_np(t) for t in res), ora, float(inp["v"].abs().max()),
               inp["q"].dtype, where=f"yat m={m} {shape}")


def oracle_forward_m(inp, causal, m):
    import oracle
    return oracle.forward("yat", inp["q"], inp["k"], inp["v"], b=inp["yat_b"], eps=inp["yat_eps"],
                          causal=causal, yat_m=m)


# ---------------------------------------------------------------- row statistics

STATS_SHAPES = [  # B, h, hkv, T_q, T_k, d, causal
    (2, 4, 2, 300, 300, 128, True),
    (1, 2, 1, 130, 130, 64, True),
    (1, 2, 2, 200, 1100, 128, False),
]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", STATS_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_row_stats_match_oracle(variant, shape):
    """Per-row entropy, fraction below 1e-6 and top-10 mass against the oracle.

    Tolerances: entropy 2e-3 absolute and top-10 mass 2e-3 relative (the
    weights come from fp32 scores of bf16 inputs and an fp32 normaliser);
    the fraction below 1e-6 may differ by keys whose weight sits within
    rounding of the threshold: at most two keys per row."""
    import oracle
    B, h, hkv, Tq, Tk, d, causal = shape
    w = _wl("stats", B, h, hkv, Tq, Tk, d, d, causal=causal, qk=2.0, seed=Tq + 5)
    inp = workloads.generate(w)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    kw = pu.params_for(variant, inp)
    _, mass, _ = attention.forward(variant, q, k, v, causal=causal, scale=w.scale, **kw)
    ent, small, top = attention.row_stats(variant, q, k, mass, causal=causal, scale=w.scale, **kw)
    torch.cuda.synchronize()
    assert attention.check_status() == 0
    e_o, s_o, t_o = oracle.row_stats(variant, inp["q"], inp["k"], inp["v"], causal=causal,
                                     scale=w.scale, **kw)
    n = np.minimum(np.arange(Tq) + 1, Tk) if causal else np.full(Tq, Tk)
    np.testing.assert_allclose(pu.to_np(ent), e_o, atol=2e-3)
    np.testing.assert_allclose(pu.to_np(top), t_o, rtol=2e-3, atol=1e-6)
    assert (np.abs(pu.to_np(small) - s_o) * n <= 2.0 + 1e-9).all()


ENT_SHAPES = [  # B, h, hkv, T_q, T_k, d, causal
    (2, 4, 2, 300, 300, 128, True),
    (1, 2, 1, 130, 130, 64, True),
    (1, 2, 2, 200, 2100, 128, False),   # two key splits: the entropy sums merge in the combine
    (1, 2, 2, 1100, 1100, 64, True),    # causal, long ragged rows
]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", ENT_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_forward_entropy_matches_oracle(variant, shape):
    """The forward's online entropy (sum f log2 f kept beside the normaliser,
    moved onto each new running max) against the oracle's per-row normalised
    entropy, at the row statistics pass's 2e-3 absolute; out and telemetry of
    the same call against the oracle as usual."""
    import oracle
    B, h, hkv, Tq, Tk, d, causal = shape
    w = _wl("ent", B, h, hkv, Tq, Tk, d, d, causal=causal, qk=2.0, seed=Tq + 9)
    inp = workloads.generate(w)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    kw = pu.params_for(variant, inp)
    out, mass, mx, ent = attention.forward_entropy(variant, q, k, v, causal=causal, scale=w.scale,
                                                   **kw)
    torch.cuda.synchronize()
    assert attention.check_status() == 0
    e_o, _, _ = oracle.row_stats(variant, inp["q"], inp["k"], inp["v"], causal=causal,
                                 scale=w.scale, **kw)
    np.testing.assert_allclose(pu.to_np(ent), e_o, atol=2e-3)
    ora = pu.run_oracle(variant, inp, causal=causal, scale=w.scale)
    pu.compare(variant, (pu.to_np(out), pu.to_np(mass), pu.to_np(mx)), ora,
               float(inp["v"].abs().max()), q.dtype, where=f"entropy forward {variant} {shape}")


def test_forward_entropy_on_near_keys():
    """Rows recomputed by the Yat near-key pass carry their entropy too."""
    import oracle
    w = _wl("ent_tied", 1, 2, 2, 300, 300, 64, 64, causal=True, qk=16.0, seed=31)
    inp = workloads.generate(w)
    inp["k"] = inp["q"].clone()
    inp["yat_b"] = np.array([0.3, 2.0], dtype=np.float32)
    inp["yat_eps"] = np.full(2, 0.05, dtype=np.float32)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    kw = pu.params_for("yat", inp)
    _, _, _, ent = attention.forward_entropy("yat", q, k, v, causal=True, **kw)
    torch.cuda.synchronize()
    e_o, _, _ = oracle.row_stats("yat", inp["q"], inp["k"], inp["v"], causal=True, **kw)
    np.testing.assert_allclose(pu.to_np(ent), e_o, atol=2e-3)


# ---------------------------------------------------------------- every width pair

WIDTH_SHAPES = [  # dtype, B, h, hkv, Tq, Tk, dk, dv, causal: widths without tensor-core tiles
    ("bf16", 1, 2, 1, 100, 100, 32, 32, True),
    ("bf16", 1, 2, 2, 70, 140, 64, 128, False),
    ("bf16", 2, 2, 1, 65, 65, 32, 64, True),
    ("bf16", 1, 2, 2, 90, 90, 128, 32, True),
    ("f32", 1, 2, 2, 80, 80, 64, 32, True),
    ("f32", 1, 2, 1, 50, 120, 32, 128, False),
]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", WIDTH_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_cuda_core_widths(variant, shape):
    """(dk, dv) pairs the tensor-core kernel has no tiles for run on the
    CUDA-core kernel (bf16 widened to fp32), each against the oracle."""
    dtype, B, h, hkv, Tq, Tk, dk, dv, causal = shape
    w = _wl("widths", B, h, hkv, Tq, Tk, dk, dv, dtype=dtype, causal=causal, seed=Tq + dk + dv)
    inp = workloads.generate(w)
    pu.full_parity(variant, inp, causal=causal, scale=w.scale, where=f"{variant} {shape}")
