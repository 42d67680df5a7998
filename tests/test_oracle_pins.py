"""Pins for the fp64 oracle: checks against what the pages and mathematics fix.

Nothing here compares the oracle with itself. The anchors are:
  * a hand-worked example (tests/golden/worked_example_tiny_ffn.txt);
  * exhaustive widening of every 16-bit pattern against numpy/torch converters,
    and hand-derived int4 nibbles / half-precision values (tests/golden/);
  * NumPy dense-matrix brute force on tiny shapes (tests/brute.py);
  * closed forms and invariants of the definitions: true ReLU mask == dense FFN,
    all-ones mask == dense, empty mask == 0, degree-2 / degree-1 homogeneity,
    sigmoid(z) > 0.5 <=> z > 0, neuron-permutation invariance, union over the
    batch, Python's stable sort for the profiler order, RMS of a constant vector.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests import brute
from tests.conftest import read_fixture, read_table
from workload.gen import quantize_int4_g128

KINDS = ["gated", "relu"]


def _store(w: np.ndarray, dtype: str):
    """Round a float64 matrix to its stored representation (raw bits) -> (stored, scales)."""
    if dtype == "f32":
        return w.astype(np.float32), None
    if dtype == "f16":
        return w.astype(np.float16).view(np.uint16), None
    if dtype == "bf16":
        t = torch.from_numpy(w.astype(np.float32)).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16).copy(), None
    if dtype == "int4g128":
        p, s = quantize_int4_g128(torch.from_numpy(w.astype(np.float32)))
        return p.numpy().copy(), s.view(torch.int16).numpy().view(np.uint16).copy()
    raise ValueError(dtype)


def rand_layer(rng, d, f, r, kind, wdtype, pdtype, bias_scale=0.5):
    L = {}
    for name in (["w_gate", "w_up", "w_down_t"] if kind == "gated" else ["w_gate", "w_down_t"]):
        st, sc = _store(rng.standard_normal((f, d)) / math.sqrt(d), wdtype)
        L[name] = st
        L["s_" + name.split("_")[1] if name != "w_down_t" else "s_down"] = sc
    L["b_gate"] = (rng.standard_normal(f) * bias_scale).astype(np.float32)
    L["p1_t"], _ = _store(rng.standard_normal((r, d)) / math.sqrt(d), pdtype)
    L["p2_t"], _ = _store(rng.standard_normal((f, r)) / math.sqrt(r), pdtype)
    L["b_pred"] = (rng.standard_normal(f) * bias_scale - 0.3).astype(np.float32)
    return L


def rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


# ------------------------------------------------------------------ widening -------------------

def test_widen_f16_exhaustive():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.widen(bits, "f16")
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_widen_bf16_exhaustive():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.widen(bits, "bf16")
    want = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_widen_hand_values():
    for typ, hexbits, val in read_table("half_values.txt"):
        got = oracle.widen(np.array([int(hexbits, 16)], np.uint16), typ)[0]
        assert got == float(val), (typ, hexbits, got, val)
        assert math.copysign(1, got) == math.copysign(1, float(val))


def test_int4_nibbles_hand_values():
    rows = read_table("int4_nibbles.txt")
    for hx, lo, hi in rows:
        packed = np.zeros((1, 64), np.uint8)
        packed[0, 0] = int(hx, 16)
        one = np.array([[0x3C00]], np.uint16)  # fp16 1.0
        w = oracle.widen(packed, "int4g128", one)
        assert w[0] == int(lo) and w[1] == int(hi), (hx, w[:2])


def test_int4_group_scales():
    # 256 elements = two groups of 128 with scales 0.5 and 3.0 (fp16 0x3800, 0x4200)
    packed = np.full((1, 128), 0x97, np.uint8)  # low 7, high -7
    scales = np.array([[0x3800, 0x4200]], np.uint16)
    w = oracle.widen(packed, "int4g128", scales)
    assert np.all(w[0:128:2] == 3.5) and np.all(w[1:128:2] == -3.5)
    assert np.all(w[128::2] == 21.0) and np.all(w[129::2] == -21.0)


def test_int4_quantisation_bound():
    # the stored reading w ~ q*s must satisfy |w - q*s| <= s/2 inside the clamp range
    rng = np.random.default_rng(3)
    w = rng.standard_normal((6, 256)) * 0.05
    p, s = _store(w, "int4g128")
    deq = oracle.widen(p, "int4g128", s).reshape(1, -1) if p.shape[0] == 1 else np.stack(
        [oracle.widen(p[i:i + 1], "int4g128", s[i:i + 1]) for i in range(p.shape[0])])
    sc = np.repeat(s.view(np.float16).astype(np.float64), 128, axis=1)
    wf = w.astype(np.float32).astype(np.float64)
    assert np.all(np.abs(wf - deq) <= sc / 2 + 1e-12 + np.abs(wf) * 2e-3)  # fp16 scale rounding slack


# ------------------------------------------------------------------ worked example -------------

def _fixture_layer():
    fx = read_fixture("worked_example_tiny_ffn.txt")
    A = lambda k: np.array(fx[k], np.float64)
    L = {k: A(k).astype(np.float32) for k in ["p1_t", "p2_t", "w_gate", "w_up", "w_down_t"]}
    L["b_pred"] = A("b_pred")[0].astype(np.float32)
    L["b_gate"] = A("b_gate")[0].astype(np.float32)
    return fx, A("u"), L


def test_worked_example_predictor():
    fx, U, L = _fixture_layer()
    pr = oracle.predict(U, L["p1_t"], L["p2_t"], L["b_pred"], "f32")
    assert np.array_equal(pr["hp"], np.array(fx["hp"]))
    assert np.array_equal(pr["z"], np.array(fx["z"]))
    assert pr["idx"].tolist() == [int(v) for v in fx["idx_union"][0]]
    for b, key in enumerate(["idx_row0", "idx_row1"]):
        prb = oracle.predict(U[b], L["p1_t"], L["p2_t"], L["b_pred"], "f32")
        assert prb["idx"].tolist() == [int(v) for v in fx[key][0]]


def test_worked_example_ffn():
    fx, U, L = _fixture_layer()
    h, y = oracle.sparse_ffn(U, L, [0, 1, 2], "gated", "f32")
    assert np.array_equal(h, np.array(fx["h_gated_union"]))
    assert np.array_equal(y, np.array(fx["y_gated_union"]))
    _, y0 = oracle.sparse_ffn(U[0], L, [0, 2], "gated", "f32")
    assert np.array_equal(y0[0], np.array(fx["y_gated_row0"][0]))
    yd = oracle.dense_ffn(U[0], L, "gated", "f32")
    assert np.array_equal(yd[0], np.array(fx["y_gated_dense_row0"][0]))
    Lr = {k: v for k, v in L.items() if k != "w_up"}
    _, yr = oracle.sparse_ffn(U[0], Lr, [0, 2], "relu", "f32")
    assert np.array_equal(yr[0], np.array(fx["y_relu_row0"][0]))


# ------------------------------------------------------------------ brute force ----------------

CASES = [
    # d, f, r, B, kind, wdtype, pdtype
    (24, 40, 8, 1, "gated", "f32", "f32"),
    (16, 70, 6, 3, "gated", "bf16", "bf16"),
    (40, 33, 12, 2, "relu", "f16", "f16"),
    (32, 64, 16, 4, "relu", "bf16", "f32"),
    (128, 50, 8, 2, "relu", "int4g128", "f16"),
    (256, 37, 16, 1, "gated", "int4g128", "f16"),
]


@pytest.mark.parametrize("d,f,r,B,kind,wdt,pdt", CASES)
def test_brute_force_tiny(d, f, r, B, kind, wdt, pdt):
    rng = np.random.default_rng(d * 7 + f)
    L = rand_layer(rng, d, f, r, kind, wdt, pdt)
    U = rng.standard_normal((B, d))
    HP, Z, M = brute.predictor(U, L["p1_t"], L["p2_t"], L["b_pred"], pdt)
    pr = oracle.predict(U, L["p1_t"], L["p2_t"], L["b_pred"], pdt)
    assert rel(pr["hp"], HP) < 1e-13 and rel(pr["z"], Z) < 1e-13
    assert np.array_equal(pr["mask"], M)
    assert 0 < pr["count"] < f  # the case exercises both branches
    Y, _ = brute.ffn_masked(U, L, M, kind, wdt)
    _, y = oracle.sparse_ffn(U, L, pr["idx"], kind, wdt)
    assert rel(y, Y) < 1e-12
    yd = oracle.dense_ffn(U, L, kind, wdt)
    Yd, _ = brute.ffn_masked(U, L, np.ones(f, bool), kind, wdt)
    assert rel(yd, Yd) < 1e-12


@pytest.mark.parametrize("kind,wdt", [("gated", "bf16"), ("relu", "f16"), ("gated", "f32"), ("relu", "int4g128")])
def test_mask_special_cases(kind, wdt):
    """True ReLU set == dense; all neurons == dense; empty set == 0 (the FFN equation)."""
    rng = np.random.default_rng(11)
    d, f, B = 128, 90, 3
    L = rand_layer(rng, d, f, 8, kind, wdt, "f32")
    U = rng.standard_normal((B, d))
    dense = oracle.dense_ffn(U, L, kind, wdt)
    truth = np.nonzero(brute.true_set(U, L, wdt))[0]
    assert 0 < truth.size < f
    _, y_true = oracle.sparse_ffn(U, L, truth, kind, wdt)
    _, y_all = oracle.sparse_ffn(U, L, np.arange(f), kind, wdt)
    _, y_none = oracle.sparse_ffn(U, L, np.zeros(0, np.int32), kind, wdt)
    assert rel(y_true, dense) < 1e-13
    assert rel(y_all, dense) < 1e-13
    assert np.all(y_none == 0.0)
    # any superset of the true set also reproduces the dense output
    extra = rng.choice(np.setdiff1d(np.arange(f), truth), size=5, replace=False)
    _, y_sup = oracle.sparse_ffn(U, L, np.sort(np.concatenate([truth, extra])), kind, wdt)
    assert rel(y_sup, dense) < 1e-13
    # dropping one true neuron does not
    _, y_drop = oracle.sparse_ffn(U, L, truth[1:], kind, wdt)
    assert rel(y_drop, dense) > 1e-6


@pytest.mark.parametrize("kind,deg", [("gated", 2), ("relu", 1)])
def test_homogeneity(kind, deg):
    rng = np.random.default_rng(5)
    d, f = 64, 80
    L = rand_layer(rng, d, f, 8, kind, "f32", "f32")
    L["b_gate"] = np.zeros(f, np.float32)
    U = rng.standard_normal((2, d))
    s = 2.5
    _, y1 = oracle.sparse_ffn(U, L, np.arange(f), kind, "f32")
    _, y2 = oracle.sparse_ffn(U * s, L, np.arange(f), kind, "f32")
    assert rel(y2, (s ** deg) * y1) < 1e-13
    # with b_pred = 0 the mask does not depend on the scale of u; with a bias it does
    p_a = oracle.predict(U, L["p1_t"], L["p2_t"], None, "f32")
    p_b = oracle.predict(U * 7.0, L["p1_t"], L["p2_t"], None, "f32")
    assert np.array_equal(p_a["idx"], p_b["idx"])


def test_sigmoid_threshold_reading():
    """sigmoid(z) > 0.5 <=> z > 0, so 'a_i > tau' with tau = 0.5 is 'logit > 0'."""
    from scipy.special import expit

    rng = np.random.default_rng(0)
    z = rng.standard_normal(10000) * 5
    assert np.array_equal(expit(z) > 0.5, z > 0)
    # tiny logits: float64 sigmoid rounds to 0.5, so evaluate at 400 digits
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 400
    for v in list(rng.standard_normal(50) * 1e-12) + [1e-300, -1e-300, 0.0]:
        sig = 1 / (1 + mpmath.exp(-mpmath.mpf(v)))
        assert (sig > mpmath.mpf("0.5")) == (v > 0), v
    # and the oracle applies it strictly: z == 0 is inactive (the worked example has such a neuron too)
    p1 = np.zeros((1, 4), np.float32)
    p2 = np.ones((3, 1), np.float32)
    pr = oracle.predict(np.ones((1, 4)), p1, p2, np.array([0.0, 1e-30, -1e-30], np.float32), "f32")
    assert pr["idx"].tolist() == [1]


def test_permutation_invariance():
    rng = np.random.default_rng(9)
    d, f, r = 48, 120, 10
    L = rand_layer(rng, d, f, r, "gated", "bf16", "bf16")
    U = rng.standard_normal((2, d))
    perm = rng.permutation(f).astype(np.int32)
    Lp = {k: (v[perm] if k in ("w_gate", "w_up", "w_down_t", "p2_t", "b_gate", "b_pred") else v) for k, v in L.items()}
    a = oracle.layer_forward(U, L, "gated", "bf16", "bf16")
    b = oracle.layer_forward(U, Lp, "gated", "bf16", "bf16")
    assert np.array_equal(np.sort(perm[b["idx"]]), a["idx"])
    assert rel(b["y"], a["y"]) < 1e-13


def test_union_over_batch():
    rng = np.random.default_rng(4)
    d, f, r = 32, 200, 8
    L = rand_layer(rng, d, f, r, "gated", "f32", "f32")
    U = rng.standard_normal((4, d))
    joint = oracle.predict(U, L["p1_t"], L["p2_t"], L["b_pred"], "f32")
    singles = [set(oracle.predict(U[b], L["p1_t"], L["p2_t"], L["b_pred"], "f32")["idx"].tolist()) for b in range(4)]
    assert set(joint["idx"].tolist()) == set().union(*singles)
    assert joint["count"] > max(len(s) for s in singles)
    # a row evaluated on the union equals that row evaluated on (union | its own true set)
    for b in range(4):
        ts = set(np.nonzero(brute.true_set(U[b:b + 1], L, "f32"))[0].tolist())
        _, y_u = oracle.sparse_ffn(U[b], L, joint["idx"], "gated", "f32")
        _, y_ut = oracle.sparse_ffn(U[b], L, sorted(set(joint["idx"].tolist()) & ts), "gated", "f32")
        assert rel(y_u, y_ut) < 1e-13


def test_hot_first_order_is_pythons_stable_sort():
    """The profiler sorts neuron ids by count, descending, with Python's stable sorted()."""
    rng = np.random.default_rng(2)
    for f in (1, 7, 500, 4099):
        counts = rng.integers(0, 12, size=f)  # many ties
        want = sorted(range(f), key=lambda i: counts[i], reverse=True)
        assert oracle.hot_first_order(counts).tolist() == want
    assert oracle.hot_first_order(np.zeros(0, np.uint32)).tolist() == []
    big = np.array([2**32 - 1, 0, 2**31, 2**31 + 1], np.uint64)
    assert oracle.hot_first_order(big).tolist() == [0, 3, 2, 1]


def test_rms_norm_closed_form():
    for c in (3.0, -0.5, 1e-4):
        x = np.full((1, 10), c)
        u = oracle.rms_norm(x, 1e-6)
        assert np.allclose(u, c / math.sqrt(c * c + 1e-6), rtol=1e-15, atol=0)
    x = np.zeros((2, 8))
    assert np.all(oracle.rms_norm(x) == 0.0)


def test_stack_reduces_to_layers():
    rng = np.random.default_rng(8)
    d, f, r = 32, 64, 8
    Ls = [rand_layer(rng, d, f, r, "relu", "f16", "f16") for _ in range(3)]
    x0 = rng.standard_normal((2, d))
    st = oracle.stack(x0, Ls, "relu", "f16", "f16", keep=True)
    x = x0.copy()
    for i, L in enumerate(Ls):
        u = brute_rms(x)
        HP, Z, M = brute.predictor(u, L["p1_t"], L["p2_t"], L["b_pred"], "f16")
        Y, _ = brute.ffn_masked(u, L, M, "relu", "f16")
        assert np.array_equal(np.nonzero(M)[0], st["idx"][i])
        x = x + Y
    assert rel(st["x_out"] - x0, x - x0) < 1e-12
    # zero W_down: the stack is the identity on x
    Z0 = [dict(L, w_down_t=np.zeros_like(L["w_down_t"])) for L in Ls]
    st0 = oracle.stack(x0, Z0, "relu", "f16", "f16")
    assert np.array_equal(st0["x_out"], x0)


def brute_rms(x, eps=1e-6):
    return x / np.sqrt((x * x).mean(axis=1, keepdims=True) + eps)


@pytest.mark.parametrize("kind,wdt,pdt", [("gated", "bf16", "bf16"), ("relu", "f16", "f16")])
def test_hot_prefix_mode(kind, wdt, pdt):
    """Hot prefix H: neurons [0, H) always active, the predictor decides the rest.

    Pins: H = 0 is the plain predictor; H = f is the dense FFN (the FFN equation over
    every neuron); any H agrees with brute force (mask = any_b(Z > 0) | i < H); and the
    layer output is the dense one whenever the true set lies inside the hot prefix plus
    the predicted tail."""
    rng = np.random.default_rng(31)
    d, f, r, B = 64, 150, 12, 3
    L = rand_layer(rng, d, f, r, kind, wdt, pdt)
    U = rng.standard_normal((B, d))
    plain = oracle.predict(U, L["p1_t"], L["p2_t"], L["b_pred"], pdt)
    zero = oracle.predict(U, L["p1_t"], L["p2_t"], L["b_pred"], pdt, hot_prefix=0)
    assert np.array_equal(zero["idx"], plain["idx"])
    _, Z, M = brute.predictor(U, L["p1_t"], L["p2_t"], L["b_pred"], pdt)
    for H in (1, 37, 149):
        pr = oracle.predict(U, L["p1_t"], L["p2_t"], L["b_pred"], pdt, hot_prefix=H)
        want = M | (np.arange(f) < H)
        assert np.array_equal(pr["mask"], want)
        assert np.array_equal(pr["idx"], np.flatnonzero(want))
        assert np.all(np.isinf(pr["z"][:, :H])) and np.array_equal(pr["z"][:, H:], plain["z"][:, H:])
        out = oracle.layer_forward(U, L, kind, wdt, pdt, hot_prefix=H)
        Y, _ = brute.ffn_masked(U, L, want, kind, wdt)
        assert rel(out["y"], Y) < 1e-12
    full = oracle.layer_forward(U, L, kind, wdt, pdt, hot_prefix=f)
    assert full["count"] == f
    assert rel(full["y"], oracle.dense_ffn(U, L, kind, wdt)) < 1e-13
    # a hot prefix that covers every truly active neuron gives the dense output too
    ts = np.flatnonzero(brute.true_set(U, L, wdt))
    out = oracle.layer_forward(U, L, kind, wdt, pdt, hot_prefix=int(ts.max()) + 1)
    assert rel(out["y"], oracle.dense_ffn(U, L, kind, wdt)) < 1e-13
