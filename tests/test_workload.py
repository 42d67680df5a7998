"""The synthetic workloads reproduce the activation statistics the pages report.

Targets: mean active fraction per workload; a hot 10% active on >= 80% of
tokens (paper walk-through page, "neuron activation power law"); 26% of neurons
carrying 80% of activations (summary page, Key Results); Zipf exponents as named
per workload.
"""
import numpy as np
import pytest
import torch

import oracle
from tests import brute
from workload import WORKLOADS, activation_probs, make_inputs, make_layer, scaled
from workload.gen import T_CALIB, ranked_probs

W = list(WORKLOADS.values())


def test_recipes_hit_targets():
    c1, c2, c3, c4, c5 = W
    p1 = ranked_probs(c1)
    assert abs(p1.mean() - 0.10) < 0.002
    assert (p1 >= 0.999).sum() >= 40  # the head of a Zipf law saturates
    p2 = ranked_probs(c2)
    n_hot = int(round(0.1 * c2.f))
    assert abs(p2.mean() - 0.10) < 0.002
    assert p2[:n_hot].min() >= 0.8 - 1e-12
    assert abs(ranked_probs(c3).mean() - 0.12) < 0.002
    p4 = ranked_probs(c4)
    k = int(round(0.26 * c4.f))
    assert abs(p4.mean() - 0.05) < 0.002
    assert abs(p4[:k].sum() / p4.sum() - 0.80) < 0.03
    assert abs(ranked_probs(c5).mean() - 0.04) < 0.002


def test_probs_are_a_seeded_permutation():
    c = W[0]
    a = activation_probs(c, 0, seed=0)
    b = activation_probs(c, 0, seed=0)
    assert np.array_equal(a, b)
    assert np.array_equal(np.sort(a), np.sort(ranked_probs(c)))
    assert not np.array_equal(a, ranked_probs(c))  # not already hot-first


def test_layer_shapes_and_dtypes():
    for w in W:
        s = scaled(w, d=256, f=300, r=32, n_layers=1)
        L = make_layer(s, 0)
        if w.wdtype == "int4g128":
            assert L["w_gate"].dtype == torch.uint8 and L["w_gate"].shape == (300, 128)
            assert L["s_gate"].dtype == torch.float16 and L["s_gate"].shape == (300, 2)
        else:
            assert L["w_gate"].shape == (300, 256)
        assert (L["w_up"] is None) == (w.kind == "relu")
        assert L["p1_t"].shape == (32, 256) and L["p2_t"].shape == (300, 32)
        assert L["b_gate"].dtype == torch.float32 and L["b_pred"].dtype == torch.float32
        assert L["counts"].dtype == torch.int32
    x = make_inputs(W[0], 3, 2)
    assert x.shape == (3, 2, 512) and x.dtype == torch.float32


def test_profiling_counts_follow_probs():
    c = scaled(W[2], d=128, f=4000, r=16, n_layers=1)
    L = make_layer(c, 0)
    p = L["p"].numpy()
    cnt = L["counts"].numpy()
    assert np.all((cnt >= 0) & (cnt <= T_CALIB))
    assert np.corrcoef(cnt / T_CALIB, p)[0, 1] > 0.99


def test_single_layer_fire_rates():
    """Full-size single-layer workload: predictor and gate fire at ~the target mean rate."""
    c = W[0]
    L = oracle.layer_numpy(make_layer(c, 0))
    X = make_inputs(c, 300, 1).numpy()[:, 0, :].astype(np.float64)
    U = X / np.sqrt((X * X).mean(axis=1, keepdims=True) + 1e-6)
    pred_rate = np.mean([oracle.predict(u, L["p1_t"], L["p2_t"], L["b_pred"], "f32")["count"] for u in U]) / c.f
    gate_rate = brute.true_set(U, L, "f32").sum() / c.f  # union over 300 rows: sanity only
    G = U @ L["w_gate"].astype(np.float64).T + L["b_gate"]
    gate_mean = (G > 0).mean()
    assert abs(pred_rate - 0.10) / 0.10 < 0.10, pred_rate
    assert abs(gate_mean - 0.10) / 0.10 < 0.10, gate_mean
    assert gate_rate > gate_mean


@pytest.mark.parametrize("name", [W[1].name])
def test_hot_prefix_rates_full_size(name):
    """ReluLLaMA-7B-shaped layer: per-neuron predictor firing tracks p; the hot 10% fires on >= ~80%."""
    c = WORKLOADS[name]
    L = oracle.layer_numpy(make_layer(c, 0))
    p = L["p"]
    X = make_inputs(c, 48, 1).numpy()[:, 0, :].astype(np.float64)
    U = X / np.sqrt((X * X).mean(axis=1, keepdims=True) + 1e-6)
    fired = np.zeros(c.f)
    counts = []
    for u in U:
        pr = oracle.predict(u, L["p1_t"], L["p2_t"], L["b_pred"], "bf16")
        fired[pr["idx"]] += 1
        counts.append(pr["count"])
    rate = fired / len(U)
    assert abs(np.mean(counts) / c.f - 0.10) / 0.10 < 0.10
    hot = np.argsort(-p, kind="stable")[: int(0.1 * c.f)]
    assert rate[hot].mean() > 0.8
