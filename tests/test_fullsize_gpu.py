"""GPU parity at the workloads' full sizes, through the same C-ABI calls and
launch configuration the benchmark uses.

Per workload: layer 0 (or more) generated at full d, f, r; the predictor's active
set compared with the oracle's outside the 1e-4 band, and the sparse FFN compared
with the oracle on the oracle's active list, for every batch size the workload
names. The ReluLLaMA-7B-shaped 32-layer stack is also run end to end through
pi_decode_stack, every layer checked teacher-forced (the oracle's layer on the GPU's
own layer input) and the free-running oracle compared where no in-band flip occurs.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_cases import TOL, band_mask, build_layers, rel_l2, rms_inputs, teacher_forced, to_dev
from workload import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu
W = list(WORKLOADS.values())
CASES = [(w.name, B) for w in W for B in w.batches]


@pytest.fixture(scope="module")
def P():
    import activation_sparse_decode_pi_gb300 as P

    return P


@pytest.mark.parametrize("name,B", CASES)
def test_layer_full_size(P, name, B):
    w = WORKLOADS[name]
    (Lg, Lo), = build_layers(w, [0])
    ffn = P.SparseFFN.from_workload(w, [Lg], max_batch=B)
    u = rms_inputs(w, B, seed=3)[0]
    u64 = u.astype(np.float64)
    ud = to_dev(u)
    idx, cnt = ffn.predict(0, ud)
    torch.cuda.synchronize()
    n = int(cnt.item())
    gi = idx[:n].cpu().numpy()
    pr = oracle.predict(u64, Lo["p1_t"], Lo["p2_t"], Lo["b_pred"], w.pdtype)
    diff = np.setxor1d(gi, pr["idx"])
    assert np.all(band_mask(pr["z"])[diff]), f"{diff.size} out-of-band mismatches"
    assert np.all(np.diff(gi) > 0)
    # the FFN on the oracle's own list
    oi = pr["idx"].astype(np.int32)
    idx_o = torch.zeros(max(1, oi.size), dtype=torch.int32, device="cuda")
    idx_o[: oi.size] = to_dev(oi)
    y = ffn.sparse_ffn(0, ud, idx_o, torch.tensor([oi.size], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    _, yo = oracle.sparse_ffn(u64, Lo, oi, w.kind, w.wdtype)
    err = rel_l2(y.cpu().numpy(), yo)
    assert err <= TOL[w.wdtype], err
    assert ffn.status() == 0
    ffn.close()
    del Lg, Lo
    torch.cuda.empty_cache()


def test_benchmark_stack_end_to_end(P):
    """All 32 layers of the ReluLLaMA-7B-shaped stack through pi_decode_stack: every layer
    checked teacher-forced, and the free-running oracle compared where no in-band flip occurs."""
    w = WORKLOADS["relullama7b_d4096_f11008_bf16_L32"]
    layers = build_layers(w, range(w.n_layers))
    ffn = P.SparseFFN.from_workload(w, [g for g, _ in layers], max_batch=1)
    X = make_inputs(w, 3, 1, seed=1000, device="cpu").numpy()
    compared = 0
    for t in range(X.shape[0]):
        counts = torch.zeros(w.n_layers, dtype=torch.int32, device="cuda")
        idx_out = torch.zeros((w.n_layers, w.f), dtype=torch.int32, device="cuda")
        xo = ffn.decode_stack(to_dev(X[t]), counts=counts, idx_out=idx_out)
        torch.cuda.synchronize()
        xt, _ = teacher_forced(P, w, layers, ffn, X[t], tag=t)
        assert np.array_equal(xt, xo.cpu().numpy())
        st = oracle.stack(X[t].astype(np.float64), [o for _, o in layers], w.kind, w.wdtype, w.pdtype)
        cg, ig = counts.cpu().numpy(), idx_out.cpu().numpy()
        same = True
        for l in range(w.n_layers):
            diff = np.setxor1d(ig[l, : cg[l]], st["idx"][l])
            if diff.size:
                assert np.all(st["zmin"][l][diff] < oracle.BAND), (t, l, diff)
                same = False
                break
        if same:
            compared += 1
            assert rel_l2(xo.cpu().numpy() - X[t], st["x_out"] - X[t]) <= TOL[w.wdtype]
    assert ffn.status() == 0
    ffn.close()


@pytest.mark.parametrize("r", [128, 256, 512])
def test_predictor_rank_sweep_full_size(P, r):
    """The predictor ranks of the rank sweep, at the benchmark workload's full d and f, layer 0."""
    import dataclasses

    w = dataclasses.replace(WORKLOADS["relullama7b_d4096_f11008_bf16_L32"], r=r)
    (Lg, Lo), = build_layers(w, [0])
    ffn = P.SparseFFN.from_workload(w, [Lg], max_batch=1)
    u = rms_inputs(w, 1, seed=9)[0]
    idx, cnt = ffn.predict(0, to_dev(u))
    torch.cuda.synchronize()
    gi = idx[: int(cnt.item())].cpu().numpy()
    pr = oracle.predict(u.astype(np.float64), Lo["p1_t"], Lo["p2_t"], Lo["b_pred"], w.pdtype)
    diff = np.setxor1d(gi, pr["idx"])
    assert np.all(band_mask(pr["z"])[diff]), f"{diff.size} out-of-band mismatches"
    # and one decode step through the persistent kernel of a 2-layer stack at this rank
    w2 = dataclasses.replace(w, n_layers=2)
    layers = build_layers(w2, range(2))
    ffn2 = P.SparseFFN.from_workload(w2, [g for g, _ in layers], max_batch=1)
    X = make_inputs(w2, 1, 1, seed=21, device="cpu").numpy()
    teacher_forced(P, w2, layers, ffn2, X[0], tag=r)
    assert ffn.status() == 0 and ffn2.status() == 0
    ffn.close()
    ffn2.close()
