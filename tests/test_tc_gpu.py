"""Tensor-core (tcgen05) path of the batched kernels.

First the operand layouts on their own: one tile product D = A * B^T through
pi_selftest_umma, with small-integer operands so that every product and sum is
exact in fp32 and the comparison with an integer matmul can be exact, for both
staging orders of A (K-major and MN-major), both 16-bit types, every N the kernels
use and one or two 64-wide K blocks.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def P():
    import activation_sparse_decode_pi_gb300 as P

    return P


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("n", [16, 32, 64, 128])
@pytest.mark.parametrize("k", [64, 128])
def test_umma_tile_exact(P, mode, dtype, n, k):
    rng = np.random.default_rng(1000 * mode + 10 * n + k + (dtype == "f16"))
    A = rng.integers(-4, 5, size=(128, k))
    B = rng.integers(-4, 5, size=(n, k))
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    a_host = A if mode == 0 else A.T
    a = torch.tensor(np.ascontiguousarray(a_host), dtype=tdt, device="cuda")
    b = torch.tensor(B, dtype=tdt, device="cuda")
    d = torch.full((128, n), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    P.pi_selftest_umma(a, b, d, mode, n, k, P.DTYPES[dtype], status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    np.testing.assert_array_equal(d.cpu().numpy(), (A @ B.T).astype(np.float32))


def test_umma_selftest_rejects_bad_shapes(P):
    a = torch.zeros((128, 64), dtype=torch.bfloat16, device="cuda")
    d = torch.zeros((128, 16), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for n, k in [(8, 64), (16, 32), (256, 64)]:
        with pytest.raises(P.PiError):
            P.pi_selftest_umma(a, a, d, 0, n, k, P.PI_BF16, st)


# ------------------------------------------------------------------ the path against the oracle
#
# Shapes where the tensor-core kernels apply (d % 128 == 0, r % 64 == 0) with a ragged
# neuron count, several 128-row tiles and stream-K splits, a predictor rank that is not a
# multiple of 128, and batches that fill NB = 16, 32, 64, 128 exactly and raggedly.
import os
from contextlib import contextmanager

import oracle
from tests.gpu_cases import TOL, band_mask, build_layers, rel_l2, rms_inputs, to_dev
from tests.test_parity_gpu import _lists, _stack_check
from workload import WORKLOADS, scaled

W = list(WORKLOADS.values())
TC_SHAPES = [dict(d=1152, f=3001, r=128), dict(d=768, f=700, r=192)]
TC_W = [1, 2, 3]   # bf16 gated, bf16 gated, fp16 non-gated


@contextmanager
def _env(**kv):
    old = {k: os.environ.get(k) for k in kv}
    try:
        for k, v in kv.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
        yield
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def _handle(P, w, layers, B, min_batch=None):
    # the tensor-core predictor too (not the optional one-launch predictor of small batches)
    with _env(PI_FFN_TC="1", PI_FFN_PRED_FUSED="0", PI_FFN_TC_MIN_BATCH=None if min_batch is None else str(min_batch)):
        return P.SparseFFN.from_workload(w, layers, max_batch=B)


def _predict_check(P, ffn, w, Lo, B, seed):
    u = rms_inputs(w, B, seed=seed)[0]
    P.pi_profile_begin(ffn.h)
    idx, cnt = ffn.predict(0, to_dev(u))
    prof = P.pi_profile_end(ffn.h)
    assert prof["rms"][1] == 1, f"tensor-core path not taken: {prof}"   # its activation split
    n = int(cnt.item())
    gi = idx[:n].cpu().numpy()
    pr = oracle.predict(u.astype(np.float64), Lo["p1_t"], Lo["p2_t"], Lo["b_pred"], w.pdtype)
    assert np.all(np.diff(gi) > 0), "active list must be ascending and unique"
    diff = np.setxor1d(gi, pr["idx"])
    assert np.all(band_mask(pr["z"])[diff]), f"{diff.size} out-of-band mismatches"
    assert ffn.status() == 0
    return u, pr


def _ffn_check(P, ffn, w, Lo, u, pr, seed):
    u64 = u.astype(np.float64)
    ud = to_dev(u)
    rng = np.random.default_rng(seed)
    for name, lst in _lists(rng, w.f, pr["idx"]).items():
        idx = torch.zeros(max(1, lst.size), dtype=torch.int32, device="cuda")
        idx[: lst.size] = to_dev(lst) if lst.size else idx[:0]
        cnt = torch.tensor([lst.size], dtype=torch.int32, device="cuda")
        y = ffn.sparse_ffn(0, ud, idx, cnt)
        y2 = ffn.sparse_ffn(0, ud, idx, cnt).clone()
        torch.cuda.synchronize()
        assert torch.equal(y, y2), "not deterministic"
        _, yo = oracle.sparse_ffn(u64, Lo, lst, w.kind, w.wdtype)
        yg = y.cpu().numpy()
        if lst.size == 0:
            assert np.all(yg == 0.0)
        else:
            err = rel_l2(yg, yo)
            assert err <= TOL[w.wdtype], (name, err)
    assert ffn.status() == 0


@pytest.mark.parametrize("B", [16, 17, 32, 64, 100])
@pytest.mark.parametrize("shape", range(len(TC_SHAPES)))
@pytest.mark.parametrize("wi", TC_W)
def test_tc_predict_and_ffn(P, wi, shape, B):
    w = scaled(W[wi], n_layers=1, **TC_SHAPES[shape])
    (Lg, Lo), = build_layers(w, [0])
    ffn = _handle(P, w, [Lg], B)
    u, pr = _predict_check(P, ffn, w, Lo, B, seed=B)
    _ffn_check(P, ffn, w, Lo, u, pr, seed=wi * 100 + B)
    ffn.close()


@pytest.mark.parametrize("B", [1, 2, 5])
def test_tc_small_batches_pad(P, B):
    """Below 16 rows (path forced on): the batch tile is padded with zero rows."""
    w = scaled(W[2], n_layers=1, **TC_SHAPES[0])
    (Lg, Lo), = build_layers(w, [0])
    ffn = _handle(P, w, [Lg], B, min_batch=1)
    u, pr = _predict_check(P, ffn, w, Lo, B, seed=7 + B)
    _ffn_check(P, ffn, w, Lo, u, pr, seed=B)
    ffn.close()


def test_tc_device_checks(P):
    w = scaled(W[3], n_layers=1, **TC_SHAPES[0])
    (Lg, Lo), = build_layers(w, [0])
    ffn = _handle(P, w, [Lg], 16)
    u = rms_inputs(w, 16)[0]
    lst = np.array([5, w.f + 7, 9, -3, 100], np.int32)
    y = ffn.sparse_ffn(0, to_dev(u), to_dev(lst), torch.tensor([5], dtype=torch.int32, device="cuda"))
    assert ffn.status() == P.PI_ERR_DEVICE_CHECK
    _, yo = oracle.sparse_ffn(u.astype(np.float64), Lo, [5, 9, 100], w.kind, w.wdtype)
    assert rel_l2(y.cpu().numpy(), yo) <= TOL[w.wdtype]
    idx = torch.arange(w.f, dtype=torch.int32, device="cuda")
    y = ffn.sparse_ffn(0, to_dev(u), idx, torch.tensor([w.f + 50], dtype=torch.int32, device="cuda"))
    assert ffn.status() == P.PI_ERR_DEVICE_CHECK
    yd = oracle.dense_ffn(u.astype(np.float64), Lo, w.kind, w.wdtype)
    assert rel_l2(y.cpu().numpy(), yd) <= TOL[w.wdtype]
    ffn.close()


@pytest.mark.parametrize("wi,B", [(1, 16), (2, 16), (3, 32), (2, 40)])
def test_tc_decode_stack(P, wi, B):
    """Free-running stack through the tensor-core kernels, with graph replay, against the oracle."""
    w = scaled(W[wi], n_layers=3, **TC_SHAPES[0])
    compared, flips = _stack_check(P, w, B, tokens=2, seed=wi)
    assert compared >= 1


@pytest.mark.parametrize("kw,ds", [(2, 1), (1, 2), (1, 1)])
@pytest.mark.parametrize("wi,B", [(2, 16), (3, 32), (1, 64)])
def test_tc_step_widths(P, kw, ds, wi, B):
    """One or two K blocks per pipeline step in the row products, one or two column slices per W_down tile."""
    w = scaled(W[wi], n_layers=1, d=1536, f=2500, r=128)   # d a multiple of 2 x 128, r of 2 x 64
    (Lg, Lo), = build_layers(w, [0])
    with _env(PI_FFN_TC_KW=str(kw), PI_FFN_TC_DS=str(ds)):
        ffn = _handle(P, w, [Lg], B)
    u, pr = _predict_check(P, ffn, w, Lo, B, seed=3 * B)
    _ffn_check(P, ffn, w, Lo, u, pr, seed=kw * 10 + ds)
    ffn.close()


@pytest.mark.parametrize("H", [100, 128, 1000, 2999, 3001])
@pytest.mark.parametrize("wi,B", [(2, 16), (3, 32)])
def test_tc_hot_prefix(P, wi, B, H):
    """Tensor-core logits with a hot prefix: the tiles start at the last 128-row boundary
    inside it, the words below are all ones, the rows in between are forced active."""
    w = scaled(W[wi], n_layers=1, **TC_SHAPES[0])
    (Lg, Lo), = build_layers(w, [0])
    ffn = _handle(P, w, [Lg], B)
    ffn.set_hot_prefix(H)
    u = rms_inputs(w, B, seed=H)[0]
    idx, cnt = ffn.predict(0, to_dev(u))
    torch.cuda.synchronize()
    gi = idx[: int(cnt.item())].cpu().numpy()
    pr = oracle.predict(u.astype(np.float64), Lo["p1_t"], Lo["p2_t"], Lo["b_pred"], w.pdtype, hot_prefix=H)
    assert np.all(np.diff(gi) > 0)
    assert np.array_equal(gi[:H], np.arange(H))
    diff = np.setxor1d(gi, pr["idx"])
    assert np.all(band_mask(pr["z"])[diff]), f"{diff.size} out-of-band mismatches"
    assert ffn.status() == 0
    ffn.close()
