"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Bars: index work (hot-first order, row permutation, active lists) bit-exact,
except active-set membership of neurons whose oracle logit lies within 1e-4 of
the threshold; FFN outputs within relative L2 1e-3 (fp32/bf16/fp16 weights) or
5e-3 (int4) of the oracle evaluated on the same active list.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_cases import TOL, band_mask, build_layers, rel_l2, rms_inputs, teacher_forced, to_dev
from workload import WORKLOADS, make_inputs, scaled

pytestmark = pytest.mark.gpu
W = list(WORKLOADS.values())
SMALL = dict(d=640, f=1007, r=72)          # several K2 words + a ragged word, several K3/K4a tiles
MID = dict(d=2304, f=3001, r=136)


@pytest.fixture(scope="module")
def P():
    import activation_sparse_decode_pi_gb300 as P

    return P


def _wl(wi, shape, n_layers=1):
    return scaled(W[wi], n_layers=n_layers, **shape)


# ------------------------------------------------------------------ offline order --------------

@pytest.mark.parametrize("f", [1, 31, 1000, 4099, 49152])
def test_hot_first_order(P, f):
    rng = np.random.default_rng(f)
    for counts in (rng.integers(0, 20, f), np.zeros(f, np.int64), np.arange(f)[::-1].copy(),
                   rng.integers(0, 2**31 - 1, f)):
        perm = P.hot_first_order(to_dev(counts.astype(np.int32)))
        assert np.array_equal(perm.cpu().numpy(), oracle.hot_first_order(counts))


@pytest.mark.parametrize("row_bytes", [16, 6, 100, 2048])
def test_permute_rows(P, row_bytes):
    rng = np.random.default_rng(row_bytes)
    rows = 777
    src = rng.integers(0, 256, (rows, row_bytes), dtype=np.uint8)
    perm = rng.permutation(rows).astype(np.int32)
    dst = P.permute_rows(to_dev(src), to_dev(perm))
    assert np.array_equal(dst.cpu().numpy(), src[perm])
    # out-of-range entries are counted and their rows left unwritten
    bad = perm.copy()
    bad[[3, 50]] = [-1, rows]
    out = torch.zeros((rows, row_bytes), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    P.pi_permute_rows(to_dev(src), out, to_dev(bad), rows, row_bytes, err)
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    assert int(err.item()) == 2
    assert np.all(o[[3, 50]] == 0)
    keep = np.setdiff1d(np.arange(rows), [3, 50])
    assert np.array_equal(o[keep], src[bad[keep]])


# ------------------------------------------------------------------ predictor -----------------

@pytest.mark.parametrize("B", [1, 3, 8, 16])
@pytest.mark.parametrize("wi", range(5))
def test_predict_small(P, wi, B):
    w = _wl(wi, SMALL)
    (Lg, Lo), = build_layers(w, [0])
    ffn = P.SparseFFN.from_workload(w, [Lg], max_batch=B)
    u = rms_inputs(w, B)[0]
    idx, cnt = ffn.predict(0, to_dev(u))
    torch.cuda.synchronize()
    n = int(cnt.item())
    gi = idx[:n].cpu().numpy()
    pr = oracle.predict(u.astype(np.float64), Lo["p1_t"], Lo["p2_t"], Lo["b_pred"], w.pdtype)
    assert 0 < pr["count"] < w.f
    assert np.all(np.diff(gi) > 0), "active list must be ascending and unique"
    diff = np.setxor1d(gi, pr["idx"])
    assert np.all(band_mask(pr["z"])[diff]), f"{diff.size} out-of-band mismatches"
    assert ffn.status() == 0
    ffn.close()


@pytest.mark.parametrize("B", [1, 2, 5, 8])
@pytest.mark.parametrize("wi", range(5))
def test_predict_fused_vs_two_kernels(P, wi, B):
    """The optional one-launch predictor of batches up to 8 (PI_FFN_PRED_FUSED=1: hidden layer over
    all SMs, a grid barrier, logits of contiguous mask words, compaction by the last CTA): against
    the oracle, and the same list as the two-kernel predictor outside the threshold band."""
    w = _wl(wi, MID)
    (Lg, Lo), = build_layers(w, [0])
    u = rms_inputs(w, B, seed=11 + B)[0]
    pr = oracle.predict(u.astype(np.float64), Lo["p1_t"], Lo["p2_t"], Lo["b_pred"], w.pdtype)
    lists = {}
    for fused in ("1", "0"):
        ffn = _with_env("PI_FFN_PRED_FUSED", fused, lambda: P.SparseFFN.from_workload(w, [Lg], max_batch=B))
        P.pi_profile_begin(ffn.h)
        idx, cnt = ffn.predict(0, to_dev(u))
        prof = P.pi_profile_end(ffn.h)
        assert (prof["pred_fused"][1] == 1) == (fused == "1"), prof
        n = int(cnt.item())
        gi = idx[:n].cpu().numpy()
        assert np.all(np.diff(gi) > 0), "active list must be ascending and unique"
        diff = np.setxor1d(gi, pr["idx"])
        assert np.all(band_mask(pr["z"])[diff]), (fused, f"{diff.size} out-of-band mismatches")
        idx2, cnt2 = ffn.predict(0, to_dev(u))
        assert int(cnt2.item()) == n and torch.equal(idx2[:n], idx[:n]), "predictor is not deterministic"
        assert ffn.status() == 0
        lists[fused] = gi
        ffn.close()
    diff = np.setxor1d(lists["1"], lists["0"])
    assert np.all(band_mask(pr["z"])[diff])


# ------------------------------------------------------------------ sparse FFN ----------------

def _lists(rng, f, pred_idx):
    sub = rng.choice(f, size=min(f, 97), replace=False).astype(np.int32)   # unsorted on purpose
    return {"predicted": pred_idx.astype(np.int32), "all": np.arange(f, dtype=np.int32),
            "empty": np.zeros(0, np.int32), "random_unsorted": sub, "single": np.array([f - 1], np.int32)}


@pytest.mark.parametrize("B", [1, 4, 16])
@pytest.mark.parametrize("wi", range(5))
def test_sparse_ffn_small(P, wi, B):
    w = _wl(wi, SMALL)
    (Lg, Lo), = build_layers(w, [0])
    ffn = P.SparseFFN.from_workload(w, [Lg], max_batch=B)
    u = rms_inputs(w, B)[0]
    u64 = u.astype(np.float64)
    pr = oracle.predict(u64, Lo["p1_t"], Lo["p2_t"], Lo["b_pred"], w.pdtype)
    rng = np.random.default_rng(wi * 10 + B)
    ud = to_dev(u)
    for name, lst in _lists(rng, w.f, pr["idx"]).items():
        idx = torch.zeros(max(1, lst.size), dtype=torch.int32, device="cuda")
        idx[: lst.size] = to_dev(lst) if lst.size else idx[:0]
        cnt = torch.tensor([lst.size], dtype=torch.int32, device="cuda")
        y = ffn.sparse_ffn(0, ud, idx, cnt)
        torch.cuda.synchronize()
        _, yo = oracle.sparse_ffn(u64, Lo, lst, w.kind, w.wdtype)
        yg = y.cpu().numpy()
        if lst.size == 0:
            assert np.all(yg == 0.0)
        else:
            err = rel_l2(yg, yo)
            assert err <= TOL[w.wdtype], (name, err)
    assert ffn.status() == 0
    ffn.close()


def test_sparse_ffn_is_deterministic(P):
    w = _wl(1, MID)
    (Lg, Lo), = build_layers(w, [0])
    ffn = P.SparseFFN.from_workload(w, [Lg], max_batch=4)
    ud = to_dev(rms_inputs(w, 4)[0])
    idx = torch.arange(w.f, dtype=torch.int32, device="cuda")
    cnt = torch.tensor([w.f], dtype=torch.int32, device="cuda")
    y1 = ffn.sparse_ffn(0, ud, idx, cnt).clone()
    y2 = ffn.sparse_ffn(0, ud, idx, cnt)
    assert torch.equal(y1, y2)
    ffn.close()


def test_device_checks(P):
    """Out-of-range list entries and counts are flagged, skipped, and never read."""
    w = _wl(0, SMALL)
    (Lg, Lo), = build_layers(w, [0])
    ffn = P.SparseFFN.from_workload(w, [Lg], max_batch=2)
    u = rms_inputs(w, 2)[0]
    lst = np.array([5, w.f + 7, 9, -3, 100], np.int32)
    y = ffn.sparse_ffn(0, to_dev(u), to_dev(lst), torch.tensor([5], dtype=torch.int32, device="cuda"))
    assert ffn.status() == P.PI_ERR_DEVICE_CHECK
    assert ffn.status() == 0   # cleared
    _, yo = oracle.sparse_ffn(u.astype(np.float64), Lo, [5, 9, 100], w.kind, w.wdtype)
    assert rel_l2(y.cpu().numpy(), yo) <= TOL[w.wdtype]
    # a count above f is clamped to f
    idx = torch.arange(w.f, dtype=torch.int32, device="cuda")
    y = ffn.sparse_ffn(0, to_dev(u), idx, torch.tensor([w.f + 50], dtype=torch.int32, device="cuda"))
    assert ffn.status() == P.PI_ERR_DEVICE_CHECK
    yd = oracle.dense_ffn(u.astype(np.float64), Lo, w.kind, w.wdtype)
    assert rel_l2(y.cpu().numpy(), yd) <= TOL[w.wdtype]
    ffn.close()


def test_host_side_rejections(P):
    w = _wl(1, SMALL)
    (Lg, Lo), = build_layers(w, [0])
    ffn = P.SparseFFN.from_workload(w, [Lg], max_batch=2)
    u = to_dev(rms_inputs(w, 2)[0])
    idx = torch.zeros(w.f, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    host = np.zeros((2, w.d), np.float32)
    with pytest.raises(P.PiError) as e:
        P.pi_predict(ffn.h, 0, host.ctypes.data, 2, idx, cnt)      # host pointer
    assert e.value.code == P.PI_ERR_INVALID_ARG
    with pytest.raises(P.PiError):
        P.pi_predict(ffn.h, 0, u.data_ptr() + 4, 1, idx, cnt)     # misaligned
    with pytest.raises(P.PiError):
        P.pi_predict(ffn.h, 0, u, 3, idx, cnt)                    # B > max_batch
    with pytest.raises(P.PiError):
        P.pi_predict(ffn.h, 1, u, 2, idx, cnt)                    # layer out of range
    with pytest.raises(P.PiError):
        P.pi_sparse_ffn(ffn.h, 0, u, 2, idx, cnt, None)           # NULL output
    # a layer whose weights would run past the end of their allocation
    big = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    seg = [s for s in torch.cuda.memory_snapshot()
           if s["address"] <= big.data_ptr() < s["address"] + s["total_size"]][0]
    end = seg["address"] + seg["total_size"]
    bad = dict(Lg)
    bad["w_gate"] = end - 4096
    with pytest.raises(P.PiError) as e:
        P.SparseFFN.from_workload(w, [bad])
    assert e.value.code == P.PI_ERR_INVALID_ARG
    ffn.close()


# ------------------------------------------------------------------ layer stack ---------------

def _stack_check(P, w, B, tokens, seed=0):
    layers = build_layers(w, range(w.n_layers), seed)
    ffn = P.SparseFFN.from_workload(w, [g for g, _ in layers], max_batch=B)
    X = make_inputs(w, tokens, B, seed, device="cpu").numpy()
    compared, flips = 0, 0
    for t in range(tokens):
        x0 = to_dev(X[t])
        counts = torch.zeros(w.n_layers, dtype=torch.int32, device="cuda")
        idx_out = torch.zeros((w.n_layers, w.f), dtype=torch.int32, device="cuda")
        xo = ffn.decode_stack(x0, counts=counts, idx_out=idx_out)
        xo2 = ffn.decode_stack(x0, counts=counts, idx_out=idx_out).clone()   # graph replay
        torch.cuda.synchronize()
        assert torch.equal(xo, xo2), "decode step is not deterministic"
        xt, _ = teacher_forced(P, w, layers, ffn, X[t], tag=(w.name, B, t))   # every layer, flips included
        assert np.array_equal(xt, xo.cpu().numpy()), "decode step with layer outputs differs"
        st = oracle.stack(X[t].astype(np.float64), [o for _, o in layers], w.kind, w.wdtype, w.pdtype)
        cg = counts.cpu().numpy()
        ig = idx_out.cpu().numpy()
        same = True
        for l in range(w.n_layers):
            gi = ig[l, : cg[l]]
            assert np.all(np.diff(gi) > 0)
            diff = np.setxor1d(gi, st["idx"][l])
            if diff.size:
                # allowed only inside the band, and then later layers no longer compare
                assert np.all(st["zmin"][l][diff] < oracle.BAND), (l, diff)
                same = False
                flips += 1
                break
        if same:
            compared += 1
            err = rel_l2(xo.cpu().numpy() - X[t], st["x_out"] - X[t])
            assert err <= TOL[w.wdtype], err
    assert ffn.status() == 0
    ffn.close()
    return compared, flips


@pytest.mark.parametrize("wi", range(5))
def test_decode_stack_small(P, wi):
    w = _wl(wi, SMALL, n_layers=3)
    for B in sorted({1, max(W[wi].batches)}):
        compared, flips = _stack_check(P, w, B, tokens=2)
        assert compared >= 1


def test_decode_stack_under_user_capture(P):
    """Inside a caller's stream capture the step is enqueued into the caller's graph."""
    w = _wl(2, SMALL, n_layers=2)
    layers = build_layers(w, range(2))
    ffn = P.SparseFFN.from_workload(w, [g for g, _ in layers], max_batch=4)
    x0 = to_dev(make_inputs(w, 1, 4).numpy()[0])
    ref = ffn.decode_stack(x0).clone()
    out = torch.empty_like(x0)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        ffn.decode_stack(x0, x_out=out, stream=s)      # warm-up outside capture
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            ffn.decode_stack(x0, x_out=out, stream=s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    ffn.close()


# ------------------------------------------------------------------ persistent decode-step kernel

STACK_SHAPE = dict(d=2048, f=3001, r=136)   # int4 rows need d % 1024 == 0 on this path


def _handle(P, w, layers, stack_kernel: bool):
    import os

    old = os.environ.get("PI_FFN_STACK_KERNEL")
    os.environ["PI_FFN_STACK_KERNEL"] = "1" if stack_kernel else "0"
    try:
        return P.SparseFFN.from_workload(w, layers, max_batch=1)
    finally:
        if old is None:
            del os.environ["PI_FFN_STACK_KERNEL"]
        else:
            os.environ["PI_FFN_STACK_KERNEL"] = old


# r % 32 == 0 with 16-bit predictor weights: the logits run on the tensor cores (mma.sync,
# staged rows from shared memory, the rest from memory); r = 136 keeps them on the CUDA cores
STACK_SHAPE_TC = dict(d=2048, f=3001, r=160)
# d * 4 bytes >= r * 4 + 8 KB: hp and the reduction scratch share u's shared-memory region
STACK_SHAPE_SHARED = dict(d=4096, f=3001, r=256)
# fewer neurons than SMs: most CTAs own one neuron (a one-row logit tile) or none
STACK_SHAPE_FEW = dict(d=1024, f=100, r=64)


def _stack_vs_oracle(P, w, layers, X, ffn, tag, hot_prefix=0):
    """One decode step per token of X against the oracle, teacher-forced layer by layer (every
    layer compared: active lists outside the band, outputs within the dtype's bar); the step is
    deterministic and the call that keeps layer outputs gives the same bits as the plain one.
    Returns the number of layers that had an in-band difference."""
    flips = 0
    for t in range(X.shape[0]):
        xo = ffn.decode_stack(to_dev(X[t]))
        xo2 = ffn.decode_stack(to_dev(X[t])).clone()
        torch.cuda.synchronize()
        assert torch.equal(xo, xo2), "decode step is not deterministic"
        xt, fl = teacher_forced(P, w, layers, ffn, X[t], hot_prefix=hot_prefix, tag=(tag, t))
        assert np.array_equal(xt, xo.cpu().numpy()), (tag, t, "layer-output call differs")
        flips += fl
    return flips


@pytest.mark.parametrize("shape", [STACK_SHAPE, STACK_SHAPE_TC, STACK_SHAPE_SHARED, STACK_SHAPE_FEW],
                         ids=["r136", "r160", "d4096", "f100"])
@pytest.mark.parametrize("wi", range(5))
def test_decode_stack_both_paths_batch1(P, wi, shape):
    """Batch 1: the single persistent kernel and the multi-kernel step both match the oracle."""
    w = _wl(wi, shape, n_layers=3)
    layers = build_layers(w, range(w.n_layers))
    X = make_inputs(w, 2, 1, seed=5, device="cpu").numpy()
    for stack_kernel in (True, False):
        ffn = _handle(P, w, [g for g, _ in layers], stack_kernel)
        P.pi_profile_begin(ffn.h)
        ffn.decode_stack(to_dev(X[0]))
        prof = P.pi_profile_end(ffn.h)
        if stack_kernel:
            assert prof["decode_stack"][1] == 1 and prof["ffn_h"][1] == 0, prof
        else:
            assert prof["decode_stack"][1] == 0 and prof["ffn_h"][1] == w.n_layers, prof
        _stack_vs_oracle(P, w, layers, X, ffn, stack_kernel)
        assert ffn.status() == 0
        ffn.close()


@pytest.mark.parametrize("group", ["1", "2", "8"])
@pytest.mark.parametrize("wi", [1, 3, 4])
def test_decode_stack_spread_neurons(P, wi, group):
    """The FFN's active neurons spread over all CTAs (one more grid barrier) or within groups of 2
    and 8 CTAs (lists exchanged through memory): the same layers against the oracle, teacher-forced,
    and repeated steps give the same bits."""
    w = _wl(wi, STACK_SHAPE, n_layers=3)
    layers = build_layers(w, range(w.n_layers))
    X = make_inputs(w, 2, 1, seed=31, device="cpu").numpy()
    ffn = _with_env("PI_FFN_STACK_BALANCE", group, lambda: _handle(P, w, [g for g, _ in layers], stack_kernel=True))
    P.pi_profile_begin(ffn.h)
    ffn.decode_stack(to_dev(X[0]))
    prof = P.pi_profile_end(ffn.h)
    assert prof["decode_stack"][1] == 1, prof
    _stack_vs_oracle(P, w, layers, X, ffn, (wi, group))
    assert ffn.status() == 0
    ffn.close()


@pytest.mark.parametrize("wi", [1, 3, 4])
def test_decode_stack_tc_logits_many_tiles(P, wi):
    """~300 owned P2 rows per CTA, all staged: more 16-row tiles than warps, each warp taking
    whole tiles (the other shapes split a tile's k range over several warps)."""
    w = _wl(wi, dict(d=1024, f=45600, r=256), n_layers=2)
    layers = build_layers(w, range(w.n_layers))
    X = make_inputs(w, 2, 1, seed=21, device="cpu").numpy()
    ffn = _handle(P, w, [g for g, _ in layers], stack_kernel=True)
    _stack_vs_oracle(P, w, layers, X, ffn, wi)
    assert ffn.status() == 0
    ffn.close()


# d 12288 with 16-bit weights: three 16-byte column chunks per thread and only two ring slots
STACK_SHAPE_WIDE = dict(d=12288, f=3001, r=144)


@pytest.mark.parametrize("wi", [1, 3])
def test_decode_stack_three_chunks_per_thread(P, wi):
    w = _wl(wi, STACK_SHAPE_WIDE, n_layers=3)
    layers = build_layers(w, range(w.n_layers))
    X = make_inputs(w, 2, 1, seed=23, device="cpu").numpy()
    ffn = _handle(P, w, [g for g, _ in layers], stack_kernel=True)
    P.pi_profile_begin(ffn.h)
    ffn.decode_stack(to_dev(X[0]))
    prof = P.pi_profile_end(ffn.h)
    assert prof["decode_stack"][1] == 1, prof
    _stack_vs_oracle(P, w, layers, X, ffn, ("wide", wi))
    assert ffn.status() == 0
    ffn.close()


@pytest.mark.parametrize("kind", ["relu", "gated"])
@pytest.mark.parametrize("d", [8192, 12288, 16384])
def test_decode_stack_int4_words_per_thread(P, d, kind):
    """int4 rows: the FFN's threads take one 32-bit word (8 columns) at a time, 2, 3 and 4 words
    of every row for d = 8192, 12288 and 16384; fc1/ReLU/fc2 and gated rows against the oracle."""
    import dataclasses

    w = dataclasses.replace(_wl(4, dict(d=d, f=3001, r=144), n_layers=2), kind=kind)
    layers = build_layers(w, range(w.n_layers))
    X = make_inputs(w, 2, 1, seed=41, device="cpu").numpy()
    ffn = _handle(P, w, [g for g, _ in layers], stack_kernel=True)
    P.pi_profile_begin(ffn.h)
    ffn.decode_stack(to_dev(X[0]))
    prof = P.pi_profile_end(ffn.h)
    assert prof["decode_stack"][1] == 1, prof
    _stack_vs_oracle(P, w, layers, X, ffn, ("int4", d, kind))
    assert ffn.status() == 0
    ffn.close()


def test_grid_barrier_gives_up_cleanly(P):
    """A barrier that can never complete times out, reports PI_ERR_TIMEOUT, and the GPU stays usable."""
    work = torch.zeros(4, dtype=torch.int32, device="cuda")
    P.pi_selftest_grid_barrier(work, 0)
    torch.cuda.synchronize()
    assert work.cpu().tolist()[2:] == [2, 0]
    work.zero_()
    P.pi_selftest_grid_barrier(work, 1)
    torch.cuda.synchronize()
    assert work.cpu().tolist()[2:] == [0, P.PI_ERR_TIMEOUT]
    # the context still runs a decode step afterwards
    w = _wl(1, SMALL, n_layers=1)
    (Lg, Lo), = build_layers(w, [0])
    ffn = P.SparseFFN.from_workload(w, [Lg], max_batch=1)
    x0 = to_dev(make_inputs(w, 1, 1).numpy()[0])
    xo = ffn.decode_stack(x0)
    torch.cuda.synchronize()
    assert torch.isfinite(xo).all()
    assert ffn.status() == 0
    ffn.close()


@pytest.mark.parametrize("wi", range(5))
def test_decode_stack_hot_neurons_bit_identical(P, wi):
    """Requesting the hot neurons' rows a layer ahead changes nothing in the output bits (hot slots
    keep every CTA on its own neurons, so the comparison runs with the FFN balancing off)."""
    w = _wl(wi, STACK_SHAPE, n_layers=3)
    layers = build_layers(w, range(w.n_layers))
    X = make_inputs(w, 3, 1, seed=11, device="cpu").numpy()
    ffn = _with_env("PI_FFN_STACK_BALANCE", "0", lambda: _handle(P, w, [g for g, _ in layers], stack_kernel=True))
    ref = []
    for t in range(X.shape[0]):
        counts = torch.zeros(w.n_layers, dtype=torch.int32, device="cuda")
        idx_out = torch.zeros((w.n_layers, w.f), dtype=torch.int32, device="cuda")
        xo = ffn.decode_stack(to_dev(X[t]), counts=counts, idx_out=idx_out)
        ref.append((xo.clone(), counts.clone(), idx_out.clone()))
    for n_hot in (1, 250, 700, w.f):
        ffn.set_hot_neurons(n_hot)
        for t in range(X.shape[0]):
            counts = torch.zeros(w.n_layers, dtype=torch.int32, device="cuda")
            idx_out = torch.zeros((w.n_layers, w.f), dtype=torch.int32, device="cuda")
            P.pi_profile_begin(ffn.h)
            xo = ffn.decode_stack(to_dev(X[t]), counts=counts, idx_out=idx_out)
            prof = P.pi_profile_end(ffn.h)
            assert prof["decode_stack"][1] == 1, prof
            assert torch.equal(xo, ref[t][0]), (n_hot, t)
            assert torch.equal(counts, ref[t][1]) and torch.equal(idx_out, ref[t][2]), (n_hot, t)
    with pytest.raises(P.PiError):
        ffn.set_hot_neurons(w.f + 1)
    assert ffn.status() == 0
    ffn.close()


def _with_env(name, value, fn):
    import os

    old = os.environ.get(name)
    os.environ[name] = value
    try:
        return fn()
    finally:
        if old is None:
            del os.environ[name]
        else:
            os.environ[name] = old


# d 1024 with f 30000 and r 1024: ~198 owned P2 rows of 2 KB per CTA, more than the ring holds
P2_WIDE_SHAPE = dict(d=1024, f=30000, r=1024)


@pytest.mark.parametrize("wi,shape", [(wi, STACK_SHAPE) for wi in range(5)] + [(1, P2_WIDE_SHAPE), (3, P2_WIDE_SHAPE)])
def test_decode_stack_p2_staging_bit_identical(P, wi, shape):
    """Copying the next layer's owned P2 rows into shared memory ahead of their logits (all of
    them, or the first ones when they do not all fit) changes nothing in the output bits: the
    logits read the same values in the same order from either place (CUDA-core logits at
    r = 136, tensor-core logits at r = 1024)."""
    w = _wl(wi, shape, n_layers=3)
    layers = build_layers(w, range(w.n_layers))
    X = make_inputs(w, 2, 1, seed=13, device="cpu").numpy()
    staged = _handle(P, w, [g for g, _ in layers], stack_kernel=True)
    plain = _with_env("PI_FFN_STACK_P2", "0", lambda: _handle(P, w, [g for g, _ in layers], stack_kernel=True))
    for H in (0, 700):
        for ffn in (staged, plain):
            ffn.set_hot_prefix(H)
        for t in range(X.shape[0]):
            outs = []
            for ffn in (staged, plain):
                counts = torch.zeros(w.n_layers, dtype=torch.int32, device="cuda")
                idx_out = torch.zeros((w.n_layers, w.f), dtype=torch.int32, device="cuda")
                P.pi_profile_begin(ffn.h)
                xo = ffn.decode_stack(to_dev(X[t]), counts=counts, idx_out=idx_out)
                prof = P.pi_profile_end(ffn.h)
                assert prof["decode_stack"][1] == 1, prof
                outs.append((xo.clone(), counts.clone(), idx_out.clone()))
            assert torch.equal(outs[0][0], outs[1][0]), (H, t)
            assert torch.equal(outs[0][1], outs[1][1]) and torch.equal(outs[0][2], outs[1][2]), (H, t)
            if H:
                cg, ig = outs[0][1].cpu().numpy(), outs[0][2].cpu().numpy()
                for l in range(w.n_layers):
                    assert np.array_equal(ig[l, :H], np.arange(H)), l
        # and the staged kernel against the oracle, layer by layer
        _stack_vs_oracle(P, w, layers, X, staged, ("staged", wi, H), hot_prefix=H)
    for ffn in (staged, plain):
        assert ffn.status() == 0
        ffn.close()


@pytest.mark.parametrize("pf", ["0", "3", "9"])
def test_decode_stack_prefetch_bits(P, pf):
    """The L2 prefetches (P1 and P2 a layer ahead, the streamed P2 rows during the FFN, none) are
    hints: the output bits are those of the default setting."""
    w = _wl(3, P2_WIDE_SHAPE, n_layers=3)
    layers = build_layers(w, range(w.n_layers))
    X = make_inputs(w, 2, 1, seed=17, device="cpu").numpy()
    ref = _handle(P, w, [g for g, _ in layers], stack_kernel=True)
    alt = _with_env("PI_FFN_STACK_PF", pf, lambda: _handle(P, w, [g for g, _ in layers], stack_kernel=True))
    for t in range(X.shape[0]):
        a = ref.decode_stack(to_dev(X[t])).clone()
        b = alt.decode_stack(to_dev(X[t])).clone()
        torch.cuda.synchronize()
        assert torch.equal(a, b), (pf, t)
    for ffn in (ref, alt):
        assert ffn.status() == 0
        ffn.close()


# ------------------------------------------------------------------ hot-prefix variant --------

def _check_list(gi, pr, H):
    assert np.all(np.diff(gi) > 0)
    assert np.array_equal(gi[: min(H, gi.size)], np.arange(min(H, gi.size)))
    diff = np.setxor1d(gi, pr["idx"])
    assert np.all(band_mask(pr["z"])[diff]), f"{diff.size} out-of-band mismatches"


@pytest.mark.parametrize("wi", range(5))
def test_hot_prefix_predict_and_stack(P, wi):
    """Neurons [0, H) active without a logit: pi_predict (batch 1 and 4) and both batch-1 stack
    paths against the oracle's hot-prefix mode."""
    w = _wl(wi, STACK_SHAPE, n_layers=2)
    layers = build_layers(w, range(w.n_layers))
    Lo0 = layers[0][1]
    X = make_inputs(w, 2, 1, seed=17, device="cpu").numpy()
    for H in (200, 1500, w.f):
        for B in (1, 4):
            ffn = P.SparseFFN.from_workload(w, [g for g, _ in layers], max_batch=B)
            ffn.set_hot_prefix(H)
            u = rms_inputs(w, B, seed=H)[0]
            idx, cnt = ffn.predict(0, to_dev(u))
            torch.cuda.synchronize()
            gi = idx[: int(cnt.item())].cpu().numpy()
            pr = oracle.predict(u.astype(np.float64), Lo0["p1_t"], Lo0["p2_t"], Lo0["b_pred"], w.pdtype, hot_prefix=H)
            _check_list(gi, pr, H)
            assert ffn.status() == 0
            ffn.close()
        for stack_kernel in (True, False):
            ffn = _handle(P, w, [g for g, _ in layers], stack_kernel)
            ffn.set_hot_prefix(H)
            _stack_vs_oracle(P, w, layers, X, ffn, (stack_kernel, H), hot_prefix=H)
            assert ffn.status() == 0
            ffn.close()
    ffn = P.SparseFFN.from_workload(w, [g for g, _ in layers], max_batch=1)
    with pytest.raises(P.PiError):
        ffn.set_hot_prefix(w.f + 1)
    ffn.close()
