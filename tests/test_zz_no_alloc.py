"""pi_sparse_ffn_noalloc: the sparse FFN for callers that cannot allocate device memory.

Such callers (code inside an allocator callback, a plugin whose host process
owns all device memory) cannot create a handle, since pi_ffn_create allocates.
The entry point keeps its scratch in a static device array of the library.
This file is collected last so that, if it fails, a run stopping at the first
failure has already run every other test; it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_cases import TOL, build_layers, rel_l2, rms_inputs, to_dev
from workload import WORKLOADS, scaled

pytestmark = pytest.mark.gpu

SHAPE = dict(d=1024, f=2752, r=128, n_layers=1)
CASES = [("relullama7b_d4096_f11008_bf16_L32", 1), ("relullama7b_d4096_f11008_bf16_L32", 2),
         ("relullama7b_d4096_f11008_bf16_L32", 3), ("opt175b_d12288_f49152_int4_L96", 1),
         ("opt175b_d12288_f49152_int4_L96", 3)]


@pytest.fixture(scope="module")
def P():
    import activation_sparse_decode_pi_gb300 as P

    return P


def _setup(P, name, B):
    w = scaled(WORKLOADS[name], **SHAPE)
    (Lg, Lo), = build_layers(w, [0])
    ffn = P.SparseFFN.from_workload(w, [Lg], max_batch=B)
    desc = P.PiFfnDesc(w.d, w.f, w.r, 1, B, P.KINDS[w.kind], P.DTYPES[w.wdtype], P.DTYPES[w.pdtype], 0.0)
    return w, Lg, Lo, ffn, desc, P.layer_weights(Lg)


@pytest.mark.parametrize("name,B", CASES, ids=[f"{n.split('_')[0]}-b{b}" for n, b in CASES])
def test_noalloc_matches_sparse_ffn_twice(P, name, B):
    """Two calls in a row (sharing the scratch) agree with pi_sparse_ffn and with the oracle."""
    w, Lg, Lo, ffn, desc, lw = _setup(P, name, B)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    us = rms_inputs(w, B, tokens=2, seed=7)
    for call in range(2):
        ud = to_dev(us[call])
        idx, cnt = ffn.predict(0, ud)
        y_ref = ffn.sparse_ffn(0, ud, idx, cnt)
        y = torch.full_like(ud, float("nan"))
        P.pi_sparse_ffn_noalloc(desc, lw, ud, B, idx, cnt, y, status)
        torch.cuda.synchronize()
        assert rel_l2(y.cpu().numpy(), y_ref.cpu().numpy()) <= TOL[w.wdtype]
        n = int(cnt.item())
        _, yo = oracle.sparse_ffn(us[call].astype(np.float64), Lo, idx[:n].cpu().numpy(), w.kind, w.wdtype)
        assert rel_l2(y.cpu().numpy(), yo) <= TOL[w.wdtype]
    assert int(status.item()) == 0
    ffn.close()


def test_noalloc_count_above_f_is_flagged(P):
    """A count above f is clamped on the device and reported in the status word."""
    w, Lg, Lo, ffn, desc, lw = _setup(P, "opt175b_d12288_f49152_int4_L96", 2)
    u = rms_inputs(w, 2, seed=3)[0]
    ud = to_dev(u)
    idx = torch.arange(w.f, dtype=torch.int32, device="cuda")
    cnt = torch.tensor([w.f + 50], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = torch.full_like(ud, float("nan"))
    P.pi_sparse_ffn_noalloc(desc, lw, ud, 2, idx, cnt, y, status)
    torch.cuda.synchronize()
    assert int(status.item()) == P.PI_ERR_DEVICE_CHECK
    yd = oracle.dense_ffn(u.astype(np.float64), Lo, w.kind, w.wdtype)
    assert rel_l2(y.cpu().numpy(), yd) <= TOL[w.wdtype]
    ffn.close()


def test_noalloc_rejects_a_short_output(P):
    """An output whose B*d floats would run past the end of its allocation is rejected on the host."""
    w, Lg, Lo, ffn, desc, lw = _setup(P, "relullama7b_d4096_f11008_bf16_L32", 2)
    ud = to_dev(rms_inputs(w, 2)[0])
    idx, cnt = ffn.predict(0, ud)
    torch.cuda.synchronize()
    big = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    seg = [s for s in torch.cuda.memory_snapshot()
           if s["address"] <= big.data_ptr() < s["address"] + s["total_size"]][0]
    end = seg["address"] + seg["total_size"]
    short_y = end - 2 * w.d * 4 + 16                          # 16 bytes short of B*d floats
    with pytest.raises(P.PiError) as e:
        P.pi_sparse_ffn_noalloc(desc, lw, ud, 2, idx, cnt, short_y)
    assert e.value.code == P.PI_ERR_INVALID_ARG
    with pytest.raises(P.PiError) as e:                       # and a short input likewise
        P.pi_sparse_ffn_noalloc(desc, lw, short_y, 2, idx, cnt, ud)
    assert e.value.code == P.PI_ERR_INVALID_ARG
    ffn.close()


def test_noalloc_rejects_sizes_beyond_its_scratch(P):
    w = WORKLOADS["opt30b_d7168_f28672_fp16_L48"]
    B = 32                                                    # 256 * 32 * 7168 * 4 bytes of partials > 16 MiB
    desc = P.PiFfnDesc(w.d, w.f, w.r, 1, B, P.KINDS[w.kind], P.DTYPES[w.wdtype], P.DTYPES[w.pdtype], 0.0)
    lw = P.PiLayerWeights()
    with pytest.raises(P.PiError) as e:
        P.pi_sparse_ffn_noalloc(desc, lw, 0, B, 0, 0, 0)
    assert e.value.code == P.PI_ERR_UNSUPPORTED
