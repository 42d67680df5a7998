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


@pytest.fixture(scope="module")
def P():
    import activation_sparse_decode_pi_gb300 as P

    return P


def test_noalloc_matches_sparse_ffn_twice(P):
    w = scaled(WORKLOADS["relullama7b_d4096_f11008_bf16_L32"], d=1024, f=2752, r=128, n_layers=1)
    (Lg, Lo), = build_layers(w, [0])
    B = 2
    ffn = P.SparseFFN.from_workload(w, [Lg], max_batch=B)
    desc = P.PiFfnDesc(w.d, w.f, w.r, 1, B, P.KINDS[w.kind], P.DTYPES[w.wdtype], P.DTYPES[w.pdtype], 0.0)
    lw = P.layer_weights(Lg)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    us = rms_inputs(w, B, tokens=2, seed=7)
    for call in range(2):                                     # two calls in a row share the scratch
        ud = to_dev(us[call])
        idx, cnt = ffn.predict(0, ud)
        y_ref = ffn.sparse_ffn(0, ud, idx, cnt)
        y = torch.full_like(ud, float("nan"))
        P.pi_sparse_ffn_noalloc(desc, lw, ud, B, idx, cnt, y, status)
        torch.cuda.synchronize()
        assert rel_l2(y.cpu().numpy(), y_ref.cpu().numpy()) <= TOL[w.wdtype]
        # and both agree with the oracle on the same list
        n = int(cnt.item())
        _, yo = oracle.sparse_ffn(us[call].astype(np.float64), Lo, idx[:n].cpu().numpy(), w.kind, w.wdtype)
        assert rel_l2(y.cpu().numpy(), yo) <= TOL[w.wdtype]
    assert int(status.item()) == 0
    ffn.close()


def test_noalloc_rejects_sizes_beyond_its_scratch(P):
    w = WORKLOADS["opt30b_d7168_f28672_fp16_L48"]
    B = 32                                                    # 256 * 32 * 7168 * 4 bytes of partials > 16 MiB
    desc = P.PiFfnDesc(w.d, w.f, w.r, 1, B, P.KINDS[w.kind], P.DTYPES[w.wdtype], P.DTYPES[w.pdtype], 0.0)
    lw = P.PiLayerWeights()
    with pytest.raises(P.PiError) as e:
        P.pi_sparse_ffn_noalloc(desc, lw, 0, B, 0, 0, 0)
    assert e.value.code == P.PI_ERR_UNSUPPORTED
