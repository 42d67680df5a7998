"""Host-side fault injection (PI_FAULT): pi_ffn_create's failure paths on a real device.

alloc: the workspace allocation fails (PI_ERR_OOM, nothing allocated); upload: a step after
the workspace exists fails (PI_ERR_CUDA) and the workspace is freed again. In both cases the
handle is NULL and the device's free memory is what it was before the call.
"""
import ctypes
import os

import pytest
import torch

from tests.gpu_cases import build_layers
from workload import WORKLOADS, scaled

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fault,code", [("alloc", 4), ("upload", 3)])
def test_create_failure_paths(fault, code):
    import activation_sparse_decode_pi_gb300 as P

    w = scaled(WORKLOADS["relullama7b_d4096_f11008_bf16_L32"], d=1024, f=2752, r=128, n_layers=1)
    (Lg, _), = build_layers(w, [0])
    desc = P.PiFfnDesc(w.d, w.f, w.r, 1, 4, P.KINDS[w.kind], P.DTYPES[w.wdtype], P.DTYPES[w.pdtype], 0.0)
    arr = (P.PiLayerWeights * 1)(P.layer_weights(Lg))
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    os.environ["PI_FAULT"] = fault
    try:
        h = ctypes.c_void_p(12345)
        rc = P._lib.pi_ffn_create(ctypes.byref(h), ctypes.byref(desc), arr)
    finally:
        del os.environ["PI_FAULT"]
    assert rc == code and h.value is None
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    # without the fault the same arguments create a handle
    ffn = P.SparseFFN.from_workload(w, [Lg], max_batch=4)
    assert ffn.h
    ffn.close()
