"""Parity of the decode step at the workloads' full d, f and r, on the kernels the benchmark
times for each batch size, checked layer by layer against the oracle (teacher-forced: layer l
of the oracle runs on the GPU's own x_l, so every layer is compared).

* batch 1 runs the persistent one-kernel step: Llama2-13B-shaped (d 5120, two 16-byte
  column chunks per thread), OPT-30B-shaped (fp16, non-gated, d 7168; only part of each
  CTA's P2 rows fit in shared memory), OPT-175B-shaped (int4 group-128, d 12288; part of
  the P2 rows staged);
* batch 2 runs the CUDA-core kernel chain, batches 4, 16 and 32 the tensor-core kernels
  (their lower batch bound is 3 at these row lengths).
A few layers of each stack are enough: every layer has the same shape and law.
"""
import dataclasses

import numpy as np
import pytest
import torch

from tests.gpu_cases import build_layers, teacher_forced, to_dev
from workload import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

CASES = [
    ("llama2_13b_d5120_f13824_bf16_L40", 1, 3),
    ("opt30b_d7168_f28672_fp16_L48", 1, 3),
    ("opt175b_d12288_f49152_int4_L96", 1, 3),
    ("llama2_13b_d5120_f13824_bf16_L40", 2, 2),
    ("llama2_13b_d5120_f13824_bf16_L40", 4, 2),
    ("llama2_13b_d5120_f13824_bf16_L40", 16, 2),
    ("opt30b_d7168_f28672_fp16_L48", 32, 2),
]


@pytest.fixture(scope="module")
def P():
    import activation_sparse_decode_pi_gb300 as P

    return P


@pytest.mark.parametrize("name,B,n_layers", CASES, ids=[f"{n.split('_')[0]}-b{b}" for n, b, _ in CASES])
def test_stack_full_size_teacher_forced(P, name, B, n_layers):
    w = dataclasses.replace(WORKLOADS[name], n_layers=n_layers)
    layers = build_layers(w, range(n_layers))
    ffn = P.SparseFFN.from_workload(w, [g for g, _ in layers], max_batch=B)
    X = make_inputs(w, 2, B, seed=4242, device="cpu").numpy()
    P.pi_profile_begin(ffn.h)
    ffn.decode_stack(to_dev(X[0]))
    prof = P.pi_profile_end(ffn.h)
    if B == 1:
        assert prof["decode_stack"][1] == 1 and prof["ffn_h"][1] == 0, prof   # the persistent kernel ran
    else:
        assert prof["decode_stack"][1] == 0 and prof["ffn_h"][1] == n_layers, prof
        # the chain normalises once per step, the tensor-core path splits each layer's input
        assert prof["rms"][1] == (1 if B == 2 else n_layers), prof
    flips = 0
    for t in range(X.shape[0]):
        xo = ffn.decode_stack(to_dev(X[t])).clone()
        xt, fl = teacher_forced(P, w, layers, ffn, X[t], tag=(name, B, t))
        assert np.array_equal(xt, xo.cpu().numpy()), (name, B, t, "layer-output call differs")
        flips += fl
    assert ffn.status() == 0
    ffn.close()
    del layers
    torch.cuda.empty_cache()
