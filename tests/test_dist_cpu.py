"""Multi-process host logic of bench.py on CPU (gloo, world size 2).

Each rank decodes its own token stream (independent sequences: the path shards
by sequence with no data-path collective). The only exchange is the job-level
timing: the max of the ranks' timed regions and the sum of their tokens.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    r, lr, ws = bench.dist_env()
    assert (r, lr, ws) == (rank, rank, world)
    ms, tokens = bench.aggregate(10.0 + 5.0 * rank, 100 * (rank + 1), world)
    bench.barrier(world)
    out[rank] = (ms, tokens)
    dist.destroy_process_group()


def test_aggregate_two_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        ms, tokens = res[rank]
        assert ms == pytest.approx(15.0)   # slowest rank bounds the job
        assert tokens == 300               # every rank's tokens count


def test_aggregate_single_process_is_identity():
    import bench

    assert bench.aggregate(12.5, 7, 1) == (12.5, 7)


def test_step_bytes_accounting():
    """Algorithmic bytes: dense predictor + per active neuron its rows (and int4 scales)."""
    import bench
    from workload import WORKLOADS

    w = WORKLOADS["relullama7b_d4096_f11008_bf16_L32"]
    pred = 1024 * 4096 * 2 + 11008 * 1024 * 2 + 11008 * 4
    assert bench.predictor_bytes(w) == pred
    assert bench.neuron_bytes(w) == 3 * 4096 * 2 + 4
    assert bench.step_bytes(w, [1000, 2000]) == 2 * pred + 3000 * (3 * 4096 * 2 + 4)
    w5 = WORKLOADS["opt175b_d12288_f49152_int4_L96"]
    assert bench.neuron_bytes(w5) == 2 * 12288 // 2 + 4 + 2 * (12288 // 128) * 2
    assert bench.kernel_bytes(w5, "pred_logits", 0, 1) == 49152 * 1024 * 2 + 49152 * 4
    # the one-launch predictor reads both predictor matrices (and the bias); the hot prefix's
    # P2 rows are not read
    assert bench.kernel_bytes(w, "pred_fused", 0, 4) == pred
    assert bench.kernel_bytes(w, "pred_fused", 0, 4, hot=100) == pred - 100 * 1024 * 2


def test_ncu_traffic_only_for_the_captured_configuration():
    """The recorded DRAM traffic is reported only for the captured configuration: the
    workload's own shape at batch 1, no hot prefix or hot slots, the captured sources;
    it scales with the layer count."""
    import dataclasses

    import bench
    from workload import WORKLOADS

    name = "opt175b_d12288_f49152_int4_L96"
    w = WORKLOADS[name]
    rec = bench.NCU_TRAFFIC[(name, "decode_stack")]
    if rec["csrc"] == bench.csrc_hash("decode_stack"):
        assert bench.ncu_traffic(w, "decode_stack") == pytest.approx(rec["bytes_per_layer"] * 96)
        assert bench.ncu_traffic(dataclasses.replace(w, n_layers=4), "decode_stack") == pytest.approx(
            rec["bytes_per_layer"] * 4)
    else:   # sources changed since the capture: no traffic figure
        assert bench.ncu_traffic(w, "decode_stack") is None
    assert bench.ncu_traffic(dataclasses.replace(w, r=128), "decode_stack") is None
    assert bench.ncu_traffic(w, "decode_stack", B=4) is None
    assert bench.ncu_traffic(w, "decode_stack", hot_prefix=100) is None
    assert bench.ncu_traffic(w, "decode_stack", n_hot=100) is None
    assert bench.ncu_traffic(w, "ffn_down") is None
    assert bench.ncu_traffic(WORKLOADS["llama2_13b_d5120_f13824_bf16_L40"], "decode_stack") is None
