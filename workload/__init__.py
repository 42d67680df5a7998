"""Seeded synthetic workloads shared by the CUDA path's tests/bench and the oracle.

This module draws inputs only. It holds none of the sparse-FFN method's
arithmetic (no predictor, no mask, no FFN): it produces weights rounded to their
stored type, calibrated biases, per-neuron activation frequencies, profiling
counts and decode-step inputs. Both sides receive the same arrays.
"""
from .gen import (  # noqa: F401
    WORKLOADS,
    Workload,
    activation_probs,
    make_inputs,
    make_layer,
    scaled,
    workload_by_name,
)
