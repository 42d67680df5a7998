"""The C-ABI library builds, loads without a GPU, exports every declared symbol,
and rejects bad descriptors on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

from tests.conftest import ROOT


@pytest.fixture(scope="module")
def P():
    import __graft_entry__

    __graft_entry__.build()
    import activation_sparse_decode_pi_gb300 as P

    return P


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(pi_[a-z0-9_]+)\s*\(", src))
    return names


def test_exports_every_declared_symbol(P):
    decl = declared_symbols()
    assert decl, "no declarations found"
    for name in decl:
        assert hasattr(P._lib, name), name
    assert decl == set(P.EXPORTS)


def test_abi_version_and_strings(P):
    assert P.pi_abi_version() == 1
    for code in range(7):
        assert P.pi_status_string(code) and P.pi_status_string(code) != "unknown status"
    assert P.pi_status_string(99) == "unknown status"


def _create(P, desc, layers=None):
    h = ctypes.c_void_p()
    rc = P._lib.pi_ffn_create(ctypes.byref(h), ctypes.byref(desc), layers)
    return rc, h.value


@pytest.mark.parametrize("fields,code", [
    (dict(d=500), 1),            # d % 8
    (dict(d=0), 1),
    (dict(f=0), 1),
    (dict(r=12), 1),             # r % 8
    (dict(n_layers=0), 1),
    (dict(max_batch=0), 1),
    (dict(max_batch=257), 1),
    (dict(kind=2), 1),
    (dict(wdtype=4), 1),
    (dict(pdtype=3), 1),         # int4 predictor not offered
    (dict(tau_logit=float("nan")), 1),
    (dict(wdtype=3, d=576), 2),  # int4 needs d % 128 == 0
    (dict(d=32768), 2),          # one staged row above the shared-memory budget
])
def test_descriptor_validation(P, fields, code):
    base = dict(d=512, f=2048, r=64, n_layers=1, max_batch=1, kind=0, wdtype=0, pdtype=0, tau_logit=0.0)
    base.update(fields)
    rc, h = _create(P, P.PiFfnDesc(**base))
    assert rc == code and h is None


def test_null_arguments(P):
    desc = P.PiFfnDesc(512, 2048, 64, 1, 1, 0, 0, 0, 0.0)
    assert P._lib.pi_ffn_create(None, ctypes.byref(desc), None) == 1
    rc, h = _create(P, desc, None)       # valid descriptor, no layer array
    assert rc == 1 and h is None
    assert P._lib.pi_predict(None, 0, None, 1, None, None, None) == 1
    assert P._lib.pi_sparse_ffn(None, 0, None, 1, None, None, None, None) == 1
    assert P._lib.pi_decode_stack(None, None, 1, None, None, None, None) == 1
    assert P._lib.pi_get_status(None) == 1
    assert P._lib.pi_hot_first_order(None, -1, None, None) == 1
    assert P._lib.pi_hot_first_order(None, 0, None, None) == 0          # empty order is a no-op
    assert P._lib.pi_permute_rows(None, None, None, -1, 16, None, None) == 1
    P._lib.pi_ffn_destroy(None)                                          # no-op


def test_injected_descriptor_fault(P):
    """PI_FAULT=badarg makes descriptor validation fail on the host: INVALID_ARG, no handle."""
    desc = P.PiFfnDesc(512, 2048, 64, 1, 1, 0, 0, 0, 0.0)
    os.environ["PI_FAULT"] = "badarg"
    try:
        rc, h = _create(P, desc, None)
    finally:
        del os.environ["PI_FAULT"]
    assert rc == 1 and h is None
    os.environ["PI_FAULT"] = "none-of-these"     # an unknown value injects nothing
    try:
        rc, h = _create(P, P.PiFfnDesc(500, 2048, 64, 1, 1, 0, 0, 0, 0.0), None)
    finally:
        del os.environ["PI_FAULT"]
    assert rc == 1 and h is None                 # the real validation (d % 8) still runs
