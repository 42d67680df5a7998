"""CPU fp64 oracle for PowerInfer-style activation-sparse FFN decode.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg import this package. It shares no code with the
CUDA library (``activation_sparse_decode_pi_gb300``) and never imports it.

The arithmetic lives in ``oracle.c`` (plain C, double precision, fixed-order
sums); this module only marshals numpy arrays and chains layers.

Steps, as the pages give them ("PowerInfer" paper walk-through page):
  * predictor (section "activation predictor", eq.  a = sigmoid(x Wp + b_p),
    active if a_i > tau), read as z = ReLU(u P1) P2 + b_p, active iff z > 0,
    union over batch rows                                   -> ``predict``
  * FFN (section "technical details", eq. FFN(x) = sigma(x W1) (.) (x W2) W3),
    sigma = ReLU, restricted to the active neurons          -> ``sparse_ffn``
    and the unrestricted definition                         -> ``dense_ffn``
  * offline profiling (code block): count-descending order, stable
                                                            -> ``hot_first_order``
  * layers chained by a parameter-free RMS pre-norm residual (the pages are
    silent about non-FFN layers; this is the reading used)  -> ``stack``
  * hot prefix (walk-through page, hot/cold neurons: a small set fires on most
    inputs; summary page, Methodology): with ``hot_prefix = H`` the neurons
    [0, H) of the hot-first order are active on every token and the
    predictor decides only [H, f)                           -> ``predict``
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build_oracle

DT = {"f32": 0, "bf16": 1, "f16": 2, "int4g128": 3}
KIND = {"gated": 0, "relu": 1}
RMS_EPS = 1e-6
BAND = 1e-4  # logits this close to the threshold may go either way

_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def lib():
    global _lib
    if _lib is None:
        path = build_oracle.build()
        L = ctypes.CDLL(path)
        L.orc_widen.argtypes = [_P, _P, ctypes.c_int, _I64, _P]
        L.orc_threads.restype = ctypes.c_int
        L.orc_predict.restype = _I64
        L.orc_predict.argtypes = [_P, ctypes.c_int, _I64, _I64, _I64, ctypes.c_int, _P, _P, _P,
                                  ctypes.c_double, _P, _P, _P, _P]
        L.orc_sparse_ffn.restype = ctypes.c_int
        L.orc_sparse_ffn.argtypes = [_P, ctypes.c_int, _I64, _I64, ctypes.c_int, ctypes.c_int,
                                     _P, _P, _P, _P, _P, _P, _P, _P, _I64, _P, _P]
        L.orc_dense_ffn.argtypes = [_P, ctypes.c_int, _I64, _I64, ctypes.c_int, ctypes.c_int,
                                    _P, _P, _P, _P, _P, _P, _P, _P]
        L.orc_rms_norm.argtypes = [_P, ctypes.c_int, _I64, ctypes.c_double, _P]
        L.orc_hot_first_order.argtypes = [_P, _I64, _P]
        _lib = L
    return _lib


def threads() -> int:
    return lib().orc_threads()


def raw(a):
    """Stored bits of a torch tensor or numpy array as a C-contiguous numpy array
    (bf16/f16 as uint16, int4 packed bytes as uint8, f32 as float32)."""
    if a is None:
        return None
    if not isinstance(a, np.ndarray):
        import torch

        t = a.detach().to("cpu").contiguous()
        if t.dtype in (torch.bfloat16, torch.float16):
            return t.view(torch.int16).numpy().view(np.uint16).copy()
        return t.numpy().copy()
    if a.dtype == np.float16:
        return np.ascontiguousarray(a).view(np.uint16)
    return np.ascontiguousarray(a)


def _ptr(a):
    return None if a is None else a.ctypes.data


def layer_numpy(layer: dict) -> dict:
    """A generator layer (torch tensors, any device) as raw numpy arrays."""
    return {k: (raw(v) if k != "p" else (None if v is None else np.asarray(v.cpu() if hasattr(v, "cpu") else v)))
            for k, v in layer.items()}


def widen(a, dtype: str, scales=None) -> np.ndarray:
    """Stored values of a 1-D array of `dtype` widened to float64 by the oracle."""
    a = raw(a)
    n = a.size * 2 if dtype == "int4g128" else a.size
    s = raw(scales)
    out = np.empty(n, np.float64)
    lib().orc_widen(_ptr(a), _ptr(s), DT[dtype], n, _ptr(out))
    return out


def _u64(u) -> np.ndarray:
    u = np.ascontiguousarray(np.asarray(u, dtype=np.float64))
    return u.reshape(1, -1) if u.ndim == 1 else u


def predict(u, p1_t, p2_t, b_pred, pdtype: str, tau: float = 0.0, hot_prefix: int = 0) -> dict:
    """Predictor hidden layer, logits, union mask and ascending active indices.

    hot_prefix = H > 0: neurons [0, H) are active without a predictor decision; their
    entries of z are returned as +inf (no logit decides them, so none lies in a band).
    """
    u = _u64(u)
    B, d = u.shape
    p1, p2 = raw(p1_t), raw(p2_t)
    r, f = p1.shape[0], p2.shape[0]
    assert p1.shape[1] == d and p2.shape[1] == r
    bp = None if b_pred is None else np.ascontiguousarray(np.asarray(raw(b_pred), np.float32))
    hp = np.empty((B, r), np.float64)
    z = np.empty((B, f), np.float64)
    mask = np.empty(f, np.uint8)
    idx = np.empty(f, np.int32)
    n = lib().orc_predict(_ptr(u), B, d, r, f, DT[pdtype], _ptr(p1), _ptr(p2), _ptr(bp), tau,
                          _ptr(hp), _ptr(z), _ptr(mask), _ptr(idx))
    mask = mask.astype(bool)
    idx = idx[:n].copy()
    if hot_prefix > 0:
        H = min(int(hot_prefix), f)
        mask[:H] = True
        z[:, :H] = np.inf
        idx = np.flatnonzero(mask).astype(np.int32)
        n = idx.size
    return {"hp": hp, "z": z, "mask": mask, "idx": idx, "count": int(n)}


def _ffn_args(layer: dict):
    g = lambda k: raw(layer.get(k))
    bg = layer.get("b_gate")
    bg = None if bg is None else np.ascontiguousarray(np.asarray(raw(bg), np.float32))
    return g("w_gate"), g("w_up"), g("w_down_t"), g("s_gate"), g("s_up"), g("s_down"), bg


def sparse_ffn(u, layer: dict, idx, kind: str, wdtype: str, d: int | None = None):
    """h[b, j] and y[b, :] over the listed neurons (any order is accepted; sums follow the list)."""
    u = _u64(u)
    B, du = u.shape
    wg, wu, wd, sg, su, sd, bg = _ffn_args(layer)
    f = wg.shape[0]
    idx = np.ascontiguousarray(np.asarray(idx, np.int32))
    n = idx.size
    h = np.empty((B, max(n, 1)), np.float64)
    y = np.empty((B, du), np.float64)
    rc = lib().orc_sparse_ffn(_ptr(u), B, du, f, KIND[kind], DT[wdtype], _ptr(wg), _ptr(wu), _ptr(wd),
                              _ptr(sg), _ptr(su), _ptr(sd), _ptr(bg), _ptr(idx), n, _ptr(h), _ptr(y))
    if rc != 0:
        raise IndexError("active index out of range")
    return h[:, :n], y


def dense_ffn(u, layer: dict, kind: str, wdtype: str):
    """The FFN definition over every neuron (no predictor, no mask)."""
    u = _u64(u)
    B, d = u.shape
    wg, wu, wd, sg, su, sd, bg = _ffn_args(layer)
    y = np.empty((B, d), np.float64)
    lib().orc_dense_ffn(_ptr(u), B, d, wg.shape[0], KIND[kind], DT[wdtype], _ptr(wg), _ptr(wu), _ptr(wd),
                        _ptr(sg), _ptr(su), _ptr(sd), _ptr(bg), _ptr(y))
    return y


def rms_norm(x, eps: float = RMS_EPS):
    x = _u64(x)
    u = np.empty_like(x)
    lib().orc_rms_norm(_ptr(x), x.shape[0], x.shape[1], eps, _ptr(u))
    return u


def hot_first_order(counts) -> np.ndarray:
    """perm[k] = neuron placed at position k: counts descending, ties by original index."""
    c = np.ascontiguousarray(np.asarray(counts).astype(np.uint32))
    perm = np.empty(c.size, np.int32)
    lib().orc_hot_first_order(_ptr(c), c.size, _ptr(perm))
    return perm


def layer_forward(u, layer: dict, kind: str, wdtype: str, pdtype: str, tau: float = 0.0,
                  hot_prefix: int = 0) -> dict:
    """One layer: predict on u, then the sparse FFN over the predicted set."""
    pr = predict(u, layer["p1_t"], layer["p2_t"], layer.get("b_pred"), pdtype, tau, hot_prefix)
    h, y = sparse_ffn(u, layer, pr["idx"], kind, wdtype)
    pr["h"], pr["y"] = h, y
    pr["zmin"] = np.abs(pr["z"]).min(axis=0) if pr["z"].size else np.zeros(0)
    return pr


def stack(x0, layers, kind: str, wdtype: str, pdtype: str, tau: float = 0.0, eps: float = RMS_EPS,
          keep: bool = False, hot_prefix: int = 0) -> dict:
    """x_{l+1} = x_l + FFN_l(u_l), u_l = rms_norm(x_l); returns x_L and per-layer traces.

    `layers` is a sequence of layer dicts or a callable layer_index -> layer dict.
    """
    x = _u64(x0).copy()
    nl = len(layers) if not callable(layers) else None
    get = layers if callable(layers) else (lambda i: layers[i])
    trace = {"idx": [], "count": [], "zmin": [], "u": [], "y": []}
    i = 0
    while nl is None or i < nl:
        try:
            layer = get(i)
        except IndexError:
            break
        if layer is None:
            break
        u = rms_norm(x, eps)
        out = layer_forward(u, layer, kind, wdtype, pdtype, tau, hot_prefix)
        trace["idx"].append(out["idx"])
        trace["count"].append(out["count"])
        trace["zmin"].append(out["zmin"])
        if keep:
            trace["u"].append(u)
            trace["y"].append(out["y"])
        x = x + out["y"]
        i += 1
    trace["x_out"] = x
    return trace
