"""NumPy brute force for tiny shapes: the method written as dense matrix algebra.

Independent of the C oracle and of the CUDA library: stored values are widened
with numpy's own float16 conversion, bit shifts for bfloat16 and nibble masks
for int4, then the whole layer is a handful of float64 matrix products:

  HP = ReLU(U P1T^T);  Z = HP P2T^T + b_p;  M = any_b(Z > tau)
  gated:     H = ReLU(U Wg^T + bg) * (U Wu^T)       non-gated: H = ReLU(U W1^T + b1)
  Y = (H * M) WdT
"""
import numpy as np


def widen(a, dtype, scales=None):
    a = np.asarray(a)
    if dtype == "f32":
        return a.astype(np.float64)
    if dtype == "f16":
        return a.view(np.float16).astype(np.float64)
    if dtype == "bf16":
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if dtype == "int4g128":
        lo = (a & 0x0F).astype(np.int16)
        hi = (a >> 4).astype(np.int16)
        lo = np.where(lo > 7, lo - 16, lo)
        hi = np.where(hi > 7, hi - 16, hi)
        q = np.stack([lo, hi], axis=-1).reshape(a.shape[0], -1).astype(np.float64)
        s = np.asarray(scales).view(np.float16).astype(np.float64)
        return q * np.repeat(s, 128, axis=1)
    raise ValueError(dtype)


def predictor(U, p1t, p2t, bp, pdtype, tau=0.0):
    P1 = widen(p1t, pdtype)
    P2 = widen(p2t, pdtype)
    HP = np.maximum(U @ P1.T, 0.0)
    Z = HP @ P2.T + (0.0 if bp is None else np.asarray(bp, np.float64))
    M = (Z > tau).any(axis=0)
    return HP, Z, M


def ffn_masked(U, layer, M, kind, wdtype):
    Wg = widen(layer["w_gate"], wdtype, layer.get("s_gate"))
    Wd = widen(layer["w_down_t"], wdtype, layer.get("s_down"))
    bg = layer.get("b_gate")
    G = U @ Wg.T + (0.0 if bg is None else np.asarray(bg, np.float64))
    if kind == "gated":
        Wu = widen(layer["w_up"], wdtype, layer.get("s_up"))
        H = np.maximum(G, 0.0) * (U @ Wu.T)
    else:
        H = np.maximum(G, 0.0)
    return (H * np.asarray(M, np.float64)) @ Wd, H


def true_set(U, layer, wdtype):
    """Neurons whose gate pre-activation is positive for some batch row."""
    Wg = widen(layer["w_gate"], wdtype, layer.get("s_gate"))
    bg = layer.get("b_gate")
    G = U @ Wg.T + (0.0 if bg is None else np.asarray(bg, np.float64))
    return (G > 0).any(axis=0)
