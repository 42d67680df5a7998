"""Shared set-up for the GPU parity tests.

Both sides receive the same generated arrays. The CUDA side reorders them
hot-first with the library's own order/permute kernels; the oracle side with
``oracle.hot_first_order`` and numpy indexing. The two orders are compared
bit-exactly before anything else is.
"""
import numpy as np
import torch

import oracle
from workload import make_inputs, make_layer

PER_NEURON = ("w_gate", "w_up", "w_down_t", "s_gate", "s_up", "s_down", "b_gate", "p2_t", "b_pred", "counts", "p")
BAND = oracle.BAND
TOL = {"f32": 1e-3, "bf16": 1e-3, "f16": 1e-3, "int4g128": 5e-3}   # rel-L2 bar on y


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def build_layers(w, layer_ids, seed=0):
    """[(gpu_layer dict of CUDA tensors, oracle layer dict of numpy arrays)] in hot-first order."""
    import activation_sparse_decode_pi_gb300 as P

    out = []
    for l in layer_ids:
        L = make_layer(w, l, seed, device="cuda")
        Lg, perm = P.apply_hot_first(L)
        perm_o = oracle.hot_first_order(L["counts"].cpu().numpy())
        assert np.array_equal(perm.cpu().numpy(), perm_o), "hot-first order differs from the oracle's"
        Lo = oracle.layer_numpy(L)
        for k in PER_NEURON:
            if Lo.get(k) is not None:
                Lo[k] = np.ascontiguousarray(Lo[k][perm_o])
        out.append((Lg, Lo))
        del L
    return out


def rms_inputs(w, B, tokens=1, seed=0):
    """u = x / rms(x) for x ~ N(0, I), rounded once to fp32: the same values for both sides."""
    x = make_inputs(w, tokens, B, seed, device="cpu").numpy().astype(np.float64)
    u = x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + oracle.RMS_EPS)
    return u.astype(np.float32)


def band_mask(z):
    """Neurons whose oracle logit lies within BAND of the threshold for some batch row."""
    return (np.abs(z) < BAND).any(axis=0)


def to_dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def teacher_forced(P, w, layers, ffn, x0, hot_prefix=0, tag=""):
    """One decode step checked layer by layer, teacher-forced.

    Layer l of the oracle runs on the GPU's own input x_l (pi_decode_stack_layers keeps every
    layer's output), so every layer is compared, including those after an in-band difference
    upstream: (1) the GPU's active list equals the oracle's outside the 1e-4 band, and (2)
    y_l = x_{l+1} - x_l is within the dtype's bar of the oracle's sparse FFN evaluated on the
    GPU's own list (an in-band difference is then not counted twice).
    Returns (x_out as numpy, number of layers with an in-band difference).
    """
    x0 = np.asarray(x0, np.float32)
    B = x0.shape[0]
    counts = torch.zeros(w.n_layers, dtype=torch.int32, device="cuda")
    idx_out = torch.zeros((w.n_layers, w.f), dtype=torch.int32, device="cuda")
    xo, xl = ffn.decode_stack_layers(to_dev(x0), counts=counts, idx_out=idx_out)
    torch.cuda.synchronize()
    assert torch.equal(xo, xl[-1]), (tag, "last layer row differs from x_out")
    xs = [x0.astype(np.float64)] + [xl[l].cpu().numpy().astype(np.float64) for l in range(w.n_layers)]
    cg, ig = counts.cpu().numpy(), idx_out.cpu().numpy()
    flips = 0
    for l in range(w.n_layers):
        Lo = layers[l][1]
        u = oracle.rms_norm(xs[l])
        pr = oracle.predict(u, Lo["p1_t"], Lo["p2_t"], Lo["b_pred"], w.pdtype, hot_prefix=hot_prefix)
        gi = ig[l, : cg[l]]
        assert np.all(np.diff(gi) > 0), (tag, l, "active list not ascending")
        if hot_prefix:
            H = min(hot_prefix, gi.size)
            assert np.array_equal(gi[:H], np.arange(H)), (tag, l, "hot prefix missing")
        diff = np.setxor1d(gi, pr["idx"])
        assert np.all(band_mask(pr["z"])[diff]), (tag, l, f"{int((~band_mask(pr['z'])[diff]).sum())} out-of-band")
        flips += int(diff.size > 0)
        _, yo = oracle.sparse_ffn(u, Lo, gi, w.kind, w.wdtype)
        err = rel_l2(xs[l + 1] - xs[l], yo)
        assert err <= TOL[w.wdtype], (tag, l, err)
    return xo.cpu().numpy(), flips
