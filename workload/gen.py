"""Synthetic workloads for PowerInfer-style activation-sparse FFN decode.

The pages measure real ReLU models (OPT, Llama2/ReluLLaMA, Falcon) on
Wikipedia/WikiText text ("PowerInfer" summary page, Experiments; the
paper walk-through page, profiling constraints). Neither the models nor the
data exist here, so these seeded draws stand in for them, with the shapes of
those models and the activation statistics the pages report:

* a power-law (Zipf) per-neuron activation frequency (walk-through page,
  "neuron activation power law"; summary page, Key Results: 26% of neurons
  carry 80% of activations; the walk-through: ~10% hot neurons active on
  >= 80% of inputs);
* weights ~ N(0, 1/d), rounded to their stored type (f32/bf16/f16) or
  int4-quantised per row in groups of 128 with fp16 scales, *before* any bias
  is computed;
* gate bias b_i = ||Wg_i|| * Phi^-1(p_i), so that P(u.Wg_i + b_i > 0) = p_i
  for u ~ N(0, I);
* predictor P1 ~ N(0, 1/d), P2 ~ N(0, 1/r) and a bias calibrated the same way
  from the mean/variance of ReLU(u.P1) so that the predictor fires on neuron i
  with probability ~ p_i;
* profiling counts ~ Binomial(T_calib, p_i): the statistic the offline
  profiler of the walk-through page (offline profiling code block) would
  collect;
* decode inputs x0 ~ N(0, I_d), independent per token.

Neurons come out in *profiling order* (Zipf ranks assigned by a seeded random
permutation), so the offline hot-first reorder has real work to do.

Everything is drawn with torch on the requested device (CPU for small cases,
CUDA for full-size ones); the same arrays are then handed to both the CUDA path
and the oracle. Substreams are keyed by (seed, workload, layer, tensor).
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field

import numpy as np
import torch

T_CALIB = 2048  # calibration tokens behind the synthetic profiling counts
P_CLIP = (1e-6, 0.999)


@dataclass(frozen=True)
class Workload:
    name: str
    wid: int              # stable id used in seeding substreams
    d: int                # model width
    f: int                # FFN width (neurons)
    r: int                # predictor rank
    n_layers: int
    kind: str             # "gated" (LLaMA-style) or "relu" (OPT/Falcon fc1->ReLU->fc2)
    wdtype: str           # "f32" | "bf16" | "f16" | "int4g128"
    pdtype: str           # "f32" | "bf16" | "f16"
    batches: tuple
    tokens: int
    freq: dict = field(default_factory=dict)
    note: str = ""


WORKLOADS = {
    w.name: w
    for w in [
        Workload(
            "ffn_d512_f2048_fp32_L1", 1, d=512, f=2048, r=64, n_layers=1, kind="gated",
            wdtype="f32", pdtype="f32", batches=(1,), tokens=1,
            freq=dict(kind="zipf", s=1.1, mean=0.10),
            note="single ReLU-gated FFN layer, oracle runs in seconds",
        ),
        Workload(
            "relullama7b_d4096_f11008_bf16_L32", 2, d=4096, f=11008, r=1024, n_layers=32,
            kind="gated", wdtype="bf16", pdtype="bf16", batches=(1,), tokens=256,
            freq=dict(kind="hot_tail", s=1.1, mean=0.10, hot_frac=0.10, hot_hi=1.0, hot_lo=0.8),
            note="ReluLLaMA-7B-shaped stack",
        ),
        Workload(
            "llama2_13b_d5120_f13824_bf16_L40", 3, d=5120, f=13824, r=1024, n_layers=40,
            kind="gated", wdtype="bf16", pdtype="bf16", batches=(1, 4, 16), tokens=256,
            freq=dict(kind="zipf", s=1.0, mean=0.12),
            note="Llama2-13B-shaped stack, union mask across the batch",
        ),
        Workload(
            "opt30b_d7168_f28672_fp16_L48", 4, d=7168, f=28672, r=1024, n_layers=48,
            kind="relu", wdtype="f16", pdtype="f16", batches=(1, 32), tokens=256,
            freq=dict(kind="cover", top=0.26, cover=0.80, mean=0.05),
            note="OPT-30B-shaped stack, non-gated",
        ),
        Workload(
            "opt175b_d12288_f49152_int4_L96", 5, d=12288, f=49152, r=1024, n_layers=96,
            kind="relu", wdtype="int4g128", pdtype="f16", batches=(1,), tokens=128,
            freq=dict(kind="zipf", s=1.2, mean=0.04),
            note="OPT-175B-shaped stack, int4 group-128 weights",
        ),
    ]
}


def workload_by_name(name: str) -> Workload:
    return WORKLOADS[name]


def scaled(w: Workload, *, d: int, f: int, r: int, n_layers: int, name: str | None = None) -> Workload:
    """Same recipe (kind, dtypes, frequency law) at a smaller shape."""
    return dataclasses.replace(
        w, name=name or f"{w.name}@d{d}_f{f}_r{r}_L{n_layers}", d=d, f=f, r=r, n_layers=n_layers
    )


# ----------------------------------------------------------------------------------------------
# activation frequencies (per rank, then assigned to neurons by a seeded permutation)
# ----------------------------------------------------------------------------------------------

def _bisect(fn, lo, hi, iters=200):
    """Root of a monotone increasing fn on [lo, hi]."""
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        if fn(mid) < 0:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def _zipf_ranked(f: int, s: float, mean: float) -> np.ndarray:
    rank = np.arange(1, f + 1, dtype=np.float64)
    base = rank ** (-s)
    c = math.exp(_bisect(lambda lc: np.minimum(1.0, math.exp(lc) * base).mean() - mean, -30.0, 30.0))
    return np.minimum(1.0, c * base)


def _hot_tail_ranked(f: int, s: float, mean: float, hot_frac: float, hot_hi: float, hot_lo: float) -> np.ndarray:
    """Hot prefix linear hot_hi -> hot_lo, then a Zipf tail capped at hot_lo.

    A pure Zipf law cannot give both a ~10% mean and a hot 10% that is active on
    >= 80% of tokens; this two-segment law gives both.
    """
    n_hot = max(1, int(round(hot_frac * f)))
    rank = np.arange(1, f + 1, dtype=np.float64)
    hot = np.linspace(hot_hi, hot_lo, n_hot)
    tail_base = rank[n_hot:] ** (-s)

    def mean_err(lc):
        tail = np.minimum(hot_lo, math.exp(lc) * tail_base)
        return (hot.sum() + tail.sum()) / f - mean

    c = math.exp(_bisect(mean_err, -30.0, 30.0))
    return np.concatenate([hot, np.minimum(hot_lo, c * tail_base)])


def _cover_ranked(f: int, top: float, cover: float, mean: float) -> np.ndarray:
    """Zipf law whose exponent makes the top `top` fraction carry `cover` of all activations."""
    k = int(round(top * f))

    def share_err(s):
        p = _zipf_ranked(f, s, mean)
        return p[:k].sum() / p.sum() - cover

    s = _bisect(share_err, 0.3, 3.0, iters=80)
    return _zipf_ranked(f, s, mean)


def ranked_probs(w: Workload) -> np.ndarray:
    fr = dict(w.freq)
    kind = fr.pop("kind")
    if kind == "zipf":
        p = _zipf_ranked(w.f, **fr)
    elif kind == "hot_tail":
        p = _hot_tail_ranked(w.f, **fr)
    elif kind == "cover":
        p = _cover_ranked(w.f, **fr)
    else:
        raise ValueError(kind)
    return np.clip(p, *P_CLIP)


def _key(seed: int, w: Workload, layer: int, tid: int) -> int:
    k = seed
    for v in (w.wid, layer, tid):
        k = (k * 1_000_003 + v + 7) % (1 << 62)
    return k


def _gen(device, seed: int, w: Workload, layer: int, tid: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_key(seed, w, layer, tid))
    return g


def activation_probs(w: Workload, layer: int, seed: int = 0) -> np.ndarray:
    """Per-neuron activation probability in profiling order (ranks randomly permuted)."""
    ranked = ranked_probs(w)
    rng = np.random.default_rng(_key(seed, w, layer, 99))
    return ranked[rng.permutation(w.f)]


# ----------------------------------------------------------------------------------------------
# weights
# ----------------------------------------------------------------------------------------------

_TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def quantize_int4_g128(wf: torch.Tensor):
    """Row-wise symmetric int4, groups of 128 along a row, fp16 scales.

    s = fp16(max|w| / 7); q = clamp(round_half_even(w / s), -7, 7); s == 0 gives q = 0.
    Packed two's-complement nibbles, the even element in the low nibble.
    Returns (packed uint8 [rows, d/2], scales fp16 [rows, d/128]).
    """
    rows, d = wf.shape
    assert d % 128 == 0
    g = wf.view(rows, d // 128, 128)
    s = (g.abs().amax(-1) / 7.0).to(torch.float16)
    sf = s.float().unsqueeze(-1)
    q = torch.where(sf > 0, torch.round(g / torch.where(sf > 0, sf, torch.ones_like(sf))), torch.zeros_like(g))
    q = q.clamp(-7, 7).to(torch.int16).view(rows, d)
    lo = q[:, 0::2] & 0xF
    hi = q[:, 1::2] & 0xF
    packed = (lo | (hi << 4)).to(torch.uint8)
    return packed.contiguous(), s.contiguous()


def dequantize_int4_g128(packed: torch.Tensor, scales: torch.Tensor) -> torch.Tensor:
    """Stored int4 values widened to fp32 (exact): only used to calibrate biases."""
    rows = packed.shape[0]
    p = packed.to(torch.int16)
    lo = p & 0xF
    hi = (p >> 4) & 0xF
    lo = torch.where(lo >= 8, lo - 16, lo)
    hi = torch.where(hi >= 8, hi - 16, hi)
    q = torch.stack([lo, hi], dim=-1).view(rows, -1).float()
    return (q.view(rows, -1, 128) * scales.float().unsqueeze(-1)).view(rows, -1)


def _weight(w: Workload, shape, std, dtype, device, seed, layer, tid):
    g = _gen(device, seed, w, layer, tid)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std
    if dtype == "int4g128":
        packed, scales = quantize_int4_g128(t)
        return packed, scales, dequantize_int4_g128(packed, scales)
    stored = t.to(_TORCH_DT[dtype]).contiguous()
    return stored, None, stored.float()


def make_layer(w: Workload, layer: int, seed: int = 0, device="cpu") -> dict:
    """All tensors of one FFN layer plus its predictor, in profiling order.

    Keys: w_gate (W1 for non-gated), w_up (None for non-gated), w_down_t (W_down
    transposed, [f x d]), s_gate/s_up/s_down (fp16 group scales for int4, else
    None), b_gate f32 [f], p1_t [r x d], p2_t [f x r], b_pred f32 [f],
    counts int32 [f] (profiling counts), p float64 [f] (activation probability).
    """
    d, f, r = w.d, w.f, w.r
    p = activation_probs(w, layer, seed)
    p_t = torch.from_numpy(p).to(device)
    out = {"p": p_t}

    wg, sg, wg_f = _weight(w, (f, d), d ** -0.5, w.wdtype, device, seed, layer, 1)
    out["w_gate"], out["s_gate"] = wg, sg
    if w.kind == "gated":
        wu, su, _ = _weight(w, (f, d), d ** -0.5, w.wdtype, device, seed, layer, 2)
        out["w_up"], out["s_up"] = wu, su
    else:
        out["w_up"], out["s_up"] = None, None
    wd, sd, _ = _weight(w, (f, d), d ** -0.5, w.wdtype, device, seed, layer, 3)
    out["w_down_t"], out["s_down"] = wd, sd

    z_p = torch.special.ndtri(p_t)  # Phi^-1(p), float64
    out["b_gate"] = (wg_f.double().norm(dim=1) * z_p).float().contiguous()
    del wg_f

    p1, _, p1_f = _weight(w, (r, d), d ** -0.5, w.pdtype, device, seed, layer, 4)
    p2, _, p2_f = _weight(w, (f, r), r ** -0.5, w.pdtype, device, seed, layer, 5)
    out["p1_t"], out["p2_t"] = p1, p2
    n1 = p1_f.double().norm(dim=1)                      # ||P1_k||, [r]
    p2d = p2_f.double()
    mu = (p2d @ n1) / math.sqrt(2 * math.pi)            # E[sum_k P2T[i,k] ReLU(u.P1_k)]
    var = (p2d * p2d) @ (n1 * n1) * (0.5 - 1.0 / (2 * math.pi))
    out["b_pred"] = (var.sqrt() * z_p - mu).float().contiguous()
    del p1_f, p2_f, p2d

    g = _gen(device, seed, w, layer, 6)
    counts = torch.binomial(torch.full((f,), float(T_CALIB), device=device, dtype=torch.float32),
                            p_t.float(), generator=g)
    out["counts"] = counts.to(torch.int32).contiguous()
    return out


def make_inputs(w: Workload, tokens: int, batch: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """Decode-step inputs x0 ~ N(0, I_d): [tokens, batch, d] float32."""
    g = _gen(device, seed, w, 10_000, 7)
    return torch.randn((tokens, batch, w.d), generator=g, device=device, dtype=torch.float32)
