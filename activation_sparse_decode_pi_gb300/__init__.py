"""Python binding of libpi_ffn.so: activation-sparse FFN decode on one GB300 (sm_103a).

Argument marshalling only. Every step of the path runs in the CUDA kernels of
libpi_ffn.so (built in-tree by ``_build.py``); there is no CPU or PyTorch
fallback, and importing this package fails if the library has not been built.

The raw C-ABI calls keep their names (``pi_ffn_create``, ``pi_predict``,
``pi_sparse_ffn``, ``pi_decode_stack``, ``pi_hot_first_order``,
``pi_permute_rows``, ``pi_get_status``, ...) and take device pointers (ints)
or CUDA torch tensors. ``SparseFFN`` wraps a handle for torch users.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpi_ffn.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python activation_sparse_decode_pi_gb300/_build.py` "
        "(or __graft_entry__.build()); there is no fallback path")

_lib = ctypes.CDLL(LIB_PATH)

PI_OK, PI_ERR_INVALID_ARG, PI_ERR_UNSUPPORTED, PI_ERR_CUDA, PI_ERR_OOM, PI_ERR_TIMEOUT, PI_ERR_DEVICE_CHECK = range(7)
PI_FFN_GATED_RELU, PI_FFN_RELU = 0, 1
PI_F32, PI_BF16, PI_F16, PI_INT4_G128 = 0, 1, 2, 3
DTYPES = {"f32": PI_F32, "bf16": PI_BF16, "f16": PI_F16, "int4g128": PI_INT4_G128}
KINDS = {"gated": PI_FFN_GATED_RELU, "relu": PI_FFN_RELU}

# every symbol include/pi_ffn.h declares
EXPORTS = (
    "pi_ffn_create", "pi_ffn_destroy", "pi_predict", "pi_sparse_ffn", "pi_decode_stack",
    "pi_hot_first_order", "pi_permute_rows", "pi_get_status", "pi_status_string", "pi_abi_version",
    "pi_profile_begin", "pi_profile_end", "pi_sparse_ffn_noalloc", "pi_selftest_grid_barrier",
    "pi_selftest_umma", "pi_ffn_set_hot_neurons", "pi_ffn_set_hot_prefix", "pi_decode_stack_layers",
    "pi_ffn_set_phase_trace",
)
PI_STACK_PHASES = 8
STACK_PHASE_NAMES = ("layer_start", "hidden_done", "logits_start", "list_ready", "first_rows", "ffn_done",
                     "reduce_start", "reduce_done")
PI_NOALLOC_SCRATCH_BYTES = 16 << 20
KERNEL_KINDS = ("rms", "pred_hidden", "pred_logits", "ffn_h", "ffn_down", "reduce", "decode_stack", "pred_fused")


class PiFfnDesc(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int32), ("f", ctypes.c_int32), ("r", ctypes.c_int32),
                ("n_layers", ctypes.c_int32), ("max_batch", ctypes.c_int32), ("kind", ctypes.c_int32),
                ("wdtype", ctypes.c_int32), ("pdtype", ctypes.c_int32), ("tau_logit", ctypes.c_float)]


class PiLayerWeights(ctypes.Structure):
    _fields_ = [("w_gate", ctypes.c_void_p), ("w_up", ctypes.c_void_p), ("w_down_t", ctypes.c_void_p),
                ("s_gate", ctypes.c_void_p), ("s_up", ctypes.c_void_p), ("s_down", ctypes.c_void_p),
                ("b_gate", ctypes.c_void_p), ("p1_t", ctypes.c_void_p), ("p2_t", ctypes.c_void_p),
                ("b_pred", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_lib.pi_ffn_create.restype = ctypes.c_int
_lib.pi_ffn_create.argtypes = [ctypes.POINTER(_P), ctypes.POINTER(PiFfnDesc), ctypes.POINTER(PiLayerWeights)]
_lib.pi_ffn_destroy.restype = None
_lib.pi_ffn_destroy.argtypes = [_P]
_lib.pi_predict.restype = ctypes.c_int
_lib.pi_predict.argtypes = [_P, _I32, _P, _I32, _P, _P, _P]
_lib.pi_sparse_ffn.restype = ctypes.c_int
_lib.pi_sparse_ffn.argtypes = [_P, _I32, _P, _I32, _P, _P, _P, _P]
_lib.pi_decode_stack.restype = ctypes.c_int
_lib.pi_decode_stack.argtypes = [_P, _P, _I32, _P, _P, _P, _P]
_lib.pi_decode_stack_layers.restype = ctypes.c_int
_lib.pi_decode_stack_layers.argtypes = [_P, _P, _I32, _P, _P, _P, _P, _P]
_lib.pi_ffn_set_phase_trace.restype = ctypes.c_int
_lib.pi_ffn_set_phase_trace.argtypes = [_P, _P, _I64]
_lib.pi_hot_first_order.restype = ctypes.c_int
_lib.pi_hot_first_order.argtypes = [_P, _I32, _P, _P]
_lib.pi_permute_rows.restype = ctypes.c_int
_lib.pi_permute_rows.argtypes = [_P, _P, _P, _I64, _I64, _P, _P]
_lib.pi_get_status.restype = ctypes.c_int
_lib.pi_get_status.argtypes = [_P]
_lib.pi_status_string.restype = ctypes.c_char_p
_lib.pi_status_string.argtypes = [ctypes.c_int]
_lib.pi_abi_version.restype = _I32
_lib.pi_abi_version.argtypes = []
_lib.pi_sparse_ffn_noalloc.restype = ctypes.c_int
_lib.pi_sparse_ffn_noalloc.argtypes = [ctypes.POINTER(PiFfnDesc), ctypes.POINTER(PiLayerWeights), _P, _I32, _P, _P,
                                       _P, _P, _P]
_lib.pi_selftest_grid_barrier.restype = ctypes.c_int
_lib.pi_selftest_grid_barrier.argtypes = [_P, _I32, _P]
_lib.pi_ffn_set_hot_prefix.restype = ctypes.c_int
_lib.pi_ffn_set_hot_prefix.argtypes = [_P, _I32]
_lib.pi_ffn_set_hot_neurons.restype = ctypes.c_int
_lib.pi_ffn_set_hot_neurons.argtypes = [_P, _I32]
_lib.pi_selftest_umma.restype = ctypes.c_int
_lib.pi_selftest_umma.argtypes = [_P, _P, _P, _I32, _I32, _I32, _I32, _P, _P]
_lib.pi_profile_begin.restype = ctypes.c_int
_lib.pi_profile_begin.argtypes = [_P]
_lib.pi_profile_end.restype = ctypes.c_int
_lib.pi_profile_end.argtypes = [_P, _P, _P, _I32]


class PiError(RuntimeError):
    def __init__(self, code: int, call: str):
        self.code = code
        super().__init__(f"{call}: {pi_status_string(code)} ({code})")


def pi_status_string(code: int) -> str:
    return _lib.pi_status_string(code).decode()


def pi_abi_version() -> int:
    return _lib.pi_abi_version()


def _ptr(x):
    """Device pointer of a CUDA tensor, an int, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(code: int, call: str):
    if code != PI_OK:
        raise PiError(code, call)


def pi_ffn_create(desc: PiFfnDesc, layers) -> int:
    arr = (PiLayerWeights * len(layers))(*layers)
    h = _P()
    _check(_lib.pi_ffn_create(ctypes.byref(h), ctypes.byref(desc), arr), "pi_ffn_create")
    return h.value


def pi_ffn_destroy(h: int) -> None:
    _lib.pi_ffn_destroy(h)


def pi_predict(h, layer, u, B, idx, count, stream=None) -> None:
    _check(_lib.pi_predict(h, layer, _ptr(u), B, _ptr(idx), _ptr(count), _stream(stream)), "pi_predict")


def pi_sparse_ffn(h, layer, u, B, idx, count, y, stream=None) -> None:
    _check(_lib.pi_sparse_ffn(h, layer, _ptr(u), B, _ptr(idx), _ptr(count), _ptr(y), _stream(stream)),
           "pi_sparse_ffn")


def pi_decode_stack(h, x0, B, x_out, counts=None, idx_out=None, stream=None) -> None:
    _check(_lib.pi_decode_stack(h, _ptr(x0), B, _ptr(x_out), _ptr(counts), _ptr(idx_out), _stream(stream)),
           "pi_decode_stack")


def pi_decode_stack_layers(h, x0, B, x_out, counts, idx_out, x_layers, stream=None) -> None:
    _check(_lib.pi_decode_stack_layers(h, _ptr(x0), B, _ptr(x_out), _ptr(counts), _ptr(idx_out), _ptr(x_layers),
                                       _stream(stream)), "pi_decode_stack_layers")


def pi_ffn_set_phase_trace(h, stamps, n_stamps=0) -> None:
    _check(_lib.pi_ffn_set_phase_trace(h, _ptr(stamps), n_stamps), "pi_ffn_set_phase_trace")


def pi_sparse_ffn_noalloc(desc, layer, u, B, idx, count, y, status=None, stream=None) -> None:
    """pi_sparse_ffn without a handle and without any device allocation (static library scratch)."""
    _check(_lib.pi_sparse_ffn_noalloc(ctypes.byref(desc), ctypes.byref(layer), _ptr(u), B, _ptr(idx), _ptr(count),
                                      _ptr(y), _ptr(status), _stream(stream)), "pi_sparse_ffn_noalloc")


def pi_selftest_grid_barrier(work, extra, stream=None) -> None:
    _check(_lib.pi_selftest_grid_barrier(_ptr(work), extra, _stream(stream)), "pi_selftest_grid_barrier")


def pi_ffn_set_hot_prefix(h, hot_prefix) -> None:
    _check(_lib.pi_ffn_set_hot_prefix(h, hot_prefix), "pi_ffn_set_hot_prefix")


def pi_ffn_set_hot_neurons(h, n_hot) -> None:
    _check(_lib.pi_ffn_set_hot_neurons(h, n_hot), "pi_ffn_set_hot_neurons")


def pi_selftest_umma(a, b, d, mode, n, k, dtype, status, stream=None) -> None:
    _check(_lib.pi_selftest_umma(_ptr(a), _ptr(b), _ptr(d), mode, n, k, dtype, _ptr(status), _stream(stream)),
           "pi_selftest_umma")


def pi_hot_first_order(counts, f, perm, stream=None) -> None:
    _check(_lib.pi_hot_first_order(_ptr(counts), f, _ptr(perm), _stream(stream)), "pi_hot_first_order")


def pi_permute_rows(src, dst, perm, rows, row_bytes, err=None, stream=None) -> None:
    _check(_lib.pi_permute_rows(_ptr(src), _ptr(dst), _ptr(perm), rows, row_bytes, _ptr(err), _stream(stream)),
           "pi_permute_rows")


def pi_get_status(h) -> int:
    return _lib.pi_get_status(h)


def pi_profile_begin(h) -> None:
    _check(_lib.pi_profile_begin(h), "pi_profile_begin")


def pi_profile_end(h) -> dict:
    """{kernel kind: (total ms, launches)} since pi_profile_begin."""
    n = len(KERNEL_KINDS)
    ms = (ctypes.c_float * n)()
    cnt = (ctypes.c_int32 * n)()
    _check(_lib.pi_profile_end(h, ms, cnt, n), "pi_profile_end")
    return {k: (float(ms[i]), int(cnt[i])) for i, k in enumerate(KERNEL_KINDS)}


# ------------------------------------------------------------------------------------------------
# torch conveniences (still only marshalling: each call is one C-ABI call)
# ------------------------------------------------------------------------------------------------

PER_NEURON = ("w_gate", "w_up", "w_down_t", "s_gate", "s_up", "s_down", "b_gate", "p2_t", "b_pred", "counts", "p")


def hot_first_order(counts):
    """perm (int32, device) for a CUDA tensor of per-neuron activation counts."""
    import torch

    c = counts.to(torch.int32).contiguous()
    perm = torch.empty_like(c)
    pi_hot_first_order(c, c.numel(), perm)
    return perm


def permute_rows(src, perm):
    """dst[k] = src[perm[k]] for a CUDA tensor (rows along dim 0)."""
    import torch

    s = src.contiguous()
    dst = torch.empty_like(s)
    rows = s.shape[0]
    row_bytes = s.numel() * s.element_size() // max(rows, 1)
    pi_permute_rows(s, dst, perm, rows, row_bytes)
    return dst


def apply_hot_first(layer: dict) -> tuple[dict, object]:
    """Offline hot-first reorder of one layer (every per-neuron array) by its profiling counts."""
    perm = hot_first_order(layer["counts"])
    out = dict(layer)
    for k in PER_NEURON:
        v = layer.get(k)
        if v is not None and hasattr(v, "is_cuda") and v.is_cuda:
            out[k] = permute_rows(v, perm)
    return out, perm


def layer_weights(layer: dict) -> PiLayerWeights:
    g = lambda k: _ptr(layer.get(k))
    return PiLayerWeights(g("w_gate"), g("w_up"), g("w_down_t"), g("s_gate"), g("s_up"), g("s_down"),
                          g("b_gate"), g("p1_t"), g("p2_t"), g("b_pred"))


class SparseFFN:
    """A pi_ffn handle over CUDA tensors (kept referenced for the handle's lifetime)."""

    def __init__(self, layers, *, d, f, r, kind, wdtype, pdtype, max_batch=1, tau=0.0):
        self.layers = list(layers)
        self.desc = PiFfnDesc(d, f, r, len(self.layers), max_batch, KINDS[kind], DTYPES[wdtype], DTYPES[pdtype],
                              tau)
        self.h = pi_ffn_create(self.desc, [layer_weights(L) for L in self.layers])

    @classmethod
    def from_workload(cls, w, layers, max_batch=1, tau=0.0):
        return cls(layers, d=w.d, f=w.f, r=w.r, kind=w.kind, wdtype=w.wdtype, pdtype=w.pdtype,
                   max_batch=max_batch, tau=tau)

    def predict(self, layer, u, idx=None, count=None, stream=None):
        import torch

        B = u.shape[0]
        idx = torch.empty(self.desc.f, dtype=torch.int32, device=u.device) if idx is None else idx
        count = torch.empty(1, dtype=torch.int32, device=u.device) if count is None else count
        pi_predict(self.h, layer, u, B, idx, count, stream)
        return idx, count

    def sparse_ffn(self, layer, u, idx, count, y=None, stream=None):
        import torch

        y = torch.empty_like(u) if y is None else y
        pi_sparse_ffn(self.h, layer, u, u.shape[0], idx, count, y, stream)
        return y

    def decode_stack(self, x0, x_out=None, counts=None, idx_out=None, stream=None):
        import torch

        x_out = torch.empty_like(x0) if x_out is None else x_out
        pi_decode_stack(self.h, x0, x0.shape[0], x_out, counts, idx_out, stream)
        return x_out

    def decode_stack_layers(self, x0, counts=None, idx_out=None, stream=None):
        """(x_out, x_layers): one decode step, and every layer's output (row l = x_{l+1})."""
        import torch

        B = x0.shape[0]
        x_out = torch.empty_like(x0)
        x_layers = torch.empty((self.desc.n_layers, B, self.desc.d), dtype=torch.float32, device=x0.device)
        pi_decode_stack_layers(self.h, x0, B, x_out, counts, idx_out, x_layers, stream)
        return x_out, x_layers

    def set_phase_trace(self, stamps) -> None:
        """Phase stamps of the persistent step into `stamps` (int64 CUDA tensor
        [n_layers, PI_STACK_PHASES, n_sm]); None turns them off."""
        pi_ffn_set_phase_trace(self.h, stamps, 0 if stamps is None else stamps.numel())

    def set_hot_neurons(self, n_hot: int) -> None:
        pi_ffn_set_hot_neurons(self.h, n_hot)

    def set_hot_prefix(self, hot_prefix: int) -> None:
        pi_ffn_set_hot_prefix(self.h, hot_prefix)

    def status(self) -> int:
        return pi_get_status(self.h)

    def close(self):
        if self.h:
            pi_ffn_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
