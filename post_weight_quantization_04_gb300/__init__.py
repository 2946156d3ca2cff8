"""GPTQ per-layer weight quantization on GB300 — Python binding of libgptq.

Thin ctypes marshalling over the C ABI declared in ``include/gptq.h``: every
function here has the C entry point's name, checks tensor shapes/dtypes/devices,
allocates outputs with PyTorch (device memory and streams only) and calls the
library on the current CUDA stream. All arithmetic runs in the library's CUDA
kernels; there is no CPU or PyTorch fallback — if the library is missing or no
GPU is present, the calls raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional, Tuple

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgptq.so")

GPTQ_F32 = 0
GPTQ_BF16 = 1

STATUS = {
    0: "GPTQ_OK", 1: "GPTQ_ERR_INVALID_ARG", 2: "GPTQ_ERR_UNSUPPORTED", 3: "GPTQ_ERR_NOT_SPD",
    4: "GPTQ_ERR_CUDA", 5: "GPTQ_ERR_TIMEOUT", 6: "GPTQ_ERR_WORKSPACE", 7: "GPTQ_ERR_NONFINITE",
}

# every symbol include/gptq.h declares
EXPORTS = [
    "gptq_hessian_create", "gptq_hessian_reset", "gptq_hessian_accumulate", "gptq_hessian_finalize",
    "gptq_hessian_destroy", "gptq_prepare_workspace_bytes", "gptq_prepare", "gptq_prepare_noalloc",
    "gptq_quantize_workspace_bytes",
    "gptq_quantize", "gptq_prune_workspace_bytes", "gptq_prune", "rtn_quantize", "gptq_packed_words_per_row", "gptq_pack", "gptq_dequant_matmul",
    "gptq_status_string", "gptq_set_status_mode", "gptq_status_mode", "gptq_status_sync",
    "gptq_launch_count", "gptq_profile_enable", "gptq_profile_read", "gptq_profile_kernel_count",
    "gptq_profile_kernel_name",
]


class GptqError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS.get(status, status)} ({_str(status)})")


class QConfig(ctypes.Structure):
    _fields_ = [("bits", ctypes.c_int32), ("group", ctypes.c_int32), ("sym", ctypes.c_int32),
                ("zero_in_range", ctypes.c_int32)]


_lib: Optional[ctypes.CDLL] = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t


def _declare(lib: ctypes.CDLL) -> None:
    sig = {
        "gptq_hessian_create": (_I, [_I64, ctypes.POINTER(_P)]),
        "gptq_hessian_reset": (_I, [_P, _P]),
        "gptq_hessian_accumulate": (_I, [_P, _P, _I, _I64, _I64, _P]),
        "gptq_hessian_finalize": (_I, [_P, _P, _P, ctypes.POINTER(_I64), _P]),
        "gptq_hessian_destroy": (_I, [_P]),
        "gptq_prepare_workspace_bytes": (_SZ, [_I64, _I]),
        "gptq_prepare": (_I, [_P, _P, _I64, _F, _I, _P, _P, _P, _P, _SZ, _P]),
        "gptq_prepare_noalloc": (_I, [_P, _P, _I64, _F, _I, _P, _P, _P, _P]),
        "gptq_quantize_workspace_bytes": (_SZ, [_I64, _I64, QConfig]),
        "gptq_quantize": (_I, [_P, _I64, _I64, _P, _P, _P, QConfig, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
        "rtn_quantize": (_I, [_P, _I64, _I64, _P, QConfig, _P, _P, _P, _P, _P, _P]),
        "gptq_prune_workspace_bytes": (_SZ, [_I64, _I64]),
        "gptq_prune": (_I, [_P, _I64, _I64, _P, _P, _P, _F, _P, _P, _P, _P, _SZ, _P]),
        "gptq_packed_words_per_row": (_I64, [_I64, _I]),
        "gptq_pack": (_I, [_P, _I64, _I64, _I, _I, _P, _P]),
        "gptq_dequant_matmul": (_I, [_P, _I64, _I64, _I64, _P, _P, _P, _P, _I64, _I64, _I, _I, _P, _I64, _P]),
        "gptq_status_string": (ctypes.c_char_p, [_I]),
        "gptq_set_status_mode": (_I, [_I]),
        "gptq_status_mode": (_I, []),
        "gptq_status_sync": (_I, [_P]),
        "gptq_launch_count": (ctypes.c_ulonglong, []),
        "gptq_profile_enable": (None, [_I]),
        "gptq_profile_read": (_I, [_P, _P, _I]),
        "gptq_profile_kernel_count": (_I, []),
        "gptq_profile_kernel_name": (ctypes.c_char_p, [_I]),
        # test hook (exported, deliberately not declared in gptq.h)
        "gptq_test_set_wait_limit_ns": (_I, [ctypes.c_ulonglong]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libgptq.so (built in-tree by ``build.py``; the environment variable GPTQ_LIB names
    another build of the same library instead); raises if it is missing."""
    global _lib
    if _lib is None:
        path = os.environ.get("GPTQ_LIB", path)
        if not os.path.exists(path):
            raise RuntimeError(f"libgptq.so not built ({path}); run post_weight_quantization_04_gb300.build")
        lib = ctypes.CDLL(path)
        _declare(lib)
        _lib = lib
    return _lib


def _str(status: int) -> str:
    try:
        return load().gptq_status_string(status).decode()
    except Exception:  # noqa: BLE001
        return "?"


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise GptqError(fn, status)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t: torch.Tensor, dtype, name: str, shape=None) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def qconfig(bits: int, group: int = 0, sym: bool = True, zero_in_range: bool = False) -> QConfig:
    return QConfig(int(bits), int(group), 1 if sym else 0, 1 if zero_in_range else 0)


def gptq_packed_words_per_row(cols: int, bits: int) -> int:
    return int(load().gptq_packed_words_per_row(cols, bits))


# ------------------------------------------------------------------------------ Hessian

class Hessian:
    """The library's accumulator: S += X^T X over token batches; H = 2 S / n."""

    def __init__(self, d: int, device=None):
        lib = load()
        self.d = int(d)
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        h = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            _check("gptq_hessian_create", lib.gptq_hessian_create(self.d, ctypes.byref(h)))
        self._h = h

    def reset(self, stream=None) -> None:
        _check("gptq_hessian_reset", load().gptq_hessian_reset(self._h, _stream(stream)))

    def accumulate(self, X: torch.Tensor, stream=None) -> None:
        if X.dim() != 2 or X.shape[1] != self.d:
            raise ValueError(f"X must be (n, {self.d})")
        if X.dtype not in (torch.bfloat16, torch.float32) or not X.is_cuda:
            raise ValueError("X must be a CUDA bf16 or fp32 tensor")
        if X.stride(1) != 1:
            raise ValueError("X rows must be contiguous")
        dt = GPTQ_BF16 if X.dtype == torch.bfloat16 else GPTQ_F32
        _check("gptq_hessian_accumulate",
               load().gptq_hessian_accumulate(self._h, _ptr(X), dt, X.shape[0], X.stride(0), _stream(stream)))

    def finalize(self, stream=None) -> Tuple[torch.Tensor, torch.Tensor, int]:
        H = torch.empty(self.d, self.d, dtype=torch.float32, device=self.device)
        diag = torch.empty(self.d, dtype=torch.float32, device=self.device)
        n = ctypes.c_int64(0)
        _check("gptq_hessian_finalize",
               load().gptq_hessian_finalize(self._h, _ptr(H), _ptr(diag), ctypes.byref(n), _stream(stream)))
        return H, diag, int(n.value)

    def close(self) -> None:
        if getattr(self, "_h", None):
            load().gptq_hessian_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001
            pass


def gptq_hessian_create(d: int, device=None) -> Hessian:
    return Hessian(d, device)


def gptq_hessian_accumulate(h: Hessian, X: torch.Tensor, stream=None) -> None:
    h.accumulate(X, stream)


def gptq_hessian_finalize(h: Hessian, stream=None):
    return h.finalize(stream)


# ------------------------------------------------------------------------------ prepare

def gptq_prepare_workspace_bytes(d: int, act_order: bool = False) -> int:
    return int(load().gptq_prepare_workspace_bytes(d, 1 if act_order else 0))


def gptq_prepare(H: torch.Tensor, diag_xtx: Optional[torch.Tensor] = None, damp: float = 0.01,
                 act_order: bool = False, ws: Optional[torch.Tensor] = None, stream=None):
    """(U, perm, dead) from H (the upper triangle is read)."""
    d = H.shape[0]
    _dev(H, torch.float32, "H", (d, d))
    if act_order:
        if diag_xtx is None:
            raise ValueError("act_order needs diag_xtx")
        _dev(diag_xtx, torch.float32, "diag_xtx", (d,))
    dev = H.device
    U = torch.empty(d, d, dtype=torch.float32, device=dev)
    perm = torch.empty(d, dtype=torch.int32, device=dev)
    dead = torch.empty(d, dtype=torch.uint8, device=dev)
    nb = gptq_prepare_workspace_bytes(d, act_order)
    if ws is None:
        ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    _check("gptq_prepare", load().gptq_prepare(_ptr(H), _ptr(diag_xtx), d, float(damp), 1 if act_order else 0,
                                               _ptr(U), _ptr(perm), _ptr(dead), _ptr(ws), ws.numel(), _stream(stream)))
    return U, perm, dead


# ----------------------------------------------------------------------------- quantize

def gptq_quantize_workspace_bytes(rows: int, cols: int, bits: int = 4, group: int = 0, sym: bool = True) -> int:
    return int(load().gptq_quantize_workspace_bytes(rows, cols, qconfig(bits, group, sym)))


def _outputs(rows, cols, bits, group, dev):
    G = -(-cols // group) if group else 1
    return {
        "codes": torch.empty(rows, cols, dtype=torch.int8, device=dev),
        "scales": torch.empty(rows, G, dtype=torch.float32, device=dev),
        "zeros": torch.empty(rows, G, dtype=torch.uint8, device=dev),
        "Wq": torch.empty(rows, cols, dtype=torch.float32, device=dev),
        "packed": torch.empty(rows, gptq_packed_words_per_row(cols, bits), dtype=torch.int32, device=dev),
    }


def gptq_quantize(W: torch.Tensor, U: torch.Tensor, perm: Optional[torch.Tensor] = None,
                  dead: Optional[torch.Tensor] = None, bits: int = 4, group: int = 0, sym: bool = True,
                  ws: Optional[torch.Tensor] = None, out: Optional[Dict[str, torch.Tensor]] = None,
                  stream=None, zero_in_range: bool = False) -> Dict[str, torch.Tensor]:
    """GPTQ's column loop on W (rows, cols) given U (loop order), perm and dead.
    zero_in_range: asymmetric grid over the min/max range widened to contain 0."""
    rows, cols = W.shape
    _dev(W, torch.float32, "W")
    _dev(U, torch.float32, "U", (cols, cols))
    if perm is not None:
        _dev(perm, torch.int32, "perm", (cols,))
    if dead is not None:
        _dev(dead, torch.uint8, "dead", (cols,))
    dev = W.device
    o = out if out is not None else _outputs(rows, cols, bits, group, dev)
    if "g_idx" not in o:
        o["g_idx"] = torch.empty(cols, dtype=torch.int32, device=dev)
    if "row_loss" not in o:
        o["row_loss"] = torch.empty(rows, dtype=torch.float32, device=dev)
    nb = gptq_quantize_workspace_bytes(rows, cols, bits, group, sym)
    if ws is None:
        ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    _check("gptq_quantize", load().gptq_quantize(
        _ptr(W), rows, cols, _ptr(U), _ptr(perm), _ptr(dead), qconfig(bits, group, sym, zero_in_range),
        _ptr(o["codes"]), _ptr(o["scales"]), _ptr(o["zeros"]), _ptr(o["g_idx"]), _ptr(o.get("Wq")),
        _ptr(o.get("packed")), _ptr(o["row_loss"]), _ptr(ws), ws.numel(), _stream(stream)))
    return o


def gptq_prune_workspace_bytes(rows: int, cols: int) -> int:
    return int(load().gptq_prune_workspace_bytes(rows, cols))


def gptq_prune(W: torch.Tensor, U: torch.Tensor, perm: Optional[torch.Tensor] = None,
               dead: Optional[torch.Tensor] = None, sparsity: float = 0.5, ws: Optional[torch.Tensor] = None,
               out: Optional[Dict[str, torch.Tensor]] = None, stream=None) -> Dict[str, torch.Tensor]:
    """Pruning with GPTQ's update: Wp (pruned and compensated, 0 where pruned), mask (uint8,
    1 where pruned) and row_loss, all in the original column order."""
    rows, cols = W.shape
    _dev(W, torch.float32, "W")
    _dev(U, torch.float32, "U", (cols, cols))
    if perm is not None:
        _dev(perm, torch.int32, "perm", (cols,))
    if dead is not None:
        _dev(dead, torch.uint8, "dead", (cols,))
    dev = W.device
    nb = gptq_prune_workspace_bytes(rows, cols)
    if ws is None:
        ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    o = out if out is not None else {
        "Wp": torch.empty(rows, cols, dtype=torch.float32, device=dev),
        "mask": torch.empty(rows, cols, dtype=torch.uint8, device=dev),
        "row_loss": torch.empty(rows, dtype=torch.float32, device=dev),
    }
    _check("gptq_prune", load().gptq_prune(
        _ptr(W), rows, cols, _ptr(U), _ptr(perm), _ptr(dead), float(sparsity), _ptr(o["Wp"]), _ptr(o.get("mask")),
        _ptr(o.get("row_loss")), _ptr(ws), ws.numel(), _stream(stream)))
    return o


def rtn_quantize(W: torch.Tensor, bits: int = 4, group: int = 0, sym: bool = True,
                 dead: Optional[torch.Tensor] = None, out: Optional[Dict[str, torch.Tensor]] = None,
                 stream=None, zero_in_range: bool = False) -> Dict[str, torch.Tensor]:
    rows, cols = W.shape
    _dev(W, torch.float32, "W")
    if dead is not None:
        _dev(dead, torch.uint8, "dead", (cols,))
    o = out if out is not None else _outputs(rows, cols, bits, group, W.device)
    _check("rtn_quantize", load().rtn_quantize(
        _ptr(W), rows, cols, _ptr(dead), qconfig(bits, group, sym, zero_in_range), _ptr(o["codes"]), _ptr(o["scales"]),
        _ptr(o["zeros"]), _ptr(o.get("Wq")), _ptr(o.get("packed")), _stream(stream)))
    return o


def gptq_pack(codes: torch.Tensor, bits: int, sym: bool = True, out: Optional[torch.Tensor] = None,
              stream=None) -> torch.Tensor:
    rows, cols = codes.shape
    _dev(codes, torch.int8, "codes")
    p = out if out is not None else torch.empty(rows, gptq_packed_words_per_row(cols, bits), dtype=torch.int32,
                                                device=codes.device)
    _check("gptq_pack", load().gptq_pack(_ptr(codes), rows, cols, bits, 1 if sym else 0, _ptr(p), _stream(stream)))
    return p


STATUS_SYNC, STATUS_DEFERRED = 0, 1


def set_status_mode(deferred: bool) -> None:
    """Deferred: the calls that synchronise to report device-side errors return once their
    work is enqueued; `status_sync` reports the first such error since its last call."""
    _check("gptq_set_status_mode", load().gptq_set_status_mode(STATUS_DEFERRED if deferred else STATUS_SYNC))


def status_sync(stream=None) -> None:
    """Synchronise the stream and raise the first device-side error recorded in deferred
    mode since the last call (clearing it)."""
    _check("gptq_status_sync", load().gptq_status_sync(_stream(stream)))


class deferred_status:
    """Context manager: deferred status reporting inside, the previous mode restored after
    (pending errors are left for `status_sync`)."""

    def __enter__(self):
        self._prev = int(load().gptq_status_mode())
        _check("gptq_set_status_mode", load().gptq_set_status_mode(STATUS_DEFERRED))
        return self

    def __exit__(self, *exc):
        load().gptq_set_status_mode(self._prev)
        return False


DQ_RELU, DQ_BF16_OUT = 1, 2


def gptq_dequant_matmul(X: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor, zeros: torch.Tensor,
                        g_idx: torch.Tensor, bits: int, out: Optional[torch.Tensor] = None, relu: bool = False,
                        out_dtype=torch.float32, stream=None) -> torch.Tensor:
    """Y = X Wq^T (optionally max(., 0)) straight from the stored form (packed codes,
    scales, zeros, g_idx); Y fp32 or bf16."""
    T, K = X.shape
    N, G = scales.shape
    _dev(X, torch.bfloat16, "X")
    _dev(packed, torch.int32, "packed", (N, gptq_packed_words_per_row(K, bits)))
    _dev(scales, torch.float32, "scales")
    _dev(zeros, torch.uint8, "zeros", (N, G))
    _dev(g_idx, torch.int32, "g_idx", (K,))
    if out_dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("out_dtype must be float32 or bfloat16")
    Y = out if out is not None else torch.empty(T, N, dtype=out_dtype, device=X.device)
    _dev(Y, out_dtype, "Y", (T, N))
    flags = (DQ_RELU if relu else 0) | (DQ_BF16_OUT if out_dtype == torch.bfloat16 else 0)
    _check("gptq_dequant_matmul", load().gptq_dequant_matmul(
        _ptr(X), T, K, K, _ptr(packed), _ptr(scales), _ptr(zeros), _ptr(g_idx), N, G, bits, flags, _ptr(Y), N,
        _stream(stream)))
    return Y


def gptq_layerwise(X: torch.Tensor, Ws, bits: int = 4, group: int = 0, sym: bool = True, damp: float = 0.01,
                   act_order: bool = False, stream=None):
    """GPTQ guide page's `apply_layerwise` on the GPU: every layer is calibrated on the
    inputs it will actually see — the bf16 outputs of the layers before it, already
    quantised — and the forward pass runs on the stored form (gptq_dequant_matmul; relu on
    the hidden layers, bf16 activations, the last layer's output fp32). Returns one dict
    per layer (its calibration input, H, U, perm, dead and the gptq_quantize outputs) and
    the network's output. Host orchestration only: every step runs in the library."""
    h = X
    layers = []
    for i, W in enumerate(Ws):
        last = i == len(Ws) - 1
        acc = Hessian(h.shape[1], h.device)
        acc.accumulate(h, stream=stream)
        H, diag, _ = acc.finalize(stream=stream)
        acc.close()
        U, perm, dead = gptq_prepare(H, diag, damp, act_order=act_order, stream=stream)
        st = gptq_quantize(W, U, perm, dead, bits, group, sym, stream=stream)
        out = gptq_dequant_matmul(h, st["packed"], st["scales"], st["zeros"], st["g_idx"], bits, relu=not last,
                                  out_dtype=torch.float32 if last else torch.bfloat16, stream=stream)
        layers.append({"input": h, "H": H, "U": U, "perm": perm, "dead": dead, **st})
        h = out
    return layers, h


def gptq_status_string(status: int) -> str:
    return _str(status)


# ------------------------------------------------------------------------- instrumentation

def gptq_launch_count() -> int:
    return int(load().gptq_launch_count())


def gptq_profile_enable(on: bool = True) -> None:
    load().gptq_profile_enable(1 if on else 0)


def gptq_profile_read() -> Dict[str, Tuple[int, float]]:
    """{kernel class: (launches, total ms)} for the launches recorded since the last read."""
    lib = load()
    n = lib.gptq_profile_kernel_count()
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_ulonglong * n)()
    _check("gptq_profile_read", lib.gptq_profile_read(ms, cnt, n))
    return {lib.gptq_profile_kernel_name(i).decode(): (int(cnt[i]), float(ms[i])) for i in range(n) if cnt[i]}


__all__ = [
    "load", "Hessian", "GptqError", "QConfig", "qconfig", "gptq_hessian_create", "gptq_hessian_accumulate",
    "gptq_hessian_finalize", "gptq_prepare", "gptq_prepare_workspace_bytes", "gptq_quantize",
    "gptq_quantize_workspace_bytes", "rtn_quantize", "gptq_pack", "gptq_packed_words_per_row",
    "gptq_dequant_matmul", "gptq_layerwise", "gptq_status_string", "gptq_launch_count", "gptq_profile_enable", "gptq_profile_read",
    "set_status_mode", "status_sync", "deferred_status", "STATUS_SYNC", "STATUS_DEFERRED",
    "EXPORTS", "LIB_PATH",
]
