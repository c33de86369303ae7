"""Thin ctypes binding of libcbq.so (include/cbq.h), same names as the C ABI.

Argument marshalling only: torch tensors give device pointers and the current
stream, numpy arrays give host pointers.  Every step of the path runs in the
library's CUDA kernels; if libcbq.so is missing this module raises instead of
computing anything another way.
"""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libcbq.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "cbq.h")

CBQ_OK, CBQ_EINVAL, CBQ_ECUDA, CBQ_ENOMEM, CBQ_EDEVICE = 0, -1, -2, -3, -4
CBQ_QK = 32
CBQ_BLOCK_BYTES = 18
CBQ_MAX_COLS = 5
CBQ_MAX_TOKENS = 5
CBQ_MAX_TOPK = 16
CBQ_DEVERR_BAD_EXPERT_ID = 0x1
CBQ_DEVERR_PIPE_TIMEOUT = 0x100
CBQ_DEVERR_DEPENDENCY_TIMEOUT = 0x200
CBQ_STATIC_SCRATCH_MAX_K = 16384
CBQ_ROUTER_MAX_E = 16384
CBQ_MAX_MMQ_COLS = 16
CBQ_HC_NHC = 4
CBQ_HC_MAX_ITERS = 1024
CBQ_HC_MAX_N = 1 << 28

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_SIGS = {
    "cbq_status_string": ([_I], ctypes.c_char_p),
    "cbq_last_cuda_error": ([], ctypes.c_char_p),
    "cbq_weights_create": ([_P, _I64, _I64, _I, _P, ctypes.POINTER(_P)], _I),
    "cbq_weights_destroy": ([_P], _I),
    "cbq_weights_info": ([_P, ctypes.POINTER(_I64), ctypes.POINTER(_I64), ctypes.POINTER(_I64)], _I),
    "cbq_quantize_act": ([_P, _I64, _I, _P, _P, _P], _I),
    "cbq_matvec_q": ([_P, _P, _P, _I, _P, _P], _I),
    "cbq_matvec": ([_P, _P, _I, _P, _P], _I),
    "cbq_matvec_host": ([_P, _P, _I, _P, _P], _I),
    "cbq_matvec_static": ([_P, _P, _I, _P, _P], _I),
    "cbq_moe_create": ([_P, _P, _I, _I64, _I64, _I, _P, ctypes.POINTER(_P)], _I),
    "cbq_moe_destroy": ([_P], _I),
    "cbq_moe_set_shared": ([_P, _P, _P, _I, _P], _I),
    "cbq_moe_info": ([_P, ctypes.POINTER(_I), ctypes.POINTER(_I64), ctypes.POINTER(_I64), ctypes.POINTER(_I64)], _I),
    "cbq_moe_matvec": ([_P, _P, _I, _P, _P, _I, _I, _P, _P], _I),
    "cbq_moe_matvec_host": ([_P, _P, _I, _P, _P, _I, _I, _P, _P], _I),
    "cbq_router_topk": ([_P, _I, _I, _I, _P, _P, _P], _I),
    "cbq_quantize_weights": ([_P, _I64, _I64, _P, _P], _I),
    "cbq_hc_sinkhorn": ([_P, _I64, _I, _P, _P], _I),
    "cbq_matmat": ([_P, _P, _I, _P, _P], _I),
    "cbq_debug_mmq_block_dots": ([_P, _P, _I, _P, _P], _I),
    "cbq_moe_matvec_logits": ([_P, _P, _I, _P, _I, _I, _P, _P], _I),
    "cbq_weights_get_error": ([_P, _P, ctypes.POINTER(ctypes.c_uint)], _I),
    "cbq_moe_get_error": ([_P, _P, ctypes.POINTER(ctypes.c_uint)], _I),
    "cbq_moe_debug_stall": ([_P, _I], _I),
    "cbq_debug_mmq_stall": ([_P, _I], _I),
    "cbq_debug_block_dots": ([_P, _P, _I, _P, _P], _I),
    "cbq_moe_debug_block_dots": ([_P, _I, _I, _P, _I, _P, _P], _I),
    "cbq_moe_set_debug": ([_P, _I], _I),
    "cbq_moe_set_stage_events": ([_P, _P, _P, _P], _I),
    "cbq_moe_debug_intermediate": ([_P, _I, _P, _P, _P, _P], _I),
}

_lib = None


class CbqError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = load()
        msg = lib.cbq_status_string(status).decode()
        cuda = lib.cbq_last_cuda_error().decode()
        super().__init__(f"{where}: {msg}" + (f" [{cuda}]" if cuda else ""))
        self.status = status


def header_functions() -> list[str]:
    """Names of the functions include/cbq.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:int|const char \*)\s*(cbq_\w+)\s*\(", text, re.M)))


def load():
    """Load libcbq.so; raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python -m verify_matvec_gb300.build`; "
                          "this package has no CPU path")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (args, res) in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _check(status: int, where: str):
    if status != CBQ_OK:
        raise CbqError(status, where)


# ----------------------------------------------------------- marshalling --

def _torch():
    import torch
    return torch


def _dev_ptr(t, dtype, name):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _host_ptr(a: np.ndarray, dtype, name):
    if not isinstance(a, np.ndarray) or a.dtype != dtype or not a.flags["C_CONTIGUOUS"]:
        raise TypeError(f"{name} must be a C-contiguous numpy {np.dtype(dtype).name} array")
    return a.ctypes.data_as(ctypes.c_void_p)


# ----------------------------------------------------------------- handles --

class Weights:
    """cbq_weights: one dense M x K codebook-4bit matrix on the device."""

    def __init__(self, blocks, M: int, K: int, stream=None):
        torch = _torch()
        lib = load()
        h = ctypes.c_void_p()
        if isinstance(blocks, torch.Tensor):
            if blocks.numel() != M * (K // CBQ_QK) * CBQ_BLOCK_BYTES:
                raise ValueError("blocks do not match M x K")
            ptr, on_dev = _dev_ptr(blocks, torch.uint8, "blocks"), 1
        else:
            blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
            if blocks.size != M * (K // CBQ_QK) * CBQ_BLOCK_BYTES:
                raise ValueError("blocks do not match M x K")
            ptr, on_dev = blocks.ctypes.data_as(ctypes.c_void_p), 0
        _check(lib.cbq_weights_create(ptr, M, K, on_dev, _stream(stream), ctypes.byref(h)), "cbq_weights_create")
        self._h = h
        self.M, self.K = M, K

    @property
    def handle(self):
        if self._h is None:
            raise ValueError("destroyed handle")
        return self._h

    def device_bytes(self) -> int:
        b = ctypes.c_int64()
        _check(load().cbq_weights_info(self.handle, None, None, ctypes.byref(b)), "cbq_weights_info")
        return b.value

    def close(self):
        if getattr(self, "_h", None) is not None:
            load().cbq_weights_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Moe:
    """cbq_moe: E experts, each a stacked gate_up (2F x H) and a down (H x F)."""

    def __init__(self, gate_up, down, E: int, H: int, F: int, stream=None):
        torch = _torch()
        lib = load()
        h = ctypes.c_void_p()
        if isinstance(gate_up, torch.Tensor):
            p1, p2, on_dev = _dev_ptr(gate_up, torch.uint8, "gate_up"), _dev_ptr(down, torch.uint8, "down"), 1
        else:
            gate_up = np.ascontiguousarray(gate_up, dtype=np.uint8)
            down = np.ascontiguousarray(down, dtype=np.uint8)
            p1, p2, on_dev = gate_up.ctypes.data_as(_P), down.ctypes.data_as(_P), 0
        nbH, nbF = H // CBQ_QK, F // CBQ_QK
        n_gu = gate_up.numel() if isinstance(gate_up, torch.Tensor) else gate_up.size
        n_dn = down.numel() if isinstance(down, torch.Tensor) else down.size
        if n_gu != E * 2 * F * nbH * CBQ_BLOCK_BYTES or n_dn != E * H * nbF * CBQ_BLOCK_BYTES:
            raise ValueError("expert blocks do not match E, H, F")
        _check(lib.cbq_moe_create(p1, p2, E, H, F, on_dev, _stream(stream), ctypes.byref(h)), "cbq_moe_create")
        self._h = h
        self.E, self.H, self.F = E, H, F
        self.shared = False

    @property
    def handle(self):
        if self._h is None:
            raise ValueError("destroyed handle")
        return self._h

    def set_shared(self, gate_up, down, stream=None):
        """cbq_moe_set_shared: a shared expert of the layer's shapes (blocks of
        one gate_up 2F x H and one down H x F), or None, None to remove it."""
        if (gate_up is None) != (down is None):
            raise ValueError("pass both gate_up and down blocks, or neither to remove the shared expert")
        torch = _torch()
        lib = load()
        if gate_up is None:
            _check(lib.cbq_moe_set_shared(self.handle, None, None, 0, _stream(stream)), "cbq_moe_set_shared")
            self.shared = False
            return
        nbH, nbF = self.H // CBQ_QK, self.F // CBQ_QK
        if isinstance(gate_up, torch.Tensor):
            p1, p2, on_dev = _dev_ptr(gate_up, torch.uint8, "gate_up"), _dev_ptr(down, torch.uint8, "down"), 1
            n_gu, n_dn = gate_up.numel(), down.numel()
        else:
            gate_up = np.ascontiguousarray(gate_up, dtype=np.uint8)
            down = np.ascontiguousarray(down, dtype=np.uint8)
            p1, p2, on_dev = gate_up.ctypes.data_as(_P), down.ctypes.data_as(_P), 0
            n_gu, n_dn = gate_up.size, down.size
        if n_gu != 2 * self.F * nbH * CBQ_BLOCK_BYTES or n_dn != self.H * nbF * CBQ_BLOCK_BYTES:
            raise ValueError("shared expert blocks do not match H, F")
        _check(lib.cbq_moe_set_shared(self.handle, p1, p2, on_dev, _stream(stream)), "cbq_moe_set_shared")
        self.shared = True

    def device_bytes(self) -> int:
        b = ctypes.c_int64()
        _check(load().cbq_moe_info(self.handle, None, None, None, ctypes.byref(b)), "cbq_moe_info")
        return b.value

    def close(self):
        if getattr(self, "_h", None) is not None:
            load().cbq_moe_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ----------------------------------------------------------- entry points --

def cbq_quantize_act(x, qx=None, dx=None, stream=None):
    """x: (n, K) float32 CUDA tensor -> (qx int8 (n, K), dx float32 (n, K/32))."""
    torch = _torch()
    x2 = x.reshape(-1, x.shape[-1])
    n, K = x2.shape
    if qx is None:
        qx = torch.empty((n, K), dtype=torch.int8, device=x.device)
    if dx is None:
        dx = torch.empty((n, K // CBQ_QK), dtype=torch.float32, device=x.device)
    _check(load().cbq_quantize_act(_dev_ptr(x2, torch.float32, "x"), K, n, _dev_ptr(qx, torch.int8, "qx"),
                                   _dev_ptr(dx, torch.float32, "dx"), _stream(stream)), "cbq_quantize_act")
    return qx, dx


def _y_out(y, n, M, device):
    torch = _torch()
    if y is None:
        y = torch.empty((n, M), dtype=torch.float32, device=device)
    return y


def cbq_matvec_q(W: Weights, qx, dx, y=None, stream=None):
    torch = _torch()
    n = qx.reshape(-1, W.K).shape[0]
    y = _y_out(y, n, W.M, qx.device)
    _check(load().cbq_matvec_q(W.handle, _dev_ptr(qx, torch.int8, "qx"), _dev_ptr(dx, torch.float32, "dx"), n,
                               _dev_ptr(y, torch.float32, "y"), _stream(stream)), "cbq_matvec_q")
    return y


def cbq_matvec(W: Weights, x, y=None, stream=None):
    torch = _torch()
    n = x.reshape(-1, W.K).shape[0]
    y = _y_out(y, n, W.M, x.device)
    _check(load().cbq_matvec(W.handle, _dev_ptr(x, torch.float32, "x"), n, _dev_ptr(y, torch.float32, "y"),
                             _stream(stream)), "cbq_matvec")
    return y


def cbq_matvec_static(W: Weights, x, y=None, stream=None):
    """cbq_matvec without touching the handle's workspace: the quantized
    activations go to the library's static per-device scratch (no device
    memory is allocated by this call)."""
    torch = _torch()
    n = x.reshape(-1, W.K).shape[0]
    y = _y_out(y, n, W.M, x.device)
    _check(load().cbq_matvec_static(W.handle, _dev_ptr(x, torch.float32, "x"), n, _dev_ptr(y, torch.float32, "y"),
                                    _stream(stream)), "cbq_matvec_static")
    return y


def cbq_matvec_host(W: Weights, x: np.ndarray, y: np.ndarray | None = None, stream=None):
    n = x.reshape(-1, W.K).shape[0]
    if y is None:
        y = np.empty((n, W.M), dtype=np.float32)
    _check(load().cbq_matvec_host(W.handle, _host_ptr(x, np.float32, "x"), n, _host_ptr(y, np.float32, "y"),
                                  _stream(stream)), "cbq_matvec_host")
    return y


def cbq_moe_matvec(L: Moe, h, ids, wts, swiglu: int = 1, y=None, stream=None):
    torch = _torch()
    n_tok, k = ids.shape
    if y is None:
        y = torch.empty((n_tok, L.H), dtype=torch.float32, device=h.device)
    _check(load().cbq_moe_matvec(L.handle, _dev_ptr(h, torch.float32, "h"), n_tok, _dev_ptr(ids, torch.int32, "ids"),
                                 _dev_ptr(wts, torch.float32, "wts"), k, int(swiglu),
                                 _dev_ptr(y, torch.float32, "y"), _stream(stream)), "cbq_moe_matvec")
    return y


def cbq_moe_set_shared(L: Moe, gate_up, down, stream=None):
    """Give L a shared expert (canonical blocks, host array or device tensor),
    or remove it with gate_up = down = None."""
    L.set_shared(gate_up, down, stream=stream)


def cbq_router_topk(logits, k: int, ids=None, wts=None, stream=None):
    """ids (n_tok, k) int32 and fp32 softmax weights of the k largest logits
    of each row of logits (n_tok, E) fp32, on the device."""
    torch = _torch()
    n_tok, E = logits.shape
    if ids is None:
        ids = torch.empty((n_tok, k), dtype=torch.int32, device=logits.device)
    if wts is None:
        wts = torch.empty((n_tok, k), dtype=torch.float32, device=logits.device)
    _check(load().cbq_router_topk(_dev_ptr(logits, torch.float32, "logits"), n_tok, E, k,
                                  _dev_ptr(ids, torch.int32, "ids"), _dev_ptr(wts, torch.float32, "wts"),
                                  _stream(stream)), "cbq_router_topk")
    return ids, wts


def cbq_moe_matvec_logits(L: Moe, h, logits, k: int, swiglu: int = 1, y=None, stream=None):
    """The routed layer from router logits (n_tok, E): top-k selection and
    softmax weights on the device, then cbq_moe_matvec."""
    torch = _torch()
    n_tok = logits.shape[0]
    if y is None:
        y = torch.empty((n_tok, L.H), dtype=torch.float32, device=h.device)
    _check(load().cbq_moe_matvec_logits(L.handle, _dev_ptr(h, torch.float32, "h"), n_tok,
                                        _dev_ptr(logits, torch.float32, "logits"), k, int(swiglu),
                                        _dev_ptr(y, torch.float32, "y"), _stream(stream)), "cbq_moe_matvec_logits")
    return y


def cbq_moe_matvec_host(L: Moe, h: np.ndarray, ids: np.ndarray, wts: np.ndarray, swiglu: int = 1,
                        y: np.ndarray | None = None, stream=None):
    n_tok, k = ids.shape
    if y is None:
        y = np.empty((n_tok, L.H), dtype=np.float32)
    _check(load().cbq_moe_matvec_host(L.handle, _host_ptr(h, np.float32, "h"), n_tok,
                                      _host_ptr(ids, np.int32, "ids"), _host_ptr(wts, np.float32, "wts"), k,
                                      int(swiglu), _host_ptr(y, np.float32, "y"), _stream(stream)),
           "cbq_moe_matvec_host")
    return y


def cbq_weights_get_error(W: Weights, stream=None) -> int:
    """Read and clear W's error word (CBQ_DEVERR_* bits) in the order of the
    stream (default: torch's current stream), then wait for that stream."""
    code = ctypes.c_uint()
    _check(load().cbq_weights_get_error(W.handle, _stream(stream), ctypes.byref(code)), "cbq_weights_get_error")
    return code.value


def cbq_moe_get_error(L: Moe, stream=None) -> int:
    """Read and clear L's error word (CBQ_DEVERR_* bits) in stream order."""
    code = ctypes.c_uint()
    _check(load().cbq_moe_get_error(L.handle, _stream(stream), ctypes.byref(code)), "cbq_moe_get_error")
    return code.value


def cbq_moe_debug_stall(L: Moe, mode: int):
    """Give-up test mode of the layer kernel (0 off; 1 a dependency never met;
    2 a weight stage never filled)."""
    _check(load().cbq_moe_debug_stall(L.handle, int(mode)), "cbq_moe_debug_stall")


def cbq_debug_mmq_stall(W: Weights, mode: int):
    """Give-up test mode of the tensor-core path (0 off; 1 the first CTA
    copies nothing, so its waits run out)."""
    _check(load().cbq_debug_mmq_stall(W.handle, int(mode)), "cbq_debug_mmq_stall")


def cbq_debug_block_dots(W: Weights, qx, s=None, stream=None):
    torch = _torch()
    n = qx.reshape(-1, W.K).shape[0]
    if s is None:
        s = torch.empty((n, W.M, W.K // CBQ_QK), dtype=torch.int32, device=qx.device)
    _check(load().cbq_debug_block_dots(W.handle, _dev_ptr(qx, torch.int8, "qx"), n, _dev_ptr(s, torch.int32, "s"),
                                       _stream(stream)), "cbq_debug_block_dots")
    return s


def cbq_moe_debug_block_dots(L: Moe, e: int, which: int, qx, s=None, stream=None):
    torch = _torch()
    M, K = (2 * L.F, L.H) if which == 0 else (L.H, L.F)
    n = qx.reshape(-1, K).shape[0]
    if s is None:
        s = torch.empty((n, M, K // CBQ_QK), dtype=torch.int32, device=qx.device)
    _check(load().cbq_moe_debug_block_dots(L.handle, e, which, _dev_ptr(qx, torch.int8, "qx"), n,
                                           _dev_ptr(s, torch.int32, "s"), _stream(stream)), "cbq_moe_debug_block_dots")
    return s


def cbq_moe_set_debug(L: Moe, keep: bool):
    _check(load().cbq_moe_set_debug(L.handle, int(bool(keep))), "cbq_moe_set_debug")


def cbq_moe_set_stage_events(L: Moe, events=None):
    """events: three torch.cuda.Event(enable_timing=True) or None to stop."""
    ptrs = [None] * 3 if events is None else [ctypes.c_void_p(ev.cuda_event) for ev in events]
    _check(load().cbq_moe_set_stage_events(L.handle, *ptrs), "cbq_moe_set_stage_events")


def cbq_moe_debug_intermediate(L: Moe, nslots: int, stream=None):
    torch = _torch()
    dev = torch.device("cuda", torch.cuda.current_device())
    a = torch.empty((nslots, L.F), dtype=torch.float32, device=dev)
    qa = torch.empty((nslots, L.F), dtype=torch.int8, device=dev)
    da = torch.empty((nslots, L.F // CBQ_QK), dtype=torch.float32, device=dev)
    _check(load().cbq_moe_debug_intermediate(L.handle, nslots, _dev_ptr(a, torch.float32, "a"),
                                             _dev_ptr(qa, torch.int8, "qa"), _dev_ptr(da, torch.float32, "da"),
                                             _stream(stream)), "cbq_moe_debug_intermediate")
    return a, qa, da


def cbq_quantize_weights(w, out=None, stream=None):
    """Canonical blocks (M, K/32, 18) uint8 of the fp32 matrix w (M, K), both
    on the device (the weight converter)."""
    torch = _torch()
    M, K = w.shape
    if out is None:
        out = torch.empty((M, K // CBQ_QK, CBQ_BLOCK_BYTES), dtype=torch.uint8, device=w.device)
    if not out.is_contiguous() or out.dtype != torch.uint8 or out.numel() != M * (K // CBQ_QK) * CBQ_BLOCK_BYTES:
        raise ValueError("out must be a contiguous uint8 tensor of M x K/32 x 18 bytes")
    _check(load().cbq_quantize_weights(_dev_ptr(w, torch.float32, "w"), M, K, ctypes.c_void_p(out.data_ptr()),
                                       _stream(stream)), "cbq_quantize_weights")
    return out


def cbq_hc_sinkhorn(logits, iters, out=None, stream=None):
    """Sinkhorn normalisation of the fp32 hyper-connection logits (..., 4, 4)
    on the device: exp(c - max c), then `iters` rounds of row and column
    normalisation; out (same shape) may be logits itself."""
    torch = _torch()
    if logits.dim() < 2 or tuple(logits.shape[-2:]) != (CBQ_HC_NHC, CBQ_HC_NHC):
        raise ValueError(f"logits must end in ({CBQ_HC_NHC}, {CBQ_HC_NHC})")
    if out is None:
        out = torch.empty_like(logits)
    if out.shape != logits.shape:
        raise ValueError("out must have the shape of logits")
    n = logits.numel() // (CBQ_HC_NHC * CBQ_HC_NHC)
    _check(load().cbq_hc_sinkhorn(_dev_ptr(logits, torch.float32, "logits"), n, int(iters),
                                  _dev_ptr(out, torch.float32, "out"), _stream(stream)), "cbq_hc_sinkhorn")
    return out


def cbq_matmat(W: Weights, x, y=None, stream=None):
    """y (n, M) fp32 = W applied to the n <= 16 fp32 columns x (n, K), by the
    tensor-core path; x and y on the device."""
    torch = _torch()
    n = x.shape[0]
    if y is None:
        y = torch.empty((n, W.M), dtype=torch.float32, device=x.device)
    _check(load().cbq_matmat(W.handle, _dev_ptr(x, torch.float32, "x"), n, _dev_ptr(y, torch.float32, "y"),
                             _stream(stream)), "cbq_matmat")
    return y


def cbq_debug_mmq_block_dots(W: Weights, qx, stream=None):
    """The exact block dots (n, M, K/32) int32 of W with int8 columns qx (n, K), by the tensor-core path."""
    torch = _torch()
    n = qx.shape[0]
    s = torch.empty((n, W.M, W.K // CBQ_QK), dtype=torch.int32, device=qx.device)
    _check(load().cbq_debug_mmq_block_dots(W.handle, _dev_ptr(qx, torch.int8, "qx"), n,
                                           _dev_ptr(s, torch.int32, "s"), _stream(stream)), "cbq_debug_mmq_block_dots")
    return s
