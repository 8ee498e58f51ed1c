"""Python binding of libmuser, the GB300 decode-FFN weight-streaming library.

Argument marshalling only: every step of the path runs in libmuser's CUDA
kernels (``csrc/``), reached through the C ABI declared in ``include/muser.h``.
PyTorch supplies device memory and streams.  There is no CPU fallback: if the
library is not built, every call raises.

The functions carry the C names.  Tensor arguments are torch tensors on the
current CUDA device (contiguous, the dtype the C ABI states); ``stream``
defaults to torch's current stream.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "MUSER_Q4_K", "MUSER_Q5_K", "MUSER_Q6_K", "QTYPES", "MuserError", "build", "library_path", "lib",
    "muser_version", "muser_last_error", "muser_block_bytes", "muser_matrix_bytes",
    "muser_dequantize", "muser_qmatvec", "muser_rms_norm", "muser_silu_mul",
    "muser_ffn_gate_up_silu", "muser_gate_up_scratch_bytes", "muser_ffn_gate_up_silu_scratch",
    "muser_qmatvec_scratch_bytes", "muser_qmatvec_scratch",
    "muser_ffn_gate_up_silu_tail", "muser_qmatvec_group", "muser_qmatvec_group_tail", "muser_scale_softcap",
    "muser_lm_head",
    "muser_fused_residual_dual_rmsnorm", "muser_scratch_bytes",
    "muser_qmatvec_residual_dual_rmsnorm", "muser_qmatvec_residual_dual_rmsnorm_static",
    "MUSER_STATIC_SCRATCH_BYTES", "MUSER_BOUNDARY_SCRATCH_BYTES", "FfnLayer", "muser_ffn_workspace_bytes", "muser_ffn_stack_launches",
    "muser_ffn_stack", "KvPlane", "muser_kv_ring_write", "muser_kv_snapshot", "muser_kv_restore", "muser_sync", "muser_debug_spin", "muser_debug_occupy",
    "muser_device_sm_count", "muser_device_status",
]

MUSER_Q4_K = 12
MUSER_Q5_K = 13
MUSER_Q6_K = 14
QTYPES = {"q4_k": MUSER_Q4_K, "q5_k": MUSER_Q5_K, "q6_k": MUSER_Q6_K}
MUSER_STATIC_SCRATCH_BYTES = 1 << 20
MUSER_BOUNDARY_SCRATCH_BYTES = 256
BLOCK_BYTES = {MUSER_Q4_K: 144, MUSER_Q5_K: 176, MUSER_Q6_K: 210}
STATUS = {0: "MUSER_OK", -1: "MUSER_ERR_INVALID_ARG", -2: "MUSER_ERR_UNSUPPORTED",
          -3: "MUSER_ERR_MISALIGNED", -4: "MUSER_ERR_CACHE_DISCONTINUITY", -5: "MUSER_ERR_CUDA",
          -6: "MUSER_ERR_TIMEOUT"}

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB = os.path.join(_PKG, "_build", "libmuser.so")
_lock = threading.Lock()
_lib = None


class MuserError(RuntimeError):
    def __init__(self, fn: str, status: int, message: str):
        super().__init__(f"{fn} -> {STATUS.get(status, status)}: {message}")
        self.status = status


def build(force: bool = False, verbose: bool = False) -> str:
    from . import buildlib as _b
    return _b.build(force=force, verbose=verbose)


def library_path() -> str:
    return _LIB


class FfnLayer(ctypes.Structure):
    _fields_ = [("w_gate", ctypes.c_void_p), ("w_up", ctypes.c_void_p), ("w_down", ctypes.c_void_p),
                ("post_norm", ctypes.c_void_p), ("next_norm", ctypes.c_void_p),
                ("gate_up_qtype", ctypes.c_int32), ("down_qtype", ctypes.c_int32)]


class KvPlane(ctypes.Structure):
    _fields_ = [("key", ctypes.c_void_p), ("value", ctypes.c_void_p), ("capacity", ctypes.c_int64),
                ("len", ctypes.c_int64), ("origin_logical", ctypes.c_int64),
                ("origin_physical", ctypes.c_int64), ("kv_dim", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("head_major", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


def lib():
    """The loaded libmuser (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB):
            raise RuntimeError(f"libmuser is not built ({_LIB} missing); call "
                               "quantized_weight_streaming_q4_gb300.build() first")
        L = ctypes.CDLL(_LIB)
        P, I, I64, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        sig = {
            "muser_version": (I, []),
            "muser_last_error": (ctypes.c_char_p, []),
            "muser_block_bytes": (SZ, [I]),
            "muser_matrix_bytes": (SZ, [I, I64, I64]),
            "muser_dequantize": (I, [I, P, I64, I64, P, P]),
            "muser_qmatvec": (I, [I, P, I64, I64, P, I, P, P]),
            "muser_qmatvec_scratch_bytes": (SZ, [I, I64, I64, I]),
            "muser_qmatvec_scratch": (I, [I, P, I64, I64, P, I, P, P, SZ, P]),
            "muser_rms_norm": (I, [P, P, P, I, I, F, P]),
            "muser_silu_mul": (I, [P, P, P, I64, P]),
            "muser_ffn_gate_up_silu": (I, [I, P, P, I64, I64, P, I, P, P]),
            "muser_gate_up_scratch_bytes": (SZ, [I, I64, I64, I]),
            "muser_ffn_gate_up_silu_scratch": (I, [I, P, P, I64, I64, P, I, P, P, SZ, P]),
            "muser_ffn_gate_up_silu_tail": (I, [I, P, P, I64, I64, P, P, P, P, P, F, F, P, I, P, P, SZ, P]),
            "muser_qmatvec_group": (I, [I, I, P, P, I64, P, I, P, P]),
            "muser_scale_softcap": (I, [P, I64, F, F, P]),
            "muser_lm_head": (I, [I, P, I64, I64, P, I, P, F, F, P]),
            "muser_qmatvec_group_tail": (I, [I, I, P, P, I64, P, P, P, P, P, F, F, P, I, P, P, SZ, P]),
    "muser_qmatvec_group_scratch_bytes": (SZ, [I, I, P, I64, I]),
    "muser_qmatvec_group_scratch": (I, [I, I, P, P, I64, P, I, P, P, SZ, P]),
            "muser_fused_residual_dual_rmsnorm": (I, [P, P, P, P, P, I, I, F, F, P]),
            "muser_scratch_bytes": (SZ, [I64, I]),
            "muser_qmatvec_residual_dual_rmsnorm": (I, [I, P, I64, I64, P, I, P, P, P, P, P, F, F, P,
                                                        SZ, P]),
            "muser_qmatvec_residual_dual_rmsnorm_static": (I, [I, P, I64, I64, P, I, P, P, P, P, F,
                                                               F, P]),
            "muser_ffn_workspace_bytes": (SZ, [I64, I64, I]),
            "muser_ffn_stack_launches": (I, [ctypes.POINTER(FfnLayer), I, I64, I64, I]),
            "muser_ffn_stack": (I, [ctypes.POINTER(FfnLayer), I, P, I64, I64, I, P, P, F, F, P, SZ,
                                    P]),
            "muser_kv_ring_write": (I, [ctypes.POINTER(KvPlane), P, P, I64, I64,
                                        ctypes.POINTER(I64), P]),
            "muser_kv_snapshot": (I, [ctypes.POINTER(KvPlane), I64, I64, P, P, P]),
            "muser_kv_restore": (I, [ctypes.POINTER(KvPlane), P, P, I64, I64, P]),
            "muser_sync": (I, [P, I]),
            "muser_debug_spin": (I, [I64, P]),
            "muser_debug_occupy": (I, [I, I64, P]),
            "muser_device_sm_count": (I, []),
            "muser_device_status": (ctypes.c_uint, [I]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
        return _lib


# ------------------------------------------------------------------ helpers
def _qt(qtype) -> int:
    return QTYPES[qtype] if isinstance(qtype, str) else int(qtype)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, rc: int) -> int:
    if rc != 0:
        msg = lib().muser_last_error()
        raise MuserError(fn, rc, msg.decode() if msg else "")
    return rc


# --------------------------------------------------------------- entry points
def muser_version() -> int:
    return lib().muser_version()


def muser_last_error() -> str:
    m = lib().muser_last_error()
    return m.decode() if m else ""


def muser_block_bytes(qtype) -> int:
    return lib().muser_block_bytes(_qt(qtype))


def muser_matrix_bytes(qtype, rows: int, cols: int) -> int:
    return lib().muser_matrix_bytes(_qt(qtype), rows, cols)


def muser_dequantize(qtype, W, rows: int, cols: int, out, stream=None) -> None:
    _check("muser_dequantize", lib().muser_dequantize(_qt(qtype), _ptr(W), rows, cols, _ptr(out),
                                                      _stream(stream)))


def muser_qmatvec(qtype, W, rows: int, cols: int, x, M: int, y, stream=None) -> None:
    _check("muser_qmatvec", lib().muser_qmatvec(_qt(qtype), _ptr(W), rows, cols, _ptr(x), M,
                                                _ptr(y), _stream(stream)))


def muser_qmatvec_scratch_bytes(qtype, rows: int, cols: int, M: int) -> int:
    return lib().muser_qmatvec_scratch_bytes(_qt(qtype), rows, cols, M)


def muser_qmatvec_scratch(qtype, W, rows: int, cols: int, x, M: int, y, scratch, scratch_bytes: int,
                          stream=None) -> None:
    _check("muser_qmatvec_scratch",
           lib().muser_qmatvec_scratch(_qt(qtype), _ptr(W), rows, cols, _ptr(x), M, _ptr(y), _ptr(scratch),
                                       scratch_bytes, _stream(stream)))


def muser_rms_norm(x, w, out, n: int, M: int, eps: float, stream=None) -> None:
    _check("muser_rms_norm", lib().muser_rms_norm(_ptr(x), _ptr(w), _ptr(out), n, M, eps,
                                                  _stream(stream)))


def muser_silu_mul(a, b, out, n: int, stream=None) -> None:
    _check("muser_silu_mul", lib().muser_silu_mul(_ptr(a), _ptr(b), _ptr(out), n, _stream(stream)))


def muser_ffn_gate_up_silu(qtype, Wg, Wu, ffn: int, hidden: int, x, M: int, mid, stream=None) -> None:
    _check("muser_ffn_gate_up_silu",
           lib().muser_ffn_gate_up_silu(_qt(qtype), _ptr(Wg), _ptr(Wu), ffn, hidden, _ptr(x), M,
                                        _ptr(mid), _stream(stream)))


def muser_gate_up_scratch_bytes(qtype, ffn: int, hidden: int, M: int) -> int:
    return lib().muser_gate_up_scratch_bytes(_qt(qtype), ffn, hidden, M)


def muser_ffn_gate_up_silu_scratch(qtype, Wg, Wu, ffn: int, hidden: int, x, M: int, mid, scratch,
                                   scratch_bytes: int, stream=None) -> None:
    _check("muser_ffn_gate_up_silu_scratch",
           lib().muser_ffn_gate_up_silu_scratch(_qt(qtype), _ptr(Wg), _ptr(Wu), ffn, hidden, _ptr(x), M,
                                                _ptr(mid), _ptr(scratch), scratch_bytes, _stream(stream)))


def muser_ffn_gate_up_silu_tail(qtype, Wg, Wu, ffn: int, hidden: int, projected, residual, w1, w2,
                                eps1: float, eps2: float, x_out, M: int, mid, scratch=None,
                                scratch_bytes: int = MUSER_BOUNDARY_SCRATCH_BYTES, residual_out=None,
                                stream=None) -> None:
    """residual_out=None updates `residual` in place (scratch: the ticket);
    otherwise the updated residual goes to residual_out."""
    _check("muser_ffn_gate_up_silu_tail",
           lib().muser_ffn_gate_up_silu_tail(_qt(qtype), _ptr(Wg), _ptr(Wu), ffn, hidden, _ptr(projected),
                                             _ptr(residual), _ptr(residual_out), _ptr(w1), _ptr(w2), eps1, eps2,
                                             _ptr(x_out), M, _ptr(mid), _ptr(scratch), scratch_bytes,
                                             _stream(stream)))


def muser_scale_softcap(logits, n: int, scale: float, cap: float, stream=None) -> None:
    _check("muser_scale_softcap", lib().muser_scale_softcap(_ptr(logits), n, scale, cap, _stream(stream)))


def muser_lm_head(qtype, W, vocab: int, hidden: int, x, M: int, logits, scale: float, cap: float,
                  stream=None) -> None:
    _check("muser_lm_head", lib().muser_lm_head(_qt(qtype), _ptr(W), vocab, hidden, _ptr(x), M, _ptr(logits),
                                                scale, cap, _stream(stream)))


def _group_arrays(Ws, rows, ys):
    n = len(Ws)
    if not (len(rows) == n == len(ys)):
        raise ValueError("one row count and one output per matrix")
    return (n, (ctypes.c_void_p * n)(*[_ptr(w) for w in Ws]), (ctypes.c_int64 * n)(*rows),
            (ctypes.c_void_p * n)(*[_ptr(y) for y in ys]))


def muser_qmatvec_group(qtype, Ws, rows, cols: int, x, M: int, ys, stream=None) -> None:
    n, wa, ra, ya = _group_arrays(Ws, rows, ys)
    _check("muser_qmatvec_group",
           lib().muser_qmatvec_group(_qt(qtype), n, wa, ra, cols, _ptr(x), M, ya, _stream(stream)))


def muser_qmatvec_group_scratch_bytes(qtype, rows, cols: int, M: int) -> int:
    n = len(rows)
    return int(lib().muser_qmatvec_group_scratch_bytes(_qt(qtype), n, (ctypes.c_int64 * n)(*rows), cols, M))


def muser_qmatvec_group_scratch(qtype, Ws, rows, cols: int, x, M: int, ys, scratch, scratch_bytes: int,
                                stream=None) -> None:
    n, wa, ra, ya = _group_arrays(Ws, rows, ys)
    _check("muser_qmatvec_group_scratch",
           lib().muser_qmatvec_group_scratch(_qt(qtype), n, wa, ra, cols, _ptr(x), M, ya, _ptr(scratch),
                                             scratch_bytes, _stream(stream)))


def muser_qmatvec_group_tail(qtype, Ws, rows, cols: int, projected, residual, w1, w2, eps1: float, eps2: float,
                             x_out, M: int, ys, scratch=None, scratch_bytes: int = MUSER_BOUNDARY_SCRATCH_BYTES,
                             residual_out=None, stream=None) -> None:
    n, wa, ra, ya = _group_arrays(Ws, rows, ys)
    _check("muser_qmatvec_group_tail",
           lib().muser_qmatvec_group_tail(_qt(qtype), n, wa, ra, cols, _ptr(projected), _ptr(residual),
                                          _ptr(residual_out), _ptr(w1), _ptr(w2), eps1, eps2, _ptr(x_out), M, ya,
                                          _ptr(scratch), scratch_bytes, _stream(stream)))


def muser_fused_residual_dual_rmsnorm(residual, src, out, w1, w2, n: int, M: int, eps1: float,
                                      eps2: float, stream=None) -> None:
    _check("muser_fused_residual_dual_rmsnorm",
           lib().muser_fused_residual_dual_rmsnorm(_ptr(residual), _ptr(src), _ptr(out), _ptr(w1),
                                                   _ptr(w2), n, M, eps1, eps2, _stream(stream)))


def muser_scratch_bytes(hidden: int, M: int) -> int:
    return lib().muser_scratch_bytes(hidden, M)


def muser_qmatvec_residual_dual_rmsnorm(qtype, Wdown, hidden: int, ffn: int, mid, M: int,
                                        projected, residual, out, w1, w2, eps1: float,
                                        eps2: float, scratch, scratch_bytes: int,
                                        stream=None) -> None:
    _check("muser_qmatvec_residual_dual_rmsnorm",
           lib().muser_qmatvec_residual_dual_rmsnorm(
               _qt(qtype), _ptr(Wdown), hidden, ffn, _ptr(mid), M, _ptr(projected),
               _ptr(residual), _ptr(out), _ptr(w1), _ptr(w2), eps1, eps2, _ptr(scratch),
               scratch_bytes, _stream(stream)))


def muser_qmatvec_residual_dual_rmsnorm_static(qtype, Wdown, hidden: int, ffn: int, mid, M: int,
                                               residual, out, w1, w2, eps1: float, eps2: float,
                                               stream=None) -> None:
    """As muser_qmatvec_residual_dual_rmsnorm, with the library's own fixed
    scratch in place of `projected` and `scratch` (see include/muser.h)."""
    _check("muser_qmatvec_residual_dual_rmsnorm_static",
           lib().muser_qmatvec_residual_dual_rmsnorm_static(
               _qt(qtype), _ptr(Wdown), hidden, ffn, _ptr(mid), M, _ptr(residual), _ptr(out),
               _ptr(w1), _ptr(w2), eps1, eps2, _stream(stream)))


def muser_ffn_workspace_bytes(hidden: int, ffn: int, M: int) -> int:
    return lib().muser_ffn_workspace_bytes(hidden, ffn, M)


def muser_ffn_stack_launches(layers, hidden: int, ffn: int, M: int) -> int:
    """Kernel launches one muser_ffn_stack call makes for these arguments."""
    if not isinstance(layers, ctypes.Array):
        layers = (FfnLayer * len(layers))(*layers)
    return lib().muser_ffn_stack_launches(layers, len(layers), hidden, ffn, M)


def muser_ffn_stack(layers, entry_norm, hidden: int, ffn: int, M: int, residual, out,
                    eps_norm: float, eps_post: float, workspace, workspace_bytes: int,
                    stream=None) -> None:
    """layers: a ctypes array of FfnLayer (host memory) or a list of FfnLayer."""
    if not isinstance(layers, ctypes.Array):
        layers = (FfnLayer * len(layers))(*layers)
    _check("muser_ffn_stack",
           lib().muser_ffn_stack(layers, len(layers), _ptr(entry_norm), hidden, ffn, M,
                                 _ptr(residual), _ptr(out), eps_norm, eps_post, _ptr(workspace),
                                 workspace_bytes, _stream(stream)))


def muser_kv_ring_write(plane: KvPlane, k, v, position: int, count: int, stream=None) -> int:
    """Appends `count` rows; returns the physical row of `position`."""
    first = ctypes.c_int64(-1)
    _check("muser_kv_ring_write",
           lib().muser_kv_ring_write(ctypes.byref(plane), _ptr(k), _ptr(v), position, count,
                                     ctypes.byref(first), _stream(stream)))
    return first.value


def muser_kv_snapshot(plane: KvPlane, first_logical: int, count: int, k_rows, v_rows,
                      stream=None) -> None:
    """Copies live logical rows first_logical..+count out as token-major binary16 rows."""
    _check("muser_kv_snapshot",
           lib().muser_kv_snapshot(ctypes.byref(plane), first_logical, count, _ptr(k_rows),
                                   _ptr(v_rows), _stream(stream)))


def muser_kv_restore(plane: KvPlane, k_rows, v_rows, origin_logical: int, length: int,
                     stream=None) -> None:
    """Installs `length` logical rows from origin_logical at rotation origin % capacity."""
    _check("muser_kv_restore",
           lib().muser_kv_restore(ctypes.byref(plane), _ptr(k_rows), _ptr(v_rows), origin_logical,
                                  length, _stream(stream)))


def muser_sync(stream=None, timeout_ms: int = -1) -> int:
    """Returns 0 or raises (MUSER_ERR_TIMEOUT is returned, not raised)."""
    rc = lib().muser_sync(_stream(stream), timeout_ms)
    if rc == -6:
        return rc
    return _check("muser_sync", rc)


def muser_debug_spin(microseconds: int, stream=None) -> None:
    _check("muser_debug_spin", lib().muser_debug_spin(microseconds, _stream(stream)))


def muser_debug_occupy(ctas: int, microseconds: int, stream=None) -> None:
    _check("muser_debug_occupy", lib().muser_debug_occupy(ctas, microseconds, _stream(stream)))


def muser_device_sm_count() -> int:
    return lib().muser_device_sm_count()


def muser_device_status(reset: bool = False) -> int:
    return lib().muser_device_status(1 if reset else 0)
