"""fp64 CPU oracle for the Muser decode-FFN weight stream.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product path (the
CUDA library ``libmuser`` and its binding) must not, and never falls back to it.

The arithmetic lives in ``oracle.c`` (plain C, built with gcc, OpenMP over
output rows).  This module builds it, wraps it with ctypes and composes the
steps of one decode-FFN block and of a stack of blocks in the order the Muser
book gives them (Ch 10 Figure 10.1 boxes 11-13; Ch 19 §19.1, §19.5).

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
(hand-worked blocks, encoder round trips, closed forms, invariants, library
routines, the book's printed examples).  The multi-layer stack is pinned only
through its pinned steps: no published stack output exists.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

Q4_K = 12
Q5_K = 13
Q6_K = 14
QTYPES = {"q4_k": Q4_K, "q5_k": Q5_K, "q6_k": Q6_K}
BLOCK_BYTES = {Q4_K: 144, Q5_K: 176, Q6_K: 210}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc, -O2, strict IEEE, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class Ring(ctypes.Structure):
    _fields_ = [("capacity", ctypes.c_int64), ("len", ctypes.c_int64),
                ("origin_logical", ctypes.c_int64), ("origin_physical", ctypes.c_int64)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            D = ctypes.c_double
            L.orc_f16_to_f64.restype = D
            L.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
            L.orc_f32_to_f16.restype = ctypes.c_uint16
            L.orc_f32_to_f16.argtypes = [ctypes.c_float]
            L.orc_f16_to_f64_array.argtypes = [P, P, I64]
            L.orc_f32_to_f16_array.argtypes = [P, P, I64]
            L.orc_q4k_block.argtypes = [P, P]
            L.orc_q6k_block.argtypes = [P, P]
            L.orc_q5k_block.argtypes = [P, P]
            L.orc_q4k_scale_min.argtypes = [P, I, P, P]
            L.orc_dequantize.argtypes = [I, P, I64, I64, P]
            L.orc_qmatvec.argtypes = [I, P, I64, I64, P, I64, P]
            L.orc_qmatvec_rows.argtypes = [I, P, I64, I64, P, I64, P, I64, P]
            L.orc_rms_norm.argtypes = [P, P, I64, I64, D, P]
            L.orc_dual_tail.argtypes = [P, P, P, P, I64, I64, D, D, P, P]
            L.orc_silu.restype = D
            L.orc_silu.argtypes = [D]
            L.orc_softcap.restype = D
            L.orc_softcap.argtypes = [D, D, D]
            L.orc_scale_softcap.argtypes = [P, I64, D, D, P]
            L.orc_silu_mul.argtypes = [P, P, I64, P]
            L.orc_gate_up_silu.argtypes = [I, P, P, I64, I64, P, I64, P]
            L.orc_ring_append.argtypes = [ctypes.POINTER(Ring), I64, ctypes.POINTER(I64)]
            L.orc_kv_write.argtypes = [ctypes.POINTER(Ring), P, P, I64, I64, I, P, P, I64, I64,
                                       ctypes.POINTER(I64)]
            L.orc_kv_snapshot.argtypes = [ctypes.POINTER(Ring), P, P, I64, I64, I, I64, I64, P, P]
            L.orc_kv_restore.argtypes = [ctypes.POINTER(Ring), P, P, I64, I64, I, P, P, I64, I64]
            L.orc_num_threads.restype = I
            L.orc_set_num_threads.argtypes = [I]
            _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _qt(qtype):
    return QTYPES[qtype] if isinstance(qtype, str) else int(qtype)


def _check(rc):
    if rc != 0:
        raise ValueError(f"oracle call failed with status {rc}")


def num_threads() -> int:
    return lib().orc_num_threads()


def set_num_threads(n: int) -> None:
    lib().orc_set_num_threads(int(n))


# ------------------------------------------------------------------ binary16
def f16_to_f64(h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, np.float64)
    lib().orc_f16_to_f64_array(_p(h), _p(out), h.size)
    return out


def f32_to_f16(f: np.ndarray) -> np.ndarray:
    f = np.ascontiguousarray(f, dtype=np.float32)
    out = np.empty(f.shape, np.uint16)
    lib().orc_f32_to_f16_array(_p(f), _p(out), f.size)
    return out


# ------------------------------------------------------------------- blocks
def q4k_block(blk: np.ndarray) -> np.ndarray:
    blk = np.ascontiguousarray(blk, dtype=np.uint8)
    assert blk.size == 144
    out = np.empty(256, np.float32)
    lib().orc_q4k_block(_p(blk), _p(out))
    return out


def q5k_block(blk: np.ndarray) -> np.ndarray:
    blk = np.ascontiguousarray(blk, dtype=np.uint8)
    assert blk.size == 176
    out = np.empty(256, np.float32)
    lib().orc_q5k_block(_p(blk), _p(out))
    return out


def q6k_block(blk: np.ndarray) -> np.ndarray:
    blk = np.ascontiguousarray(blk, dtype=np.uint8)
    assert blk.size == 210
    out = np.empty(256, np.float32)
    lib().orc_q6k_block(_p(blk), _p(out))
    return out


def q4k_scale_min(packed12: np.ndarray, j: int):
    packed12 = np.ascontiguousarray(packed12, dtype=np.uint8)
    sc, mn = ctypes.c_int(), ctypes.c_int()
    lib().orc_q4k_scale_min(_p(packed12), j, ctypes.byref(sc), ctypes.byref(mn))
    return sc.value, mn.value


def dequantize(qtype, W: np.ndarray, rows: int, cols: int) -> np.ndarray:
    W = np.ascontiguousarray(W, dtype=np.uint8)
    out = np.empty((rows, cols), np.float32)
    _check(lib().orc_dequantize(_qt(qtype), _p(W), rows, cols, _p(out)))
    return out


# ------------------------------------------------------------------- matvec
def qmatvec(qtype, W: np.ndarray, rows: int, cols: int, x: np.ndarray) -> np.ndarray:
    """y[M, rows] = x[M, cols] . W^T, fp64 sums rounded to binary32."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    M = x.shape[0]
    y = np.empty((M, rows), np.float32)
    _check(lib().orc_qmatvec(_qt(qtype), _p(W), rows, cols, _p(x), M, _p(y)))
    return y


def qmatvec_rows(qtype, W: np.ndarray, rows: int, cols: int, ridx, x: np.ndarray) -> np.ndarray:
    """y[M, len(ridx)]: the matvec sums for the listed output rows only."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    ridx = np.ascontiguousarray(ridx, dtype=np.int64)
    M = x.shape[0]
    y = np.empty((M, ridx.size), np.float32)
    _check(lib().orc_qmatvec_rows(_qt(qtype), _p(W), rows, cols, _p(ridx), ridx.size, _p(x), M,
                                  _p(y)))
    return y


# -------------------------------------------------------------------- norms
def rms_norm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    M, n = x.shape
    out = np.empty_like(x)
    lib().orc_rms_norm(_p(x), _p(w), n, M, eps, _p(out))
    return out


def dual_tail(resid: np.ndarray, src: np.ndarray, w1: np.ndarray, w2: np.ndarray,
              eps1: float = 1e-8, eps2: float = 1e-5):
    """Returns (updated residual, next-norm output), both binary32 [M, n]."""
    resid = np.ascontiguousarray(np.atleast_2d(resid), dtype=np.float32)
    src = np.ascontiguousarray(np.atleast_2d(src), dtype=np.float32)
    w1 = np.ascontiguousarray(w1, dtype=np.float32)
    w2 = np.ascontiguousarray(w2, dtype=np.float32)
    M, n = resid.shape
    assert src.shape == (M, n)
    r_out = np.empty_like(resid)
    out = np.empty_like(resid)
    lib().orc_dual_tail(_p(resid), _p(src), _p(w1), _p(w2), n, M, eps1, eps2, _p(r_out), _p(out))
    return r_out, out


# --------------------------------------------------------------------- SiLU
# The LM head's logit scale and soft cap (Ch 10 Figure 10.1 box 15): x 0.196116
# (1/sqrt(26)), then 20 * tanh(l / 20).
LOGIT_SCALE = 0.196116
SOFTCAP = 20.0


def softcap(l: float, scale: float = LOGIT_SCALE, cap: float = SOFTCAP) -> float:
    return lib().orc_softcap(float(l), float(scale), float(cap))


def scale_softcap(logits: np.ndarray, scale: float = LOGIT_SCALE, cap: float = SOFTCAP) -> np.ndarray:
    l = np.ascontiguousarray(logits, dtype=np.float32)
    out = np.empty_like(l)
    lib().orc_scale_softcap(_p(l), l.size, float(scale), float(cap), _p(out))
    return out


def lm_head(qtype, W: np.ndarray, vocab: int, hidden: int, x: np.ndarray, scale: float = LOGIT_SCALE,
            cap: float = SOFTCAP) -> np.ndarray:
    """Ch 10 Figure 10.1 boxes 14-15: binary32 logits W . x, then scale and cap."""
    return scale_softcap(qmatvec(qtype, W, vocab, hidden, x), scale, cap)


def silu(z: float) -> float:
    return lib().orc_silu(float(z))


def silu_mul(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    b = np.ascontiguousarray(b, dtype=np.float32)
    assert a.shape == b.shape
    out = np.empty_like(a)
    lib().orc_silu_mul(_p(a), _p(b), a.size, _p(out))
    return out


def gate_up_silu(qtype, Wg, Wu, ffn: int, hidden: int, x: np.ndarray) -> np.ndarray:
    Wg = np.ascontiguousarray(Wg, dtype=np.uint8)
    Wu = np.ascontiguousarray(Wu, dtype=np.uint8)
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    M = x.shape[0]
    mid = np.empty((M, ffn), np.float32)
    _check(lib().orc_gate_up_silu(_qt(qtype), _p(Wg), _p(Wu), ffn, hidden, _p(x), M, _p(mid)))
    return mid


# ----------------------------------------------------- FFN block and stack
def down_tail(qtype, Wd, hidden: int, ffn: int, mid: np.ndarray, resid: np.ndarray, w1, w2,
              eps1: float = 1e-8, eps2: float = 1e-5):
    """Ch 19: p = W_down . mid, then the dual-eps tail.  Returns (p, resid', out)."""
    p = qmatvec(qtype, Wd, hidden, ffn, mid)
    r_out, out = dual_tail(resid, p, w1, w2, eps1, eps2)
    return p, r_out, out


def ffn_layer(x: np.ndarray, resid: np.ndarray, layer: dict, w_next: np.ndarray, hidden: int,
              ffn: int, down_qtype="q6_k", eps1: float = 1e-8, eps2: float = 1e-5):
    """One decode-FFN layer on its normed input x (Ch 10 Figure 10.1 boxes 11-13).

    mid = silu(Wg.x) * (Wu.x); p = Wd.mid; resid += w1*rms_norm(p, eps1);
    out = w_next * rms_norm(resid, eps2).  Returns (resid', out, mid, p).
    """
    mid = gate_up_silu("q4_k", layer["Wg"], layer["Wu"], ffn, hidden, x)
    p, r_out, out = down_tail(down_qtype, layer["Wd"], hidden, ffn, mid, resid, layer["w1"],
                              w_next, eps1, eps2)
    return r_out, out, mid, p


def ffn_block(resid: np.ndarray, w_in: np.ndarray, layer: dict, w_next: np.ndarray, hidden: int,
              ffn: int, down_qtype="q6_k", eps_norm: float = 1e-5, eps_post: float = 1e-8):
    """A whole decode-FFN block from the residual: the input RMSNorm (Ch 2 §2.6
    rms_norm, eps 1e-5) and then ffn_layer.  Returns (x, mid, p, resid', out)."""
    x = rms_norm(resid, w_in, eps_norm)
    r_out, out, mid, p = ffn_layer(x, resid, layer, w_next, hidden, ffn, down_qtype, eps_post,
                                   eps_norm)
    return x, mid, p, r_out, out


def ffn_stack(resid: np.ndarray, w_in0: np.ndarray, layers, w_nexts, hidden: int, ffn: int,
              down_qtype="q6_k", eps_norm: float = 1e-5, eps_post: float = 1e-8,
              keep_outputs: bool = False):
    """The layer loop of Ch 10 §10.3-§10.4: the entry norm runs once (layer 0);
    every later layer's normed input is the previous tail's second output, whose
    weight is that next layer's input norm (the output norm after the last).

    `layers` and `w_nexts` may be sequences or callables(layer_index).
    Returns (resid_final, out_final[, per-layer outputs])."""
    get_layer = layers if callable(layers) else (lambda i: layers[i])
    get_next = w_nexts if callable(w_nexts) else (lambda i: w_nexts[i])
    n_layers = len(layers) if not callable(layers) else None
    x = rms_norm(resid, w_in0, eps_norm)
    r = np.ascontiguousarray(np.atleast_2d(resid), dtype=np.float32)
    outs = []
    i = 0
    while n_layers is None or i < n_layers:
        L = get_layer(i)
        if L is None:
            break
        r, x, _, _ = ffn_layer(x, r, L, get_next(i), hidden, ffn, down_qtype, eps_post, eps_norm)
        if keep_outputs:
            outs.append((r.copy(), x.copy()))
        i += 1
    return (r, x, outs) if keep_outputs else (r, x)


# ------------------------------------------------------------------ KV ring
def ring_append(ring: Ring, position: int):
    w = ctypes.c_int64()
    rc = lib().orc_ring_append(ctypes.byref(ring), position, ctypes.byref(w))
    return rc, w.value


def kv_write(ring: Ring, key: np.ndarray, value: np.ndarray, kv_dim: int, head_dim: int,
             head_major: bool, k: np.ndarray, v: np.ndarray, position: int):
    """Appends len(k) rows; returns (status, first physical row written)."""
    k = np.ascontiguousarray(np.atleast_2d(k), dtype=np.float32)
    v = np.ascontiguousarray(np.atleast_2d(v), dtype=np.float32)
    assert key.dtype == np.uint16 and value.dtype == np.uint16
    first = ctypes.c_int64(-1)
    rc = lib().orc_kv_write(ctypes.byref(ring), _p(key), _p(value), kv_dim, head_dim,
                            int(bool(head_major)), _p(k), _p(v), position, k.shape[0],
                            ctypes.byref(first))
    return rc, first.value


def kv_snapshot(ring: Ring, key: np.ndarray, value: np.ndarray, kv_dim: int, head_dim: int,
                head_major: bool, first: int, count: int):
    """Ch 15 §15.6: live logical rows first..first+count-1 as token-major binary16
    rows; returns (status, k_rows, v_rows)."""
    assert key.dtype == np.uint16 and value.dtype == np.uint16
    kr = np.zeros((count, kv_dim), np.uint16)
    vr = np.zeros((count, kv_dim), np.uint16)
    rc = lib().orc_kv_snapshot(ctypes.byref(ring), _p(key), _p(value), kv_dim, head_dim,
                               int(bool(head_major)), first, count, _p(kr), _p(vr))
    return rc, kr, vr


def kv_restore(ring: Ring, key: np.ndarray, value: np.ndarray, kv_dim: int, head_dim: int,
               head_major: bool, k_rows: np.ndarray, v_rows: np.ndarray, origin: int) -> int:
    """Ch 15 §15.6: installs len(k_rows) logical rows from `origin` at rotation
    origin % capacity; updates `ring` on success.  Returns the status."""
    kr = np.ascontiguousarray(k_rows, dtype=np.uint16).reshape(-1, kv_dim)
    vr = np.ascontiguousarray(v_rows, dtype=np.uint16).reshape(-1, kv_dim)
    assert kr.shape == vr.shape
    return lib().orc_kv_restore(ctypes.byref(ring), _p(key), _p(value), kv_dim, head_dim,
                                int(bool(head_major)), _p(kr), _p(vr), origin, kr.shape[0])
