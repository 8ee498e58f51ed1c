"""Seeded synthetic inputs for the decode-FFN weight stream.

This module is shared by the parity tests, the CPU oracle runs and ``bench.py``.
It draws bytes and numbers and nothing else: it holds none of the method's
arithmetic (no dequantisation, no matvec, no normalisation, no SiLU).  Where a
workload needs a derived input, e.g. the FFN intermediate silu(a)*b, the
generator returns the raw factors and each side computes the derived value
with its own code.

Block field positions follow the super-block layouts the Muser book describes
("How to Write an Inference Engine", Ch 19 §19.3: Q4_K is 144 bytes and Q6_K is
210 bytes per 256 weights).  Only where a field sits in the block is used here:

* Q4_K: bytes [0,2) f16 d, [2,4) f16 dmin, [4,16) the twelve bytes that pack
  eight 6-bit sub-block scales and eight 6-bit mins, [16,144) 128 bytes of
  4-bit codes.  Every one of the 96 bits of the packed scale bytes belongs to
  exactly one 6-bit field, and every code byte holds two 4-bit codes, so
  "every 6-bit scale/min and every 4-bit code uniform" is the same thing as
  "those bytes uniform": the generator draws uniform bytes.
* Q6_K: bytes [0,128) low 4-bit code nibbles, [128,192) high 2-bit code
  fields, [192,208) sixteen int8 sub-block scales, [208,210) f16 d.  Uniform
  nibbles and 2-bit fields are again uniform bytes.

Randomness: numpy's PCG64 bit generator seeded from a SeedSequence built from
(base seed, workload id, layer, tensor id).  PCG64's raw output is platform
independent, so the x86 development host and the aarch64 GPU host draw the
same bytes.
"""
from __future__ import annotations

import numpy as np

Q4K_BLOCK_BYTES = 144
Q6K_BLOCK_BYTES = 210
Q5K_BLOCK_BYTES = 176
QK = 256  # weights per super-block

# tensor ids inside one layer's stream family
T_GATE, T_UP, T_DOWN = 0, 1, 2
T_X, T_RESID, T_W_IN, T_W1, T_W2, T_A, T_B, T_K, T_V = 10, 11, 12, 13, 14, 15, 16, 17, 18
# attention side of a layer: Q, K, V, gate and output projections, the
# attention output fed to o_proj, and the post-attention norm weight
T_WQ, T_WK, T_WV, T_WAG, T_WO, T_ATTN, T_W_POST_ATTN = 20, 21, 22, 23, 24, 25, 26


def _bitgen(seed, workload: int, layer: int, tensor: int) -> np.random.PCG64:
    return np.random.PCG64(np.random.SeedSequence([int(seed), int(workload), int(layer), int(tensor)]))


def _gen(seed, workload, layer, tensor) -> np.random.Generator:
    return np.random.Generator(_bitgen(seed, workload, layer, tensor))


def _uniform_bytes(bg: np.random.PCG64, n: int) -> np.ndarray:
    words = bg.random_raw((n + 7) // 8)
    return words.view(np.uint8)[:n]


def _f16_bits(values: np.ndarray) -> np.ndarray:
    """Round float64 draws to binary16 (numpy's conversion is round-to-nearest-even)."""
    return values.astype(np.float16).view(np.uint16)


def q4k_matrix(rows: int, cols: int, *, seed=0, workload=0, layer=0, tensor=T_DOWN,
               d_range=(0.001, 0.01), dmin_range=(0.0, 0.005)) -> np.ndarray:
    """A Q4_K matrix as uint8[rows, cols/256*144], rows of consecutive super-blocks.

    Field distributions: f16 d ~ U(d_range), f16 dmin ~ U(dmin_range), 6-bit
    scales and mins uniform on 0..63, 4-bit codes uniform on 0..15.
    """
    if cols % QK:
        raise ValueError("cols must be a multiple of 256")
    nb = rows * (cols // QK)
    bg = _bitgen(seed, workload, layer, tensor)
    blk = _uniform_bytes(bg, nb * Q4K_BLOCK_BYTES).reshape(nb, Q4K_BLOCK_BYTES).copy()
    g = np.random.Generator(bg)
    d = _f16_bits(g.uniform(d_range[0], d_range[1], nb))
    dmin = _f16_bits(g.uniform(dmin_range[0], dmin_range[1], nb))
    blk[:, 0:2] = d.view(np.uint8).reshape(nb, 2)
    blk[:, 2:4] = dmin.view(np.uint8).reshape(nb, 2)
    return blk.reshape(rows, (cols // QK) * Q4K_BLOCK_BYTES)


def q5k_matrix(rows: int, cols: int, *, seed=0, workload=0, layer=0, tensor=T_DOWN,
               d_range=(0.001, 0.01), dmin_range=(0.0, 0.005)) -> np.ndarray:
    """A Q5_K matrix as uint8[rows, cols/256*176]: Q4_K's field distributions
    (f16 d, dmin, uniform 6-bit scales and mins) with 5-bit codes uniform on
    0..31 (uniform code and fifth-bit bytes)."""
    if cols % QK:
        raise ValueError("cols must be a multiple of 256")
    nb = rows * (cols // QK)
    bg = _bitgen(seed, workload, layer, tensor)
    blk = _uniform_bytes(bg, nb * Q5K_BLOCK_BYTES).reshape(nb, Q5K_BLOCK_BYTES).copy()
    g = np.random.Generator(bg)
    d = _f16_bits(g.uniform(d_range[0], d_range[1], nb))
    dmin = _f16_bits(g.uniform(dmin_range[0], dmin_range[1], nb))
    blk[:, 0:2] = d.view(np.uint8).reshape(nb, 2)
    blk[:, 2:4] = dmin.view(np.uint8).reshape(nb, 2)
    return blk.reshape(rows, (cols // QK) * Q5K_BLOCK_BYTES)


def q6k_matrix(rows: int, cols: int, *, seed=0, workload=0, layer=0, tensor=T_DOWN,
               d_range=(0.0005, 0.005), scale_range=(-32, 31)) -> np.ndarray:
    """A Q6_K matrix as uint8[rows, cols/256*210].

    Field distributions: 4-bit low codes and 2-bit high codes uniform, the 16
    int8 sub-block scales uniform integers on scale_range (inclusive), f16 d ~
    U(d_range).
    """
    if cols % QK:
        raise ValueError("cols must be a multiple of 256")
    nb = rows * (cols // QK)
    bg = _bitgen(seed, workload, layer, tensor)
    blk = _uniform_bytes(bg, nb * Q6K_BLOCK_BYTES).reshape(nb, Q6K_BLOCK_BYTES).copy()
    g = np.random.Generator(bg)
    sc = g.integers(scale_range[0], scale_range[1] + 1, size=(nb, 16), dtype=np.int64).astype(np.int8)
    blk[:, 192:208] = sc.view(np.uint8)
    d = _f16_bits(g.uniform(d_range[0], d_range[1], nb))
    blk[:, 208:210] = d.view(np.uint8).reshape(nb, 2)
    return blk.reshape(rows, (cols // QK) * Q6K_BLOCK_BYTES)


def qmatrix(qtype: str, rows: int, cols: int, **kw) -> np.ndarray:
    if qtype == "q4_k":
        return q4k_matrix(rows, cols, **kw)
    if qtype == "q5_k":
        return q5k_matrix(rows, cols, **kw)
    if qtype == "q6_k":
        return q6k_matrix(rows, cols, **kw)
    raise ValueError(qtype)


def normal(shape, *, seed=0, workload=0, layer=0, tensor=T_X) -> np.ndarray:
    """f32 draws from N(0, 1)."""
    return _gen(seed, workload, layer, tensor).standard_normal(shape, dtype=np.float32)


def norm_weight(n: int, *, seed=0, workload=0, layer=0, tensor=T_W1) -> np.ndarray:
    """f32 RMSNorm weight ~ 1 + N(0, 0.1)."""
    g = _gen(seed, workload, layer, tensor)
    return (1.0 + 0.1 * g.standard_normal(n)).astype(np.float32)


def ffn_mid_factors(n: int, M: int = 1, *, seed=0, workload=0, layer=0):
    """The two N(0,1) f32 factors (a, b) of an FFN intermediate silu(a)*b.

    The product itself is computed by each consumer with its own SiLU.
    """
    a = normal((M, n), seed=seed, workload=workload, layer=layer, tensor=T_A)
    b = normal((M, n), seed=seed, workload=workload, layer=layer, tensor=T_B)
    return a, b


# ---------------------------------------------------------------- workloads
HIDDEN = 6656
FFN = 19968
N_LAYERS = 52
EPS_POST = 1e-8
EPS_NORM = 1e-5

WORKLOADS = {
    # id: description
    0: "q4k_matvec_512x2048",
    1: "q4k_down_6656x19968_tail",
    2: "q6k_down_6656x19968_tail",
    3: "ffn_block_m1",
    4: "ffn_stack52_m16",
    5: "kv_ring_rows",
    6: "attn_projections_m1_m16",
    7: "lm_head_202048x6656",
}


def matvec_case(rows=512, cols=2048, M=1, qtype="q4_k", *, seed=0, workload=0):
    """Workload 0 shape by default: one quantized matrix and an N(0,1) input."""
    W = qmatrix(qtype, rows, cols, seed=seed, workload=workload, layer=0, tensor=T_DOWN)
    x = normal((M, cols), seed=seed, workload=workload, layer=0, tensor=T_X)
    return W, x


def down_tail_case(qtype="q4_k", hidden=HIDDEN, ffn=FFN, M=1, *, seed=0, workload=None, layer=0):
    """Workloads 1 and 2: W_down, the FFN intermediate factors, residual, norm weights."""
    if workload is None:
        workload = 1 if qtype == "q4_k" else 2
    W = qmatrix(qtype, hidden, ffn, seed=seed, workload=workload, layer=layer, tensor=T_DOWN)
    a, b = ffn_mid_factors(ffn, M, seed=seed, workload=workload, layer=layer)
    resid = normal((M, hidden), seed=seed, workload=workload, layer=layer, tensor=T_RESID)
    w1 = norm_weight(hidden, seed=seed, workload=workload, layer=layer, tensor=T_W1)
    w2 = norm_weight(hidden, seed=seed, workload=workload, layer=layer, tensor=T_W2)
    return dict(W=W, a=a, b=b, resid=resid, w1=w1, w2=w2)


def ffn_layer(layer: int, hidden=HIDDEN, ffn=FFN, *, seed=0, workload=3, down_qtype="q6_k"):
    """One FFN layer's weights: gate/up Q4_K [ffn x hidden], down [hidden x ffn], post-FFN norm."""
    Wg = q4k_matrix(ffn, hidden, seed=seed, workload=workload, layer=layer, tensor=T_GATE)
    Wu = q4k_matrix(ffn, hidden, seed=seed, workload=workload, layer=layer, tensor=T_UP)
    Wd = qmatrix(down_qtype, hidden, ffn, seed=seed, workload=workload, layer=layer, tensor=T_DOWN)
    w1 = norm_weight(hidden, seed=seed, workload=workload, layer=layer, tensor=T_W1)
    return dict(Wg=Wg, Wu=Wu, Wd=Wd, w1=w1)


# The attention-side projections of the Muser book's model (Ch 10 Figure 10.1
# boxes 4 and 9): Q and gate [6656 -> 4096], K and V [6656 -> 256], o_proj
# [4096 -> 6656].
Q_DIM = 4096
KV_DIM = 256
ATTN_WORKLOAD = 6


def attn_layer(layer: int, hidden=HIDDEN, *, seed=0, workload=ATTN_WORKLOAD):
    """One layer's attention-side weights, all Q4_K with the Q4_K field recipe,
    and its post-attention norm weight."""
    kw = dict(seed=seed, workload=workload, layer=layer)
    return dict(Wq=q4k_matrix(Q_DIM, hidden, tensor=T_WQ, **kw), Wk=q4k_matrix(KV_DIM, hidden, tensor=T_WK, **kw),
                Wv=q4k_matrix(KV_DIM, hidden, tensor=T_WV, **kw), Wg=q4k_matrix(Q_DIM, hidden, tensor=T_WAG, **kw),
                Wo=q4k_matrix(hidden, Q_DIM, tensor=T_WO, **kw),
                w_post=norm_weight(hidden, tensor=T_W_POST_ATTN, **kw))


def attn_output(M: int, layer: int = 0, *, seed=0, workload=ATTN_WORKLOAD):
    """A stand-in for the gated attention output that o_proj reads: N(0,1)
    f32 [M x 4096] (attention itself is outside this path)."""
    return normal((M, Q_DIM), seed=seed, workload=workload, layer=layer, tensor=T_ATTN)


def input_norm_weight(layer: int, hidden=HIDDEN, *, seed=0, workload=3):
    """Input (pre-FFN) norm weight of `layer`; layer == n_layers gives the output norm."""
    return norm_weight(hidden, seed=seed, workload=workload, layer=layer, tensor=T_W_IN)


def residual_rows(M: int, hidden=HIDDEN, *, seed=0, workload=3):
    return normal((M, hidden), seed=seed, workload=workload, layer=0, tensor=T_RESID)


def kv_rows(count: int, kv_dim: int, *, seed=0, workload=5, step=0):
    k = normal((count, kv_dim), seed=seed, workload=workload, layer=step, tensor=T_K)
    v = normal((count, kv_dim), seed=seed, workload=workload, layer=step, tensor=T_V)
    return k, v
