"""GPU parity of every libmuser entry point against the fp64 oracle, through
the C ABI, on seeded inputs that span several tiles and ragged tails.

Bit-exact: dequantised weights, one-hot matvec columns, K/V planes and ring
metadata.  Floating point: the path's bound (tests/gpu_util.py)."""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import assert_close, check_canary, dev, host, nan_like
from tests.kquant_pack import pack_q4k, pack_q5k, pack_q6k

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import quantized_weight_streaming_q4_gb300 as mu  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mu.build()
    mu.lib()
    torch.cuda.init()
    yield
    torch.cuda.synchronize()


def _qmatvec(qtype, W, rows, cols, x, canary=64):
    M = x.shape[0]
    Wd, xd = dev(W), dev(x)
    y = nan_like((M, rows), extra=canary)
    mu.muser_qmatvec(qtype, Wd, rows, cols, xd, M, y)
    out = host(y[:M * rows]).reshape(M, rows)
    check_canary(y, M * rows)
    return out


# ------------------------------------------------------------ dequantize
@pytest.mark.parametrize("qtype", ["q4_k", "q5_k", "q6_k"])
@pytest.mark.parametrize("rows,cols", [(1, 256), (37, 768), (512, 2048), (300, 6656)])
def test_dequantize_bit_exact(qtype, rows, cols):
    W = synth.qmatrix(qtype, rows, cols, seed=rows + cols)
    out = nan_like((rows, cols), extra=16)
    mu.muser_dequantize(qtype, dev(W), rows, cols, out)
    got = host(out[:rows * cols]).reshape(rows, cols)
    check_canary(out, rows * cols)
    ref = oracle.dequantize(qtype, W, rows, cols)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_dequantize_extreme_blocks_bit_exact():
    rng = np.random.default_rng(0)
    blocks4 = [pack_q4k(65504.0, 2.0 ** -24, [63] * 8, [63] * 8, list(range(16)) * 16),
               pack_q4k(2.0 ** -24, 65504.0, [63] * 8, [0] * 8, [15] * 256),
               pack_q4k(6.1e-5, 3.0e-7, rng.integers(0, 64, 8), rng.integers(0, 64, 8), rng.integers(0, 16, 256)),
               pack_q4k(0.0, 0.0, [5] * 8, [5] * 8, [7] * 256)]
    W4 = np.concatenate(blocks4).reshape(1, -1)
    out = nan_like((1, 1024))
    mu.muser_dequantize("q4_k", dev(W4), 1, 1024, out)
    assert np.array_equal(host(out).view(np.uint32), oracle.dequantize("q4_k", W4, 1, 1024).ravel().view(np.uint32))
    blocks6 = [pack_q6k(65504.0, [127] * 8 + [-128] * 8, list(range(64)) * 4),
               pack_q6k(2.0 ** -24, rng.integers(-128, 128, 16), rng.integers(0, 64, 256)),
               pack_q6k(1.0, [-128] * 16, [0] * 256)]
    W6 = np.concatenate(blocks6 + [blocks6[0]]).reshape(1, -1)
    out = nan_like((1, 1024))
    mu.muser_dequantize("q6_k", dev(W6), 1, 1024, out)
    assert np.array_equal(host(out).view(np.uint32), oracle.dequantize("q6_k", W6, 1, 1024).ravel().view(np.uint32))
    blocks5 = [pack_q5k(65504.0, 2.0 ** -24, [63] * 8, [63] * 8, list(range(32)) * 8),
               pack_q5k(2.0 ** -24, 65504.0, [63] * 8, [0] * 8, [31] * 256),
               pack_q5k(6.1e-5, 3.0e-7, rng.integers(0, 64, 8), rng.integers(0, 64, 8), rng.integers(0, 32, 256)),
               pack_q5k(0.0, 0.0, [5] * 8, [5] * 8, [17] * 256)]
    W5 = np.concatenate(blocks5).reshape(1, -1)
    out = nan_like((1, 1024))
    mu.muser_dequantize("q5_k", dev(W5), 1, 1024, out)
    assert np.array_equal(host(out).view(np.uint32), oracle.dequantize("q5_k", W5, 1, 1024).ravel().view(np.uint32))


# ---------------------------------------------------------------- matvec
@pytest.mark.parametrize("qtype", ["q4_k", "q5_k", "q6_k"])
@pytest.mark.parametrize("rows,cols", [(512, 2048), (37, 768), (5, 256), (1, 512), (997, 6656),
                                       (300, 19968)])
def test_qmatvec_m1(qtype, rows, cols):
    W = synth.qmatrix(qtype, rows, cols, seed=3 * rows + cols)
    x = synth.normal((1, cols), seed=rows, tensor=synth.T_X)
    got = _qmatvec(qtype, W, rows, cols, x)
    ref = oracle.qmatvec(qtype, W, rows, cols, x)
    assert_close(got, ref, f"{qtype} {rows}x{cols} M=1", scaled=True)


@pytest.mark.parametrize("qtype", ["q4_k", "q5_k", "q6_k"])
@pytest.mark.parametrize("cols", [26624, 26880])   # the one-token kernel's widest rows, and one block more
@pytest.mark.parametrize("M", [1, 16])
def test_qmatvec_width_limits(qtype, cols, M):
    rows = 37 if M == 1 else 64
    W = synth.qmatrix(qtype, rows, cols, seed=cols + M)
    x = synth.normal((M, cols), seed=cols, tensor=synth.T_X)
    got = _qmatvec(qtype, W, rows, cols, x)
    ref = oracle.qmatvec(qtype, W, rows, cols, x)
    assert_close(got, ref, f"{qtype} {rows}x{cols} M={M}", scaled=True)


@pytest.mark.parametrize("qtype", ["q4_k", "q5_k", "q6_k"])
def test_qmatvec_input_dynamic_range(qtype):
    # every 64-input slice takes its own power-of-two scale: slices 1e-30 to
    # 1e30 apart, all-zero slices, a slice with one nonzero input, binary32
    # subnormal inputs, and inputs of magnitude 1e30 (the kernels keep the
    # sums of each 32-input sub-block in binary32, times a 6-bit min)
    rows, cols = 96, 2048
    W = synth.qmatrix(qtype, rows, cols, seed=11)
    base = synth.normal((3, cols), seed=12, tensor=synth.T_X)
    x = base.copy()
    scales = np.float32(10.0) ** np.arange(-30, 32, 2, dtype=np.float32)
    for sl in range(cols // 64):
        x[0, 64 * sl:64 * sl + 64] *= scales[sl % scales.size]
    x[0, 0:64] = 0.0
    x[0, 128:192] = 0.0
    x[0, 130] = 3.0
    x[1] *= np.float32(1e-41)   # subnormal binary32 inputs
    x[2] *= np.float32(2e30)
    for m in range(3):
        got = _qmatvec(qtype, W, rows, cols, x[m:m + 1])
        ref = oracle.qmatvec(qtype, W, rows, cols, x[m:m + 1])
        assert np.isfinite(got).all()
        if m == 1:
            # the subnormal row: only the bound's absolute part is meaningful
            assert np.max(np.abs(got - ref)) <= 1e-30
        else:
            assert_close(got, ref, f"{qtype} dynamic range row {m}", scaled=True)


def test_qmatvec_q5k_full_shape_sampled_rows():
    # the bench's Q5_K launch: a 6656 x 19968 matrix at M = 1, every 23rd row
    # and the last one against the oracle
    rows, cols = 6656, 19968
    W = synth.q5k_matrix(rows, cols, seed=0, workload=3, layer=0)
    x = synth.normal((1, cols), seed=0, workload=3, tensor=synth.T_X)
    got = _qmatvec("q5_k", W, rows, cols, x)
    ridx = np.array(list(range(0, rows, 23)) + [rows - 1], np.int64)
    ref = oracle.qmatvec_rows("q5_k", W, rows, cols, ridx, x)
    assert_close(got[:, ridx], ref, "q5_k 6656x19968 sampled rows", scaled=True)


@pytest.mark.parametrize("qtype", ["q4_k", "q5_k", "q6_k"])
@pytest.mark.parametrize("M", [2, 3, 5, 8, 16])
@pytest.mark.parametrize("rows,cols", [(100, 768), (37, 2048)])
def test_qmatvec_multirow(qtype, M, rows, cols):
    W = synth.qmatrix(qtype, rows, cols, seed=M + rows)
    x = synth.normal((M, cols), seed=M, tensor=synth.T_X)
    got = _qmatvec(qtype, W, rows, cols, x)
    ref = oracle.qmatvec(qtype, W, rows, cols, x)
    assert_close(got, ref, f"{qtype} {rows}x{cols} M={M}", scaled=True)


@pytest.mark.parametrize("qtype,rows,cols", [("q4_k", 4096, 6656), ("q4_k", 256, 6656), ("q4_k", 6656, 4096),
                                            ("q4_k", 1000, 2048), ("q6_k", 6656, 19968), ("q6_k", 264, 1280),
                                            # enough units per SM for the prebuilt B image, with a partial last tile
                                            ("q4_k", 9999, 6656), ("q6_k", 6600, 19968)])
@pytest.mark.parametrize("M", [3, 16])
def test_qmatvec_scratch_split(qtype, rows, cols, M):
    # the attention-side shapes at several rows of x, split over every SM with
    # caller scratch; rows sampled against the oracle, the scratch left zeroed
    W = synth.qmatrix(qtype, rows, cols, seed=rows + M)
    x = synth.normal((M, cols), seed=M + 1, tensor=synth.T_X)
    nscr = mu.muser_qmatvec_scratch_bytes(qtype, rows, cols, M)
    assert nscr > 0
    scratch = torch.zeros(nscr // 4 + 64, dtype=torch.float32, device="cuda")
    scratch[nscr // 4:] = 777.0
    y = nan_like((M, rows), extra=64)
    Wd, xd = dev(W), dev(x)
    for _ in range(2):  # the second call runs on the scratch the first one left
        mu.muser_qmatvec_scratch(qtype, Wd, rows, cols, xd, M, y, scratch, nscr)
        got = host(y[:M * rows]).reshape(M, rows)
        check_canary(y, M * rows)
        ridx = np.unique(np.r_[np.arange(0, rows, max(1, rows // 200)), rows - 1])
        ref = oracle.qmatvec_rows(qtype, W, rows, cols, ridx, x)
        assert_close(got[:, ridx], ref, f"{qtype} {rows}x{cols} M={M} split", scaled=True)
        sc = host(scratch)
        assert not np.any(sc[:nscr // 4]), "scratch not left zeroed"
        assert np.all(sc[nscr // 4:] == 777.0), "write past the scratch"
    assert mu.muser_device_status() == 0


@pytest.mark.parametrize("qtype", ["q4_k", "q5_k", "q6_k"])
def test_qmatvec_one_hot_columns_bit_exact(qtype):
    # x = e_j picks column j of the dequantised matrix exactly (one product by
    # 1.0, every other term an exact zero), so every code and scale position
    # of the kernels' layout arithmetic is pinned against the oracle.
    rows, cols = 64, 768
    W = synth.qmatrix(qtype, rows, cols, seed=77)
    dense = oracle.dequantize(qtype, W, rows, cols)
    Wd = dev(W)
    y = nan_like((16, rows))
    js = list(range(0, cols, 5)) + [cols - 1]
    for j in js:  # M = 1 path
        x = np.zeros((1, cols), np.float32)
        x[0, j] = 1.0
        mu.muser_qmatvec(qtype, Wd, rows, cols, dev(x), 1, y)
        got = host(y[:rows])
        assert np.array_equal(got.view(np.uint32) & 0x7FFFFFFF, dense[:, j].view(np.uint32) & 0x7FFFFFFF), j
    for base in range(0, cols, 16):  # M = 16 path: sixteen one-hot rows at once
        x = np.zeros((16, cols), np.float32)
        for m in range(16):
            x[m, base + m] = 1.0
        mu.muser_qmatvec(qtype, Wd, rows, cols, dev(x), 16, y)
        got = host(y).reshape(16, rows)
        ref = dense[:, base:base + 16].T
        assert np.array_equal(got.view(np.uint32) & 0x7FFFFFFF, ref.view(np.uint32) & 0x7FFFFFFF), base


# ------------------------------------------------------- gate / up / SiLU
@pytest.mark.parametrize("M", [1, 4, 16])
@pytest.mark.parametrize("with_scratch", [False, True])
def test_ffn_gate_up_silu(M, with_scratch):
    """Without scratch the tensor-core kernel (M > 1) takes whole row tiles;
    with it the tiles' super-blocks split over SMs (ragged ffn in both)."""
    ffn, hidden = 2000 + M, 6656
    Wg = synth.q4k_matrix(ffn, hidden, seed=M, tensor=synth.T_GATE)
    Wu = synth.q4k_matrix(ffn, hidden, seed=M, tensor=synth.T_UP)
    x = oracle.rms_norm(synth.normal((M, hidden), seed=M), synth.norm_weight(hidden, seed=M), 1e-5)
    mid = nan_like((M, ffn), extra=32)
    if with_scratch:
        nscr = mu.muser_gate_up_scratch_bytes("q4_k", ffn, hidden, M)
        scratch = torch.zeros(max(nscr, 16) // 4, dtype=torch.float32, device="cuda")
        mu.muser_ffn_gate_up_silu_scratch("q4_k", dev(Wg), dev(Wu), ffn, hidden, dev(x), M, mid, scratch, nscr)
        assert not host(scratch).any(), "scratch must be left zeroed"
    else:
        mu.muser_ffn_gate_up_silu("q4_k", dev(Wg), dev(Wu), ffn, hidden, dev(x), M, mid)
    got = host(mid[:M * ffn]).reshape(M, ffn)
    check_canary(mid, M * ffn)
    ref = oracle.gate_up_silu("q4_k", Wg, Wu, ffn, hidden, x)
    assert_close(got, ref, f"gate_up_silu M={M}", scaled=True)


def boundary_case(M, ffn, hidden=6656):
    """Inputs of the fused layer boundary: gate/up, a residual row, a large
    projected row (as the down projection makes it) and the two norm weights."""
    Wg = synth.q4k_matrix(ffn, hidden, seed=40 + M, tensor=synth.T_GATE)
    Wu = synth.q4k_matrix(ffn, hidden, seed=40 + M, tensor=synth.T_UP)
    r = synth.normal((M, hidden), seed=41, tensor=synth.T_RESID)
    p = synth.normal((M, hidden), seed=41, tensor=synth.T_X) * np.float32(2.5e6)
    w1 = synth.norm_weight(hidden, seed=42, tensor=synth.T_W1)
    w2 = synth.norm_weight(hidden, seed=42, tensor=synth.T_W2)
    return Wg, Wu, r, p, w1, w2


def ticket_scratch():
    return torch.zeros(mu.MUSER_BOUNDARY_SCRATCH_BYTES // 4, dtype=torch.int32, device="cuda")


@pytest.mark.parametrize("M,ffn", [(1, 19968), (1, 2001), (3, 2003)])
@pytest.mark.parametrize("form", ["in_place", "residual_out"])
def test_ffn_gate_up_silu_tail(M, ffn, form):
    """The layer boundary: the previous tail then gate/up/SiLU.  One row of x
    runs the tail inside the gate/up kernel (every block computes x; in place,
    the block that takes the last ticket writes residual and x_out); M = 3
    runs the two calls.  With residual_out the input residual is left as it
    was."""
    hidden = 6656
    Wg, Wu, r, p, w1, w2 = boundary_case(M, ffn, hidden)
    rd, x_out, mid = dev(r), nan_like((M, hidden), extra=32), nan_like((M, ffn), extra=32)
    tk = ticket_scratch()
    r_out = nan_like((M, hidden), extra=32) if form == "residual_out" else None
    mu.muser_ffn_gate_up_silu_tail("q4_k", dev(Wg), dev(Wu), ffn, hidden, dev(p), rd, dev(w1), dev(w2),
                                   1e-8, 1e-5, x_out, M, mid, tk if r_out is None else None, residual_out=r_out)
    assert not host(tk).any(), "the ticket must be left zeroed"
    r_ref, x_ref = oracle.dual_tail(r, p, w1, w2, 1e-8, 1e-5)
    mid_ref = oracle.gate_up_silu("q4_k", Wg, Wu, ffn, hidden, x_ref)
    if r_out is not None:
        assert np.array_equal(host(rd).reshape(M, hidden), r), "residual_out form: the input row is read only"
        check_canary(r_out, M * hidden)
        rd = r_out[:M * hidden]
    assert_close(host(rd).reshape(M, hidden), r_ref, "tail residual")
    assert_close(host(x_out[:M * hidden]).reshape(M, hidden), x_ref, "tail x_out")
    assert_close(host(mid[:M * ffn]).reshape(M, ffn), mid_ref, f"gate_up_silu after the tail M={M}", scaled=True)
    check_canary(x_out, M * hidden)
    check_canary(mid, M * ffn)
    assert mu.muser_device_status() == 0


@pytest.mark.parametrize("M", [3, 16])
def test_ffn_gate_up_silu_scratch_b_image_ragged(M):
    """Gate/up with caller scratch at a row count whose units exceed 8 per SM
    (the B operand image path) and whose last tile is partial: equal to the
    oracle; the scratch (image region included) left zeroed and not overrun."""
    ffn, hidden = 9999, 6656
    Wg = synth.q4k_matrix(ffn, hidden, seed=M, tensor=synth.T_GATE)
    Wu = synth.q4k_matrix(ffn, hidden, seed=M, tensor=synth.T_UP)
    x = oracle.rms_norm(synth.normal((M, hidden), seed=M + 3), synth.norm_weight(hidden, seed=M + 3), 1e-5)
    nscr = mu.muser_gate_up_scratch_bytes("q4_k", ffn, hidden, M)
    scratch = torch.zeros(nscr // 4 + 64, dtype=torch.float32, device="cuda")
    scratch[nscr // 4:] = 777.0
    mid = nan_like((M, ffn), extra=32)
    mu.muser_ffn_gate_up_silu_scratch("q4_k", dev(Wg), dev(Wu), ffn, hidden, dev(x), M, mid, scratch, nscr)
    ref = oracle.gate_up_silu("q4_k", Wg, Wu, ffn, hidden, x)
    assert_close(host(mid[:M * ffn]).reshape(M, ffn), ref, f"gate_up_silu image path M={M}", scaled=True)
    check_canary(mid, M * ffn)
    sc = host(scratch)
    assert not np.any(sc[:nscr // 4]), "scratch not left zeroed"
    assert np.all(sc[nscr // 4:] == 777.0), "write past the scratch"
    assert mu.muser_device_status() == 0


def start_blocks_late(stream, ms=30):
    """Keep all but 8 SMs busy for `ms` on another stream (bounded), then let
    the host wait 5 ms so those blocks hold their SMs before anything else is
    enqueued: a one-block-per-SM kernel enqueued next on `stream` starts 8
    blocks at once and the rest about 25 ms later."""
    import time
    sms = mu.muser_device_sm_count()
    busy = torch.cuda.Stream()
    mu.muser_debug_occupy(1, 0, busy)       # loads the kernel before the timed use
    busy.synchronize()
    torch.cuda.synchronize()
    mu.muser_debug_occupy(max(1, sms - 8), ms * 1000, busy)
    time.sleep(0.005)
    return busy


@pytest.mark.parametrize("reps", [2])
@pytest.mark.parametrize("form", ["in_place", "residual_out"])
def test_ffn_gate_up_silu_tail_blocks_start_late(reps, form):
    """The fused boundary updates the residual in place while every block reads
    it.  With most blocks starting ~25 ms after the first ones, a block that
    read the already-updated row would add the tail twice: residual, x_out and
    mid must still equal the oracle's (Ch 19 §19.4: one update of `hidden`).
    Two calls in a row check that the ticket is left at zero."""
    M, ffn, hidden = 1, 19968, 6656
    Wg, Wu, r, p, w1, w2 = boundary_case(M, ffn, hidden)
    r_ref, x_ref = oracle.dual_tail(r, p, w1, w2, 1e-8, 1e-5)
    mid_ref = oracle.gate_up_silu("q4_k", Wg, Wu, ffn, hidden, x_ref)
    dWg, dWu, dp, dw1, dw2 = dev(Wg), dev(Wu), dev(p), dev(w1), dev(w2)
    tk = ticket_scratch()
    s = torch.cuda.current_stream()
    for call in range(reps):
        rd, x_out, mid = dev(r), nan_like((M, hidden)), nan_like((M, ffn))
        r_out = nan_like((M, hidden)) if form == "residual_out" else None
        busy = start_blocks_late(s)
        mu.muser_ffn_gate_up_silu_tail("q4_k", dWg, dWu, ffn, hidden, dp, rd, dw1, dw2, 1e-8, 1e-5, x_out, M,
                                       mid, tk, residual_out=r_out, stream=s)
        torch.cuda.synchronize()
        busy.synchronize()
        if r_out is not None:
            assert np.array_equal(host(rd).reshape(M, hidden), r)
            rd = r_out
        assert_close(host(rd).reshape(M, hidden), r_ref, f"residual with late blocks (call {call})")
        assert_close(host(x_out).reshape(M, hidden), x_ref, f"x_out with late blocks (call {call})")
        assert_close(host(mid).reshape(M, ffn), mid_ref, f"mid with late blocks (call {call})", scaled=True)
        assert not host(tk).any(), "the ticket must be left zeroed"
    assert mu.muser_device_status() == 0


@pytest.mark.parametrize("form", ["in_place", "residual_out"])
def test_group_tail_blocks_start_late(form):
    """The attention-side group with the previous tail in its launch, under
    the same late block starts: residual, x_out and the four projections."""
    H = 6656
    A = synth.attn_layer(2, H)
    names, rows = ("Wq", "Wk", "Wv", "Wg"), (synth.Q_DIM, synth.KV_DIM, synth.KV_DIM, synth.Q_DIM)
    r = synth.residual_rows(1, H, workload=synth.ATTN_WORKLOAD)
    p = synth.normal((1, H), seed=8, workload=synth.ATTN_WORKLOAD, tensor=synth.T_X) * np.float32(3e5)
    w1 = synth.norm_weight(H, seed=8, workload=synth.ATTN_WORKLOAD, tensor=synth.T_W1)
    w2 = synth.norm_weight(H, seed=8, workload=synth.ATTN_WORKLOAD, tensor=synth.T_W2)
    r_ref, x_ref = oracle.dual_tail(r, p, w1, w2, 1e-8, 1e-5)
    rd, x_out = dev(r), nan_like((1, H))
    ys = [nan_like((1, n)) for n in rows]
    tk = ticket_scratch()
    s = torch.cuda.current_stream()
    r_out = nan_like((1, H)) if form == "residual_out" else None
    busy = start_blocks_late(s)
    mu.muser_qmatvec_group_tail("q4_k", [dev(A[n]) for n in names], rows, H, dev(p), rd, dev(w1), dev(w2),
                                1e-8, 1e-5, x_out, 1, ys, tk, residual_out=r_out, stream=s)
    torch.cuda.synchronize()
    busy.synchronize()
    if r_out is not None:
        assert np.array_equal(host(rd).reshape(1, H), r)
        rd = r_out
    assert_close(host(rd).reshape(1, H), r_ref, "residual with late blocks")
    assert_close(host(x_out).reshape(1, H), x_ref, "x_out with late blocks")
    for name, n, y in zip(names, rows, ys):
        assert_close(host(y).reshape(1, n), oracle.qmatvec("q4_k", A[name], n, H, x_ref),
                     f"{name} with late blocks", scaled=True)
    assert not host(tk).any()
    assert mu.muser_device_status() == 0


def test_silu_mul_and_rms_norm():
    a, b = synth.ffn_mid_factors(19968, 3, seed=9)
    out = nan_like((3, 19968))
    mu.muser_silu_mul(dev(a), dev(b), out, a.size)
    assert_close(host(out).reshape(3, -1), oracle.silu_mul(a, b), "silu_mul")
    x = synth.normal((5, 6656), seed=10) * np.float32(7.0)
    w = synth.norm_weight(6656, seed=10)
    o = nan_like((5, 6656))
    mu.muser_rms_norm(dev(x), dev(w), o, 6656, 5, 1e-5)
    assert_close(host(o).reshape(5, -1), oracle.rms_norm(x, w, 1e-5), "rms_norm")


# ------------------------------------------------------------- dual tail
def test_tail_worked_example_from_book():
    r = dev(np.array([[1, 2, 3, 4]], np.float32))
    p = dev(np.array([[4, 0, 0, 0]], np.float32))
    ones = dev(np.ones(4, np.float32))
    out = nan_like((1, 4))
    mu.muser_fused_residual_dual_rmsnorm(r, p, out, ones, ones, 4, 1, 1e-8, 1e-5)
    np.testing.assert_allclose(host(r)[0], [3, 2, 3, 4], atol=1e-6)
    np.testing.assert_allclose(host(out), [0.973, 0.649, 0.973, 1.297], atol=1e-3)


@pytest.mark.parametrize("M,n", [(1, 6656), (16, 6656), (3, 4100)])
def test_fused_residual_dual_rmsnorm(M, n):
    r = synth.normal((M, n), seed=n + M, tensor=synth.T_RESID)
    p = synth.normal((M, n), seed=n + M, tensor=synth.T_X) * np.float32(2.5e6)
    w1 = synth.norm_weight(n, seed=M, tensor=synth.T_W1)
    w2 = synth.norm_weight(n, seed=M, tensor=synth.T_W2)
    rd, out = dev(r), nan_like((M, n))
    mu.muser_fused_residual_dual_rmsnorm(rd, dev(p), out, dev(w1), dev(w2), n, M, 1e-8, 1e-5)
    r_ref, out_ref = oracle.dual_tail(r, p, w1, w2, 1e-8, 1e-5)
    assert_close(host(rd), r_ref, "tail residual")
    assert_close(host(out).reshape(M, n), out_ref, "tail out")


def test_tail_zero_projection_keeps_residual_bit_exact():
    n = 6656
    r = synth.normal((2, n), seed=1, tensor=synth.T_RESID)
    rd = dev(r)
    out = nan_like((2, n))
    w = dev(synth.norm_weight(n, seed=1))
    mu.muser_fused_residual_dual_rmsnorm(rd, dev(np.zeros_like(r)), out, w, w, n, 2, 1e-8, 1e-5)
    assert np.array_equal(host(rd), r)


@pytest.mark.parametrize("qtype", ["q4_k", "q6_k"])
@pytest.mark.parametrize("M,small_scratch", [(1, False), (1, True), (3, False), (16, False)])
def test_down_projection_with_fused_tail(qtype, M, small_scratch):
    """M > 1 with full scratch runs the tensor-core kernel (tiles split over
    all SMs); M = 1, or the 256-byte minimum, the CUDA-core kernels."""
    hidden, ffn = 6656, 19968 if M == 1 else 2048
    case = synth.down_tail_case(qtype, hidden, ffn, M, seed=5)
    a, b = case["a"], case["b"]
    mid_d = nan_like((M, ffn))
    mu.muser_silu_mul(dev(a), dev(b), mid_d, a.size)
    mid_ref = oracle.silu_mul(a, b)
    Wd, w1, w2 = dev(case["W"]), dev(case["w1"]), dev(case["w2"])
    resid = dev(case["resid"])
    proj, out = nan_like((M, hidden)), nan_like((M, hidden))
    nscr = 256 if small_scratch else mu.muser_scratch_bytes(hidden, M)
    scratch = torch.zeros(nscr // 4 + 4, dtype=torch.float32, device="cuda")
    p_ref, r_ref, o_ref = oracle.down_tail(qtype, case["W"], hidden, ffn, mid_ref, case["resid"],
                                           case["w1"], case["w2"])
    mu.muser_qmatvec_residual_dual_rmsnorm(qtype, Wd, hidden, ffn, mid_d, M, proj, resid, out, w1,
                                           w2, 1e-8, 1e-5, scratch, nscr)
    assert_close(host(proj).reshape(M, hidden), p_ref, "projected", scaled=True)
    assert_close(host(resid), r_ref, "residual")
    assert_close(host(out).reshape(M, hidden), o_ref, "next-norm output")
    assert not host(scratch).any(), "scratch must be left zeroed"
    # a second call on the updated residual (scratch reuse) matches the oracle too
    _, r_ref2, o_ref2 = oracle.down_tail(qtype, case["W"], hidden, ffn, mid_ref, r_ref,
                                         case["w1"], case["w2"])
    mu.muser_qmatvec_residual_dual_rmsnorm(qtype, Wd, hidden, ffn, mid_d, M, proj, resid, out, w1,
                                           w2, 1e-8, 1e-5, scratch, nscr)
    assert_close(host(resid), r_ref2, "residual (second call)")
    assert_close(host(out).reshape(M, hidden), o_ref2, "output (second call)")
    assert mu.muser_device_status() == 0


# ---------------------------------------------------------------- KV ring
def _plane_pair(cap, kv_dim, head_dim, head_major):
    key = torch.full((cap * kv_dim,), 0xDEAD, dtype=torch.int32, device="cuda").to(torch.int16)
    val = key.clone()
    plane = mu.KvPlane(key.data_ptr(), val.data_ptr(), cap, 0, 0, 0, kv_dim, head_dim,
                       1 if head_major else 0, 0)
    ring = oracle.Ring(cap, 0, 0, 0)
    okey = np.full(cap * kv_dim, 0xDEAD, np.uint16)
    oval = okey.copy()
    return key, val, plane, ring, okey, oval


@pytest.mark.parametrize("head_major", [False, True])
@pytest.mark.parametrize("cap", [32, 2048])
def test_kv_ring_write_bit_exact(head_major, cap):
    kv_dim, head_dim = 256, 128
    key, val, plane, ring, okey, oval = _plane_pair(cap, kv_dim, head_dim, head_major)
    pos = 0
    counts = [1, 1, 30, 1, 1, 5, cap + 3, 1, 2]   # crosses the wrap, and one batch > capacity
    for step, count in enumerate(counts):
        k, v = synth.kv_rows(count, kv_dim, seed=step, step=step)
        k[0, :3] = [70000.0, -1e-9, 65519.0]  # overflow, underflow, tie cases
        first = mu.muser_kv_ring_write(plane, dev(k), dev(v), pos, count)
        rc, ofirst = oracle.kv_write(ring, okey, oval, kv_dim, head_dim, head_major, k, v, pos)
        assert rc == 0 and first == ofirst
        assert (plane.len, plane.origin_logical, plane.origin_physical) == (
            ring.len, ring.origin_logical, ring.origin_physical)
        pos += count
    assert np.array_equal(host(key).view(np.uint16), okey)
    assert np.array_equal(host(val).view(np.uint16), oval)


def test_kv_ring_discontinuity_leaves_planes_untouched():
    key, val, plane, ring, okey, oval = _plane_pair(32, 256, 128, False)
    k, v = synth.kv_rows(40, 256, seed=1)
    mu.muser_kv_ring_write(plane, dev(k), dev(v), 0, 40)
    before = (host(key).copy(), host(val).copy(), plane.len, plane.origin_logical, plane.origin_physical)
    for bad in (39, 41, 0):
        with pytest.raises(mu.MuserError) as ei:
            mu.muser_kv_ring_write(plane, dev(k[:1]), dev(v[:1]), bad, 1)
        assert ei.value.status == -4
    after = (host(key), host(val), plane.len, plane.origin_logical, plane.origin_physical)
    assert np.array_equal(before[0], after[0]) and np.array_equal(before[1], after[1])
    assert before[2:] == after[2:]


def _u16(t):
    return host(t).view(np.uint16)


def _rows_buf(n, kv_dim, offset=0, canary=24):
    """int16 device rows [n*kv_dim] starting `offset` halves into a buffer, canaries after."""
    buf = torch.full((offset + n * kv_dim + canary,), 0x7777, dtype=torch.int16, device="cuda")
    return buf, buf[offset:offset + n * kv_dim]


def _check_rows_canary(buf, offset, n, kv_dim):
    b = host(buf)
    assert np.all(b[:offset] == 0x7777) and np.all(b[offset + n * kv_dim:] == 0x7777)


@pytest.mark.parametrize("head_major", [False, True])
@pytest.mark.parametrize("cap,kv_dim,head_dim,offset", [(2048, 256, 128, 0), (37, 256, 128, 0),
                                                       (37, 256, 128, 1), (29, 6, 3, 0)])
def test_kv_snapshot_and_restore_bit_exact(head_major, cap, kv_dim, head_dim, offset):
    key, val, plane, ring, okey, oval = _plane_pair(cap, kv_dim, head_dim, head_major)
    pos = 0
    for step, count in enumerate([5, cap - 2, 3, cap // 3 + 1]):   # wraps, origins not 0
        k, v = synth.kv_rows(count, kv_dim, seed=40 + step, step=step)
        mu.muser_kv_ring_write(plane, dev(k), dev(v), pos, count)
        assert oracle.kv_write(ring, okey, oval, kv_dim, head_dim, head_major, k, v, pos)[0] == 0
        pos += count
    assert np.array_equal(_u16(key), okey) and plane.origin_logical == ring.origin_logical > 0
    o0, n = plane.origin_logical, plane.len
    # the whole window, and a sub-range that crosses the physical end of the plane
    split = (cap - plane.origin_physical) - 2
    for first, count in [(o0, n), (o0 + split, min(7, n - split)), (o0 + n - 1, 1)]:
        kb, kr = _rows_buf(count, kv_dim, offset)
        vb, vr = _rows_buf(count, kv_dim, offset)
        mu.muser_kv_snapshot(plane, first, count, kr, vr)
        rc, ok, ov = oracle.kv_snapshot(ring, okey, oval, kv_dim, head_dim, head_major, first, count)
        assert rc == 0
        assert np.array_equal(_u16(kr).reshape(count, kv_dim), ok)
        assert np.array_equal(_u16(vr).reshape(count, kv_dim), ov)
        _check_rows_canary(kb, offset, count, kv_dim)
        _check_rows_canary(vb, offset, count, kv_dim)
    # restore the whole window into a fresh plane pair, at its own origin and at another one
    kb, kr = _rows_buf(n, kv_dim, offset)
    vb, vr = _rows_buf(n, kv_dim, offset)
    mu.muser_kv_snapshot(plane, o0, n, kr, vr)
    _, ok, ov = oracle.kv_snapshot(ring, okey, oval, kv_dim, head_dim, head_major, o0, n)
    for origin in (o0, o0 + 5 * cap + 3, 0):
        key2 = torch.full((cap * kv_dim,), 0x3C3C, dtype=torch.int16, device="cuda")
        val2 = key2.clone()
        plane2 = mu.KvPlane(key2.data_ptr(), val2.data_ptr(), cap, 1, 9, 9, kv_dim, head_dim,
                            1 if head_major else 0, 0)
        ring2 = oracle.Ring(cap, 1, 9, 9)
        okey2 = np.full(cap * kv_dim, 0x3C3C, np.uint16)
        oval2 = okey2.copy()
        mu.muser_kv_restore(plane2, kr, vr, origin, n)
        assert oracle.kv_restore(ring2, okey2, oval2, kv_dim, head_dim, head_major, ok, ov, origin) == 0
        assert (plane2.len, plane2.origin_logical, plane2.origin_physical) == (
            ring2.len, ring2.origin_logical, ring2.origin_physical) == (n, origin, origin % cap)
        assert np.array_equal(_u16(key2), okey2) and np.array_equal(_u16(val2), oval2)
        if origin == o0:
            # restored at its own origin, the pair is the live one, slot for slot
            assert np.array_equal(okey2, okey) and np.array_equal(oval2, oval)
            # and it keeps appending as the live ring does
            k, v = synth.kv_rows(4, kv_dim, seed=77)
            mu.muser_kv_ring_write(plane2, dev(k), dev(v), o0 + n, 4)
            mu.muser_kv_ring_write(plane, dev(k), dev(v), o0 + n, 4)
            assert np.array_equal(_u16(key2), _u16(key)) and np.array_equal(_u16(val2), _u16(val))
            assert (plane2.len, plane2.origin_logical, plane2.origin_physical) == (
                plane.len, plane.origin_logical, plane.origin_physical)


@pytest.mark.parametrize("head_major,cap,n,origin", [(True, 131072, 130815, 0),        # a NoPE plane
                                                     (False, 2048, 2048, 128767)])     # a wrapped SWA ring
def test_kv_restore_full_session_plane(head_major, cap, n, origin):
    # the bench's session shapes (kv_dim 256, two KV heads of 128): the whole
    # plane pair against the oracle, byte for byte, and the snapshot back
    kv_dim, head_dim = 256, 128
    rng = np.random.default_rng(cap + n)
    kr = rng.integers(0, 1 << 16, (n, kv_dim), dtype=np.uint16)
    vr = rng.integers(0, 1 << 16, (n, kv_dim), dtype=np.uint16)
    key = torch.full((cap * kv_dim,), 0x1234, dtype=torch.int16, device="cuda")
    val = key.clone()
    plane = mu.KvPlane(key.data_ptr(), val.data_ptr(), cap, 0, 0, 0, kv_dim, head_dim, 1 if head_major else 0, 0)
    dk, dv = dev(kr.view(np.int16)), dev(vr.view(np.int16))
    mu.muser_kv_restore(plane, dk, dv, origin, n)
    ring = oracle.Ring(cap, 0, 0, 0)
    okey = np.full(cap * kv_dim, 0x1234, np.uint16)
    oval = okey.copy()
    assert oracle.kv_restore(ring, okey, oval, kv_dim, head_dim, head_major, kr, vr, origin) == 0
    assert (plane.len, plane.origin_logical, plane.origin_physical) == (
        ring.len, ring.origin_logical, ring.origin_physical)
    assert np.array_equal(_u16(key), okey) and np.array_equal(_u16(val), oval)
    back_k = torch.empty(n * kv_dim, dtype=torch.int16, device="cuda")
    back_v = torch.empty_like(back_k)
    mu.muser_kv_snapshot(plane, origin, n, back_k, back_v)
    assert np.array_equal(_u16(back_k).reshape(n, kv_dim), kr)
    assert np.array_equal(_u16(back_v).reshape(n, kv_dim), vr)


def test_kv_snapshot_and_restore_reject_without_writing():
    key, val, plane, ring, okey, oval = _plane_pair(32, 256, 128, True)
    k, v = synth.kv_rows(40, 256, seed=5)
    mu.muser_kv_ring_write(plane, dev(k), dev(v), 0, 40)
    kb, kr = _rows_buf(4, 256)
    vb, vr = _rows_buf(4, 256)
    for first in (7, 37, 100):
        with pytest.raises(mu.MuserError) as ei:
            mu.muser_kv_snapshot(plane, first, 4, kr, vr)
        assert ei.value.status == -1
    _check_rows_canary(kb, 0, 0, 256)
    before = (_u16(key).copy(), plane.len, plane.origin_logical, plane.origin_physical)
    with pytest.raises(mu.MuserError):
        mu.muser_kv_restore(plane, kr, vr, 0, 33)
    assert np.array_equal(_u16(key), before[0])
    assert (plane.len, plane.origin_logical, plane.origin_physical) == before[1:]


# ----------------------------------------------------------------- sync
def test_sync_bounded_wait_times_out_then_completes():
    s = torch.cuda.Stream()
    mu.muser_debug_spin(300_000, s)   # a bounded 0.3 s kernel
    assert mu.muser_sync(s, 20) == -6
    assert mu.muser_sync(s, -1) == 0
    assert mu.muser_sync(s, 1000) == 0


def test_device_status_clean():
    torch.cuda.synchronize()
    assert mu.muser_device_status() == 0


# ------------------------------------------------ LM head scale + soft cap
def test_scale_softcap_in_place():
    rng = np.random.default_rng(11)
    logits = (rng.standard_normal(70001) * np.float32(80)).astype(np.float32)
    logits[:4] = [0.0, -0.0, 3.0e4, -3.0e4]
    d = dev(logits)
    mu.muser_scale_softcap(d, logits.size, oracle.LOGIT_SCALE, oracle.SOFTCAP)
    assert_close(host(d), oracle.scale_softcap(logits), "scale_softcap")


@pytest.mark.parametrize("qtype", ["q6_k", "q4_k"])
@pytest.mark.parametrize("M,xscale", [(1, 0.02), (1, 1.0), (3, 0.02)])
def test_lm_head(qtype, M, xscale):
    """Logits in the cap's curved range (x scaled down) and saturated; one
    row of x runs the cap as the matvec's epilogue, three rows separately."""
    vocab, hidden = 20011, 6656
    W = synth.qmatrix(qtype, vocab, hidden, seed=61)
    x = (oracle.rms_norm(synth.normal((M, hidden), seed=62), synth.norm_weight(hidden, seed=62), 1e-5)
         * np.float32(xscale)).astype(np.float32)
    logits = nan_like((M, vocab), extra=32)
    mu.muser_lm_head(qtype, dev(W), vocab, hidden, dev(x), M, logits, oracle.LOGIT_SCALE, oracle.SOFTCAP)
    ref = oracle.lm_head(qtype, W, vocab, hidden, x)
    assert_close(host(logits[:M * vocab]).reshape(M, vocab), ref, f"lm_head {qtype} M={M} x*{xscale}")
    check_canary(logits, M * vocab)
    assert mu.muser_device_status() == 0


def test_lm_head_full_vocabulary():
    """The book's LM head shape, 202,048 x 6,656 (Q6_K, 1.09 GB), every logit."""
    vocab, hidden = 202048, 6656
    W = synth.q6k_matrix(vocab, hidden, seed=63)
    x = (oracle.rms_norm(synth.normal((1, hidden), seed=64), synth.norm_weight(hidden, seed=64), 1e-5)
         * np.float32(0.02)).astype(np.float32)
    logits = nan_like((1, vocab), extra=32)
    Wd = dev(W)
    mu.muser_lm_head("q6_k", Wd, vocab, hidden, dev(x), 1, logits, oracle.LOGIT_SCALE, oracle.SOFTCAP)
    ref = oracle.lm_head("q6_k", W, vocab, hidden, x)
    assert_close(host(logits[:vocab]).reshape(1, vocab), ref, "lm_head 202048 x 6656")
    check_canary(logits, vocab)
    del Wd
    torch.cuda.empty_cache()


def test_q6k_scale_outside_the_tensor_core_range_is_flagged():
    """Q6_K scales are exact in the tensor-core kernel's binary16 products only
    on [-62, 62].  A matrix with one scale of 100: one row of x takes it exactly
    (the oracle's result, no flag); 16 rows through the tensor-core kernel set
    bit 4 of the device status instead of failing silently."""
    rows, cols = 1024, 2048
    W = synth.q6k_matrix(rows, cols, seed=5)
    Wbig = W.copy()
    Wbig[37, 192 + 3] = np.uint8(100)       # row 37, super-block 0, sub-block 3: scale 100
    x1 = synth.normal((1, cols), seed=6, tensor=synth.T_X)
    assert mu.muser_device_status(1) == 0
    y1 = nan_like((1, rows))
    mu.muser_qmatvec("q6_k", dev(Wbig), rows, cols, dev(x1), 1, y1)
    assert_close(host(y1).reshape(1, rows), oracle.qmatvec("q6_k", Wbig, rows, cols, x1), "M=1 scale 100",
                 scaled=True)
    assert mu.muser_device_status() == 0, "the one-token kernel takes any int8 scale"
    x16 = synth.normal((16, cols), seed=7, tensor=synth.T_X)
    nscr = mu.muser_qmatvec_scratch_bytes("q6_k", rows, cols, 16)
    scratch = torch.zeros(max(nscr, 16) // 4 + 4, dtype=torch.float32, device="cuda")
    y16 = nan_like((16, rows))
    mu.muser_qmatvec_scratch("q6_k", dev(W), rows, cols, dev(x16), 16, y16, scratch, nscr)
    assert mu.muser_device_status() == 0, "in-range scales leave the status clean"
    mu.muser_qmatvec_scratch("q6_k", dev(Wbig), rows, cols, dev(x16), 16, y16, scratch, nscr)
    torch.cuda.synchronize()
    assert mu.muser_device_status(1) == 4, "an out-of-range scale on the tensor-core path is flagged"
    assert mu.muser_device_status() == 0
