"""Pins for the oracle's matvec, RMSNorm, dual-eps tail, SiLU and FFN composition.

Pinned against: numpy fp64 dense products (library routine) on the
dequantised weights, brute force on tiny integer-valued cases computed from the
block FIELDS (not from the decoder), closed forms, invariants, scipy's logistic
function, and the worked tail example printed in the Muser book (Ch 19 §19.3).
"""
import json
import os

import numpy as np
import pytest

import oracle
import synth
from tests.kquant_pack import pack_q4k, pack_q6k


# ------------------------------------------------------------------ matvec
@pytest.mark.parametrize("qtype", ["q4_k", "q6_k"])
@pytest.mark.parametrize("M", [1, 3, 16])
def test_matvec_equals_dense_fp64_product(qtype, M):
    rows, cols = 37, 1024
    W = synth.qmatrix(qtype, rows, cols, seed=21)
    x = synth.normal((M, cols), seed=21, tensor=synth.T_X)
    y = oracle.qmatvec(qtype, W, rows, cols, x)
    dense = oracle.dequantize(qtype, W, rows, cols).astype(np.float64)
    ref = (x.astype(np.float64) @ dense.T).astype(np.float32)
    # both are fp64 sums of the same products; after rounding to f32 they may
    # differ by at most one unit in the last place
    assert np.all(np.abs(y.view(np.int32).astype(np.int64) - ref.view(np.int32).astype(np.int64)) <= 1)
    assert np.mean(y == ref) > 0.99


def _brute_q4k(fields, x):
    # sum over weights of (d*sc*q - dmin*m) * x computed from the fields
    tot = 0.0
    for (d, dmin, sc, mn, q), xb in zip(fields, x.reshape(-1, 256)):
        for i in range(256):
            j = i // 32
            tot += (d * sc[j] * q[i] - dmin * mn[j]) * float(xb[i])
    return tot


@pytest.mark.parametrize("rows,cols", [(1, 256), (2, 512), (3, 768)])
def test_q4k_matvec_brute_force_tiny(rows, cols):
    rng = np.random.default_rng(rows)
    nsb = cols // 256
    W = np.zeros((rows, nsb * 144), np.uint8)
    fields = []
    for r in range(rows):
        fr = []
        for b in range(nsb):
            f = (1.0, 1.0, rng.integers(0, 4, 8), rng.integers(0, 4, 8), rng.integers(0, 16, 256))
            W[r, b * 144:(b + 1) * 144] = pack_q4k(*f)
            fr.append(f)
        fields.append(fr)
    x = rng.integers(-3, 4, size=cols).astype(np.float32)
    y = oracle.qmatvec("q4_k", W, rows, cols, x)[0]
    for r in range(rows):
        assert y[r] == _brute_q4k(fields[r], x)   # small integers: exact


@pytest.mark.parametrize("rows,cols", [(1, 256), (2, 512), (3, 768)])
def test_q6k_matvec_brute_force_tiny(rows, cols):
    rng = np.random.default_rng(100 + rows)
    nsb = cols // 256
    W = np.zeros((rows, nsb * 210), np.uint8)
    ref = np.zeros(rows)
    x = rng.integers(-3, 4, size=cols).astype(np.float32)
    for r in range(rows):
        for b in range(nsb):
            sc = rng.integers(-4, 4, 16)
            q = rng.integers(0, 64, 256)
            W[r, b * 210:(b + 1) * 210] = pack_q6k(1.0, sc, q)
            for i in range(256):
                ref[r] += sc[i // 16] * (q[i] - 32) * float(x[b * 256 + i])
    y = oracle.qmatvec("q6_k", W, rows, cols, x)[0]
    assert np.array_equal(y.astype(np.float64), ref)


def test_q4k_all_zero_codes_closed_form():
    # q = 0 everywhere: y = -sum_j dmin*m_j*(sum of x over sub-block j)
    rng = np.random.default_rng(5)
    dmin = 0.125
    mn = rng.integers(0, 64, 8)
    blk = pack_q4k(0.75, dmin, rng.integers(0, 64, 8), mn, [0] * 256)
    x = rng.standard_normal(256).astype(np.float32)
    y = oracle.qmatvec("q4_k", blk.reshape(1, -1), 1, 256, x)[0, 0]
    ref = -sum(dmin * mn[j] * float(np.sum(x[32 * j:32 * j + 32].astype(np.float64))) for j in range(8))
    assert y == np.float32(ref)


def test_matvec_zero_scales_give_exact_zero():
    W = synth.q4k_matrix(8, 512, seed=9)
    Wz = W.reshape(8, 2, 144).copy()
    Wz[:, :, 0:4] = 0
    y = oracle.qmatvec("q4_k", Wz.reshape(8, -1), 8, 512, synth.normal((2, 512), seed=9))
    assert np.all(y == 0.0)


def test_matvec_linearity():
    W = synth.q6k_matrix(16, 512, seed=13)
    x1 = synth.normal((1, 512), seed=13, tensor=1)
    x2 = synth.normal((1, 512), seed=13, tensor=2)
    y = oracle.qmatvec("q6_k", W, 16, 512, np.concatenate([x1, x2, 2.5 * x1 + x2]))
    np.testing.assert_allclose(y[2], 2.5 * y[0] + y[1], rtol=1e-5, atol=1e-3)


def test_matvec_rows_subset_matches_full():
    W = synth.q4k_matrix(40, 768, seed=2)
    x = synth.normal((3, 768), seed=2)
    full = oracle.qmatvec("q4_k", W, 40, 768, x)
    idx = np.array([0, 7, 39, 12])
    sub = oracle.qmatvec_rows("q4_k", W, 40, 768, idx, x)
    assert np.array_equal(sub, full[:, idx])


def test_byte_accounting_matches_book(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "byte_accounting.json")))
    nsb = synth.FFN // 256
    assert nsb == g["w_down_row_superblocks"]
    assert nsb * 144 == g["q4k_row_bytes"] and nsb * 210 == g["q6k_row_bytes"]
    assert synth.HIDDEN * nsb * 144 == g["q4k_w_down_bytes"]
    assert synth.HIDDEN * nsb * 210 == g["q6k_w_down_bytes"]
    assert synth.FFN * 4 == g["ffn_mid_bytes"] and synth.HIDDEN * 4 == g["projected_bytes"]
    W = synth.q4k_matrix(2, synth.FFN, seed=0)
    assert W.shape == (2, g["q4k_row_bytes"])


# ------------------------------------------------------------- norm / tail
def test_tail_worked_example_from_book(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "tail_worked_example.json")))
    r = np.array([g["residual"]], np.float32)
    p = np.array([g["projected"]], np.float32)
    r_out, out = oracle.dual_tail(r, p, np.array(g["post_weight"], np.float32),
                                  np.array(g["next_weight"], np.float32), g["eps1"], g["eps2"])
    np.testing.assert_allclose(r_out[0], g["printed_residual_after_add"], atol=1e-6)
    np.testing.assert_allclose(out[0], g["printed_next_input"], atol=g["abs_tol"])
    rms = np.sqrt(np.mean(r_out[0].astype(np.float64) ** 2))
    assert abs(rms - g["printed_rms_of_residual"]) < 1e-3
    post = oracle.rms_norm(p, np.ones(4, np.float32), g["eps1"])
    np.testing.assert_allclose(post[0], g["printed_post_norm"], atol=1e-6)


def test_rms_norm_invariant_mean_square():
    # mean((out/w)^2) = ms/(ms+eps) exactly in real arithmetic
    x = synth.normal((4, 6656), seed=1) * np.float32(3.0)
    w = synth.norm_weight(6656, seed=1)
    for eps in (1e-5, 1e-8, 0.5):
        out = oracle.rms_norm(x, w, eps).astype(np.float64)
        ms = np.mean(x.astype(np.float64) ** 2, axis=1)
        got = np.mean((out / w.astype(np.float64)) ** 2, axis=1)
        np.testing.assert_allclose(got, ms / (ms + eps), rtol=1e-6)


def test_rms_norm_scale_invariance_and_zero():
    x = synth.normal((1, 512), seed=4)
    w = synth.norm_weight(512, seed=4)
    a = oracle.rms_norm(x, w, 1e-12)
    b = oracle.rms_norm(np.float32(1024.0) * x, w, 1e-12)
    np.testing.assert_allclose(a, b, rtol=2e-7)
    assert np.all(oracle.rms_norm(np.zeros((1, 8), np.float32), np.ones(8, np.float32), 1e-5) == 0)


def test_tail_special_cases():
    n = 6656
    r = synth.normal((2, n), seed=8, tensor=synth.T_RESID)
    w1 = synth.norm_weight(n, seed=8, tensor=synth.T_W1)
    w2 = synth.norm_weight(n, seed=8, tensor=synth.T_W2)
    # p = 0: the residual is unchanged bit for bit
    r_out, out = oracle.dual_tail(r, np.zeros_like(r), w1, w2)
    assert np.array_equal(r_out, r)
    np.testing.assert_array_equal(out, oracle.rms_norm(r, w2, 1e-5))
    # r = p = 0: everything is zero
    r_out, out = oracle.dual_tail(np.zeros_like(r), np.zeros_like(r), w1, w2)
    assert np.all(r_out == 0) and np.all(out == 0)


def test_tail_invariants():
    n = 6656
    r = synth.normal((3, n), seed=12, tensor=synth.T_RESID)
    p = synth.normal((3, n), seed=12, tensor=synth.T_X) * np.float32(1e3)
    w1 = synth.norm_weight(n, seed=12, tensor=synth.T_W1)
    w2 = synth.norm_weight(n, seed=12, tensor=synth.T_W2)
    r_out, out = oracle.dual_tail(r, p, w1, w2, 1e-8, 1e-5)
    h = r_out.astype(np.float64)
    # post-norm invariant: mean(((h - r)/w1)^2) = mp/(mp + eps1) (up to the f32 rounding of h)
    mp = np.mean(p.astype(np.float64) ** 2, axis=1)
    d = (h - r.astype(np.float64)) / w1.astype(np.float64)
    np.testing.assert_allclose(np.mean(d ** 2, axis=1), mp / (mp + 1e-8), rtol=1e-5)
    # next-norm invariant on the stored h
    ms = np.mean(h ** 2, axis=1)
    got = np.mean((out.astype(np.float64) / w2.astype(np.float64)) ** 2, axis=1)
    np.testing.assert_allclose(got, ms / (ms + 1e-5), rtol=1e-6)
    # scaling p leaves the result unchanged up to the eps term
    r2, out2 = oracle.dual_tail(r, np.float32(64.0) * p, w1, w2, 1e-8, 1e-5)
    np.testing.assert_allclose(out2, out, rtol=1e-6, atol=1e-6)


# -------------------------------------------------------------------- SiLU
def test_silu_values():
    from scipy.special import expit
    z = np.concatenate([np.linspace(-40, 40, 2001), [0.0, 1e-30, -1e-30, 700.0, -700.0, -800.0]])
    got = np.array([oracle.silu(v) for v in z])
    ref = z * expit(z)
    np.testing.assert_allclose(got, ref, rtol=1e-14, atol=1e-300)
    assert oracle.silu(0.0) == 0.0
    for v in (0.3, 2.0, 17.5):
        assert abs((oracle.silu(v) - oracle.silu(-v)) - v) < 1e-14 * max(1.0, v)
    assert oracle.silu(80.0) == 80.0 and abs(oracle.silu(-80.0)) < 1e-30


def test_silu_mul_rounds_once():
    from scipy.special import expit
    a = synth.normal((1, 4096), seed=3, tensor=synth.T_A)
    b = synth.normal((1, 4096), seed=3, tensor=synth.T_B)
    got = oracle.silu_mul(a, b)
    a64 = a.astype(np.float64)
    ref = (a64 * expit(a64) * b.astype(np.float64)).astype(np.float32)
    assert np.max(np.abs(got.view(np.int32).astype(np.int64) - ref.view(np.int32).astype(np.int64))) <= 1


# ------------------------------------------------------- FFN composition
def test_ffn_block_is_the_composition_of_its_steps():
    hidden, ffn = 512, 1024
    layer = synth.ffn_layer(0, hidden, ffn, seed=31)
    w_in = synth.input_norm_weight(0, hidden, seed=31)
    w_next = synth.input_norm_weight(1, hidden, seed=31)
    r = synth.residual_rows(2, hidden, seed=31)
    x, mid, p, r_out, out = oracle.ffn_block(r, w_in, layer, w_next, hidden, ffn)
    x2 = oracle.rms_norm(r, w_in, 1e-5)
    g = oracle.qmatvec("q4_k", layer["Wg"], ffn, hidden, x2)
    u = oracle.qmatvec("q4_k", layer["Wu"], ffn, hidden, x2)
    mid2 = oracle.silu_mul(g, u)
    p2 = oracle.qmatvec("q6_k", layer["Wd"], hidden, ffn, mid2)
    r2, out2 = oracle.dual_tail(r, p2, layer["w1"], w_next, 1e-8, 1e-5)
    for a, b in [(x, x2), (mid, mid2), (p, p2), (r_out, r2), (out, out2)]:
        assert np.array_equal(a, b)


def test_ffn_stack_rows_are_independent():
    hidden, ffn, L = 256, 512, 3
    layers = [synth.ffn_layer(i, hidden, ffn, seed=41, workload=4) for i in range(L)]
    w_in = [synth.input_norm_weight(i, hidden, seed=41, workload=4) for i in range(L + 1)]
    r = synth.residual_rows(4, hidden, seed=41, workload=4)
    rf, of = oracle.ffn_stack(r, w_in[0], layers, w_in[1:], hidden, ffn)
    rs, os_ = oracle.ffn_stack(r[2:3], w_in[0], layers, w_in[1:], hidden, ffn)
    assert np.array_equal(rf[2:3], rs) and np.array_equal(of[2:3], os_)


# ------------------------------------------------- LM head scale + soft cap
def test_softcap_constants_are_the_pages_values():
    # Ch 10 Figure 10.1 box 15 prints "x 0.196116 (1/sqrt(26)), then 20 tanh(l/20)"
    assert oracle.LOGIT_SCALE == 0.196116 and oracle.SOFTCAP == 20.0
    assert abs(oracle.LOGIT_SCALE - 26 ** -0.5) < 5e-7


def test_softcap_closed_forms():
    s, c = oracle.LOGIT_SCALE, oracle.SOFTCAP
    assert oracle.softcap(0.0) == 0.0
    for l in (1e-3, 0.7, 13.0, 250.0, 4.0e3):
        assert oracle.softcap(-l) == -oracle.softcap(l)                # odd
        assert abs(oracle.softcap(l)) <= c and (l > 500 or abs(oracle.softcap(l)) < c)  # bounded by the cap
        t = l * s / c                                                  # tanh through exp, another formula
        assert abs(oracle.softcap(l) - c * np.expm1(2 * t) / (np.exp(2 * t) + 1)) <= 1e-12 * c
    assert abs(oracle.softcap(1e-7) / 1e-7 - s) < 1e-9                # slope at 0 is the scale
    assert oracle.softcap(1e5) == c and oracle.softcap(-1e5) == -c     # saturates at the cap
    l = 37.25                                                          # inverse: atanh undoes it
    assert abs(np.arctanh(oracle.softcap(l) / c) * c / s - l) < 1e-9


def test_scale_softcap_rounds_once_and_lm_head_composes():
    rng = np.random.default_rng(5)
    logits = (rng.standard_normal(4099) * 60).astype(np.float32)
    got = oracle.scale_softcap(logits)
    ref = np.array([oracle.softcap(float(v)) for v in logits], np.float64).astype(np.float32)
    assert np.array_equal(got, ref)
    W = synth.q6k_matrix(300, 512, seed=3)
    x = synth.normal((2, 512), seed=3)
    assert np.array_equal(oracle.lm_head("q6_k", W, 300, 512, x),
                          oracle.scale_softcap(oracle.qmatvec("q6_k", W, 300, 512, x)))
