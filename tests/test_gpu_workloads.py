"""The five workloads at their full sizes, on the GPU, against the oracle.

0: Q4_K 512x2048 matvec; 1/2: Q4_K / Q6_K W_down 6656x19968 + dual-eps tail;
3: one decode-FFN block (M = 1, gate/up Q4_K, down Q6_K); 4: 52 layers at
M = 16 (and M = 1, the benchmark's stack): every layer teacher-forced on the
oracle's own layer input, plus the end-to-end stack (a 3-layer slice end to
end at the per-layer bound)."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import assert_close, check_canary, dev, host, nan_like

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import quantized_weight_streaming_q4_gb300 as mu  # noqa: E402

H, F = synth.HIDDEN, synth.FFN


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mu.build()
    mu.lib()
    torch.cuda.init()


def test_workload0_q4k_matvec_512x2048():
    W, x = synth.matvec_case(512, 2048, 1, "q4_k", seed=0, workload=0)
    y = nan_like((1, 512))
    mu.muser_qmatvec("q4_k", dev(W), 512, 2048, dev(x), 1, y)
    assert_close(host(y).reshape(1, 512), oracle.qmatvec("q4_k", W, 512, 2048, x), "workload 0", scaled=True)


@pytest.mark.parametrize("qtype,wl", [("q4_k", 1), ("q6_k", 2)])
def test_workloads_1_2_down_projection_and_tail(qtype, wl):
    case = synth.down_tail_case(qtype, H, F, 1, seed=0, workload=wl)
    mid = nan_like((1, F))
    mu.muser_silu_mul(dev(case["a"]), dev(case["b"]), mid, F)
    mid_ref = oracle.silu_mul(case["a"], case["b"])
    assert_close(host(mid).reshape(1, F), mid_ref, "ffn_mid", scaled=True)
    resid = dev(case["resid"])
    proj, out = nan_like((1, H)), nan_like((1, H))
    nscr = mu.muser_scratch_bytes(H, 1)
    scratch = torch.zeros(nscr // 4, dtype=torch.float32, device="cuda")
    mu.muser_qmatvec_residual_dual_rmsnorm(qtype, dev(case["W"]), H, F, mid, 1, proj, resid, out,
                                           dev(case["w1"]), dev(case["w2"]), 1e-8, 1e-5, scratch,
                                           nscr)
    p_ref, r_ref, o_ref = oracle.down_tail(qtype, case["W"], H, F, mid_ref, case["resid"],
                                           case["w1"], case["w2"])
    assert_close(host(proj).reshape(1, H), p_ref, f"workload {wl} projected", scaled=True)
    assert_close(host(resid), r_ref, f"workload {wl} residual")
    assert_close(host(out).reshape(1, H), o_ref, f"workload {wl} output")


def _layer_dev(L, w_next):
    d = {k: dev(v) for k, v in L.items()}
    d["w_next"] = dev(w_next)
    return d


def _ffn_layer_struct(d, down_qtype="q6_k"):
    return mu.FfnLayer(d["Wg"].data_ptr(), d["Wu"].data_ptr(), d["Wd"].data_ptr(),
                       d["w1"].data_ptr(), d["w_next"].data_ptr(), mu.MUSER_Q4_K,
                       mu.QTYPES[down_qtype])


def test_workload3_ffn_block_m1():
    L = synth.ffn_layer(0, H, F, seed=0, workload=3)
    w_in = synth.input_norm_weight(0, H, seed=0, workload=3)
    w_next = synth.input_norm_weight(1, H, seed=0, workload=3)
    r = synth.residual_rows(1, H, seed=0, workload=3)
    x_ref, mid_ref, p_ref, r_ref, o_ref = oracle.ffn_block(r, w_in, L, w_next, H, F)
    d = _layer_dev(L, w_next)
    # the public one-call path
    ws_bytes = mu.muser_ffn_workspace_bytes(H, F, 1)
    ws = torch.zeros(ws_bytes // 4, dtype=torch.float32, device="cuda")
    resid, out = dev(r), nan_like((1, H))
    mu.muser_ffn_stack([_ffn_layer_struct(d)], dev(w_in), H, F, 1, resid, out, 1e-5, 1e-8, ws,
                       ws_bytes)
    assert_close(host(resid), r_ref, "block residual")
    assert_close(host(out).reshape(1, H), o_ref, "block output")
    # the same block step by step, every intermediate against the oracle
    resid2, x, mid = dev(r), nan_like((1, H)), nan_like((1, F))
    proj, out2 = nan_like((1, H)), nan_like((1, H))
    mu.muser_rms_norm(resid2, dev(w_in), x, H, 1, 1e-5)
    assert_close(host(x).reshape(1, H), x_ref, "normed input")
    mu.muser_ffn_gate_up_silu("q4_k", d["Wg"], d["Wu"], F, H, x, 1, mid)
    assert_close(host(mid).reshape(1, F), mid_ref, "ffn_mid", scaled=True)
    scratch = torch.zeros(64, dtype=torch.float32, device="cuda")
    mu.muser_qmatvec_residual_dual_rmsnorm("q6_k", d["Wd"], H, F, mid, 1, proj, resid2, out2,
                                           d["w1"], d["w_next"], 1e-8, 1e-5, scratch, 256)
    assert_close(host(proj).reshape(1, H), p_ref, "projected", scaled=True)
    assert_close(host(resid2), r_ref, "residual")
    assert_close(host(out2).reshape(1, H), o_ref, "output")


def _stack(n_layers, M, rows_checked, seed=0):
    wl = 4
    w_in0 = synth.input_norm_weight(0, H, seed=seed, workload=wl)
    r = synth.residual_rows(M, H, seed=seed, workload=wl)
    x_ref = oracle.rms_norm(r[rows_checked], w_in0, 1e-5)
    r_ref = r[rows_checked].copy()
    keep, structs = [], []
    for l in range(n_layers):
        L = synth.ffn_layer(l, H, F, seed=seed, workload=wl)
        w_next = synth.input_norm_weight(l + 1, H, seed=seed, workload=wl)
        d = _layer_dev(L, w_next)
        keep.append(d)
        structs.append(_ffn_layer_struct(d))
        r_ref, x_ref, _, _ = oracle.ffn_layer(x_ref, r_ref, L, w_next, H, F)
        del L
    ws_bytes = mu.muser_ffn_workspace_bytes(H, F, M)
    ws = torch.zeros(ws_bytes // 4, dtype=torch.float32, device="cuda")
    resid, out = dev(r), nan_like((M, H))
    mu.muser_ffn_stack(structs, dev(w_in0), H, F, M, resid, out, 1e-5, 1e-8, ws, ws_bytes)
    got_r = host(resid)
    got_o = host(out).reshape(M, H)
    assert np.isfinite(got_r).all() and np.isfinite(got_o).all()
    del keep
    return got_r[rows_checked], got_o[rows_checked], r_ref, x_ref


@pytest.mark.parametrize("M", [3, 16])
def test_small_stack_several_rows(M):
    """Two layers at hidden 512, ffn 1280 through muser_ffn_stack: partial
    gate/up tiles split over CTAs, Q6_K down rows of 5 blocks (1050 bytes, the
    worst row alignment), several rows of x."""
    hidden, ffn, wl = 512, 1280, 3
    w_in0 = synth.input_norm_weight(0, hidden, seed=7, workload=wl)
    r = synth.residual_rows(M, hidden, seed=7, workload=wl)
    x_ref, r_ref = oracle.rms_norm(r, w_in0, 1e-5), r.copy()
    keep, structs = [], []
    for l in range(2):
        L = synth.ffn_layer(l, hidden, ffn, seed=7, workload=wl)
        w_next = synth.input_norm_weight(l + 1, hidden, seed=7, workload=wl)
        d = _layer_dev(L, w_next)
        keep.append(d)
        structs.append(_ffn_layer_struct(d))
        r_ref, x_ref, _, _ = oracle.ffn_layer(x_ref, r_ref, L, w_next, hidden, ffn)
    ws_bytes = mu.muser_ffn_workspace_bytes(hidden, ffn, M)
    ws = torch.zeros(ws_bytes // 4, dtype=torch.float32, device="cuda")
    resid, out = dev(r), nan_like((M, hidden))
    mu.muser_ffn_stack(structs, dev(w_in0), hidden, ffn, M, resid, out, 1e-5, 1e-8, ws, ws_bytes)
    assert_close(host(resid).reshape(M, hidden), r_ref, f"2-layer residual M={M}")
    assert_close(host(out).reshape(M, hidden), x_ref, f"2-layer output M={M}")
    assert not host(ws).reshape(-1)[-(mu.muser_scratch_bytes(hidden, M) // 4):].any(), "scratch left zeroed"
    assert mu.muser_device_status() == 0
    del keep


def test_workload4_stack_slice_all_rows():
    rows = np.arange(16)
    gr, go, rr, orf = _stack(3, 16, rows)
    assert_close(gr, rr, "3-layer stack residual (16 rows)")
    assert_close(go, orf, "3-layer stack output (16 rows)")


# The 52-layer stack amplifies rounding chaotically on some rows: one-ulp
# binary32 nudges on the input of the fp64 oracle itself move its layer-51
# residual by up to ~6e-3 of the row's RMS (rows whose gates sit deep in
# SiLU's exponential tail), while other rows do not amplify at all (~5e-7).
# So (1) every layer is held to the path's bound teacher-forced -- the GPU
# layer runs on the oracle's own input of that layer -- at M = 16 and M = 1;
# (2) a second oracle trajectory from nudged inputs classifies each row from
# the oracle alone; stable rows are held to the path's bound end to end,
# chaotic rows to finiteness and their RMS (error reported).
STABLE = 1e-5        # oracle self-sensitivity (max |dr| / rms) below which a row is stable
CHAOTIC_RMS = 0.05   # chaotic rows: |rms(gpu) - rms(oracle)| / rms(oracle)


def _nudge(r):
    r2 = r.copy()
    r2.view(np.int32)[:, ::7] += 1
    return r2


def test_workload4_52_layers_teacher_forced_and_end_to_end():
    """M = 16 (workload 4) and M = 1 (the benchmark's stack) through 52 layers."""
    wl, M = 4, 16
    w_in0 = synth.input_norm_weight(0, H, seed=0, workload=wl)
    r0 = synth.residual_rows(M, H, seed=0, workload=wl)
    rr = np.concatenate([r0, _nudge(r0)])           # oracle: true and nudged trajectories
    xx = oracle.rms_norm(rr, w_in0, 1e-5)
    keep, structs = [], []
    mid16, proj16, out16 = nan_like((16, F)), nan_like((16, H)), nan_like((16, H))
    mid1, proj1, out1 = nan_like((1, F)), nan_like((1, H)), nan_like((1, H))
    nscr = mu.muser_scratch_bytes(H, 16)
    scratch = torch.zeros(nscr // 4, dtype=torch.float32, device="cuda")
    for l in range(synth.N_LAYERS):
        L = synth.ffn_layer(l, H, F, seed=0, workload=wl)
        w_next = synth.input_norm_weight(l + 1, H, seed=0, workload=wl)
        d = _layer_dev(L, w_next)
        keep.append(d)
        structs.append(_ffn_layer_struct(d))
        r_next, x_next, mid_o, p_o = oracle.ffn_layer(xx, rr, L, w_next, H, F)
        # teacher-forced GPU layer at M = 16 and M = 1 on the oracle's input
        for Mt, mid, proj, out in ((16, mid16, proj16, out16), (1, mid1, proj1, out1)):
            xg, rg = dev(xx[:Mt]), dev(rr[:Mt])
            mu.muser_ffn_gate_up_silu("q4_k", d["Wg"], d["Wu"], F, H, xg, Mt, mid)
            assert_close(host(mid).reshape(-1, F)[:Mt], mid_o[:Mt], f"layer {l} mid M={Mt}", scaled=True)
            mu.muser_qmatvec_residual_dual_rmsnorm("q6_k", d["Wd"], H, F, mid, Mt, proj, rg, out,
                                                   d["w1"], d["w_next"], 1e-8, 1e-5, scratch, nscr)
            assert_close(host(proj).reshape(-1, H)[:Mt], p_o[:Mt], f"layer {l} projected M={Mt}", scaled=True)
            assert_close(host(rg), r_next[:Mt], f"layer {l} residual M={Mt}")
            assert_close(host(out).reshape(-1, H)[:Mt], x_next[:Mt], f"layer {l} output M={Mt}")
        rr, xx = r_next, x_next
        del L
    assert not host(scratch).any()
    r_ref, x_ref = rr[:M], xx[:M]
    rms = np.sqrt(np.mean(r_ref.astype(np.float64) ** 2, axis=1))
    sens = np.abs(rr[M:].astype(np.float64) - r_ref).max(axis=1) / rms
    stable = sens < STABLE
    assert stable.sum() >= 4 and (~stable).sum() >= 1
    ws_bytes = mu.muser_ffn_workspace_bytes(H, F, M)
    ws = torch.zeros(ws_bytes // 4, dtype=torch.float32, device="cuda")
    for Mt, rows in ((16, np.arange(16)), (1, np.array([int(np.argmax(stable))])),
                     (1, np.array([int(np.argmin(stable))]))):
        resid, out = dev(r0[rows]), nan_like((Mt, H))
        ws.zero_()
        mu.muser_ffn_stack(structs, dev(w_in0), H, F, Mt, resid, out, 1e-5, 1e-8, ws, ws_bytes)
        gr, go = host(resid), host(out).reshape(Mt, H)
        assert np.isfinite(gr).all() and np.isfinite(go).all()
        for i, row in enumerate(rows):
            err = np.abs(gr[i].astype(np.float64) - r_ref[row]).max() / rms[row]
            print(f"52-layer M={Mt} row {row}: oracle self-sensitivity {sens[row]:.1e}, "
                  f"gpu max |err|/rms {err:.1e} ({'stable' if stable[row] else 'chaotic'})")
            if stable[row]:
                assert_close(gr[i:i + 1], r_ref[row:row + 1], f"52-layer residual row {row} M={Mt}")
                assert_close(go[i:i + 1], x_ref[row:row + 1], f"52-layer output row {row} M={Mt}")
            else:
                g_rms = np.sqrt(np.mean(gr[i].astype(np.float64) ** 2))
                assert abs(g_rms - rms[row]) / rms[row] < CHAOTIC_RMS
    del keep
    torch.cuda.empty_cache()


# ---------------------------------------------- attention-side projections
@pytest.mark.parametrize("M", [1, 16])
def test_attention_side_projections_and_first_tail(M):
    """The rest of a layer's weight stream at the book's shapes (Ch 10 Figure
    10.1 boxes 4, 9 and 10): Q, K, V and gate [6656 -> 4096/256/256/4096] on
    the normed residual, then o_proj [4096 -> 6656] with the first dual-eps
    tail (post-attention norm, then the FFN input norm).  Attention itself is
    outside the path; o_proj reads a seeded stand-in for its output."""
    A = synth.attn_layer(0, H)
    r = synth.residual_rows(M, H, workload=synth.ATTN_WORKLOAD)
    w_in = synth.input_norm_weight(0, H, workload=synth.ATTN_WORKLOAD)
    w_ffn = synth.input_norm_weight(1, H, workload=synth.ATTN_WORKLOAD)
    x = oracle.rms_norm(r, w_in, 1e-5)
    xd = dev(x)
    for name, rows in (("Wq", synth.Q_DIM), ("Wk", synth.KV_DIM), ("Wv", synth.KV_DIM), ("Wg", synth.Q_DIM)):
        y = nan_like((M, rows), extra=16)
        mu.muser_qmatvec("q4_k", dev(A[name]), rows, H, xd, M, y)
        ref = oracle.qmatvec("q4_k", A[name], rows, H, x)
        assert_close(host(y[:M * rows]).reshape(M, rows), ref, f"{name} M={M}", scaled=True)
        check_canary(y, M * rows)
    attn = synth.attn_output(M)
    nscr = mu.muser_scratch_bytes(H, M)
    scratch = torch.zeros(nscr // 4, dtype=torch.float32, device="cuda")
    rd, proj, out = dev(r), nan_like((M, H)), nan_like((M, H))
    mu.muser_qmatvec_residual_dual_rmsnorm("q4_k", dev(A["Wo"]), H, synth.Q_DIM, dev(attn), M, proj, rd, out,
                                           dev(A["w_post"]), dev(w_ffn), 1e-8, 1e-5, scratch, nscr)
    p_ref, r_ref, o_ref = oracle.down_tail("q4_k", A["Wo"], H, synth.Q_DIM, attn, r, A["w_post"], w_ffn)
    assert_close(host(proj).reshape(M, H), p_ref, f"o_proj M={M}", scaled=True)
    assert_close(host(rd), r_ref, f"post-attention residual M={M}")
    assert_close(host(out).reshape(M, H), o_ref, f"FFN input M={M}")
    assert not host(scratch).any()
    assert mu.muser_device_status() == 0


@pytest.mark.parametrize("M", [1, 3])
@pytest.mark.parametrize("with_tail", [False, "in_place", "residual_out"])
def test_attention_projection_group(M, with_tail):
    """Q, K, V and gate as one group (one launch at M = 1), optionally after
    the previous sub-block's tail: equal to the tail and four matvecs."""
    A = synth.attn_layer(1, H)
    names, rows = ("Wq", "Wk", "Wv", "Wg"), (synth.Q_DIM, synth.KV_DIM, synth.KV_DIM, synth.Q_DIM)
    ys = [nan_like((M, n), extra=16) for n in rows]
    if with_tail:
        r = synth.residual_rows(M, H, workload=synth.ATTN_WORKLOAD)
        p = synth.normal((M, H), seed=7, workload=synth.ATTN_WORKLOAD, tensor=synth.T_X) * np.float32(3e5)
        w1 = synth.norm_weight(H, seed=7, workload=synth.ATTN_WORKLOAD, tensor=synth.T_W1)
        w2 = synth.norm_weight(H, seed=7, workload=synth.ATTN_WORKLOAD, tensor=synth.T_W2)
        rd, x_out = dev(r), nan_like((M, H), extra=16)
        tk = torch.zeros(mu.MUSER_BOUNDARY_SCRATCH_BYTES // 4, dtype=torch.int32, device="cuda")
        r_out = nan_like((M, H), extra=16) if with_tail == "residual_out" else None
        mu.muser_qmatvec_group_tail("q4_k", [dev(A[n]) for n in names], rows, H, dev(p), rd, dev(w1), dev(w2),
                                    1e-8, 1e-5, x_out, M, ys, tk, residual_out=r_out)
        assert not host(tk).any(), "the ticket must be left zeroed"
        r_ref, x = oracle.dual_tail(r, p, w1, w2, 1e-8, 1e-5)
        if r_out is not None:
            assert np.array_equal(host(rd).reshape(M, H), r), "residual_out form: the input row is read only"
            check_canary(r_out, M * H)
            rd = r_out[:M * H]
        assert_close(host(rd).reshape(M, H), r_ref, "tail residual")
        assert_close(host(x_out[:M * H]).reshape(M, H), x, "tail x_out")
        check_canary(x_out, M * H)
    else:
        x = oracle.rms_norm(synth.residual_rows(M, H, workload=synth.ATTN_WORKLOAD),
                            synth.input_norm_weight(0, H, workload=synth.ATTN_WORKLOAD), 1e-5)
        mu.muser_qmatvec_group("q4_k", [dev(A[n]) for n in names], rows, H, dev(x), M, ys)
    for name, n, y in zip(names, rows, ys):
        ref = oracle.qmatvec("q4_k", A[name], n, H, x)
        assert_close(host(y[:M * n]).reshape(M, n), ref, f"{name} in the group M={M}", scaled=True)
        check_canary(y, M * n)
    assert mu.muser_device_status() == 0


@pytest.mark.parametrize("M", [3, 16])
@pytest.mark.parametrize("case", ["attention", "ragged", "tail", "tail_in_place"])
def test_group_scratch_one_tensor_core_launch(M, case):
    """Several rows of x with group scratch: the group's matrices run as one
    tensor-core launch, each matrix starting a 128-row tile (ragged row counts
    leave partial tiles inside the virtual matrix); every output equals the
    oracle's matvec, canaries stay, the scratch is left zeroed.  With the
    tail (residual_out or in place), the tail kernel also writes the launch's
    B image of its output (rows of the image past M stay zero)."""
    if case == "ragged":
        rows = (200, 72, 328, 136)
        mats = [synth.q4k_matrix(r, H, seed=M, layer=i, tensor=synth.T_GATE) for i, r in enumerate(rows)]
    else:
        A = synth.attn_layer(2, H)
        rows = (synth.Q_DIM, synth.KV_DIM, synth.KV_DIM, synth.Q_DIM)
        mats = [A[n] for n in ("Wq", "Wk", "Wv", "Wg")]
    nscr = mu.muser_qmatvec_group_scratch_bytes("q4_k", rows, H, M)
    assert nscr > 0, "the group takes the one-launch tensor-core path"
    scratch = torch.zeros(nscr // 4 + 4, dtype=torch.float32, device="cuda")
    ys = [nan_like((M, n), extra=16) for n in rows]
    if case.startswith("tail"):
        r = synth.residual_rows(M, H, workload=synth.ATTN_WORKLOAD)
        p = synth.normal((M, H), seed=9, workload=synth.ATTN_WORKLOAD, tensor=synth.T_X) * np.float32(3e5)
        w1 = synth.norm_weight(H, seed=9, workload=synth.ATTN_WORKLOAD, tensor=synth.T_W1)
        w2 = synth.norm_weight(H, seed=9, workload=synth.ATTN_WORKLOAD, tensor=synth.T_W2)
        in_place = case == "tail_in_place"
        rd, x_out = dev(r), nan_like((M, H), extra=16)
        r_out = None if in_place else nan_like((M, H), extra=16)
        mu.muser_qmatvec_group_tail("q4_k", [dev(m) for m in mats], rows, H, dev(p), rd, dev(w1), dev(w2), 1e-8,
                                    1e-5, x_out, M, ys, scratch, nscr, residual_out=r_out)
        r_ref, x = oracle.dual_tail(r, p, w1, w2, 1e-8, 1e-5)
        if in_place:
            assert_close(host(rd).reshape(M, H), r_ref, "tail residual (in place)")
        else:
            assert_close(host(r_out[:M * H]).reshape(M, H), r_ref, "tail residual")
            check_canary(r_out, M * H)
            assert np.array_equal(host(rd).reshape(M, H), r)
        assert_close(host(x_out[:M * H]).reshape(M, H), x, "tail x_out")
        check_canary(x_out, M * H)
    else:
        x = oracle.rms_norm(synth.normal((M, H), seed=M + 1), synth.norm_weight(H, seed=M + 1), 1e-5)
        mu.muser_qmatvec_group_scratch("q4_k", [dev(m) for m in mats], rows, H, dev(x), M, ys, scratch, nscr)
    for i, (m, n, y) in enumerate(zip(mats, rows, ys)):
        ref = oracle.qmatvec("q4_k", m, n, H, x)
        assert_close(host(y[:M * n]).reshape(M, n), ref, f"matrix {i} of the group ({case}) M={M}", scaled=True)
        check_canary(y, M * n)
    assert not host(scratch).any(), "scratch must be left zeroed"
    assert mu.muser_device_status() == 0


@pytest.mark.parametrize("form", ["residual_out", "in_place"])
def test_group_tail_image_short_row_two_rows(form):
    """The tail that writes the grouped launch's B image, at a row of 2,048
    (one float4 per thread of its block) and the fewest rows of x (M = 2, so
    14 of the image's 16 rows stay as the zero-filled scratch has them), on a
    group of ragged Q4_K matrices large enough to take the image (8 units of
    128 rows x 256 inputs per SM): residual, x_out and every output equal the
    oracle's tail and matvecs; canaries stay; the scratch is left zeroed."""
    M, cols = 2, 2048
    rows = (9000, 4040, 5000, 1480)  # 155 tiles of 128 rows: 1,240 units over 8 super-blocks
    mats = [synth.q4k_matrix(r, cols, seed=21, layer=i, tensor=synth.T_GATE) for i, r in enumerate(rows)]
    nscr = mu.muser_qmatvec_group_scratch_bytes("q4_k", rows, cols, M)
    assert nscr > 0
    scratch = torch.zeros(nscr // 4 + 4, dtype=torch.float32, device="cuda")
    r = synth.normal((M, cols), seed=22, workload=synth.ATTN_WORKLOAD, tensor=synth.T_X)
    p = synth.normal((M, cols), seed=23, workload=synth.ATTN_WORKLOAD, tensor=synth.T_X) * np.float32(40.0)
    w1 = synth.norm_weight(cols, seed=24, workload=synth.ATTN_WORKLOAD, tensor=synth.T_W1)
    w2 = synth.norm_weight(cols, seed=24, workload=synth.ATTN_WORKLOAD, tensor=synth.T_W2)
    rd, x_out = dev(r), nan_like((M, cols), extra=16)
    r_out = nan_like((M, cols), extra=16) if form == "residual_out" else None
    ys = [nan_like((M, n), extra=16) for n in rows]
    mu.muser_qmatvec_group_tail("q4_k", [dev(m) for m in mats], rows, cols, dev(p), rd, dev(w1), dev(w2), 1e-8,
                                1e-5, x_out, M, ys, scratch, nscr, residual_out=r_out)
    r_ref, x = oracle.dual_tail(r, p, w1, w2, 1e-8, 1e-5)
    got_r = host(rd).reshape(M, cols) if r_out is None else host(r_out[:M * cols]).reshape(M, cols)
    assert_close(got_r, r_ref, "tail residual")
    assert_close(host(x_out[:M * cols]).reshape(M, cols), x, "tail x_out")
    check_canary(x_out, M * cols)
    for i, (m, n, y) in enumerate(zip(mats, rows, ys)):
        assert_close(host(y[:M * n]).reshape(M, n), oracle.qmatvec("q4_k", m, n, cols, x),
                     f"matrix {i} after the image-writing tail", scaled=True)
        check_canary(y, M * n)
    assert not host(scratch).any(), "scratch must be left zeroed"
    assert mu.muser_device_status() == 0


def test_group_scratch_edges():
    """muser_qmatvec_group_scratch refuses scratch below its size before any
    launch; the group tail at several rows with only the 256-byte ticket scratch
    runs one launch per matrix and still equals the oracle; one row of x needs
    no group scratch (size 0) and takes the one-token kernel."""
    M = 4
    A = synth.attn_layer(3, H)
    names, rows = ("Wq", "Wk", "Wv", "Wg"), (synth.Q_DIM, synth.KV_DIM, synth.KV_DIM, synth.Q_DIM)
    mats = [dev(A[n]) for n in names]
    x = oracle.rms_norm(synth.normal((M, H), seed=11), synth.norm_weight(H, seed=11), 1e-5)
    nscr = mu.muser_qmatvec_group_scratch_bytes("q4_k", rows, H, M)
    assert nscr > 0 and mu.muser_qmatvec_group_scratch_bytes("q4_k", rows, H, 1) == 0
    small = torch.zeros(nscr // 8, dtype=torch.float32, device="cuda")
    ys = [nan_like((M, n), extra=16) for n in rows]
    with pytest.raises(RuntimeError, match="scratch"):
        mu.muser_qmatvec_group_scratch("q4_k", mats, rows, H, dev(x), M, ys, small, nscr // 2)
    for n, y in zip(rows, ys):
        assert torch.isnan(y[:M * n]).all(), "nothing launched"
    # the tail at several rows with the ticket scratch only: one launch per matrix
    r = synth.residual_rows(M, H, workload=synth.ATTN_WORKLOAD)
    p = synth.normal((M, H), seed=12, workload=synth.ATTN_WORKLOAD, tensor=synth.T_X) * np.float32(3e5)
    w1 = synth.norm_weight(H, seed=12, workload=synth.ATTN_WORKLOAD, tensor=synth.T_W1)
    w2 = synth.norm_weight(H, seed=12, workload=synth.ATTN_WORKLOAD, tensor=synth.T_W2)
    tk = torch.zeros(mu.MUSER_BOUNDARY_SCRATCH_BYTES // 4, dtype=torch.int32, device="cuda")
    rd, x_out = dev(r), nan_like((M, H), extra=16)
    mu.muser_qmatvec_group_tail("q4_k", mats, rows, H, dev(p), rd, dev(w1), dev(w2), 1e-8, 1e-5, x_out, M, ys, tk)
    r_ref, xr = oracle.dual_tail(r, p, w1, w2, 1e-8, 1e-5)
    assert_close(host(rd).reshape(M, H), r_ref, "tail residual (per-matrix path)")
    for name, n, y in zip(names, rows, ys):
        assert_close(host(y[:M * n]).reshape(M, n), oracle.qmatvec("q4_k", A[name], n, H, xr),
                     f"{name} per-matrix path", scaled=True)
        check_canary(y, M * n)
    assert not host(tk).any()
    assert mu.muser_device_status() == 0
