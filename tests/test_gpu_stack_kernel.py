"""The one-token decode-FFN stack as one persistent launch (muser_ffn_stack at
M = 1 with Q4_K gate/up and Q6_K down) against the oracle's layer loop
(Ch 10 §10.3-§10.4): every layer's gate/up/SiLU, down projection and dual-eps
tail, the residual relayed between two buffers (odd and even layer counts),
shapes with idle slice threads, and the widest down row the kernel takes."""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import assert_close, dev, host, nan_like

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import quantized_weight_streaming_q4_gb300 as mu  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mu.build()
    mu.lib()
    torch.cuda.init()


def run_stack(n_layers, hidden, ffn, seed, wl=4, reps=1):
    """n_layers seeded layers through muser_ffn_stack at M = 1 and through the
    oracle; returns (gpu residual, gpu out, oracle residual, oracle out,
    launches)."""
    w_in0 = synth.input_norm_weight(0, hidden, seed=seed, workload=wl)
    r = synth.residual_rows(1, hidden, seed=seed, workload=wl)
    x_ref, r_ref = oracle.rms_norm(r, w_in0, 1e-5), r.copy()
    keep, structs = [], []
    for l in range(n_layers):
        L = synth.ffn_layer(l, hidden, ffn, seed=seed, workload=wl)
        w_next = synth.input_norm_weight(l + 1, hidden, seed=seed, workload=wl)
        d = {k: dev(v) for k, v in L.items()}
        d["w_next"] = dev(w_next)
        keep.append(d)
        structs.append(mu.FfnLayer(d["Wg"].data_ptr(), d["Wu"].data_ptr(), d["Wd"].data_ptr(), d["w1"].data_ptr(),
                                   d["w_next"].data_ptr(), mu.MUSER_Q4_K, mu.MUSER_Q6_K))
        r_ref, x_ref, _, _ = oracle.ffn_layer(x_ref, r_ref, L, w_next, hidden, ffn)
    arr = (mu.FfnLayer * n_layers)(*structs)
    launches = mu.muser_ffn_stack_launches(arr, hidden, ffn, 1)
    ws_bytes = mu.muser_ffn_workspace_bytes(hidden, ffn, 1)
    # the workspace need not be zeroed by the caller for this path; fill it
    # with garbage to check that nothing depends on its contents
    ws = torch.full((ws_bytes // 4,), -7.0, dtype=torch.float32, device="cuda")
    outs = []
    for _ in range(reps):
        resid, out = dev(r), nan_like((1, hidden), extra=16)
        mu.muser_ffn_stack(arr, dev(w_in0), hidden, ffn, 1, resid, out, 1e-5, 1e-8, ws, ws_bytes)
        outs.append((host(resid).reshape(1, hidden), host(out)))
    del keep
    return outs, r_ref, x_ref, launches


@pytest.mark.parametrize("n_layers", [1, 2, 3])
def test_stack_one_launch_small(n_layers):
    """hidden 512, ffn 1024: 8 gate/up slices, 52 row groups of 8 threads;
    odd and even layer counts (the relay starts in the workspace or in the
    caller's buffer and always ends in the caller's)."""
    hidden, ffn = 512, 1024
    outs, r_ref, x_ref, launches = run_stack(n_layers, hidden, ffn, seed=11)
    assert launches == 1
    for i, (gr, go) in enumerate(outs):
        assert_close(gr, r_ref, f"{n_layers}-layer residual")
        assert_close(go[:hidden].reshape(1, hidden), x_ref, f"{n_layers}-layer output")
        assert np.all(go[hidden:] == 12345.0), "write past the output row"
    assert mu.muser_device_status() == 0


@pytest.mark.parametrize("hidden,ffn,n_layers", [(2304, 2560, 3), (6656, 24576, 2), (6656, 19968, 2)])
def test_stack_one_launch_shapes(hidden, ffn, n_layers):
    """Ragged slice counts (hidden 2304: 36 slices, 11 row groups and 20 idle
    threads; ffn 2560: 10 super-blocks per down row), the widest down row the
    kernel takes (ffn 24576: 384 slices over 416 threads), and the model's
    shape with an even layer count; two calls in a row on one workspace."""
    outs, r_ref, x_ref, launches = run_stack(n_layers, hidden, ffn, seed=12, reps=2)
    assert launches == 1
    for i, (gr, go) in enumerate(outs):
        assert_close(gr, r_ref, f"residual {hidden}x{ffn} call {i}")
        assert_close(go[:hidden].reshape(1, hidden), x_ref, f"output {hidden}x{ffn} call {i}")
    assert mu.muser_device_status() == 0


def test_stack_launch_counts():
    """The persistent path is taken for one row of Q4_K/Q6_K layers only; the
    counts of the per-projection paths follow their compositions."""
    fake = mu.FfnLayer(16, 32, 48, 64, 80, mu.MUSER_Q4_K, mu.MUSER_Q6_K)
    arr = (mu.FfnLayer * 52)(*([fake] * 52))
    assert mu.muser_ffn_stack_launches(arr, 6656, 19968, 1) == 1
    # several rows: per layer gate/up and down as tensor-core matvecs (each
    # with its B image built before and cleared after: three launches) and the
    # tail, which from layer 0 on also builds the next gate/up's image (one
    # launch fewer per later layer)
    assert mu.muser_ffn_stack_launches(arr, 6656, 19968, 16) == 1 + 7 + 6 * 51
    q4down = mu.FfnLayer(16, 32, 48, 64, 80, mu.MUSER_Q4_K, mu.MUSER_Q4_K)
    arr2 = (mu.FfnLayer * 2)(q4down, q4down)
    assert mu.muser_ffn_stack_launches(arr2, 6656, 19968, 1) == 2 + 2 * 2
    # ffn not a multiple of 512: the per-projection kernels
    assert mu.muser_ffn_stack_launches(arr, 6656, 19968 + 256, 1) == 2 + 2 * 52
