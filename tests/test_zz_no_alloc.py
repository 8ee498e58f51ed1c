"""The down projection + dual-eps tail with the library's own fixed scratch
(muser_qmatvec_residual_dual_rmsnorm_static) against the entry point that
takes caller-owned scratch and against the oracle, through the C ABI, on two
calls in a row.

The file name sorts last, so in a full run these cases execute after every
other GPU test has used the library in the same process; they also pass when
run alone in a fresh process."""
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
    yield
    torch.cuda.synchronize()


# (qtype, M, hidden, ffn): the one-token Q6_K and Q4_K shapes of the 6656 x
# 19968 layer (counter-based tail), the 16-row shape, and the largest
# M * hidden the fixed scratch holds (16 x 16380 = 262080 floats).
CASES = [("q6_k", 1, 6656, 19968), ("q4_k", 1, 6656, 19968), ("q6_k", 16, 6656, 2048),
         ("q4_k", 16, 16380, 256)]


@pytest.mark.parametrize("qtype,M,hidden,ffn", CASES)
def test_static_scratch_matches_caller_scratch(qtype, M, hidden, ffn):
    case = synth.down_tail_case(qtype, hidden, ffn, M, seed=23)
    Wd, w1, w2 = dev(case["W"]), dev(case["w1"]), dev(case["w2"])
    mid = nan_like((M, ffn))
    mu.muser_silu_mul(dev(case["a"]), dev(case["b"]), mid, M * ffn)

    # the entry point with caller-owned projected rows and scratch
    nscr = mu.muser_scratch_bytes(hidden, M)
    scratch = torch.zeros(nscr // 4 + 4, dtype=torch.float32, device="cuda")
    proj = nan_like((M, hidden))
    r_ref, o_ref = dev(case["resid"]), nan_like((M, hidden))
    mu.muser_qmatvec_residual_dual_rmsnorm(qtype, Wd, hidden, ffn, mid, M, proj, r_ref, o_ref,
                                           w1, w2, 1e-8, 1e-5, scratch, nscr)
    r_ref = host(r_ref).reshape(M, hidden).astype(np.float64)
    o_ref = host(o_ref).reshape(M, hidden).astype(np.float64)
    # the oracle on the same intermediate row (Ch 19 §19.4-§19.5)
    mid_h = host(mid).reshape(M, ffn)
    _, r_orc, o_orc = oracle.down_tail(qtype, case["W"], hidden, ffn, mid_h, case["resid"], case["w1"], case["w2"])

    # two calls in a row on the same inputs: the second sees what the first
    # left in the shared array
    for call in (1, 2):
        r, o = dev(case["resid"]), nan_like((M, hidden))
        mu.muser_qmatvec_residual_dual_rmsnorm_static(qtype, Wd, hidden, ffn, mid, M, r, o, w1, w2,
                                                      1e-8, 1e-5)
        assert_close(host(r).reshape(M, hidden), r_ref, f"residual (call {call})")
        assert_close(host(o).reshape(M, hidden), o_ref, f"next-norm output (call {call})")
        assert_close(host(r).reshape(M, hidden), r_orc, f"residual vs oracle (call {call})")
        assert_close(host(o).reshape(M, hidden), o_orc, f"next-norm output vs oracle (call {call})")
    assert mu.muser_device_status() == 0


def test_static_scratch_rejects_sizes_beyond_its_limit():
    W = torch.zeros(16384 * 144 // 4, dtype=torch.float32, device="cuda")
    v = torch.zeros(16 * 16384, dtype=torch.float32, device="cuda")
    with pytest.raises(mu.MuserError, match="M \\* hidden <= 262080"):
        mu.muser_qmatvec_residual_dual_rmsnorm_static("q4_k", W, 16384, 256, v, 16, v, v[8:],
                                                      v, v, 1e-8, 1e-5)
