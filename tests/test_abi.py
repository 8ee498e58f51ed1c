"""The C ABI without a GPU: libmuser builds for sm_103a, loads, exports every
function include/muser.h declares, and its host-side argument checks fail
closed (no CUDA call is reached on these paths)."""
import ctypes
import os
import re
import shutil

import pytest

import quantized_weight_streaming_q4_gb300 as mu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "muser.h")

needs_nvcc = pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="nvcc not available")


@pytest.fixture(scope="module")
def L():
    mu.build()
    return mu.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(muser_[a-z0-9_]+)\s*\(", text)))


@needs_nvcc
def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 15
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing


@needs_nvcc
def test_sizes_and_version(L):
    assert mu.muser_version() == 2
    assert mu.muser_block_bytes("q4_k") == 144 and mu.muser_block_bytes("q6_k") == 210
    assert mu.muser_block_bytes("q5_k") == 176 and mu.muser_block_bytes(13) == 176
    assert mu.muser_matrix_bytes("q5_k", 6656, 19968) == 6656 * 78 * 176
    assert mu.muser_block_bytes(7) == 0
    assert mu.muser_matrix_bytes("q4_k", 6656, 19968) == 74760192
    assert mu.muser_matrix_bytes("q6_k", 6656, 19968) == 109025280
    assert mu.muser_matrix_bytes("q4_k", 1, 300) == 0
    assert mu.muser_scratch_bytes(6656, 1) >= 16
    assert mu.muser_ffn_workspace_bytes(6656, 19968, 16) >= 4 * (2 * 16 * 6656 + 16 * 19968 + 16 * 6656)


FAKE = 1 << 20  # an aligned, never-dereferenced pointer value


@needs_nvcc
@pytest.mark.parametrize("args,status", [
    ((99, FAKE, 8, 256, FAKE, 1, FAKE), -2),         # unknown quant type
    ((12, None, 8, 256, FAKE, 1, FAKE), -1),         # NULL weights
    ((12, FAKE, 8, 300, FAKE, 1, FAKE), -1),         # cols not a multiple of 256
    ((12, FAKE, 0, 256, FAKE, 1, FAKE), -1),         # no rows
    ((12, FAKE + 4, 8, 256, FAKE, 1, FAKE), -3),     # misaligned weights
    ((12, FAKE, 8, 256, FAKE + 8, 1, FAKE), -3),     # misaligned x
    ((12, FAKE, 8, 256, FAKE, 0, FAKE), -1),         # M = 0
    ((14, FAKE, 8, 256, FAKE, 17, FAKE), -1),        # M = 17
])
def test_qmatvec_rejects_bad_arguments(L, args, status):
    rc = L.muser_qmatvec(*args, None)
    assert rc == status
    assert mu.muser_last_error()


@needs_nvcc
def test_tail_and_fused_reject_bad_arguments(L):
    assert L.muser_fused_residual_dual_rmsnorm(FAKE, FAKE, FAKE, FAKE, FAKE, 6, 1, 1e-8, 1e-5, None) == -1
    assert L.muser_fused_residual_dual_rmsnorm(FAKE, FAKE, FAKE, FAKE, FAKE, 8, 1, 0.0, 1e-5, None) == -1
    assert L.muser_fused_residual_dual_rmsnorm(FAKE, FAKE, FAKE, FAKE, FAKE, 8, 1, 1e-8, 1e-5, None) == -1  # out aliases residual
    rc = L.muser_qmatvec_residual_dual_rmsnorm(12, FAKE, 6656, 19968, FAKE, 1, FAKE, FAKE + 256, FAKE + 512,
                                               FAKE, FAKE, 1e-8, 1e-5, FAKE, 8, None)
    assert rc == -1 and "scratch" in mu.muser_last_error()
    # every call below fails validation before any launch (fake pointers are never used)
    assert L.muser_ffn_gate_up_silu(14, FAKE, FAKE, 100, 6600, FAKE, 1, FAKE, None) == -1


@needs_nvcc
def test_qmatvec_scratch_host_checks(L):
    # one row of x needs no scratch; checks run before any size query
    assert mu.muser_qmatvec_scratch_bytes("q4_k", 4096, 6656, 1) == 0
    assert mu.muser_qmatvec_scratch_bytes("q4_k", 4096, 6656, 17) == 0
    assert L.muser_qmatvec_scratch(99, FAKE, 8, 256, FAKE, 3, FAKE, FAKE, 1 << 20, None) == -2
    assert L.muser_qmatvec_scratch(12, FAKE, 8, 256, FAKE, 0, FAKE, FAKE, 1 << 20, None) == -1
    assert L.muser_qmatvec_scratch(12, FAKE, 8, 256, FAKE + 4, 3, FAKE, FAKE, 1 << 20, None) == -3


@needs_nvcc
def test_q5k_only_where_supported(L):
    # Q5_K is taken by the plain matvec and dequantisation; the FFN, tail,
    # group and LM-head calls reject it before any launch
    assert L.muser_qmatvec(13, FAKE + 4, 8, 256, FAKE, 1, FAKE, None) == -3   # passes the type check
    assert L.muser_ffn_gate_up_silu(13, FAKE, FAKE, 256, 256, FAKE, 1, FAKE, None) == -2
    rc = L.muser_qmatvec_residual_dual_rmsnorm(13, FAKE, 256, 256, FAKE, 1, FAKE, FAKE + 4096, FAKE + 8192,
                                               FAKE, FAKE, 1e-8, 1e-5, FAKE, 1024, None)
    assert rc == -2 and "Q5_K" not in mu.muser_last_error().split("(")[1]
    assert L.muser_lm_head(13, FAKE, 512, 256, FAKE, 1, FAKE, 0.2, 20.0, None) == -2


@needs_nvcc
def test_stack_rejects_bad_layers(L):
    layer = mu.FfnLayer(FAKE, FAKE, FAKE + 4, FAKE, FAKE, 12, 14)   # misaligned down matrix
    arr = (mu.FfnLayer * 1)(layer)
    ws = mu.muser_ffn_workspace_bytes(512, 1024, 1)
    rc = L.muser_ffn_stack(arr, 1, FAKE, 512, 1024, 1, FAKE, FAKE * 2, 1e-5, 1e-8, FAKE * 4, ws, None)
    assert rc == -3
    rc = L.muser_ffn_stack(arr, 0, FAKE, 512, 1024, 1, FAKE, FAKE * 2, 1e-5, 1e-8, FAKE * 4, ws, None)
    assert rc == -1
    good = (mu.FfnLayer * 1)(mu.FfnLayer(FAKE, FAKE, FAKE, FAKE, FAKE, 12, 14))
    rc = L.muser_ffn_stack(good, 1, FAKE, 512, 1024, 1, FAKE, FAKE * 2, 1e-5, 1e-8, FAKE * 4, ws - 16, None)
    assert rc == -1 and "workspace" in mu.muser_last_error()


@needs_nvcc
def test_kv_ring_discontinuity_fails_closed_without_touching_the_plane(L):
    plane = mu.KvPlane(FAKE, FAKE * 2, 2048, 2048, 5, 5, 256, 128, 0, 0)
    first = ctypes.c_int64(-7)
    for bad in (2052, 2054, 0):
        rc = L.muser_kv_ring_write(ctypes.byref(plane), FAKE, FAKE, bad, 1, ctypes.byref(first), None)
        assert rc == -4
        assert "discontinuity" in mu.muser_last_error()
        assert (plane.len, plane.origin_logical, plane.origin_physical) == (2048, 5, 5)
        assert first.value == -7
    # zero rows at the right position is a no-op that reports the write row
    rc = L.muser_kv_ring_write(ctypes.byref(plane), None, None, 2053, 0, ctypes.byref(first), None)
    assert rc == 0 and first.value == 5
    # inconsistent metadata is rejected
    bad_plane = mu.KvPlane(FAKE, FAKE, 32, 40, 0, 0, 256, 128, 0, 0)
    assert L.muser_kv_ring_write(ctypes.byref(bad_plane), FAKE, FAKE, 40, 1, None, None) == -1


@needs_nvcc
def test_kv_snapshot_and_restore_fail_closed(L):
    plane = mu.KvPlane(FAKE, FAKE * 2, 2048, 2048, 5000, 904, 256, 128, 1, 0)
    # rows outside the live window 5000..7047
    for first, count in ((4999, 1), (5000, 2049), (7047, 2), (7048, 1), (6000, -1)):
        rc = L.muser_kv_snapshot(ctypes.byref(plane), first, count, FAKE, FAKE, None)
        assert rc == -1 and "live window" in mu.muser_last_error()
    # an empty range inside the window launches nothing
    assert L.muser_kv_snapshot(ctypes.byref(plane), 7048, 0, None, None, None) == 0
    for origin, n in ((-1, 1), (0, 2049), (10, -1)):
        rc = L.muser_kv_restore(ctypes.byref(plane), FAKE, FAKE, origin, n, None)
        assert rc == -1
        assert (plane.len, plane.origin_logical, plane.origin_physical) == (2048, 5000, 904)
    assert L.muser_kv_restore(ctypes.byref(plane), None, None, 0, 3, None) == -1
    assert L.muser_kv_restore(ctypes.byref(plane), FAKE + 1, FAKE, 0, 3, None) == -3
    assert (plane.len, plane.origin_logical, plane.origin_physical) == (2048, 5000, 904)
    # an empty window sets only the metadata, at the rotation origin % capacity
    assert L.muser_kv_restore(ctypes.byref(plane), None, None, 4100, 0, None) == 0
    assert (plane.len, plane.origin_logical, plane.origin_physical) == (0, 4100, 4)
    bad_plane = mu.KvPlane(FAKE, FAKE, 32, 40, 0, 0, 256, 128, 0, 0)
    assert L.muser_kv_restore(ctypes.byref(bad_plane), FAKE, FAKE, 0, 1, None) == -1
    # detached rows that overlap a plane, or each other, are rejected before any launch
    plane = mu.KvPlane(FAKE, FAKE * 2, 64, 64, 0, 0, 256, 128, 0, 0)     # planes: 32 KB each
    rows = FAKE * 4
    for k_rows, v_rows in ((FAKE + 512, rows), (rows, FAKE * 2 + 32768 - 2), (rows, rows + 1024)):
        assert L.muser_kv_restore(ctypes.byref(plane), k_rows, v_rows, 0, 8, None) == -1
        assert "overlap" in mu.muser_last_error()
        assert L.muser_kv_snapshot(ctypes.byref(plane), 0, 8, k_rows, v_rows, None) == -1
    assert (plane.len, plane.origin_logical, plane.origin_physical) == (64, 0, 0)


@needs_nvcc
def test_group_calls_fail_closed(L):
    P3 = ctypes.c_void_p * 4
    R4 = ctypes.c_int64 * 4
    W = P3(FAKE, FAKE, FAKE, FAKE)
    rows = R4(4096, 256, 256, 4096)
    y = P3(FAKE * 2, FAKE * 3, FAKE * 4, FAKE * 5)
    g = L.muser_qmatvec_group
    assert g(12, 0, W, rows, 6656, FAKE * 6, 1, y, None) == -1          # no matrices
    assert g(12, 5, W, rows, 6656, FAKE * 6, 1, y, None) == -1          # more than four
    assert g(12, 4, None, rows, 6656, FAKE * 6, 1, y, None) == -1       # no weight array
    assert g(13, 4, W, rows, 6656, FAKE * 6, 1, y, None) == -2          # Q5_K is not a group type
    assert g(12, 4, W, rows, 6600, FAKE * 6, 1, y, None) == -1          # cols not a multiple of 256
    assert g(12, 4, W, rows, 6656, FAKE * 6, 17, y, None) == -1         # M = 17
    assert g(12, 4, P3(FAKE, FAKE + 8, FAKE, FAKE), rows, 6656, FAKE * 6, 1, y, None) == -3
    assert g(12, 4, W, rows, 6656, FAKE * 6, 1, P3(FAKE * 2, FAKE * 3 + 4, FAKE * 4, FAKE * 5), None) == -3
    gs = L.muser_qmatvec_group_scratch
    assert gs(12, 0, W, rows, 6656, FAKE * 6, 16, y, FAKE * 11, 1 << 20, None) == -1   # no matrices
    assert gs(12, 4, W, rows, 6656, FAKE * 6, 17, y, FAKE * 11, 1 << 20, None) == -1   # M = 17
    assert gs(12, 4, W, rows, 6656, FAKE * 6 + 4, 16, y, FAKE * 11, 1 << 20, None) == -3   # misaligned x
    assert L.muser_qmatvec_group_scratch_bytes(14, 4, rows, 6656, 16) == 0   # Q6_K: per matrix
    assert L.muser_qmatvec_group_scratch_bytes(12, 4, rows, 6656, 1) == 0    # one row: the one-token kernel
    t = L.muser_qmatvec_group_tail
    args = (12, 4, W, rows, 6656)
    S = (FAKE * 11, 256)                                                 # the ticket scratch
    pr = (FAKE * 6, FAKE * 7, None, FAKE * 8, FAKE * 9)                  # projected, residual, residual_out, w1, w2
    assert t(*args, *pr, 1e-8, 1e-5, FAKE * 7, 1, y, *S, None) == -1     # x_out == residual
    assert t(*args, *pr, 0.0, 1e-5, FAKE * 10, 1, y, *S, None) == -1     # eps1 = 0
    assert t(*args, FAKE * 6, FAKE * 6, None, FAKE * 8, FAKE * 9, 1e-8, 1e-5, FAKE * 10, 1, y, *S,
             None) == -1                                                 # projected == residual
    assert t(*args, *pr, 1e-8, 1e-5, FAKE * 10, 1, y, None, 256, None) == -1   # in place without scratch
    assert t(*args, *pr, 1e-8, 1e-5, FAKE * 10, 1, y, FAKE * 11, 255, None) == -1
    assert t(*args, *pr, 1e-8, 1e-5, FAKE * 10, 1, y, FAKE * 11 + 4, 256, None) == -3   # misaligned scratch
    assert t(*args, FAKE * 6, FAKE * 7, FAKE * 7, FAKE * 8, FAKE * 9, 1e-8, 1e-5, FAKE * 10, 1, y, None, 0,
             None) == -1                                                 # residual_out == residual
    assert t(*args, FAKE * 6, FAKE * 7, FAKE * 10, FAKE * 8, FAKE * 9, 1e-8, 1e-5, FAKE * 10, 1, y, None, 0,
             None) == -1                                                 # residual_out == x_out
    assert t(*args, FAKE * 6, FAKE * 7, FAKE * 12 + 4, FAKE * 8, FAKE * 9, 1e-8, 1e-5, FAKE * 10, 1, y, None, 0,
             None) == -3                                                 # misaligned residual_out


@needs_nvcc
def test_scale_softcap_and_lm_head_fail_closed(L):
    sc = L.muser_scale_softcap
    assert sc(FAKE, 8, 0.2, 0.0, None) == -1                 # cap must be > 0
    assert sc(FAKE, 8, float("nan"), 20.0, None) == -1       # scale must be finite
    assert sc(FAKE, 8, 0.2, float("inf"), None) == -1
    assert sc(FAKE, -1, 0.2, 20.0, None) == -1
    assert sc(FAKE + 4, 8, 0.2, 20.0, None) == -3
    assert sc(FAKE, 0, 0.2, 20.0, None) == 0                 # nothing to do, nothing launched
    lm = L.muser_lm_head
    assert lm(14, FAKE, 202048, 6656, FAKE * 2, 1, FAKE * 3, 0.196116, -1.0, None) == -1
    assert lm(14, FAKE, 202048, 6656, FAKE * 2, 0, FAKE * 3, 0.196116, 20.0, None) == -1
    assert lm(14, FAKE, 202048, 6600, FAKE * 2, 1, FAKE * 3, 0.196116, 20.0, None) == -1
    assert lm(99, FAKE, 202048, 6656, FAKE * 2, 1, FAKE * 3, 0.196116, 20.0, None) == -2


@needs_nvcc
def test_fused_layer_boundary_and_static_scratch_fail_closed(L):
    f = L.muser_ffn_gate_up_silu_tail
    base = (12, FAKE, FAKE * 2, 19968, 6656, FAKE * 3, FAKE * 4, None, FAKE * 5, FAKE * 6)
    S = (FAKE * 9, 256)                                              # the ticket scratch
    assert f(*base, 1e-8, 1e-5, FAKE * 4, 1, FAKE * 8, *S, None) == -1   # x_out aliases the residual
    assert f(*base, 1e-8, -1.0, FAKE * 7, 1, FAKE * 8, *S, None) == -1   # eps2 < 0
    assert f(*base, 1e-8, 1e-5, FAKE * 7, 0, FAKE * 8, *S, None) == -1   # M = 0
    assert f(14, FAKE, FAKE * 2, 19968, 6656, FAKE * 3, FAKE * 4, None, FAKE * 5, FAKE * 6, 1e-8, 1e-5,
             FAKE * 7, 1, FAKE * 8 + 4, *S, None) == -3                   # misaligned mid
    assert f(*base, 1e-8, 1e-5, FAKE * 7, 1, FAKE * 8, None, 256, None) == -1        # in place without scratch
    assert f(*base, 1e-8, 1e-5, FAKE * 7, 1, FAKE * 8, FAKE * 9, 128, None) == -1    # too small
    assert "scratch" in mu.muser_last_error()
    out = (12, FAKE, FAKE * 2, 19968, 6656, FAKE * 3, FAKE * 4)
    assert f(*out, FAKE * 3, FAKE * 5, FAKE * 6, 1e-8, 1e-5, FAKE * 7, 1, FAKE * 8, None, 0,
             None) == -1                                             # residual_out == projected
    assert "residual_out" in mu.muser_last_error()
    assert f(*out, FAKE * 10 + 8, FAKE * 5, FAKE * 6, 1e-8, 1e-5, FAKE * 7, 1, FAKE * 8, None, 0,
             None) == -3                                             # misaligned residual_out
    st = L.muser_qmatvec_residual_dual_rmsnorm_static
    # M * hidden above the static array's 262,080 floats
    assert st(14, FAKE, 65536, 19968, FAKE * 2, 16, FAKE * 3, FAKE * 4, FAKE * 5, FAKE * 6, 1e-8, 1e-5,
              None) == -1
    assert "static" in mu.muser_last_error() or "scratch" in mu.muser_last_error()


@needs_nvcc
def test_debug_spin_bound(L):
    assert L.muser_debug_spin(11 * 1000 * 1000, None) == -1
    assert L.muser_debug_occupy(4, 11 * 1000 * 1000, None) == -1     # over 10 s
    assert L.muser_debug_occupy(0, 1000, None) == -1                 # no blocks
    assert L.muser_debug_occupy(5000, 1000, None) == -1              # too many blocks


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    monkeypatch.setattr(mu, "_lib", None)
    monkeypatch.setattr(mu, "_LIB", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        mu.lib()


@needs_nvcc
def test_static_scratch_entry_rejects_oversize_before_any_cuda_call(L):
    # 16 x 16384 floats of projected rows exceed the library's fixed scratch
    rc = L.muser_qmatvec_residual_dual_rmsnorm_static(12, FAKE, 16384, 256, FAKE, 16, FAKE, FAKE * 2,
                                                      FAKE, FAKE, 1e-8, 1e-5, None)
    assert rc == -1 and "262080" in mu.muser_last_error()
    assert L.muser_qmatvec_residual_dual_rmsnorm_static(12, FAKE, 6656, 19968, FAKE, 1, FAKE, FAKE,
                                                        FAKE, FAKE, 1e-8, 1e-5, None) == -1  # out aliases residual
