"""Helpers of the GPU parity tests (test-only)."""
import numpy as np

# The parity bound of the path: max relative error 1e-3 with an absolute floor
# of 1e-4 (elementwise |gpu - oracle| <= 1e-4 * S + 1e-3 * |oracle|).  S = 1
# for normalised outputs; for raw projection outputs (whose magnitude grows
# with the row length and the weights) S = max(1, rms of that output row), so
# the floor is 1e-4 of the output's own scale.
RTOL = 1e-3
ATOL = 1e-4


def dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    import torch
    torch.cuda.synchronize()
    return t.detach().cpu().numpy()


def nan_like(shape, extra=0):
    """A NaN-poisoned f32 device buffer with `extra` canary elements after it."""
    import torch
    n = int(np.prod(shape))
    buf = torch.full((n + extra,), float("nan"), dtype=torch.float32, device="cuda")
    if extra:
        buf[n:] = 12345.0
    return buf


def check_canary(buf, n):
    tail = host(buf[n:])
    assert np.all(tail == 12345.0), "write past the end of an output buffer"


def assert_close(g, o, what, scaled=False):
    g = np.asarray(g, dtype=np.float64).reshape(np.shape(o))
    o = np.asarray(o, dtype=np.float64)
    assert not np.isnan(g).any(), f"{what}: NaN in GPU output (unwritten or invalid element)"
    if scaled:
        o2 = np.atleast_2d(o)
        S = np.maximum(1.0, np.sqrt(np.mean(o2 ** 2, axis=-1, keepdims=True)))
        S = np.broadcast_to(S, o2.shape).reshape(o.shape)
    else:
        S = 1.0
    err = np.abs(g - o)
    bound = ATOL * S + RTOL * np.abs(o)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err / bound), o.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements outside "
                             f"|g-o| <= {ATOL}*S + {RTOL}*|o|; worst at {i}: gpu {g[i]!r} "
                             f"oracle {o[i]!r}")


def max_rel(g, o):
    g = np.asarray(g, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    return float(np.max(np.abs(g - o) / np.maximum(np.abs(o), 1e-30)))
