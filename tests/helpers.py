"""Shared helpers of the test suite (not part of the library)."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def ensure_lib():
    """Builds libmoex.so if it is missing (the CPU ABI tests need the file)."""
    import moe_expert_gb300 as mx
    if not os.path.exists(mx.LIB_PATH):
        from moe_expert_gb300 import build
        build.build()
    return mx.lib()


def to_np(t):
    return t.detach().cpu().numpy()


def assert_within(got, ref, A, what=""):
    """|got - ref| <= 1e-5 * A + 1e-6 elementwise (the GEMV pass rule)."""
    from oracle.gemv import tolerance
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref)
    tol = tolerance(np.asarray(A, dtype=np.float64))
    bad = err > tol
    if bad.any():
        i = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst at {i}: "
                             f"got {got[i]!r} ref {ref[i]!r} err {err[i]:.3g} tol {tol[i]:.3g}")
    return float((err / np.maximum(tol, 1e-30)).max())
