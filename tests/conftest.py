import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


import pytest  # noqa: E402


@pytest.fixture(scope="session")
def cb():
    """The built CUDA library's Python binding (GPU tests only)."""
    import torch

    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without CUDA")
    from rag_kv_cache_gb300.build import build

    build()
    import rag_kv_cache_gb300 as cbm

    return cbm


def assert_close_bf16(got, ref, atol=2e-2, rtol=1e-2, what=""):
    """|got - ref| <= atol + rtol * |ref| elementwise (the blend's bf16 tolerance)."""
    import numpy as np

    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = np.abs(got - ref)
    lim = atol + rtol * np.abs(ref)
    bad = err > lim
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} elements outside tolerance; "
                           f"max abs err {err.max():.3e}")


def assert_close_attention(got, ref, vscale, what="attention"):
    """Attention tolerance: |got - ref| <= 2e-2 * max(1, vscale) + 1e-2 * |ref|.

    vscale = sum_j p_j |v_j| (from the oracle). The kernel rounds the softmax
    weights p to bf16 (relative error <= 2^-9) before the PV product, so its
    error is bounded by about 2^-8 * vscale: the absolute part of the bf16
    tolerance scales with the values attended to once they exceed unit size.
    """
    import numpy as np

    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    lim = 2e-2 * np.maximum(1.0, vscale) + 1e-2 * np.abs(ref)
    bad = err > lim
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} elements outside tolerance; "
                           f"max abs err {err.max():.3e}; max err/limit {(err / lim).max():.3f}")


# Attention elements measured against the fixed bf16 bound |got - ref| <= 2e-2 + 1e-2 |ref|
# (without the widening by sum_j p_j |v_j| above), per compared case. Written as JSON to the
# path in CB_PARITY_REPORT at the end of the session, when that variable is set.
STRICT_ATTENTION = []


def record_strict_attention(what, got, ref):
    import numpy as np

    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    lim = 2e-2 + 1e-2 * np.abs(ref)
    STRICT_ATTENTION.append({"case": what, "elements": int(err.size), "outside_fixed_bound": int((err > lim).sum()),
                             "max_err_over_limit": float((err / lim).max()) if err.size else 0.0,
                             "max_abs_err": float(err.max()) if err.size else 0.0})


def pytest_sessionfinish(session, exitstatus):
    path = os.environ.get("CB_PARITY_REPORT")
    if path and STRICT_ATTENTION:
        import json

        with open(path, "w") as f:
            json.dump(STRICT_ATTENTION, f, indent=1)
