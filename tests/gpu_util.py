"""Helpers shared by the GPU parity tests (no method arithmetic here)."""
import numpy as np
import pytest
import torch


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def lib():
    require_gpu()
    from chunked_linear_attention_gb300 import _build
    _build.build()
    import chunked_linear_attention_gb300 as cla
    cla.library()
    cla.set_wait_limit_ns(200_000_000)
    return cla


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def rel_l2(x, r) -> float:
    x = np.asarray(x, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    return float(np.linalg.norm(x - r) / max(np.linalg.norm(r), 1e-300))


def max_rel(x, r) -> float:
    """max |x - r| / max |r| over the tensor."""
    x = np.asarray(x, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    return float(np.max(np.abs(x - r)) / max(np.max(np.abs(r)), 1e-300))


def assert_status_ok(cla):
    st = cla.device_status()
    assert st == 0, f"device status {st}: {cla.status_string(st)}"
