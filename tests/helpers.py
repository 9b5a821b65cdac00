"""Shared helpers for the parity tests: metrics and tensor conversion."""
import numpy as np
import torch

# Output tolerance against the oracle's quantized-math result (fp64):
# relative L2 <= 5e-3 and max abs <= 2e-3.
REL_L2 = 5e-3
MAX_ABS = 2e-3


def f32(t: torch.Tensor) -> np.ndarray:
    """Exact fp32 numpy copy of an f16/bf16/fp32 tensor."""
    return t.detach().float().cpu().numpy()


def np_(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b.ravel())
    return float(np.linalg.norm((a - b).ravel()) / (den if den > 0 else 1.0))


def max_abs(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.abs(a - b).max()) if a.size else 0.0


def assert_close(gpu, ref, what="output", rel=REL_L2, abs_=MAX_ABS):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu) == np.isfinite(ref)), "%s: finiteness differs" % what
    fin = np.isfinite(ref)
    assert np.array_equal(gpu[~fin], ref[~fin]), "%s: non-finite entries differ" % what
    r, m = rel_l2(gpu[fin], ref[fin]), max_abs(gpu[fin], ref[fin])
    assert r <= rel and m <= abs_, "%s: rel-L2 %.3g (<= %.1g), max-abs %.3g (<= %.1g)" % (
        what, r, rel, m, abs_)
    return r, m
