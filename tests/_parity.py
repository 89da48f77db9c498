"""Comparison helpers for the GPU-vs-oracle parity tests.

Metric (stated with the tolerances next to each test): for O, dQ, dK, dV the
max-abs error normalised by the oracle tensor's RMS; for LSE the absolute max
error over finite entries, and -inf entries must coincide exactly.
"""
import numpy as np

# Tolerances for the two input precisions (fp32 inputs use the 3xTF32 path).
TOL = {
    "f32": {"O": 2e-3, "LSE": 1e-3, "grad": 5e-3},
    "bf16": {"O": 2e-2, "LSE": 1e-2, "grad": 2e-2},
}


def to_np(t):
    return t.detach().float().cpu().double().numpy()


def rms_err(got, ref):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite values in GPU output"
    rms = np.sqrt(np.mean(ref ** 2))
    if rms == 0.0:
        return float(np.abs(got - ref).max(initial=0.0))
    return float(np.abs(got - ref).max(initial=0.0) / rms)


def lse_err(got, ref):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    ninf_ref = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), ninf_ref), "-inf rows differ"
    fin = ~ninf_ref
    assert np.all(np.isfinite(got[fin])), "non-finite LSE on a non-empty row"
    return float(np.abs(got[fin] - ref[fin]).max(initial=0.0))
