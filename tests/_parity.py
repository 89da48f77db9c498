"""Comparison helpers for the GPU-vs-oracle parity tests.

Metric (stated with the tolerances next to each test): for O, dQ, dK, dV the
max-abs error normalised by the oracle tensor's RMS; for LSE the absolute max
error over finite entries, and -inf entries must coincide exactly.
"""
import numpy as np

# Tolerances for the two input precisions (fp32 inputs: either f32_mma form).
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


BF16_U = 2.0 ** -8  # unit roundoff of bf16 (8 significant bits, round to nearest)


def delta_perturbation_bounds(q, k, do, o_ref, lse_ref, scale, causal, window):
    """Per-element bounds on how far dQ and dK move when the backward is given O
    rounded to bf16 (bf16 outputs: the O a caller stores and passes back).

    The backward forms Delta_i = sum_d dO_id O_id from the O it is given. Rounding O to
    bf16 moves each element by at most u |O_id| (u = 2^-8), so Delta_i moves by at
    most e_i = u sum_d |dO_id O_id|, and dS_ij = P_ij (dP_ij - Delta_i) by P_ij e_i.
    Through dQ_i = scale sum_j dS_ij K_j and dK_j = scale sum_i dS_ij Q_i (summed over
    a kv head's query heads):
        |delta dQ_id| <= scale e_i sum_j P_ij |K_jd|
        |delta dK_jd| <= scale sum_i P_ij e_i |Q_id|
    with P_ij = exp(scale q_i . k_j - LSE_i) on the visible pairs (query i sees key j
    iff (not causal or j <= i) and (window == 0 or j >= i - window + 1)). dV does not
    involve Delta. Inputs: CPU tensors / arrays in the oracle's layout [B, heads, S, D];
    o_ref and lse_ref the oracle's forward outputs. Returns (bound_dq, bound_dk)."""
    qn, kn, don = (np.asarray(t.double().numpy() if hasattr(t, "double") else t, np.float64)
                   for t in (q, k, do))
    o_ref, lse_ref = np.asarray(o_ref, np.float64), np.asarray(lse_ref, np.float64)
    B, H, Sq, D = qn.shape
    HKV, Sk = kn.shape[1], kn.shape[2]
    rep = H // HKV
    i = np.arange(Sq)[:, None]
    j = np.arange(Sk)[None, :]
    vis = np.ones((Sq, Sk), bool)
    if causal:
        vis &= j <= i
    if window:
        vis &= j >= i - window + 1
    bq = np.zeros_like(qn)
    bk = np.zeros_like(kn)
    for b in range(B):
        for h in range(H):
            g = h // rep
            lse = lse_ref[b, h]
            live = np.isfinite(lse)
            s = scale * (qn[b, h] @ kn[b, g].T) - np.where(live, lse, 0.0)[:, None]
            p = np.where(vis & live[:, None], np.exp(np.minimum(s, 0.0)), 0.0)
            e = BF16_U * np.sum(np.abs(don[b, h]) * np.abs(o_ref[b, h]), axis=1)
            bq[b, h] = scale * e[:, None] * (p @ np.abs(kn[b, g]))
            bk[b, g] += scale * (p.T @ (e[:, None] * np.abs(qn[b, h])))
    return bq, bk


def bf16_output_excess(got, ref, extra=0.0):
    """max over elements of |got - ref| - u |ref| - extra, in units of RMS(ref) (of 1
    where ref is identically 0, as rms_err does): the error left once bf16's rounding
    of each stored element (u = 2^-8) and a derived perturbation `extra` are allowed."""
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite values in GPU output"
    rms = np.sqrt(np.mean(ref ** 2))
    ex = np.abs(got - ref) - BF16_U * np.abs(ref) - extra
    return float(ex.max(initial=0.0) / (rms if rms > 0.0 else 1.0))
