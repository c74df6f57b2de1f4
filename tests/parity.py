"""Comparison helpers for GPU-vs-oracle parity tests.

Tolerances: floating-point outputs (per-layer residual stream, logits)
must satisfy max|gpu - oracle| <= 2e-3 * max|oracle|; greedy tokens must
agree wherever the oracle's top-2 logit gap exceeds 1e-2 (elsewhere the
oracle's token is fed to both sides so the runs stay aligned).  Dequantised
weights and KV-fork copies are compared bit for bit.
"""
import numpy as np

REL_TOL = 2e-3
GAP = 1e-2


def rel_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = np.max(np.abs(ref))
    return float(np.max(np.abs(got - ref)) / (scale if scale > 0 else 1.0))


def assert_close(got, ref, what: str, tol: float = REL_TOL):
    e = rel_err(got, ref)
    assert e <= tol, f"{what}: max abs err / Linf = {e:.3e} > {tol:.1e}"
    return e


def check_greedy(gpu_logits, ref_logits, what: str):
    ref = np.asarray(ref_logits, dtype=np.float64)
    top = np.argsort(ref)[-2:]
    gap = ref[top[1]] - ref[top[0]]
    g = int(np.argmax(np.asarray(gpu_logits)))
    o = int(np.argmax(ref))
    if gap > GAP:
        assert g == o, f"{what}: greedy token {g} != oracle {o} (gap {gap:.3g})"
    return o
