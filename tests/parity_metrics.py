"""Pass metrics for comparing a CUDA result with the oracle.

* max relative error of a tensor: max_i |g_i - r_i| / max_i |r_i|, with the
  bound 1e-4 for fp32 and 2e-2 for bf16 (fp32 accumulation);
* "same argmax along every output row": rows are the last axis; a row whose
  argmax differs is accepted only when the two candidates are a near-tie in
  the reference, |r[a_g] - r[a_r]| <= tol * max|r| (ties break to the lowest
  index, as numpy does).
"""
import numpy as np

TOL = {"f32": 1e-4, "bf16": 2e-2}


def as_f64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().float().cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def max_rel_err(got, ref) -> float:
    got, ref = as_f64(got), as_f64(ref)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    scale = np.abs(ref).max()
    if scale == 0:
        return float(np.abs(got).max())
    return float(np.abs(got - ref).max() / scale)


def argmax_violations(got, ref, tol) -> int:
    got, ref = as_f64(got), as_f64(ref)
    if got.ndim == 1 or got.shape[-1] < 2:
        return 0
    g2 = got.reshape(-1, got.shape[-1])
    r2 = ref.reshape(-1, ref.shape[-1])
    ag = g2.argmax(1)
    ar = r2.argmax(1)
    bad = np.nonzero(ag != ar)[0]
    if bad.size == 0:
        return 0
    gap = np.abs(r2[bad, ag[bad]] - r2[bad, ar[bad]])
    return int((gap > tol * np.abs(ref).max()).sum())


def assert_close(name, got, ref, tol):
    err = max_rel_err(got, ref)
    assert err <= tol, f"{name}: max relative error {err:.3e} > {tol:.1e}"
    viol = argmax_violations(got, ref, tol)
    assert viol == 0, f"{name}: {viol} rows with a different argmax (not a near-tie)"
    return err
