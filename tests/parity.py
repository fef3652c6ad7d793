"""Tolerances and comparison helpers for the GPU-vs-oracle parity tests.

The stated bars:
* bf16 inputs with fp32 accumulation: max |O - O_ref| <= 1e-2, and
  |LSE - LSE_ref| <= 1e-3 * max(1, |LSE_ref|).  The floor keeps the relative
  bound meaningful near LSE = 0.
* fp32 inputs: max |O - O_ref| <= 1e-5, and the same floored form with 1e-5
  for LSE.

States (m, l, O~) are compared in their canonical form, relative to the
exact running max:
* |m - m_ref| <= tol_lse * max(1, |m_ref|)
* |l - l_ref| <= tol_l * l_ref
* |O~ - O~_ref| <= tol_o * l_ref, elementwise.  O~ is a weighted sum with
  total weight l, so its error scales with l.

Gradients (bf16 inputs only) are compared per tensor against the largest
reference magnitude: max |dX - dX_ref| <= 2e-2 * max |dX_ref|.  Each
product in the backward rounds one operand to bf16 (P for dV, dS for dQ
and dK), a relative error of at most 2^-9 per term; summed over the keys
(or queries) with mixed signs, the error of an output element stays a few
times 2^-9 of the largest |term| sums, which the bar covers with margin.
"""
import numpy as np

TOL = {
    "bf16": {"o": 1e-2, "lse": 1e-3, "l": 2e-3, "grad": 2e-2},
    "f32": {"o": 1e-5, "lse": 1e-5, "l": 1e-5},
}


def _np(x):
    import torch

    if isinstance(x, torch.Tensor):
        return x.detach().cpu().to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def check_output(out, lse, ref_out, ref_lse, kind):
    """max |O - O_ref| and the floored relative LSE error against the bars."""
    t = TOL[kind]
    out, lse = _np(out), _np(lse)
    assert out.shape == ref_out.shape and lse.shape == ref_lse.shape
    assert np.isfinite(out).all(), "non-finite output"
    err_o = np.abs(out - ref_out).max() if out.size else 0.0
    fin = np.isfinite(ref_lse)
    assert (np.isneginf(lse) == ~fin).all(), "LSE -inf pattern differs"
    err_l = (np.abs(lse[fin] - ref_lse[fin]) / np.maximum(1.0, np.abs(ref_lse[fin]))).max() \
        if fin.any() else 0.0
    assert err_o <= t["o"], f"max |O - O_ref| = {err_o:.3e} > {t['o']}"
    assert err_l <= t["lse"], f"LSE rel err = {err_l:.3e} > {t['lse']}"
    return err_o, err_l


def check_state(m, l, o, ref, kind):
    t = TOL[kind]
    m, l, o = _np(m), _np(l), _np(o)
    mr, lr, orf = ref
    assert (np.isneginf(m) == np.isneginf(mr)).all(), "m -inf pattern differs"
    fin = np.isfinite(mr)
    if fin.any():
        em = (np.abs(m[fin] - mr[fin]) / np.maximum(1.0, np.abs(mr[fin]))).max()
        assert em <= t["lse"], f"m err {em:.3e}"
        el = (np.abs(l[fin] - lr[fin]) / lr[fin]).max()
        assert el <= t["l"], f"l rel err {el:.3e}"
        eo = (np.abs(o - orf)[fin] / lr[fin][:, None]).max()
        assert eo <= t["o"], f"O~ err / l = {eo:.3e}"
    # rows with no allowed key keep the identity state
    assert (l[~fin] == 0).all() and (o[~fin] == 0).all()


def check_grad(x, ref, name="grad"):
    """max |x - ref| <= TOL["bf16"]["grad"] * max |ref| (the gradient bar)."""
    x = _np(x)
    ref = np.asarray(ref, dtype=np.float64)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    assert np.isfinite(x).all(), f"non-finite {name}"
    scale = np.abs(ref).max() if ref.size else 0.0
    err = np.abs(x - ref).max() if ref.size else 0.0
    assert err <= TOL["bf16"]["grad"] * max(scale, 1e-30), \
        f"{name}: max err {err:.3e} > {TOL['bf16']['grad']} x {scale:.3e}"
    return err / max(scale, 1e-30)


def assert_fused_matches(out, lse, ref_out, ref_lse):
    """The fused bf16 ring against the same ring run step by step: the same
    products and the same state updates in the same order, so they differ
    only in the last fp32 roundings of the finalize (out = O~ / l, and LSE
    from the log2-unit max)."""
    import torch

    assert (out - ref_out).abs().max().item() <= 1e-6
    fin = torch.isfinite(ref_lse)
    assert torch.equal(torch.isfinite(lse), fin)
    err = ((lse - ref_lse).abs() / ref_lse.abs().clamp(min=1.0))[fin]
    assert err.numel() == 0 or err.max().item() <= 1e-6
