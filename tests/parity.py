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

Gradients (bf16 inputs only) are compared element by element against the
oracle's absolute-term sum A of that element (the same sum with every term
replaced by its absolute value; see oracle/attention.c):
    |dX - dX_ref| <= 2^-7 * A + 1e-6 * max A.
Why this form: every product of the backward rounds one operand to bf16
(P for dV, dS for dQ and dK; D comes from the forward's O, whose P was
rounded too), a relative error of at most 2^-9 per term.  The standard
error bound of a sum is a multiple of the unit error times the sum of the
|terms|, not times |sum|: elements whose terms cancel (a late causal key
that few queries see, a query row whose dS nearly sums away) have a small
|dX_ref| but not a small error.  A model of the kernel's roundings in fp64
(P and dS rounded to bf16, O from bf16 P) stays below 3.3e-3 * A on every
element of the test cases, so 2^-7 = 7.8e-3 leaves a 2.4x margin.  A wrong
element is usually off by |dX_ref|, whose median is 4e-2 * A, and a key
whose gradient is dropped is off by 0.1-0.9 of its A: both fail.  The
1e-6 * max A floor only covers entries with no allowed pair (A = 0).
tests/test_grad_bar_host.py plants such mistakes in the oracle's gradients
on the CPU and checks that this bar rejects them.
"""
import numpy as np

TOL = {
    "bf16": {"o": 1e-2, "lse": 1e-3, "l": 2e-3, "grad": 2.0 ** -7, "grad_floor": 1e-6},
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


def grad_errors(x, ref, scale):
    """|x - ref| / (2^-7 A + 1e-6 max A) per element: the gradient bar's
    ratio (<= 1 passes), and the largest |x - ref| / A."""
    t = TOL["bf16"]
    x = _np(x)
    ref = np.asarray(ref, dtype=np.float64)
    scale = np.asarray(scale, dtype=np.float64)
    assert x.shape == ref.shape == scale.shape, (x.shape, ref.shape, scale.shape)
    if not ref.size:
        return np.zeros(0), 0.0
    err = np.abs(x - ref)
    bar = t["grad"] * scale + t["grad_floor"] * scale.max()
    ratio = np.where(bar > 0, err / np.where(bar > 0, bar, 1.0), np.where(err > 0, np.inf, 0.0))
    rel = (err / np.where(scale > 0, scale, np.inf)).max()
    return ratio, float(rel)


def check_grad(x, ref, scale, name="grad"):
    """|x - ref| <= 2^-7 * scale + 1e-6 * max(scale), element by element,
    where scale is the oracle's absolute-term sum of each element (the
    gradient bar; see the module docstring).  Returns max |x - ref| / scale."""
    xs = _np(x)
    assert np.isfinite(xs).all(), f"non-finite {name}"
    ratio, rel = grad_errors(xs, ref, scale)
    if ratio.size and ratio.max() > 1.0:
        i = np.unravel_index(int(ratio.argmax()), ratio.shape)
        raise AssertionError(
            f"{name}: element {i} off by {abs(xs[i] - ref[i]):.3e} (ref {ref[i]:.3e}, "
            f"absolute-term sum {scale[i]:.3e}); bar 2^-7 of that sum; {int((ratio > 1).sum())} "
            f"elements over")
    return rel


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
