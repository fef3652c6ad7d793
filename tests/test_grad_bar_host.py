"""The gradient bar (parity.check_grad) on the CPU: it must reject the
mistakes a backward ring can plausibly make, and accept the rounding a
correct bf16 kernel makes.

Every mistake is planted in the oracle's own gradients ("Ring Attention：把
超长序列沿设备环流动", section "Backward 需要让梯度也沿环传播": each
(Q block, K/V block) pair adds to dQ, dK and dV):
* the last key tile's dK and dV never written (a dropped tile);
* the pairs of the last query block never folded into dK and dV (a ring
  step skipped), computed by the oracle with that block's rows left out;
* D = rowsum(dO * O) left out of dS;
* the wrong KV head for a query head (h % Hkv instead of h // g).
The accepted case is a model of the kernel's roundings in fp64: P and dS
rounded to bf16 before their products, O of the forward from bf16 P.
"""
import numpy as np
import pytest
import torch

import oracle
from blockwise_online_softmax_gb300 import inputs
from parity import check_grad, grad_errors

N, P, HQ, HKV, D = 256, 4, 4, 2, 32
C = N // P


@pytest.fixture(scope="module")
def case():
    q, k, v = inputs.make_random(N, HQ, HKV, D, seed=71)
    g = inputs.randn_chunked((N, HQ, D), 71, 3).to(torch.bfloat16)
    refs, scales, lse = oracle.backward_with_scales(q, k, v, g, causal=True)
    return q, k, v, g, refs, scales


def _fails(x, ref, a):
    with pytest.raises(AssertionError):
        check_grad(x, ref, a)


def _bf16(x):
    return torch.from_numpy(x).to(torch.float32).to(torch.bfloat16).double().numpy()


def _rounded_backward(q, k, v, g):
    """fp64 backward with the kernel's bf16 roundings: forward O = bf16(P) V / l,
    then P and dS rounded to bf16 before the products that read them."""
    q, k, v, g = (t.double().numpy() for t in (q, k, v, g))
    sc = 1.0 / np.sqrt(D)
    grp = HQ // HKV
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    allowed = np.tril(np.ones((N, N), dtype=bool))
    for h in range(HQ):
        kh = h // grp
        s = np.where(allowed, q[:, h] @ k[:, kh].T * sc, -np.inf)
        m = s.max(1, keepdims=True)
        p = np.exp(s - m)
        l = p.sum(1, keepdims=True)
        o = _bf16(p) @ v[:, kh] / l
        pn = np.exp(s - (m + np.log(l)))
        dvec = (g[:, h] * o).sum(1, keepdims=True)
        dv[:, kh] += _bf16(pn).T @ g[:, h]
        ds = _bf16(pn * (g[:, h] @ v[:, kh].T - dvec) * sc)
        dq[:, h] = ds @ k[:, kh]
        dk[:, kh] += ds.T @ q[:, h]
    return dq, dk, dv


def test_the_kernels_rounding_passes(case):
    q, k, v, g, refs, scales = case
    for x, r, a in zip(_rounded_backward(q, k, v, g), refs, scales):
        ratio, rel = grad_errors(x, r, a)
        assert ratio.max() <= 0.6, ratio.max()   # well inside the bar
        check_grad(x, r, a)


def test_a_dropped_last_key_tile_fails(case):
    _, _, _, _, (dq, dk, dv), (aq, ak, av) = case
    for x, r, a in ((dk, dk, ak), (dv, dv, av)):
        bad = x.copy()
        bad[-C:] = 0.0
        _fails(bad, r, a)


def test_a_dropped_last_key_fails_and_the_old_global_bar_missed_it(case):
    # The last key is seen by one query row: its gradient is tiny next to
    # the largest one, so a bar scaled by max |ref| (the old form) accepts
    # a zero there.  The element-wise bar does not.
    _, _, _, _, (_, dk, _), (_, ak, _) = case
    bad = dk.copy()
    bad[-1] = 0.0
    assert np.abs(bad - dk).max() <= 2e-2 * np.abs(dk).max()
    _fails(bad, dk, ak)


def test_a_skipped_ring_step_fails(case):
    # dK and dV without the pairs of the last query block: the oracle run
    # with that block's rows left out (LSE = -inf drops a row's terms).
    q, k, v, g, (_, dk, dv), (_, ak, av) = case
    _, lse, dvec = oracle.grad_q(q, k, v, g, causal=True)
    lse = lse.copy()
    lse[-C:] = -np.inf
    bad_k, bad_v = oracle.grad_kv(q, k, v, g, lse, dvec, causal=True)
    _fails(bad_k, dk, ak)
    _fails(bad_v, dv, av)


def test_a_dropped_d_term_fails(case):
    q, k, v, g, (_, dk, _), (_, ak, _) = case
    _, lse, dvec = oracle.grad_q(q, k, v, g, causal=True)
    bad_k, _ = oracle.grad_kv(q, k, v, g, lse, np.zeros_like(dvec), causal=True)
    _fails(bad_k, dk, ak)


def test_a_wrong_head_mapping_fails(case):
    # Query head h read KV head h % HKV instead of h // (HQ / HKV): the same
    # as the right mapping with the query heads permuted.
    q, k, v, g, (dq, _, _), (aq, _, _) = case
    perm = np.array([0, 2, 1, 3])
    bad, _, _, _ = oracle.backward(q[:, perm], k, v, g[:, perm], causal=True)
    _fails(bad[:, np.argsort(perm)], dq, aq)
