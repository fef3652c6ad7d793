"""fp64 numpy restatement of the blockwise online-softmax algebra -- TEST
INFRASTRUCTURE ONLY (see the package docstring for who may import it).

It follows the pages' own steps, in their order and notation:

* ``block_update`` is the per-block recurrence.  The source is "Ring
  Attention Paper Breakdown: Blockwise Distributed Transformers for
  Near-Infinite Context", section "3. Cross-Device Online Softmax
  Accumulator Math", steps 1-7: S = Q K^T / sqrt(d); m~ = rowmax(S);
  m' = max(m, m~); alpha = exp(m - m'); P = exp(S - m'); l' = alpha l +
  rowsum(P); O' = diag(alpha) O + P V.  "Ring Attention Math Deep", section
  "Accumulation math, step by step", states the same recurrence.
* ``identity_state`` is (m, l, O) = (-inf, 0, 0).  The source is the
  xf_ring_attention page, section "End-to-end flow": the accumulator starts
  at negative infinity, zero and zero, the identity of the merge.
* ``merge`` combines two partial states.  It takes the new max, rescales
  each side by exp(m_side - m_new), and adds.  The source is the
  xf_ring_attention page, section "The architecture: every piece explained"
  (the online softmax accumulator paragraph).
* ``finalize`` divides the accumulated O~ by l once the last block has been
  folded in ("Ring Attention Math Deep", section "Accumulation math, step
  by step").  LSE = m + ln l is the row log-sum-exp that
  "Ring Attention：把超长序列沿设备环流动", section "Backward
  需要让梯度也沿环传播", keeps for the backward pass.

Readings where the pages are silent:
* alpha = 0 when m = -inf.  In the worked example of "Ring Attention Math
  Deep" ("Accumulation math, step by step") the first block sets the max
  to 2 from an empty state and its rescale factor is zero.
* A row with no allowed key so far (m' = -inf) keeps its state: alpha = 1
  and P = 0, so (-inf) - (-inf) is never formed.
* finalize with l = 0 gives O = 0 and LSE = -inf.

States are tuples (m [n, h], l [n, h], o [n, h, d]) of float64 arrays.
"""
from __future__ import annotations

import numpy as np


def identity_state(nrows: int, heads: int, d: int):
    return (np.full((nrows, heads), -np.inf), np.zeros((nrows, heads)),
            np.zeros((nrows, heads, d)))


def _widen(x) -> np.ndarray:
    if not isinstance(x, np.ndarray):
        import torch

        x = x.detach().cpu().to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def scores(q, k, *, causal: bool, q_pos, k_pos, scale: float | None = None) -> np.ndarray:
    """S[r, h, t] = (q_r,h . k_t,kv(h)) * scale, -inf where causally masked."""
    q = _widen(q)
    k = _widen(k)
    nq, hq, d = q.shape
    nk, hkv, _ = k.shape
    group = hq // hkv
    kx = np.repeat(k, group, axis=1)  # query head h reads KV head h // group
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    s = np.einsum("rhx,thx->rht", q, kx) * scale
    if causal:
        qp = np.asarray(q_pos, dtype=np.int64)
        kp = np.asarray(k_pos, dtype=np.int64)
        allowed = kp[None, :] <= qp[:, None]  # [nq, nk]
        s = np.where(allowed[:, None, :], s, -np.inf)
    return s


def block_update(state, q, k, v, *, causal: bool, q_pos, k_pos, scale: float | None = None,
                 return_terms: bool = False):
    """Fold one K/V block into the running state (steps 1-7 of the
    recurrence, in that order).  With ``return_terms`` it also returns
    (alpha, P) so tests can read the intermediates the pages print."""
    m, l, o = state
    v = _widen(v)
    hq = m.shape[1]
    group = hq // v.shape[1]
    vx = np.repeat(v, group, axis=1)
    # 1. local block score
    s = scores(q, k, causal=causal, q_pos=q_pos, k_pos=k_pos, scale=scale)
    # 2. block row max (-inf for a row with no allowed key in this block)
    m_tilde = s.max(axis=2) if s.shape[2] > 0 else np.full(m.shape, -np.inf)
    # 3. global running max
    m_new = np.maximum(m, m_tilde)
    empty = np.isneginf(m_new)
    m_ref = np.where(empty, 0.0, m_new)
    # 4. rescaling factor (alpha = 0 when m = -inf; 1 for a still-empty row)
    alpha = np.where(empty, 1.0, np.exp(m - m_ref))
    # 5. local block exponentials
    p = np.exp(s - m_ref[:, :, None])
    # 6. running normalizer
    l_new = alpha * l + p.sum(axis=2)
    # 7. running output rescale and accumulate
    o_new = alpha[:, :, None] * o + np.einsum("rht,thx->rhx", p, vx)
    if return_terms:
        return (m_new, l_new, o_new), alpha, p
    return m_new, l_new, o_new


def merge(a, b):
    """a (+) b: new max, each side rescaled by exp(m_side - m_new), then added."""
    ma, la, oa = a
    mb, lb, ob = b
    m = np.maximum(ma, mb)
    empty = np.isneginf(m)
    m_ref = np.where(empty, 0.0, m)
    ea = np.exp(ma - m_ref)
    eb = np.exp(mb - m_ref)
    return m, ea * la + eb * lb, ea[..., None] * oa + eb[..., None] * ob


def finalize(state):
    """O = O~ / l and LSE = m + ln l."""
    m, l, o = state
    pos = l > 0
    safe = np.where(pos, l, 1.0)
    out = np.where(pos[..., None], o / safe[..., None], 0.0)
    lse = np.where(pos, m + np.log(safe), -np.inf)
    return out, lse


def ring_forward(q, k, v, *, P: int, causal: bool, order=None, scale: float | None = None):
    """The ring schedule on one host: virtual rank i keeps Q_i and folds
    K/V block j = (i - s) mod P at step s.  The source is "Ring Attention
    Math Deep", section "The ring schedule: passing K/V around".  Under
    causal masking a block strictly in the future of Q_i is skipped, per
    "Ring Attention：把超长序列沿设备环流动", section "Causal Attention
    让环不再完全对称".  ``order`` (optional) is a list, per rank, of the
    block indices to visit, so tests can permute the ring order.  Returns
    ``(O, LSE)`` in fp64."""
    q = _widen(q)
    k = _widen(k)
    v = _widen(v)
    n, hq, d = q.shape
    if n % P:
        raise ValueError("N must be a multiple of P")
    c = n // P
    out = np.zeros((n, hq, d))
    lse = np.zeros((n, hq))
    for i in range(P):
        rows = slice(i * c, (i + 1) * c)
        qpos = np.arange(i * c, (i + 1) * c)
        st = identity_state(c, hq, d)
        visit = order[i] if order is not None else [(i - s) % P for s in range(P)]
        for j in visit:
            if causal and j > i:
                continue  # the whole block is in the future: skipped
            kv = slice(j * c, (j + 1) * c)
            st = block_update(st, q[rows], k[kv], v[kv], causal=causal, q_pos=qpos,
                              k_pos=np.arange(j * c, (j + 1) * c), scale=scale)
        out[rows], lse[rows] = finalize(st)
    return out, lse
