"""Pins for the CPU oracle.  These tests run on CPU only.

Each test ties the oracle to a fact that does not come from the oracle
itself:
* the worked example the pages print,
* special cases that reduce to library routines (scipy softmax and
  logsumexp),
* closed forms,
* brute force in exact arithmetic,
* invariants.
Each test is chosen so that a plausible slip fails it: a dropped scale, a
wrong sign, a wrong head or row index, an off-by-one in the causal mask, or
a transposed operand.
"""
import itertools
import math
from fractions import Fraction

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from oracle import online
from blockwise_online_softmax_gb300 import inputs


def _example(golden):
    g = golden("worked_example.txt")
    s = np.array(g["block_A.s"] + g["block_B.s"], dtype=np.float32)
    v = np.array(g["block_A.v"] + g["block_B.v"], dtype=np.float32)
    # d = 1, q = 1, scale = 1: the score of key t is exactly k_t.
    q = np.ones((1, 1, 1), dtype=np.float32)
    k = s.reshape(4, 1, 1)
    vv = v.reshape(4, 1, 1)
    return g, q, k, vv


# --- the worked example ("Ring Attention Math Deep", "A worked numeric example")

def test_worked_example_dense_output(golden):
    g, q, k, v = _example(golden)
    out, lse = oracle.attention(q, k, v, causal=False, scale=1.0)
    assert abs(out[0, 0, 0] - g["out"]) <= g["tol"]
    assert abs(out[0, 0, 0] - g["direct"]) <= g["tol"]
    # the full-set state equals the page's state after block B
    m, l, o = oracle.partial_state(q, k, v, causal=False, scale=1.0)
    assert m[0, 0] == g["after_B.m"]
    assert abs(l[0, 0] - g["after_B.l"]) <= g["tol"]
    assert abs(o[0, 0, 0] - g["after_B.o"]) <= g["tol"]
    # LSE is consistent with the state: ln of the sum of exp(scores)
    assert abs(lse[0, 0] - (m[0, 0] + math.log(l[0, 0]))) < 1e-12


def test_worked_example_block_A_state(golden):
    g, q, k, v = _example(golden)
    m, l, o = oracle.partial_state(q, k[:2], v[:2], causal=False, scale=1.0)
    assert m[0, 0] == g["after_A.m"]
    assert abs(l[0, 0] - g["after_A.l"]) <= g["tol"]
    assert abs(o[0, 0, 0] - g["after_A.o"]) <= g["tol"]


def test_worked_example_online_intermediates(golden):
    g, q, k, v = _example(golden)
    st = online.identity_state(1, 1, 1)
    pos = np.arange(4)
    st, alpha, p = online.block_update(st, q, k[:2], v[:2], causal=False, q_pos=[0],
                                       k_pos=pos[:2], scale=1.0, return_terms=True)
    assert st[0][0, 0] == g["after_A.m"] and alpha[0, 0] == g["after_A.alpha"]
    np.testing.assert_allclose(p[0, 0], g["after_A.p"], atol=g["tol"])
    assert abs(st[1][0, 0] - g["after_A.l"]) <= g["tol"]
    assert abs(st[2][0, 0, 0] - g["after_A.o"]) <= g["tol"]
    st, alpha, p = online.block_update(st, q, k[2:], v[2:], causal=False, q_pos=[0],
                                       k_pos=pos[2:], scale=1.0, return_terms=True)
    assert st[0][0, 0] == g["after_B.m"]
    assert abs(alpha[0, 0] - g["after_B.alpha"]) <= g["tol"]
    np.testing.assert_allclose(p[0, 0], g["after_B.p"], atol=g["tol"])
    assert abs(st[1][0, 0] - g["after_B.l"]) <= g["tol"]
    assert abs(st[2][0, 0, 0] - g["after_B.o"]) <= g["tol"]
    out, _ = online.finalize(st)
    assert abs(out[0, 0, 0] - g["out"]) <= g["tol"]


def test_worked_example_merge_and_finalize(golden):
    g, q, k, v = _example(golden)
    a = oracle.partial_state(q, k[:2], v[:2], causal=False, scale=1.0)
    b = oracle.partial_state(q, k[2:], v[2:], causal=False, scale=1.0)
    for x, y in ((a, b), (b, a)):
        m, l, o = online.merge(x, y)
        assert m[0, 0] == g["after_B.m"]
        assert abs(l[0, 0] - g["after_B.l"]) <= g["tol"]
        assert abs(o[0, 0, 0] - g["after_B.o"]) <= g["tol"]
        out, _ = online.finalize((m, l, o))
        assert abs(out[0, 0, 0] - g["out"]) <= g["tol"]


# --- special cases that reduce to library routines

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_onehot_values_return_softmax_rows(causal, dtype):
    """With v_t = e_t (one-hot), row r of O is row r of softmax(S).  It is
    checked against scipy.special.softmax of a numpy matmul, per head,
    with GQA.  The shapes are non-square (nq != nk, d != nk) so a transposed
    operand cannot pass."""
    nq, nk, hq, hkv, d = 7, 12, 4, 2, 16
    g = torch.Generator().manual_seed(3)
    q = torch.randn(nq, hq, d, generator=g).to(dtype)
    k = torch.randn(nk, hkv, d, generator=g).to(dtype)
    v = torch.zeros(nk, hkv, d, dtype=dtype)
    for t in range(nk):
        v[t, :, t] = 1.0
    q_pos = np.arange(nq) + 3  # queries sit at positions 3..9, keys at 0..11
    out, lse = oracle.attention(q, k, v, causal=causal, q_pos=q_pos)
    qd = q.to(torch.float64).numpy()
    kd = k.to(torch.float64).numpy()
    for h in range(hq):
        s = qd[:, h, :] @ kd[:, h // (hq // hkv), :].T / math.sqrt(d)
        if causal:
            s = np.where(np.arange(nk)[None, :] <= q_pos[:, None], s, -np.inf)
        ref = scipy.special.softmax(s, axis=1)
        np.testing.assert_allclose(out[:, h, :nk], ref, rtol=0, atol=1e-13)
        np.testing.assert_allclose(out[:, h, nk:], 0.0, atol=0)
        np.testing.assert_allclose(lse[:, h], scipy.special.logsumexp(s, axis=1), atol=1e-12)


def test_gqa_equals_repeated_kv_heads():
    """Query head h reads KV head h // (hq/hkv): the same as MHA with each
    KV head repeated hq/hkv times in a row (np.repeat)."""
    q, k, v = inputs.make_random(40, 6, 2, 8, dtype=torch.float32, seed=5)
    o1, l1 = oracle.attention(q, k, v, causal=True)
    kr = np.repeat(k.numpy(), 3, axis=1)
    vr = np.repeat(v.numpy(), 3, axis=1)
    o2, l2 = oracle.attention(q, kr, vr, causal=True)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    # and not the interleaved convention h % hkv
    kt = np.tile(k.numpy(), (1, 3, 1))
    vt = np.tile(v.numpy(), (1, 3, 1))
    o3, _ = oracle.attention(q, kt, vt, causal=True)
    assert np.abs(o1 - o3).max() > 1e-2


# --- closed forms

def test_equal_keys_give_running_mean():
    """If every key is the same vector, every allowed score is equal.  The
    weights are then uniform: causal row r gets mean(v_0..v_r), and the
    non-causal rows get the global mean."""
    n, h, d = 33, 2, 8
    g = torch.Generator().manual_seed(7)
    q = torch.randn(n, h, d, generator=g)
    k = torch.randn(1, h, d, generator=g).expand(n, h, d).contiguous()
    v = torch.randn(n, h, d, generator=g)
    out, lse = oracle.attention(q, k, v, causal=True)
    vd = v.double().numpy()
    running_mean = np.cumsum(vd, axis=0) / np.arange(1, n + 1)[:, None, None]
    np.testing.assert_allclose(out, running_mean, atol=1e-13)
    s = (q.double() * k.double()).sum(-1).numpy() / math.sqrt(d)
    np.testing.assert_allclose(lse, s + np.log(np.arange(1, n + 1))[:, None], atol=1e-12)
    out_nc, _ = oracle.attention(q, k, v, causal=False)
    np.testing.assert_allclose(out_nc, np.broadcast_to(vd.mean(0), out_nc.shape), atol=1e-13)


def test_causal_row_zero_is_its_own_value():
    q, k, v = inputs.make_random(16, 3, 3, 8, dtype=torch.float32, seed=2)
    out, lse = oracle.attention(q, k, v, causal=True)
    np.testing.assert_array_equal(out[0], v[0].double().numpy())
    s00 = (q[0].double() * k[0].double()).sum(-1).numpy() / math.sqrt(8)
    np.testing.assert_allclose(lse[0], s00, atol=1e-14)


def test_dominant_key_large_logits():
    """Scores scaled by 100 (|s| up to ~1e3): no overflow, and the output is
    the value of the arg-max key to machine precision."""
    q, k, v = inputs.make_random(20, 2, 2, 8, dtype=torch.float32, seed=11, scale=1.0)
    q = q * 100.0
    out, lse = oracle.attention(q, k, v, causal=False)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    s = np.einsum("rhx,thx->rht", q.double().numpy(), k.double().numpy()) / math.sqrt(8)
    top = s.argmax(axis=2)
    srt = np.sort(s, axis=2)
    gap = srt[:, :, -1] - srt[:, :, -2]
    for r in range(20):
        for h in range(2):
            if gap[r, h] > 40:  # runner-up weight < e^-40
                np.testing.assert_allclose(out[r, h], v[top[r, h], h].double().numpy(),
                                           atol=1e-15)
                np.testing.assert_allclose(lse[r, h], srt[r, h, -1], atol=1e-15)


def test_values_all_one_give_one():
    q, k, _ = inputs.make_random(50, 4, 2, 16, dtype=torch.bfloat16, seed=4)
    v = torch.ones(50, 2, 16, dtype=torch.bfloat16)
    for causal in (False, True):
        out, _ = oracle.attention(q, k, v, causal=causal)
        np.testing.assert_allclose(out, 1.0, atol=1e-14)


# --- brute force in exact arithmetic

def test_brute_force_exact_rationals_tiny():
    """Tiny inputs with integer scores: sum_t e^{s_t} v_t / sum_t e^{s_t} with
    no max shift.  Evaluated as exact rationals in x = e (scores in 0..3 give
    powers of e, a polynomial ratio), then turned to float once.  This needs
    no exp() and no floating-point order."""
    # d = 1, scale = 1: score(r, t) = q_r * k_t, integers in [-3, 3]
    qv = [1, -1, 2, 0, 1]
    kv = [0, 1, -1, 1, 2, -2]
    # values exactly representable in float32, so the inputs are exact too
    vv = [Fraction(1), Fraction(-2), Fraction(3, 2), Fraction(5), Fraction(-3, 8), Fraction(2)]
    q = np.array(qv, dtype=np.float32).reshape(5, 1, 1)
    k = np.array(kv, dtype=np.float32).reshape(6, 1, 1)
    v = np.array([float(x) for x in vv], dtype=np.float32).reshape(6, 1, 1)
    for causal in (False, True):
        out, lse = oracle.attention(q, k, v, causal=causal, scale=1.0)
        for r in range(5):
            allowed = [t for t in range(6) if not causal or t <= r]
            # ratio of polynomials in e with exponents s + 8 (all >= 0)
            num = {}
            den = {}
            for t in allowed:
                p = qv[r] * kv[t] + 8
                num[p] = num.get(p, Fraction(0)) + vv[t]
                den[p] = den.get(p, Fraction(0)) + 1

            def ev(poly):
                return math.fsum(float(c) * math.e ** p for p, c in poly.items())
            assert abs(out[r, 0, 0] - ev(num) / ev(den)) < 1e-13
            assert abs(lse[r, 0] - (math.log(ev(den)) - 8)) < 1e-13


def test_brute_force_pairs_no_max_shift():
    """Explicit (r, t) loops in pure Python with math.fsum, no max shift,
    on random tiny inputs with causal and GQA."""
    nq, hq, hkv, d = 9, 4, 2, 4
    g = torch.Generator().manual_seed(21)
    q = torch.randn(nq, hq, d, generator=g)
    k = torch.randn(nq, hkv, d, generator=g)
    v = torch.randn(nq, hkv, d, generator=g)
    out, lse = oracle.attention(q, k, v, causal=True)
    qd, kd, vd = q.tolist(), k.tolist(), v.tolist()
    for r in range(nq):
        for h in range(hq):
            kh = h // 2
            w = []
            for t in range(r + 1):
                s = math.fsum(qd[r][h][x] * kd[t][kh][x] for x in range(d)) / math.sqrt(d)
                w.append(math.exp(s))
            den = math.fsum(w)
            for x in range(d):
                num = math.fsum(w[t] * vd[t][kh][x] for t in range(r + 1))
                assert abs(out[r, h, x] - num / den) < 1e-13
            assert abs(lse[r, h] - math.log(den)) < 1e-13


# --- invariants

def test_permutation_equivariance():
    """Non-causal: permuting key/value rows together leaves O unchanged, and
    permuting the query rows permutes the output rows."""
    q, k, v = inputs.make_random(24, 2, 1, 8, dtype=torch.float32, seed=9)
    out, lse = oracle.attention(q, k, v, causal=False)
    perm = np.random.default_rng(0).permutation(24)
    out_k, lse_k = oracle.attention(q, k[perm], v[perm], causal=False)
    np.testing.assert_allclose(out_k, out, atol=1e-14)
    np.testing.assert_allclose(lse_k, lse, atol=1e-14)
    out_q, _ = oracle.attention(q[perm], k, v, causal=False)
    np.testing.assert_array_equal(out_q, out[perm])


def test_linear_in_values_and_shift_in_scores():
    q, k, v = inputs.make_random(16, 2, 2, 8, dtype=torch.float32, seed=13)
    out, lse = oracle.attention(q, k, v, causal=True)
    out3, lse3 = oracle.attention(q, k, v * 4.0, causal=True)
    np.testing.assert_allclose(out3, 4.0 * out, atol=1e-13)
    np.testing.assert_array_equal(lse3, lse)
    # Append a constant coordinate (1 in q, c in k).  Every score of row r
    # moves by c / sqrt(d'), so O stays and LSE shifts by the same amount.
    c = 3.0
    q2 = torch.cat([q, torch.ones(16, 2, 1)], dim=2)
    k2 = torch.cat([k, torch.full((16, 2, 1), c)], dim=2)
    v2 = torch.cat([v, torch.zeros(16, 2, 1)], dim=2)
    sc = 1.0 / math.sqrt(8)
    out2, lse2 = oracle.attention(q2, k2, v2, causal=True, scale=sc)
    np.testing.assert_allclose(out2[..., :8], out, atol=1e-13)
    np.testing.assert_allclose(lse2, lse + c * sc, atol=1e-13)


def test_rows_subset_positions_and_threads():
    q, k, v = inputs.make_random(30, 2, 1, 8, dtype=torch.bfloat16, seed=17)
    full, full_lse = oracle.attention(q, k, v, causal=True, threads=1)
    rows = np.array([29, 0, 7, 7, 15])
    sub, sub_lse = oracle.attention(q, k, v, causal=True, rows=rows, threads=4)
    np.testing.assert_array_equal(sub, full[rows])
    np.testing.assert_array_equal(sub_lse, full_lse[rows])
    pos = np.arange(30)
    exp_, exp_lse = oracle.attention(q, k, v, causal=True, q_pos=pos, k_pos=pos)
    np.testing.assert_array_equal(exp_, full)
    # bf16 bit patterns are widened exactly: same as passing float32 values
    f32, _ = oracle.attention(q.float(), k.float(), v.float(), causal=True)
    np.testing.assert_array_equal(f32, full)


def test_row_without_allowed_key():
    q, k, v = inputs.make_random(4, 1, 1, 8, dtype=torch.float32, seed=1)
    m, l, o = oracle.partial_state(q, k, v, causal=True, q_pos=[0, 1, 5, 9],
                                   k_pos=[2, 3, 4, 5])
    assert np.isneginf(m[0, 0]) and l[0, 0] == 0 and not o[0].any()
    assert np.isneginf(m[1, 0]) and l[1, 0] == 0
    out, lse = oracle.attention(q, k, v, causal=True, q_pos=[0, 1, 5, 9], k_pos=[2, 3, 4, 5])
    assert np.isneginf(lse[0, 0]) and not out[0].any()
    assert np.isfinite(lse[2:]).all()


def test_online_ring_equals_dense():
    """The pages' blockwise ring (fp64 recurrence) equals the dense definition."""
    q, k, v = inputs.make_random(64, 4, 2, 8, dtype=torch.bfloat16, seed=23)
    for causal in (False, True):
        ref, ref_lse = oracle.attention(q, k, v, causal=causal)
        out, lse = online.ring_forward(q, k, v, P=4, causal=causal)
        np.testing.assert_allclose(out, ref, atol=1e-12)
        np.testing.assert_allclose(lse, ref_lse, atol=1e-12)


def test_ring_order_and_merge_order_independence():
    """Any order of visiting the blocks, and any order of merging the block
    states, gives the same result (all 4! orders, within 1e-12)."""
    q, k, v = inputs.make_random(32, 2, 2, 8, dtype=torch.float32, seed=29)
    ref, ref_lse = oracle.attention(q, k, v, causal=False)
    for perm in itertools.permutations(range(4)):
        out, lse = online.ring_forward(q, k, v, P=4, causal=False, order=[list(perm)] * 4)
        np.testing.assert_allclose(out, ref, atol=1e-12)
        np.testing.assert_allclose(lse, ref_lse, atol=1e-12)
    # merge of block partial states, from the C oracle, in every order
    parts = [oracle.partial_state(q, k[j * 8:(j + 1) * 8], v[j * 8:(j + 1) * 8], causal=False)
             for j in range(4)]
    for perm in itertools.permutations(range(4)):
        st = online.identity_state(32, 2, 8)
        for j in perm:
            st = online.merge(st, parts[j])
        out, lse = online.finalize(st)
        np.testing.assert_allclose(out, ref, atol=1e-12)
        np.testing.assert_allclose(lse, ref_lse, atol=1e-12)


def test_identity_state_is_neutral():
    q, k, v = inputs.make_random(8, 2, 2, 4, dtype=torch.float32, seed=31)
    st = oracle.partial_state(q, k, v, causal=True)
    e = online.identity_state(8, 2, 4)
    for a, b in ((st, e), (e, st)):
        m, l, o = online.merge(a, b)
        np.testing.assert_array_equal(m, st[0])
        np.testing.assert_array_equal(l, st[1])
        np.testing.assert_array_equal(o, st[2])


def test_normalize_then_average_is_wrong():
    """Normalizing each block on its own and then averaging is not attention
    ("Ring Attention Math Deep", "Causal masking, load balance, and other
    wrinkles").  The oracle tells the two apart."""
    q, k, v = inputs.make_random(32, 2, 2, 8, dtype=torch.float32, seed=37)
    ref, _ = oracle.attention(q, k, v, causal=False)
    blocks = [oracle.attention(q, k[j * 8:(j + 1) * 8], v[j * 8:(j + 1) * 8], causal=False)[0]
              for j in range(4)]
    wrong = sum(blocks) / 4
    assert np.abs(wrong - ref).max() > 1e-2


# --- masks beyond causal: window, packed documents, padding ("Ring Attention：
# 把超长序列沿设备环流动", "正确性测试应覆盖哪些边界")

def _rand(n, h, d, seed):
    g = np.random.default_rng(seed)
    return g.standard_normal((n, h, d)).astype(np.float32)


def test_causal_window_one_is_the_own_value():
    # With causal and window 1 a row sees only itself: O = v_r, LSE = s_rr.
    q, k, v = _rand(40, 2, 8, 1), _rand(40, 2, 8, 2), _rand(40, 2, 8, 3)
    out, lse = oracle.attention(q, k, v, causal=True, window=1)
    assert np.array_equal(out, v.astype(np.float64))
    s_rr = (q.astype(np.float64) * k.astype(np.float64)).sum(-1) / math.sqrt(8)
    assert np.abs(lse - s_rr).max() < 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_window_equals_the_explicit_key_slice(causal):
    # Row r with window W sees exactly the keys r-W+1 .. r+W-1 (.. r if
    # causal).  Hand the oracle that slice, positions kept, with no window.
    n, W = 57, 6
    q, k, v = _rand(n, 3, 4, 4), _rand(n, 3, 4, 5), _rand(n, 3, 4, 6)
    out, lse = oracle.attention(q, k, v, causal=causal, window=W)
    for r in range(n):
        lo, hi = max(0, r - W + 1), (r + 1 if causal else min(n, r + W))
        o2, l2 = oracle.attention(q[r:r + 1], k[lo:hi], v[lo:hi], causal=False)
        assert np.abs(out[r] - o2[0]).max() < 1e-13
        assert np.abs(lse[r] - l2[0]).max() < 1e-13


def test_window_wider_than_the_sequence_changes_nothing():
    q, k, v = _rand(33, 2, 8, 7), _rand(33, 2, 8, 8), _rand(33, 2, 8, 9)
    for causal in (False, True):
        a = oracle.attention(q, k, v, causal=causal)
        b = oracle.attention(q, k, v, causal=causal, window=33)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("causal", [False, True])
def test_packed_documents_equal_separate_sequences(causal):
    lens = [5, 1, 17, 9]
    n = sum(lens)
    q, k, v = _rand(n, 2, 8, 10), _rand(n, 2, 8, 11), _rand(n, 2, 8, 12)
    doc = np.repeat(np.arange(len(lens)), lens)
    out, lse = oracle.attention(q, k, v, causal=causal, q_doc=doc, k_doc=doc)
    at = 0
    for ln in lens:
        o2, l2 = oracle.attention(q[at:at + ln], k[at:at + ln], v[at:at + ln], causal=causal)
        assert np.abs(out[at:at + ln] - o2).max() < 1e-13
        assert np.abs(lse[at:at + ln] - l2).max() < 1e-13
        at += ln


def test_padding_rows_see_nothing_and_are_not_seen():
    n, pad = 30, 7
    q, k, v = _rand(n, 2, 8, 13), _rand(n, 2, 8, 14), _rand(n, 2, 8, 15)
    doc = np.where(np.arange(n) < n - pad, 0, -1)
    out, lse = oracle.attention(q, k, v, causal=True, q_doc=doc, k_doc=doc)
    assert (out[n - pad:] == 0).all() and np.isneginf(lse[n - pad:]).all()
    o2, l2 = oracle.attention(q[:n - pad], k[:n - pad], v[:n - pad], causal=True)
    assert np.abs(out[:n - pad] - o2).max() < 1e-13
    assert np.abs(lse[:n - pad] - l2).max() < 1e-13


def test_positions_not_indices_decide_the_mask():
    # Permuting rows together with their positions changes nothing but the
    # row order: the mask reads positions, not indices.
    n, W = 48, 9
    q, k, v = _rand(n, 2, 8, 16), _rand(n, 2, 8, 17), _rand(n, 2, 8, 18)
    doc = np.repeat([0, 1, 2], [20, 12, 16])
    perm = np.random.default_rng(19).permutation(n)
    a = oracle.attention(q, k, v, causal=True, window=W, q_doc=doc, k_doc=doc)
    b = oracle.attention(q[perm], k[perm], v[perm], causal=True, window=W, q_pos=perm,
                         k_pos=perm, q_doc=doc[perm], k_doc=doc[perm])
    assert np.abs(b[0] - a[0][perm]).max() < 1e-13
    assert np.abs(b[1] - a[1][perm]).max() < 1e-13


# --- gradients (the backward ring: "Ring Attention：把超长序列沿设备环流动",
# "Backward 需要让梯度也沿环传播")

def _loss(q, k, v, dout, **kw):
    out, _ = oracle.attention(q, k, v, **kw)
    return float((out * dout.astype(np.float64)).sum())


@pytest.mark.parametrize("kw", [dict(causal=False), dict(causal=True),
                                dict(causal=True, window=3),
                                dict(causal=False, q_doc=np.array([0, 0, 1, 1, 1, 2]),
                                     k_doc=np.array([0, 0, 1, 1, 1, 2]))])
def test_gradients_match_finite_differences(kw):
    """Central differences of the forward oracle's loss sum(dout * O) pin
    every element of dQ, dK and dV (GQA 2:1)."""
    rng = np.random.default_rng(41)
    q = rng.standard_normal((6, 2, 3)).astype(np.float32)
    k = rng.standard_normal((6, 1, 3)).astype(np.float32)
    v = rng.standard_normal((6, 1, 3)).astype(np.float32)
    g = rng.standard_normal((6, 2, 3)).astype(np.float32)
    dq, dk, dv, _ = oracle.backward(q, k, v, g, **kw)
    h = np.float32(2.0 ** -9)
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] = x[idx] + h
            xm[idx] = x[idx] - h
            step = float(xp[idx]) - float(xm[idx])  # exact after fp32 rounding
            args = {"q": q, "k": k, "v": v}
            lp = _loss(**{**args, name: xp}, dout=g, **kw)
            lm = _loss(**{**args, name: xm}, dout=g, **kw)
            fd = (lp - lm) / step
            assert abs(fd - grad[idx]) < 2e-5 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])


def test_gradients_single_key_per_row():
    # Causal window 1: each row's softmax is the constant 1, so dQ = dK = 0
    # and dV_t gathers dout of row t over the heads of its group.
    rng = np.random.default_rng(43)
    q = rng.standard_normal((9, 4, 8)).astype(np.float32)
    k = rng.standard_normal((9, 2, 8)).astype(np.float32)
    v = rng.standard_normal((9, 2, 8)).astype(np.float32)
    g = rng.standard_normal((9, 4, 8)).astype(np.float32)
    dq, dk, dv, _ = oracle.backward(q, k, v, g, causal=True, window=1)
    assert np.abs(dq).max() < 1e-15 and np.abs(dk).max() < 1e-15
    want = g.astype(np.float64).reshape(9, 2, 2, 8).sum(2)
    assert np.abs(dv - want).max() < 1e-13


def test_gradients_equal_values_give_zero_dq_dk():
    # Equal value rows: O does not depend on the softmax weights.
    rng = np.random.default_rng(45)
    q = rng.standard_normal((12, 2, 8)).astype(np.float32)
    k = rng.standard_normal((12, 2, 8)).astype(np.float32)
    v = np.repeat(rng.standard_normal((1, 2, 8)).astype(np.float32), 12, axis=0)
    g = rng.standard_normal((12, 2, 8)).astype(np.float32)
    dq, dk, _, _ = oracle.backward(q, k, v, g, causal=True)
    assert np.abs(dq).max() < 1e-12 and np.abs(dk).max() < 1e-12


def test_gradient_sums_and_d_identity():
    # sum_t dV_t = sum of dout over the group's rows; sum_t dK_t = 0 (each
    # row's dS sums to zero); D_r = dout_r . O_r.
    rng = np.random.default_rng(47)
    n = 40
    q = rng.standard_normal((n, 6, 16)).astype(np.float32)
    k = rng.standard_normal((n, 2, 16)).astype(np.float32)
    v = rng.standard_normal((n, 2, 16)).astype(np.float32)
    g = rng.standard_normal((n, 6, 16)).astype(np.float32)
    dq, lse, dvec = oracle.grad_q(q, k, v, g, causal=True)
    dk, dv = oracle.grad_kv(q, k, v, g, lse, dvec, causal=True)
    gsum = g.astype(np.float64).reshape(n, 2, 3, 16).sum((0, 2))
    assert np.abs(dv.sum(0) - gsum).max() < 1e-12
    assert np.abs(dk.sum(0)).max() < 1e-12
    out, lse2 = oracle.attention(q, k, v, causal=True)
    assert np.abs(dvec - (out * g.astype(np.float64)).sum(-1)).max() < 1e-12
    assert np.abs(lse - lse2).max() < 1e-13


def test_gradients_gqa_equal_summed_repeated_heads():
    rng = np.random.default_rng(49)
    q = rng.standard_normal((20, 4, 8)).astype(np.float32)
    k = rng.standard_normal((20, 2, 8)).astype(np.float32)
    v = rng.standard_normal((20, 2, 8)).astype(np.float32)
    g = rng.standard_normal((20, 4, 8)).astype(np.float32)
    dq, dk, dv, _ = oracle.backward(q, k, v, g, causal=True)
    kr, vr = np.repeat(k, 2, axis=1), np.repeat(v, 2, axis=1)
    dq2, dk2, dv2, _ = oracle.backward(q, kr, vr, g, causal=True)
    assert np.abs(dq - dq2).max() < 1e-13
    assert np.abs(dk - dk2.reshape(20, 2, 2, 8).sum(2)).max() < 1e-13
    assert np.abs(dv - dv2.reshape(20, 2, 2, 8).sum(2)).max() < 1e-13


def test_gradient_rows_and_keys_subsets():
    rng = np.random.default_rng(51)
    q = rng.standard_normal((30, 2, 8)).astype(np.float32)
    k = rng.standard_normal((30, 1, 8)).astype(np.float32)
    v = rng.standard_normal((30, 1, 8)).astype(np.float32)
    g = rng.standard_normal((30, 2, 8)).astype(np.float32)
    dq, dk, dv, lse = oracle.backward(q, k, v, g, causal=True)
    rows = np.array([29, 0, 7])
    dq_r, lse_r, _ = oracle.grad_q(q, k, v, g, causal=True, rows=rows, threads=2)
    assert np.array_equal(dq_r, dq[rows]) and np.array_equal(lse_r, lse[rows])
    _, lse_a, d_a = oracle.grad_q(q, k, v, g, causal=True)
    dk_k, dv_k = oracle.grad_kv(q, k, v, g, lse_a, d_a, causal=True, keys=[3, 29], threads=3)
    assert np.array_equal(dk_k, dk[[3, 29]]) and np.array_equal(dv_k, dv[[3, 29]])


# --- absolute-term sums of the gradients (error scales; Higham, "Accuracy and
# Stability of Numerical Algorithms", ch. 3).  Each is a gradient's sum with
# every term replaced by its absolute value.

def _grad_case(seed, n=24, hq=4, hkv=2, d=8):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((n, hq, d)).astype(np.float32)
    k = rng.standard_normal((n, hkv, d)).astype(np.float32)
    v = rng.standard_normal((n, hkv, d)).astype(np.float32)
    g = rng.standard_normal((n, hq, d)).astype(np.float32)
    return q, k, v, g


@pytest.mark.parametrize("kw", [dict(causal=False), dict(causal=True),
                                dict(causal=True, window=5)])
def test_abs_scales_bound_the_gradients(kw):
    # Triangle inequality: |sum x_i| <= sum |x_i|, element by element; the
    # gradients are the oracle's own (pinned above).
    q, k, v, g = _grad_case(53)
    grads, scales, _ = oracle.backward_with_scales(q, k, v, g, **kw)
    plain = oracle.backward(q, k, v, g, **kw)[:3]
    for x, y, a in zip(grads, plain, scales):
        assert np.array_equal(x, y)
        assert (np.abs(x) <= a * (1 + 1e-12)).all()
        assert (a > 0).all()


def test_abs_scales_equal_the_gradient_when_every_term_is_positive():
    # dout >= 0: every term of dV_t (P_rt dO_r) is >= 0, so A_dV = dV.  With
    # v >= 0 too, every dP and O is >= 0, so D's absolute sum is D.
    q, k, v, g = _grad_case(55)
    g, v = np.abs(g), np.abs(v)
    dq, lse, dvec, dq_abs, d_abs = oracle.grad_q(q, k, v, g, causal=True, absolute=True)
    dk, dv, dk_abs, dv_abs = oracle.grad_kv(q, k, v, g, lse, dvec, causal=True,
                                            d_abs_all=d_abs)
    assert np.abs(dv_abs - dv).max() <= 1e-13 * np.abs(dv).max()
    assert np.abs(d_abs - dvec).max() <= 1e-13 * np.abs(dvec).max()


def test_abs_scales_closed_form_with_one_key_per_row():
    # Causal window 1: row r sees key r alone, so P = 1 and D = dP.  Then
    # A_D,r = sum_x |dO_rx||v_rx| and A_S,rr = 2 A_D,r, so
    # A_dQ,r = scale 2 A_D,r |k_r|, A_dK,t = scale sum_h 2 A_D,t,h |q_t,h|,
    # A_dV,t = sum_h |dO_t,h| over the query heads h of t's KV head.
    q, k, v, g = _grad_case(57, n=9, hq=4, hkv=2, d=8)
    _, (aq, ak, av), _ = oracle.backward_with_scales(q, k, v, g, causal=True, window=1)
    sc = 1.0 / math.sqrt(8)
    q64, k64, v64, g64 = (x.astype(np.float64) for x in (q, k, v, g))
    vh = np.repeat(v64, 2, axis=1)                  # value row of each query head
    kh = np.repeat(k64, 2, axis=1)
    a_d = (np.abs(g64) * np.abs(vh)).sum(-1)        # [n, hq]
    want_q = sc * 2 * a_d[..., None] * np.abs(kh)
    want_k = (sc * 2 * a_d[..., None] * np.abs(q64)).reshape(9, 2, 2, 8).sum(2)
    want_v = np.abs(g64).reshape(9, 2, 2, 8).sum(2)
    assert np.abs(aq - want_q).max() <= 1e-13 * want_q.max()
    assert np.abs(ak - want_k).max() <= 1e-13 * want_k.max()
    assert np.abs(av - want_v).max() <= 1e-13 * want_v.max()


def test_abs_scales_ignore_coordinate_signs_and_scale_with_dout():
    # Flipping the sign of coordinate x of dO in every row, or of v in every
    # key, changes the gradients but none of the absolute sums (P depends on
    # q and k only).  Scaling dO by -2 scales every absolute sum by 2.
    q, k, v, g = _grad_case(59)
    base_g, base_a, _ = oracle.backward_with_scales(q, k, v, g, causal=True)
    rng = np.random.default_rng(61)
    fg = np.where(rng.random(g.shape[-1]) < 0.5, -1, 1).astype(np.float32)
    fv = np.where(rng.random(v.shape[-1]) < 0.5, -1, 1).astype(np.float32)
    assert (fg < 0).any() and (fv < 0).any()
    grads, scales, _ = oracle.backward_with_scales(q, k, v * fv, g * fg, causal=True)
    for a, b in zip(scales, base_a):
        assert np.abs(a - b).max() <= 1e-12 * b.max()
    assert np.abs(grads[0] - base_g[0]).max() > 1e-3   # the gradients did change
    _, scaled, _ = oracle.backward_with_scales(q, k, v, -2 * g, causal=True)
    for a, b in zip(scaled, base_a):
        assert np.abs(a - 2 * b).max() <= 1e-12 * b.max()


def test_abs_scales_rows_and_keys_subsets():
    q, k, v, g = _grad_case(63, n=30)
    _, (aq, ak, av), _ = oracle.backward_with_scales(q, k, v, g, causal=True)
    rows = np.array([29, 0, 7])
    _, _, _, aq_r, _ = oracle.grad_q(q, k, v, g, causal=True, rows=rows, absolute=True)
    assert np.array_equal(aq_r, aq[rows])
    _, lse, dvec, _, d_abs = oracle.grad_q(q, k, v, g, causal=True, absolute=True)
    _, _, ak_k, av_k = oracle.grad_kv(q, k, v, g, lse, dvec, causal=True, keys=[3, 29],
                                      d_abs_all=d_abs, threads=3)
    assert np.array_equal(ak_k, ak[[3, 29]]) and np.array_equal(av_k, av[[3, 29]])
