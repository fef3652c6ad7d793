"""Element offsets past 2^31 and 2^32.

One sequence of 1,048,576 tokens with 40 query heads over 8 KV heads at
d = 128 gives Q, O and the O~ state 5.4e9 elements each, so every flat
index (row * heads + head) * d past the 2^31 and 2^32 marks must be
computed in 64 bits.  Checked on the fused ring forward, on the one-step
block update (which loads and stores its state in HBM) with the finalize
in place, and on the merge: every output element written (outputs start
as NaN), and the rows that straddle both marks, plus block edges and
seeded random rows, against the oracle.  The backward (320 query heads)
and decode (5M keys) get tensors of the same size their own way."""
import numpy as np
import pytest
import torch

import oracle
from oracle import online
from parity import check_grad, check_output, check_state

import blockwise_online_softmax_gb300 as ra
from blockwise_online_softmax_gb300 import build, inputs

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = torch.device("cuda:0")
N, P, HEADS, KV_HEADS, D = 1 << 20, 64, 40, 8, 128
C = N // P
ROW_ELEMS = HEADS * D  # elements of one token row of Q or O


def straddling_rows(n_rows):
    """Rows whose elements cross 2^31 and 2^32, block edges, the last row,
    and four seeded random rows from the upper half."""
    rows = {0, C - 1, C, n_rows - 1}
    for mark in (1 << 31, 1 << 32):
        r = mark // ROW_ELEMS
        rows |= {r - 1, r, r + 1}
    rng = np.random.default_rng(2024)
    rows |= set(rng.integers(n_rows // 2, n_rows, size=4).tolist())
    return np.array(sorted(r for r in rows if 0 <= r < n_rows), dtype=np.int64)


@pytest.fixture(scope="module")
def big():
    build.build()
    assert N * HEADS * D > (1 << 32)
    q, k, v = inputs.make_random(N, HEADS, KV_HEADS, D, seed=77)
    yield q, k, v, q.to(DEV), k.to(DEV), v.to(DEV)
    torch.cuda.empty_cache()


def test_fused_ring_forward_past_2_32_elements(big):
    q, k, v, qd, kd, vd = big
    out = torch.full((N, HEADS, D), float("nan"), device=DEV)
    lse = torch.full((N, HEADS), float("nan"), device=DEV)
    ra.ra_ring_forward(qd, kd, vd, P=P, causal=True, out=out, lse=lse)
    ra.ra_device_status()
    # Causal: every row sees at least its own key, so every element is
    # written and finite.
    assert not out.isnan().any().item() and torch.isfinite(lse).all().item()
    rows = straddling_rows(N)
    idx = torch.from_numpy(rows).to(DEV)
    got_out, got_lse = out.index_select(0, idx).cpu(), lse.index_select(0, idx).cpu()
    del out, lse
    torch.cuda.empty_cache()
    ref_out, ref_lse = oracle.attention(q, k, v, causal=True, rows=rows)
    check_output(got_out, got_lse, ref_out, ref_lse, "bf16")


def test_block_update_state_and_finalize_past_2_32_elements(big):
    # All N query rows (positions 4096 + r) against two K/V blocks of 4096
    # keys (positions 0..4095, then 4096..8191): the second update loads
    # the state the first stored, and masks rows r < 4095.  The finalize
    # writes in place over the state.
    q, k, v, qd, kd, vd = big
    ck = 4096
    m = torch.full((N, HEADS), float("nan"), device=DEV)
    l = torch.full((N, HEADS), float("nan"), device=DEV)
    o = torch.full((N, HEADS, D), float("nan"), device=DEV)
    ra.ra_state_init(m, l, o)
    for b in range(2):
        ra.ra_block_update_masked(qd, kd[b * ck:(b + 1) * ck], vd[b * ck:(b + 1) * ck], m, l, o,
                                  q_off=ck, kv_off=b * ck, causal=True)
    out, lse = ra.ra_finalize(m, l, o, out=o, lse=m)
    ra.ra_device_status()
    assert not out.isnan().any().item() and torch.isfinite(lse).all().item()
    rows = straddling_rows(N)
    idx = torch.from_numpy(rows).to(DEV)
    got_out, got_lse = out.index_select(0, idx).cpu(), lse.index_select(0, idx).cpu()
    del m, l, o, out, lse
    torch.cuda.empty_cache()
    ref_out, ref_lse = oracle.attention(q, k[:2 * ck], v[:2 * ck], causal=True,
                                        q_pos=ck + np.arange(N), k_pos=np.arange(2 * ck),
                                        rows=rows)
    check_output(got_out, got_lse, ref_out, ref_lse, "bf16")


def test_merge_past_2_32_elements():
    # Two random states of N rows; some (row, head) entries of either side,
    # at the marks, are the identity (m = -inf, l = 0, O~ = 0).
    build.build()
    g = torch.Generator(device=DEV).manual_seed(31)
    rows = straddling_rows(N)
    sides = []
    for s in range(2):
        m = torch.randn((N, HEADS), generator=g, device=DEV) * 2.0
        l = torch.rand((N, HEADS), generator=g, device=DEV) + 0.5
        o = torch.randn((N, HEADS, D), generator=g, device=DEV)
        empty = torch.from_numpy(rows[s::3]).to(DEV)
        m[empty, s] = float("-inf")
        l[empty, s] = 0.0
        o[empty, s] = 0.0
        sides.append((m, l, o))
    idx = torch.from_numpy(rows).to(DEV)
    host = [tuple(t.index_select(0, idx).cpu().double().numpy() for t in side) for side in sides]
    (ma, la, oa), (mb, lb, ob) = sides
    ra.ra_merge(ma, la, oa, mb, lb, ob)
    ra.ra_device_status()
    del sides, mb, lb, ob
    torch.cuda.empty_cache()
    assert not oa.isnan().any().item()
    got = tuple(t.index_select(0, idx).cpu() for t in (ma, la, oa))
    check_state(*got, online.merge(host[0], host[1]), "f32")


def test_backward_past_2_32_elements():
    # 131,072 tokens with 320 query heads over 8 KV heads: Q, dout, O and
    # dQ hold 5.4e9 elements.  Causal with a 1024-key window (the offsets
    # are what is tested, the window keeps it cheap).  dQ on the rows that
    # straddle the marks, element by element; dK and dV through properties
    # that hold at any size (sum of dV over keys = summed dout per KV head,
    # sum of dK = 0).
    build.build()
    n, p, heads, kv_heads, w = 1 << 17, 16, 320, 8, 1024
    assert n * heads * D > (1 << 32)
    q, k, v = inputs.make_random(n, heads, kv_heads, D, seed=78)
    g = inputs.randn_chunked((n, heads, D), 78, 3, dtype=torch.bfloat16)
    qd, kd, vd, gd = q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV)
    out, lse = ra.ra_ring_forward_masked(qd, kd, vd, P=p, causal=True, window=w)
    dq = torch.full((n, heads, D), float("nan"), device=DEV)
    dq, dk, dv = ra.ra_ring_backward_masked(qd, kd, vd, out, lse, gd, P=p, causal=True,
                                            window=w, dq=dq)
    ra.ra_device_status()
    del qd, gd, out, lse
    assert not dq.isnan().any().item()
    rows = {0, n // p - 1, n // p, n - 1}
    for mark in (1 << 31, 1 << 32):
        r = mark // (heads * D)
        rows |= {r - 1, r, r + 1}
    rows = np.array(sorted(rows), dtype=np.int64)
    got = dq.index_select(0, torch.from_numpy(rows).to(DEV)).cpu()
    del dq
    torch.cuda.empty_cache()
    ref, _, _, ref_abs, _ = oracle.grad_q(q, k, v, g, causal=True, rows=rows, window=w,
                                          absolute=True)
    check_grad(got, ref, ref_abs, "dq")
    gv = g.view(n, kv_heads, heads // kv_heads, D)
    gsum = sum(gv[t:t + 8192].double().sum((0, 2)) for t in range(0, n, 8192))
    dv_sum = dv.double().sum(0).cpu()
    assert (dv_sum - gsum).abs().max().item() <= 2e-2 * gsum.abs().max().item()
    dk_sum = dk.double().sum(0).cpu()
    assert dk_sum.abs().max().item() <= 2.0 ** -8 * np.sqrt(n) * dk.abs().max().item()


def test_decode_past_2_32_elements():
    # Two new tokens (32 query heads over 8 KV heads) after a history of
    # 5,242,880 tokens in 80 shards: K and V hold 5.4e9 elements each.
    build.build()
    w = inputs.DecodeWorkload("decode-5m", seed=79, n_q=2, heads=32, kv_heads=8, d=D,
                              n_kv=5 << 20, P=80)
    assert w.n_kv * w.kv_heads * w.d > (1 << 32)
    q, k, v = inputs.make_decode(w)
    out, lse = ra.ra_decode_forward(q.to(DEV), k.to(DEV), v.to(DEV), P=w.P)
    ra.ra_device_status()
    torch.cuda.empty_cache()
    ref_out, ref_lse = oracle.attention(q, k, v, causal=True,
                                        q_pos=w.n_kv - w.n_q + np.arange(w.n_q))
    check_output(out, lse, ref_out, ref_lse, "bf16")
