"""GPU parity of the backward ring (dQ, dK, dV) against the fp64 gradient
oracle ("Ring Attention：把超长序列沿设备环流动", section "Backward 需要让梯度也
沿环传播").  The GPU recomputes the softmax from its own forward's LSE; the
oracle computes everything from the inputs alone."""
import numpy as np
import pytest
import torch

import oracle
from parity import check_grad

import blockwise_online_softmax_gb300 as ra
from blockwise_online_softmax_gb300 import binding, inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from blockwise_online_softmax_gb300 import build

    build.build()
    binding.lib()
    yield
    torch.cuda.empty_cache()


def doc_ids(N, doc_lens, n_valid):
    ids = np.zeros(N, dtype=np.int64)
    if doc_lens is not None:
        ids[:] = -1
        at = 0
        for dd, ln in enumerate(doc_lens):
            ids[at:at + ln] = dd
            at += ln
    if n_valid is not None:
        ids[n_valid:] = -1
    return ids


def run(N, P, heads, kv_heads, d, causal, layout="contiguous", window=0, n_valid=None,
        docs=None, seed=0):
    q, k, v = inputs.make_random(N, heads, kv_heads, d, seed=seed)
    dout = inputs.randn_chunked((N, heads, d), seed, 3).to(torch.bfloat16)
    pos = binding.layout_positions(N, P, layout)
    ql, kl, vl, gl = q[pos], k[pos], v[pos], dout[pos]
    cu = None
    if docs is not None:
        cu = torch.tensor(np.concatenate([[0], np.cumsum(docs)]), dtype=torch.int32, device=DEV)
    kw = dict(P=P, layout=layout, causal=causal, window=window,
              n_valid=-1 if n_valid is None else n_valid, cu_seqlens=cu)
    qd, kd, vd, gd = ql.to(DEV), kl.to(DEV), vl.to(DEV), gl.to(DEV)
    out, lse = ra.ra_ring_forward_masked(qd, kd, vd, **kw)
    dq, dk, dv = ra.ra_ring_backward_masked(qd, kd, vd, out, lse, gd, **kw)
    ra.ra_device_status()
    okw = {}
    if docs is not None or n_valid is not None:
        ids = doc_ids(N, docs, n_valid)[pos.numpy()]
        okw = dict(q_doc=ids, k_doc=ids)
    refs, scales, _ = oracle.backward_with_scales(ql, kl, vl, gl, causal=causal, window=window,
                                                  q_pos=pos.numpy(), k_pos=pos.numpy(), **okw)
    for name, x, r, a in zip(("dq", "dk", "dv"), (dq, dk, dv), refs, scales):
        check_grad(x, r, a, name)


CASES = [
    # N, P, heads, kv_heads, d, causal
    (1024, 4, 2, 1, 128, True),
    (1024, 4, 2, 2, 64, False),
    (768, 3, 4, 2, 128, True),
    (600, 3, 2, 1, 128, True),   # c = 200: ragged tiles
    (256, 1, 2, 2, 64, True),    # one block
    (130, 2, 1, 1, 128, True),   # c = 65 < one tile
    (768, 3, 6, 2, 64, True),    # GQA 3:1, six query heads
    (512, 2, 3, 3, 128, False),  # odd head count
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"N{c[0]}-P{c[1]}-h{c[2]}/{c[3]}-d{c[4]}"
                         f"-{'c' if c[5] else 'nc'}")
def test_backward_matches_oracle(case):
    N, P, heads, kv_heads, d, causal = case
    run(N, P, heads, kv_heads, d, causal, seed=N + d)


MASKED = [
    dict(layout="zigzag"),
    dict(layout="striped"),
    dict(window=300),
    dict(docs=[300, 1, 400, 323]),
    dict(n_valid=1000),
    dict(layout="zigzag", window=200, docs=[512, 400, 100], n_valid=1012),
]


@pytest.mark.parametrize("kw", MASKED, ids=lambda k: "-".join(f"{a}" for a in k))
def test_masked_backward_matches_oracle(kw):
    run(1024, 4, 4, 2, 128, True, seed=7, **kw)


def test_backward_non_causal_window():
    run(1024, 4, 2, 1, 64, False, window=150, seed=9)


def test_backward_is_deterministic():
    N, P = 1024, 4
    q, k, v = (t.to(DEV) for t in inputs.make_random(N, 4, 2, 128, seed=11))
    g = inputs.randn_chunked((N, 4, 128), 11, 3).to(torch.bfloat16).to(DEV)
    out, lse = ra.ra_ring_forward(q, k, v, P=P, causal=True)
    a = ra.ra_ring_backward(q, k, v, out, lse, g, P=P, causal=True)
    b = ra.ra_ring_backward(q, k, v, out, lse, g, P=P, causal=True)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_backward_block_count_does_not_change_the_result():
    # Each P is within the bar of the oracle, so two of them are within
    # twice the bar of each other.
    N = 1024
    qh, kh, vh = inputs.make_random(N, 2, 1, 128, seed=13)
    gh = inputs.randn_chunked((N, 2, 128), 13, 3).to(torch.bfloat16)
    q, k, v, g = (t.to(DEV) for t in (qh, kh, vh, gh))
    _, scales, _ = oracle.backward_with_scales(qh, kh, vh, gh, causal=True)
    ref = None
    for P in (1, 2, 4, 8):
        out, lse = ra.ra_ring_forward(q, k, v, P=P, causal=True)
        res = ra.ra_ring_backward(q, k, v, out, lse, g, P=P, causal=True)
        torch.cuda.synchronize()
        if ref is None:
            ref = res
        for x, y, a in zip(res, ref, scales):
            a = torch.from_numpy(a)
            bar = 2 * (2.0 ** -7 * a + 1e-6 * a.max())
            assert ((x.cpu().double() - y.cpu().double()).abs() <= bar).all()


def test_backward_with_300_ranks():
    """P = 300 ranks of two rows each: 300 ring steps of mostly empty or
    one-tile work, the gradients accumulating in HBM across the steps.  They
    are those of the P = 4 ring (the same attention) and of the oracle."""
    N, P, heads, kv_heads, d = 600, 300, 2, 1, 64
    q, k, v = inputs.make_random(N, heads, kv_heads, d, seed=41)
    g = inputs.randn_chunked((N, heads, d), 41, 3).to(torch.bfloat16)
    qd, kd, vd, gd = q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV)
    grads = {}
    for p in (P, 4):
        out, lse = ra.ra_ring_forward(qd, kd, vd, P=p, causal=True)
        grads[p] = ra.ra_ring_backward(qd, kd, vd, out, lse, gd, P=p, causal=True)
    ra.ra_device_status()
    refs, scales, _ = oracle.backward_with_scales(q, k, v, g, causal=True)
    for name, x, y, r, a in zip(("dq", "dk", "dv"), grads[P], grads[4], refs, scales):
        check_grad(x, r, a, name)
        check_grad(y, r, a, name + " (P = 4)")


@pytest.mark.slow
def test_backward_mha_8k():
    w = inputs.WORKLOADS["mha-8k"]
    run(w.N, w.P, w.heads, w.kv_heads, w.d, w.causal, seed=w.seed)


@pytest.mark.slow
def test_backward_gqa_128k_sampled():
    """gqa-128k at full size: dQ on sampled rows against the oracle; dK, dV
    through properties that hold at any size (sum of dV = summed dout per KV
    head, sum of dK = 0, both over all keys)."""
    w = inputs.WORKLOADS["gqa-128k"]
    q, k, v = inputs.make_workload(w)
    g = inputs.randn_chunked((w.N, w.heads, w.d), w.seed, 3).to(torch.bfloat16)
    qd, kd, vd, gd = q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV)
    out, lse = ra.ra_ring_forward(qd, kd, vd, P=w.P, causal=True)
    dq, dk, dv = ra.ra_ring_backward(qd, kd, vd, out, lse, gd, P=w.P, causal=True)
    ra.ra_device_status()
    rows = inputs.sample_rows(w, random_per_block=2)
    got = dq.index_select(0, torch.from_numpy(rows).to(DEV)).cpu()
    ref, _, _, ref_abs, _ = oracle.grad_q(q, k, v, g, causal=True, rows=rows, absolute=True)
    check_grad(got, ref, ref_abs, "dq")
    gsum = g.double().view(w.N, w.kv_heads, w.heads // w.kv_heads, w.d).sum((0, 2))
    dv_sum = dv.double().sum(0).cpu()
    assert (dv_sum - gsum).abs().max().item() <= 2e-2 * gsum.abs().max().item()
    # sum_t dK_t is 0 exactly; the GPU's per-element errors (bf16 dS, at most
    # 2^-9 relative) add up like a random walk over the N keys.
    dk_sum = dk.double().sum(0).cpu()
    assert dk_sum.abs().max().item() <= 2.0 ** -8 * np.sqrt(w.N) * dk.abs().max().item()


@pytest.mark.slow
def test_backward_gqa_128k_window_sampled_keys():
    """gqa-128k at full size, causal with a 1024-key window: dQ on sampled
    rows, and dK, dV on sampled keys, element by element against the
    oracle.  Key k is seen only by queries [k, k + W), so the oracle needs
    their LSE and D alone; the other rows' entries are NaN, which would
    poison any result that used them.  Every key tile of the dK/dV kernel
    walks 32 query tiles (8 per query head of its group)."""
    w = inputs.WORKLOADS["gqa-128k"]
    W = 1024
    q, k, v = inputs.make_workload(w)
    g = inputs.randn_chunked((w.N, w.heads, w.d), w.seed, 3).to(torch.bfloat16)
    qd, kd, vd, gd = q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV)
    out, lse = ra.ra_ring_forward_masked(qd, kd, vd, P=w.P, causal=True, window=W)
    dq, dk, dv = ra.ra_ring_backward_masked(qd, kd, vd, out, lse, gd, P=w.P, causal=True,
                                            window=W)
    ra.ra_device_status()
    c = w.c
    keys = np.array([0, 1, c - 1, c, 3 * c + 777, 8 * c - 1, 8 * c, 11 * c + 4000,
                     w.N - W - 1, w.N - 1], dtype=np.int64)
    need = np.unique(np.concatenate([np.arange(kk, min(w.N, kk + W)) for kk in keys]))
    dq_ref, lse_rows, d_rows, dq_abs, d_abs_rows = oracle.grad_q(
        q, k, v, g, causal=True, rows=need, window=W, absolute=True)
    lse_all = np.full((w.N, w.heads), np.nan)
    d_all = np.full((w.N, w.heads), np.nan)
    d_abs_all = np.full((w.N, w.heads), np.nan)
    lse_all[need] = lse_rows
    d_all[need] = d_rows
    d_abs_all[need] = d_abs_rows
    dk_ref, dv_ref, dk_abs, dv_abs = oracle.grad_kv(q, k, v, g, lse_all, d_all, causal=True,
                                                    keys=keys, window=W, d_abs_all=d_abs_all)
    sel = torch.from_numpy(keys).to(DEV)
    check_grad(dk.index_select(0, sel).cpu(), dk_ref, dk_abs, "dk")
    check_grad(dv.index_select(0, sel).cpu(), dv_ref, dv_abs, "dv")
    rows = need[::97]
    check_grad(dq.index_select(0, torch.from_numpy(rows).to(DEV)).cpu(),
               dq_ref[::97], dq_abs[::97], "dq")


@pytest.mark.slow
def test_backward_mha_8k_window_and_documents():
    w = inputs.WORKLOADS["mha-8k"]
    run(w.N, w.P, w.heads, w.kv_heads, w.d, True, layout="zigzag", window=2000,
        docs=[3000, 17, 4000, 1175], seed=w.seed + 1)
