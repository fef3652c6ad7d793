"""GPU parity of the zigzag and striped layouts and of the masks beyond
causal (sliding window, packed documents, padding with a valid length)
against the CPU oracle.

The library gets the layout and the mask as arguments (cu_seqlens, n_valid,
window); the oracle gets only per-row positions and per-row document ids,
with -1 for padding.  The two descriptions share nothing but the inputs.
The layouts come from "Ring Attention Paper Breakdown", section 5, and
"RingAttention: Scaling LLM Context to 10M Tokens", section "Causal
Masking: Striped and Zig-Zag RingAttention"; the masks are the cases that
"Ring Attention：把超长序列沿设备环流动" lists under
"正确性测试应覆盖哪些边界".
"""
import numpy as np
import pytest
import torch

import oracle
from parity import check_output, check_state, assert_fused_matches

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
    """Document id of every position: -1 past the documents or n_valid."""
    ids = np.full(N, -1, dtype=np.int64)
    if doc_lens is None:
        ids[:] = 0
    else:
        at = 0
        for d, ln in enumerate(doc_lens):
            ids[at:at + ln] = d
            at += ln
    if n_valid is not None:
        ids[n_valid:] = -1
    return ids


def run_case(N, P, layout, causal, window, n_valid, doc_lens, heads, kv_heads, d, dtype, seed):
    # Sequence-order inputs, laid out for the ring: row r holds position pos[r].
    q, k, v = inputs.make_random(N, heads, kv_heads, d, dtype=dtype, seed=seed)
    pos = binding.layout_positions(N, P, layout)
    ql, kl, vl = q[pos], k[pos], v[pos]
    cu = None
    if doc_lens is not None:
        cu = torch.tensor(np.concatenate([[0], np.cumsum(doc_lens)]), dtype=torch.int32,
                          device=DEV)
    out, lse = ra.ra_ring_forward_masked(
        ql.to(DEV), kl.to(DEV), vl.to(DEV), P=P, layout=layout, causal=causal, window=window,
        n_valid=-1 if n_valid is None else n_valid, cu_seqlens=cu)
    ra.ra_device_status()
    ids = doc_ids(N, doc_lens, n_valid)[pos.numpy()]
    use_docs = doc_lens is not None or n_valid is not None
    ref_out, ref_lse = oracle.attention(ql, kl, vl, causal=causal, window=window,
                                        q_pos=pos.numpy(), k_pos=pos.numpy(),
                                        q_doc=ids if use_docs else None,
                                        k_doc=ids if use_docs else None)
    kind = "bf16" if dtype == torch.bfloat16 else "f32"
    check_output(out, lse, ref_out, ref_lse, kind)
    return out, lse


DOCS = [300, 1, 700, 500, 547]  # sums to 2048
CASES = [
    # N, P, layout, causal, window, n_valid, docs, heads, kv_heads, d, dtype
    (2048, 4, "zigzag", True, 0, None, None, 4, 2, 128, torch.bfloat16),
    (2048, 4, "striped", True, 0, None, None, 4, 2, 128, torch.bfloat16),
    (2048, 4, "zigzag", False, 0, None, None, 2, 1, 64, torch.bfloat16),
    (1536, 3, "striped", False, 0, None, None, 2, 2, 64, torch.bfloat16),
    (1200, 4, "zigzag", True, 0, None, None, 2, 1, 128, torch.bfloat16),  # c = 300, h = 150
    (2048, 8, "contiguous", True, 300, None, None, 4, 2, 128, torch.bfloat16),
    (2048, 4, "contiguous", False, 200, None, None, 2, 2, 64, torch.bfloat16),
    (2048, 4, "zigzag", True, 700, None, None, 2, 1, 128, torch.bfloat16),
    (2048, 4, "striped", True, 37, None, None, 2, 1, 128, torch.bfloat16),
    (2048, 4, "contiguous", True, 0, None, DOCS, 4, 2, 128, torch.bfloat16),
    (2048, 4, "zigzag", True, 0, None, DOCS, 2, 2, 128, torch.bfloat16),
    (2048, 4, "striped", False, 0, None, DOCS, 2, 1, 64, torch.bfloat16),
    (2048, 4, "contiguous", True, 0, 2048 - 77, None, 2, 2, 128, torch.bfloat16),
    (2048, 4, "striped", False, 0, 1500, None, 2, 2, 64, torch.bfloat16),
    (2048, 4, "zigzag", True, 256, 2000, [900, 3, 1000, 97], 4, 1, 128, torch.bfloat16),
    # d = 64, causal: a document starts inside query tile 0 of a pair, so
    # query tile 1 sees keys in the first ring step only and tile 0 runs
    # alone through the later steps (the fused ring rotates three score
    # buffers between the two tiles at d = 64).
    (4096, 4, "contiguous", True, 0, None, [1000, 17, 2355, 724], 2, 2, 64, torch.bfloat16),
    (4096, 4, "zigzag", True, 1500, None, [1000, 17, 2355, 724], 2, 1, 64, torch.bfloat16),
    (1024, 4, "zigzag", True, 100, 1000, [500, 11, 489], 2, 1, 64, torch.float32),
    (1024, 4, "contiguous", False, 64, 999, None, 2, 2, 128, torch.float32),
    (1024, 4, "striped", True, 0, None, [512, 512], 2, 2, 64, torch.float32),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[2]}-{'c' if c[3] else 'nc'}-w{c[4]}"
                         f"-v{c[5]}-{'docs' if c[6] else 'nodoc'}-d{c[9]}-{str(c[10])[6:]}")
def test_masked_ring_matches_oracle(case):
    N, P, layout, causal, window, n_valid, docs, heads, kv_heads, d, dtype = case
    run_case(N, P, layout, causal, window, n_valid, docs, heads, kv_heads, d, dtype,
             seed=N + P + window)


def test_plain_arguments_reproduce_the_plain_ring_bit_for_bit():
    q, k, v = (t.to(DEV) for t in inputs.make_random(2048, 4, 2, 128, seed=3))
    for causal in (False, True):
        a = ra.ra_ring_forward(q, k, v, P=4, causal=causal)
        b = ra.ra_ring_forward_masked(q, k, v, P=4, causal=causal, n_valid=2048)
        torch.cuda.synchronize()
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_layouts_give_the_same_attention():
    # The same sequence, laid out three ways, gives the same per-position
    # result (up to the rounding of a different ring order).
    N, P = 2048, 8
    q, k, v = inputs.make_random(N, 2, 1, 128, seed=23)
    res = {}
    for layout in ("contiguous", "zigzag", "striped"):
        pos = binding.layout_positions(N, P, layout)
        out, lse = ra.ra_ring_forward_masked(q[pos].to(DEV), k[pos].to(DEV), v[pos].to(DEV), P=P,
                                             layout=layout, causal=True)
        inv = torch.argsort(pos).to(DEV)
        res[layout] = (out[inv], lse[inv])
    for layout in ("zigzag", "striped"):
        assert (res[layout][0] - res["contiguous"][0]).abs().max().item() < 1e-2
        assert (res[layout][1] - res["contiguous"][1]).abs().max().item() < 1e-3


def test_every_query_alone_in_its_document():
    # ndocs = N: each row sees only itself, so O = v_row and LSE = s_rr.
    N, P = 512, 4
    q, k, v = inputs.make_random(N, 2, 2, 64, seed=29)
    cu = torch.arange(N + 1, dtype=torch.int32, device=DEV)
    out, lse = ra.ra_ring_forward_masked(q.to(DEV), k.to(DEV), v.to(DEV), P=P, causal=False,
                                         cu_seqlens=cu)
    torch.cuda.synchronize()
    # P = 2^(tiny) rounds to 1 in bf16; l keeps the fp32 value 1 - O(1e-8).
    assert (out.cpu() - v.float()).abs().max().item() < 1e-5
    s = (q.double() * k.double()).sum(-1) / 8.0
    assert (lse.cpu().double() - s).abs().max().item() < 1e-3


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_masked_block_update_unequal_blocks(dtype):
    """One pair with c_q != c_kv at arbitrary positions, window and
    documents: the state equals the oracle's partial state."""
    c_q, c_kv, heads, kv_heads, d = 200, 900, 4, 2, 128
    q_off, kv_off = 1000, 350
    q, _, _ = inputs.make_random(c_q, heads, kv_heads, d, dtype=dtype, seed=31)
    _, k, v = inputs.make_random(c_kv, heads, kv_heads, d, dtype=dtype, seed=32)
    docs = [0, 700, 1100, 1300]  # positions: documents [0,700), [700,1100), [1100,1300)
    cu = torch.tensor(docs, dtype=torch.int32, device=DEV)
    window = 500
    m = torch.empty(c_q, heads, device=DEV)
    l = torch.empty(c_q, heads, device=DEV)
    o = torch.empty(c_q, heads, d, device=DEV)
    ra.ra_state_init(m, l, o)
    ra.ra_block_update_masked(q.to(DEV), k.to(DEV), v.to(DEV), m, l, o, q_off=q_off,
                              kv_off=kv_off, causal=True, window=window, n_valid=1250,
                              cu_seqlens=cu)
    ra.ra_device_status()
    qp = np.arange(q_off, q_off + c_q)
    kp = np.arange(kv_off, kv_off + c_kv)

    def ids(p):
        x = np.searchsorted(np.array(docs), p, side="right") - 1
        return np.where((p < 1250) & (p < docs[-1]), x, -1)

    ref = oracle.partial_state(q, k, v, causal=True, window=window, q_pos=qp, k_pos=kp,
                               q_doc=ids(qp), k_doc=ids(kp))
    check_state(m, l, o, ref, "bf16" if dtype == torch.bfloat16 else "f32")


def test_masked_steps_equal_the_masked_forward():
    N, P = 1024, 4
    q, k, v = (t.to(DEV) for t in inputs.make_random(N, 2, 1, 64, seed=37))
    cu = torch.tensor([0, 100, 1024], dtype=torch.int32, device=DEV)
    kw = dict(layout="zigzag", causal=True, window=300, n_valid=1000, cu_seqlens=cu)
    ref_out, ref_lse = ra.ra_ring_forward_masked(q, k, v, P=P, **kw)
    m = torch.empty(N, 2, device=DEV)
    l = torch.empty(N, 2, device=DEV)
    o = torch.empty(N, 2, 64, device=DEV)
    ra.ra_state_init(m, l, o)
    for s in range(P):
        ra.ra_ring_step_masked(q, k, v, m, l, o, P=P, s=s, **kw)
    out, lse = ra.ra_finalize(m, l, o)
    torch.cuda.synchronize()
    # The masked forward (bf16) is one fused launch; the steps above do the
    # same products and state updates, with the state in HBM between them.
    assert_fused_matches(ref_out, ref_lse, out, lse)


@pytest.mark.slow
def test_zigzag_gqa_large_sampled_rows():
    """The gqa-128k shape (N = 131072, P = 16, 32/8 heads, d = 128), zigzag
    layout, causal: sampled rows over their full key range."""
    w = inputs.WORKLOADS["gqa-128k"]
    q, k, v = inputs.make_workload(w)
    pos = binding.layout_positions(w.N, w.P, "zigzag")
    ql, kl, vl = q[pos], k[pos], v[pos]
    del q, k, v
    out, lse = ra.ra_ring_forward_masked(ql.to(DEV), kl.to(DEV), vl.to(DEV), P=w.P,
                                         layout="zigzag", causal=True)
    rows = inputs.sample_rows(w, random_per_block=4)
    idx = torch.from_numpy(rows).to(DEV)
    got_out, got_lse = out.index_select(0, idx).cpu(), lse.index_select(0, idx).cpu()
    del out, lse
    torch.cuda.empty_cache()
    ref_out, ref_lse = oracle.attention(ql, kl, vl, causal=True, q_pos=pos.numpy(),
                                        k_pos=pos.numpy(), rows=rows)
    check_output(got_out, got_lse, ref_out, ref_lse, "bf16")


@pytest.mark.slow
def test_masked_gqa_128k_sampled_rows():
    """The gqa-128k shape with the zigzag layout, a 16384-token causal window
    and 32 packed documents: sampled rows over their full allowed key range."""
    w = inputs.WORKLOADS["gqa-128k"]
    q, k, v = inputs.make_workload(w)
    pos = binding.layout_positions(w.N, w.P, "zigzag")
    rng = np.random.default_rng(77)
    cuts = np.sort(rng.choice(np.arange(1, w.N), size=31, replace=False))
    bounds = np.concatenate([[0], cuts, [w.N]])
    cu = torch.tensor(bounds, dtype=torch.int32, device=DEV)
    ql, kl, vl = q[pos], k[pos], v[pos]
    del q, k, v
    out, lse = ra.ra_ring_forward_masked(ql.to(DEV), kl.to(DEV), vl.to(DEV), P=w.P,
                                         layout="zigzag", causal=True, window=16384,
                                         cu_seqlens=cu)
    ra.ra_device_status()
    rows = inputs.sample_rows(w, random_per_block=4)
    idx = torch.from_numpy(rows).to(DEV)
    got_out, got_lse = out.index_select(0, idx).cpu(), lse.index_select(0, idx).cpu()
    del out, lse
    torch.cuda.empty_cache()
    ids = (np.searchsorted(bounds, np.arange(w.N), side="right") - 1)[pos.numpy()]
    ref_out, ref_lse = oracle.attention(ql, kl, vl, causal=True, window=16384, q_pos=pos.numpy(),
                                        k_pos=pos.numpy(), q_doc=ids, k_doc=ids, rows=rows)
    check_output(got_out, got_lse, ref_out, ref_lse, "bf16")
