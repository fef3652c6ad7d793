"""GPU parity of the ring forward (init, P ring steps, finalize) against the
CPU oracle.  The five named workloads are checked, in the launch
configuration the benchmark times: the two small ones on every output, the
three large ones on sampled rows over each row's full key range.  Ragged
and degenerate shapes, invariants, resume from a saved state, and the
host-buffer entry point are covered too."""
import numpy as np
import pytest
import torch

import oracle
from parity import TOL, check_output, assert_fused_matches

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


def kind_of(dtype):
    return "bf16" if dtype == torch.bfloat16 else "f32"


def run_ring(q, k, v, P, causal):
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    out, lse = ra.ra_ring_forward(qd, kd, vd, P=P, causal=causal)
    ra.ra_device_status()
    return out, lse


@pytest.mark.parametrize("name", ["tiny-exact", "mha-8k"])
def test_small_workloads_every_output(name):
    w = inputs.WORKLOADS[name]
    q, k, v = inputs.make_workload(w)
    out, lse = run_ring(q, k, v, w.P, w.causal)
    ref_out, ref_lse = oracle.attention(q, k, v, causal=w.causal)
    check_output(out, lse, ref_out, ref_lse, w.dtype)


@pytest.mark.slow
@pytest.mark.parametrize("name,random_rows", [("mha-32k-scaled-keys", 16), ("gqa-128k", 16),
                                              ("mha-1m-planted", 4)])
def test_large_workloads_sampled_rows(name, random_rows):
    w = inputs.WORKLOADS[name]
    q, k, v = inputs.make_workload(w)
    rows = inputs.sample_rows(w, random_per_block=random_rows)
    out, lse = run_ring(q, k, v, w.P, w.causal)
    idx = torch.from_numpy(rows).to(DEV)
    got_out = out.index_select(0, idx).cpu()
    got_lse = lse.index_select(0, idx).cpu()
    del out, lse
    torch.cuda.empty_cache()
    ref_out, ref_lse = oracle.attention(q, k, v, causal=w.causal, rows=rows)
    check_output(got_out, got_lse, ref_out, ref_lse, w.dtype)


SHAPES = [
    # N, P, heads, kv_heads, d, dtype, causal
    (600, 3, 4, 2, 128, torch.bfloat16, True),    # c = 200: ragged tail tile
    (600, 3, 4, 2, 128, torch.bfloat16, False),
    (1000, 5, 2, 1, 64, torch.bfloat16, True),    # MQA, d = 64
    (256, 1, 2, 2, 128, torch.bfloat16, True),    # P = 1: a single block
    (130, 2, 1, 1, 128, torch.bfloat16, True),    # c = 65 < one tile
    (8, 8, 1, 1, 64, torch.bfloat16, True),       # c = 1
    # head counts for every grouping of the fused launch order (chunks of
    # 4, 2 or 1 heads), including chunks that straddle two KV heads
    (1024, 4, 3, 1, 128, torch.bfloat16, True),   # odd: chunks of 1, GQA 3:1
    (1536, 3, 6, 2, 64, torch.bfloat16, True),    # chunks of 2, three of them
    (1024, 4, 12, 4, 128, torch.bfloat16, True),  # chunks of 4 over groups of 3
    (768, 2, 5, 5, 64, torch.bfloat16, False),    # odd, non-causal
    (1536, 6, 3, 1, 64, torch.float32, True),     # fp32 path, GQA 3:1
    (768, 2, 2, 2, 128, torch.float32, False),    # fp32, d = 128
]


@pytest.mark.parametrize("shape", SHAPES)
def test_ring_shapes_match_oracle(shape):
    N, P, heads, kv_heads, d, dtype, causal = shape
    q, k, v = inputs.make_random(N, heads, kv_heads, d, dtype=dtype, seed=N + P + d)
    out, lse = run_ring(q, k, v, P, causal)
    ref_out, ref_lse = oracle.attention(q, k, v, causal=causal)
    check_output(out, lse, ref_out, ref_lse, kind_of(dtype))


def test_empty_sequence():
    z = torch.zeros(0, 2, 64, dtype=torch.bfloat16, device=DEV)
    out, lse = ra.ra_ring_forward(z, z, z, P=4, causal=True)
    assert out.shape == (0, 2, 64) and lse.shape == (0, 2)


def test_large_logits_stay_finite():
    q, k, v = inputs.make_random(1024, 2, 2, 128, dtype=torch.bfloat16, seed=77)
    q = (q.float() * 30).to(torch.bfloat16)  # scores of several hundred
    out, lse = run_ring(q, k, v, 4, True)
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    ref_out, ref_lse = oracle.attention(q, k, v, causal=True)
    check_output(out, lse, ref_out, ref_lse, "bf16")


def test_values_all_one_give_one():
    q, k, _ = inputs.make_random(2048, 4, 2, 128, dtype=torch.bfloat16, seed=5)
    v = torch.ones(2048, 2, 128, dtype=torch.bfloat16)
    out, _ = run_ring(q, k, v, 8, True)
    assert (out - 1).abs().max().item() <= TOL["bf16"]["o"]


def test_block_count_does_not_change_the_result():
    q, k, v = inputs.make_random(2048, 2, 1, 128, dtype=torch.bfloat16, seed=9)
    ref_out, ref_lse = oracle.attention(q, k, v, causal=True)
    outs = []
    for P in (1, 2, 4, 8, 16):
        out, lse = run_ring(q, k, v, P, True)
        check_output(out, lse, ref_out, ref_lse, "bf16")
        outs.append(out)
    for x in outs[1:]:
        assert (x - outs[0]).abs().max().item() <= TOL["bf16"]["o"]


def stepwise_ring(q, k, v, P, causal, save_after=None):
    """init + ra_ring_step for s = 0..P-1 + finalize.  With save_after = k,
    the (m, l, O~) state goes to the host after step k, the device copies
    are overwritten with NaN, and the state is restored (checkpoint and
    resume)."""
    N, heads, d = q.shape
    m = torch.empty(N, heads, device=DEV)
    l = torch.empty(N, heads, device=DEV)
    o = torch.empty(N, heads, d, device=DEV)
    ra.ra_state_init(m, l, o)
    for s in range(P):
        ra.ra_ring_step(q, k, v, m, l, o, P=P, s=s, causal=causal)
        if s == save_after:
            saved = [x.cpu() for x in (m, l, o)]
            for x in (m, l, o):
                x.fill_(float("nan"))
            for x, y in zip((m, l, o), saved):
                x.copy_(y)
    out, lse = ra.ra_finalize(m, l, o)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_ring_equals_its_steps_and_resumes_from_saved_state(dtype):
    """init + ra_ring_step for s = 0..P-1 + finalize gives the same bits
    when the (m, l, O~) state is saved to the host after step 1 and restored
    (checkpoint and resume).  ra_ring_forward equals that composition bit
    for bit in fp32 (it is that composition); in bf16 it is one fused launch
    that keeps the state on chip, equal up to the finalize's roundings."""
    N, P, heads, kv_heads, d = 1024, 4, 2, 1, 64
    q, k, v = (t.to(DEV) for t in inputs.make_random(N, heads, kv_heads, d, dtype=dtype, seed=13))
    ref_out, ref_lse = ra.ra_ring_forward(q, k, v, P=P, causal=True)
    out0, lse0 = stepwise_ring(q, k, v, P, True)
    out, lse = stepwise_ring(q, k, v, P, True, save_after=1)
    assert torch.equal(out, out0) and torch.equal(lse, lse0)
    if dtype == torch.float32:
        assert torch.equal(out, ref_out)
        assert torch.equal(lse, ref_lse)
    else:
        assert_fused_matches(ref_out, ref_lse, out, lse)


def test_ring_equals_single_pair_calls():
    """The all-ranks ring step computes, for every rank, the same bits as
    per-pair ra_block_update calls made in ring order (and the fused ring
    matches both up to the finalize's roundings)."""
    N, P, heads, d = 768, 3, 2, 128
    q, k, v = (t.to(DEV) for t in inputs.make_random(N, heads, heads, d, seed=15))
    ref_out, ref_lse = stepwise_ring(q, k, v, P, True)
    fused_out, fused_lse = ra.ra_ring_forward(q, k, v, P=P, causal=True)
    assert_fused_matches(fused_out, fused_lse, ref_out, ref_lse)
    c = N // P
    for i in range(P):
        m = torch.empty(c, heads, device=DEV)
        l = torch.empty(c, heads, device=DEV)
        o = torch.empty(c, heads, d, device=DEV)
        ra.ra_state_init(m, l, o)
        for s in range(P):
            j = (i - s) % P
            if j > i:
                continue
            sl = slice(i * c, (i + 1) * c)
            kv = slice(j * c, (j + 1) * c)
            ra.ra_block_update(q[sl], k[kv], v[kv], m, l, o, q_off=i * c, kv_off=j * c,
                               causal=True)
        out, lse = ra.ra_finalize(m, l, o)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out[i * c:(i + 1) * c])
        assert torch.equal(lse, ref_lse[i * c:(i + 1) * c])


@pytest.mark.parametrize("shape", [
    (1024, 4, 2, 128, True, True),     # 2 KV-head groups, pinned
    (4096, 32, 8, 128, True, True),    # 4 groups of 2 KV heads (the gqa-128k grouping)
    (2048, 6, 3, 64, False, True),     # 3 groups, pageable host memory
    (1000, 8, 8, 64, True, False),     # 4 groups, non-causal, ragged last block
])
def test_host_buffer_entry_point(shape):
    """The host-buffer ring (bf16: KV-head groups pipelined against their
    copies) gives the device ring's bits."""
    N, heads, kv_heads, d, pinned, causal = shape
    q, k, v = inputs.make_random(N, heads, kv_heads, d, dtype=torch.bfloat16, seed=19)
    if pinned:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    P = 4 if N % 4 == 0 else 8
    out_h, lse_h = ra.ra_ring_forward_host(q, k, v, P=P, causal=causal)
    out_d, lse_d = run_ring(q, k, v, P, causal)
    assert not out_h.is_cuda
    assert torch.equal(out_h, out_d.cpu()) and torch.equal(lse_h, lse_d.cpu())


def test_scratch_pool_keeps_and_releases_staging():
    """The host-buffer call's device staging comes from the library's pool:
    it stays cached after the call (a second call of the same size adds
    nothing) and goes back to the driver on release."""
    N, heads, kv_heads, d = 4096, 8, 2, 128
    q, k, v = inputs.make_random(N, heads, kv_heads, d, dtype=torch.bfloat16, seed=23)
    q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    staging = N * heads * d * 2 + 2 * N * kv_heads * d * 2 + N * heads * (d + 1) * 4
    out1, lse1 = ra.ra_ring_forward_host(q, k, v, P=4, causal=True)
    torch.cuda.synchronize()
    held = ra.ra_cached_memory()
    assert held >= staging
    out2, lse2 = ra.ra_ring_forward_host(q, k, v, P=4, causal=True)
    torch.cuda.synchronize()
    assert ra.ra_cached_memory() == held
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)
    ra.ra_release_cached_memory()
    assert ra.ra_cached_memory() == 0


def test_more_than_256_ranks_takes_the_step_path():
    """bf16 with P > 256 (beyond the fused launch's visit table) runs one
    launch per ring step; it gives the attention of the fused P = 256 ring
    and of the oracle on sampled rows."""
    N, heads, kv_heads, d = 10240, 2, 1, 64
    q, k, v = inputs.make_random(N, heads, kv_heads, d, seed=29)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    got = trace_counts(lambda: ra.ra_ring_forward(qd, kd, vd, P=320, causal=True))
    assert got["ring_fused_bf16"][0] == 0 and got["block_update_bf16"][0] == 320
    out, lse = ra.ra_ring_forward(qd, kd, vd, P=320, causal=True)
    out_f, lse_f = ra.ra_ring_forward(qd, kd, vd, P=256, causal=True)
    ra.ra_device_status()
    assert (out - out_f).abs().max().item() <= TOL["bf16"]["o"]
    rows = np.array([0, 1, 31, 32, 5000, 10239])
    idx = torch.from_numpy(rows).to(DEV)
    ref_out, ref_lse = oracle.attention(q, k, v, causal=True, rows=rows)
    check_output(out.index_select(0, idx).cpu(), lse.index_select(0, idx).cpu(), ref_out, ref_lse,
                 "bf16")


def trace_counts(run):
    ra.ra_trace_reset()
    ra.ra_trace_enable(True)
    try:
        run()
        got = {kind: ra.ra_trace_query(kind)
               for kind in ("ring_fused_bf16", "ring_fused_f32", "block_update_bf16",
                            "block_update_f32", "state_init", "finalize")}
    finally:
        ra.ra_trace_enable(False)
        ra.ra_trace_reset()
    return got


@pytest.mark.parametrize("shape", [
    # N, heads, kv_heads, d, P, layout, window
    (16384, 8, 2, 128, 4, "contiguous", 0),
    (8192, 8, 8, 64, 8, "contiguous", 0),
    (12288, 4, 1, 128, 6, "zigzag", 3000),
])
def test_fused_ring_is_bitwise_repeatable(shape):
    """The fused ring forward gives the same bits on every run: its order
    of operations is fixed, so a difference would mean a race (an mbarrier
    phase read two phases late, a TMEM buffer overwritten early)."""
    N, heads, kv_heads, d, P, layout, window = shape
    q, k, v = inputs.make_random(N, heads, kv_heads, d, seed=N + d)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    runs = []
    for _ in range(4):
        out, lse = ra.ra_ring_forward_masked(qd, kd, vd, P=P, layout=layout, causal=True,
                                             window=window)
        runs.append((out.clone(), lse.clone()))
    ra.ra_device_status()
    for out, lse in runs[1:]:
        assert torch.equal(out, runs[0][0]) and torch.equal(lse, runs[0][1])


def test_trace_counts_launches():
    """bf16 and fp32: the whole ring is one fused launch (tcgen05, FFMA)."""
    q, k, v = (t.to(DEV) for t in inputs.make_random(1024, 2, 2, 128, seed=21))
    got = trace_counts(lambda: ra.ra_ring_forward(q, k, v, P=4, causal=True))
    assert [got[x][0] for x in ("ring_fused_bf16", "block_update_bf16", "state_init",
                                "finalize")] == [1, 0, 0, 0]
    assert got["ring_fused_bf16"][1] > 0
    q, k, v = (t.to(DEV) for t in inputs.make_random(1024, 2, 2, 64, dtype=torch.float32,
                                                     seed=21))
    got = trace_counts(lambda: ra.ra_ring_forward(q, k, v, P=4, causal=True))
    assert [got[x][0] for x in ("ring_fused_f32", "ring_fused_bf16", "block_update_f32",
                                "state_init", "finalize")] == [1, 0, 0, 0, 0]
    assert got["ring_fused_f32"][1] > 0
