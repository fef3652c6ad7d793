"""GPU parity of the decode / short-query path against the CPU oracle.

A few query tokens meet a long K/V history held as P shards: each shard's
partial state, then the global merge reduction ("Ring Attention：把超长序列
沿设备环流动", section "训练与推理的适用方式不同").  The oracle sees only
the plain definition over the whole history."""
import numpy as np
import pytest
import torch

import oracle
from parity import check_output, check_state

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


def qkv(n_q, heads, kv_heads, d, n_kv, seed, scale=1.0):
    q, _, _ = inputs.make_random(n_q, heads, kv_heads, d, seed=seed, scale=scale)
    _, k, v = inputs.make_random(n_kv, heads, kv_heads, d, seed=seed + 1, scale=scale)
    return q, k, v


CASES = [
    # n_q, heads, kv_heads, d, n_kv, P, causal, window
    (1, 32, 8, 128, 5000, 4, True, 0),
    (4, 32, 8, 128, 20000, 8, True, 0),      # 16 rows per KV head
    (2, 8, 1, 64, 3001, 3, True, 0),         # MQA, ragged shards
    (1, 4, 4, 128, 777, 1, False, 0),        # MHA, one shard, non-causal
    (3, 12, 4, 64, 10000, 5, True, 1000),    # sliding window
    (16, 16, 16, 128, 4096, 2, True, 0),     # 16 new tokens, causal among them
    (1, 8, 2, 128, 31, 7, True, 0),          # fewer keys than a tile; empty shards
    # more than 4 rows per KV head: the tensor-core chunks
    (32, 32, 8, 128, 9000, 4, True, 0),      # 128 rows per KV head
    (100, 4, 4, 64, 3000, 3, True, 0),       # 100 rows, MHA, d = 64
    (8, 64, 8, 128, 20000, 16, True, 2048),  # 64 rows, windowed
    (5, 8, 8, 128, 777, 2, False, 0),        # 5 rows, non-causal, ragged
    (3, 32, 8, 64, 130, 8, True, 0),         # 12 rows, shards shorter than a tile
    # more than 128 rows per KV head: several 128-row tiles
    (64, 32, 8, 128, 6000, 4, True, 0),      # 256 rows: two full tiles of 32 tokens
    (50, 12, 4, 64, 4000, 3, True, 700),     # g = 3: tiles of 42 tokens, the last partial
    (300, 2, 2, 128, 2000, 2, False, 0),     # MHA: three tiles of 128 tokens, non-causal
    (20, 256, 2, 64, 1000, 2, True, 0),      # g = 128: one token per tile
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"q{c[0]}-h{c[1]}/{c[2]}-d{c[3]}-kv{c[4]}"
                         f"-P{c[5]}-{'c' if c[6] else 'nc'}-w{c[7]}")
def test_decode_forward_matches_oracle(case):
    n_q, heads, kv_heads, d, n_kv, P, causal, window = case
    q, k, v = qkv(n_q, heads, kv_heads, d, n_kv, seed=n_kv + n_q)
    q_off = n_kv - n_q
    out, lse = ra.ra_decode_forward(q.to(DEV), k.to(DEV), v.to(DEV), P=P, q_off=q_off,
                                    causal=causal, window=window)
    ra.ra_device_status()
    ref_out, ref_lse = oracle.attention(q, k, v, causal=causal, window=window,
                                        q_pos=q_off + np.arange(n_q), k_pos=np.arange(n_kv))
    check_output(out, lse, ref_out, ref_lse, "bf16")


def test_decode_shard_count_does_not_change_the_result():
    q, k, v = qkv(2, 16, 4, 128, 9000, seed=5)
    res = [ra.ra_decode_forward(q.to(DEV), k.to(DEV), v.to(DEV), P=P) for P in (1, 2, 7, 64)]
    ref_out, ref_lse = oracle.attention(q, k, v, causal=True, q_pos=8998 + np.arange(2))
    for out, lse in res:
        check_output(out, lse, ref_out, ref_lse, "bf16")


def test_decode_partial_accumulates_over_shards():
    """Two ra_decode_partial calls into one state equal the oracle's partial
    state over both shards; keys past the queries are masked by position."""
    n_q, heads, kv_heads, d = 3, 8, 2, 128
    q, k, v = qkv(n_q, heads, kv_heads, d, 6000, seed=9)
    q_off = 4000  # the queries sit inside the history: later keys are masked
    m = torch.empty(n_q, heads, device=DEV)
    l = torch.empty(n_q, heads, device=DEV)
    o = torch.empty(n_q, heads, d, device=DEV)
    ra.ra_state_init(m, l, o)
    qd = q.to(DEV)
    for lo, hi in ((0, 2500), (2500, 6000)):
        ra.ra_decode_partial(qd, k[lo:hi].to(DEV), v[lo:hi].to(DEV), m, l, o, q_off=q_off,
                             kv_off=lo, causal=True)
    ra.ra_device_status()
    ref = oracle.partial_state(q, k, v, causal=True, q_pos=q_off + np.arange(n_q))
    check_state(m, l, o, ref, "bf16")


def test_decode_without_keys():
    q = torch.randn(2, 4, 64).to(torch.bfloat16).to(DEV)
    z = torch.zeros(0, 2, 64, dtype=torch.bfloat16, device=DEV)
    out, lse = ra.ra_decode_forward(q, z, z, P=4)
    torch.cuda.synchronize()
    assert (out == 0).all() and torch.isneginf(lse).all()


@pytest.mark.parametrize("window", [0, 3])
def test_decode_rows_that_see_no_key(window):
    """Query positions before the first key (q_off < 0, causal) see no key:
    the reduction over the shards gives out = 0 and lse = -inf for them and
    the plain result for the others."""
    n_q, heads, kv_heads, d, n_kv = 6, 8, 2, 128, 700
    q, k, v = qkv(n_q, heads, kv_heads, d, n_kv, seed=41)
    q_off = -3  # positions -3 .. 2
    out, lse = ra.ra_decode_forward(q.to(DEV), k.to(DEV), v.to(DEV), P=5, q_off=q_off,
                                    causal=True, window=window)
    ra.ra_device_status()
    ref_out, ref_lse = oracle.attention(q, k, v, causal=True, window=window,
                                        q_pos=q_off + np.arange(n_q), k_pos=np.arange(n_kv))
    assert np.isneginf(ref_lse[:3]).all() and np.isfinite(ref_lse[3:]).all()
    check_output(out, lse, ref_out, ref_lse, "bf16")
    assert (out[:3].cpu() == 0).all()


def test_decode_is_bitwise_repeatable():
    """Chunk kernel and reduction have a fixed order of operations: every
    run gives the same bits."""
    q, k, v = qkv(4, 32, 8, 128, 50000, seed=17)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    runs = [ra.ra_decode_forward(qd, kd, vd, P=16, q_off=50000 - 4) for _ in range(4)]
    ra.ra_device_status()
    for out, lse in runs[1:]:
        assert torch.equal(out, runs[0][0]) and torch.equal(lse, runs[0][1])


def test_decode_large_logits_stay_finite():
    q, k, v = qkv(1, 8, 8, 128, 4000, seed=11)
    k = (k.float() * 20).to(torch.bfloat16)
    out, lse = ra.ra_decode_forward(q.to(DEV), k.to(DEV), v.to(DEV), P=4)
    ref_out, ref_lse = oracle.attention(q, k, v, causal=True, q_pos=np.array([3999]))
    check_output(out, lse, ref_out, ref_lse, "bf16")


@pytest.mark.slow
def test_decode_one_million_keys():
    """The decode workload at full size: 1 query token, 32/8 heads, d = 128,
    a history of 1,048,576 keys in 64 shards."""
    w = inputs.DECODE_WORKLOADS["decode-1m"]
    q, k, v = inputs.make_decode(w)
    out, lse = ra.ra_decode_forward(q.to(DEV), k.to(DEV), v.to(DEV), P=w.P)
    ra.ra_device_status()
    ref_out, ref_lse = oracle.attention(q, k, v, causal=True,
                                        q_pos=w.n_kv - w.n_q + np.arange(w.n_q))
    check_output(out, lse, ref_out, ref_lse, "bf16")


@pytest.mark.slow
def test_decode_four_tokens_one_million_keys():
    w = inputs.DECODE_WORKLOADS["decode-1m-q4"]
    q, k, v = inputs.make_decode(w)
    out, lse = ra.ra_decode_forward(q.to(DEV), k.to(DEV), v.to(DEV), P=w.P)
    ra.ra_device_status()
    ref_out, ref_lse = oracle.attention(q, k, v, causal=True,
                                        q_pos=w.n_kv - w.n_q + np.arange(w.n_q))
    check_output(out, lse, ref_out, ref_lse, "bf16")
