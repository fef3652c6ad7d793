"""Host-side checks of the token layouts and of the masked calls' argument
checks.  No GPU is needed.

The layouts are those of "Ring Attention Paper Breakdown", section "5.
Causal Masking Imbalance & Striped / ZigZag Attention", and "RingAttention:
Scaling LLM Context to 10M Tokens", section "Causal Masking: Striped and
Zig-Zag RingAttention": striped puts token t on rank t mod P, zigzag gives
rank i the chunks i and 2P-1-i of 2P.  Both pages state that these make the
causal work of every rank equal; the balance tests below check that claim
on the positions the library uses, by counting allowed pairs.
"""
import ctypes

import numpy as np
import pytest

from blockwise_online_softmax_gb300 import binding

FAKE = 0x10000


@pytest.fixture(scope="module")
def lib():
    from blockwise_online_softmax_gb300 import build

    build.build()
    return binding.lib()


@pytest.mark.parametrize("layout", ["contiguous", "zigzag", "striped"])
def test_positions_are_a_permutation_increasing_inside_blocks(layout):
    N, P = 96, 4
    pos = binding.layout_positions(N, P, layout).numpy()
    assert sorted(pos.tolist()) == list(range(N))
    blocks = pos.reshape(P, N // P)
    assert (np.diff(blocks, axis=1) > 0).all()


def test_zigzag_and_striped_match_the_pages_assignment():
    N, P = 80, 5
    c, h = N // P, N // (2 * P)
    z = binding.layout_positions(N, P, "zigzag").numpy().reshape(P, c)
    for i in range(P):
        want = list(range(i * h, (i + 1) * h)) + list(range((2 * P - 1 - i) * h, (2 * P - i) * h))
        assert z[i].tolist() == want
    s = binding.layout_positions(N, P, "striped").numpy().reshape(P, c)
    for i in range(P):
        assert (s[i] % P == i).all()


def _causal_pairs(pos, P, i, j):
    c = pos.shape[0] // P
    qp = pos[i * c:(i + 1) * c]
    kp = pos[j * c:(j + 1) * c]
    return int((kp[None, :] <= qp[:, None]).sum())


def test_zigzag_balances_causal_work_at_every_step():
    N, P = 128, 4
    pos = binding.layout_positions(N, P, "zigzag").numpy()
    for s in range(P):
        work = [_causal_pairs(pos, P, i, (i - s) % P) for i in range(P)]
        assert len(set(work)) == 1, (s, work)
    naive = binding.layout_positions(N, P, "contiguous").numpy()
    work = [_causal_pairs(naive, P, i, (i - 1) % P) for i in range(P)]
    assert len(set(work)) > 1  # the imbalance the layouts remove


def test_striped_balances_causal_work_within_one_block_row():
    # Striped ranks differ by at most c pairs (one diagonal) at any step.
    N, P = 128, 4
    c = N // P
    pos = binding.layout_positions(N, P, "striped").numpy()
    for s in range(P):
        work = [_causal_pairs(pos, P, i, (i - s) % P) for i in range(P)]
        assert max(work) - min(work) <= c
        assert min(work) >= c * (c - 1) // 2


def test_layout_argument_errors():
    with pytest.raises(ValueError):
        binding.layout_positions(10, 3, "zigzag")
    with pytest.raises(ValueError):
        binding.layout_positions(12, 2, "diagonal")
    with pytest.raises(ValueError):
        binding.layout_positions(6, 2, "zigzag")  # c = 3 is odd


def ring_fwd_masked(lib, N=1024, P=4, layout=0, causal=1, window=0, n_valid=-1, cu=FAKE,
                    ndocs=0, d=64, heads=2, kv_heads=2, dtype=1):
    return lib.ra_ring_forward_masked(FAKE, FAKE, FAKE, FAKE, FAKE, N, P, layout, causal, window,
                                      n_valid, cu, ndocs, d, heads, kv_heads, dtype, None)


@pytest.mark.parametrize("kw, msg", [
    (dict(layout=3), b"layout"),
    (dict(causal=2), b"causal"),
    (dict(window=-1), b"window"),
    (dict(ndocs=-2), b"ndocs"),
    (dict(ndocs=2, cu=None), b"NULL cu_seqlens"),
    (dict(ndocs=2, cu=FAKE + 2), b"aligned"),
    (dict(layout=1, N=12, P=4), b"odd"),
    (dict(N=1000, P=3), b"multiple of P"),
])
def test_masked_ring_rejects_bad_arguments(lib, kw, msg):
    assert ring_fwd_masked(lib, **kw) == -1
    assert msg in lib.ra_last_error()


def test_masked_block_update_rejects_bad_arguments(lib):
    def call(c_q=256, c_kv=256, layout=1, P=4, qb=0, kb=1):
        return lib.ra_block_update_masked(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, c_q, c_kv, 64, 2, 2,
                                          layout, P, qb, kb, 0, 0, 1, 0, -1, None, 0, 1, None)
    assert call(c_kv=128) == -1 and b"zigzag" in lib.ra_last_error()
    assert call(c_q=255, c_kv=255) == -1 and b"even" in lib.ra_last_error()
    assert call(kb=4) == -1 and b"range" in lib.ra_last_error()
    assert call(layout=2, P=0) == -1 and b"P=0" in lib.ra_last_error()
    # contiguous ignores P and the block indices; zero-size is a no-op
    assert call(c_q=0, layout=0, P=0, kb=9) == 0


def test_masked_zero_size_is_a_no_op(lib):
    assert lib.ra_ring_forward_masked(None, None, None, None, None, 0, 4, 1, 1, 16, 5, None, 0,
                                      64, 2, 2, 1, None) == 0
    assert lib.ra_ring_step_masked(None, None, None, None, None, None, 0, 4, 0, 2, 0, 0, -1, None,
                                   0, 64, 2, 2, 1, None) == 0


def test_decode_rejects_bad_arguments(lib):
    def fwd(n_q=1, heads=32, kv_heads=8, d=128, dtype=1, P=4, window=0):
        return lib.ra_decode_forward(FAKE, FAKE, FAKE, FAKE, FAKE, n_q, 1000, P, 999, 1, window,
                                     d, heads, kv_heads, dtype, None)
    assert fwd(heads=258, kv_heads=2) == -2 and b"exceeds 128" in lib.ra_last_error()
    assert fwd(n_q=(1 << 24) + 1) == -2 and b"2^24" in lib.ra_last_error()
    assert fwd(n_q=1 << 24, heads=256, kv_heads=2) == -2 and b"2^31" in lib.ra_last_error()
    assert fwd(dtype=0) == -2 and b"bf16" in lib.ra_last_error()
    assert fwd(P=0) == -1 and b"P=0" in lib.ra_last_error()
    assert fwd(window=-3) == -1 and b"window" in lib.ra_last_error()
    assert fwd(d=96) == -2
    assert lib.ra_decode_forward(None, None, None, None, None, 0, 1000, 4, 0, 1, 0, 128, 32, 8,
                                 1, None) == 0  # n_q = 0: nothing to do
    assert lib.ra_decode_partial(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 0, 128, 32, 8, 0, 0, 1,
                                 0, 1, None) == 0  # n_kv = 0: the state stays


def test_decode_workload_sizes():
    from blockwise_online_softmax_gb300 import inputs

    w = inputs.DECODE_WORKLOADS["decode-1m"]
    assert w.kv_bytes() == 2 * (1 << 20) * 8 * 128 * 2
    assert w.flops() == 4.0 * 128 * 32 * (1 << 20)
