"""The allocation-free ring forward (ra_ring_forward_noalloc).

It is meant for callers that cannot let the library allocate device
memory, such as an application that keeps the whole GPU in its own pool.
The call keeps its l state in a fixed device array inside the library.
This file runs last (pytest collects it after the others).  It must pass
on its own in a fresh process and after the rest of the suite.  It checks
that two calls in a row, through the C ABI, match ra_ring_forward (and,
for the fp32 case, the oracle directly), including a case with P > 256,
the step-by-step ring that keeps its l state in the fixed array, that
neither torch's allocator nor the library's scratch pool grows over those
calls, and that sizes over the fixed limit are refused.
"""
import ctypes

import pytest
import torch

from parity import check_output

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
LIMIT = 1 << 22  # N * heads entries of the fixed scratch


@pytest.fixture(scope="module")
def lib():
    from blockwise_online_softmax_gb300 import binding, build

    build.build()
    return binding.lib()


def _call(L, q, k, v, out, lse, P, causal):
    N, heads, d = q.shape
    return L.ra_ring_forward_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
        ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(lse.data_ptr()), N, P, int(causal), d, heads, k.shape[1],
        1 if q.dtype == torch.bfloat16 else 0, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("shape", [
    # N, P, heads, kv_heads, d, dtype, causal
    (4096, 4, 8, 2, 128, torch.bfloat16, True),
    (1000, 5, 2, 2, 64, torch.bfloat16, False),
    (1536, 6, 3, 1, 64, torch.float32, True),
    # P > 256: the step-by-step ring, the calls that use the fixed array
    (600, 300, 2, 1, 64, torch.bfloat16, True),
])
def test_two_calls_match_ring_forward(lib, shape):
    import blockwise_online_softmax_gb300 as ra
    import oracle
    from blockwise_online_softmax_gb300 import inputs

    N, P, heads, kv_heads, d, dtype, causal = shape
    q_h, k_h, v_h = inputs.make_random(N, heads, kv_heads, d, dtype=dtype, seed=N)
    q, k, v = (t.to(DEV) for t in (q_h, k_h, v_h))
    ref_out, ref_lse = ra.ra_ring_forward(q, k, v, P=P, causal=causal)
    oracle_ref = oracle.attention(q_h, k_h, v_h, causal=causal) if dtype == torch.float32 else None
    tol = 1e-2 if dtype == torch.bfloat16 else 1e-5
    outs = [torch.full((N, heads, d), float("nan"), device=DEV) for _ in range(2)]
    lses = [torch.full((N, heads), float("nan"), device=DEV) for _ in range(2)]
    torch.cuda.synchronize()
    torch_before = torch.cuda.memory_allocated(DEV)
    pool_before = ra.ra_cached_memory()
    for out, lse in zip(outs, lses):
        assert _call(lib, q, k, v, out, lse, P, causal) == 0, lib.ra_last_error()
        assert lib.ra_device_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == 0
    torch.cuda.synchronize()
    # Nothing was allocated by either call: not through torch, not from the
    # library's scratch pool.
    assert torch.cuda.memory_allocated(DEV) == torch_before
    assert ra.ra_cached_memory() == pool_before
    for out, lse in zip(outs, lses):
        assert (out - ref_out).abs().max().item() <= tol
        rel = (lse - ref_lse).abs() / ref_lse.abs().clamp(min=1.0)
        assert rel.max().item() <= (1e-3 if dtype == torch.bfloat16 else 1e-5)
        if oracle_ref is not None:
            check_output(out, lse, oracle_ref[0], oracle_ref[1], "f32")


def test_over_the_limit_is_refused(lib):
    # N * heads one block over the fixed scratch: refused before any launch.
    # The pointers are NULL, so no call can reach a buffer: were the size
    # check ever moved behind the pointer check, the call would fail with
    # the NULL-pointer message instead and this test would say so.
    N, heads = LIMIT // 4 + 256, 4
    rc = lib.ra_ring_forward_noalloc(None, None, None, None, None, N, 1, 1, 64, heads, heads, 1,
                                     None)
    assert rc == -2, lib.ra_last_error()  # RA_ERR_UNSUPPORTED
    assert b"fixed scratch" in lib.ra_last_error()
