"""The allocation-free ring forward (ra_ring_forward_noalloc).

It is meant for callers that cannot let the library allocate device
memory, such as an application that keeps the whole GPU in its own pool.
The call keeps its l state in a fixed device array inside the library.
This file runs last (pytest collects it after the others).  It must pass
on its own in a fresh process and after the rest of the suite.  It checks
that two calls in a row, through the C ABI, match ra_ring_forward, and that
sizes over the fixed limit are refused.
"""
import ctypes

import pytest
import torch

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
])
def test_two_calls_match_ring_forward(lib, shape):
    import blockwise_online_softmax_gb300 as ra
    from blockwise_online_softmax_gb300 import inputs

    N, P, heads, kv_heads, d, dtype, causal = shape
    q, k, v = (t.to(DEV) for t in inputs.make_random(N, heads, kv_heads, d, dtype=dtype, seed=N))
    ref_out, ref_lse = ra.ra_ring_forward(q, k, v, P=P, causal=causal)
    tol = 1e-2 if dtype == torch.bfloat16 else 1e-5
    for _ in range(2):
        out = torch.full((N, heads, d), float("nan"), device=DEV)
        lse = torch.full((N, heads), float("nan"), device=DEV)
        assert _call(lib, q, k, v, out, lse, P, causal) == 0, lib.ra_last_error()
        assert lib.ra_device_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == 0
        assert (out - ref_out).abs().max().item() <= tol
        rel = (lse - ref_lse).abs() / ref_lse.abs().clamp(min=1.0)
        assert rel.max().item() <= (1e-3 if dtype == torch.bfloat16 else 1e-5)


def test_over_the_limit_is_refused(lib):
    # N * heads one block over the fixed scratch: refused before any launch.
    N, heads = LIMIT // 4 + 256, 4
    q = torch.zeros(1, dtype=torch.bfloat16, device=DEV)
    rc = lib.ra_ring_forward_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(q.data_ptr()),
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(q.data_ptr()),
        ctypes.c_void_p(q.data_ptr()), N, 1, 1, 64, heads, heads, 1, None)
    assert rc == -2  # RA_ERR_UNSUPPORTED
    assert b"fixed scratch" in lib.ra_last_error()
