"""Host-side checks of the C ABI that need no GPU.  The library must load,
export every function include/ra.h declares, and reject bad arguments
before any CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from blockwise_online_softmax_gb300 import build as b
    from blockwise_online_softmax_gb300 import binding

    b.build()
    return binding.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "ra.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ra_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("ra_state_init", "ra_block_update", "ra_merge", "ra_finalize",
                     "ra_ring_forward"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(os.path.join(ROOT, "blockwise_online_softmax_gb300", "libra.so"))
    missing = [n for n in declared_functions() if not hasattr(raw, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol():
    from blockwise_online_softmax_gb300 import binding

    assert set(declared_functions()) <= set(binding._SIGNATURES)


def test_status_strings(lib):
    assert lib.ra_abi_version() == 3
    for code, name in ((0, b"RA_OK"), (-1, b"RA_ERR_INVALID"), (-2, b"RA_ERR_UNSUPPORTED"),
                       (-3, b"RA_ERR_CUDA"), (-4, b"RA_ERR_TIMEOUT"), (-5, b"RA_ERR_ALLOC")):
        assert lib.ra_status_string(code) == name


# Argument checks run before any CUDA call, so they work without a GPU.
# Pointers are fake but never dereferenced.
FAKE = 0x10000


@pytest.mark.parametrize("args, code, msg", [
    # (c, d, heads, kv_heads, dtype)
    ((128, 96, 1, 1, 1), -2, b"head dim"),
    ((128, 64, 4, 3, 1), -1, b"multiple of kv_heads"),
    ((128, 64, 0, 1, 1), -1, b"heads"),
    ((128, 64, 2, 0, 1), -1, b"kv_heads"),
    ((128, 64, 2, 2, 7), -1, b"dtype"),
    ((-1, 64, 2, 2, 1), -1, b"negative"),
])
def test_block_update_rejects_bad_arguments(lib, args, code, msg):
    c, d, heads, kv_heads, dtype = args
    rc = lib.ra_block_update(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, c, d, heads, kv_heads, 0, 0, 1,
                             dtype, None)
    assert rc == code
    assert msg in lib.ra_last_error()


def test_null_and_misaligned_pointers_rejected(lib):
    rc = lib.ra_block_update(None, FAKE, FAKE, FAKE, FAKE, FAKE, 128, 64, 1, 1, 0, 0, 0, 1, None)
    assert rc == -1 and b"NULL" in lib.ra_last_error()
    rc = lib.ra_block_update(FAKE + 4, FAKE, FAKE, FAKE, FAKE, FAKE, 128, 64, 1, 1, 0, 0, 0, 1,
                             None)
    assert rc == -1 and b"aligned" in lib.ra_last_error()
    rc = lib.ra_merge(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 8, 4, 128, 2, None)
    assert rc == -1 and b"aligned" in lib.ra_last_error()


def test_ring_arguments(lib):
    rc = lib.ra_ring_forward(FAKE, FAKE, FAKE, FAKE, FAKE, 1000, 3, 1, 64, 2, 2, 1, None)
    assert rc == -1 and b"multiple of P" in lib.ra_last_error()
    rc = lib.ra_ring_forward(FAKE, FAKE, FAKE, FAKE, FAKE, 1024, 0, 1, 64, 2, 2, 1, None)
    assert rc == -1 and b"P=0" in lib.ra_last_error()
    rc = lib.ra_ring_step(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1024, 4, 4, 1, 64, 2, 2, 1, None)
    assert rc == -1 and b"ring step" in lib.ra_last_error()
    rc = lib.ra_ring_forward_host(None, FAKE, FAKE, FAKE, FAKE, 1024, 4, 1, 64, 2, 2, 1, None)
    assert rc == -1


def test_zero_size_work_is_a_no_op(lib):
    # c == 0 / N == 0 returns RA_OK without touching memory or the GPU.
    assert lib.ra_block_update(None, None, None, None, None, None, 0, 64, 1, 1, 0, 0, 1, 1,
                               None) == 0
    assert lib.ra_ring_forward(None, None, None, None, None, 0, 4, 1, 128, 8, 8, 1, None) == 0
    assert lib.ra_state_init(None, None, None, 0, 64, 1, None) == 0
    assert lib.ra_merge(None, None, None, None, None, None, 0, 64, 1, None) == 0
    assert lib.ra_finalize(None, None, None, None, None, 0, 64, 1, None) == 0


def test_cached_memory_arguments(lib):
    assert lib.ra_cached_memory(None) == -1
    assert b"NULL" in lib.ra_last_error()


def test_trace_controls(lib):
    assert lib.ra_trace_enable(0) == 0
    assert lib.ra_trace_reset() == 0
    n = ctypes.c_longlong(-1)
    ms = ctypes.c_double(-1)
    assert lib.ra_trace_query(1, ctypes.addressof(n), ctypes.addressof(ms)) == 0
    assert n.value == 0 and ms.value == 0.0
    assert lib.ra_trace_query(99, ctypes.addressof(n), ctypes.addressof(ms)) == -1


def test_binding_marshalling_errors():
    import torch

    from blockwise_online_softmax_gb300 import binding

    q = torch.zeros(8, 2, 64)
    with pytest.raises(ValueError):
        binding.ra_ring_forward(q, q, q, P=2, causal=True)  # CPU tensors are refused
    with pytest.raises(ValueError):
        binding._shapes(q, torch.zeros(8, 2, 32), torch.zeros(8, 2, 32))


def test_noalloc_size_limit_is_checked_before_the_pointers(lib):
    # ra_ring_forward_noalloc refuses N * heads above its fixed scratch
    # (4,194,304 entries) before it looks at the pointers, so NULL pointers
    # give the size error; at the limit they give the NULL-pointer error.
    limit = 1 << 22
    for dtype in (0, 1):
        rc = lib.ra_ring_forward_noalloc(None, None, None, None, None, limit // 4 + 256, 1, 1, 64,
                                         4, 4, dtype, None)
        assert rc == -2 and b"fixed scratch" in lib.ra_last_error()
        rc = lib.ra_ring_forward_noalloc(None, None, None, None, None, limit // 4, 1, 1, 64, 4, 4,
                                         dtype, None)
        assert rc == -1 and b"NULL" in lib.ra_last_error()
