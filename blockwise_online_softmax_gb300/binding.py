"""Thin Python binding over ``libra.so``.  The functions carry the C ABI's
names (include/ra.h).  This module only marshals arguments: it takes torch
tensors, passes raw pointers, sizes and the stream, and turns status codes
into exceptions.  Every step of the computation runs in the library's CUDA
kernels.  There is no fallback.  If ``libra.so`` is missing, the first call
raises ``RaError``.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libra.so")

RA_OK = 0
RA_ERR_INVALID = -1
RA_ERR_UNSUPPORTED = -2
RA_ERR_CUDA = -3
RA_ERR_TIMEOUT = -4
RA_ERR_ALLOC = -5
RA_F32 = 0
RA_BF16 = 1
LAYOUTS = {"contiguous": 0, "zigzag": 1, "striped": 2}
ABI_VERSION = 3
KERNEL_KINDS = {
    "state_init": 0,
    "block_update_bf16": 1,
    "block_update_f32": 2,
    "merge": 3,
    "finalize": 4,
    "decode_split": 5,
    "decode_combine": 6,
    "bwd_pre": 7,
    "bwd_dq": 8,
    "bwd_dkdv": 9,
    "ring_fused_bf16": 10,
    "ring_fused_f32": 11,
}

_lock = threading.Lock()
_lib = None


class RaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} [{status}]")
        self.status = status


_SIGNATURES = {
    # name: (argtypes, restype)
    "ra_state_init": ("PPPLiiP", "i"),
    "ra_block_update": ("PPPPPPLiiiLLiiP", "i"),
    "ra_merge": ("PPPPPPLiiP", "i"),
    "ra_finalize": ("PPPPPLiiP", "i"),
    "ra_ring_step": ("PPPPPPLiiiiiiiP", "i"),
    "ra_ring_forward": ("PPPPPLiiiiiiP", "i"),
    "ra_ring_forward_host": ("PPPPPLiiiiiiP", "i"),
    "ra_ring_forward_noalloc": ("PPPPPLiiiiiiP", "i"),
    "ra_block_update_masked": ("PPPPPPLLiiiiiiiLLiLLPiiP", "i"),
    "ra_ring_step_masked": ("PPPPPPLiiiiLLPiiiiiP", "i"),
    "ra_ring_forward_masked": ("PPPPPLiiiLLPiiiiiP", "i"),
    "ra_decode_partial": ("PPPPPPLLiiiLLiLiP", "i"),
    "ra_ring_backward": ("PPPPPPPPPLiiiiiiP", "i"),
    "ra_ring_backward_masked": ("PPPPPPPPPLiiiLLPiiiiiP", "i"),
    "ra_decode_forward": ("PPPPPLLiLiLiiiiP", "i"),
    "ra_device_status": ("P", "i"),
    "ra_selftest_wait_timeout": ("LP", "i"),
    "ra_cached_memory": ("P", "i"),
    "ra_release_cached_memory": ("", "i"),
    "ra_trace_enable": ("i", "i"),
    "ra_trace_reset": ("", "i"),
    "ra_trace_query": ("iPP", "i"),
    "ra_status_string": ("i", "s"),
    "ra_last_error": ("", "s"),
    "ra_abi_version": ("", "i"),
}
_CT = {"P": ctypes.c_void_p, "L": ctypes.c_longlong, "i": ctypes.c_int, "s": ctypes.c_char_p}


def lib():
    """Load libra.so once.  Raise RaError if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RaError(RA_ERR_UNSUPPORTED,
                              f"{LIB_PATH} is not built; run __graft_entry__.build() "
                              "(nvcc, sm_103a)")
            L = ctypes.CDLL(LIB_PATH)
            for name, (args, res) in _SIGNATURES.items():
                f = getattr(L, name)
                f.argtypes = [_CT[c] for c in args]
                f.restype = _CT[res]
            if L.ra_abi_version() != ABI_VERSION:
                raise RaError(RA_ERR_UNSUPPORTED, "libra.so ABI version mismatch; rebuild it")
            _lib = L
    return _lib


def _check(rc: int):
    if rc != RA_OK:
        L = lib()
        raise RaError(rc, f"{L.ra_status_string(rc).decode()}: {L.ra_last_error().decode()}")


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: torch.Tensor, name: str, dtype=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (token-major)")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _qkv_dtype(q: torch.Tensor) -> int:
    if q.dtype == torch.bfloat16:
        return RA_BF16
    if q.dtype == torch.float32:
        return RA_F32
    raise TypeError(f"q/k/v must be bfloat16 or float32, got {q.dtype}")


def _shapes(q, k, v):
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3:
        raise ValueError("q, k, v must be [rows, heads, d] (token-major)")
    if k.shape != v.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("k and v must match in shape, and q, k, v in dtype")
    if q.shape[2] != k.shape[2]:
        raise ValueError("q and k must share the head dim")
    return q.shape[0], q.shape[1], k.shape[1], q.shape[2]


def _state_shapes(m, l, o, rows, heads, d):
    for name, t, shp in (("m", m, (rows, heads)), ("l", l, (rows, heads)),
                         ("o", o, (rows, heads, d))):
        if tuple(t.shape) != shp:
            raise ValueError(f"{name} must have shape {shp}, got {tuple(t.shape)}")


def ra_state_init(m, l, o, stream=None):
    rows, heads, d = o.shape
    _state_shapes(m, l, o, rows, heads, d)
    _check(lib().ra_state_init(_dev(m, "m", torch.float32), _dev(l, "l", torch.float32),
                               _dev(o, "o", torch.float32), rows, d, heads, _stream(stream)))


def ra_block_update(q, k, v, m, l, o, *, q_off: int = 0, kv_off: int = 0, causal: bool = False,
                    stream=None):
    c, heads, kv_heads, d = _shapes(q, k, v)
    if k.shape[0] != c:
        raise ValueError("the query block and the K/V block must have the same length c")
    _state_shapes(m, l, o, c, heads, d)
    _check(lib().ra_block_update(
        _dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(m, "m", torch.float32),
        _dev(l, "l", torch.float32), _dev(o, "o", torch.float32), c, d, heads, kv_heads,
        int(q_off), int(kv_off), int(bool(causal)), _qkv_dtype(q), _stream(stream)))


def ra_merge(m_a, l_a, o_a, m_b, l_b, o_b, stream=None):
    rows, heads, d = o_a.shape
    _state_shapes(m_a, l_a, o_a, rows, heads, d)
    _state_shapes(m_b, l_b, o_b, rows, heads, d)
    _check(lib().ra_merge(_dev(m_a, "m_a", torch.float32), _dev(l_a, "l_a", torch.float32),
                          _dev(o_a, "o_a", torch.float32), _dev(m_b, "m_b", torch.float32),
                          _dev(l_b, "l_b", torch.float32), _dev(o_b, "o_b", torch.float32),
                          rows, d, heads, _stream(stream)))


def ra_finalize(m, l, o, out=None, lse=None, stream=None):
    rows, heads, d = o.shape
    _state_shapes(m, l, o, rows, heads, d)
    if out is None:
        out = torch.empty_like(o)
    if lse is None:
        lse = torch.empty_like(m)
    _state_shapes(lse, lse, out, rows, heads, d)
    _check(lib().ra_finalize(_dev(m, "m", torch.float32), _dev(l, "l", torch.float32),
                             _dev(o, "o", torch.float32), _dev(out, "out", torch.float32),
                             _dev(lse, "lse", torch.float32), rows, d, heads, _stream(stream)))
    return out, lse


def ra_ring_step(q, k, v, m, l, o, *, P: int, s: int, causal: bool, stream=None):
    N, heads, kv_heads, d = _shapes(q, k, v)
    if k.shape[0] != N:
        raise ValueError("q, k and v must cover the same N tokens")
    _state_shapes(m, l, o, N, heads, d)
    _check(lib().ra_ring_step(
        _dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(m, "m", torch.float32),
        _dev(l, "l", torch.float32), _dev(o, "o", torch.float32), N, int(P), int(s),
        int(bool(causal)), d, heads, kv_heads, _qkv_dtype(q), _stream(stream)))


def ra_ring_forward(q, k, v, *, P: int, causal: bool, out=None, lse=None, stream=None):
    """Returns (out [N, heads, d] fp32, lse [N, heads] fp32)."""
    N, heads, kv_heads, d = _shapes(q, k, v)
    if k.shape[0] != N:
        raise ValueError("q, k and v must cover the same N tokens")
    if out is None:
        out = torch.empty((N, heads, d), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((N, heads), dtype=torch.float32, device=q.device)
    _state_shapes(lse, lse, out, N, heads, d)
    _check(lib().ra_ring_forward(
        _dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(out, "out", torch.float32),
        _dev(lse, "lse", torch.float32), N, int(P), int(bool(causal)), d, heads, kv_heads,
        _qkv_dtype(q), _stream(stream)))
    return out, lse


def _layout(layout) -> int:
    if isinstance(layout, str):
        if layout not in LAYOUTS:
            raise ValueError(f"layout must be one of {sorted(LAYOUTS)}, got {layout!r}")
        return LAYOUTS[layout]
    return int(layout)


def _docs(cu_seqlens):
    """Device pointer and document count of an int32 cu_seqlens tensor (or None)."""
    if cu_seqlens is None:
        return 0, 0
    if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2:
        raise ValueError("cu_seqlens must be 1-D with ndocs + 1 >= 2 entries")
    return _dev(cu_seqlens, "cu_seqlens", torch.int32), cu_seqlens.numel() - 1


def layout_positions(N: int, P: int, layout="contiguous") -> torch.Tensor:
    """Global sequence position held by each row of a ring tensor of N rows
    under `layout` (int64, CPU).  Host index arithmetic for callers that lay
    their tensors out; x_layout = x[argsort(positions)] is not needed, since
    x_layout[r] = x[positions[r]]."""
    lay = _layout(layout)
    if N % P:
        raise ValueError("N must be a multiple of P")
    c = N // P
    r = torch.arange(c, dtype=torch.int64)
    out = []
    for b in range(P):
        if lay == 0:
            out.append(b * c + r)
        elif lay == 1:
            if c % 2:
                raise ValueError("zigzag needs an even block length N / P")
            h = c // 2
            out.append(torch.where(r < h, b * h + r, (2 * P - 1 - b) * h + (r - h)))
        else:
            out.append(r * P + b)
    return torch.cat(out)


def ra_block_update_masked(q, k, v, m, l, o, *, layout="contiguous", P: int = 1,
                           q_block: int = 0, kv_block: int = 0, q_off: int = 0, kv_off: int = 0,
                           causal: bool = False, window: int = 0, n_valid: int = -1,
                           cu_seqlens=None, stream=None):
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3 or k.shape != v.shape:
        raise ValueError("q: [c_q, heads, d]; k, v: [c_kv, kv_heads, d]")
    if k.dtype != q.dtype or v.dtype != q.dtype or q.shape[2] != k.shape[2]:
        raise ValueError("q, k, v must share dtype and head dim")
    c_q, heads, d = q.shape
    c_kv, kv_heads = k.shape[0], k.shape[1]
    _state_shapes(m, l, o, c_q, heads, d)
    cu_ptr, ndocs = _docs(cu_seqlens)
    _check(lib().ra_block_update_masked(
        _dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(m, "m", torch.float32),
        _dev(l, "l", torch.float32), _dev(o, "o", torch.float32), c_q, c_kv, d, heads, kv_heads,
        _layout(layout), int(P), int(q_block), int(kv_block), int(q_off), int(kv_off),
        int(bool(causal)), int(window), int(n_valid), cu_ptr, ndocs, _qkv_dtype(q),
        _stream(stream)))


def ra_ring_step_masked(q, k, v, m, l, o, *, P: int, s: int, layout="contiguous",
                        causal: bool = False, window: int = 0, n_valid: int = -1,
                        cu_seqlens=None, stream=None):
    N, heads, kv_heads, d = _shapes(q, k, v)
    if k.shape[0] != N:
        raise ValueError("q, k and v must cover the same N tokens")
    _state_shapes(m, l, o, N, heads, d)
    cu_ptr, ndocs = _docs(cu_seqlens)
    _check(lib().ra_ring_step_masked(
        _dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(m, "m", torch.float32),
        _dev(l, "l", torch.float32), _dev(o, "o", torch.float32), N, int(P), int(s),
        _layout(layout), int(bool(causal)), int(window), int(n_valid), cu_ptr, ndocs, d, heads,
        kv_heads, _qkv_dtype(q), _stream(stream)))


def ra_ring_forward_masked(q, k, v, *, P: int, layout="contiguous", causal: bool = False,
                           window: int = 0, n_valid: int = -1, cu_seqlens=None, out=None,
                           lse=None, stream=None):
    """Returns (out [N, heads, d] fp32, lse [N, heads] fp32), rows in q's order."""
    N, heads, kv_heads, d = _shapes(q, k, v)
    if k.shape[0] != N:
        raise ValueError("q, k and v must cover the same N tokens")
    if out is None:
        out = torch.empty((N, heads, d), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((N, heads), dtype=torch.float32, device=q.device)
    _state_shapes(lse, lse, out, N, heads, d)
    cu_ptr, ndocs = _docs(cu_seqlens)
    _check(lib().ra_ring_forward_masked(
        _dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(out, "out", torch.float32),
        _dev(lse, "lse", torch.float32), N, int(P), _layout(layout), int(bool(causal)),
        int(window), int(n_valid), cu_ptr, ndocs, d, heads, kv_heads, _qkv_dtype(q),
        _stream(stream)))
    return out, lse


def ra_ring_backward_masked(q, k, v, out, lse, dout, *, P: int, layout="contiguous",
                            causal: bool = False, window: int = 0, n_valid: int = -1,
                            cu_seqlens=None, dq=None, dk=None, dv=None, stream=None):
    """Gradients (dq [N, heads, d], dk, dv [N, kv_heads, d], fp32) of the
    ring forward whose outputs are out, lse, for the upstream gradient dout
    (bf16, like q).  Same layout and mask arguments as the forward."""
    N, heads, kv_heads, d = _shapes(q, k, v)
    if k.shape[0] != N:
        raise ValueError("q, k and v must cover the same N tokens")
    _state_shapes(lse, lse, out, N, heads, d)
    if tuple(dout.shape) != (N, heads, d) or dout.dtype != q.dtype:
        raise ValueError("dout must match q in shape and dtype")
    if dq is None:
        dq = torch.empty((N, heads, d), dtype=torch.float32, device=q.device)
    if dk is None:
        dk = torch.empty((N, kv_heads, d), dtype=torch.float32, device=q.device)
    if dv is None:
        dv = torch.empty((N, kv_heads, d), dtype=torch.float32, device=q.device)
    cu_ptr, ndocs = _docs(cu_seqlens)
    _check(lib().ra_ring_backward_masked(
        _dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(out, "out", torch.float32),
        _dev(lse, "lse", torch.float32), _dev(dout, "dout"), _dev(dq, "dq", torch.float32),
        _dev(dk, "dk", torch.float32), _dev(dv, "dv", torch.float32), N, int(P),
        _layout(layout), int(bool(causal)), int(window), int(n_valid), cu_ptr, ndocs, d, heads,
        kv_heads, _qkv_dtype(q), _stream(stream)))
    return dq, dk, dv


def ra_ring_backward(q, k, v, out, lse, dout, *, P: int, causal: bool, dq=None, dk=None,
                     dv=None, stream=None):
    """ra_ring_backward_masked with the contiguous layout and no extra mask."""
    N, heads, kv_heads, d = _shapes(q, k, v)
    _state_shapes(lse, lse, out, N, heads, d)
    if tuple(dout.shape) != (N, heads, d) or dout.dtype != q.dtype:
        raise ValueError("dout must match q in shape and dtype")
    if dq is None:
        dq = torch.empty((N, heads, d), dtype=torch.float32, device=q.device)
    if dk is None:
        dk = torch.empty((N, kv_heads, d), dtype=torch.float32, device=q.device)
    if dv is None:
        dv = torch.empty((N, kv_heads, d), dtype=torch.float32, device=q.device)
    _check(lib().ra_ring_backward(
        _dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(out, "out", torch.float32),
        _dev(lse, "lse", torch.float32), _dev(dout, "dout"), _dev(dq, "dq", torch.float32),
        _dev(dk, "dk", torch.float32), _dev(dv, "dv", torch.float32), N, int(P),
        int(bool(causal)), d, heads, kv_heads, _qkv_dtype(q), _stream(stream)))
    return dq, dk, dv


def _decode_shapes(q, k, v):
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3 or k.shape != v.shape:
        raise ValueError("q: [n_q, heads, d]; k, v: [n_kv, kv_heads, d]")
    if k.dtype != q.dtype or v.dtype != q.dtype or q.shape[2] != k.shape[2]:
        raise ValueError("q, k, v must share dtype and head dim")
    return q.shape[0], q.shape[1], k.shape[0], k.shape[1], q.shape[2]


def ra_decode_partial(q, k, v, m, l, o, *, q_off: int, kv_off: int = 0, causal: bool = True,
                      window: int = 0, stream=None):
    """Fold one K/V shard into the state (m, l, o) of n_q query rows, in place."""
    n_q, heads, n_kv, kv_heads, d = _decode_shapes(q, k, v)
    _state_shapes(m, l, o, n_q, heads, d)
    _check(lib().ra_decode_partial(
        _dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(m, "m", torch.float32),
        _dev(l, "l", torch.float32), _dev(o, "o", torch.float32), n_q, n_kv, d, heads, kv_heads,
        int(q_off), int(kv_off), int(bool(causal)), int(window), _qkv_dtype(q), _stream(stream)))


def ra_decode_forward(q, k, v, *, P: int, q_off: int | None = None, causal: bool = True,
                      window: int = 0, out=None, lse=None, stream=None):
    """Decode attention of q [n_q, heads, d] against k, v [n_kv, kv_heads, d]
    held as P shards.  q_off defaults to n_kv - n_q (the new tokens are the
    last ones of the history).  Returns (out [n_q, heads, d], lse [n_q, heads])."""
    n_q, heads, n_kv, kv_heads, d = _decode_shapes(q, k, v)
    if q_off is None:
        q_off = n_kv - n_q
    if out is None:
        out = torch.empty((n_q, heads, d), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((n_q, heads), dtype=torch.float32, device=q.device)
    _state_shapes(lse, lse, out, n_q, heads, d)
    kp = _dev(k, "k") if n_kv else 0
    vp = _dev(v, "v") if n_kv else 0
    _check(lib().ra_decode_forward(
        _dev(q, "q"), kp, vp, _dev(out, "out", torch.float32), _dev(lse, "lse", torch.float32),
        n_q, n_kv, int(P), int(q_off), int(bool(causal)), int(window), d, heads, kv_heads,
        _qkv_dtype(q), _stream(stream)))
    return out, lse


def ra_ring_forward_noalloc(q, k, v, *, P: int, causal: bool, out=None, lse=None,
                            stream=None):
    """ra_ring_forward with its l scratch in the library's fixed device array
    (N * heads <= 4,194,304).  It calls no allocator inside the library.
    The output tensors, when not passed in, are still created here by torch.
    Calls that overlap on the GPU share that array and race."""
    N, heads, kv_heads, d = _shapes(q, k, v)
    if k.shape[0] != N:
        raise ValueError("q, k and v must cover the same N tokens")
    if out is None:
        out = torch.empty((N, heads, d), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((N, heads), dtype=torch.float32, device=q.device)
    _state_shapes(lse, lse, out, N, heads, d)
    _check(lib().ra_ring_forward_noalloc(
        _dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(out, "out", torch.float32),
        _dev(lse, "lse", torch.float32), N, int(P), int(bool(causal)), d, heads, kv_heads,
        _qkv_dtype(q), _stream(stream)))
    return out, lse


def ra_ring_forward_host(q, k, v, *, P: int, causal: bool, out=None, lse=None, stream=None):
    """ra_ring_forward on CPU tensors.  Pinned memory makes the copies
    asynchronous DMA.  The call returns when out and lse are on the host."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CPU tensor")
    N, heads, kv_heads, d = _shapes(q, k, v)
    if out is None:
        out = torch.empty((N, heads, d), dtype=torch.float32, pin_memory=q.is_pinned())
    if lse is None:
        lse = torch.empty((N, heads), dtype=torch.float32, pin_memory=q.is_pinned())
    _check(lib().ra_ring_forward_host(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), N, int(P),
        int(bool(causal)), d, heads, kv_heads, _qkv_dtype(q), _stream(stream)))
    return out, lse


def ra_device_status(stream=None):
    _check(lib().ra_device_status(_stream(stream)))


def ra_selftest_wait_timeout(limit_cycles: int, stream=None) -> int:
    return lib().ra_selftest_wait_timeout(int(limit_cycles), _stream(stream))


def ra_cached_memory() -> int:
    """Bytes the library's scratch pool holds on the current device."""
    n = ctypes.c_longlong(0)
    _check(lib().ra_cached_memory(ctypes.addressof(n)))
    return int(n.value)


def ra_release_cached_memory():
    _check(lib().ra_release_cached_memory())


def ra_trace_enable(on: bool = True):
    _check(lib().ra_trace_enable(int(bool(on))))


def ra_trace_reset():
    _check(lib().ra_trace_reset())


def ra_trace_query(kind) -> tuple[int, float]:
    """Returns (launches, total device ms) of one kernel kind since the last reset."""
    k = KERNEL_KINDS[kind] if isinstance(kind, str) else int(kind)
    n = ctypes.c_longlong(0)
    ms = ctypes.c_double(0.0)
    _check(lib().ra_trace_query(k, ctypes.addressof(n), ctypes.addressof(ms)))
    return n.value, ms.value
