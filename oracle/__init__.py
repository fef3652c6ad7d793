"""CPU oracle for blockwise online-softmax attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library and its Python
binding never import it, and nothing here imports them.  The two sides share
only the seeded input generator, which holds none of the method's arithmetic.

Contents
--------
* ``attention.c`` is the dense fp64 definition (see its header), built with
  gcc into ``liboracle.so`` and loaded through ctypes.  ``partial_state`` and
  ``attention`` below wrap it.
* ``online.py`` restates, in fp64 numpy, the pages' own blockwise recurrence,
  merge and finalize.  The invariant tests use it, and it serves as the
  oracle for the state-level calls (block update, merge, finalize).

Pins
----
``tests/test_oracle.py`` pins every function here to facts other than the
code itself: the worked example the pages print, special cases that reduce
to library routines, closed forms, brute force and invariants.  No function
is unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32 = 0
BF16 = 1


def build_library(force: bool = False) -> str:
    """Compile ``attention.c`` with gcc into ``liboracle.so`` next to it."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build_library()
            lib = ctypes.CDLL(_LIB_PATH)
            f = lib.oracle_partial_state_masked
            P = ctypes.c_void_p
            LL = ctypes.c_longlong
            f.argtypes = [P, P, P, ctypes.c_int, LL, LL, ctypes.c_int, ctypes.c_int,
                          ctypes.c_int, ctypes.c_double, ctypes.c_int, LL, P, P, P, P, P, LL,
                          P, P, P, ctypes.c_int]
            f.restype = ctypes.c_int
            gq = lib.oracle_grad_q
            gq.argtypes = [P, P, P, P, ctypes.c_int, LL, LL, ctypes.c_int, ctypes.c_int,
                           ctypes.c_int, ctypes.c_double, ctypes.c_int, LL, P, P, P, P, P, LL,
                           P, P, P, P, P, ctypes.c_int]
            gq.restype = ctypes.c_int
            gkv = lib.oracle_grad_kv
            gkv.argtypes = [P, P, P, P, ctypes.c_int, LL, LL, ctypes.c_int, ctypes.c_int,
                            ctypes.c_int, ctypes.c_double, ctypes.c_int, LL, P, P, P, P, P, P,
                            P, LL, P, P, P, P, P, ctypes.c_int]
            gkv.restype = ctypes.c_int
            lib.oracle_abi_version.restype = ctypes.c_int
            if lib.oracle_abi_version() != 4:
                raise RuntimeError("liboracle.so is stale; rebuild it")
            _lib = lib
    return _lib


def _as_input(x):
    """Accept a numpy float32 array, a numpy uint16 array of bf16 bit
    patterns, or a CPU torch tensor (float32 or bfloat16)."""
    if not isinstance(x, np.ndarray):
        import torch  # local import: only needed for tensor inputs

        t = x.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            x = t.view(torch.int16).numpy().view(np.uint16)
        elif t.dtype == torch.float32:
            x = t.numpy()
        else:
            raise TypeError(f"oracle takes float32 or bfloat16, got {t.dtype}")
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, F32
    if x.dtype == np.uint16:
        return x, BF16
    raise TypeError(f"oracle takes float32 or bf16 bit patterns (uint16), got {x.dtype}")


def partial_state(q, k, v, *, causal: bool, q_pos=None, k_pos=None, rows=None,
                  scale: float | None = None, threads: int | None = None, window: int = 0,
                  q_doc=None, k_doc=None):
    """Partial online-softmax state of query rows against a key set, in fp64.

    q: [nq, hq, d]; k, v: [nk, hkv, d] (token-major).  ``q_pos``/``k_pos``
    are global token positions (default: the index).  ``rows`` selects the
    query rows (default: all).  ``window`` > 0 allows only keys with
    |q_pos - k_pos| < window.  ``q_doc``/``k_doc`` are per-row document ids
    (both or neither); a key is allowed only within its query's document,
    and id -1 marks a padding row that sees and is seen by nothing.
    Returns ``(m, l, o)`` of shapes ``[nrows, hq]``, ``[nrows, hq]`` and
    ``[nrows, hq, d]``, as defined in ``attention.c``.  The default scale is
    1/sqrt(d).
    """
    qa, dt = _as_input(q)
    ka, dk = _as_input(k)
    va, dv = _as_input(v)
    if not (dt == dk == dv):
        raise TypeError("q, k and v must share one dtype")
    if qa.ndim != 3 or ka.ndim != 3 or va.ndim != 3:
        raise ValueError("q, k, v must be 3-D token-major arrays")
    nq, hq, d = qa.shape
    nk, hkv, dk_ = ka.shape
    if va.shape != ka.shape or dk_ != d:
        raise ValueError("shape mismatch between q, k and v")
    if rows is None:
        rows = np.arange(nq, dtype=np.int64)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    qp = None if q_pos is None else np.ascontiguousarray(np.asarray(q_pos, dtype=np.int64))
    kp = None if k_pos is None else np.ascontiguousarray(np.asarray(k_pos, dtype=np.int64))
    if qp is not None and qp.shape != (nq,):
        raise ValueError("q_pos must have one entry per query row")
    if kp is not None and kp.shape != (nk,):
        raise ValueError("k_pos must have one entry per key")
    if (q_doc is None) != (k_doc is None):
        raise ValueError("give both q_doc and k_doc, or neither")
    qd = None if q_doc is None else np.ascontiguousarray(np.asarray(q_doc, dtype=np.int64))
    kd = None if k_doc is None else np.ascontiguousarray(np.asarray(k_doc, dtype=np.int64))
    if qd is not None and (qd.shape != (nq,) or kd.shape != (nk,)):
        raise ValueError("q_doc / k_doc must have one entry per row")
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    if threads is None:
        threads = os.cpu_count() or 1
    nr = rows.shape[0]
    m = np.empty((nr, hq), dtype=np.float64)
    l = np.empty((nr, hq), dtype=np.float64)
    o = np.empty((nr, hq, d), dtype=np.float64)

    def ptr(a):
        return None if a is None else a.ctypes.data_as(ctypes.c_void_p)

    rc = _load().oracle_partial_state_masked(
        ptr(qa), ptr(ka), ptr(va), dt, nq, nk, hq, hkv, d, float(scale), int(bool(causal)),
        int(window), ptr(qp), ptr(kp), ptr(qd), ptr(kd), ptr(rows), nr, ptr(m), ptr(l), ptr(o),
        int(threads))
    if rc != 0:
        raise ValueError(f"oracle_partial_state failed with code {rc}")
    return m, l, o


def attention(q, k, v, *, causal: bool, q_pos=None, k_pos=None, rows=None,
              scale: float | None = None, threads: int | None = None, window: int = 0,
              q_doc=None, k_doc=None):
    """Dense attention O = softmax(q k^T * scale) v and its row log-sum-exp.

    Returns ``(O [nrows, hq, d], LSE [nrows, hq])`` in fp64.  A row with no
    allowed key gets O = 0 and LSE = -inf.
    """
    m, l, o = partial_state(q, k, v, causal=causal, q_pos=q_pos, k_pos=k_pos, rows=rows,
                            scale=scale, threads=threads, window=window, q_doc=q_doc,
                            k_doc=k_doc)
    with np.errstate(divide="ignore", invalid="ignore"):
        out = np.where(l[..., None] > 0, o / np.where(l > 0, l, 1.0)[..., None], 0.0)
        lse = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return out, lse


# ------------------------------------------------------------------ gradients
def _grad_inputs(q, k, v, dout, q_pos, k_pos, q_doc, k_doc, scale):
    qa, dt = _as_input(q)
    ka, dk_ = _as_input(k)
    va, dv_ = _as_input(v)
    ga, dg = _as_input(dout)
    if not (dt == dk_ == dv_ == dg):
        raise TypeError("q, k, v and dout must share one dtype")
    nq, hq, d = qa.shape
    nk, hkv, _ = ka.shape
    if ga.shape != qa.shape or va.shape != ka.shape or ka.shape[2] != d:
        raise ValueError("shape mismatch between q, k, v and dout")

    def arr(x, n):
        if x is None:
            return None
        a = np.ascontiguousarray(np.asarray(x, dtype=np.int64))
        if a.shape != (n,):
            raise ValueError("positions and document ids need one entry per row")
        return a

    qp, kp = arr(q_pos, nq), arr(k_pos, nk)
    if (q_doc is None) != (k_doc is None):
        raise ValueError("give both q_doc and k_doc, or neither")
    qd, kd = arr(q_doc, nq), arr(k_doc, nk)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    return qa, ka, va, ga, dt, nq, nk, hq, hkv, d, qp, kp, qd, kd, float(scale)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def grad_q(q, k, v, dout, *, causal: bool, rows=None, q_pos=None, k_pos=None, window: int = 0,
           q_doc=None, k_doc=None, scale: float | None = None, threads: int | None = None,
           absolute: bool = False):
    """dQ, LSE and D = sum_t P dP of the listed query rows (default: all),
    for the loss sum(dout * O).  Shapes [nrows, hq, d], [nrows, hq],
    [nrows, hq]; fp64.  The definition is in ``attention.c``.

    With ``absolute=True`` two more arrays follow: the absolute-term sums
    of dQ ([nrows, hq, d]) and of D ([nrows, hq]), the error scales defined
    in ``attention.c`` (each sum with every term replaced by its absolute
    value)."""
    qa, ka, va, ga, dt, nq, nk, hq, hkv, d, qp, kp, qd, kd, sc = _grad_inputs(
        q, k, v, dout, q_pos, k_pos, q_doc, k_doc, scale)
    rows = np.arange(nq, dtype=np.int64) if rows is None else np.ascontiguousarray(
        np.asarray(rows, dtype=np.int64))
    nr = rows.shape[0]
    dq = np.empty((nr, hq, d))
    lse = np.empty((nr, hq))
    dvec = np.empty((nr, hq))
    dq_abs = np.empty((nr, hq, d)) if absolute else None
    d_abs = np.empty((nr, hq)) if absolute else None
    rc = _load().oracle_grad_q(_ptr(qa), _ptr(ka), _ptr(va), _ptr(ga), dt, nq, nk, hq, hkv, d,
                               sc, int(bool(causal)), int(window), _ptr(qp), _ptr(kp), _ptr(qd),
                               _ptr(kd), _ptr(rows), nr, _ptr(dq), _ptr(lse), _ptr(dvec),
                               _ptr(dq_abs), _ptr(d_abs), int(threads or os.cpu_count() or 1))
    if rc != 0:
        raise ValueError(f"oracle_grad_q failed with code {rc}")
    if absolute:
        return dq, lse, dvec, dq_abs, d_abs
    return dq, lse, dvec


def grad_kv(q, k, v, dout, lse_all, d_all, *, causal: bool, keys=None, q_pos=None, k_pos=None,
            window: int = 0, q_doc=None, k_doc=None, scale: float | None = None,
            threads: int | None = None, d_abs_all=None):
    """dK and dV of the listed keys (default: all), [nkeys, hkv, d] fp64,
    given LSE and D of every query row (from ``grad_q`` over all rows).

    Given ``d_abs_all`` (the absolute-term sums of D of every query row,
    from ``grad_q(absolute=True)``), two more arrays follow: the
    absolute-term sums of dK and of dV."""
    qa, ka, va, ga, dt, nq, nk, hq, hkv, d, qp, kp, qd, kd, sc = _grad_inputs(
        q, k, v, dout, q_pos, k_pos, q_doc, k_doc, scale)
    lse_all = np.ascontiguousarray(np.asarray(lse_all, dtype=np.float64))
    d_all = np.ascontiguousarray(np.asarray(d_all, dtype=np.float64))
    if lse_all.shape != (nq, hq) or d_all.shape != (nq, hq):
        raise ValueError("lse_all and d_all must be [nq, hq]")
    keys = np.arange(nk, dtype=np.int64) if keys is None else np.ascontiguousarray(
        np.asarray(keys, dtype=np.int64))
    nkk = keys.shape[0]
    dk = np.empty((nkk, hkv, d))
    dv = np.empty((nkk, hkv, d))
    absolute = d_abs_all is not None
    if absolute:
        d_abs_all = np.ascontiguousarray(np.asarray(d_abs_all, dtype=np.float64))
        if d_abs_all.shape != (nq, hq):
            raise ValueError("d_abs_all must be [nq, hq]")
    dk_abs = np.empty((nkk, hkv, d)) if absolute else None
    dv_abs = np.empty((nkk, hkv, d)) if absolute else None
    rc = _load().oracle_grad_kv(_ptr(qa), _ptr(ka), _ptr(va), _ptr(ga), dt, nq, nk, hq, hkv, d,
                                sc, int(bool(causal)), int(window), _ptr(qp), _ptr(kp), _ptr(qd),
                                _ptr(kd), _ptr(lse_all), _ptr(d_all), _ptr(keys), nkk, _ptr(dk),
                                _ptr(dv), _ptr(d_abs_all), _ptr(dk_abs), _ptr(dv_abs),
                                int(threads or os.cpu_count() or 1))
    if rc != 0:
        raise ValueError(f"oracle_grad_kv failed with code {rc}")
    if absolute:
        return dk, dv, dk_abs, dv_abs
    return dk, dv


def backward(q, k, v, dout, *, causal: bool, **kw):
    """All gradients of sum(dout * attention(q, k, v)): (dq, dk, dv, lse)."""
    dq, lse, dvec = grad_q(q, k, v, dout, causal=causal, **kw)
    dk, dv = grad_kv(q, k, v, dout, lse, dvec, causal=causal, **kw)
    return dq, dk, dv, lse


def backward_with_scales(q, k, v, dout, *, causal: bool, **kw):
    """The gradients and their absolute-term sums (the error scales of
    ``attention.c``): ((dq, dk, dv), (dq_abs, dk_abs, dv_abs), lse)."""
    dq, lse, dvec, dq_abs, d_abs = grad_q(q, k, v, dout, causal=causal, absolute=True, **kw)
    dk, dv, dk_abs, dv_abs = grad_kv(q, k, v, dout, lse, dvec, causal=causal, d_abs_all=d_abs,
                                     **kw)
    return (dq, dk, dv), (dq_abs, dk_abs, dv_abs), lse
