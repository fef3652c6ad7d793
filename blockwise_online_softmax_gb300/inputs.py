"""Seeded synthetic inputs, shared by the CUDA path's tests and benchmark and
by the CPU oracle.  This module only draws and lays out random numbers.  It
holds none of the attention arithmetic.

Recipe (the same for every workload)
------------------------------------
* Tensors are Q ``[N, Hq, d]``, K ``[N, Hkv, d]`` and V ``[N, Hkv, d]``,
  token-major with batch 1.  Each gets a tensor id: Q = 0, K = 1, V = 2.
* Each tensor is filled with fp32 standard normals in flat (row-major)
  order, in chunks of 2^22 elements.  Chunk b of tensor t comes from its
  own CPU ``torch.Generator`` seeded with ``(seed << 20) | (t << 16) | b``,
  using ``torch.randn``.  The chunks are independent, so they are drawn in
  parallel, and the result does not depend on the thread count.
* The workload's extra draws are the row picks for scaled or planted keys,
  each a ``randperm`` of the block length.  They come from a second CPU
  generator seeded with ``seed + 1000``, in the order given below.  The
  picks can then be found again without redrawing the big tensors.
* Apply the multiplications in fp32.
* Last, cast to the workload dtype (``.to(torch.bfloat16)`` rounds to
  nearest even).  The oracle and the GPU both read the cast tensors.

The five workloads, with sizes as the pages' long-context discussion
motivates them, are listed in ``WORKLOADS``.  Blocks are contiguous:
virtual rank i holds tokens [i*c, (i+1)*c).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

CHUNK = 1 << 22


def randn_chunked(shape, seed: int, tensor_id: int, threads: int | None = None, *,
                  scale: float = 1.0, dtype=torch.float32) -> torch.Tensor:
    """fp32 standard normals, filled chunk by chunk (see the module recipe).

    With ``scale`` and ``dtype`` each chunk is multiplied in fp32 and cast
    as it is drawn: the same values as ``(randn_chunked(...) * scale)
    .to(dtype)``, without the whole fp32 tensor in memory at once."""
    out = torch.empty(shape, dtype=dtype)
    flat = out.view(-1)
    n = flat.numel()
    nchunks = (n + CHUNK - 1) // CHUNK
    if nchunks >= (1 << 16) or not (0 <= tensor_id < 16) or seed < 0:
        raise ValueError("tensor too large or bad seed / tensor id for the chunked recipe")
    direct = dtype == torch.float32 and scale == 1.0

    def fill(b):
        g = torch.Generator().manual_seed((seed << 20) | (tensor_id << 16) | b)
        part = flat[b * CHUNK:(b + 1) * CHUNK]
        if direct:
            torch.randn(part.shape, generator=g, out=part)
        else:
            x = torch.randn(part.shape, generator=g)
            if scale != 1.0:
                x *= scale
            part.copy_(x)

    if nchunks <= 1:
        for b in range(nchunks):
            fill(b)
    else:
        with ThreadPoolExecutor(max_workers=threads or os.cpu_count() or 1) as ex:
            list(ex.map(fill, range(nchunks)))
    return out


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    heads: int
    kv_heads: int
    d: int
    N: int
    P: int
    dtype: str  # "f32" or "bf16"
    causal: bool
    recipe: str = "iid"  # iid | scaled_keys | half | planted
    notes: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def c(self) -> int:
        return self.N // self.P

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def flops_causal_adjusted(self) -> float:
        """4*d FLOPs per allowed (q, k) pair per query head, with the causal
        pair count taken as N^2/2 (the metric's convention)."""
        pairs = self.N * self.N / (2.0 if self.causal else 1.0)
        return 4.0 * self.d * self.heads * pairs

    def flops_exact(self) -> float:
        """Same convention, exact pair count N(N+1)/2 under causal masking."""
        pairs = self.N * (self.N + 1) / 2.0 if self.causal else float(self.N) * self.N
        return 4.0 * self.d * self.heads * pairs


WORKLOADS = {
    "tiny-exact": Workload(
        "tiny-exact", seed=0, heads=1, kv_heads=1, d=64, N=1024, P=4, dtype="f32",
        causal=False, notes="fp32 exactness case, non-causal"),
    "mha-8k": Workload(
        "mha-8k", seed=1, heads=8, kv_heads=8, d=64, N=8192, P=8, dtype="bf16", causal=True),
    "mha-32k-scaled-keys": Workload(
        "mha-32k-scaled-keys", seed=2, heads=32, kv_heads=32, d=128, N=32768, P=8,
        dtype="bf16", causal=True, recipe="scaled_keys",
        notes="1% of key rows of blocks P/2..P-1 scaled x8",
        extra={"frac": 0.01, "factor": 8.0}),
    "gqa-128k": Workload(
        "gqa-128k", seed=3, heads=32, kv_heads=8, d=128, N=131072, P=16, dtype="bf16",
        causal=True, recipe="half", notes="GQA 32/8, values N(0,1)*0.5"),
    "mha-1m-planted": Workload(
        "mha-1m-planted", seed=4, heads=8, kv_heads=8, d=128, N=1048576, P=64,
        dtype="bf16", causal=True, recipe="planted",
        notes="blocks j = 0 mod 8 carry 16 keys scaled x20",
        extra={"every": 8, "count": 16, "factor": 20.0}),
}


def scaled_key_rows(w: Workload, g: torch.Generator):
    """Row picks for the scaled-keys recipe.  For each block j in [P/2, P)
    (the outer loop) and each KV head (the inner loop), take round(frac*c)
    distinct rows from randperm(c)."""
    c = w.c
    count = int(round(w.extra["frac"] * c))
    picks = []
    for j in range(w.P // 2, w.P):
        for h in range(w.kv_heads):
            idx = torch.randperm(c, generator=g)[:count]
            picks.append((j, h, idx + j * c))
    return picks


def planted_key_rows(w: Workload, g: torch.Generator):
    """Row picks for the planted-keys recipe.  For each block j with
    j % every == 0 (the outer loop) and each KV head (the inner loop), take
    ``count`` distinct rows from randperm(c)."""
    c = w.c
    picks = []
    for j in range(0, w.P, w.extra["every"]):
        for h in range(w.kv_heads):
            idx = torch.randperm(c, generator=g)[: w.extra["count"]]
            picks.append((j, h, idx + j * c))
    return picks


def pick_generator(w: Workload) -> torch.Generator:
    return torch.Generator().manual_seed(w.seed + 1000)


def make_workload(w: Workload | str):
    """Return (q, k, v) CPU tensors of the workload's dtype, token-major.

    Each tensor is drawn, modified and cast before the next one, so only
    one fp32 tensor (K, whose rows the recipe may scale) is alive at a
    time; Q and V are cast chunk by chunk."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    if w.recipe not in ("iid", "scaled_keys", "half", "planted"):
        raise ValueError(f"unknown recipe {w.recipe}")
    dt = w.torch_dtype
    half = w.recipe == "half"

    q = randn_chunked((w.N, w.heads, w.d), w.seed, 0, scale=0.5 if half else 1.0, dtype=dt)
    k = randn_chunked((w.N, w.kv_heads, w.d), w.seed, 1)
    if w.recipe == "scaled_keys":
        for _, h, rows in scaled_key_rows(w, pick_generator(w)):
            k[rows, h, :] *= w.extra["factor"]
    elif w.recipe == "planted":
        for _, h, rows in planted_key_rows(w, pick_generator(w)):
            k[rows, h, :] *= w.extra["factor"]
    elif half:
        k *= 0.5
    k = k.to(dt)
    v = randn_chunked((w.N, w.kv_heads, w.d), w.seed, 2, scale=0.5 if half else 1.0, dtype=dt)
    return q, k, v


def make_random(N: int, heads: int, kv_heads: int, d: int, *, dtype=torch.bfloat16,
                seed: int = 0, scale: float = 1.0):
    """iid N(0,1)*scale case: Q [N,Hq,d], K and V [N,Hkv,d] (module recipe)."""
    q = randn_chunked((N, heads, d), seed, 0, scale=scale, dtype=dtype)
    k = randn_chunked((N, kv_heads, d), seed, 1, scale=scale, dtype=dtype)
    v = randn_chunked((N, kv_heads, d), seed, 2, scale=scale, dtype=dtype)
    return q, k, v


def sample_rows(w: Workload | str, *, random_per_block: int = 16, seed: int = 12345,
                after_planted: int = 8) -> np.ndarray:
    """Query rows to check at full size.  Per block i: local rows {0, 1, 127,
    128, c/2, c-1}, plus ``random_per_block`` seeded random rows.  For the
    scaled or planted recipes, add the ``after_planted`` rows that follow
    the first picked key row of one block per picked block.  Returns sorted
    unique global row indices."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    c = w.c
    rng = np.random.default_rng(seed)
    rows = []
    for i in range(w.P):
        base = i * c
        fixed = [0, 1, 127, 128, c // 2, c - 1]
        rows.extend(base + r for r in fixed if 0 <= r < c)
        rows.extend((base + rng.integers(0, c, size=random_per_block)).tolist())
    if w.recipe in ("scaled_keys", "planted") and after_planted > 0:
        g = pick_generator(w)
        picks = scaled_key_rows(w, g) if w.recipe == "scaled_keys" else planted_key_rows(w, g)
        seen = set()
        for j, h, idx in picks:
            if j in seen:
                continue
            seen.add(j)
            r0 = int(idx.min())
            rows.extend(r for r in range(r0, min(r0 + after_planted, w.N)))
    return np.unique(np.asarray(rows, dtype=np.int64))


# ------------------------------------------------------------------ decode
@dataclass(frozen=True)
class DecodeWorkload:
    """A decode step: n_q new query tokens against a K/V history of n_kv
    tokens (the new ones included, so the queries sit at positions
    n_kv - n_q .. n_kv - 1) held as P shards.  Causal.  Same recipe as
    above: Q, K, V are tensor ids 0, 1, 2 of ``seed``, times ``scale``,
    cast to bf16."""
    name: str
    seed: int
    n_q: int
    heads: int
    kv_heads: int
    d: int
    n_kv: int
    P: int
    scale: float = 1.0
    notes: str = ""

    def kv_bytes(self) -> int:
        """K and V, read once: the algorithmic HBM traffic of the step."""
        return 2 * self.n_kv * self.kv_heads * self.d * 2

    def flops(self) -> float:
        """4*d per allowed (query, key) pair per query head."""
        keys = sum(self.n_kv - self.n_q + i + 1 for i in range(self.n_q))
        return 4.0 * self.d * self.heads * keys


DECODE_WORKLOADS = {
    "decode-1m": DecodeWorkload(
        "decode-1m", seed=5, n_q=1, heads=32, kv_heads=8, d=128, n_kv=1 << 20, P=64,
        notes="one new token after a 1M-token history in 64 shards, GQA 32/8"),
    "decode-1m-q4": DecodeWorkload(
        "decode-1m-q4", seed=6, n_q=4, heads=32, kv_heads=8, d=128, n_kv=1 << 20, P=64,
        notes="four new tokens (a short query block) after a 1M-token history"),
}


def make_decode(w: DecodeWorkload | str):
    """(q [n_q, heads, d], k, v [n_kv, kv_heads, d]) bf16 CPU tensors."""
    if isinstance(w, str):
        w = DECODE_WORKLOADS[w]
    bf = torch.bfloat16
    q = randn_chunked((w.n_q, w.heads, w.d), w.seed, 0, scale=w.scale, dtype=bf)
    k = randn_chunked((w.n_kv, w.kv_heads, w.d), w.seed, 1, scale=w.scale, dtype=bf)
    v = randn_chunked((w.n_kv, w.kv_heads, w.d), w.seed, 2, scale=w.scale, dtype=bf)
    return q, k, v
