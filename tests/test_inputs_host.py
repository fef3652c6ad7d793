"""The synthetic input recipes (no GPU): the five workloads have the sizes
and draws they are stated with, and the scaled and planted keys land on
the rows, blocks and KV heads the recipes name, scaled by exactly their
factor, with every other value left as drawn."""
import numpy as np
import pytest
import torch

from blockwise_online_softmax_gb300 import inputs


def test_named_workloads():
    w = inputs.WORKLOADS
    assert [(x.heads, x.kv_heads, x.d, x.N, x.P, x.dtype, x.causal)
            for x in (w["tiny-exact"], w["mha-8k"], w["mha-32k-scaled-keys"], w["gqa-128k"],
                      w["mha-1m-planted"])] == [
        (1, 1, 64, 1024, 4, "f32", False),
        (8, 8, 64, 8192, 8, "bf16", True),
        (32, 32, 128, 32768, 8, "bf16", True),
        (32, 8, 128, 131072, 16, "bf16", True),
        (8, 8, 128, 1048576, 64, "bf16", True),
    ]
    assert w["gqa-128k"].flops_causal_adjusted() == 4 * 32 * 128 * 131072 ** 2 / 2


def test_scaled_key_picks_of_the_32k_workload():
    """1% of each (block, KV head)'s keys, blocks P/2 .. P-1 only."""
    w = inputs.WORKLOADS["mha-32k-scaled-keys"]
    picks = inputs.scaled_key_rows(w, inputs.pick_generator(w))
    assert len(picks) == (w.P - w.P // 2) * w.kv_heads
    assert {(j, h) for j, h, _ in picks} == {(j, h) for j in range(w.P // 2, w.P)
                                             for h in range(w.kv_heads)}
    for j, h, rows in picks:
        r = rows.numpy()
        assert len(r) == round(0.01 * w.c) == 41
        assert len(set(r.tolist())) == len(r)
        assert (r >= j * w.c).all() and (r < (j + 1) * w.c).all()


def test_planted_key_picks_of_the_1m_workload():
    """16 keys of each KV head in every eighth block (j = 0, 8, ..., 56)."""
    w = inputs.WORKLOADS["mha-1m-planted"]
    picks = inputs.planted_key_rows(w, inputs.pick_generator(w))
    assert sorted({j for j, _, _ in picks}) == list(range(0, 64, 8))
    assert len(picks) == 8 * w.kv_heads
    for j, h, rows in picks:
        r = rows.numpy()
        assert len(r) == 16 and len(set(r.tolist())) == 16
        assert (r >= j * w.c).all() and (r < (j + 1) * w.c).all()


@pytest.mark.parametrize("recipe, extra", [
    ("scaled_keys", {"frac": 0.01, "factor": 8.0}),
    ("planted", {"every": 2, "count": 7, "factor": 20.0}),
])
def test_recipe_scales_exactly_the_picked_keys(recipe, extra):
    """A small workload under the same recipe: K rows at the picks are the
    drawn values times the factor (rounded to bf16 once, after the
    product); every other K value, and all of Q and V, are the drawn values
    rounded to bf16."""
    w = inputs.Workload("t", seed=11, heads=4, kv_heads=2, d=64, N=4096, P=8, dtype="bf16",
                        causal=True, recipe=recipe, extra=extra)
    q, k, v = inputs.make_workload(w)
    raw_q = inputs.randn_chunked((w.N, w.heads, w.d), w.seed, 0)
    raw_k = inputs.randn_chunked((w.N, w.kv_heads, w.d), w.seed, 1)
    raw_v = inputs.randn_chunked((w.N, w.kv_heads, w.d), w.seed, 2)
    assert torch.equal(q, raw_q.to(torch.bfloat16)) and torch.equal(v, raw_v.to(torch.bfloat16))
    picks = (inputs.scaled_key_rows if recipe == "scaled_keys" else
             inputs.planted_key_rows)(w, inputs.pick_generator(w))
    picked = np.zeros((w.N, w.kv_heads), dtype=bool)
    for _, h, rows in picks:
        picked[rows.numpy(), h] = True
    assert picked.sum() == sum(len(r) for _, _, r in picks) > 0
    expect = raw_k.clone()
    mask = torch.from_numpy(picked)
    expect[mask] = raw_k[mask] * extra["factor"]
    assert torch.equal(k, expect.to(torch.bfloat16))
    # the picked rows really changed
    assert not torch.equal(k[mask], raw_k[mask].to(torch.bfloat16))


def test_half_recipe_halves_every_tensor():
    w = inputs.Workload("h", seed=5, heads=4, kv_heads=2, d=64, N=1024, P=4, dtype="bf16",
                        causal=True, recipe="half")
    q, k, v = inputs.make_workload(w)
    for t, (shape, tid) in zip((q, k, v), (((w.N, w.heads, w.d), 0), ((w.N, w.kv_heads, w.d), 1),
                                           ((w.N, w.kv_heads, w.d), 2))):
        assert torch.equal(t, (inputs.randn_chunked(shape, w.seed, tid) * 0.5).to(torch.bfloat16))


def test_draws_do_not_depend_on_the_thread_count():
    a = inputs.randn_chunked((3 * inputs.CHUNK // 64 + 5, 64), 9, 1, threads=1)
    b = inputs.randn_chunked((3 * inputs.CHUNK // 64 + 5, 64), 9, 1, threads=4)
    assert torch.equal(a, b)
    # chunk 0 is torch.randn from its own generator
    g = torch.Generator().manual_seed((9 << 20) | (1 << 16) | 0)
    assert torch.equal(a.reshape(-1)[:inputs.CHUNK], torch.randn(inputs.CHUNK, generator=g))


def test_chunkwise_cast_equals_the_whole_tensor_cast():
    # Scale and cast per chunk (no whole fp32 tensor) give the recipe's
    # values: the fp32 draw, times the scale in fp32, then the cast.
    shape = (2 * inputs.CHUNK // 64 + 7, 64)
    whole = inputs.randn_chunked(shape, 4, 2)
    for scale, dtype in ((1.0, torch.bfloat16), (0.5, torch.bfloat16), (3.0, torch.float32)):
        got = inputs.randn_chunked(shape, 4, 2, scale=scale, dtype=dtype)
        assert got.dtype == dtype
        assert torch.equal(got, (whole * scale).to(dtype))
    q, k, v = inputs.make_random(300, 3, 1, 64, seed=6, scale=2.0)
    assert torch.equal(q, (inputs.randn_chunked((300, 3, 64), 6, 0) * 2.0).to(torch.bfloat16))
    assert torch.equal(v, (inputs.randn_chunked((300, 1, 64), 6, 2) * 2.0).to(torch.bfloat16))
