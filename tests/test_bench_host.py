"""Host-side checks of bench.py's bookkeeping that need no GPU: the DRAM
traffic records are reported only for the kernel source they were taken
on, the clock window padding, and the parity check's row choice."""
import numpy as np
import pytest
import torch

import bench
import oracle
from blockwise_online_softmax_gb300 import inputs


@pytest.mark.parametrize("workload, profile, files, lo, hi", [
    # fused forward: at least Q, K, V read once (1.61 GB) and O, LSE written
    # once (2.16 GB); K/V re-reads that miss L2 add to the reads
    ("gqa-128k", "ring_fused_bf16_traffic.md", bench.FORWARD_SOURCES, 3.7e9, 2e10),
    # decode: K and V read once (4.295 GB) plus the small partial states
    ("decode-1m", "decode_tc_traffic.md", bench.DECODE_SOURCES, 4.29e9, 4.31e9),
])
def test_traffic_records_are_plausible(workload, profile, files, lo, hi):
    """A record taken on the current kernel sources is reported and lies
    in its plausible range; a stale one (the kernel changed since its
    capture) is not reported at all, which is what bench.py relies on."""
    val = bench.recorded_traffic(workload, profile, files)
    if val is None:
        pytest.skip(f"{profile} was captured on other kernel sources; recapture it")
    assert lo < val < hi


def test_traffic_record_needs_its_own_digest():
    # A record checked against another kernel's sources does not count, and
    # a workload the record does not list gives nothing.
    assert bench.recorded_traffic("gqa-128k", "ring_fused_bf16_traffic.md",
                                  bench.DECODE_SOURCES) is None
    assert bench.recorded_traffic("decode-1m", "decode_tc_traffic.md") is None
    assert bench.recorded_traffic("mha-8k", "ring_fused_bf16_traffic.md") is None
    assert bench.recorded_traffic("gqa-128k", "no_such_profile.md") is None


def test_digests_differ_per_kernel():
    assert bench.kernel_digest() != bench.kernel_digest(bench.DECODE_SOURCES)
    assert len(bench.kernel_digest()) == 16


def test_clock_padding_only_for_short_regions():
    assert bench.pad_seconds(0.1, 5) == bench.CLOCK_PAD_S  # 0.5 s region
    assert bench.pad_seconds(0.3, 5) == 0.0                # 1.5 s region
    clk = bench.note_window({"sm_mhz": 2000.0}, 0.5)
    assert "untimed steps" in clk["window"]
    assert bench.note_window({"sm_mhz": 2000.0}, 0.0)["window"] == "timed region"


def test_parity_check_takes_every_row_of_a_small_workload():
    """On the fp32 exactness workload the check covers all 1024 rows, and
    it catches one wrong output row that sampling could miss."""
    w = inputs.WORKLOADS["tiny-exact"]
    q, k, v = inputs.make_workload(w)
    ref_o, ref_l = oracle.attention(q, k, v, causal=w.causal)
    out = torch.from_numpy(ref_o).float()
    lse = torch.from_numpy(ref_l).float()
    good = bench.parity_check(w, q, k, v, out, lse)
    assert good["all_rows"] and good["rows"] == w.N and good["pass"]
    bad = out.clone()
    bad[777, 0, 5] += 1e-3  # row 777 is none of the fixed rows {0, 1, 127, 128, c/2, c-1} of a block
    res = bench.parity_check(w, q, k, v, bad, lse)
    assert not res["pass"] and res["max_abs_o"] == pytest.approx(1e-3, rel=1e-2)


def test_both_arms_describe_the_workload_identically():
    # The reference arm and the GPU arm print the same config dict, key for
    # key, so a reader (or a script) can tell they ran the same workload.
    for name, w in inputs.WORKLOADS.items():
        a, b = bench.forward_config(w, 1), bench.forward_config(w, 1)
        assert a == b and a["workload"] == name
        for key in ("N", "P", "c", "heads", "kv_heads", "d", "causal", "recipe", "seed"):
            assert key in a


def test_l2_flush_only_for_workloads_that_fit_in_l2():
    W = inputs.WORKLOADS
    assert bench.needs_l2_flush(W["tiny-exact"]) and bench.needs_l2_flush(W["mha-8k"])
    for name in ("mha-32k-scaled-keys", "gqa-128k", "mha-1m-planted"):
        assert not bench.needs_l2_flush(W[name])
        assert bench.footprint_bytes(W[name]) > 2 * bench.L2_BYTES
    assert bench.L2_FLUSH_BYTES > 2 * bench.L2_BYTES
    assert "written between timed steps" in bench.forward_config(W["mha-8k"], 1)["l2"]


def test_state_kernel_bytes():
    # m and l (8 bytes) plus d fp32 values per state (row, head).
    b = bench.state_bytes(128)
    assert b == {"state_init": 520, "merge": 3 * 520, "finalize": 520 + 516}
    assert bench.state_bytes(64)["merge"] == 3 * 264


def test_head_slice_is_the_same_problem_on_fewer_heads():
    w = bench.head_slice(inputs.WORKLOADS["mha-8k"], 2)
    assert (w.heads, w.kv_heads, w.N, w.P) == (2, 2, 8192, 8)
    q, k, v = bench.workload_inputs(w)
    fq, fk, fv = inputs.make_workload(inputs.WORKLOADS["mha-8k"])
    assert torch.equal(q, fq[:, :2]) and torch.equal(k, fk[:, :2]) and torch.equal(v, fv[:, :2])
    g = bench.head_slice(inputs.WORKLOADS["gqa-128k"], 8)
    assert (g.heads, g.kv_heads) == (8, 2)
    with pytest.raises(SystemExit):
        bench.head_slice(inputs.WORKLOADS["gqa-128k"], 6)
