"""The byte models behind the benchmark's roofline figures (no GPU): the algorithmic bytes
of a decode step and of a prefill chunk, checked against their closed forms on the bench
workload and on small hand-counted cases."""
import torch

import bench


def test_decode_bytes_of_the_bench_workload():
    """32 832 tokens (2 052 pages of 16), 32 MHA heads, 128 full pages kept per head: boxes
    2052 * 32 * 512 B, kept K/V 32 * 128 * 16 tokens * 512 B, q and out 32 * 256 B each,
    lse 32 * 4 B."""
    L = 32832
    tokens = 32 * 128 * 16
    want = 2052 * 32 * 512 + tokens * 512 + 2 * 32 * 256 + 32 * 4
    assert bench.decode_bytes([L], tokens, 1, 32, 32) == want == 67_190_912


def test_selected_tokens_count_a_partial_last_page():
    idx = torch.tensor([[[0, 2, -1]]], dtype=torch.int32)
    cnt = torch.tensor([[2]], dtype=torch.int32)
    assert bench.selected_tokens(idx, cnt, [40], page=16) == 16 + 8


def test_prefill_bytes_closed_forms():
    # a 32K prompt into an empty cache: K and V read and written once, 2 048 fresh boxes
    rows = 2 * 32768 * 32 * 256
    assert bench.prefill_bytes(1, 32768, 32, 16, [0]) == 2 * rows + 2048 * 32 * 512
    # 20 tokens from length 5: pages 0 and 1 are touched, page 0's box is read too
    assert bench.prefill_bytes(1, 20, 4, 16, [5]) == 2 * (2 * 20 * 4 * 256) + 2 * 4 * 512 + 4 * 512
    # page-aligned start: no box is read
    assert bench.prefill_bytes(2, 16, 1, 16, [16, 32]) == 2 * (2 * 2 * 16 * 256) + 2 * 512


def test_clock_summary_reads_throttle_reasons_and_busy_clock():
    """nvidia-smi lines (csv, no units): the median SM clock over samples under load (above
    half the maximum), the maximum, and every throttle reason seen active."""
    c = bench.ClockSampler(0)
    c.lines = [
        "345, 2070, 150.2, 0x0000000000000001, Not Active, Not Active, Not Active, Not Active",
        "2070, 2070, 900.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "1980, 2070, 1350.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "2010, 2070, 1200.0, 0x0000000000000000, Active, Not Active, Not Active, Not Active",
        "garbage line",
    ]
    s = c.summary()
    assert s["sm_max_mhz"] == 2070.0
    assert s["sm_mhz"] == 2010.0             # median of 2070, 1980, 2010 (345 is idle)
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert s["samples"] == 4
    c.lines = []
    assert c.summary() is None
