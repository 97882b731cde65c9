"""Host-side arithmetic of bench.py (no GPU): the FLOP and byte counts it
reports against, and the routing statistics of its JSON line."""
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from token_dispatch_grouped_gb300 import inputs as I  # noqa: E402


def test_flop_count_is_the_layer_formula():
    s = I.WORKLOADS["mixtral"]
    TK = s.T * s.K
    # 18 TK d h for the expert GEMMs (fwd 6, bwd 12) + 6 T d E for the router
    assert bench.flops_per_step(s) == 18 * TK * s.d * s.h + 6 * s.T * s.d * s.E
    ng = I.WORKLOADS["moeblaze_conf7"]
    assert bench.flops_per_step(ng) == 12 * ng.T * ng.K * ng.d * ng.h + 6 * ng.T * ng.d * ng.E


def test_memory_kernel_bytes_and_routed_buffer():
    s = I.WORKLOADS["mixtral"]
    b = bench.memory_kernel_bytes(s)
    TK, d = s.T * s.K, s.d
    assert b["combine"][1] == TK * d * 2 + TK * 8 + s.T * d * 2
    assert b["router_dwg"][1] == s.T * d * 2 + TK * 12 + s.E * d * 4
    assert "router_dwg_mma" in b["router_dwg"][0] and "router_dwg" in b["router_dwg"][0]
    # the routed [T*K, d] bf16 buffer the layer never allocates: 64 MiB here
    assert TK * d * 2 == 64 * 2**20


def test_routing_stats_counts_partial_tiles():
    # Mixtral-like: six experts just above 1024 rows get a fifth, nearly empty tile
    counts = torch.tensor([1030, 1025, 1038, 1026, 1027, 1029, 1001, 1016], dtype=torch.int32)
    st = bench.routing_stats(counts)
    assert st["min_rows"] == 1001 and st["max_rows"] == 1038 and st["empty_experts"] == 0
    assert st["m_tiles_256"] == 6 * 5 + 2 * 4
    assert st["m_tiles_256_packed"] == (int(counts.sum()) + 255) // 256
    # pair tiles for the 1024 (or 768) rows of whole tiles, a 128-row single-CTA tile
    # for each remainder of 1..14 rows, a 256-row tile for the 233- and 248-row ones
    assert st["mma_rows_issued"] == 6 * (1024 + 128) + 2 * 1024
    assert st["mma_rows_pairs_only"] == 38 * 256 and st["routed_rows"] == int(counts.sum())
    z = bench.routing_stats(torch.tensor([0, 512, 0, 257], dtype=torch.int32))
    assert z["empty_experts"] == 2 and z["m_tiles_256"] == 2 + 2


def test_peak_rule_burst_for_short_or_full_clock_regions():
    peaks = {"bf16": 1932.0, "bf16_sus": 1741.0}
    full = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0}
    capped = {"sm_mhz": 1650.0, "sm_max_mhz": 2070.0}
    assert bench.choose_bf16_peak(peaks, 130.0, capped) == (1932.0, "burst")     # short region
    assert bench.choose_bf16_peak(peaks, 5000.0, full) == (1932.0, "burst")      # at max clock
    assert bench.choose_bf16_peak(peaks, 5000.0, capped) == (1741.0, "sustained")
    assert bench.choose_bf16_peak(peaks, 5000.0, {"sm_mhz": None, "sm_max_mhz": None}) == \
        (1741.0, "sustained")
