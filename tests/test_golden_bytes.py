"""The byte accounting behind the bench's roofline against numbers the pages print."""
import json
from pathlib import Path

from quantized_matmul_speculative_gb300 import workloads

GOLDEN = json.loads((Path(__file__).parent / "golden" / "page_byte_counts.json").read_text())


def test_metadata_share_matches_pages():
    g = GOLDEN["metadata_share"]
    N, K = 4096, 8192
    shares = {}
    for gs, printed in g["printed_percent"].items():
        gs = int(gs)
        share = 100.0 * workloads.meta_bytes(N, K, gs) / workloads.call_bytes(N, K, g["bits"], gs)
        assert abs(share - printed) <= g["printed_precision_percent"][str(gs)], (gs, share)
        shares[gs] = share
    assert abs(shares[32] / shares[128] - g["g32_over_g128_printed"]) <= g["g32_over_g128_precision"]


def test_microbench_roofline_time_matches_pages():
    r = GOLDEN["microbench_roofline"]
    nbytes = workloads.call_bytes(r["N"], r["K"], r["bits"], r["group_size"])
    ms = nbytes / (r["roofline_gbs"] * 1e9) * 1e3
    assert abs(ms - r["printed_ms"]) <= r["printed_precision_ms"], ms
