"""The synthetic workloads keep the shapes the pages print.

tests/golden/granularity_table.txt holds the granularity and activated-share
table of the SonicMoE page (section "MoE 的两个核心趋势").  The
DeepSeek-V3-style workload must reproduce that row (d/n = 3.50, k/E = 3.13 %)
and the Mixtral-style workload the 2-of-8 routing of the Mixtral family (25 %);
its d and n are the 8x7B member's, so its d/n is not the 8x22B row's.  The
fine-grained 7B workload runs at the microbatch the page's kernel table quotes
(section "Kernel 级性能": microbatch 32768).
"""
import os

from mixture_experts_layer_93_b300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "granularity_table.txt")


def _table():
    rows = {}
    with open(GOLDEN, encoding="utf-8") as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            model, share, gran = (c.strip() for c in line.split("|"))
            rows[model] = (float(share), float(gran))
    return rows


def test_table_parses():
    rows = _table()
    assert set(rows) == {"Mixtral 8x22B", "DBRX", "DeepSeek-V3", "Kimi K2", "gpt-oss-120b"}


def test_dsv3_workload_matches_printed_row():
    share, gran = _table()["DeepSeek-V3"]
    cfg = I.CONFIGS["dsv3"]
    # printed to two decimals: within half a unit of the last digit
    assert abs(cfg.d / cfg.n - gran) <= 0.005 + 1e-12
    assert abs(100.0 * cfg.k / cfg.E - share) <= 0.005 + 1e-12


def test_mixtral_workload_routing_share():
    share, _ = _table()["Mixtral 8x22B"]
    cfg = I.CONFIGS["mixtral"]
    assert abs(100.0 * cfg.k / cfg.E - share) <= 0.05 + 1e-12


def test_b7_microbatch():
    assert I.CONFIGS["b7"].T == 32768
