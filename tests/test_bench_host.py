"""Host-side pieces of bench.py that need no GPU: the clock-record summary that decides
whether a timed run counts (throttle reasons, median SM clock) and the peak table."""
import bench


def test_clock_rows_median_and_no_reason():
    text = "\n".join(f"0, {mhz}, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active"
                     for mhz in (2070, 2055, 2070))
    c = bench.parse_clocks(text)
    assert c == dict(sm_mhz=2070.0, sm_max_mhz=2070.0, reasons=[], samples=3)


def test_clock_rows_report_every_reason_seen():
    text = ("0, 1980, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active\n"
            "0, 1800, 2070, 1400.0, 0x8, Active, Not Active, Not Active, Not Active\n"
            "0, 2070, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active\n")
    c = bench.parse_clocks(text)
    assert c["reasons"] == ["hw_slowdown", "sw_power_cap"] and c["sm_mhz"] == 1980.0 and c["samples"] == 3


def test_clock_rows_skip_unreadable_lines():
    c = bench.parse_clocks("0, [N/A], 2070, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active\n\n")
    assert c["samples"] == 0 and c["sm_mhz"] is None


def test_peaks_have_every_denominator():
    p = bench.load_peaks()
    assert p["src"] in ("measured", "fallback") and p["hbm"] > 0 and p["tf"] > 0 and p["tf_sus"] > 0
