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


def test_algorithmic_bytes_per_unit_follow_from_the_tensors():
    """Per (token x value head) unit at D=128: bf16 q, k (one key head per two value heads), v, o,
    do; fp32 g, beta; fp32 dq, dk (per key head), dv, dg, dbeta. The roofline's byte counts are
    these sums, not measured traffic."""
    D, bf16, f32, group = bench.D, 2, 4, bench.HV // bench.HK
    qk = 2 * D * bf16 // group            # q and k, shared by the group's value heads
    v = o = do = D * bf16
    gates = 2 * f32                       # g (scalar gate) and beta
    grads = 2 * D * f32 // group + D * f32 + 2 * f32   # dq, dk; dv; dg, dbeta
    model = bench.KERNEL_MODEL
    assert model["chunk_prep"][0] == qk + v + gates
    assert model["chunk_scan_fwd"][0] == o
    assert model["chunk_scan_bwd"][0] == do
    assert model["chunk_grad"][0] == qk + v + do + gates + grads
    assert bench.STEP_BYTES == (qk + v + o + gates + model["chunk_grad"][0]) * bench.UNITS


def test_step_flops_are_forward_plus_vjp_products():
    """Forward 6 D^2 + 10 C D and VJP 14 D^2 + 28 C D + 4 C^2 flops per unit (the tensor-core
    products of the chunk algebra, 2 flops per multiply-add)."""
    D, C = bench.D, bench.C
    assert bench.STEP_FLOPS == ((6 * D * D + 10 * C * D) + (14 * D * D + 28 * C * D + 4 * C * C)) * bench.UNITS
