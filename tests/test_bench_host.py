"""Host-side logic of bench.py that needs no GPU: which repeat is reported and
how the clock records of several timed regions combine."""
import bench


def test_median_run_picks_the_middle_repeat_with_its_kernel_times():
    runs = [{"total_ms": 9.0, "per_kernel_ms": {"fwd": 3.0}},
            {"total_ms": 7.0, "per_kernel_ms": {"fwd": 2.0}},
            {"total_ms": 8.0, "per_kernel_ms": {"fwd": 2.5}}]
    r = bench.median_run(runs)
    assert r["total_ms"] == 8.0 and r["per_kernel_ms"]["fwd"] == 2.5
    # an even count takes the lower middle
    assert bench.median_run(runs[:2])["total_ms"] == 7.0


def test_merge_clocks_keeps_every_throttle_reason():
    a = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "power_w_max": 900.0,
         "samples": 5}
    b = {"sm_mhz": 1900.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"],
         "power_w_max": 1300.0, "samples": 4}
    c = {"sm_mhz": 2000.0, "sm_max_mhz": 2070.0, "reasons": ["hw_slowdown"],
         "power_w_max": None, "samples": 6}
    m = bench.merge_clocks([a, b, c])
    assert m["sm_mhz"] == 2000.0 and m["sm_max_mhz"] == 2070.0
    assert m["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert m["power_w_max"] == 1300.0 and m["samples"] == 15


def test_merge_clocks_without_samples():
    m = bench.merge_clocks([{"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"],
                             "samples": 0}])
    assert m["reasons"] == ["unsampled"]


def test_e2e_slots_and_steps():
    """The end-to-end sessions get enough slots to compute through a host-link
    pause of E2E_RIDE_MS, within a quarter of the free memory, and about a
    second of timed steps."""
    import bench
    gib = 1 << 30
    per_slot = lambda n: n * 908 * (1 << 20)  # noqa: E731 -- the long workload's slots
    # 6.4 ms steps: ceil(80 / 6.4) + 1 = 14 slots (12.4 GiB of 270 GiB free)
    assert bench.e2e_slots(0, 6.4, per_slot, 270 * gib, 16) == 14
    # short steps: capped at the session's maximum
    assert bench.e2e_slots(0, 0.05, per_slot, 270 * gib, 16) == 16
    # long steps: at least two
    assert bench.e2e_slots(0, 500.0, per_slot, 270 * gib, 16) == 2
    # little free memory: fewer slots, never below two
    assert bench.e2e_slots(0, 6.4, per_slot, 16 * gib, 16) == 4
    assert bench.e2e_slots(0, 6.4, per_slot, 1 * gib, 16) == 2
    # an explicit request is clamped to the session's range
    assert bench.e2e_slots(40, 6.4, per_slot, 270 * gib, 16) == 16
    assert bench.e2e_slots(1, 6.4, per_slot, 270 * gib, 16) == 2
    # not yet timed: 8 ms assumed
    assert bench.e2e_slots(0, None, per_slot, 270 * gib, 16) == 11
    assert bench.e2e_steps(1.0, 6.4) == 157
    assert bench.e2e_steps(1.0, 0.04) == 1000
    assert bench.e2e_steps(1.0, 900.0) == 3
    assert bench.e2e_steps(1.0, None) == 125
