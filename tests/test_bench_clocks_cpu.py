"""Clock record of the benchmark's timed region, on CPU with fake samples: the summary takes the
median SM clock over both sources and reports every throttle reason either source saw (the ones
that make a measurement invalid must never be dropped)."""
import bench


def _smi(mhz, hw=False, hw_thermal=False, sw_thermal=False, power=False):
    act = lambda b: "Active" if b else "Not Active"
    return ["0", str(mhz), "2070", "950.00", "0x0", act(hw), act(hw_thermal), act(sw_thermal), act(power)]


def test_no_samples_is_reported():
    assert bench.summarize_clocks([], [], None)["reasons"] == ["no samples"]


def test_median_and_max_over_both_sources():
    out = bench.summarize_clocks([_smi(1900)], [(2070.0, 0), (2070.0, 0), (2000.0, 0)], 2070.0)
    assert out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0
    assert out["samples"] == 4 and out["reasons"] == []
    assert out["sources"] == {"nvidia_smi_100ms": 1, "nvml_2ms": 3}


def test_reasons_from_nvml_bits():
    # NVML clock-event reason bits: 0x4 sw power cap, 0x8 hw slowdown, 0x20 sw thermal, 0x40 hw thermal
    out = bench.summarize_clocks([], [(2070.0, 0x4), (1500.0, 0x8 | 0x40), (1600.0, 0x20)], 2070.0)
    assert out["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap", "sw_thermal_slowdown"]


def test_reasons_from_nvidia_smi_rows():
    out = bench.summarize_clocks([_smi(2070, power=True), _smi(1800, sw_thermal=True)], [], None)
    assert out["reasons"] == ["sw_power_cap", "sw_thermal_slowdown"]
    assert out["sm_max_mhz"] == 2070.0


def test_sampler_without_driver_library_degrades():
    s = bench.ClockSampler(0)
    s.start()
    out = s.stop()
    assert "sm_mhz" in out and "reasons" in out


def test_sampler_leaves_no_temp_file(monkeypatch):
    # without nvidia-smi (or with it) the sampler's temp file is gone after stop()
    import os

    import bench

    def no_smi(*a, **k):
        raise FileNotFoundError("nvidia-smi")

    monkeypatch.setattr(bench.subprocess, "Popen", no_smi)
    c = bench.ClockSampler(0)
    c.start()
    path = c.path
    assert path is not None and os.path.exists(path)
    c.stop()
    assert not os.path.exists(path)
