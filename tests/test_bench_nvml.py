"""bench.py's NVML records, checked on the CPU against a fake NVML library: the energy record
(TFLOP per joule from the board's cumulative energy counter, the pages' energy comparison;
spbcomputers.ru ZYFA article, "Цифры") and the in-process clock sampler.  Only read queries exist in
bench.py; the fake records every call so the test can check that nothing else was asked."""
import bench


class FakeNvml:
    """Answers NVML's read queries from fixed values; unknown attributes raise AttributeError, as a
    missing symbol does in ctypes."""

    READS = {"nvmlInit_v2", "nvmlDeviceGetHandleByUUID", "nvmlDeviceGetHandleByIndex_v2", "nvmlDeviceGetClockInfo",
             "nvmlDeviceGetMaxClockInfo", "nvmlDeviceGetPowerUsage", "nvmlDeviceGetCurrentClocksEventReasons",
             "nvmlDeviceGetTotalEnergyConsumption"}

    def __init__(self, energy_mj=(1000, 4000), sm=1800, sm_max=2070, power_mw=1390000, reasons=0x4, fail=()):
        self.calls = []
        self.energy = list(energy_mj)
        self.values = {"nvmlDeviceGetClockInfo": sm, "nvmlDeviceGetMaxClockInfo": sm_max,
                       "nvmlDeviceGetPowerUsage": power_mw, "nvmlDeviceGetCurrentClocksEventReasons": reasons}
        self.fail = set(fail)

    def __getattr__(self, name):
        if name not in self.READS:
            raise AttributeError(name)

        def fn(*args):
            self.calls.append(name)
            if name in self.fail:
                return 999
            if name == "nvmlInit_v2":
                return 0
            if name.startswith("nvmlDeviceGetHandle"):
                return 0
            out = args[-1]._obj
            out.value = self.energy.pop(0) if name == "nvmlDeviceGetTotalEnergyConsumption" else self.values[name]
            return 0
        return fn


def test_energy_record_from_the_counter():
    meter = bench.EnergyCounter(0, lib=FakeNvml(energy_mj=(1_000, 31_000)))
    e0, e1 = meter.read_mj(), meter.read_mj()
    rec = bench.energy_block(e0, e1, steps=10, flops_per_step=8.796e12, seconds=0.02)
    # 30 J over 10 steps of 8.796e12 FLOP: 2.932 TFLOP/J, 3 J per step, 1.5 kW over 20 ms
    assert abs(rec["tflop_per_joule"] - 8.796e13 / 30 / 1e12) < 1e-12
    assert abs(rec["joules_per_step"] - 3.0) < 1e-12 and abs(rec["avg_power_w"] - 1500.0) < 1e-9


def test_energy_unavailable_is_reported_not_invented():
    meter = bench.EnergyCounter(0, lib=FakeNvml(fail={"nvmlDeviceGetTotalEnergyConsumption"}))
    assert meter.read_mj() is None
    assert "unavailable" in bench.energy_block(meter.read_mj(), meter.read_mj(), 10, 1e12, 1.0)
    assert "unavailable" in bench.energy_block(5_000, 5_000, 10, 1e12, 1.0)       # the counter did not move
    no_lib = bench.EnergyCounter(0, lib=FakeNvml(fail={"nvmlInit_v2"}))
    assert no_lib.read_mj() is None


def test_nvml_sampler_summarises_the_window_and_names_reasons():
    fake = FakeNvml(sm=1815, reasons=0x4 | 0x8)
    nv = bench.Nvml(0, lib=fake)
    assert nv.ok
    s = bench.NvmlSampler(nv)
    for _ in range(3):
        s.sample()
    t0 = s.rows[0][0]
    s.rows.append((t0 + 10.0, 2070.0, 2070.0, 180.0, set()))              # after the window
    s.mark(t0 - 1e-3, t0 + 1.0)
    rec = s.stop()
    assert rec["samples"] == 3 and rec["samples_in_window"] and rec["sm_mhz"] == 1815
    assert rec["sm_max_mhz"] == 2070 and rec["power_w_median"] == 1390.0
    assert rec["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert set(fake.calls) <= FakeNvml.READS                                # read queries only


def test_nvml_handle_falls_back_to_the_index_and_reports_failure():
    fake = FakeNvml(fail={"nvmlDeviceGetHandleByUUID"})
    assert bench.Nvml(0, 3, lib=fake).ok
    bad = bench.Nvml(0, lib=FakeNvml(fail={"nvmlDeviceGetHandleByUUID", "nvmlDeviceGetHandleByIndex_v2"}))
    assert not bad.ok and bad.sm_mhz() is None and bad.energy_mj() is None
