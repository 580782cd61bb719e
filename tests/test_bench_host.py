"""Host-side logic of bench.py, without a GPU: the clock record parsed from
nvidia-smi lines, the staleness rule of the committed DRAM-traffic figure, the
code-only hash it rests on, the whole-job throughput, and the burst / sustained
legs of the roofline (against a fake device clock)."""
import datetime

import pytest

import bench


def _line(ts, sm, smax, power, reasons=("Not Active",) * 4):
    return ", ".join([ts.strftime("%Y/%m/%d %H:%M:%S.%f")[:-3], str(sm), str(smax), str(power), "0x0", *reasons])


def test_clock_record_keeps_only_samples_inside_the_timed_region():
    t0 = datetime.datetime(2026, 1, 2, 3, 4, 5)
    s = bench.ClockSampler(0)
    s.proc = None
    s.t_begin = t0 + datetime.timedelta(seconds=1)
    s.t_end = t0 + datetime.timedelta(seconds=2)
    s.lines = [
        _line(t0, 2070, 2070, 150.0),  # before the region: idle clock, ignored
        _line(t0 + datetime.timedelta(seconds=1.1), 1800, 2070, 900.0,
              ("Not Active", "Not Active", "Not Active", "Active")),
        _line(t0 + datetime.timedelta(seconds=1.5), 1750, 2070, 950.0),
        _line(t0 + datetime.timedelta(seconds=1.9), 1790, 2070, 940.0),
        _line(t0 + datetime.timedelta(seconds=2.5), 300, 2070, 90.0,
              ("Active", "Not Active", "Not Active", "Not Active")),  # after: ignored
        "garbage line",
    ]

    class _Done:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    s.proc = _Done()
    rec = s.stop()
    assert rec["samples"] == 3
    assert rec["sm_mhz"] == 1790.0
    assert rec["sm_mhz_min"] == 1750.0
    assert rec["sm_max_mhz"] == 2070.0
    assert rec["power_w_max"] == 950.0
    # the hw_slowdown sample lies outside the region; sw_power_cap inside it counts
    assert rec["reasons"] == ["sw_power_cap"]


def test_clock_record_without_nvidia_smi_says_so():
    s = bench.ClockSampler(0)
    rec = s.stop()
    assert rec["sm_mhz"] is None and rec["reasons"] == ["nvidia-smi unavailable"]


def test_code_only_drops_comments_and_layout_but_not_code():
    a = 'int x = 1;  // one\n/* block\n comment */ int y = "a//b";\n'
    b = 'int x = 1;\nint y = "a//b"; // other words\n'
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only("int x = 1;") != bench._code_only("int x = 2;")
    # a comment marker inside a string literal is code
    assert '"a//b"' in bench._code_only(a)


def test_traffic_figure_is_dropped_when_the_kernel_changes(monkeypatch, tmp_path):
    f = tmp_path / "traffic.txt"
    f.write_text("# comment: ignored\nsource_sha256_16: 0123456789abcdef\n"
                 "dram_bytes_per_full_launch: 763224960\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    monkeypatch.setattr(bench, "source_hash", lambda: "0123456789abcdef")
    assert bench.traffic_from_profile() == 763224960.0
    monkeypatch.setattr(bench, "source_hash", lambda: "fedcba9876543210")
    assert bench.traffic_from_profile() is None


@pytest.mark.parametrize("world", [1, 2, 8])
def test_whole_job_throughput_counts_every_rank(world):
    # every rank does the same work in the slowest rank's time
    assert bench.whole_job_tflops(2.0e12, world, 1000.0) == pytest.approx(2.0 * world)


def test_nvml_clock_record_window_and_reason_bits():
    # the in-process sampler keeps samples inside the timed region only and
    # decodes the clock-event reason bits of each kept sample
    s = bench.NvmlClockSampler.__new__(bench.NvmlClockSampler)
    s.period, s.max_mhz, s.thread, s.power_instant = 0.005, 2070.0, None, True
    s._stop = bench.threading.Event()
    s.t_begin, s.t_end = 10.0, 11.0
    s.samples = [
        (9.9, 2070.0, 120.0, 0x0),          # before the region
        (10.1, 1800.0, 1380.0, 0x4),        # sw_power_cap
        (10.5, 1755.0, 1395.0, 0x4 | 0x0),
        (10.9, 1790.0, 1390.0, 0x0),
        (11.2, 600.0, 90.0, 0x8 | 0x40),    # after: hw_slowdown / hw_thermal_slowdown not counted
    ]
    rec = s.stop()
    assert rec["samples"] == 3
    assert rec["sm_mhz"] == 1790.0 and rec["sm_mhz_min"] == 1755.0 and rec["sm_max_mhz"] == 2070.0
    assert rec["power_w_max"] == 1395.0
    assert rec["reasons"] == ["sw_power_cap"]
    assert "NVML" in rec["window"] and "instantaneous" in rec["window"]


class _FakeNvml:
    """NVML calls of one sample: SM clock 1740 MHz, one-second average power
    900 W, instantaneous power 1391.5 W as a field value (or refused)."""

    def __init__(self, serve_field, value_type=1):
        self.serve_field, self.value_type, self.field_calls = serve_field, value_type, 0

    def nvmlDeviceGetClockInfo(self, h, kind, out):
        out._obj.value = 1740
        return 0

    def nvmlDeviceGetPowerUsage(self, h, out):
        out._obj.value = 900000
        return 0

    def nvmlDeviceGetFieldValues(self, h, n, fv):
        import ctypes
        self.field_calls += 1
        v = fv._obj
        assert n == 1 and v.fieldId == 186
        if not self.serve_field:
            v.nvmlReturn = 3  # NVML_ERROR_NOT_SUPPORTED
            return 0
        v.nvmlReturn, v.valueType = 0, self.value_type
        if self.value_type == 0:
            v.value = ctypes.c_ulonglong.from_buffer_copy(ctypes.c_double(1391500.0)).value
        else:
            v.value = 1391500
        return 0


def _nvml_sampler(lib):
    import ctypes
    s = bench.NvmlClockSampler.__new__(bench.NvmlClockSampler)
    s.ct, s.lib, s.h, s.power_instant = ctypes, lib, None, True
    s.reason_fn = lambda h, out: (setattr(out._obj, "value", 0x4), 0)[1]
    return s


@pytest.mark.parametrize("value_type", [0, 1, 3])
def test_nvml_sample_takes_the_instantaneous_power_field(value_type):
    s = _nvml_sampler(_FakeNvml(True, value_type))
    _, mhz, power, reasons = s._one()
    assert mhz == 1740.0 and power == pytest.approx(1391.5) and reasons == 0x4
    assert s.power_instant


def test_nvml_sample_falls_back_to_the_average_power_once_the_field_is_refused():
    lib = _FakeNvml(False)
    s = _nvml_sampler(lib)
    assert s._one()[2] == pytest.approx(900.0) and not s.power_instant
    assert s._one()[2] == pytest.approx(900.0) and lib.field_calls == 1  # not asked again


def test_nvml_sampler_without_the_driver_falls_back():
    # no NVML here: the sampler reports itself unusable and clock_sampler
    # falls back to the nvidia-smi reader
    s = bench.NvmlClockSampler(None, None)
    if not s.ok:
        class _T:
            class cuda:
                @staticmethod
                def get_device_properties(i):
                    raise RuntimeError("no GPU")
        assert isinstance(bench.clock_sampler(_T, 0), bench.ClockSampler)


class _FakeDevice:
    """Device clock of a fake torch: every attention launch advances it by the
    next duration (ms) from a list."""

    def __init__(self, durations):
        self.now, self.durations, self.launches = 0.0, list(durations), 0

    def launch(self):
        self.now += self.durations[min(self.launches, len(self.durations) - 1)]
        self.launches += 1


def _fake_torch(dev):
    class Event:
        def __init__(self, enable_timing=False):
            self.t = None

        def record(self, stream=None):
            self.t = dev.now

        def elapsed_time(self, other):
            return other.t - self.t

    class Cuda:
        pass

    cuda = Cuda()
    cuda.Event = Event
    cuda.current_stream = lambda: None
    cuda.synchronize = lambda: None

    class Torch:
        pass

    t = Torch()
    t.cuda = cuda
    return t


def _fake_bss(dev, status=0):
    class Bss:
        @staticmethod
        def sparse_attention_split(*a):
            dev.launch()

        @staticmethod
        def get_device_status():
            return status

        @staticmethod
        def status_string(s):
            return f"status {s}"

    return Bss


class _FakeSampler:
    def start(self):
        pass

    def mark_begin(self):
        pass

    def mark_end(self):
        pass

    def stop(self):
        return {"sm_mhz": 1740.0, "reasons": ["sw_power_cap"], "samples": 9}


def test_power_regimes_time_each_end_of_the_ramp_against_its_own_peak(monkeypatch):
    monkeypatch.setattr(bench.time, "sleep", lambda s: None)
    monkeypatch.setattr(bench, "clock_sampler", lambda torch, idx: _FakeSampler())
    # three bursts (5.0, 5.4, 5.2 ms), then every launch 6.0 ms (the settled regime)
    dev = _FakeDevice([5.0, 5.4, 5.2, 6.0])
    peaks = {"bf16_tflops": 2000.0, "bf16_tflops_sustained": 1500.0}
    flops = 10e12
    out = bench.power_regimes(_fake_bss(dev), _fake_torch(dev), *[None] * 9, flops, peaks, 0, sustain_s=0.12)
    b, s = out["burst"], out["sustained"]
    assert b["ms"] == pytest.approx(5.2)  # median of the three
    assert b["achieved"] == pytest.approx(flops / 5.2e-3 / 1e12)
    assert b["peak"] == 2000.0 and b["frac"] == pytest.approx(b["achieved"] / 2000.0)
    # 0.12 s / 2 / 5.2 ms -> 11 launches a half; only the second half is timed
    assert s["launches"] == 11 and dev.launches == 3 + 2 * 11
    assert s["ms"] == pytest.approx(6.0)
    assert s["peak"] == 1500.0 and s["frac"] == pytest.approx(flops / 6.0e-3 / 1e12 / 1500.0)
    assert s["clocks"]["reasons"] == ["sw_power_cap"]


def test_power_regimes_refuse_a_device_error(monkeypatch):
    monkeypatch.setattr(bench.time, "sleep", lambda s: None)
    monkeypatch.setattr(bench, "clock_sampler", lambda torch, idx: _FakeSampler())
    dev = _FakeDevice([5.0])
    with pytest.raises(RuntimeError, match="power-regime"):
        bench.power_regimes(_fake_bss(dev, status=3), _fake_torch(dev), *[None] * 9, 1e12,
                            {"bf16_tflops": 1.0, "bf16_tflops_sustained": 1.0}, 0, sustain_s=0.05)
