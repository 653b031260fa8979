"""bench.py's host-side helpers on CPU: the algorithmic byte count behind
every GB/s figure, the peak lookup behind the roofline fraction, and the
clock-sample summary that decides whether a run's clocks were clean."""

import json
import os

import bench


def test_gemv_bytes_closed_form():
    """N*K/2 codes + N*G*2 scales + N*G/2 zero points + M*K*2 x + M*N*2 y at
    4 bits, group 128, asymmetric, one token (worked by hand per shape)."""
    assert bench.gemv_bytes(4096, 4096) == 8_388_608 + 262_144 + 65_536 + 8_192 + 8_192 == 8_732_672
    assert bench.gemv_bytes(11008, 4096) == 23_455_232
    assert bench.gemv_bytes(4096, 11008) == 23_455_232
    assert bench.gemv_bytes(8192, 8192) == 34_897_920
    assert bench.gemv_bytes(1024, 8192) == 4_376_576
    assert bench.gemv_bytes(28672, 8192) == 122_101_760
    # symmetric: no zero points; 8 bits: a byte per code and per zero point;
    # 3 bits: 3/8 byte per code, zero points still nibbles
    assert bench.gemv_bytes(4096, 4096, sym=True) == 8_732_672 - 65_536
    assert bench.gemv_bytes(4096, 4096, bits=8) == 16_777_216 + 262_144 + 131_072 + 16_384
    assert bench.gemv_bytes(4096, 4096, bits=3) == 6_291_456 + 262_144 + 65_536 + 16_384
    # more tokens add only activations and outputs
    assert bench.gemv_bytes(4096, 4096, M=16) - bench.gemv_bytes(4096, 4096) == 15 * (4096 * 2 + 4096 * 2)


def test_llama2_7b_step_bytes():
    """32 layers x (q, k, v, o 4096x4096; gate, up 11008x4096; down 4096x11008)."""
    per_layer = 4 * bench.gemv_bytes(4096, 4096) + 3 * bench.gemv_bytes(11008, 4096)
    assert 32 * per_layer == 3_369_484_288


def test_measured_peaks_reads_the_file_or_falls_back(tmp_path, monkeypatch):
    path = os.path.join(bench.ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        assert bench.measured_peaks() == (float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peaks() == (bench.FALLBACK_HBM_GBPS, bench.FALLBACK_BF16_TFLOPS, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6000.5, "bf16_tflops": 1700}))
    assert bench.measured_peaks() == (6000.5, 1700.0, "measured")


def sampler_with(samples, max_mhz=2032.0):
    # no NVML here: the constructor records why and keeps no handle
    s = bench.ClockSampler(None, None)
    s.samples = list(samples)
    s.max_mhz = max_mhz
    return s


def test_clock_summary_median_max_and_reasons():
    rows = [(True, 2032.0, 0x0), (True, 1980.0, 0x4), (True, 2010.0, 0x0),
            (False, 900.0, 0x8)]  # outside the timed region: ignored
    s = sampler_with(rows).summary()
    assert s["sm_mhz"] == 2010.0 and s["sm_max_mhz"] == 2032.0 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"] and s["min_mhz"] == 1980.0
    hot = sampler_with(rows + [(True, 1500.0, 0x40)]).summary()
    assert hot["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    slow = sampler_with([(True, 2000.0, 0x8 | 0x20)]).summary()
    assert slow["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_clock_summary_without_samples():
    s = bench.ClockSampler(None, None).summary()
    assert s["sm_mhz"] is None and s["reasons"] == ["unsampled"] and s["error"]
    outside = sampler_with([(False, 2032.0, 0)]).summary()
    assert outside["reasons"] == ["unsampled"]
