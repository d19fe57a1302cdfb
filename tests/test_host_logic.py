"""Host-side logic that needs no GPU: the benchmark's clock-record checks and traffic-record lookup,
and the seeded input recipe shared by the oracle and the CUDA path."""
import hashlib
import os

import numpy as np
import pytest
import torch

import bench
import workloads as wl


# ---------------------------------------------------------------- bench host logic

@pytest.mark.parametrize("summary,expect", [
    ({"sm_mhz": 1560.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}, []),
    ({"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}, []),
    ({"sm_mhz": 1400.0, "sm_max_mhz": 2070.0, "reasons": ["hw_slowdown", "sw_power_cap"]}, ["hw_slowdown"]),
    ({"sm_mhz": 1400.0, "sm_max_mhz": 2070.0, "reasons": ["sw_thermal_slowdown", "hw_thermal_slowdown"]},
     ["hw_thermal_slowdown", "sw_thermal_slowdown"]),
    ({"sm_mhz": 1005.0, "sm_max_mhz": 2070.0, "reasons": []}, ["sm_clock_low_without_reason"]),
    ({"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}, []),
])
def test_clock_suspect(summary, expect):
    assert bench.clock_suspect(summary) == expect


def test_clock_sampler_summary_parses_nvidia_smi_lines():
    s = bench.ClockSampler(0)
    s.lines = [
        "0, 2070, 2070, 150.0, 0x0, Not Active, Not Active, Not Active, Not Active",  # idle before load
        "0, 1560, 2070, 960.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 1550, 2070, 955.5, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 1580, 2070, 940.0, 0x4, Not Active, Not Active, Not Active, Active",
        "garbage line",
    ]
    out = s.summary()
    assert out["sm_mhz"] == 1560.0  # median of the loaded samples only
    assert out["sm_max_mhz"] == 2070.0 and out["reasons"] == ["sw_power_cap"]
    assert out["samples"] == 4 and out["power_w_max"] == 960.0
    assert bench.ClockSampler(0).summary()["reasons"] == ["unsampled"]


def test_load_traffic_follows_the_kernel_source(tmp_path, monkeypatch):
    src = tmp_path / "scaling_quantization_gemm_gb300" / "csrc"
    src.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (src / "gemm.cu").write_bytes(b"// kernel source v1\n")
    sha = hashlib.sha1(b"// kernel source v1\n").hexdigest()
    (tmp_path / "profiles" / "traffic.txt").write_text(
        f"kernel=gemm_tensor_pair_kernel bytes_per_launch=123456 source=gemm.cu source_sha1={sha} workload=w\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_traffic("gemm_tensor_pair_kernel") == 123456
    assert bench.load_traffic("another_kernel") is None
    (src / "gemm.cu").write_bytes(b"// kernel source v2\n")  # changed since the capture: no traffic
    assert bench.load_traffic("gemm_tensor_pair_kernel") is None
    os.remove(tmp_path / "profiles" / "traffic.txt")
    assert bench.load_traffic("gemm_tensor_pair_kernel") is None


# ---------------------------------------------------------------- input recipe

def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.standard_normal(50000) * 1e3, np.exp2(rng.uniform(-120, 120, 50000)),
                        # exact ties between two bf16 values
                        (np.arange(1, 3000, dtype=np.uint32) << 16 | 0x8000).view(np.float32).astype(np.float64)])
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(wl.bf16_bits(v), ref)


def test_generation_does_not_depend_on_chunking(monkeypatch):
    whole = wl.normal(np.random.default_rng(5), 64, 96, 0.5)
    monkeypatch.setattr(wl, "CHUNK_ELEMS", 96 * 5)  # five rows per draw
    assert np.array_equal(wl.normal(np.random.default_rng(5), 64, 96, 0.5), whole)


def test_current_scaling_workload_outliers():
    X, W = wl.linear_fwd_current()
    x = wl.bf16_to_f32(X)
    assert np.count_nonzero(np.abs(x) == 30.0) == 8
    assert np.abs(x[np.abs(x) != 30.0]).max() < 0.2  # N(0, 0.02^2) elsewhere
    assert X.shape == (256, 1024) and W.shape == (1024, 1024)
    X2, W2 = wl.linear_fwd_current()
    assert np.array_equal(X, X2) and np.array_equal(W, W2)  # seeded


def test_delayed_activation_grows_with_t():
    s = [float(np.std(wl.bf16_to_f32(wl.delayed_activation(t, 256, 256)))) for t in (0, 5, 10)]
    assert s[0] == pytest.approx(1.0, rel=0.02) and s[1] == pytest.approx(1.5, rel=0.02)
    assert s[2] == pytest.approx(2.0, rel=0.02)
