"""The bench's algorithmic work per launch, against closed forms written out here.

Every roofline fraction the bench reports divides these counts by a measured time, so a
wrong count would misstate every figure.  FLOPs are 2·M·N·K per GEMM (one multiply and one
add per term); bytes count each operand once, C read only when beta != 0 and written once.
The FFN counts are the pages' own: about 103 GFLOP against 128 MiB touched
("Operator & Runtime", chapter introduction and section 5.2.1).
"""
import pytest

import bench
from dense_gemm_sm_gb300 import inputs


def spec(name):
    return bench.Workload.spec(name, inputs)


def test_fp32_counts():
    s = spec("sgemm_4096")
    assert s["unit"] == "TFLOPS" and s["bound"] == "alu"
    assert s["flops"] == 137_438_953_472                        # 2 * 4096^3
    assert s["algo_bytes"] == 4 * 4 * 4096 * 4096               # A, B, C read (beta 0.5), C written
    r = spec("sgemm_ragged")
    M, N, K = 1000, 3000, 777
    assert r["flops"] == 2 * M * N * K == 4_662_000_000
    assert r["algo_bytes"] == 4 * (M * K + K * N + 2 * M * N)


def test_ffn_counts_are_the_pages_figures():
    s = spec("ffn_bf16")
    assert s["flops"] == 103_079_215_104                        # ~103 GFLOP
    assert s["algo_bytes"] == 128 * 2 ** 20                     # X 8 MiB + W 96 MiB + C 24 MiB
    g = spec("ffn_gate_up")
    assert g["flops"] == 2 * 103_079_215_104                    # two projections
    assert g["algo_bytes"] == 2 * (1024 * 4096 + 2 * 4096 * 12288 + 1024 * 12288)


@pytest.mark.parametrize("M", [1, 4, 16])
def test_decode_counts_and_unit(M):
    s = spec(f"decode_m{M}")
    assert s["unit"] == "GB/s" and s["bound"] == "hbm"
    assert s["algo_bytes"] == 2 * (M * 4096 + 4096 * 12288 + M * 12288)
    assert s["flops"] == 2 * M * 12288 * 4096
    # GB/s = algorithmic bytes / time: the W stream of 96 MiB dominates.
    w = bench.Workload.__new__(bench.Workload)
    w.__dict__.update(s)
    assert w.metric_value(20e-6) == pytest.approx(s["algo_bytes"] / 20e-6 / 1e9)


def test_batched_qk_counts():
    s = spec("qk_batched")
    b, S, D = 64, 2048, 128
    assert s["flops"] == 2 * b * S * S * D == 68_719_476_736
    assert s["algo_bytes"] == 2 * b * 2 * S * D + 4 * b * S * S  # BF16 Q and K, FP32 C
    w = bench.Workload.__new__(bench.Workload)
    w.__dict__.update(s)
    assert w.metric_value(1e-3) == pytest.approx(68.719476736)


class _FakeCuda:
    """Stands in for torch.cuda in the roofline's SM-count query (no GPU here)."""

    def __init__(self, sms):
        self.sms = sms

    def current_device(self):
        return 0

    def get_device_properties(self, dev):
        return type("Props", (), {"multi_processor_count": self.sms})()


@pytest.mark.parametrize("sms", [152, 148])
def test_roofline_peaks(sms):
    # Kernels are timed in isolation, so tensor work is measured against the burst BF16
    # figure (FP8: twice it); the FP32 CUDA-core peak uses the device's own SM count.
    peaks = dict(hbm_gbs=6698.5, bf16=1929.9, bf16_sustained=1761.4, sm_max_mhz=2070.0,
                 source="measured")
    fake_torch = type("T", (), {"cuda": _FakeCuda(sms)})()

    def wl(name):
        w = bench.Workload.__new__(bench.Workload)
        w.__dict__.update(spec(name), name=name, torch=fake_torch)
        return w

    r = wl("sgemm_4096").roofline(2.0e-3, peaks, None)
    assert r["bound"] == "alu"
    assert r["peak"] == pytest.approx(sms * 128 * 2 * 2070e6 / 1e12, abs=0.05)
    assert r["frac"] == pytest.approx((2 * 4096 ** 3 / 2.0e-3 / 1e12) / r["peak"], rel=1e-3)
    assert wl("ffn_bf16").roofline(60e-6, peaks, None)["peak"] == pytest.approx(1929.9)
    assert wl("fp8_ffn").roofline(40e-6, peaks, None)["peak"] == pytest.approx(2 * 1929.9)
    d = wl("decode_m1").roofline(19e-6, peaks, None)
    assert d["bound"] == "hbm" and d["peak"] == pytest.approx(6698.5)
