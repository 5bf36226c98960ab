"""bench.py's host-side arithmetic (no GPU): the roofline denominators and the
list of workloads the default run measures beside the contract's."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from dense_gemm_epilogues_gb300 import inputs as I  # noqa: E402

PEAKS = {"bf16_tflops": 1897.1, "bf16_tflops_sustained": 1690.9, "hbm_gbs": 6789.0, "source": "measured"}


def test_short_unthrottled_region_divides_by_the_burst_peak():
    pk, src = bench.choose_tensor_peak(PEAKS, {"samples_under_load": 5, "power_cap_samples_under_load": 0},
                                       0.054)
    assert pk == PEAKS["bf16_tflops"] and "burst" in src


@pytest.mark.parametrize("timed_s,capped,under", [(0.8, 40, 50), (3.0, 10, 50), (3.0, 0, 0)])
def test_sustained_peak_needs_a_long_region_mostly_at_the_power_cap(timed_s, capped, under):
    pk, _ = bench.choose_tensor_peak(PEAKS, {"samples_under_load": under,
                                             "power_cap_samples_under_load": capped}, timed_s)
    assert pk == PEAKS["bf16_tflops"]


def test_long_capped_region_divides_by_the_sustained_peak():
    pk, src = bench.choose_tensor_peak(PEAKS, {"samples_under_load": 50, "power_cap_samples_under_load": 40},
                                       3.0)
    assert pk == PEAKS["bf16_tflops_sustained"] and "sustained" in src


def test_ffma_peak_from_unit_counts_and_clock():
    # 152 SMs x 128 lanes x 2 flops x 2.07 GHz
    assert bench.ffma_peak_tflops(152, 2070.0) == pytest.approx(80.5478, rel=1e-4)


def test_algorithmic_bytes_of_the_fc_layer():
    p = I.fc_bf16_8192x4096x11008()
    want = 8192 * 4096 * 2 + 4096 * 11008 * 2 + 8192 * 11008 * 2 + 11008 * 4
    assert bench.algorithmic_bytes(p, I.ELEM_BYTES) == want


def test_algorithmic_bytes_count_c_when_it_is_read():
    p = I.square_fp16_8192("TN")
    assert bench.algorithmic_bytes(p, I.ELEM_BYTES) == 2 * 8192 * 8192 * 2 + 2 * 8192 * 8192 * 4


def test_default_run_measures_every_other_workload():
    names = [w[0] for w in bench.config_workloads()]
    # config 1, the FC layer, int8, SGEMM, the five squares of the sweep, the skinny shape
    assert len(names) == 10 and len(set(names)) == 10
    bounds = {w[0]: w[3] for w in bench.config_workloads()}
    assert bounds["skinny_gemm_f16_tn_16384x64x16384"] == "hbm"
    assert bounds["sgemm_f32_tn_4096_bias_relu"] == "alu"
    sweep = sorted(w[1].M for w in bench.config_workloads() if w[0].startswith("sweep_"))
    assert sweep == [512, 1024, 2048, 4096, 16384]


def test_theoretical_peak_at_the_ncu_clock():
    """The second denominator from the committed counters: flops per
    tensor-active cycle per SM (8192 for fp16 tcgen05 on GB300) times the SMs
    and the clock ncu saw; the launch under ncu as a fraction of it matches the
    tensor-pipe share."""
    c = bench.measured_counters()
    if "sm_cycles_active" not in c:
        pytest.skip("counters stale for the current kernel sources")
    t = bench.theoretical_at_clock(c, 2.0 * 8192 ** 3, 152)
    assert abs(t["flops_per_tensor_cycle_per_sm"] - 8192) < 0.01 * 8192, t
    assert 1900 < t["peak"] < 2100 and 0.8 < t["frac"] < 0.95, t
    assert abs(t["frac"] - c["tensor_pipe_active_pct"] / 100.0) < 0.02, t
    assert bench.theoretical_at_clock({}, 1.0, 152) is None


def test_vs_cublas_mode_is_a_separate_entry(monkeypatch):
    """--vs-cublas selects the comparison routine, which prints no contract line, and
    its graph helper orders its side stream after the stream that wrote the inputs."""
    monkeypatch.setattr(sys, "argv", ["bench.py", "--vs-cublas"])
    args = bench.parse_args()
    assert args.vs_cublas and args.case is None
    import inspect
    src = inspect.getsource(bench._graph_us)
    assert "wait_stream" in src
    assert "run_vs_cublas" in inspect.getsource(bench.main)
