"""bench.py's host logic (no GPU): the record it prints stays complete and short.

The driver keeps only the end of the benchmark's output, so the secondary
figures are printed again as one short JSON line after the headline; it must
stay well under that window.  Both arms (the CUDA path and the CPU-oracle
reference arm) must describe their workload with the same `config`.
"""
import json

import bench
import workloads


def fake_also():
    clocks = {"sm_mhz": 1440.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 12,
              "window": "timed region"}
    small = {"tflops": 7.3, "gpu_us_per_launch": 4.6032, "single_call_us": 18.43,
             "launch_overhead_us": 13.8, "roofline_us": 0.077, "roofline_frac": 0.0168,
             "launch_floor_us": 0.66, "launch_floor": "graph of 20 empty kernels",
             "timing": "x" * 120, "kernel": "tma", "staged": 0}
    also = {
        "sustained_square8192_bf16": {"tflops": 1601.234, "launches": 4200, "seconds": 2.51,
                                      "frac_of_sustained_peak": 0.9438, "peak": 1696.4,
                                      "peak_source": "measured", "clocks": clocks,
                                      "tflops_per_ghz": 1111.97,
                                      "torch_matmul": {"tflops": 1650.2, "seconds": 2.6,
                                                       "clocks": dict(clocks, sm_mhz=1425.0),
                                                       "tflops_per_ghz": 1158.0, "what": "w" * 60}},
        "square4096_bf16": {"tflops": 1633.21, "pct_of_peak": 86.3, "median_ms": 0.084,
                            "torch_matmul_tflops": 1756.2, "torch_matmul": "y" * 80},
        "skinny16x4096x14336_bf16": {"gbs": 6133.3, "pct_of_hbm_peak": 90.51,
                                     "torch_matmul_gbs": 5578.0, "timing": "z" * 80},
        "gemm256_f16": dict(small),
        "ragged1023x1000x1029_f16": dict(small),
    }
    for n in ("softmax65536x1000_f32", "softmax4096x32768_f32"):
        also[n] = {"gbs": 6486.1, "pct_of_hbm_peak": 95.7, "torch_softmax_gbs": 6405.2}
    for n in ("attn_bh16_s8192_d64_bf16_causal", "attn_bh16_s8192_d64_bf16",
              "attn_bh16_s8192_d128_bf16_causal"):
        also[n] = {"tflops": 799.4, "pct_of_peak": 42.2, "torch_sdpa_tflops": 292.0}
    return also


def test_summary_line_is_short_and_complete():
    also = fake_also()
    line = json.dumps({"secondary": bench.summary(also)})
    assert len(line) < 1300, len(line)
    summ = json.loads(line)["secondary"]
    assert set(summ) == set(also)
    assert summ["skinny16x4096x14336_bf16"]["gbs"] == 6133.0
    assert summ["sustained_square8192_bf16"]["clock_samples"] == 12
    assert summ["sustained_square8192_bf16"]["per_ghz"] == 1112.0
    assert summ["sustained_square8192_bf16"]["matmul_per_ghz"] == 1158.0
    assert summ["gemm256_f16"]["floor_us"] == 0.66
    assert summ["square4096_bf16"]["matmul"] == 1756.2


def test_both_arms_share_one_config():
    w = workloads.WORKLOADS[bench.HEADLINE]
    assert bench.headline_config(w, 1) == bench.headline_config(w, 1)
    cfg = bench.headline_config(w, 1)
    assert cfg["workload"] == "square8192_bf16" and (cfg["M"], cfg["N"], cfg["K"]) == (8192,) * 3
    assert bench.SAMPLE_ROWS <= w.M
