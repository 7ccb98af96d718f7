"""The benchmark's JSON line stays short enough for a reader that keeps only
the last 3 KB of the output, with every workload's entry in it (CPU only: the
line is assembled from a workload detail of the size a full run produces)."""

import json

import bench


def _verbose_entry(name, i):
    # every key a workload's detail may carry, with unrounded values and the
    # longest strings the benchmark writes
    return {
        "value": 1234.56789012345 + i, "unit": "TFLOP/s", "ms_per_call": 0.398765432109876,
        "us_per_call": 22.6345678901, "us_per_graph_replay": 21.0123456789, "us_per_call_in_graph": 26.7345678,
        "paths": "simt+simt", "achieved_gbs": 5928.123456789, "frac": 0.71349876543, "peak": 40.0765432,
        "frac_of_write_peak": 0.83456789012, "bound": "tensor", "kernels_per_call": 4,
        "l2": "weights (3.8 GB int8) larger than L2", "types": "input torch.bfloat16, weights int8, block K",
        "stream_probe": {"write_gbs": 6400.1, "write_bulk_gbs": 6722.3, "copy_gbs": 6690.2},
        "cpu_baseline": {"value": 0.0432198765, "unit": "TOP/s", "cores": 16, "kind": "oracle",
                         "sample": "512 tokens x 512 cols"},
    }


def test_line_with_every_workload_fits_3_kb():
    extras = {name: _verbose_entry(name, i) for i, (_, name, _) in enumerate(bench.PER_CONFIG)}
    per_config = bench.per_config_entries({"value": 1687.0, "unit": "TFLOP/s", "ms_per_call": 0.6516,
                                           "frac": 0.9633}, extras)
    assert set(per_config) == {"2_gemm_bf16"} | {key for key, _, _ in bench.PER_CONFIG}
    assert all("value" in v for v in per_config.values())
    # the other keys of the line, with values of the size a full run writes
    line = {
        "metric": bench.METRIC, "value": 1687.455758142748, "unit": "TFLOP/s", "per_config": per_config,
        "n_gpus": 1, "steps": 1000, "warmup": 20, "ms_per_step": 0.6515795288085937, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic, seeded",
        "config": {"workload": "gemm_bf16", "M": 8192, "N": 8192, "K": 8192, "transB": 1, "alpha": 0.5,
                   "beta": 2.0, "C": [1, 8192], "parallelism": "replicas x1", "l2": "A+B 256 MiB > L2"},
        "roofline": {"bound": "tensor", "achieved": 1687.0, "peak": 1751.8, "unit": "TFLOP/s", "frac": 0.9633,
                     "traffic": 1223205472.0, "peak_kind": "measured bf16_tflops_sustained",
                     "frac_of_burst": 0.8737},
        "cpu_baseline": {"value": 0.04815, "unit": "TFLOP/s", "cores": 16, "kind": "oracle",
                         "sample": "256 of 8192 rows, C++ oracle (plain double loops)"},
        "e2e": {"value": 754.8, "unit": "TFLOP/s", "ms_per_step": 1.457, "h2d_bytes_per_step": 268451840,
                "d2h_bytes_per_step": 134217728, "host_link_gbs": 276.4},
        "gpu_launches": 1000,
        "clocks": {"sm_mhz": 1627.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 33},
        "device_status": "MM_OK",
    }
    n = len(json.dumps(line))
    assert n < 3000, n


def test_error_of_other_workloads_is_kept_short():
    per_config = bench.per_config_entries({"value": 1.0}, {"error": "RuntimeError: " + "x" * 1000})
    assert len(per_config["error"]) == 200
