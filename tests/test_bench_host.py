"""Host-side pieces of bench.py that need no GPU: the FLOP count behind the headline number,
the ncu traffic lookup and its source-hash guard, and the roofline denominators."""
import json
import os
import re

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_layer_flops_is_the_sum_of_the_step_products():
    """2 m n k for every product of one forward and backward: Y = X W^T, U = X A^T, U B^T;
    dX = dY W, V = dY B, V A; dA = V^T X, dB = dY^T U."""
    for M, N, K, r in [(4096, 4096, 4096, 16), (8192, 14336, 4096, 64), (16, 256, 512, 8), (3, 5, 7, 2)]:
        products = [(M, N, K), (M, r, K), (M, N, r),
                    (M, K, N), (M, r, N), (M, K, r),
                    (r, K, M), (N, r, M)]
        assert bench.layer_flops(M, N, K, r) == sum(2.0 * m * n * k for m, n, k in products)


def test_traffic_lookup_follows_the_recorded_kernel_hash():
    with open(os.path.join(ROOT, "profiles", "fused_gemm_llama8b_attn.json")) as f:
        side = json.load(f)
    sha, dram = side["kernel_source_sha256"], float(side["dram_bytes_per_launch_avg"])
    # the sidecar belongs to a summary that exists beside it
    assert os.path.exists(os.path.join(ROOT, "profiles", side["summary"]))
    assert bench.traffic_from_profile(sha) == dram
    assert bench.traffic_from_profile("0" * 64) is None
    # the hash covers a non-empty stretch of the kernel source
    assert re.fullmatch(r"[0-9a-f]{64}", bench.fused_kernel_source_sha() or "")


def test_peaks_come_from_the_measured_file():
    p = bench.load_peaks()
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        m = json.load(open(path))
        assert p["source"] == "measured"
        assert p["hbm_gbs"] == m["hbm_gbs"] and p["bf16_tflops"] == m["bf16_tflops"]
    else:
        assert p["source"] == "fallback"


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` (the oracle on this host's cores) prints one JSON line with
    the benchmark contract's keys, on the same metric and workload as the GPU arm."""
    import subprocess
    import sys
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert (d["steps"], d["warmup"], d["n_gpus"]) == (1, 3, 1)
    assert d["config"]["workload"] == bench.WORKLOAD and d["vs_baseline"] is None and d["data"] == "synthetic"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == bench.host_threads() and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == "TFLOP/s"
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_cpu_baseline_reports_one_thread_and_every_thread():
    """The oracle timed on one host thread and on all of them, the core count stated, on the
    small layer (whole-matrix quantize + dequantize, a few tokens of the layer)."""
    import oracle
    from bit_nf4_quantized_36_b300 import synth
    inp = synth.tiny_inputs()
    M, N, K = inp.shape
    ref = oracle.nf4_quantize(inp.W)
    What = oracle.nf4_dequantize(ref["packed"], ref["qcode"], ref["c2"], ref["mu"], N, K)
    cb = bench.oracle_baseline(inp, What, bench.layer_flops(M, N, K, inp.A.shape[0]), tokens=2)
    assert cb["kind"] == "oracle" and cb["cores"] == bench.host_threads() >= 1
    assert cb["value"] > 0 and cb["single_core"]["value"] > 0 and cb["single_core"]["cores"] == 1
    assert "whole" in cb["sample"] and "not sampled" in cb["sample"]


def test_run_threads_runs_every_job_once():
    seen = []
    out = bench.run_threads([lambda i=i: seen.append(i) or i * i for i in range(7)], 3)
    assert out == [i * i for i in range(7)] and sorted(seen) == list(range(7))
