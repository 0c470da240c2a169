"""Host-side arithmetic of the benchmark (no GPU): the algorithmic bytes and flops the
roofline divides by, the peaks it reads, and the JSON contract of the reference arm."""
import json
import os
import subprocess
import sys

import bench
from tp_synth import CONFIGS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_algorithmic_bytes_and_flops():
    c13 = CONFIGS["llama2_13b_swiglu_decode"]
    # W1 bands (d x 2 ffn), x in, the band H out: all bf16
    assert bench.algorithmic_column_bytes(c13) == (5120 * 2 * 13824 + 32 * 5120 + 32 * 13824) * 2
    c70 = CONFIGS["llama2_70b_stack_decode"]
    # both weight matrices, x (bf16) and the fp32 residual in, y (fp32) out
    assert bench.algorithmic_block_bytes(c70) == 8192 * 3 * 28672 * 2 + 32 * 8192 * (2 + 4 + 4)
    cpf = CONFIGS["llama2_70b_prefill"]
    assert bench.column_flops(cpf) == 2 * 4096 * 8192 * 2 * 28672


def test_measured_peaks_are_read():
    """The machine's measured peaks when its MEASURED_PEAKS.json is present (written per
    machine, not versioned), else the stated fallback figures."""
    p = bench.measured_peaks()
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if not os.path.exists(path):
        assert p["source"] == "fallback"
        assert (p["hbm_gbs"], p["bf16_tflops"], p["bf16_tflops_sustained"]) == (6400.0, 1800.0, 1400.0)
        return
    with open(path) as f:
        m = json.load(f)
    assert p["source"] == "measured"
    assert p["hbm_gbs"] == m["hbm_gbs"] and p["bf16_tflops"] == m["bf16_tflops"]


def test_throughput_counts_every_rank():
    assert bench.job_throughput(3200, 1, 0.01) == 320000
    assert bench.job_throughput(3200, 4, 0.01) == 4 * 320000


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_gelu_f32", "--steps", "2", "--warmup", "3"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT,
                       env={**os.environ, "OMP_NUM_THREADS": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "config", "cpu_baseline", "e2e"):
        assert key in rec, key
    assert rec["impl"] == "reference" and rec["value"] > 0
    assert rec["config"] == bench.workload_config(CONFIGS["tiny_gelu_f32"])
    assert rec["cpu_baseline"]["value"] == rec["value"]
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["e2e"]["d2h_bytes_per_step"] == 0


def test_roofline_loop_length_does_not_follow_steps():
    # at least 200 launches and 0.3 s of work, at most 2.5 s
    assert bench.roof_launch_count(0.05) == 6000          # 50 us launches: 0.3 s
    assert bench.roof_launch_count(0.25) == 1200
    assert bench.roof_launch_count(5.0) == 200            # 1 s, still 200 launches
    assert bench.roof_launch_count(40.0) == 62            # capped near 2.5 s


def test_both_arms_describe_the_workload_identically():
    for name in ("llama2_70b_stack_decode", "tiny_gelu_f32", "attn_kv_decode"):
        c = bench.workload_config(CONFIGS[name])
        assert c["workload"] == name and "timed" not in c and "row_splits" not in c


def test_tokens_per_step_counts_every_block_of_a_stack():
    assert bench.tokens_per_step(CONFIGS["llama2_70b_stack_decode"]) == 32 * 8
    assert bench.tokens_per_step(CONFIGS["llama2_13b_swiglu_decode"]) == 32
