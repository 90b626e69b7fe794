"""CPU checks of bench.py's arithmetic and of its reference-arm JSON line.

The per-token algorithmic bytes and tensor work are the figures the roofline fractions are
taken against (q, k, g, v, o and beta per token and head, plus the fp32 state; the chunk
form's products at C = 64); they are pinned here to their closed forms at d = 128.
"""
import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_algorithmic_bytes_of_the_prefill_workload():
    tokens, H, d = 4 * 8192, 32, 128
    per_tok = (3 * d + 2 * d) * 2 + 2            # q, k, g, v, o in bf16, and beta
    assert per_tok == 1282
    got = bench.algorithmic_bytes(tokens, H, d, d, 2, 4, False)
    assert got == tokens * H * per_tok + 4 * H * d * d * 4
    assert got == 1352663040
    # a given initial state is read as well as the final state written
    assert bench.algorithmic_bytes(tokens, H, d, d, 2, 4, True) == got + 4 * H * d * d * 4


def test_chunk_flops_per_token():
    # 3 state products of 2 d^2 (K S, Q S, Kp^T U) + A, M, T(beta K), T(beta V), M U at C = 64
    assert bench.chunk_flops(1, 1, 128, 128) == 6 * 128 * 128 + 64 * (4 * 128 + 3 * 128)
    assert bench.chunk_flops(1, 1, 128, 128) == 155648


def test_reference_arm_prints_the_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--ref-step-s", "0.2"], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference"
    assert line["config"]["workload"] == "prefill_b4_h32_t8192"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["value"] > 0 and line["e2e"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
