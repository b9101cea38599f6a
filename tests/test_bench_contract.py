"""The parts of bench.py that need no GPU: the reference arm's JSON line on
the smallest workload, the launch count it claims per call, and the byte
counts behind its rooflines."""
import importlib.util
import json
import os
import subprocess
import sys

import kda_inputs as KI

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_reference_arm_line_on_tiny_workload():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_T64_H1", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["dtype"] == "f64"
    assert line["value"] > 0 and line["unit"] == "tokens/s" and line["higher_is_better"]
    assert line["config"]["workload"] == "tiny_T64_H1"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s",
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


class _Args:
    recurrent_impl = None


def test_launches_per_call():
    b = load_bench()
    n = {name: b.launches_per_call(w, _Args) for name, w in KI.WORKLOADS.items()}
    # intra-chunk kernel, its exact-form companion, recurrent kernel
    assert n["fixed_T8192_H64"] == 3 and n["fixed_T8192_H96"] == 3
    assert n["varlen16_T8192_H64"] == 4            # + the cu_seqlens prologue
    assert n["long_T131072_H32"] == 5              # + the segment scan's maps and combine (P = 6)
    assert b.scan_segments(32, 8192, 152) == 6 and b.scan_segments(64, 512, 152) == 1
    args = _Args()
    args.recurrent_impl = 3                        # 64-token split: intra-chunk + recurrent
    assert b.launches_per_call(KI.WORKLOADS["long_T131072_H32"], args) == 2
    args.recurrent_impl = 4                        # 64-token fused: one cooperative kernel
    assert b.launches_per_call(KI.WORKLOADS["varlen16_T8192_H64"], args) == 2


def test_backward_byte_counts():
    b = load_bench()
    # q, k, v, dO bf16 + g, beta read; dq, dk, dv, dg, dbeta written (fp32)
    assert b.BWD_TOKEN_HEAD_BYTES == 4 * 256 + 512 + 4 + 4 * 512 + 4
    assert b.BWD_UNIT_BYTES == 3 * 65536
