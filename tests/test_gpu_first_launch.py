"""The first launch of each kernel in a fresh process must be right too.

A process's first launch of a kernel is its slowest (the module is loaded
lazily, caches are cold), which is when a wait that passes on the parity of a
phase one too early shows: the tcgen05 prefill kernel once read O before the
PV products of a query tile had landed, on first launches only.  Each case
runs in its own child process and compares that process's first call with
the oracle."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, numpy as np
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
from gpu_util import DevWorkload, as_f64, assert_parity, oracle_rows
from paged_kv_attention_02_gb300 import workloads as wl
cfg = wl.Config({name!r}, *{args!r}, pages_per_seq={pps})
w = wl.make_workload(cfg, poison=True)
ref = oracle_rows(w, window={window}).out   # first, as a caller's own host work would be
dw = DevWorkload(w)
out, err = dw.run(window={window})          # the first launch of this process
assert err == 0, err
assert_parity(as_f64(out), ref, dw.fp8, {name!r})
print("ok")
"""

# (name, Config args after the name, pages_per_seq, window): the tcgen05
# prefill kernel with and without its window terms, the tcgen05 split kernel,
# the decode and verify tiles.
CASES = [
    ("prefill_tc_window", (3, 300, 8, 2, 128, 16, 0, 209, "fixed:300,1000,2500"), 160, 257),
    ("prefill_tc_plain", (2, 384, 8, 2, 128, 16, 0, 210, "fixed:384,2000"), 160, 0),
    ("split_tc05_verify", (6, 8, 32, 8, 128, 16, 1, 211, "fixed:8,900,2000,3100,40,5000"), 320, 0),
    ("tile_decode", (8, 1, 32, 8, 128, 16, 0, 212, "fixed:1,17,700,1025,2048,3000,4100,5000"), 320, 0),
    ("tile_verify_d256", (4, 8, 16, 2, 256, 32, 0, 213, "fixed:8,700,2100,4000"), 130, 0),
    ("prefill_fp8_window", (3, 300, 8, 2, 128, 16, 1, 214, "fixed:300,1000,2500"), 160, 257),
    ("prefill_fp8_plain", (2, 384, 8, 2, 128, 16, 1, 215, "fixed:384,2000"), 160, 0),
    ("prefill_d256_window", (2, 300, 16, 2, 256, 32, 0, 216, "fixed:300,1500"), 60, 257),
    ("prefill_d256_plain", (1, 384, 16, 2, 256, 32, 0, 217, "fixed:2000"), 70, 0),
    ("prefill_fp8_d256_window", (2, 300, 16, 2, 256, 32, 1, 218, "fixed:300,1500"), 60, 257),
    ("prefill_fp8_d256_plain", (1, 384, 16, 2, 256, 32, 1, 219, "fixed:2000"), 70, 0),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_first_launch_in_a_fresh_process_matches_oracle(case):
    name, args, pps, window = case
    code = CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"), name=name, args=args, pps=pps,
                        window=window)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-4000:]
