#!/usr/bin/env python
"""Benchmark of paged-KV attention on one GB300 per process.

Workload (default): the batched decode step -- 256 sequences x rows=1,
n_head=32, n_head_kv=8, head_dim=128, page_size=16, context lengths uniform in
[512, 8192], bf16 KV ~ N(0,1), random-permutation page table (seeded).  A step
is one rad_attn_paged call over the whole batch (split kernel + in-kernel
combine), replayed from a CUDA graph as a decode program is.

Metric: KV bytes read per second (GB/s), the algorithmic bytes of one call --
every visible key's K and V rows for every KV head, plus page-table entries
(and per-page scales for fp8) -- divided by the device time of a call.  Also
reported: context tokens attended per second, rows per second, and the
fraction of the measured HBM copy bandwidth.

Under torchrun (N > 1) every rank runs its own independent batch (its own
seed): the op shards by sequence with no data-path exchange, so scaling is
weak; `value` is the sum of all ranks' bytes over the slowest rank's time.

--impl reference times the fp64 CPU oracle (the only other implementation of
the op there is) on a bounded sample of the same workload, on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import glob
import json
import os
import statistics
import subprocess
import sys
import threading
import time
from dataclasses import replace

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_attention_02_gb300 import workloads as wl  # noqa: E402

METRIC = "paged-decode KV GB/s and seq-tokens/s (fraction of GB300 HBM peak) at 1 GPU"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0

# DRAM traffic per launch of the dominant kernel plus the combine (and the
# item-order kernel where the call runs one), from the committed ncu captures
# (a capture of fewer sequences scaled by the KV bytes where the workload is
# too large to capture), valid only while the sources that kernel is built
# from hash to `src_sha256`.
_BF16_SPLIT_SOURCES = ("split_bf16_tc05.cuh", "sched.cuh", "attn_tile.cuh", "tc05.cuh", "ptx.cuh", "combine.cuh",
                       "launch.cuh", "tile_configs.cuh", "kern_split_bf16_tc05.cu", "kern_split_bf16_tc05_d256.cu")
_E4M3_SPLIT_SOURCES = ("split_tc05.cuh", "sched.cuh", "attn_tile.cuh", "tc05.cuh", "ptx.cuh", "combine.cuh",
                       "launch.cuh", "tile_configs.cuh", "kern_split_tc05.cu", "kern_split_tc05_d256.cu")
_BF16_PREFILL_SOURCES = ("prefill_pair.cuh", "prefill_tc05.cuh", "attn_tile.cuh", "tc05.cuh", "ptx.cuh",
                         "tile_configs.cuh", "kern_prefill_pair.cu", "kern_prefill_tc05_d256.cu")
_FP8_PREFILL_SOURCES = ("prefill_fp8.cuh", "prefill_tc05.cuh", "sched.cuh", "attn_tile.cuh", "tc05.cuh", "ptx.cuh",
                        "tile_configs.cuh", "kern_prefill_fp8.cu", "kern_prefill_fp8_d256.cu")
NCU_TRAFFIC: dict[str, dict] = {
    "batched_decode": {"bytes_per_launch": 4522011744, "sources": _BF16_SPLIT_SOURCES,
                       "src_sha256": "8bed5860df4e7fd28ba80b09164f9fc677126ba6cd8fe4255139580dad95172c",
                       "capture": "64 sequences, scaled by the KV bytes (x 4.3412)"},
    "hybrid_decode": {"bytes_per_launch": 2284209889, "sources": _BF16_SPLIT_SOURCES,
                      "src_sha256": "8bed5860df4e7fd28ba80b09164f9fc677126ba6cd8fe4255139580dad95172c",
                      "capture": "32 sequences, scaled by the KV bytes (x 3.8372)"},
    "spec_verify": {"bytes_per_launch": 1246796429, "sources": _E4M3_SPLIT_SOURCES,
                    "src_sha256": "905400cfdeb263ce7ff3e9ed8df80ba87a68170b8ccfcd213d85a184c767a7d2",
                    "capture": "16 sequences, scaled by the KV bytes (x 4.4698)"},
    "tiny_decode": {"bytes_per_launch": 679168, "sources": _BF16_SPLIT_SOURCES,
                    "src_sha256": "8bed5860df4e7fd28ba80b09164f9fc677126ba6cd8fe4255139580dad95172c",
                    "capture": "the whole workload"},
    "prefill_chunk": {"bytes_per_launch": 51_253_760, "sources": _BF16_PREFILL_SOURCES,
                      "src_sha256": "c8486b490e146bf5cc9cf675cb49b485f11b6a5be0116df2fb05e21946855e8f",
                      "capture": "the whole workload (K/V re-reads served by L2)"},
    "prefill_chunk_fp8": {"bytes_per_launch": 33_652_224, "sources": _FP8_PREFILL_SOURCES,
                          "src_sha256": "bfdae5aaa1f5c0033858df83a8b67ba4fb4a94e94246b34d21d02d9d53ea2373",
                          "capture": "the whole workload (K/V re-reads served by L2)"},
    "prefill_chunk_d256": {"bytes_per_launch": 33_628_928, "sources": _BF16_PREFILL_SOURCES,
                           "src_sha256": "c8486b490e146bf5cc9cf675cb49b485f11b6a5be0116df2fb05e21946855e8f",
                           "capture": "the whole workload (K/V re-reads served by L2)"},
    "prefill_chunk_d256_fp8": {"bytes_per_launch": 25_282_048, "sources": _FP8_PREFILL_SOURCES,
                               "src_sha256": "bfdae5aaa1f5c0033858df83a8b67ba4fb4a94e94246b34d21d02d9d53ea2373",
                               "capture": "the whole workload (K/V re-reads served by L2)"},
    "hybrid_decode_fp8": {"bytes_per_launch": 1355983132, "sources": _E4M3_SPLIT_SOURCES,
                          "src_sha256": "905400cfdeb263ce7ff3e9ed8df80ba87a68170b8ccfcd213d85a184c767a7d2",
                          "capture": "32 sequences, scaled by the KV bytes (x 4.1277)"},
}


def kernel_source_hash(names=None) -> str:
    """sha256 over the named files of csrc/ (all of them by default), in name order."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_attention_02_gb300", "csrc")
    paths = sorted(glob.glob(os.path.join(csrc, "*"))) if names is None else \
        [os.path.join(csrc, n) for n in sorted(names)]
    for p in paths:
        with open(p, "rb") as f:
            h.update(os.path.basename(p).encode())
            h.update(f.read())
    return h.hexdigest()


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="batched_decode", choices=sorted(wl.CONFIGS))
    ap.add_argument("--no-graph", action="store_true", help="launch eagerly instead of graph replay")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle CPU-baseline budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--max-groups", type=int, default=0,
                    help="draw only N sequences (a smaller pool, for profiling)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only --workload, not the other configurations beside it")
    return ap.parse_args()


# ---------------------------------------------------------------- distributed plumbing
def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def rank_config(name: str, rank: int) -> wl.Config:
    """Each rank draws its own batch (weak scaling): rank r uses seed + 1000 r."""
    cfg = wl.CONFIGS[name]
    return cfg if rank == 0 else replace(cfg, seed=cfg.seed + 1000 * rank)


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, period_ms: int = 50):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 f"-lms={period_ms}", f"-i={device_index}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        win = [p for (t, p) in self.samples if t0 <= t <= t1]
        if not win and self.samples:   # a very short window: the nearest samples
            win = [min(self.samples, key=lambda s: abs(s[0] - (t0 + t1) / 2))[1]]
        mhz = [num(p[1]) for p in win if num(p[1]) is not None]
        mx = [num(p[2]) for p in win if num(p[2]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for p in win:
            for i, n in enumerate(names):
                if p[5 + i].lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(mhz) if mhz else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(win)}


# ---------------------------------------------------------------- peaks
def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


FALLBACK_BF16_TFLOPS = 1900.0


def tensor_peak():
    """Dense bf16 tensor TFLOP/s: the measured burst figure (a kernel timed on
    its own), else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, "fallback"


# ---------------------------------------------------------------- oracle timing (CPU)
def time_oracle(w: wl.Workload, groups_idx) -> tuple[float, int]:
    import oracle
    sub = w.select_groups(groups_idx)
    extra = {}
    q = sub.q
    if sub.ragged:
        q, cu, mask = sub.packed()
        extra = dict(cu_seqlens=cu, tree_mask=mask)
    elif sub.tree_mask is not None:
        extra = dict(tree_mask=sub.tree_mask)
    t0 = time.perf_counter()
    oracle.attn_paged_rows(q, sub.k_pool, sub.v_pool, sub.page_table, sub.seq_lens,
                           k_scales=sub.k_scales, v_scales=sub.v_scales, **extra, **sub.call_args())
    return time.perf_counter() - t0, wl.kv_bytes(sub)


def cpu_baseline(w: wl.Workload, budget_s: float) -> dict:
    import oracle
    oracle.build()
    t1, _ = time_oracle(w, [0])
    n = int(max(1, min(w.groups, budget_s / max(t1, 1e-3))))
    idx = list(range(n))
    dt, nbytes = time_oracle(w, idx)
    return {"value": nbytes / dt / 1e9, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"{n} of {w.groups} sequences (all rows and heads), one oracle call, fp64",
            "seconds": round(dt, 3)}


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = wl.make_workload(rank_config(args.workload, 0))
    t1, _ = time_oracle(w, [0])
    per_step = max(0.2, min(3.0, 150.0 / max(1, args.steps + args.warmup)))
    n = int(max(1, min(w.groups, per_step / max(t1, 1e-3))))
    rng = np.random.default_rng(12345)
    for _ in range(args.warmup):
        time_oracle(w, rng.choice(w.groups, n, replace=False))
    total_t, total_b = 0.0, 0
    for _ in range(args.steps):
        dt, nb = time_oracle(w, rng.choice(w.groups, n, replace=False))
        total_t += dt
        total_b += nb
    value = total_b / total_t / 1e9
    cores = oracle.max_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w, l2="not applicable: the oracle runs on the host cores"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{n} random sequences of {w.groups} per step, all rows and heads"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm
L2_BYTES = 129 * 10**6        # GB300 L2
FLUSH_BYTES = 256 * 2**20     # written before each timed step of a workload that fits in L2
L2_LARGE = "inputs larger than L2 (no flush): the KV pools exceed the 129 MB L2"
L2_FLUSHED = ("inputs smaller than twice the 129 MB L2: a 256 MB buffer is written before every timed "
              "step (L2 flush) and each step is timed alone, the flush outside its events")


def fits_l2(w: wl.Workload) -> bool:
    """Whether the step's inputs could stay resident in L2 between steps."""
    return int(w.k_pool.nbytes + w.v_pool.nbytes + w.q.nbytes + w.page_table.nbytes) < 2 * L2_BYTES


def workload_config(w: wl.Workload, l2: str | None = None) -> dict:
    c = w.cfg
    rows = f"rows {c.q_lens} (ragged, cu_seqlens)" if c.q_lens else f"rows={c.rows}"
    tree = f", {'ragged ' if c.q_lens else ''}draft trees (random forests, tree_mask)" if c.tree else ""
    return {"workload": f"{c.name}: {w.groups} seqs x {rows}{tree}, n_head={c.n_head}, "
                        f"n_head_kv={c.n_head_kv}, head_dim={c.head_dim}, page_size={c.page_size}, "
                        f"ctx {c.lens}, {'fp8-e4m3' if c.kv_dtype else 'bf16'} KV, seed {c.seed}",
            "groups": w.groups, "rows": c.rows, "n_head": c.n_head, "n_head_kv": c.n_head_kv,
            "head_dim": c.head_dim, "page_size": c.page_size, "num_pages": w.num_pages,
            "kv_pool_bytes": int(w.k_pool.nbytes + w.v_pool.nbytes),
            "l2": l2 if l2 is not None else (L2_FLUSHED if fits_l2(w) else L2_LARGE)}


# The configurations of the op's headline measurement: the batched decode is the
# metric's own configuration, the others are measured beside it in the same run.
PER_CONFIG = ["tiny_decode", "batched_decode", "hybrid_decode", "spec_verify", "prefill_chunk"]
PREWINDOW_S = 1.0   # untimed replays before a timed window, with the clock sampler running


class Step:
    """One workload on the device: its inputs, one call of the op through the
    C ABI, and (unless disabled) the call captured in a CUDA graph."""

    def __init__(self, w: wl.Workload, dev, use_graph: bool):
        from paged_kv_attention_02_gb300 import binding as b
        self.w = w
        c = w.cfg
        self.fp8 = c.kv_dtype == wl.KV_FP8_E4M3

        def to_dev(a, as_bf16=False):
            t = torch.from_numpy(np.ascontiguousarray(a))
            if as_bf16:
                t = t.view(torch.int16).view(torch.bfloat16)
            return t.to(dev)

        # ragged and tree calls go through rad_attn_paged_ex with their offsets / mask words
        self.general = w.ragged or w.tree_mask is not None
        q_np, cu_np, mask_np = w.q, None, None
        if w.ragged:
            q_np, cu_np, mask_np = w.packed()
        elif w.tree_mask is not None:
            mask_np = w.tree_mask.reshape(-1)
        self.q_np, self.cu_np, self.mask_np = q_np, cu_np, mask_np
        self.q = to_dev(q_np.view(np.int16), True)
        self.cu = None if cu_np is None else to_dev(cu_np)
        self.mask = None if mask_np is None else to_dev(mask_np.view(np.int32))
        self.total_rows = int(q_np.shape[0]) if w.ragged else 0
        self.k = to_dev(w.k_pool) if self.fp8 else to_dev(w.k_pool.view(np.int16), True)
        self.v = to_dev(w.v_pool) if self.fp8 else to_dev(w.v_pool.view(np.int16), True)
        self.ks = to_dev(w.k_scales) if self.fp8 else None
        self.vs = to_dev(w.v_scales) if self.fp8 else None
        self.table = to_dev(w.page_table)
        self.lens = to_dev(w.seq_lens)
        self.out = torch.empty(tuple(self.q.shape), dtype=torch.bfloat16, device=dev)
        shape = b.shape_args(w.groups, c.rows, c.n_head, c.n_head_kv, c.head_dim, c.page_size, w.pages_per_seq,
                             c.kv_dtype, ragged=w.ragged, tree=w.tree_mask is not None, total_rows=self.total_rows)
        self.ws = torch.empty(max(1, b.ex_workspace_bytes(shape)), dtype=torch.uint8, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.stream = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(self.stream):
            self.call()
        torch.cuda.synchronize()
        assert int(self.err.item()) == 0, f"{c.name}: error word {int(self.err.item())}"
        self.step = self.call
        if use_graph:
            self.graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.graph, stream=self.stream):
                self.call()
            self.step = self.graph.replay
        # a workload whose inputs fit in L2 is timed step by step, each after an L2 flush
        self.flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev) if fits_l2(w) else None

    def call(self, qq=None, tt=None, ll=None, oo=None, cc=None, mm=None):
        from paged_kv_attention_02_gb300 import binding as b
        c = self.w.cfg
        qq = self.q if qq is None else qq
        tt = self.table if tt is None else tt
        ll = self.lens if ll is None else ll
        oo = self.out if oo is None else oo
        if self.general:
            b.attn_paged_general(qq, self.k, self.v, tt, ll, rows=c.rows, n_head=c.n_head, n_head_kv=c.n_head_kv,
                                 head_dim=c.head_dim, page_size=c.page_size, scale=c.scale, kv_dtype=c.kv_dtype,
                                 k_scales=self.ks, v_scales=self.vs, cu_seqlens=self.cu if cc is None else cc,
                                 tree_mask=self.mask if mm is None else mm, total_rows=self.total_rows, out=oo,
                                 workspace=self.ws, err_word=self.err, stream=self.stream)
            return
        b.attn_paged(qq, self.k, self.v, tt, ll, rows=c.rows, n_head=c.n_head, n_head_kv=c.n_head_kv,
                     head_dim=c.head_dim, page_size=c.page_size, scale=c.scale, kv_dtype=c.kv_dtype,
                     k_scales=self.ks, v_scales=self.vs, out=oo, workspace=self.ws, err_word=self.err,
                     stream=self.stream)

    def timed(self, fn, steps: int) -> float:
        """ms per step of fn over `steps` steps on the step's stream (CUDA
        events on that stream)."""
        st = self.stream
        if self.flush_buf is None:
            a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(st)
            with torch.cuda.stream(st):
                for _ in range(steps):
                    fn()
            z.record(st)
            torch.cuda.synchronize()
            return a.elapsed_time(z) / steps
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        with torch.cuda.stream(st):
            for a, z in pairs:
                self.flush_buf.fill_(1)
                a.record(st)
                fn()
                z.record(st)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(z) for a, z in pairs) / steps

    def prewindow(self, seconds: float):
        """Untimed replays of the step (with the flush where the step is
        timed after one) for about `seconds`, so the clock sampler sees the
        GPU under this load before the timed window."""
        with torch.cuda.stream(self.stream):
            self.step()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        self.timed(self.step, 1)
        one = max(time.perf_counter() - t0, 1e-5)
        n = int(min(200000, max(1, seconds / one)))
        t_end = time.perf_counter() + seconds
        while time.perf_counter() < t_end:
            with torch.cuda.stream(self.stream):
                for _ in range(min(n, 2000)):
                    if self.flush_buf is not None:
                        self.flush_buf.fill_(1)
                    self.step()
            torch.cuda.synchronize()


def measure_device(st: Step, steps: int, warmup: int, world: int, sampler: ClockSampler | None) -> dict:
    """Warm-up, an untimed pre-window under the clock sampler, then exactly
    `steps` timed replays bracketed by a barrier and a synchronize."""
    with torch.cuda.stream(st.stream):
        for _ in range(max(3, warmup)):
            st.step()
    torch.cuda.synchronize()
    pre0 = time.time()
    st.prewindow(PREWINDOW_S)
    torch.cuda.synchronize()
    barrier(world)
    wall0 = time.time()
    ms = st.timed(st.step, steps)
    wall1 = time.time()
    barrier(world)
    assert int(st.err.item()) == 0
    clocks = None
    if sampler is not None:
        time.sleep(0.12)   # the sample taken at the window's end
        timed = sampler.summary(wall0, wall1)
        pre = sampler.summary(pre0, wall0)
        clocks = {"sm_mhz": timed["sm_mhz"], "sm_max_mhz": timed["sm_max_mhz"],
                  "reasons": sorted(set(timed["reasons"]) | set(pre["reasons"])), "samples": timed["samples"],
                  "prewindow": dict(pre, seconds=round(wall0 - pre0, 3),
                                    note="untimed replays of the same step right before the timed window")}
        both = sampler.summary(pre0, wall1)
        clocks["samples_under_load"] = both["samples"]
        clocks["sm_mhz_under_load"] = both["sm_mhz"]
    return {"ms": ms, "clocks": clocks}


def roofline_of(w: wl.Workload, ms: float, desc: str) -> dict:
    nbytes = wl.kv_bytes(w) + wl.aux_bytes(w)
    tr = NCU_TRAFFIC.get(w.cfg.name)
    traffic = tr["bytes_per_launch"] if tr and tr.get("src_sha256") == kernel_source_hash(tr["sources"]) else None
    if "split_len=0" in desc:
        # a prefill chunk (no splits): bound by the tensor pipe, not by HBM
        tpeak, tpeak_src = tensor_peak()
        flops = wl.attended_flops(w)
        t_ach = flops / (ms * 1e-3) / 1e12
        return {"bound": "tensor", "achieved": t_ach, "peak": tpeak, "unit": "TFLOP/s", "frac": t_ach / tpeak,
                "traffic": traffic, "peak_source": tpeak_src, "algorithmic_flops_per_launch": flops,
                "kv_bytes_per_launch": nbytes}
    peak, peak_src = hbm_peak()
    achieved = nbytes / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": traffic, "peak_source": peak_src, "algorithmic_bytes_per_launch": nbytes,
            "kv_bytes_per_launch": wl.kv_bytes(w), "aux_bytes_per_launch": wl.aux_bytes(w)}


def config_entry(w: wl.Workload, ms: float, clocks, graph: bool) -> dict:
    """One configuration's figures, for the per_config table."""
    desc = describe(w)
    rl = roofline_of(w, ms, desc)
    nbytes = wl.kv_bytes(w) + wl.aux_bytes(w)
    return {"workload": workload_config(w)["workload"], "ms_per_step": ms,
            "kv_gbs": nbytes / (ms * 1e-3) / 1e9,
            "seq_tokens_per_s": float(w.seq_lens.astype(np.int64).sum()) / (ms * 1e-3),
            "rows_per_s": float(w.rows_of().sum()) / (ms * 1e-3),
            "roofline": {k: rl[k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic")},
            "l2": L2_FLUSHED if fits_l2(w) else L2_LARGE, "graph": graph, "clocks": clocks,
            "kernel": desc.split(" family=")[0]}


def make_bench_workload(name: str, rank: int, max_groups: int = 0) -> wl.Workload:
    cfg = rank_config(name, rank)
    subset = max_groups and max_groups < cfg.groups
    if subset and not cfg.q_lens:
        cfg = replace(cfg, groups=max_groups)
    w = wl.make_workload(cfg)
    if subset and cfg.q_lens:
        # a ragged step keeps its mix: sequences spread evenly over the call order
        w = wl.compact_pool(
            w.select_groups(np.unique(np.linspace(0, cfg.groups - 1, max_groups).round().astype(int))))
    return w


def run_ours(args, rank, world, local):
    from paged_kv_attention_02_gb300.build import build_library

    build_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = make_bench_workload(args.workload, rank, args.max_groups)
    c = w.cfg
    fp8 = c.kv_dtype == wl.KV_FP8_E4M3
    st = Step(w, dev, not args.no_graph)

    sampler = ClockSampler(local)
    # ---- device-resident timing
    dm = measure_device(st, args.steps, args.warmup, world, sampler)
    ms = dm["ms"]

    # ---- end to end: per-step inputs from pinned host memory, result back to host
    q_h = torch.from_numpy(st.q_np.view(np.int16)).view(torch.bfloat16).pin_memory()
    t_h = torch.from_numpy(w.page_table).pin_memory()
    l_h = torch.from_numpy(w.seq_lens).pin_memory()
    o_h = torch.empty(st.out.shape, dtype=torch.bfloat16).pin_memory()
    q_d, t_d, l_d = torch.empty_like(st.q), torch.empty_like(st.table), torch.empty_like(st.lens)
    # per-step row offsets and mask words travel with the step's other inputs
    c_h = None if st.cu is None else torch.from_numpy(st.cu_np).pin_memory()
    m_h = None if st.mask is None else torch.from_numpy(st.mask_np.view(np.int32)).pin_memory()
    c_d = None if st.cu is None else torch.empty_like(st.cu)
    m_d = None if st.mask is None else torch.empty_like(st.mask)

    def e2e_step():
        q_d.copy_(q_h, non_blocking=True)
        t_d.copy_(t_h, non_blocking=True)
        l_d.copy_(l_h, non_blocking=True)
        if c_d is not None:
            c_d.copy_(c_h, non_blocking=True)
        if m_d is not None:
            m_d.copy_(m_h, non_blocking=True)
        st.call(q_d, t_d, l_d, st.out, c_d, m_d)
        o_h.copy_(st.out, non_blocking=True)

    with torch.cuda.stream(st.stream):
        for _ in range(max(3, args.warmup)):
            e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = st.timed(e2e_step, args.steps)
    barrier(world)
    h2d = q_h.numel() * 2 + t_h.numel() * 4 + l_h.numel() * 4
    h2d += (0 if c_h is None else c_h.numel() * 4) + (0 if m_h is None else m_h.numel() * 4)
    d2h = o_h.numel() * 2

    nbytes = wl.kv_bytes(w) + wl.aux_bytes(w)
    tokens = int(w.seq_lens.astype(np.int64).sum())
    ms_max = reduce_max(ms, world)
    e2e_max = reduce_max(e2e_ms, world)
    tot_bytes = reduce_sum(float(nbytes), world)
    tot_tokens = reduce_sum(float(tokens), world)
    tot_rows = reduce_sum(float(w.rows_of().sum()), world)

    # ---- the other configurations, device-resident, one GPU only
    per_config = None
    if world == 1 and not args.no_per_config and not args.max_groups:
        per_config = {args.workload: config_entry(w, ms, dm["clocks"], not args.no_graph)}
        del st
        torch.cuda.empty_cache()
        for name in PER_CONFIG:
            if name == args.workload:
                continue
            wo = make_bench_workload(name, rank)
            so = Step(wo, dev, not args.no_graph)
            mo = measure_device(so, args.steps, args.warmup, world, sampler)
            per_config[name] = config_entry(wo, mo["ms"], mo["clocks"], not args.no_graph)
            del so, wo
            torch.cuda.empty_cache()
    sampler.stop()
    if rank != 0:
        return
    value = tot_bytes / (ms_max * 1e-3) / 1e9
    peak, _ = hbm_peak()
    desc = describe(w)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp8e4m3" if fp8 else "bf16", "data": "synthetic",
        "config": dict(workload_config(w), graph=not args.no_graph),
        "seq_tokens_per_s": tot_tokens / (ms_max * 1e-3),
        "rows_per_s": tot_rows / (ms_max * 1e-3),
        "hbm_frac": value / world / peak,
        "roofline": roofline_of(w, ms, desc),
        "clocks": dm["clocks"],
        "e2e": {"value": tot_bytes / (e2e_max * 1e-3) / 1e9, "unit": UNIT, "ms_per_step": e2e_max,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "note": "KV pools resident (persistent state); q, page table, seq_lens in and out back per step"},
        "gpu_launches": args.steps * launches_per_step(w),
        "kernel": desc,
    }
    if per_config is not None:
        line["per_config"] = per_config
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def describe(w) -> str:
    """The library's description of the kernels a call of this workload runs."""
    from paged_kv_attention_02_gb300 import binding as b
    c = w.cfg
    return b.ex_describe(b.shape_args(w.groups, c.rows, c.n_head, c.n_head_kv, c.head_dim, c.page_size,
                                      w.pages_per_seq, c.kv_dtype, ragged=w.ragged,
                                      tree=w.tree_mask is not None))


def launches_per_step(w) -> int:
    """Kernels one call launches: the attention kernel, plus the split combine
    when a sequence of the call's capacity can span more than one split, plus
    the tile map of a ragged call, plus the item-order kernel of a split call
    that runs one (a uniform call with more than two items per SM)."""
    import torch
    c = w.cfg
    desc = describe(w)
    kernels = (desc.count("attn_tile family") + desc.count("attn_split_tc05 ") + desc.count("attn_split_bf16_tc05 ")
               + desc.count("attn_prefill_tc05 "))
    split_len = int(desc.split("split_len=")[1].split()[0])
    combines = desc.count("attn_combine") if split_len > 0 and w.pages_per_seq * c.page_size > split_len else 0
    order = 0
    if "item_order" in desc:
        m = c.rows * (c.n_head // c.n_head_kv)
        qt = int(desc.split("tile_rows=")[1].split()[0])
        n_items = w.groups * c.n_head_kv * (-(-m // qt)) * (-(-(w.pages_per_seq * c.page_size) // split_len))
        sms = torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 152
        order = int(n_items > 2 * sms)
    return kernels + combines + order + int("ragged_tile_map" in desc)


def main():
    args = parse_args()
    rank, world, local = dist_init()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
