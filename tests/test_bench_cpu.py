"""Host-side logic of bench.py, on CPU: which workloads are timed after an L2
flush, what the line's `l2` note says, and where the roofline peaks come from."""
import json
import os
from types import SimpleNamespace

import bench
from paged_kv_attention_02_gb300 import workloads as wl


def _sized(kv_bytes, q_bytes=1 << 20, table_bytes=1 << 16):
    """A stand-in workload with arrays of the given sizes (only .nbytes is read)."""
    half = SimpleNamespace(nbytes=kv_bytes // 2)
    return SimpleNamespace(k_pool=half, v_pool=half, q=SimpleNamespace(nbytes=q_bytes),
                           page_table=SimpleNamespace(nbytes=table_bytes))


def test_inputs_that_fit_twice_in_l2_are_flushed_and_larger_ones_are_not():
    assert bench.fits_l2(_sized(1 << 20))                        # the tiny decode's 1 MB pool
    assert bench.fits_l2(_sized(34 * 10**6, q_bytes=17 * 10**6))  # a prefill chunk's pools and rows
    assert not bench.fits_l2(_sized(4_500 * 10**6))              # the batched decode's pools
    edge = 2 * bench.L2_BYTES
    assert not bench.fits_l2(_sized(edge, q_bytes=0, table_bytes=0))
    assert bench.fits_l2(_sized(edge - 2, q_bytes=0, table_bytes=0))


def test_the_flush_buffer_is_larger_than_l2():
    assert bench.FLUSH_BYTES > bench.L2_BYTES


def test_the_l2_note_names_the_method_that_ran():
    w = wl.make_workload("tiny_decode")
    assert bench.workload_config(w)["l2"] == bench.L2_FLUSHED
    assert bench.workload_config(w, l2="host")["l2"] == "host"
    big = _sized(4_500 * 10**6)
    assert bench.fits_l2(big) is False
    assert "exceed" in bench.L2_LARGE and "flush" in bench.L2_FLUSHED


def test_roofline_peaks_come_from_the_measured_file():
    with open(os.path.join(bench.ROOT, "MEASURED_PEAKS.json")) as f:
        peaks = json.load(f)
    assert bench.hbm_peak() == (float(peaks["hbm_gbs"]), "measured")
    assert bench.tensor_peak() == (float(peaks["bf16_tflops"]), "measured")


def test_traffic_figures_name_existing_kernel_sources():
    # each recorded ncu traffic figure is tied to files that exist, and is
    # reported only while they hash to the recorded value
    csrc = os.path.join(bench.ROOT, "paged_kv_attention_02_gb300", "csrc")
    for name, tr in bench.NCU_TRAFFIC.items():
        assert name in wl.CONFIGS
        assert tr["bytes_per_launch"] > 0 and len(tr["src_sha256"]) == 64
        for f in tr["sources"]:
            assert os.path.exists(os.path.join(csrc, f)), f
    assert bench.kernel_source_hash(["ptx.cuh"]) != bench.kernel_source_hash(["tc05.cuh"])


def test_launches_per_step_counts_every_kernel_of_a_call():
    # shape-only stand-ins (the real workloads hold GBs): the split kernel, its combine
    # when a sequence can span splits, the order kernel of a sorted call, the tile map of
    # a ragged one
    def shape(name):
        c = wl.CONFIGS[name]
        return SimpleNamespace(cfg=c, groups=c.groups, pages_per_seq=c.pages_per_seq,
                               ragged=c.q_lens is not None, tree_mask=object() if c.tree else None)
    assert bench.launches_per_step(shape("tiny_decode")) == 1      # one split per sequence
    assert bench.launches_per_step(shape("batched_decode")) == 2   # split order: kernel + combine
    assert bench.launches_per_step(shape("spec_verify")) == 3      # + the order kernel
    assert bench.launches_per_step(shape("tree_verify")) == 3
    assert bench.launches_per_step(shape("hybrid_decode_fp8")) == 3
    assert bench.launches_per_step(shape("mixed_step")) == 3       # tile map + kernel + combine
    assert bench.launches_per_step(shape("prefill_chunk")) == 1
