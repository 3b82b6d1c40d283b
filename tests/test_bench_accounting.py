"""The benchmark's algorithmic work per launch (the roofline numerators) and
its throughput arithmetic, checked on the CPU against counts made here by
walking the queries and their visible positions one by one."""
import numpy as np
import pytest

import bench
import synth


def _walk(lay, H, K, kv_row, fp8):
    """Per-launch work by explicit enumeration: every (query, visible
    position) pair scored, every selected key attended, every cache row of a
    sequence read at most once per launch."""
    idx_pairs = mla_keys = 0
    rows_read = 0
    for b in range(lay.num_seqs):
        sel_b = 0
        for t in range(int(lay.q_start[b]), int(lay.q_start[b + 1])):
            vis = int(lay.q_pos[t]) + 1
            idx_pairs += vis
            sel = min(vis, K)
            mla_keys += sel
            sel_b += sel
        rows_read += min(sel_b, int(lay.q_pos[lay.q_start[b + 1] - 1]) + 1)
    key_bytes = 128 * (1 if fp8 else 2) + (4 if fp8 else 0)
    seq_len = sum(int(lay.q_pos[lay.q_start[b + 1] - 1]) + 1 for b in range(lay.num_seqs))
    # prefill rows beyond 16K positions: the select-only F layer (no score
    # matrix; sampled scores, a 2K-entry candidate list and K indices per row)
    select_only = max(int(lay.q_start[b + 1] - lay.q_start[b]) for b in range(lay.num_seqs)) > 1 \
        and lay.max_len > 16384
    sampled = 0
    for t in range(lay.num_q):
        tiles = int(lay.q_pos[t]) // 128 + 1
        sampled += min(tiles, min(max(tiles // 64, 32), 64)) * 128
    return {
        "indexer_flops": 2.0 * 32 * 128 * idx_pairs,
        "indexer_bytes": seq_len * key_bytes + lay.num_q * 32 * (128 * (1 if fp8 else 2) + 4)
        + (0 if select_only else idx_pairs * 4),
        "topk_bytes": (sampled * 4 + lay.num_q * (2 * K * 8 + K * 4)) if select_only
        else idx_pairs * 4 + lay.num_q * K * 4,
        "mla_flops": 2.0 * H * (576 + 512) * mla_keys,
        "mla_bytes": rows_read * kv_row + lay.num_q * H * (576 + 512) * 2,
    }


@pytest.mark.parametrize("case", ["prefill", "decode", "chunked", "long_prefill"])
@pytest.mark.parametrize("kv_row", [1152, 656])
def test_algorithmic_work_matches_an_explicit_count(case, kv_row):
    if case == "prefill":
        lay, H, K = synth.make_layout([512], [512]), 16, 64
    elif case == "decode":
        lay, H, K = synth.make_layout([5000, 300, 2048], [1, 1, 1]), 64, 2048
    elif case == "chunked":
        lay, H, K = synth.make_layout([3000, 700], [200, 50]), 64, 256
    else:  # rows beyond 16K positions: the select-only F layer
        lay, H, K = synth.make_layout([20000, 17000], [24, 8]), 64, 2048
    for fp8 in (False, True):
        w = bench.algorithmic(lay, {"H": H, "K": K}, fp8, kv_row)
        ref = _walk(lay, H, K, kv_row, fp8)
        assert w["indexer"]["flops"] == ref["indexer_flops"]
        assert w["indexer"]["bytes"] == ref["indexer_bytes"]
        assert w["topk"]["bytes"] == ref["topk_bytes"]
        assert w["sparse_mla"]["flops"] == ref["mla_flops"]
        assert w["sparse_mla"]["bytes"] == ref["mla_bytes"]


def test_decode_reads_each_selected_row_once():
    # one query per sequence: a decode launch reads min(len, K) rows per sequence
    lay = synth.make_layout([100000, 1000], [1, 1])
    w = bench.algorithmic(lay, {"H": 64, "K": 2048}, False)
    assert w["sparse_mla"]["bytes"] == (2048 + 1000) * 1152 + 2 * 64 * 1088 * 2


def test_bounds_and_throughput():
    peaks = {"hbm": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "src": "measured"}
    prefill = bench.algorithmic(synth.make_layout([8192], [8192]), {"H": 64, "K": 2048}, False)
    decode = bench.algorithmic(synth.make_layout([131072] * 4, [1] * 4), {"H": 64, "K": 2048}, False)
    assert bench.kernel_bound("sparse_mla", prefill["sparse_mla"], peaks, False)[0] == "tensor"
    assert bench.kernel_bound("indexer", decode["indexer"], peaks, False)[0] == "hbm"
    assert bench.kernel_bound("sparse_mla", decode["sparse_mla"], peaks, False)[0] == "hbm"
    assert bench.kernel_bound("topk", prefill["topk"], peaks, False)[0] == "hbm"
    # whole-job rate: every replica processes the workload; time = the slowest rank
    assert bench.replica_throughput(8192, 20, 4, 250.0) == pytest.approx(4 * 8192 * 20 / 0.25)
    assert bench.slowest_rank_ms(12.5, 1) == 12.5


def test_every_workload_is_described():
    assert set(bench.DESCR) == set(synth.WORKLOADS)
    for name, text in bench.DESCR.items():
        assert text and "KV latent" not in text  # the KV dtype is its own config key


def test_tensor_peak_follows_the_timed_region():
    peaks = {"hbm": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "src": "measured"}
    # a short timed region runs at the burst clock, a long one under the power cap
    assert bench.tensor_peak(peaks, False, 0.25)[0] == 1900.0
    assert bench.tensor_peak(peaks, False, 10.0)[0] == 1700.0
    # FP8 indexer: the nominal 2x ratio without a measured FP8 GEMM, else the measurement
    assert bench.tensor_peak(peaks, True, 0.25)[0] == 3800.0
    peaks["fp8"] = 3500.0
    assert bench.tensor_peak(peaks, True, 0.25)[0] == 3500.0
    assert bench.tensor_peak(peaks, True, 10.0)[0] == pytest.approx(3500.0 * 1700 / 1900)
    work = {"flops": 1e12, "bytes": 1e6}
    assert bench.kernel_bound("sparse_mla", work, peaks, False, 0.25)[:2] == ("tensor", 1900.0)


def test_kernel_records_count_work_per_unit_not_per_launch():
    """An F layer whose indexer takes three launches (the select-only path)
    is one unit of indexer work: the achieved rate divides one unit's work by
    the summed time of its launches, and the scan + gather figure adds the
    units' bytes over the summed times."""
    peaks = {"hbm": 1000.0, "bf16": 100.0, "bf16_src": "x", "hbm_src": "y", "fp8": 200.0,
             "fp8_src": "z", "bf16_sustained": 90.0}
    work = {"indexer": {"flops": 0.0, "bytes": 2.0e9}, "sparse_mla": {"flops": 0.0, "bytes": 1.0e9}}
    units = bench.step_units("FSSS", 10)
    assert units == {"indexer": 10, "topk": 10, "sparse_mla": 40}
    prof = {"indexer": (30.0, 30), "sparse_mla": (40.0, 40)}  # ms, launches
    orig = bench.kernel_bound
    bench.kernel_bound = lambda name, w, p, fp8, t: ("hbm", p["hbm"], "GB/s", "test")
    try:
        k = bench.kernel_records(prof, work, peaks, False, 1.0, units=units)
        per_launch = bench.kernel_records(prof, work, peaks, False, 1.0)
    finally:
        bench.kernel_bound = orig
    # 3 ms per F layer for 2 GB: 666.67 GB/s; per launch it would read 2000 GB/s
    assert k["indexer"]["ms_per_unit"] == 3.0 and k["indexer"]["ms_per_launch"] == 1.0
    assert k["indexer"]["achieved"] == pytest.approx(666.67, abs=0.01)
    assert per_launch["indexer"]["achieved"] == pytest.approx(2000.0)
    assert k["sparse_mla"]["achieved"] == pytest.approx(1000.0)
    assert k["indexer"]["share"] == pytest.approx(30.0 / 70.0, abs=1e-4)
    sg = bench.scan_gather_record(k, work, peaks)
    assert sg["achieved"] == pytest.approx((10 * 2.0e9 + 40 * 1.0e9) / 0.070 / 1e9, abs=0.05)
