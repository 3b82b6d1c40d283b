"""GPU parity of the hot/cold KV path through the C ABI: the plan kernel
against the oracle's plan step by step (rows, slot tables, stamps, position
map and fetch lists bit for bit, with overlapping selections, duplicates,
invalid entries and an overflowing sequence), the swap-in from pinned host
memory (contiguous and paged cold caches), attention over hot rows
bit-identical to attention over the full device cache, and the hot group
call identical to the plain group call."""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import synth  # noqa: E402
from gpu_helpers import bf16_dev, device_layers, make_batch  # noqa: E402

dsa = pytest.importorskip("dsa_indexer_indexshare_gb300")
DEV = torch.device("cuda:0")


def _state_np(st):
    return {"slot_pos": st.slot_pos.cpu().numpy(), "slot_stamp": st.slot_stamp.cpu().numpy(),
            "pos_slot": st.pos_slot.cpu().numpy()}


def _trace_idx(rng, lay, K, pool):
    """Selections drawn mostly from a per-sequence pool of recent positions
    (so steps overlap), sometimes fresh; -1 padded, unsorted."""
    idx = np.full((lay.num_q, K), -1, np.int32)
    seq_of = np.searchsorted(lay.q_start, np.arange(lay.num_q), side="right") - 1
    for t in range(lay.num_q):
        n = int(lay.q_pos[t]) + 1
        b = seq_of[t]
        m = min(n, K - int(rng.integers(0, 3)))
        fresh = rng.choice(n, min(n, 4 * K), replace=False)
        cand = np.concatenate([pool[b][pool[b] < n], fresh]) if rng.random() < 0.8 else fresh
        _, first = np.unique(cand, return_index=True)
        cand = cand[np.sort(first)]
        idx[t, :m] = rng.permutation(cand[:max(m, 1)])[:m]
        pool[b] = np.unique(np.concatenate([pool[b], idx[t, :m]]))[-2 * K:]
    return idx


def _compare(st_gpu, st_ref):
    g = _state_np(st_gpu)
    for key in ("slot_pos", "slot_stamp", "pos_slot"):
        assert np.array_equal(g[key], st_ref[key]), key


@pytest.mark.parametrize("hot_slots,K,step0", [(400, 128, 0), (6144, 2048, 0),
                                               (400, 128, (1 << 24) - 3)])
def test_hot_plan_matches_oracle_over_steps(hot_slots, K, step0):
    """step0 > 0 starts the step numbers just below 2^24, so the stamps cross
    a digit of the kernel's radix select over them."""
    rng = np.random.default_rng(hot_slots)
    if K == 2048:  # decode-shaped: 16 sequences of ~100K positions, one query each
        lens = rng.integers(98304, 131073, 16)
        lay = synth.make_layout(list(lens), [1] * 16)
    else:
        lay = synth.make_layout([5000, 900, 3000], [2, 1, 3])
    batch = make_batch(dsa, lay, DEV)
    st = dsa.HotState(lay.num_seqs, hot_slots, lay.max_len, DEV)
    ref = oracle.hot_state(lay.num_seqs, hot_slots, lay.max_len)
    pool = [np.zeros(0, np.int64) for _ in range(lay.num_seqs)]
    ws = dsa.workspace(256, DEV)
    for i in range(4 if K == 2048 else 8):
        step = step0 + i
        idx = _trace_idx(rng, lay, K, pool)
        rows = dsa.dsa_hot_plan(torch.from_numpy(idx).to(DEV), batch, st, step, ws=ws)
        assert dsa.status_fetch(ws) == 0
        ref, rrows, rfetch, err = oracle.hot_plan(idx, lay.q_start, lay.q_pos, ref, step, hot_slots)
        assert not err
        assert np.array_equal(rows.cpu().numpy(), rrows)
        assert st.fetch_lists() == [list(map(tuple, f)) for f in rfetch]
        _compare(st, ref)


def test_hot_plan_overflow_and_invalid_entries():
    lay = synth.make_layout([400, 400], [1, 1])  # both queries at position 399
    hot, K = 8, 9
    batch = make_batch(dsa, lay, DEV)
    st = dsa.HotState(lay.num_seqs, hot, lay.max_len, DEV)
    ref = oracle.hot_state(lay.num_seqs, hot, lay.max_len)
    ws = dsa.workspace(256, DEV)
    first = np.array([[1, 2, 3, 4, 5, -1, -1, -1, -1],
                      [10, 11, 12, 13, -1, -1, -1, -1, -1]], np.int32)
    dsa.dsa_hot_plan(torch.from_numpy(first).to(DEV), batch, st, 0, ws=ws)
    assert dsa.status_fetch(ws) == 0
    ref, _, _, _ = oracle.hot_plan(first, lay.q_start, lay.q_pos, ref, 0, hot)
    # sequence 0: 2 hits + 7 misses > 6 unused slots (overflow); sequence 1
    # proceeds, but its entry 500 lies beyond its query's position
    second = np.array([[1, 2, 20, 21, 22, 23, 24, 25, 26],
                       [10, 30, 31, 500, -1, -1, -1, -1, -1]], np.int32)
    rows = dsa.dsa_hot_plan(torch.from_numpy(second).to(DEV), batch, st, 1, ws=ws)
    raw = ctypes.c_int32(0)
    s = dsa.lib.dsa_status_fetch(dsa._ptr(ws), dsa._stream(None, DEV), ctypes.byref(raw))
    assert s == dsa.DSA_ERR_DEVICE_INDEX and raw.value == 2 | 8
    ref, rrows, rfetch, err = oracle.hot_plan(second, lay.q_start, lay.q_pos, ref, 1, hot)
    assert err == {"overflow", "index"} and (rrows[0] == -1).all()
    assert np.array_equal(rows.cpu().numpy(), rrows)
    assert st.fetch_lists() == [list(map(tuple, f)) for f in rfetch]
    _compare(st, ref)


def _cold_layers(host_kv_list, table=None, R=0, lay=None):
    """Cold caches in pinned host memory, in the contiguous or a paged layout."""
    out = []
    for kv in host_kv_list:
        a = kv
        if table is not None:
            nblk = int(table.max()) + 1
            a = np.zeros((nblk * R,) + kv.shape[1:], kv.dtype)
            for b in range(lay.num_seqs):
                for s in range(int(lay.seq_len[b])):
                    a[oracle.paged_row(table, R, b, s)] = kv[int(lay.seq_row0[b]) + s]
        a = np.ascontiguousarray(a)
        t = (torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16
             else torch.from_numpy(a))
        out.append(t.pin_memory())
    return out


@pytest.mark.parametrize("layout", ["contiguous", "paged"])
@pytest.mark.parametrize("kv_fp8", [False, True])
def test_fetch_and_attention_over_hot_rows(layout, kv_fp8):
    lay = synth.make_layout([2000, 1300], [2, 1])
    K, hot = 256, 700
    host = synth.host_layers(lay, "SS", 64, ints=False, seed=21)
    kvs = [oracle.kv_fp8_quantize(L["kv"]) if kv_fp8 else L["kv"] for L in host]
    table, R = None, 0
    if layout == "paged":
        R = 256
        nb = [(int(n) + R - 1) // R for n in lay.seq_len]
        ids = np.random.default_rng(3).permutation(sum(nb) + 2)
        table = np.full((lay.num_seqs, lay.max_len // R), -1, np.int32)
        k = 0
        for b, n in enumerate(nb):
            table[b, :n] = ids[k:k + n]
            k += n
        batch = dsa.Batch(lay.q_start, lay.q_pos, None, lay.max_len, device=DEV,
                          block_table=table, block_rows=R)
    else:
        batch = make_batch(dsa, lay, DEV)
    cold = _cold_layers(kvs, table, R, lay)
    dsa.dsa_hot_touch(cold, stride=4096, device=DEV)  # reads only: the caches stay as they were
    row_w = dsa.KV_ROW_FP8 if kv_fp8 else dsa.KV_ROW
    dt = torch.uint8 if kv_fp8 else torch.bfloat16
    hot_kv = [torch.zeros((lay.num_seqs * hot, row_w), dtype=dt, device=DEV) for _ in kvs]
    st = dsa.HotState(lay.num_seqs, hot, lay.max_len, DEV)
    ref = oracle.hot_state(lay.num_seqs, hot, lay.max_len)
    ref_hot = [np.zeros((lay.num_seqs * hot, row_w), kvs[0].dtype) for _ in kvs]
    full_batch = make_batch(dsa, lay, DEV)
    full_dev = [torch.from_numpy(kv).to(DEV) if kv_fp8 else bf16_dev(kv, DEV) for kv in kvs]
    rng = np.random.default_rng(8)
    pool = [np.zeros(0, np.int64) for _ in range(lay.num_seqs)]
    ws = dsa.workspace(1 << 20, DEV)
    for step in range(3):
        idx = _trace_idx(rng, lay, K, pool)
        idx_d = torch.from_numpy(idx).to(DEV)
        rows = dsa.dsa_hot_plan(idx_d, batch, st, step, ws=ws)
        dsa.dsa_hot_fetch(st, batch, cold, hot_kv, ws=ws)
        assert dsa.status_fetch(ws) == 0
        ref, rrows, rfetch, _ = oracle.hot_plan(idx, lay.q_start, lay.q_pos, ref, step, hot)
        for l, kv in enumerate(kvs):
            oracle.hot_fetch(rfetch, kv, lambda b, e: int(lay.seq_row0[b]) + e, ref_hot[l], hot)
            got = hot_kv[l].cpu()
            got = (got.view(torch.int16).numpy().view(np.uint16) if not kv_fp8 else got.numpy())
            assert np.array_equal(got, ref_hot[l])
        for l, L in enumerate(host):
            ql, qr = bf16_dev(L["q_lat"], DEV), bf16_dev(L["q_rope"], DEV)
            o_hot, l_hot = dsa.dsa_sparse_mla_attn_rows(ql, qr, hot_kv[l], rows, batch, scale=1 / 16,
                                                        ws=ws)
            o_full, l_full = dsa.dsa_sparse_mla_attn(ql, qr, full_dev[l], idx_d, full_batch,
                                                     scale=1 / 16, ws=ws)
            assert torch.equal(o_hot, o_full) and torch.equal(l_hot, l_full)
        assert dsa.status_fetch(ws) == 0


@pytest.mark.parametrize("types,kv_fp8", [("FSSS", False), ("FSSSFSSS", True)])
def test_group_forward_hot_equals_group_forward(types, kv_fp8):
    lay = synth.make_layout([3000, 2200], [1, 1])
    K, hot = 512, 1536
    host = synth.host_layers(lay, types, 64, ints=False, seed=31)
    layers_full = device_layers(host, DEV)
    if kv_fp8:
        for L in layers_full:
            L["kv"] = dsa.dsa_kv_fp8_quantize(L["kv"])
    batch = make_batch(dsa, lay, DEV)
    g_full = dsa.Group(types, layers_full, k=K, scale=1 / 16, with_lse=True)
    cold = [L["kv"].cpu().pin_memory() for L in layers_full]
    row_w = dsa.KV_ROW_FP8 if kv_fp8 else dsa.KV_ROW
    layers_hot = [dict(L, kv=torch.zeros((lay.num_seqs * hot, row_w), dtype=L["kv"].dtype,
                                         device=DEV)) for L in layers_full]
    g_hot = dsa.Group(types, layers_hot, k=K, scale=1 / 16, with_lse=True)
    spans = [dsa.HotState(lay.num_seqs, hot, lay.max_len, DEV) for c in types if c == "F"]
    hg = dsa.HotGroup(spans, cold, num_q=lay.num_q, k=K, device=DEV)
    ws_f = dsa.workspace(g_full.workspace_size(batch), DEV)
    ws_h = dsa.workspace(g_hot.workspace_size(batch), DEV)
    outs_f, lses_f, idx_f = dsa.indexshare_group_forward(g_full, batch, ws=ws_f)
    dsa.status_fetch(ws_f)
    for step in range(3):  # the first step misses everything, the next ones hit
        outs_h, lses_h, idx_h = dsa.indexshare_group_forward_hot(g_hot, batch, hg, step, ws=ws_h)
        dsa.status_fetch(ws_h)
        assert torch.equal(idx_h, idx_f)
        for a, b in zip(outs_h, outs_f):
            assert torch.equal(a, b)
        for a, b in zip(lses_h, lses_f):
            assert torch.equal(a, b)
        n_fetch = sum(int(s.fetch_count.sum()) for s in spans)
        assert (n_fetch > 0) == (step == 0)
