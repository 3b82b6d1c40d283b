"""Pins of the oracle's hot/cold KV plan and swap-in (a GPU hot buffer of a
few thousand slots per sequence, the full cache in host memory, selected rows
swapped in after the top-K): a hand-worked four-slot trace, the overflow
case, invariants checked against bookkeeping kept by the test from the index
history alone (every selected position resident, hits never move, evictions
least recently used), and attention through the hot rows equal to attention
over the full cache."""
import numpy as np

import oracle
import synth


def _plan(idx, q_start, q_pos, st, step, hot):
    return oracle.hot_plan(np.asarray(idx, np.int32), q_start, q_pos, st, step, hot)


def test_hand_worked_four_slot_trace():
    hot, q_start, q_pos = 4, [0, 1], [100]
    st = oracle.hot_state(1, hot, 128)
    # step 0: two misses take the two empty slots of lowest index
    st, rows, fetch, err = _plan([[5, 9, -1]], q_start, q_pos, st, 0, hot)
    assert not err and fetch == [[(5, 0), (9, 1)]] and rows.tolist() == [[0, 1, -1]]
    # step 1: 9 hits (slot 1); empty slots 2, 3 are older than slot 0 (stamp 0)
    st, rows, fetch, err = _plan([[9, 2, 7]], q_start, q_pos, st, 1, hot)
    assert fetch == [[(2, 2), (7, 3)]] and rows.tolist() == [[1, 2, 3]]
    assert st["slot_pos"][0].tolist() == [5, 9, 2, 7]
    assert st["slot_stamp"][0].tolist() == [0, 1, 1, 1]
    # step 2: 7 and 5 hit; of the unused slots 1 and 2 (both stamp 1) the
    # lower index goes: 9 leaves, 4 enters slot 1
    st, rows, fetch, err = _plan([[7, 4, 5]], q_start, q_pos, st, 2, hot)
    assert fetch == [[(4, 1)]] and rows.tolist() == [[3, 1, 0]]
    assert st["slot_pos"][0].tolist() == [5, 4, 2, 7]
    assert st["slot_stamp"][0].tolist() == [2, 2, 1, 2]
    assert st["pos_slot"][0, 9] == -1 and st["pos_slot"][0, 4] == 1
    # step 3: 2 and 4 hit; unused slots 0 and 3 share stamp 2: slot 0 (5) goes
    st, rows, fetch, err = _plan([[9, 2, 4]], q_start, q_pos, st, 3, hot)
    assert fetch == [[(9, 0)]] and rows.tolist() == [[0, 2, 1]]
    assert st["pos_slot"][0, 5] == -1
    # step 4: one miss, slot 3 (stamp 2) is the least recently used unused slot
    st, rows, fetch, err = _plan([[9, 11, -1]], q_start, q_pos, st, 4, hot)
    assert fetch == [[(11, 3)]] and st["slot_pos"][0].tolist() == [9, 4, 2, 11]
    # steps 5, 6: hits only, leaving stamps [6, 6, 5, 4]
    st, _, fetch, _ = _plan([[2, -1, -1]], q_start, q_pos, st, 5, hot)
    st, _, fetch, _ = _plan([[9, 4, -1]], q_start, q_pos, st, 6, hot)
    assert fetch == [[]] and st["slot_stamp"][0].tolist() == [6, 6, 5, 4]
    # step 7: the two least recently used slots are 3 (stamp 4) and 2 (stamp 5);
    # they are handed out in slot order, so the first miss gets slot 2
    st, rows, fetch, err = _plan([[70, 71, -1]], q_start, q_pos, st, 7, hot)
    assert fetch == [[(70, 2), (71, 3)]] and rows.tolist() == [[2, 3, -1]]
    assert st["slot_pos"][0].tolist() == [9, 4, 70, 71]
    assert st["pos_slot"][0, 2] == -1 and st["pos_slot"][0, 11] == -1


def test_two_sequences_duplicates_and_first_appearance_order():
    hot = 3
    q_start, q_pos = [0, 2, 3], [50, 51, 20]
    st = oracle.hot_state(2, hot, 64)
    idx = [[4, 8, -1], [8, 6, 4],    # sequence 0: 4, 8, 6 in first-appearance order
           [20, 0, 3]]               # sequence 1
    st, rows, fetch, err = _plan(idx, q_start, q_pos, st, 7, hot)
    assert not err
    assert fetch == [[(4, 0), (8, 1), (6, 2)], [(20, 0), (0, 1), (3, 2)]]
    assert rows.tolist() == [[0, 1, -1], [1, 2, 0], [3, 4, 5]]


def test_overflow_and_invalid_entries():
    hot, q_start, q_pos = 4, [0, 2], [30, 31]
    st0 = oracle.hot_state(1, hot, 64)
    st, rows, fetch, err = _plan([[1, 3, 6], [8, 10, 6]], q_start, q_pos, st0, 0, hot)
    assert err == {"overflow"} and fetch == [[]] and (rows == -1).all()
    assert (st["slot_pos"] == -1).all() and (st["pos_slot"] == -1).all()
    # one hit plus four misses need four slots besides the hit's: overflow too
    st1, _, _, _ = _plan([[6, -1, -1], [-1, -1, -1]], q_start, q_pos, st0, 0, hot)
    st, rows, fetch, err = _plan([[1, 3, 6], [8, 10, 6]], q_start, q_pos, st1, 1, hot)
    assert err == {"overflow"} and (rows == -1).all()
    assert np.array_equal(st["slot_pos"], st1["slot_pos"]) and np.array_equal(st["pos_slot"], st1["pos_slot"])
    # a position beyond the query's own is an error and is skipped
    st, rows, fetch, err = _plan([[1, 31, -1], [2, 40, -1]], q_start, q_pos, st0, 0, hot)
    assert err == {"index"} and rows.tolist() == [[0, -1, -1], [1, -1, -1]]
    assert fetch == [[(1, 0), (2, 1)]]


def test_invariants_over_a_random_trace():
    rng = np.random.default_rng(5)
    S, hot, L, K, nq = 3, 48, 400, 16, 2
    q_start = np.arange(S + 1) * nq
    st = oracle.hot_state(S, hot, L)
    last_use = [dict() for _ in range(S)]        # position -> last step it was selected
    resident = [set() for _ in range(S)]
    for step in range(60):
        q_pos = rng.integers(200, L, S * nq).astype(np.int32)
        idx = np.full((S * nq, K), -1, np.int32)
        for t in range(S * nq):
            # mostly from a small hot set, sometimes fresh positions
            pool = rng.choice(60, K, replace=False) if rng.random() < 0.7 else rng.choice(200, K, replace=False)
            n = rng.integers(K // 2, K + 1)
            idx[t, :n] = pool[:n]
        before = {key: v.copy() for key, v in st.items()}
        st, rows, fetch, err = _plan(idx, q_start, q_pos, st, step, hot)
        assert not err
        for b in range(S):
            sel = {int(e) for e in idx[nq * b: nq * b + nq].ravel() if e >= 0}
            sp, ps = st["slot_pos"][b], st["pos_slot"][b]
            # bijection between occupied slots and resident positions
            occ = {int(p): s for s, p in enumerate(sp) if p >= 0}
            assert occ == {p: int(ps[p]) for p in np.flatnonzero(ps >= 0)}
            # every selected position resident, rows decode to it
            for t in range(nq * b, nq * b + nq):
                for k in range(K):
                    e = idx[t, k]
                    if e >= 0:
                        assert rows[t, k] == b * hot + ps[e]
                    else:
                        assert rows[t, k] == -1
            # hits keep their slot; misses are exactly the selected non-residents
            for e in sel & resident[b]:
                assert ps[e] == before["pos_slot"][b][e]
            assert {e for e, _ in fetch[b]} == sel - resident[b]
            # evicted positions were used no later than any kept, unused one
            new_res = set(occ)
            evicted = resident[b] - new_res
            kept_idle = new_res - sel
            if evicted and kept_idle:
                assert max(last_use[b][e] for e in evicted) <= min(last_use[b][e] for e in kept_idle)
            for e in sel:
                last_use[b][e] = step
            resident[b] = new_res


def test_attention_through_hot_rows_equals_full_cache():
    lay = synth.make_layout([700, 500], [2, 1])
    host = synth.host_layers(lay, "S", 16, ints=False, seed=9)[0]
    hot, K = 200, 64
    rng = np.random.default_rng(4)
    st = oracle.hot_state(lay.num_seqs, hot, lay.max_len)
    hot_kv = np.zeros((lay.num_seqs * hot, 576), np.uint16)
    rows_all = np.arange(lay.num_q, dtype=np.int32)
    pos, key0 = oracle.row_metadata(lay.q_start, lay.q_pos, lay.seq_row0, rows_all)
    for step in range(4):
        idx = np.full((lay.num_q, K), -1, np.int32)
        for t in range(lay.num_q):
            n = int(lay.q_pos[t]) + 1
            idx[t] = np.sort(rng.choice(min(n, 150 + 40 * step), K, replace=False))
        st, rows, fetch, err = oracle.hot_plan(idx, lay.q_start, lay.q_pos, st, step, hot)
        assert not err
        oracle.hot_fetch(fetch, host["kv"], lambda b, e: int(lay.seq_row0[b]) + e, hot_kv, hot)
        ref = oracle.sparse_mla(host["q_lat"], host["q_rope"], host["kv"], rows_all, key0, idx, 1 / 16)
        got = oracle.sparse_mla(host["q_lat"], host["q_rope"], hot_kv, rows_all,
                                np.zeros_like(key0), rows, 1 / 16)
        assert np.array_equal(ref[0], got[0]) and np.array_equal(ref[1], got[1])
