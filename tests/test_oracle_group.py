"""Pins for the oracle's IndexShare group loop and the pages' printed numbers.

"GLM-5.2 架构深度拆解" CH 2.1 (indexer_types: 3 full + 3 shared, then 18
groups of 1 full + 3 shared = 21 full + 57 shared), CH 2.2 (S layers skip the
indexer and reuse the nearest F layer's indices), CH 2.3 (indexer FLOPs ratio
21/78 = 0.269), CH 7.3 (all layers full = the every-layer-indexer model).
"""
import json
import os

import numpy as np
import pytest

import oracle
import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden", "pages_numbers.json")


def glm52_indexer_types(g):
    lp = g["layer_pattern"]
    return ("F" * lp["cold_start"]["full"] + "S" * lp["cold_start"]["shared"]
            + lp["group"] * lp["main_loop_groups"])


def test_printed_layer_pattern_and_flops_ratio():
    g = json.load(open(GOLD))
    types = glm52_indexer_types(g)
    full = oracle.parse_layer_types(types)
    assert len(full) == g["layer_pattern"]["total_layers"]
    assert sum(full) == g["layer_pattern"]["total_full"]
    assert len(full) - sum(full) == g["layer_pattern"]["total_shared"]
    r = g["indexer_flops_ratio"]
    assert round(sum(full) / len(full), r["ratio_decimals"]) == r["ratio"]
    # one indexer pass per group of four in the main loop
    assert types[6:10] == "FSSS" and g["indexer_shape"]["share_every"] == 4


def test_printed_kv_row_and_scale():
    g = json.load(open(GOLD))
    kvb = g["kv_bytes_per_token_per_layer_bf16"]
    assert (synth.DL + synth.DR) * 2 == kvb["bytes"] and synth.DL == kvb["latent"]
    assert synth.DR == kvb["rope"]
    m = g["mla_shape"]
    assert 1 / np.sqrt(m["qk_head_dim"]) == m["softmax_scale"]
    assert (synth.HI, synth.DI) == (g["indexer_shape"]["heads"], g["indexer_shape"]["dim"])


def test_layer_types_validation():
    for bad in ("", "SFSS", "FXS", "fsss"):
        with pytest.raises(ValueError):
            oracle.parse_layer_types(bad)
    assert oracle.parse_layer_types("FSSSFSSS") == [True, False, False, False] * 2


def _tiny(layer_types, T=96, H=4, seed=0):
    lay = synth.make_layout([T], [T])
    layers = synth.host_layers(lay, layer_types, H, ints=True, seed=seed)
    rows = np.arange(lay.num_q, dtype=np.int32)
    pos, key0 = oracle.row_metadata(lay.q_start, lay.q_pos, lay.seq_row0, rows)
    return lay, layers, rows, pos, key0


def test_shared_layers_reuse_the_full_layers_indices(monkeypatch):
    lay, layers, rows, pos, key0 = _tiny("FSSSFSSS")
    calls = []
    real = oracle.indexer_scores
    monkeypatch.setattr(oracle, "indexer_scores", lambda *a, **k: calls.append(1) or real(*a, **k))
    res = oracle.group_forward("FSSSFSSS", layers, rows, pos, key0, lay.max_len, 16, 1 / 16)
    assert len(calls) == 2                       # one indexer pass per F layer
    for l in (1, 2, 3):
        assert res["idx"][l].tobytes() == res["idx"][0].tobytes()
    for l in (5, 6, 7):
        assert res["idx"][l].tobytes() == res["idx"][4].tobytes()
    # an S layer is plain sparse MLA of its own cache over the F layer's buffer
    o, s = oracle.sparse_mla(layers[2]["q_lat"], layers[2]["q_rope"], layers[2]["kv"], rows,
                             key0, res["idx"][0], 1 / 16)
    assert np.array_equal(o, res["out"][2]) and np.array_equal(s, res["lse"][2])


def test_all_full_is_independent_dsa_layers():
    lay, layers, rows, pos, key0 = _tiny("FFFF", seed=1)
    res = oracle.group_forward("FFFF", layers, rows, pos, key0, lay.max_len, 16, 1 / 16)
    for l in range(4):
        one = oracle.group_forward("F", [layers[l]], rows, pos, key0, lay.max_len, 16, 1 / 16)
        assert np.array_equal(one["out"][0], res["out"][l])
        assert np.array_equal(one["idx"][0], res["idx"][l])
    # different layers' indexers pick different sets on random data
    assert not np.array_equal(res["idx"][0], res["idx"][1])


def test_short_prefix_rows_select_everything():
    lay, layers, rows, pos, key0 = _tiny("FS", T=40)
    res = oracle.group_forward("FS", layers, rows, pos, key0, lay.max_len, 16, 1 / 16)
    idx = res["idx"][0]
    for t in range(16):                          # pos + 1 <= K: all visible positions
        assert idx[t, :t + 1].tolist() == list(range(t + 1))
        assert (idx[t, t + 1:] == -1).all()
    assert (idx[16:] >= 0).all()
