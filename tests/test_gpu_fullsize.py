"""Full-size parity in the launch configuration the benchmark times.

Each workload is built exactly as bench.py builds it (seeded device inputs,
one indexshare_group_forward call per F-led span) and sampled query rows are
recomputed by the oracle from host copies of the same inputs.  Rows are
independent, so parity on sampled rows is parity of those rows.  The oracle
reads the indexer keys of the sampled rows' sequences in full, and of each
layer's KV cache only the rows it attends to (gathered on the device and
copied out), so that long contexts fit in host memory.

* indices (Gaussian scores): the GPU set may differ from the oracle's only at
  positions whose oracle score lies within 1e-3 of the K-th score;
* attention outputs: within 2e-2 * max|ref| for rows whose index set equals
  the oracle's (a near-tie swap changes the sparse set, and with it the
  output, legitimately; such rows are validated through their index set);
* sparse MLA alone: the oracle's own index rows are fed to the GPU kernel for
  the sampled rows, and the outputs must agree within the same bound;
* FP8 indexer: the library quantiser's codes obey the comparison rule
  against the oracle's definition (tests/fp8_rule.py) on every sampled query
  vector and a sample of key rows; the oracle then scores the library's codes;
* FP8 KV latent: the library's 656-byte rows equal the oracle's quantisation
  of the same bf16 rows (the quantiser rounds the exact quotient), and the
  oracle reads their dequantised values;
* hot/cold KV (decode shape, 6144 hot slots): the hot group call equals the
  device-resident group call bit for bit over steps that miss and hit.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.slow]

import oracle  # noqa: E402
import synth  # noqa: E402
from fp8_rule import check_fp8_rows  # noqa: E402
from gpu_helpers import (assert_close, assert_topk_within_band, bits,  # noqa: E402
                         oracle_attention_gathered)

dsa = pytest.importorskip("dsa_indexer_indexshare_gb300")
DEV = torch.device("cuda:0")
SCALE = 1 / 16
KEY_RULE_ROWS = 1 << 17   # key rows per F layer checked by the FP8 comparison rule


def _seq_spans(lay, rows):
    """Sequences of the sampled rows, each as (first cache row, length, base
    in the compact host copy of the indexer keys)."""
    seq = np.searchsorted(lay.q_start, rows, side="right") - 1
    spans, base = {}, 0
    for b in sorted(set(seq.tolist())):
        n = int(lay.q_pos[lay.q_start[b + 1] - 1]) + 1
        spans[b] = (int(lay.seq_row0[b]), n, base)
        base += n
    return seq, spans


def _compact(t, spans):
    return torch.cat([t[r0:r0 + n] for (r0, n, _) in spans.values()]).contiguous()


def _oracle_indices(lay, L, rows, seq, spans, fp8, rng):
    """Oracle scores and top-K of one F layer for the sampled rows."""
    rt = torch.as_tensor(rows, device=DEV)
    pos = lay.q_pos[rows].astype(np.int32)
    key0 = np.array([spans[b][2] for b in seq], np.int64)
    w = L["w"].index_select(0, rt).cpu().numpy()
    if fp8:
        q_bf16 = bits(L["q_idx_bf16"].index_select(0, rt))
        qc = L["q_idx"].index_select(0, rt).cpu().numpy()
        qs = L["q_scale"].index_select(0, rt).cpu().numpy()
        check_fp8_rows(qc.reshape(-1, 128), qs.reshape(-1), q_bf16.reshape(-1, 128),
                       what="query codes")
        kc = _compact(L["k_idx"], spans).cpu().numpy()
        ks = _compact(L["k_scale"], spans).cpu().numpy()
        pick = np.sort(rng.choice(kc.shape[0], min(KEY_RULE_ROWS, kc.shape[0]), replace=False))
        kb = bits(_compact(L["k_idx_bf16"], spans)[torch.as_tensor(pick, device=DEV)])
        check_fp8_rows(kc[pick], ks[pick], kb, what="key codes")
        sc = oracle.indexer_scores(qc, w, kc, np.arange(len(rows), dtype=np.int32), pos, key0,
                                   lay.max_len, dtype=1, q_scale=qs, k_scale=ks)
    else:
        sc = oracle.indexer_scores(bits(L["q_idx"].index_select(0, rt)), w,
                                   bits(_compact(L["k_idx"], spans)),
                                   np.arange(len(rows), dtype=np.int32), pos, key0, lay.max_len)
    return sc, oracle.topk(sc, pos + 1, int(L["K"]))


def _oracle_attention(lay, L, rows, seq, idx):
    """Oracle sparse MLA of one layer for the sampled rows over `idx`."""
    return oracle_attention_gathered(L["q_lat"], L["q_rope"], L["kv"], rows, lay.seq_row0[seq], idx,
                                     SCALE, kv_bf16=L.get("kv_bf16"))


def _run(name, sample, kv_fp8=False):
    cfg = dict(synth.WORKLOADS[name])
    lay = synth.workload_layout(name)
    types, H, K = cfg["layers"], cfg["H"], cfg["K"]
    fp8 = bool(cfg.get("fp8"))
    layers = synth.device_layers(lay, types, H, device=DEV, seed=0)
    for L in layers:
        L["K"] = K
        if fp8 and "q_idx" in L:
            L["q_idx_bf16"], L["k_idx_bf16"] = L["q_idx"], L["k_idx"]
            qc, qs = dsa.dsa_fp8_quantize(L["q_idx"])
            kc, ks = dsa.dsa_fp8_quantize(L["k_idx"])
            L.update(q_idx=qc, q_scale=qs, k_idx=kc, k_scale=ks)
        if kv_fp8:
            L["kv_bf16"] = L["kv"]
            L["kv"] = dsa.dsa_kv_fp8_quantize(L["kv"])
    batch = dsa.Batch(lay.q_start, lay.q_pos, lay.seq_row0, lay.max_len, device=DEV)
    rows = np.array(sorted(set(r for r in sample if 0 <= r < lay.num_q)), np.int64)
    seq, spans = _seq_spans(lay, rows)
    rng = np.random.default_rng(99)
    lens = lay.q_pos[rows].astype(np.int64) + 1
    rt = torch.as_tensor(rows, device=DEV)
    f_layers = [l for l, c in enumerate(types) if c == "F"]
    starts = f_layers + [len(types)]
    for gi in range(len(f_layers)):
        lo, hi = starts[gi], starts[gi + 1]
        sc, ref_idx = _oracle_indices(lay, layers[lo], rows, seq, spans, fp8, rng)
        group = dsa.Group(types[lo:hi], [{k: v for k, v in L.items() if not k.endswith("_bf16")
                                          and k != "K"} for L in layers[lo:hi]], k=K, scale=SCALE)
        ws = dsa.workspace(group.workspace_size(batch), DEV)
        outs, _, idx = dsa.indexshare_group_forward(group, batch, ws=ws)
        torch.cuda.synchronize()
        dsa.status_fetch(ws)
        got_idx = idx.index_select(0, rt).cpu().numpy()
        assert_topk_within_band(got_idx, sc, lens, K, what=f"{name} F layer {lo}")
        same = np.array([np.array_equal(got_idx[i], ref_idx[i]) for i in range(len(rows))])
        for l in range(lo, hi):
            ref_o, ref_lse = _oracle_attention(lay, layers[l], rows, seq, ref_idx)
            if same.any():
                got = outs[l - lo].index_select(0, torch.as_tensor(rows[same], device=DEV))
                assert_close(got.float().cpu().numpy(), ref_o[same], 2e-2, f"{name} layer {l}")
            if l == lo:
                # sparse MLA alone with the oracle's indices in the sampled rows
                idx_in = idx.clone()
                idx_in[rt] = torch.from_numpy(ref_idx).to(DEV)
                o, lse = dsa.dsa_sparse_mla_attn(layers[l]["q_lat"], layers[l]["q_rope"],
                                                 layers[l]["kv"], idx_in, batch, scale=SCALE)
                o = o.index_select(0, rt).float().cpu().numpy()
                assert_close(o, ref_o, 2e-2, f"{name} sparse MLA layer {l}")
                lse = lse.index_select(0, rt).cpu().numpy()
                assert np.allclose(lse, ref_lse, rtol=0, atol=1e-3 * max(1.0, np.abs(ref_lse).max()))
        del group, ws, outs, idx
    del layers
    torch.cuda.empty_cache()


def _decode_sample(name, n):
    """About n rows of a decode workload (one query per sequence): its
    longest and shortest sequences and others spread evenly."""
    lay = synth.workload_layout(name)
    pick = {int(np.argmax(lay.seq_len)), int(np.argmin(lay.seq_len))}
    pick |= set(np.linspace(0, lay.num_q - 1, n - 2).astype(int).tolist())
    return sorted(pick)


def test_prefill8k_full_size():
    _run("prefill8k", [0, 1, 2, 100, 2046, 2047, 2048, 2049, 3000, 4095, 4096, 5000, 6143, 7000,
                       8190, 8191])


def test_decode64_full_size():
    _run("decode64", _decode_sample("decode64", 18))


def test_chunked_full_size():
    _run("chunked", [0, 1, 1000, 2047, 2048, 3000, 4094, 4095])


def test_decode1m_fp8_full_size():
    _run("decode1m", [0, 1, 2, 3])


def test_decode64_fp8_kv_full_size():
    _run("decode64", _decode_sample("decode64", 8), kv_fp8=True)


def test_decode8_hot_cold_equals_resident():
    cfg = dict(synth.WORKLOADS["decode8"])
    lay = synth.workload_layout("decode8")
    types, H, K = cfg["layers"], cfg["H"], cfg["K"]
    layers = synth.device_layers(lay, types, H, device=DEV, seed=0)
    batch = dsa.Batch(lay.q_start, lay.q_pos, lay.seq_row0, lay.max_len, device=DEV)
    slots = 6144
    # a second indexer query set, so that one step selects other positions
    g2 = torch.Generator(device=DEV)
    g2.manual_seed(77)
    layers2 = [dict(L) for L in layers]
    layers2[0]["q_idx"] = (torch.randn(layers[0]["q_idx"].shape, generator=g2, device=DEV)
                           / np.sqrt(128)).to(torch.bfloat16)
    res = [dsa.Group(types, ls, k=K, scale=SCALE) for ls in (layers, layers2)]
    cold = []
    for L in layers:
        h = torch.empty(L["kv"].shape, dtype=L["kv"].dtype, pin_memory=True)
        h.copy_(L["kv"])
        cold.append(h)
    hot_kv = [torch.zeros((lay.num_seqs * slots, 576), dtype=torch.bfloat16, device=DEV) for _ in layers]
    hot = [dsa.Group(types, [dict(L, kv=hk) for L, hk in zip(ls, hot_kv)], k=K, scale=SCALE)
           for ls in (layers, layers2)]
    spans = [dsa.HotState(lay.num_seqs, slots, lay.max_len, DEV)]
    hg = dsa.HotGroup(spans, cold, num_q=lay.num_q, k=K, device=DEV)
    ws = dsa.workspace(res[0].workspace_size(batch), DEV)
    for step, which in enumerate((0, 1, 0, 0)):
        outs_r, _, idx_r = dsa.indexshare_group_forward(res[which], batch, ws=ws)
        outs_r = [o.clone() for o in outs_r]
        idx_r = idx_r.clone()
        outs_h, _, idx_h = dsa.indexshare_group_forward_hot(hot[which], batch, hg, step, ws=ws)
        dsa.status_fetch(ws)
        assert torch.equal(idx_h, idx_r)
        for a, b in zip(outs_h, outs_r):
            assert torch.equal(a, b)
        fetched = int(spans[0].fetch_count.sum())
        # steps 0 and 1 select new positions; steps 2 and 3 repeat step 0's
        # selection, still resident (2 x 2048 rows fit in 6144 slots): all hit
        assert (fetched > 0) == (step < 2)
