"""GPU parity of the FP8 indexer variant against the bf16 pipeline: the
group call with the library's FP8 quantiser on the indexer inputs stays
within 6e-2 * max|ref| of the oracle run on the unquantised bf16 inputs, on
inputs with a planted set of relevant positions (see synth's
planted_host_layers and plant_device): on a small two-sequence case and at
the 1M-context decode shape."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import synth  # noqa: E402
from gpu_helpers import bits, device_layers, make_batch, oracle_attention_gathered  # noqa: E402

dsa = pytest.importorskip("dsa_indexer_indexshare_gb300")
DEV = torch.device("cuda:0")


def test_fp8_indexer_group_within_6e2_of_bf16_oracle():
    lay = synth.make_layout([3000, 1200], [2, 2])
    K, types = 512, "FSSS"
    host, planted = synth.planted_host_layers(lay, types, 64, m=64, seed=21)
    layers = device_layers(host, DEV)
    for L in layers:
        if "q_idx" in L:
            qc, qs = dsa.dsa_fp8_quantize(L["q_idx"])
            kc, ks = dsa.dsa_fp8_quantize(L["k_idx"])
            L.update(q_idx=qc, q_scale=qs, k_idx=kc, k_scale=ks)
    batch = make_batch(dsa, lay, DEV)
    g = dsa.Group(types, layers, k=K, scale=1 / 16)
    ws = dsa.workspace(g.workspace_size(batch), DEV)
    outs, _, idx = dsa.indexshare_group_forward(g, batch, ws=ws)
    torch.cuda.synchronize()
    dsa.status_fetch(ws)
    rows = np.arange(lay.num_q, dtype=np.int32)
    pos, key0 = oracle.row_metadata(lay.q_start, lay.q_pos, lay.seq_row0, rows)
    ref = oracle.group_forward(types, host, rows, pos, key0, lay.max_len, K, 1 / 16, idx_dtype=0)
    got_idx = idx.cpu().numpy()
    seq_of = np.searchsorted(lay.q_start, rows, side="right") - 1
    for t in range(lay.num_q):
        assert set(planted[seq_of[t]].tolist()) <= set(got_idx[t].tolist())
    for l in range(4):
        got = outs[l].float().cpu().numpy()
        err = np.abs(got - ref["out"][l]).max()
        assert err <= 6e-2 * np.abs(ref["out"][l]).max(), (l, err)


@pytest.mark.slow
def test_fp8_indexer_group_within_6e2_at_the_1m_decode_shape():
    # the 1M-context decode workload's shape (4 sequences of 1,048,576
    # positions, one query each, K = 2048, FSSS, 64 heads) with the same
    # planted construction (m = 64 positions per sequence); every query row
    # and every layer is compared with the oracle on the unquantised bf16
    # indexer inputs.  The oracle reads the whole indexer key cache of the
    # four sequences and, of each layer's KV cache, the rows it selects.
    lay = synth.workload_layout("decode1m")
    K, types, H = 2048, "FSSS", 64
    layers = synth.device_layers(lay, types, H, device=DEV, seed=5)
    planted = synth.plant_device(layers, lay, types, m=64, seed=5)
    L0 = layers[0]
    qc, qs = dsa.dsa_fp8_quantize(L0["q_idx"])
    kc, ks = dsa.dsa_fp8_quantize(L0["k_idx"])
    g_layers = [dict(L) for L in layers]
    g_layers[0].update(q_idx=qc, q_scale=qs, k_idx=kc, k_scale=ks)
    batch = make_batch(dsa, lay, DEV)
    g = dsa.Group(types, g_layers, k=K, scale=1 / 16)
    ws = dsa.workspace(g.workspace_size(batch), DEV)
    outs, _, idx = dsa.indexshare_group_forward(g, batch, ws=ws)
    torch.cuda.synchronize()
    dsa.status_fetch(ws)
    del kc, ks, g_layers
    rows = np.arange(lay.num_q, dtype=np.int32)
    pos, key0 = oracle.row_metadata(lay.q_start, lay.q_pos, lay.seq_row0, rows)
    sc = oracle.indexer_scores(bits(L0["q_idx"]), L0["w"].cpu().numpy(), bits(L0["k_idx"]), rows, pos,
                               key0, lay.max_len)
    ref_idx = oracle.topk(sc, pos + 1, K)
    got_idx = idx.cpu().numpy()
    for t in range(lay.num_q):  # one query per sequence
        p = set(planted[t].tolist())
        assert len(p) == 64 and p <= set(ref_idx[t].tolist()) and p <= set(got_idx[t].tolist())
    for l in range(4):
        ref_o, _ = oracle_attention_gathered(layers[l]["q_lat"], layers[l]["q_rope"], layers[l]["kv"],
                                             rows, lay.seq_row0, ref_idx, 1 / 16)
        got = outs[l].float().cpu().numpy()
        err = np.abs(got - ref_o).max()
        assert err <= 6e-2 * np.abs(ref_o).max(), (l, err, np.abs(ref_o).max())
