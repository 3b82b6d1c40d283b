"""GPU parity of the FP8 indexer variant against the bf16 pipeline: the
group call with the library's FP8 quantiser on the indexer inputs stays
within 6e-2 * max|ref| of the oracle run on the unquantised bf16 inputs, on
inputs with a planted set of relevant positions (see synth's
planted_host_layers)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import synth  # noqa: E402
from gpu_helpers import device_layers, make_batch  # noqa: E402

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
