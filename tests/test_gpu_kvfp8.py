"""GPU parity of the FP8 KV latent path through the C ABI: the KV quantiser
bit for bit against the oracle; sparse MLA over FP8 rows bit for bit against
the bf16 kernel run on the oracle's dequantised rows (same bf16 operands),
and within the attention tolerance against the oracle; the group call with
FP8 caches, contiguous and paged."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import synth  # noqa: E402
from gpu_helpers import assert_close, bf16_dev, device_layers, make_batch  # noqa: E402

dsa = pytest.importorskip("dsa_indexer_indexshare_gb300")
DEV = torch.device("cuda:0")


def _kv_rows(n, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, 576)).astype(np.float32) / np.float32(np.sqrt(512))
    x[3, :128] = 0             # an all-zero group
    x[4, 128:256] *= 1e3       # a large group
    x[5, 256:384] *= 1e-4      # a small one (subnormal E4M3 codes)
    return synth.f32_to_bf16_bits(x)


def test_kv_quantiser_bit_exact():
    kv = _kv_rows(5000, 1)
    got = dsa.dsa_kv_fp8_quantize(bf16_dev(kv, DEV)).cpu().numpy()
    assert np.array_equal(got, oracle.kv_fp8_quantize(kv))


def _indices(lay, K, seed):
    rng = np.random.default_rng(seed)
    idx = np.full((lay.num_q, K), -1, np.int32)
    for t in range(lay.num_q):
        n = int(lay.q_pos[t]) + 1
        idx[t, :min(n, K)] = np.sort(rng.choice(n, min(n, K), replace=False))
    return idx


@pytest.mark.parametrize("case", ["prefill", "decode"])
def test_sparse_mla_fp8_kv(case):
    if case == "prefill":
        lay, K = synth.make_layout([1500], [300]), 512
    else:
        lay, K = synth.make_layout([3000, 9000, 700], [1, 1, 1]), 2048  # cluster split-K
    host = synth.host_layers(lay, "S", 64, ints=False, seed=2)[0]
    kv8 = oracle.kv_fp8_quantize(host["kv"])
    kv_deq = oracle.kv_fp8_dequantize(kv8)
    idx = torch.from_numpy(_indices(lay, K, 3)).to(DEV)
    batch = make_batch(dsa, lay, DEV)
    ql, qr = bf16_dev(host["q_lat"], DEV), bf16_dev(host["q_rope"], DEV)
    o8, l8 = dsa.dsa_sparse_mla_attn(ql, qr, torch.from_numpy(kv8).to(DEV), idx, batch,
                                     scale=1 / 16)
    ob, lb = dsa.dsa_sparse_mla_attn(ql, qr, bf16_dev(kv_deq, DEV), idx, batch, scale=1 / 16)
    assert torch.equal(o8, ob) and torch.equal(l8, lb)
    rows = np.arange(lay.num_q, dtype=np.int32)
    pos, key0 = oracle.row_metadata(lay.q_start, lay.q_pos, lay.seq_row0, rows)
    ref_o, _ = oracle.sparse_mla(host["q_lat"], host["q_rope"], kv_deq, rows, key0,
                                 idx.cpu().numpy(), 1 / 16)
    assert_close(o8.float().cpu().numpy(), ref_o, 2e-2, "FP8 KV out")


@pytest.mark.parametrize("paged", [False, True])
def test_group_fp8_kv_matches_bf16_on_dequantised(paged):
    lay = synth.make_layout([1200, 700], [200, 100])
    types, K = "FSSS", 256
    host = synth.host_layers(lay, types, 64, ints=False, seed=4)
    deq = [dict(L, kv=oracle.kv_fp8_dequantize(oracle.kv_fp8_quantize(L["kv"]))) for L in host]
    lay_batch = make_batch(dsa, lay, DEV)
    table = None
    if paged:  # identity-free layout: blocks of 256 positions in reverse order
        R = 256
        nb = [(int(n) + R - 1) // R for n in lay.seq_len]
        total = sum(nb)
        ids = np.arange(total)[::-1]
        table = np.full((lay.num_seqs, lay.max_len // R), -1, np.int32)
        phys = np.empty(lay.rows, np.int64)
        k = 0
        for b, n in enumerate(lay.seq_len):
            table[b, :nb[b]] = ids[k:k + nb[b]]
            s = np.arange(int(n))
            phys[int(lay.seq_row0[b]) + s] = table[b, s // R].astype(np.int64) * R + s % R
            k += nb[b]
        lay_batch = dsa.Batch(lay.q_start, lay.q_pos, None, lay.max_len, device=DEV,
                              block_table=table, block_rows=R)

    def place(a):  # logical rows -> the batch layout's rows
        if table is None:
            return a
        out = np.zeros((sum((int(n) + 255) // 256 for n in lay.seq_len) * 256,) + a.shape[1:],
                       a.dtype)
        out[phys] = a
        return out

    results = []
    for hl, fp8 in ((deq, False), (host, True)):
        layers = device_layers([dict(L, kv=place(L["kv"]), **({"k_idx": place(L["k_idx"])}
                                                            if "k_idx" in L else {}))
                                for L in hl], DEV)
        if fp8:
            for L, h in zip(layers, hl):
                L["kv"] = torch.from_numpy(place(oracle.kv_fp8_quantize(h["kv"]))).to(DEV)
        g = dsa.Group(types, layers, k=K, scale=1 / 16, with_lse=True)
        ws = dsa.workspace(g.workspace_size(lay_batch), DEV)
        outs, lses, idx = dsa.indexshare_group_forward(g, lay_batch, ws=ws)
        torch.cuda.synchronize()
        dsa.status_fetch(ws)
        results.append(([o.clone() for o in outs], idx.clone()))
    (ob, ib), (o8, i8) = results
    assert torch.equal(ib, i8)
    for a, b in zip(ob, o8):
        assert torch.equal(a, b)
