"""The select-only F layer (prefill rows longer than 16K positions): the
indexer's epilogue keeps only the keys at or above a cutoff taken from a
sample of each row, the top-K is resolved from those lists, and rows whose
sample misleads take the score matrix and the exact top-K instead.  Through
the group call, against the oracle's scores and top-K ("GLM-5.2 架构深度拆解"
CH 2.2: top-2048 per query; "GLM-5 -> 5.1 -> 5.2" section 10: the indices
written once per group).

Scores are made exact: every head of every query is the unit vector e0 and
only head 0 has weight 1, so score(t, s) = ReLU(k[s, 0]) with k[s, 0] a
small integer (exact in bf16 and in fp32).  The cases:
  * random integers 0..255 (many ties: the position tie-break decides), on
    rows of 30-40K positions and on rows of 300K;
  * a drift, k[s, 0] = s // 1000, so the selected keys all lie in the last
    key chunk and overflow its segments of the capture list (the fallback);
  * a misleading sample: a large value planted only inside the tiles the
    sample reads (22 keys of each), so that fewer than K keys clear the
    cutoff (the fallback), with K = 4096;
  * the FP8 indexer on Gaussian vectors (codes from the library's quantiser,
    scored by the oracle; equal up to the tie band).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import synth  # noqa: E402
from gpu_helpers import assert_topk_within_band, bf16_dev, bits, make_batch  # noqa: E402

dsa = pytest.importorskip("dsa_indexer_indexshare_gb300")
DEV = torch.device("cuda:0")


def _layers(lay, k0, dev):
    """One F layer with score(t, s) = ReLU(k0[s]) (k0 small integers)."""
    nq, rows = lay.num_q, lay.rows
    q = np.zeros((nq, 32, 128), np.float32)
    q[:, :, 0] = 1.0
    w = np.zeros((nq, 32), np.float32)
    w[:, 0] = 1.0
    k = np.zeros((rows, 128), np.float32)
    k[:, 0] = k0
    host = {"q_idx": synth.f32_to_bf16_bits(q), "w": w, "k_idx": synth.f32_to_bf16_bits(k)}
    d = {"q_idx": bf16_dev(host["q_idx"], dev), "w": torch.from_numpy(w).to(dev),
         "k_idx": bf16_dev(host["k_idx"], dev),
         "q_lat": torch.zeros((nq, 64, 512), dtype=torch.bfloat16, device=dev),
         "q_rope": torch.zeros((nq, 64, 64), dtype=torch.bfloat16, device=dev),
         "kv": torch.zeros((rows, 576), dtype=torch.bfloat16, device=dev)}
    return host, d


def _group_indices(lay, d, K):
    batch = make_batch(dsa, lay, DEV)
    group = dsa.Group("F", [d], k=K, scale=1 / 16)
    ws = dsa.workspace(group.workspace_size(batch), DEV)
    _, _, idx = dsa.indexshare_group_forward(group, batch, ws=ws)
    torch.cuda.synchronize()
    dsa.status_fetch(ws)
    return idx.cpu().numpy()


def _oracle_topk(lay, host, K, **kw):
    rows = np.arange(lay.num_q, dtype=np.int32)
    pos, key0 = oracle.row_metadata(lay.q_start, lay.q_pos, lay.seq_row0, rows)
    sc = oracle.indexer_scores(host["q_idx"], host["w"], host["k_idx"], rows, pos, key0,
                               lay.max_len, **kw)
    return sc, pos + 1, oracle.topk(sc, pos + 1, K)


def _per_seq(lay, f):
    """k0 for every cache row: f(position) within each sequence."""
    k0 = np.zeros(lay.rows, np.float32)
    for b in range(lay.num_seqs):
        n = int(lay.seq_len[b])
        k0[int(lay.seq_row0[b]):int(lay.seq_row0[b]) + n] = f(np.arange(n))
    return k0


@pytest.mark.parametrize("case", ["random", "drift", "long"])
def test_select_only_equals_oracle_topk(case):
    # "long": rows beyond 262,144 positions, whose taken positions are sorted
    # into order rather than compacted from a bitmap over the row
    lens, counts = ([300000, 20000], [8, 8]) if case == "long" else ([40000, 30000], [16, 8])
    lay = synth.make_layout(lens, counts)
    rng = np.random.default_rng(5)
    if case in ("random", "long"):
        k0 = rng.integers(0, 256, lay.rows).astype(np.float32)
    else:
        k0 = _per_seq(lay, lambda s: (s // 1000).astype(np.float32))
    host, d = _layers(lay, k0, DEV)
    got = _group_indices(lay, d, 2048)
    _, _, ref = _oracle_topk(lay, host, 2048)
    assert np.array_equal(got, ref)


def test_select_only_misleading_sample_takes_the_exact_path():
    # one block of 8 queries at the end of a 40000-position row: the sample
    # reads 32 tiles of 128 keys, tile i starting at 128 * floor(i * 313 / 32)
    L, K = 40000, 4096
    lay = synth.make_layout([L], [8])
    rng = np.random.default_rng(6)
    k0 = rng.integers(0, 4, lay.rows).astype(np.float32)
    T = (L - 1) // 128 + 1
    for i in range(32):
        start = (i * T // 32) * 128
        k0[start:start + 22] = 100.0
    host, d = _layers(lay, k0, DEV)
    got = _group_indices(lay, d, K)
    _, _, ref = _oracle_topk(lay, host, K)
    assert np.array_equal(got, ref)


def test_select_only_fp8_indexer_within_tie_band():
    lay = synth.make_layout([36000], [24])
    rng = np.random.default_rng(7)
    q = (rng.standard_normal((lay.num_q, 32, 128)) / np.sqrt(128)).astype(np.float32)
    k = (rng.standard_normal((lay.rows, 128)) / np.sqrt(128)).astype(np.float32)
    w = rng.standard_normal((lay.num_q, 32)).astype(np.float32)
    qc, qs = dsa.dsa_fp8_quantize(bf16_dev(synth.f32_to_bf16_bits(q), DEV))
    kc, ks = dsa.dsa_fp8_quantize(bf16_dev(synth.f32_to_bf16_bits(k), DEV))
    d = {"q_idx": qc, "q_scale": qs, "w": torch.from_numpy(w).to(DEV), "k_idx": kc, "k_scale": ks,
         "q_lat": torch.zeros((lay.num_q, 64, 512), dtype=torch.bfloat16, device=DEV),
         "q_rope": torch.zeros((lay.num_q, 64, 64), dtype=torch.bfloat16, device=DEV),
         "kv": torch.zeros((lay.rows, 576), dtype=torch.bfloat16, device=DEV)}
    got = _group_indices(lay, d, 2048)
    host = {"q_idx": qc.cpu().numpy(), "w": w, "k_idx": kc.cpu().numpy()}
    sc, lens, _ = _oracle_topk(lay, host, 2048, dtype=1, q_scale=qs.cpu().numpy(),
                               k_scale=ks.cpu().numpy())
    assert_topk_within_band(got, sc, lens, 2048, what="select-only fp8")
