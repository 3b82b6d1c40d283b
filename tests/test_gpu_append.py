"""GPU parity of the indexer cache append (RoPE, then the FP8 quantiser for
the FP8 indexer) through the C ABI: keys written at their cache rows in the
contiguous and in the paged layout, queries prepared for a batch.  Both sides
rotate in fp64 with the same frequencies and round once to bf16, so the bf16
results and the FP8 codes and scales are compared bit for bit."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import synth  # noqa: E402
from gpu_helpers import bf16_dev, bits, make_batch  # noqa: E402

dsa = pytest.importorskip("dsa_indexer_indexshare_gb300")
DEV = torch.device("cuda:0")
FREQ = oracle.rope_inv_freq(8e6)


def _new_keys(lay, n, seed):
    """n new keys at random (sequence, position) pairs of the layout, positions
    spread up to each sequence's length, plus each sequence's last position."""
    rng = np.random.default_rng(seed)
    seq = rng.integers(0, lay.num_seqs, n).astype(np.int32)
    pos = (rng.random(n) * lay.seq_len[seq]).astype(np.int32)
    seq[: lay.num_seqs] = np.arange(lay.num_seqs)
    pos[: lay.num_seqs] = lay.seq_len - 1
    # distinct destination rows (a repeated row would be written twice)
    _, keep = np.unique(np.stack([seq, pos], 1), axis=0, return_index=True)
    keep = np.sort(keep)
    x = synth.f32_to_bf16_bits(rng.standard_normal((keep.size, 128)).astype(np.float32) * 2)
    return seq[keep], pos[keep], x


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("paged", [False, True])
def test_append_keys_bit_exact(fp8, paged):
    lay = synth.make_layout([1048576, 70001, 300], [1, 1, 1])
    seq, pos, x = _new_keys(lay, 3000, seed=31 + 2 * fp8 + paged)
    if paged:
        R = 1024
        nblk = [(int(n) + R - 1) // R for n in lay.seq_len]
        total = sum(nblk) + 5
        ids = np.random.default_rng(7).permutation(total)
        table = np.full((lay.num_seqs, lay.max_len // R), -1, np.int32)
        k = 0
        for b_, nb in enumerate(nblk):
            table[b_, :nb] = ids[k:k + nb]
            k += nb
        rows = np.array([oracle.paged_row(table, R, s, p) for s, p in zip(seq, pos)], np.int64)
        batch = dsa.Batch(lay.q_start, lay.q_pos, None, lay.max_len, device=DEV,
                          block_table=table, block_rows=R)
        nrows = total * R
    else:
        rows = lay.seq_row0[seq] + pos
        batch = make_batch(dsa, lay, DEV)
        nrows = lay.rows
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    fill = 0x5A
    if fp8:
        cache = torch.full((nrows, 128), fill, dtype=torch.uint8, device=DEV)
        scale = torch.full((nrows,), -1.0, dtype=torch.float32, device=DEV)
    else:
        cache = torch.full((nrows, 128), fill, dtype=torch.int16, device=DEV).view(torch.bfloat16)
        scale = None
    ws = dsa.workspace(256, DEV)
    dsa.dsa_indexer_append_keys(bf16_dev(x, DEV), T(seq), T(pos), batch, cache, FREQ,
                                k_scale=scale, ws=ws)
    assert dsa.status_fetch(ws) == 0
    ref = oracle.indexer_append(x, pos, FREQ, fp8)
    if fp8:
        got_c, got_s = cache.cpu().numpy(), scale.cpu().numpy()
        assert np.array_equal(got_c[rows], ref[0]) and np.array_equal(got_s[rows], ref[1])
        others = np.setdiff1d(np.arange(nrows), rows)
        assert (got_c[others] == fill).all() and (got_s[others] == -1.0).all()
    else:
        got = bits(cache)
        assert np.array_equal(got[rows], ref)
        others = np.setdiff1d(np.arange(nrows), rows)
        assert (got[others] == fill).all()


@pytest.mark.parametrize("fp8", [False, True])
def test_prepare_queries_bit_exact(fp8):
    lay = synth.make_layout([1048576, 4097, 129], [3, 2, 1])
    rng = np.random.default_rng(41)
    q = synth.f32_to_bf16_bits(rng.standard_normal((lay.num_q, 32, 128)).astype(np.float32))
    batch = make_batch(dsa, lay, DEV)
    got = dsa.dsa_indexer_prepare_queries(bf16_dev(q, DEV), batch, FREQ, fp8=fp8)
    posv = np.repeat(lay.q_pos, 32)
    ref = oracle.indexer_append(q.reshape(-1, 128), posv, FREQ, fp8)
    if fp8:
        assert np.array_equal(got[0].cpu().numpy().reshape(-1, 128), ref[0])
        assert np.array_equal(got[1].cpu().numpy().reshape(-1), ref[1])
    else:
        assert np.array_equal(bits(got).reshape(-1, 128), ref)


def test_append_reports_rows_outside_the_cache():
    lay = synth.make_layout([1000], [1])
    seq = np.array([0, 0, 0], np.int32)
    pos = np.array([5, 999, 7], np.int32)
    x = synth.f32_to_bf16_bits(np.ones((3, 128), np.float32))
    cache = torch.zeros((998, 128), dtype=torch.bfloat16, device=DEV)  # row 999 is missing
    ws = dsa.workspace(256, DEV)
    T = lambda a: torch.from_numpy(a).to(DEV)
    dsa.dsa_indexer_append_keys(bf16_dev(x, DEV), T(seq), T(pos), make_batch(dsa, lay, DEV), cache,
                                FREQ, ws=ws)
    with pytest.raises(dsa.DsaError) as e:
        dsa.status_fetch(ws)
    assert e.value.status == dsa.DSA_ERR_DEVICE_INDEX
    ref = oracle.indexer_append(x[[0, 2]], pos[[0, 2]], FREQ, False)
    assert np.array_equal(bits(cache)[[5, 7]], ref)  # the valid keys were written
