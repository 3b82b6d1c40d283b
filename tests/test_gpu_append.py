"""GPU parity of the indexer cache append (RoPE, then the FP8 quantiser for
the FP8 indexer) through the C ABI: keys written at their cache rows in the
contiguous and in the paged layout, queries prepared for a batch.

bf16 results: the oracle rotates in fp64 and rounds once to bf16; the kernel
rounds its own value of the same rotation once.  They are compared bit for
bit, except that a result may differ by one bf16 unit where the fp64 value
lies within 2^-44 * (|x0| + |x1|) of the midpoint between two bf16 values
(the two computations' error bounds: the kernel's rotation and the libm
sin/cos of each side), so that no difference in the last bits of fp64
arithmetic can fail the test spuriously.  FP8 results: the codes and scales
obey the comparison rule of tests/fp8_rule.py against the oracle's
quantisation of the oracle's bf16 RoPE output."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import synth  # noqa: E402
from fp8_rule import check_fp8_rows  # noqa: E402
from gpu_helpers import bf16_dev, bits, make_batch  # noqa: E402

dsa = pytest.importorskip("dsa_indexer_indexshare_gb300")
DEV = torch.device("cuda:0")
FREQ = oracle.rope_inv_freq(8e6)


def assert_rope_bf16(got, ref, x, pos):
    """got, ref: bf16 bits [n, 128] of the kernel and the oracle for inputs x
    (bf16 bits [n, 128]) at positions pos [n]."""
    got = np.asarray(got, np.uint16).reshape(-1, 128)
    ref = np.asarray(ref, np.uint16).reshape(-1, 128)
    diff = np.argwhere(got != ref)
    if diff.size == 0:
        return
    xv = synth.bf16_bits_to_f32(np.asarray(x).reshape(-1, 128)).astype(np.float64)
    for r, d in diff:
        assert d < 64, f"row {r} dim {d}: a copied entry differs"
        i = d // 2
        a = float(pos[r]) * FREQ[i]
        x0, x1 = xv[r, 2 * i], xv[r, 2 * i + 1]
        v = x0 * np.cos(a) - x1 * np.sin(a) if d % 2 == 0 else x0 * np.sin(a) + x1 * np.cos(a)
        g, f = int(got[r, d]), int(ref[r, d])
        assert abs(g - f) == 1 and (g >> 15) == (f >> 15), f"row {r} dim {d}: not one bf16 unit"
        lo, hi = sorted((synth.bf16_bits_to_f32(np.array([g], np.uint16))[0],
                         synth.bf16_bits_to_f32(np.array([f], np.uint16))[0]))
        mid = (float(lo) + float(hi)) / 2
        assert abs(v - mid) <= 2.0 ** -44 * (abs(x0) + abs(x1)), (
            f"row {r} dim {d}: value {v!r} is not within the band of the midpoint {mid!r}")
    assert len(diff) <= max(1, 1e-6 * got.size)


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
    if fp8:
        got_c, got_s = cache.cpu().numpy(), scale.cpu().numpy()
        check_fp8_rows(got_c[rows], got_s[rows], oracle.rope_bf16(x, pos, FREQ), what="appended keys")
        others = np.setdiff1d(np.arange(nrows), rows)
        assert (got_c[others] == fill).all() and (got_s[others] == -1.0).all()
    else:
        got = bits(cache)
        assert_rope_bf16(got[rows], oracle.indexer_append(x, pos, FREQ, False), x, pos)
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
    if fp8:
        check_fp8_rows(got[0].cpu().numpy().reshape(-1, 128), got[1].cpu().numpy().reshape(-1),
                       oracle.rope_bf16(q.reshape(-1, 128), posv, FREQ), what="prepared queries")
    else:
        assert_rope_bf16(bits(got).reshape(-1, 128),
                         oracle.indexer_append(q.reshape(-1, 128), posv, FREQ, False),
                         q.reshape(-1, 128), posv)


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
    assert_rope_bf16(bits(cache)[[5, 7]], ref, x[[0, 2]], pos[[0, 2]])  # the valid keys were written
