"""GPU parity of each hot-path step against the oracle, through the C ABI.

Bars: integer-valued inputs give bit-exact scores and index
sets; Gaussian inputs give index sets that differ only within 1e-3 of the
K-th score; attention outputs within 2e-2 * max|ref| (bf16)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import synth  # noqa: E402
from fp8_rule import check_fp8_rows  # noqa: E402
from gpu_helpers import (assert_close, assert_topk_within_band, bf16_dev, bits,  # noqa: E402
                         device_layers, make_batch)

dsa = pytest.importorskip("dsa_indexer_indexshare_gb300")
DEV = torch.device("cuda:0")


def rows_meta(lay, rows):
    return oracle.row_metadata(lay.q_start, lay.q_pos, lay.seq_row0, rows)


LAYOUTS = {
    "prefill512": ([512], [512]),
    "ragged3": ([300, 77, 1000], [300, 5, 129]),
    "decode5": ([1, 129, 1000, 4097, 256], [1, 1, 1, 1, 1]),
    "empty_middle": ([200, 50, 333], [17, 0, 40]),
}


@pytest.mark.parametrize("name", list(LAYOUTS))
def test_indexer_scores_bit_exact_on_integers(name):
    lay = synth.make_layout(*LAYOUTS[name])
    host = synth.host_layers(lay, "F", 16, ints=True, seed=3)[0]
    d = device_layers([host], DEV)[0]
    batch = make_batch(dsa, lay, DEV)
    ws = dsa.workspace(256, DEV)
    sc = dsa.dsa_indexer_scores(d["q_idx"], d["w"], d["k_idx"], batch, ws=ws)
    dsa.status_fetch(ws)
    rows = np.arange(lay.num_q, dtype=np.int32)
    pos, key0 = rows_meta(lay, rows)
    ref = oracle.indexer_scores(host["q_idx"], host["w"], host["k_idx"], rows, pos, key0, lay.max_len)
    got = sc.cpu().numpy().astype(np.float64)
    assert np.array_equal(got, ref)


def test_indexer_scores_gaussian_fp32_accuracy():
    lay = synth.make_layout([1000], [1000])
    host = synth.host_layers(lay, "F", 16, ints=False, seed=4)[0]
    d = device_layers([host], DEV)[0]
    batch = make_batch(dsa, lay, DEV)
    sc = dsa.dsa_indexer_scores(d["q_idx"], d["w"], d["k_idx"], batch).cpu().numpy()
    rows = np.arange(lay.num_q, dtype=np.int32)
    pos, key0 = rows_meta(lay, rows)
    ref = oracle.indexer_scores(host["q_idx"], host["w"], host["k_idx"], rows, pos, key0, lay.max_len)
    fin = np.isfinite(ref)
    assert np.array_equal(fin, np.isfinite(sc))
    # fp32 tensor-core accumulation of exact bf16 products + fp32 head reduction
    assert np.abs(sc[fin] - ref[fin]).max() <= 1e-5 * np.abs(ref[fin]).max()


def _topk_case(lens, qcounts, K, values, seed):
    lay = synth.make_layout(lens, qcounts)
    rng = np.random.default_rng(seed)
    if values == "ties":
        sc = rng.integers(-3, 4, (lay.num_q, lay.max_len)).astype(np.float32)
    elif values == "gauss":
        sc = rng.standard_normal((lay.num_q, lay.max_len)).astype(np.float32)
    elif values == "signed_zeros":  # +0 and -0 are equal scores: ties go to the lower position
        sc = rng.choice(np.array([0.0, -0.0, 1.0, -1.0], np.float32), (lay.num_q, lay.max_len),
                        p=[0.45, 0.45, 0.02, 0.08])
    else:  # constant rows
        sc = np.zeros((lay.num_q, lay.max_len), np.float32)
    sc[0, : min(5, sc.shape[1])] = -np.inf
    batch = make_batch(dsa, lay, DEV)
    ws = dsa.workspace(dsa.lib.dsa_topk_workspace_size(batch.c, K), DEV)
    got = dsa.dsa_topk(torch.from_numpy(sc).to(DEV), batch, K, ws=ws).cpu().numpy()
    dsa.status_fetch(ws)
    lens_q = lay.q_pos.astype(np.int64) + 1
    ref = oracle.topk(sc.astype(np.float64), lens_q.astype(np.int32), K)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("values", ["ties", "gauss", "const", "signed_zeros"])
def test_topk_bit_exact_short_rows(values):
    _topk_case([3000], [3000], 64, values, 1)          # one CTA per row, 256 threads
    _topk_case([5000, 20000], [40, 60], 2048, values, 2)  # 1024-thread rows, pos+1 <= K rows


@pytest.mark.parametrize("values", ["ties", "gauss", "const", "signed_zeros"])
def test_topk_bit_exact_long_rows(values):
    # fewer than 80 rows beyond 16K positions: cutoff / capture /
    # resolve-and-write launches (constant and 7-valued rows overflow the
    # capture list and go to the fallback); rows beyond 262,144 positions
    # are sorted into order rather than compacted from a bitmap
    _topk_case([40000, 70001, 131072], [1, 1, 1], 2048, values, 3)
    _topk_case([1 << 20, 300000], [1, 1], 2048, values, 4)
    # 79 rows: the same path; 103 rows: one persistent CTA per SM
    _topk_case([20000, 17000, 131072], [40, 36, 3], 2048, values, 7)
    _topk_case([20000, 17000, 131072], [60, 40, 3], 2048, values, 8)


@pytest.mark.parametrize("values", ["ties", "gauss"])
def test_topk_bit_exact_sort_widths(values):
    # the ordered write's sort at each width: few long rows (512 threads)
    # with K = 300 (one entry per thread) and 4096 (eight); the persistent
    # kernel (1024 threads, 80 rows) on a row beyond its 917,504-position
    # bitmap (two entries per thread at K = 2048).  Integer rows overflow
    # the few-rows capture and take the persistent kernel's sort instead.
    _topk_case([300000, 270000], [1, 1], 300, values, 11)
    _topk_case([300000, 270000], [1, 1], 4096, values, 12)
    _topk_case([1000000] + [20000] * 79, [1] * 80, 2048, values, 13)


@pytest.mark.parametrize("values", ["ties", "gauss", "const", "signed_zeros"])
def test_topk_bit_exact_many_long_rows(values):
    # hundreds of rows beyond 16K positions: one persistent CTA per SM, two
    # reads per row (constant rows overflow the member buffer and rescan);
    # the second sequence's rows have pos + 1 <= K
    _topk_case([40000, 1500], [390, 20], 2048, values, 6)


@pytest.mark.parametrize("values", ["ties", "gauss", "const", "signed_zeros"])
def test_topk_bit_exact_few_short_rows_cluster(values):
    _topk_case([9000, 16000, 3000], [1, 2, 1], 512, values, 5)  # cluster of 8, staged


def _mla_case(lens, qcounts, H, K, ints, seed, sample=None, bad_index=False, holes=False):
    lay = synth.make_layout(lens, qcounts)
    host = synth.host_layers(lay, "S", H, ints=ints, seed=seed)[0]
    rng = np.random.default_rng(seed)
    # indices: a random distinct subset of visible positions, ascending, -1 padded
    idx = np.full((lay.num_q, K), -1, np.int32)
    for t in range(lay.num_q):
        n = int(lay.q_pos[t]) + 1
        take = min(n, K)
        sel = np.sort(rng.choice(n, take, replace=False))
        if holes and take > 10:
            sel = sel[: take // 2]
        idx[t, : len(sel)] = sel
    if bad_index:
        idx[0, 0] = int(lay.q_pos[0]) + 5       # beyond the causal range
    d = device_layers([host], DEV)[0]
    batch = make_batch(dsa, lay, DEV)
    ws = dsa.workspace(dsa.lib.dsa_sparse_mla_workspace_size(batch.c, H, K), DEV)
    out, lse = dsa.dsa_sparse_mla_attn(d["q_lat"], d["q_rope"], d["kv"], torch.from_numpy(idx).to(DEV),
                                       batch, scale=1 / 16, ws=ws)
    if bad_index:
        with pytest.raises(dsa.DsaError) as e:
            dsa.status_fetch(ws)
        assert e.value.status == dsa.DSA_ERR_DEVICE_INDEX
        idx[0, 0] = -1
    else:
        dsa.status_fetch(ws)
    rows = np.arange(lay.num_q, dtype=np.int32) if sample is None else np.asarray(sample, np.int32)
    pos, key0 = rows_meta(lay, rows)
    ref_o, ref_l = oracle.sparse_mla(host["q_lat"][rows], host["q_rope"][rows], host["kv"],
                                     np.arange(len(rows), dtype=np.int32), key0, idx[rows], 1 / 16)
    got = out.float().cpu().numpy()[rows]
    assert_close(got, ref_o, 2e-2, "out")
    gl = lse.cpu().numpy()[rows]
    assert np.allclose(gl, ref_l, rtol=0, atol=1e-3 * max(1.0, np.abs(ref_l).max()))


def test_mla_h16_k64_integers():
    _mla_case([300], [300], 16, 64, True, 5)


def test_mla_h64_k2048_gaussian_prefill():
    sample = [0, 1, 126, 127, 128, 2046, 2047, 2048, 2049, 2599]
    _mla_case([2600], [2600], 64, 2048, False, 6, sample=sample)


def test_mla_h64_decode_split_clusters():
    # 4 tokens: clusters of 16 CTAs (partial results combined through L2;
    # the short rows leave some CTAs without blocks)
    _mla_case([100000, 3000, 2047, 4100], [1, 1, 1, 1], 64, 2048, False, 7)
    # 6 tokens: clusters of 8 CTAs
    _mla_case([3000 + 517 * i for i in range(6)], [1] * 6, 64, 2048, False, 10)
    # 24 tokens: clusters of 4 CTAs
    lens = [2100 + 157 * i for i in range(24)]
    _mla_case(lens, [1] * 24, 64, 2048, False, 9, sample=[0, 5, 11, 23])


def test_mla_holes_and_bad_index():
    _mla_case([700, 300], [20, 30], 64, 256, False, 8, holes=True, bad_index=True)


def test_mla_h16_ragged_batch():
    _mla_case([300, 77, 1000], [300, 5, 129], 16, 128, False, 9)


def _mla_both_kernels(lens, qcounts, K, seed, holes=False, bad_pos=None, sample=(), page_rows=0):
    """64 heads, bf16 rows, at least twice as many tokens as SMs: the
    persistent grid and the CTA-per-token kernel give bit-identical outputs
    and lse (on paged caches also equal to the contiguous cache's); sampled
    rows match the oracle; a query at an invalid position gets zeros and
    lse = -inf from both (and the batch error)."""
    lay = synth.make_layout(lens, qcounts)
    assert lay.num_q >= 2 * torch.cuda.get_device_properties(DEV).multi_processor_count
    H = 64
    host = synth.host_layers(lay, "S", H, ints=False, seed=seed)[0]
    rng = np.random.default_rng(seed)
    idx = np.full((lay.num_q, K), -1, np.int32)
    for t in range(lay.num_q):
        n = int(lay.q_pos[t]) + 1
        take = min(n, K)
        sel = np.sort(rng.choice(n, take, replace=False))
        if holes and t % 3 == 0 and take > 10:
            sel = sel[: take // 2]
        idx[t, : len(sel)] = sel
    q_pos = lay.q_pos.copy()
    if bad_pos is not None:
        q_pos[bad_pos] = lay.max_len  # outside [0, max_len)
    d = device_layers([host], DEV)[0]
    idx_d = torch.from_numpy(idx).to(DEV)
    contiguous = dsa.Batch(lay.q_start, q_pos, lay.seq_row0, lay.max_len, device=DEV)

    def run(batch, kv, persistent):
        out = torch.full((lay.num_q, H, 512), 3.0, dtype=torch.bfloat16, device=DEV)
        lse = torch.full((lay.num_q, H), 5.0, dtype=torch.float32, device=DEV)
        ws = dsa.workspace(dsa.lib.dsa_sparse_mla_workspace_size(batch.c, H, K), DEV)
        dsa.set_mla_persistent(persistent)
        try:
            dsa.dsa_sparse_mla_attn(d["q_lat"], d["q_rope"], kv, idx_d, batch, scale=1 / 16,
                                    out=out, lse=lse, ws=ws)
        finally:
            dsa.set_mla_persistent(True)
        if bad_pos is None:
            dsa.status_fetch(ws)
        else:
            with pytest.raises(dsa.DsaError) as e:
                dsa.status_fetch(ws)
            assert e.value.status == dsa.DSA_ERR_DEVICE_INDEX
        return bits(out), lse.cpu().numpy()

    if page_rows:
        table, (kv_paged,) = _page(lay, [host["kv"]], page_rows, seed=seed + 1)
        batch = dsa.Batch(lay.q_start, q_pos, None, lay.max_len, device=DEV, block_table=table,
                          block_rows=page_rows)
        kv = bf16_dev(kv_paged, DEV)
    else:
        batch, kv = contiguous, d["kv"]
    (op, lp), (ot, lt) = run(batch, kv, True), run(batch, kv, False)
    assert np.array_equal(op, ot), "outputs differ between the two kernels"
    assert np.array_equal(lp.view(np.uint32), lt.view(np.uint32)), "lse differs between the two kernels"
    if page_rows:
        oc, lc = run(contiguous, d["kv"], True)
        assert np.array_equal(op, oc) and np.array_equal(lp.view(np.uint32), lc.view(np.uint32)), \
            "paged and contiguous caches give different results"
    if bad_pos is not None:
        assert not op[bad_pos].any() and np.all(lp[bad_pos] == -np.inf)
    rows = np.asarray([r for r in sample if r != bad_pos], np.int32)
    pos, key0 = rows_meta(lay, rows)
    ref_o, ref_l = oracle.sparse_mla(host["q_lat"][rows], host["q_rope"][rows], host["kv"],
                                     np.arange(len(rows), dtype=np.int32), key0, idx[rows], 1 / 16)
    o = op[rows].view(np.uint16).astype(np.uint32) << 16
    assert_close(o.view(np.float32), ref_o, 2e-2, "out")
    assert np.allclose(lp[rows], ref_l, rtol=0, atol=1e-3 * max(1.0, np.abs(ref_l).max()))


def test_mla_persistent_grid_matches_per_token_kernel():
    # three sequences of unequal query counts, short index rows and holes
    _mla_both_kernels([3000, 700, 1500], [400, 300, 1000], 512, 21, holes=True,
                      sample=[0, 1, 399, 400, 699, 700, 1100, 1699])
    # 200 sequences (one of 200 queries, 199 of one): 40000 work items, more
    # than 256 per SM, so the grid outgrows the SM count; most items are past
    # their sequence's end; one query at an invalid position
    _mla_both_kernels([300] + [50] * 199, [200] + [1] * 199, 128, 22, bad_pos=5,
                      sample=[0, 4, 6, 199, 200, 398])
    # 304 sequences, one of 400 queries and 303 of one: 121,600 work items over
    # 475 CTAs for 703 tokens, so some CTAs get an empty list
    _mla_both_kernels([500] + [30] * 303, [400] + [1] * 303, 64, 27,
                      sample=[0, 1, 399, 400, 702])
    # paged caches (blocks of 128 positions over a permuted pool): two sequences
    _mla_both_kernels([2500, 1300], [700, 400], 1024, 23, holes=True, page_rows=128,
                      sample=[0, 1, 699, 700, 1099])


@pytest.mark.parametrize("types", ["FSSS", "FFFF", "FSSSFSSS"])
def test_group_tiny_bit_exact_indices(types):
    lay = synth.workload_layout("tiny")
    H, K = 16, 64
    host = synth.host_layers(lay, types, H, ints=True, seed=11)
    layers = device_layers(host, DEV)
    batch = make_batch(dsa, lay, DEV)
    group = dsa.Group(types, layers, k=K, scale=1 / 16, with_lse=True)
    ws = dsa.workspace(group.workspace_size(batch), DEV)
    dsa.launch_counts_reset()
    outs, lses, idx = dsa.indexshare_group_forward(group, batch, ws=ws)
    torch.cuda.synchronize()
    counts = dsa.launch_counts()
    dsa.status_fetch(ws)
    nf = types.count("F")
    assert counts["indexer"] == nf and counts["topk"] == nf and counts["sparse_mla"] == len(types)
    rows = np.arange(lay.num_q, dtype=np.int32)
    pos, key0 = rows_meta(lay, rows)
    ref = oracle.group_forward(types, host, rows, pos, key0, lay.max_len, K, 1 / 16)
    assert np.array_equal(idx.cpu().numpy(), ref["idx"][-1])
    for l in range(len(types)):
        assert_close(outs[l].float().cpu().numpy(), ref["out"][l], 2e-2, f"layer {l}")
    # an S layer is the standalone sparse MLA over the same buffer, bit for bit
    # (indices of the last F layer are in idx_buf after the call)
    last_f = types.rfind("F")
    for l in range(last_f, len(types)):
        o, _ = dsa.dsa_sparse_mla_attn(layers[l]["q_lat"], layers[l]["q_rope"], layers[l]["kv"], idx,
                                       batch, scale=1 / 16)
        assert torch.equal(o, outs[l])


def _page(lay, arrays, R, seed, spare=3):
    """Paged copies of per-position cache arrays (rows in the layout's
    contiguous order): every sequence's blocks of R positions land in a
    random permutation of physical blocks, with spare blocks left unused.
    Returns the block table and the paged arrays."""
    rng = np.random.default_rng(seed)
    lens = [int(n) for n in lay.seq_len]
    nblk = [(n + R - 1) // R for n in lens]
    bps = lay.max_len // R + (lay.max_len % R != 0)
    total = sum(nblk) + spare
    ids = rng.permutation(total)
    table = np.full((len(lens), bps), -1, np.int32)
    paged = [np.zeros((total * R,) + a.shape[1:], a.dtype) for a in arrays]
    k = 0
    for b, n in enumerate(lens):
        r0 = int(lay.seq_row0[b])
        for j in range(nblk[b]):
            table[b, j] = ids[k]
            m = min(R, n - j * R)
            for a, pa in zip(arrays, paged):
                pa[ids[k] * R: ids[k] * R + m] = a[r0 + j * R: r0 + j * R + m]
            k += 1
    return table, paged


def test_paged_caches_match_contiguous_and_oracle():
    # two sequences, blocks of 256 positions scattered over a permuted pool
    lay = synth.make_layout([700, 400], [300, 200])
    types, H, K, R = "FSSS", 16, 64, 256
    host = synth.host_layers(lay, types, H, ints=True, seed=21)
    keys = ["kv", "k_idx"]
    table = None
    paged_host = []
    for l, L in enumerate(host):
        arrs = [L[k] for k in keys if k in L]
        table, parr = _page(lay, arrs, R, seed=22)  # same table for every layer
        P = dict(L)
        for k, a in zip([k for k in keys if k in L], parr):
            P[k] = a
            # the oracle's row map gives back the logical cache
            assert np.array_equal(oracle.logical_cache(a, table, R, lay.seq_len), L[k])
        paged_host.append(P)
    contiguous = make_batch(dsa, lay, DEV)
    paged = dsa.Batch(lay.q_start, lay.q_pos, None, lay.max_len, device=DEV, block_table=table,
                      block_rows=R)
    results = []
    for hl, batch in ((host, contiguous), (paged_host, paged)):
        layers = device_layers(hl, DEV)
        group = dsa.Group(types, layers, k=K, scale=1 / 16, with_lse=True)
        ws = dsa.workspace(group.workspace_size(batch), DEV)
        outs, lses, idx = dsa.indexshare_group_forward(group, batch, ws=ws)
        torch.cuda.synchronize()
        dsa.status_fetch(ws)
        results.append(([o.clone() for o in outs], idx.clone()))
    (oc, ic), (op, ip) = results
    assert torch.equal(ic, ip)
    for a, b_ in zip(oc, op):
        assert torch.equal(a, b_)
    rows = np.arange(lay.num_q, dtype=np.int32)
    pos, key0 = rows_meta(lay, rows)
    ref = oracle.group_forward(types, host, rows, pos, key0, lay.max_len, K, 1 / 16)
    assert np.array_equal(ip.cpu().numpy(), ref["idx"][-1])
    for l in range(len(types)):
        assert_close(op[l].float().cpu().numpy(), ref["out"][l], 2e-2, f"paged layer {l}")


def test_paged_fp8_indexer_scores_match_contiguous():
    lay = synth.make_layout([1500, 2300], [3, 2])
    host = synth.host_layers(lay, "F", 16, ints=False, seed=23)[0]
    qc, qs = oracle.fp8_quantize_rows(host["q_idx"].reshape(-1, 128))
    kc, ks = oracle.fp8_quantize_rows(host["k_idx"])
    R = 512
    table, (kcp, ksp) = _page(lay, [kc, ks], R, seed=24)
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    qc_d, qs_d, w_d = T(qc.reshape(lay.num_q, 32, 128)), T(qs.reshape(lay.num_q, 32)), T(host["w"])
    sc = dsa.dsa_indexer_scores(qc_d, w_d, T(kc), make_batch(dsa, lay, DEV), q_scale=qs_d,
                                k_scale=T(ks))
    paged = dsa.Batch(lay.q_start, lay.q_pos, None, lay.max_len, device=DEV, block_table=table,
                      block_rows=R)
    scp = dsa.dsa_indexer_scores(qc_d, w_d, T(kcp), paged, q_scale=qs_d, k_scale=T(ksp))
    assert torch.equal(sc, scp)


def test_fp8_quantiser_matches_definition():
    # the library's fp32 quantiser against the oracle's definition (fp64
    # rotation, nearest fp32 scale, nearest E4M3 code): equal codes except a
    # code step within the fp32 error bound of an E4M3 rounding boundary,
    # and those rare (tests/fp8_rule.py states the rule and its bound)
    rng = np.random.default_rng(12)
    x = rng.standard_normal((20011, 128)).astype(np.float32) / np.sqrt(128)
    x[7] = 0
    x[8] *= 1e4
    x[9, :3] = [1e-30, -3e38, 2.5]
    x[10] = 0
    x[10, 5] = -1.0
    xb = synth.f32_to_bf16_bits(x)
    codes, scale = dsa.dsa_fp8_quantize(bf16_dev(xb, DEV))
    r = check_fp8_rows(codes.cpu().numpy(), scale.cpu().numpy(), xb, what="dsa_fp8_quantize")
    assert r["code_exceptions"] <= 1e-3 * r["codes"]


def test_fp8_indexer_scores_and_topk():
    lay = synth.make_layout([1500, 2300], [1, 1])
    host = synth.host_layers(lay, "F", 16, ints=False, seed=13)[0]
    qc, qs = oracle.fp8_quantize_rows(host["q_idx"].reshape(-1, 128))
    kc, ks = oracle.fp8_quantize_rows(host["k_idx"])
    qc = qc.reshape(lay.num_q, 32, 128)
    qs = qs.reshape(lay.num_q, 32)
    batch = make_batch(dsa, lay, DEV)
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    sc = dsa.dsa_indexer_scores(T(qc), T(host["w"]), T(kc), batch, q_scale=T(qs), k_scale=T(ks))
    rows = np.arange(lay.num_q, dtype=np.int32)
    pos, key0 = rows_meta(lay, rows)
    ref = oracle.indexer_scores(qc, host["w"], kc, rows, pos, key0, lay.max_len, dtype=1,
                                q_scale=qs, k_scale=ks)
    got = sc.cpu().numpy()
    fin = np.isfinite(ref)
    assert np.array_equal(fin, np.isfinite(got))
    assert np.abs(got[fin] - ref[fin]).max() <= 1e-5 * np.abs(ref[fin]).max()
    idx = dsa.dsa_topk(sc, batch, 512).cpu().numpy()
    assert_topk_within_band(idx, ref, pos + 1, 512, what="fp8")


def test_bounded_wait_reports_timeout_and_context_survives():
    ws = dsa.workspace(256, DEV)
    dsa.set_wait_timeout_ns(1_000_000)  # 1 ms
    try:
        dsa.dsa_selftest_wait_timeout(ws)
        with pytest.raises(dsa.DsaError) as e:
            dsa.status_fetch(ws)
        assert e.value.status == dsa.DSA_ERR_TIMEOUT
    finally:
        dsa.set_wait_timeout_ns(2_000_000_000)
    # the context is still usable
    test_indexer_scores_bit_exact_on_integers("decode5")


def test_host_argument_errors():
    lay = synth.make_layout([300], [3])
    batch = make_batch(dsa, lay, DEV)
    z = torch.zeros((lay.num_q, 32, 128), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(dsa.DsaError) as e:
        dsa.dsa_topk(torch.zeros((3, lay.max_len), device=DEV), batch, 5000)
    assert e.value.status == dsa.DSA_ERR_UNSUPPORTED
    ql = torch.zeros((3, 32, 512), dtype=torch.bfloat16, device=DEV)
    qr = torch.zeros((3, 32, 64), dtype=torch.bfloat16, device=DEV)
    kv = torch.zeros((300, 576), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(dsa.DsaError) as e:
        dsa.dsa_sparse_mla_attn(ql, qr, kv, torch.zeros((3, 64), dtype=torch.int32, device=DEV),
                                batch, scale=1 / 16)
    assert e.value.status == dsa.DSA_ERR_UNSUPPORTED
    # paged layout: blocks must be a power of two >= 128 and the table must cover max_len
    for table, rows in (([[0, 1, 2]], 384), ([[0]], 128), ([[0, 1, 2]], 64)):
        bad = dsa.Batch(lay.q_start, lay.q_pos, None, lay.max_len, device=DEV,
                        block_table=np.asarray(table, np.int32), block_rows=rows)
        with pytest.raises(dsa.DsaError) as e:
            dsa.dsa_indexer_scores(z, torch.zeros((3, 32), device=DEV),
                                   torch.zeros((300, 128), dtype=torch.bfloat16, device=DEV), bad)
        assert e.value.status == dsa.DSA_ERR_INVALID_ARG
    del z
