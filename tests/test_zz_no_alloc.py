"""The allocation-free F-layer entry point (dsa_indexer_topk_noalloc).

Callers that cannot allocate device memory (a host framework that owns all of
it, or a serving loop that must not call cudaMalloc/cudaFree because those
can synchronise the device) use this entry point instead of
dsa_indexer_scores + dsa_topk with a workspace.  Here it is called through
the C ABI twice in a row and each result is compared with the workspace
entry points on the same inputs (index sets identical), and with the oracle:
bit for bit on integer-valued inputs, within the tie band on Gaussian and
FP8 inputs.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import synth  # noqa: E402
from gpu_helpers import assert_topk_within_band, device_layers, make_batch  # noqa: E402

dsa = pytest.importorskip("dsa_indexer_indexshare_gb300")
DEV = torch.device("cuda:0")
CASES = [([300, 9000, 20000, 4097, 129], [1, 1, 1, 1, 1]),   # decode-like rows
         ([2500, 700], [40, 700])]                           # prefill-like rows


def _noalloc(L, batch, k, idx, status, dt=None, k_rows=None):
    fn = dsa.lib.dsa_indexer_topk_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
                                           ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.c_void_p]
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
    stream = ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    return fn(p(L["q_idx"]), p(L.get("q_scale")), p(L["w"]), p(L["k_idx"]), p(L.get("k_scale")),
              L["k_idx"].shape[0] if k_rows is None else k_rows,
              dsa.DSA_BF16 if dt is None else dt, batch.c, k, p(idx), p(status), stream)


def _oracle_scores(lay, host, fp8=False):
    rows = np.arange(lay.num_q, dtype=np.int32)
    pos, key0 = oracle.row_metadata(lay.q_start, lay.q_pos, lay.seq_row0, rows)
    return oracle.indexer_scores(host["q_idx"], host["w"], host["k_idx"], rows, pos, key0,
                                 lay.max_len, dtype=1 if fp8 else 0, q_scale=host.get("q_scale"),
                                 k_scale=host.get("k_scale")), pos + 1


@pytest.mark.parametrize("ints", [True, False])
def test_noalloc_matches_workspace_entry_points_and_oracle_twice(ints):
    K = 512
    for call, (lens, qc) in enumerate(CASES):
        lay = synth.make_layout(lens, qc)
        host = synth.host_layers(lay, "F", 16, ints=ints, seed=21 + call)[0]
        L = device_layers([host], DEV)[0]
        batch = make_batch(dsa, lay, DEV)
        ref = dsa.dsa_topk(dsa.dsa_indexer_scores(L["q_idx"], L["w"], L["k_idx"], batch), batch, K)
        idx = torch.full((lay.num_q, K), -7, dtype=torch.int32, device=DEV)
        status = torch.full((1,), 99, dtype=torch.int32, device=DEV)
        assert _noalloc(L, batch, K, idx, status) == dsa.DSA_OK
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(idx, ref)
        sc, lens_q = _oracle_scores(lay, host)
        if ints:  # fp32 scores are exact: the index sets are the oracle's, bit for bit
            assert np.array_equal(idx.cpu().numpy(), oracle.topk(sc, lens_q, K))
        else:
            assert_topk_within_band(idx.cpu().numpy(), sc, lens_q, K, what="noalloc")


def test_noalloc_fp8_indexer_twice():
    K = 256
    for call, (lens, qc) in enumerate(CASES):
        lay = synth.make_layout(lens, qc)
        host = synth.host_layers(lay, "F", 16, ints=False, seed=31 + call)[0]
        L = device_layers([host], DEV)[0]
        qc8, qs = dsa.dsa_fp8_quantize(L["q_idx"])
        kc8, ks = dsa.dsa_fp8_quantize(L["k_idx"])
        L8 = {"q_idx": qc8, "q_scale": qs, "w": L["w"], "k_idx": kc8, "k_scale": ks}
        batch = make_batch(dsa, lay, DEV)
        ref = dsa.dsa_topk(dsa.dsa_indexer_scores(qc8, L["w"], kc8, batch, q_scale=qs, k_scale=ks),
                           batch, K)
        idx = torch.full((lay.num_q, K), -7, dtype=torch.int32, device=DEV)
        status = torch.full((1,), 99, dtype=torch.int32, device=DEV)
        assert _noalloc(L8, batch, K, idx, status, dt=dsa.DSA_FP8_E4M3) == dsa.DSA_OK
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(idx, ref)
        # the oracle on the same codes and scales
        h8 = {"q_idx": qc8.cpu().numpy(), "q_scale": qs.cpu().numpy(), "w": host["w"],
              "k_idx": kc8.cpu().numpy(), "k_scale": ks.cpu().numpy()}
        sc, lens_q = _oracle_scores(lay, h8, fp8=True)
        assert_topk_within_band(idx.cpu().numpy(), sc, lens_q, K, what="noalloc fp8")


def test_noalloc_rejects_what_the_workspace_entry_points_reject():
    lay = synth.make_layout([1 << 20] * 17, [1] * 17)   # 17 rows x 1M scores > 48 MiB
    batch = dsa.Batch(lay.q_start, lay.q_pos, lay.seq_row0, lay.max_len, device=DEV)
    L = {"q_idx": torch.zeros((17, 32, 128), dtype=torch.bfloat16, device=DEV),
         "w": torch.zeros((17, 32), device=DEV),
         "k_idx": torch.zeros((1024, 128), dtype=torch.bfloat16, device=DEV)}
    idx = torch.zeros((17, 64), dtype=torch.int32, device=DEV)
    assert _noalloc(L, batch, 64, idx, None) == dsa.DSA_ERR_WORKSPACE
    assert b"exceeds the fixed" in dsa.lib.dsa_last_error_string()
    small = make_batch(dsa, synth.make_layout([300], [1]), DEV)
    # the same codes as dsa_indexer_scores / dsa_topk for the same mistakes
    assert _noalloc(L, small, 64, idx, None, k_rows=1 << 31) == dsa.DSA_ERR_UNSUPPORTED
    assert _noalloc(L, small, 5000, idx, None) == dsa.DSA_ERR_UNSUPPORTED
    assert _noalloc(L, small, 64, idx, None, dt=dsa.DSA_FP8_E4M3) == dsa.DSA_ERR_INVALID_ARG
    assert b"q_scale" in dsa.lib.dsa_last_error_string()
