"""The allocation-free F-layer entry point (dsa_indexer_topk_noalloc).

Callers that cannot allocate device memory (a host framework that owns all of
it, or a serving loop that must not call cudaMalloc/cudaFree because those
can synchronise the device) use this entry point instead of
dsa_indexer_scores + dsa_topk with a workspace.  Here it is called through
the C ABI twice in a row and each result is compared with the workspace
entry points on the same inputs: index sets must be identical, the same bar
as the other top-K tests.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import synth  # noqa: E402
from gpu_helpers import device_layers, make_batch  # noqa: E402

dsa = pytest.importorskip("dsa_indexer_indexshare_gb300")
DEV = torch.device("cuda:0")


def _noalloc(lib, L, batch, k, idx, status):
    fn = lib.dsa_indexer_topk_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
                                           ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.c_void_p]
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
    stream = ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    return fn(p(L["q_idx"]), None, p(L["w"]), p(L["k_idx"]), None, L["k_idx"].shape[0],
              dsa.DSA_BF16, batch.c, k, p(idx), p(status), stream)


@pytest.mark.parametrize("ints", [True, False])
def test_noalloc_matches_workspace_entry_points_twice(ints):
    cases = [([300, 9000, 20000, 4097, 129], [1, 1, 1, 1, 1]),   # decode-like rows
             ([2500, 700], [40, 700])]                           # prefill-like rows
    for call, (lens, qc) in enumerate(cases):
        lay = synth.make_layout(lens, qc)
        host = synth.host_layers(lay, "F", 16, ints=ints, seed=21 + call)[0]
        L = device_layers([host], DEV)[0]
        batch = make_batch(dsa, lay, DEV)
        K = 512
        ref = dsa.dsa_topk(dsa.dsa_indexer_scores(L["q_idx"], L["w"], L["k_idx"], batch), batch, K)
        idx = torch.full((lay.num_q, K), -7, dtype=torch.int32, device=DEV)
        status = torch.full((1,), 99, dtype=torch.int32, device=DEV)
        assert _noalloc(dsa.lib, L, batch, K, idx, status) == dsa.DSA_OK
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(idx, ref)


def test_noalloc_rejects_batches_beyond_the_fixed_array():
    lay = synth.make_layout([1 << 20] * 17, [1] * 17)   # 17 rows x 1M scores > 48 MiB
    batch = dsa.Batch(lay.q_start, lay.q_pos, lay.seq_row0, lay.max_len, device=DEV)
    L = {"q_idx": torch.zeros((17, 32, 128), dtype=torch.bfloat16, device=DEV),
         "w": torch.zeros((17, 32), device=DEV),
         "k_idx": torch.zeros((1024, 128), dtype=torch.bfloat16, device=DEV)}
    idx = torch.zeros((17, 64), dtype=torch.int32, device=DEV)
    assert _noalloc(dsa.lib, L, batch, 64, idx, None) == dsa.DSA_ERR_WORKSPACE
