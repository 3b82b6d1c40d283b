"""Shared helpers of the GPU parity tests: device copies of the seeded
inputs, host copies of device tensors, and the tolerance checks."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth


def bf16_dev(a, dev):
    """bf16 bit patterns (numpy uint16) -> device torch.bfloat16."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)


def bits(t):
    """device/host torch.bfloat16 -> numpy uint16 bit patterns."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def device_layers(host_layers, dev):
    out = []
    for L in host_layers:
        d = {k: bf16_dev(L[k], dev) for k in ("q_lat", "q_rope", "kv")}
        if "q_idx" in L:
            d.update(q_idx=bf16_dev(L["q_idx"], dev), k_idx=bf16_dev(L["k_idx"], dev),
                     w=torch.from_numpy(np.ascontiguousarray(L["w"])).to(dev))
        out.append(d)
    return out


def make_batch(dsa, lay, dev):
    return dsa.Batch(lay.q_start, lay.q_pos, lay.seq_row0, lay.max_len, device=dev)


def assert_close(got, ref, rel, what=""):
    """max |got - ref| <= rel * max |ref| (the bound used for attention outputs)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    scale = np.abs(ref).max()
    err = np.abs(got - ref).max() if ref.size else 0.0
    assert err <= rel * scale + 1e-30, f"{what}: max err {err:.3e} > {rel} * {scale:.3e}"
    return err / max(scale, 1e-30)


def assert_topk_within_band(got_idx, scores, lens, K, rel=1e-3, what=""):
    """Top-K parity on real-valued scores: the GPU set may differ from the
    exact set only at positions whose exact score lies within rel * |I_K| of
    the K-th largest exact score I_K (the tie band).  scores are the
    oracle's fp64 scores of the same rows."""
    got_idx = np.asarray(got_idx)
    for i in range(got_idx.shape[0]):
        n = int(lens[i])
        g = got_idx[i]
        take = min(n, K)
        assert (g[:take] >= 0).all() and (g[take:] == -1).all(), f"{what} row {i}: padding"
        sel = g[:take]
        assert len(np.unique(sel)) == take and (sel < n).all(), f"{what} row {i}: not a set"
        if n <= K:
            assert np.array_equal(np.sort(sel), np.arange(n)), f"{what} row {i}"
            continue
        row = scores[i, :n]
        kth = np.sort(row)[::-1][K - 1]
        band = rel * abs(kth)
        exact = np.zeros(n, bool)
        exact[oracle.topk(row[None], [n], K)[0]] = True
        mine = np.zeros(n, bool)
        mine[sel] = True
        diff = np.nonzero(exact != mine)[0]
        bad = diff[np.abs(row[diff] - kth) > band]
        assert bad.size == 0, (f"{what} row {i}: {bad.size} positions differ outside the band "
                               f"(e.g. s={bad[:5]}, scores {row[bad[:5]]}, kth {kth})")


def oracle_attention_gathered(q_lat, q_rope, kv, rows, base_rows, idx, scale, kv_bf16=None):
    """Oracle sparse MLA for query rows `rows` of device tensors q_lat, q_rope
    over their index rows idx [n, K] (positions, -1 padded), reading only the
    cache rows they select: base_rows[i] + idx[i, j] of the device cache kv,
    gathered on the device into a compact host copy [n * K, 576].  FP8 KV
    rows (uint8 [rows, 656]) are checked against the oracle's quantisation of
    the same rows of kv_bf16 and read through the oracle's dequantisation.
    Returns (out [n, H, 512], lse [n, H]) in fp64."""
    idx = np.asarray(idx)
    n, K = idx.shape
    dev = kv.device
    rt = torch.as_tensor(np.asarray(rows, np.int64), device=dev)
    cache_rows = np.asarray(base_rows, np.int64)[:, None] + np.maximum(idx, 0)
    cr = torch.as_tensor(cache_rows.reshape(-1), device=dev)
    if kv.dtype == torch.uint8:
        codes = kv.index_select(0, cr).cpu().numpy()
        assert np.array_equal(codes, oracle.kv_fp8_quantize(bits(kv_bf16.index_select(0, cr))))
        kvh = oracle.kv_fp8_dequantize(codes)
    else:
        kvh = bits(kv.index_select(0, cr))
    local = np.where(idx >= 0, np.arange(K)[None, :], -1).astype(np.int32)
    return oracle.sparse_mla(bits(q_lat.index_select(0, rt)), bits(q_rope.index_select(0, rt)), kvh,
                             np.arange(n, dtype=np.int32), np.arange(n, dtype=np.int64) * K, local,
                             scale)
