"""CPU oracle for the DSA layer group with IndexShare (test infrastructure).

Only the tests, the smoke check and the benchmark's CPU-baseline leg use
this package; the product library never imports it.  It wraps the plain C
restatement in ``oracle.c`` (fp64 arithmetic on the exact input values) with
numpy marshalling, plus the group loop of the method:

* an F layer computes indexer scores and keeps the top-K positions, writing
  them into the group's index buffer;
* every layer (F or S) runs sparse MLA over that buffer with its own cache
  ("GLM-5.2 架构深度拆解" CH 2.2 and 2.4; "GLM-5 -> 5.1 -> 5.2" section 10).

Functions whose results are pinned by tests against values fixed by the
pages or by mathematics are listed in ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

P_U8 = ctypes.POINTER(ctypes.c_uint8)


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, OpenMP, no FP contraction)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            L.oracle_e4m3_decode.restype = dbl
            L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.oracle_e4m3_encode.restype = ctypes.c_uint8
            L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            L.oracle_e4m3_encode_f64.restype = ctypes.c_uint8
            L.oracle_e4m3_encode_f64.argtypes = [dbl]
            L.oracle_e4m3_encode_array.argtypes = [vp, i64, vp]
            L.oracle_e4m3_decode_array.argtypes = [vp, i64, vp]
            L.oracle_fp8_block_scale.restype = ctypes.c_float
            L.oracle_fp8_block_scale.argtypes = [dbl]
            L.oracle_hadamard128_f64.argtypes = [vp, vp]
            L.oracle_fp8_rotate_rows.argtypes = [vp, i64, vp]
            L.oracle_fp8_quantize_rows.argtypes = [vp, i64, vp, vp]
            L.oracle_f64_to_bf16.argtypes = [ctypes.c_double]
            L.oracle_f64_to_bf16.restype = ctypes.c_uint16
            L.oracle_rope_bf16.argtypes = [vp, vp, i64, ctypes.c_int, ctypes.c_int, vp, vp]
            L.oracle_kv_fp8_quantize.argtypes = [vp, i64, vp]
            L.oracle_kv_fp8_dequantize.argtypes = [vp, i64, vp]
            L.oracle_indexer_scores.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp,
                                                vp, vp, vp, vp, vp, vp, ctypes.c_int, i64, vp]
            L.oracle_topk.argtypes = [vp, i64, vp, ctypes.c_int, ctypes.c_int, vp]
            L.oracle_sparse_mla.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, vp,
                                            vp, vp, ctypes.c_int, vp, ctypes.c_int, dbl, vp, vp]
            L.oracle_dense_mla.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, vp,
                                           vp, vp, vp, ctypes.c_int, dbl, vp, vp]
            L.oracle_num_threads.restype = ctypes.c_int
            _lib = L
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(lib().oracle_num_threads())


# ---------------------------------------------------------------- FP8 / Hadamard
def e4m3_decode(codes) -> np.ndarray:
    """E4M3 codes -> their exact values (fp64; NaN for 0x7F / 0xFF)."""
    c, pc = _c(codes, np.uint8)
    out = np.empty(c.shape, np.float64)
    lib().oracle_e4m3_decode_array(pc, c.size, out.ctypes.data_as(ctypes.c_void_p))
    return out


def e4m3_encode(x) -> np.ndarray:
    """Values -> the nearest E4M3 codes (ties to even, saturating at +-448).
    fp32 inputs are taken as fp32 values; anything else as fp64 values."""
    x = np.asarray(x)
    if x.dtype != np.float32:
        x = x.astype(np.float64)
    v, pv = _c(x.astype(np.float64), np.float64)   # fp32 -> fp64 is exact
    out = np.empty(v.shape, np.uint8)
    lib().oracle_e4m3_encode_array(pv, v.size, out.ctypes.data_as(ctypes.c_void_p))
    return out


def fp8_block_scale(amax: float) -> np.float32:
    """amax / 448 as the nearest fp32 (1 for amax == 0): a block's FP8 scale."""
    return np.float32(lib().oracle_fp8_block_scale(float(amax)))


def hadamard128_f64(v) -> np.ndarray:
    v, pv = _c(v, np.float64)
    assert v.shape == (128,)
    out = np.empty(128, np.float64)
    lib().oracle_hadamard128_f64(pv, out.ctypes.data_as(ctypes.c_void_p))
    return out


def fp8_rotate_rows(x_bf16_bits) -> np.ndarray:
    """H_128 x / sqrt(128) (fp64) of rows of 128 bf16 values: [rows, 128]."""
    x, px = _c(x_bf16_bits, np.uint16)
    rows = x.size // 128
    y = np.empty((rows, 128), np.float64)
    lib().oracle_fp8_rotate_rows(px, rows, y.ctypes.data_as(ctypes.c_void_p))
    return y


def fp8_quantize_rows(x_bf16_bits):
    """Hadamard-rotate and FP8-quantise rows of 128 bf16 values, from the
    definition (fp64 rotation, fp32 scale nearest to amax/448, nearest E4M3).
    Returns (codes uint8 [rows,128], scale float32 [rows])."""
    x, px = _c(x_bf16_bits, np.uint16)
    rows = x.size // 128
    q = np.empty((rows, 128), np.uint8)
    s = np.empty(rows, np.float32)
    lib().oracle_fp8_quantize_rows(px, rows, q.ctypes.data_as(ctypes.c_void_p),
                                   s.ctypes.data_as(ctypes.c_void_p))
    return q, s


def f64_to_bf16(x: float) -> int:
    """One fp64 value rounded to a bf16 bit pattern (nearest, ties to even)."""
    return int(lib().oracle_f64_to_bf16(float(x)))


def rope_inv_freq(theta: float, rope_dims: int = 64) -> np.ndarray:
    """theta^(-2i/rope_dims), i < rope_dims/2: the rotary frequencies of a
    base theta (8e6 for GLM-5.2, "GLM-5.2 架构深度拆解" CH 1.1)."""
    return np.power(float(theta), -2.0 * np.arange(rope_dims // 2) / rope_dims)


def rope_bf16(x_bf16_bits, pos, inv_freq, rope_dims: int = 64):
    """Interleaved RoPE of the first rope_dims entries of each row of x (bf16
    bits, [n, dim]) at positions pos [n], fp64, rounded once to bf16."""
    x, px = _c(np.asarray(x_bf16_bits).reshape(len(pos), -1), np.uint16)
    n, dim = x.shape
    p, pp = _c(pos, np.int32)
    f, pf = _c(inv_freq, np.float64)
    assert f.size >= rope_dims // 2
    out = np.empty_like(x)
    lib().oracle_rope_bf16(px, pp, n, dim, rope_dims, pf, out.ctypes.data_as(ctypes.c_void_p))
    return out


def indexer_append(x_bf16_bits, pos, inv_freq, fp8: bool):
    """What the cache append writes for indexer vectors (rows of 128): RoPE
    (rounded to bf16), then for FP8 the Hadamard + E4M3 quantiser.  Returns
    bf16 bits, or (codes, scales)."""
    r = rope_bf16(x_bf16_bits, pos, inv_freq, 64)
    return fp8_quantize_rows(r) if fp8 else r


def kv_fp8_quantize(kv_bf16_bits):
    """bf16 KV rows [rows, 576] -> FP8 KV rows uint8 [rows, 656]: four groups
    of 128 latent dims as E4M3 codes, four fp32 scales, the bf16 RoPE key."""
    x, px = _c(np.asarray(kv_bf16_bits).reshape(-1, 576), np.uint16)
    rows = x.shape[0]
    out = np.empty((rows, 656), np.uint8)
    lib().oracle_kv_fp8_quantize(px, rows, out.ctypes.data_as(ctypes.c_void_p))
    return out


def kv_fp8_dequantize(kv_fp8):
    """FP8 KV rows uint8 [rows, 656] -> the bf16 rows [rows, 576] (bits) the
    attention reads: the fp32 product code * scale rounded to bf16, the RoPE
    key as is."""
    x, px = _c(np.asarray(kv_fp8).reshape(-1, 656), np.uint8)
    rows = x.shape[0]
    out = np.empty((rows, 576), np.uint16)
    lib().oracle_kv_fp8_dequantize(px, rows, out.ctypes.data_as(ctypes.c_void_p))
    return out


# ---------------------------------------------------------------- batch helpers
def row_metadata(q_start, q_pos, seq_row0, rows):
    """Per listed query row: its absolute position and the cache row of its
    sequence's position 0."""
    q_start = np.asarray(q_start, np.int64)
    rows = np.asarray(rows, np.int64)
    seq = np.searchsorted(q_start, rows, side="right") - 1
    row_pos = np.asarray(q_pos, np.int64)[rows].astype(np.int32)
    row_key0 = np.asarray(seq_row0, np.int64)[seq]
    return row_pos, row_key0


def paged_row(block_table, block_rows, seq, s):
    """Cache row of position s of sequence seq in a paged cache: the table
    names the block holding positions [j*block_rows, (j+1)*block_rows) of the
    sequence, and the position keeps its offset inside the block
    (PagedAttention over the compressed MLA KV, "GLM-5.2 架构深度拆解" CH 4.4).
    -1 when the table has no block for it (negative id or beyond the table)."""
    bt = np.asarray(block_table)
    j = int(s) // int(block_rows)
    if j >= bt.shape[1] or bt[seq, j] < 0:
        return -1
    return int(bt[seq, j]) * int(block_rows) + int(s) % int(block_rows)


def logical_cache(paged, block_table, block_rows, seq_lens):
    """The contiguous cache a paged one stands for: positions 0..seq_lens[b]-1
    of every sequence b, back to back in sequence order (row seq_row0[b] + s
    with seq_row0 the running sum of seq_lens, the layout the functions
    below take).  Row by row through paged_row."""
    paged = np.asarray(paged)
    out = np.empty((int(np.sum(seq_lens)),) + paged.shape[1:], paged.dtype)
    r = 0
    for b, n in enumerate(seq_lens):
        for s in range(int(n)):
            out[r] = paged[paged_row(block_table, block_rows, b, s)]
            r += 1
    return out


# ---------------------------------------------------------------- hot / cold KV
def hot_state(num_seqs, hot_slots, max_len):
    """An empty hot buffer: slot_pos [S, hot] (position held, -1 empty),
    slot_stamp [S, hot] (last step that used the slot, -1 never) and
    pos_slot [S, max_len] (slot holding each position, -1 none)."""
    return {"slot_pos": np.full((num_seqs, hot_slots), -1, np.int32),
            "slot_stamp": np.full((num_seqs, hot_slots), -1, np.int32),
            "pos_slot": np.full((num_seqs, max_len), -1, np.int32)}


def hot_plan(idx, q_start, q_pos, state, step, hot_slots):
    """One step of the HiSparse-style hot buffer ("GLM-5.2 / 总览" glossary
    entry HiSparse: a GPU "hot" KV of 6144 slots, the full KV in CPU pinned
    memory, rows swapped in on demand after the DSA top-K).

    Per sequence b, over the valid entries e = idx[t, k] (0 <= e <= q_pos[t])
    of its queries, taken query by query and slot by slot:
      1. a resident position (pos_slot[e] >= 0) is a hit: its slot's stamp
         becomes `step`;
      2. the other positions are misses, kept in order of first appearance;
      3. the m misses need m slots: among the slots whose stamp is below
         `step` (not used at this step), the m least recently used ones
         (smallest stamp, then lowest slot index); more misses than such
         slots is an overflow: the sequence changes no slot and all its rows
         are -1;
      4. the chosen slots, taken in increasing slot index, receive the misses
         in order: the slot's old position (if any) leaves, the miss enters,
         the stamp becomes `step`; (position, slot) goes on the fetch list;
      5. rows[t, k] = b * hot_slots + pos_slot[e] (-1 for -1 padding and for
         invalid entries).
    `step` must exceed every step used before with this state.  Returns
    (new state, rows [Nq, K] int32, fetch list per sequence, set of errors
    among {"index", "overflow"})."""
    st = {key: np.array(v, copy=True) for key, v in state.items()}
    idx = np.asarray(idx)
    q_start = np.asarray(q_start)
    q_pos = np.asarray(q_pos)
    nq, K = idx.shape
    max_len = st["pos_slot"].shape[1]
    rows = np.full((nq, K), -1, np.int32)
    fetch, errors = [], set()
    for b in range(len(q_start) - 1):
        sp, ss, ps = st["slot_pos"][b], st["slot_stamp"][b], st["pos_slot"][b]
        entries = []
        for t in range(int(q_start[b]), int(q_start[b + 1])):
            for k in range(K):
                e = int(idx[t, k])
                if e == -1:
                    continue
                if e < 0 or e > int(q_pos[t]) or e >= max_len:
                    errors.add("index")
                    continue
                entries.append((t, k, e))
        misses, seen = [], set()
        for _, _, e in entries:
            if ps[e] >= 0:
                ss[ps[e]] = step
            elif e not in seen:
                seen.add(e)
                misses.append(e)
        free = [s for s in range(hot_slots) if ss[s] < step]
        if len(misses) > len(free):
            errors.add("overflow")
            fetch.append([])
            continue
        lru = sorted(free, key=lambda s: (int(ss[s]), s))[:len(misses)]
        moves = []
        for e, s in zip(misses, sorted(lru)):
            if sp[s] >= 0:
                ps[sp[s]] = -1
            ps[e], sp[s], ss[s] = s, e, step
            moves.append((e, s))
        fetch.append(moves)
        for t, k, e in entries:
            rows[t, k] = b * hot_slots + ps[e]
    return st, rows, fetch, errors


def hot_fetch(fetch, cold_kv, cold_row, hot_kv, hot_slots):
    """Swap-in: for every (position e, slot s) of sequence b's fetch list,
    hot_kv[b * hot_slots + s] = cold_kv[cold_row(b, e)] (in place)."""
    for b, moves in enumerate(fetch):
        for e, s in moves:
            hot_kv[b * hot_slots + s] = cold_kv[cold_row(b, e)]
    return hot_kv


# ---------------------------------------------------------------- the method
def indexer_scores(q_idx, w, k_idx, rows, row_pos, row_key0, max_len, *, dtype=0,
                   q_scale=None, k_scale=None, Hi=None, Di=None):
    """Scores [len(rows), max_len] in fp64; -inf beyond each row's position.
    dtype 0: q_idx/k_idx are bf16 bit patterns (uint16); dtype 1: E4M3 codes
    (uint8) with q_scale [num_q, Hi] and k_scale [rows] (float32)."""
    q_idx = np.asarray(q_idx)
    Hi = q_idx.shape[-2] if Hi is None else Hi
    Di = q_idx.shape[-1] if Di is None else Di
    et = np.uint16 if dtype == 0 else np.uint8
    q_idx, pq = _c(q_idx, et)
    k_idx, pk = _c(k_idx, et)
    w, pw = _c(w, np.float32)
    qs, pqs = _c(q_scale if q_scale is not None else np.zeros(1), np.float32)
    ks, pks = _c(k_scale if k_scale is not None else np.zeros(1), np.float32)
    rows, pr = _c(rows, np.int32)
    row_pos, pp = _c(row_pos, np.int32)
    row_key0, p0 = _c(row_key0, np.int64)
    out = np.empty((rows.size, int(max_len)), np.float64)
    lib().oracle_indexer_scores(Hi, Di, dtype, pq, pqs, pw, pk, pks, pr, pp, p0, rows.size,
                                int(max_len), out.ctypes.data_as(ctypes.c_void_p))
    return out


def topk(scores, lens, K):
    """Top-K positions per row (ties: lower position), ascending, -1 padded."""
    scores, ps = _c(scores, np.float64)
    lens, pl = _c(lens, np.int32)
    n = lens.size
    out = np.empty((n, K), np.int32)
    lib().oracle_topk(ps, scores.shape[-1], pl, n, K, out.ctypes.data_as(ctypes.c_void_p))
    return out


def sparse_mla(q_lat, q_rope, kv, rows, row_key0, idx, scale):
    """Sparse MLA for the listed rows: (out [n,H,Dl] fp64, lse [n,H] fp64)."""
    q_lat = np.asarray(q_lat)
    H, Dl = q_lat.shape[-2], q_lat.shape[-1]
    Dr = np.asarray(q_rope).shape[-1]
    q_lat, pql = _c(q_lat, np.uint16)
    q_rope, pqr = _c(q_rope, np.uint16)
    kv, pkv = _c(kv, np.uint16)
    rows, pr = _c(rows, np.int32)
    row_key0, p0 = _c(row_key0, np.int64)
    idx, pi = _c(idx, np.int32)
    n, K = idx.shape
    out = np.empty((n, H, Dl), np.float64)
    lse = np.empty((n, H), np.float64)
    lib().oracle_sparse_mla(H, Dl, Dr, pql, pqr, pkv, pr, p0, n, pi, K, float(scale),
                            out.ctypes.data_as(ctypes.c_void_p), lse.ctypes.data_as(ctypes.c_void_p))
    return out, lse


def dense_mla(q_lat, q_rope, kv, rows, row_pos, row_key0, scale):
    q_lat = np.asarray(q_lat)
    H, Dl = q_lat.shape[-2], q_lat.shape[-1]
    Dr = np.asarray(q_rope).shape[-1]
    q_lat, pql = _c(q_lat, np.uint16)
    q_rope, pqr = _c(q_rope, np.uint16)
    kv, pkv = _c(kv, np.uint16)
    rows, pr = _c(rows, np.int32)
    row_pos, pp = _c(row_pos, np.int32)
    row_key0, p0 = _c(row_key0, np.int64)
    n = rows.size
    out = np.empty((n, H, Dl), np.float64)
    lse = np.empty((n, H), np.float64)
    lib().oracle_dense_mla(H, Dl, Dr, pql, pqr, pkv, pr, pp, p0, n, float(scale),
                           out.ctypes.data_as(ctypes.c_void_p), lse.ctypes.data_as(ctypes.c_void_p))
    return out, lse


def parse_layer_types(layer_types: str):
    """'F' = full layer (runs the indexer), 'S' = shared layer (reuses the
    nearest preceding F layer's indices).  The first layer must be F."""
    if not layer_types or any(c not in "FS" for c in layer_types) or layer_types[0] != "F":
        raise ValueError(f"bad layer_types {layer_types!r}")
    return [c == "F" for c in layer_types]


def group_forward(layer_types, layers, rows, row_pos, row_key0, max_len, K, scale, *,
                  idx_dtype=0, keep_scores=False):
    """One layer group for the listed query rows.

    layers[l] is a dict with q_lat, q_rope, kv and, on F layers, q_idx, w,
    k_idx (plus q_scale, k_scale for the FP8 indexer).  Returns a dict with
    per-layer outputs, lse, the index buffer each layer used, and the scores
    of each F layer when keep_scores is set."""
    full = parse_layer_types(layer_types)
    lens = np.minimum(np.asarray(row_pos, np.int64) + 1, int(max_len)).astype(np.int32)
    res = {"out": [], "lse": [], "idx": [], "scores": [], "kth": []}
    idx = None
    for l, is_full in enumerate(full):
        L = layers[l]
        if is_full:
            sc = indexer_scores(L["q_idx"], L["w"], L["k_idx"], rows, row_pos, row_key0, max_len,
                                dtype=idx_dtype, q_scale=L.get("q_scale"), k_scale=L.get("k_scale"))
            idx = topk(sc, lens, K)
            if keep_scores:
                res["scores"].append(sc)
        o, s = sparse_mla(L["q_lat"], L["q_rope"], L["kv"], rows, row_key0, idx, scale)
        res["out"].append(o)
        res["lse"].append(s)
        res["idx"].append(idx)
    return res
