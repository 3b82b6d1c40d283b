"""Python binding of libdsa, the GB300 DSA attention layer group with IndexShare.

Argument marshalling only: every function here forwards to the C entry point of
the same name in ``include/dsa.h`` and every step of the computation runs in
the library's CUDA kernels.  PyTorch provides device memory and the stream.
There is no fallback: importing this package fails if ``libdsa.so`` has not
been built, and a call fails if its kernel cannot run.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_float, c_int, c_int32, c_int64, c_size_t, c_uint64, c_void_p

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsa.so")

DSA_OK, DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED, DSA_ERR_WORKSPACE = 0, 1, 2, 3
DSA_ERR_CUDA, DSA_ERR_TIMEOUT, DSA_ERR_DEVICE_INDEX, DSA_ERR_HOT_OVERFLOW = 4, 5, 6, 7
DSA_BF16, DSA_FP8_E4M3 = 0, 1
INDEX_HEADS, INDEX_DIM, LATENT, ROPE, KV_ROW, KV_ROW_FP8 = 32, 128, 512, 64, 576, 656
STATUS_BYTES = 256
LAUNCH_KINDS = ("indexer", "topk", "sparse_mla", "combine", "fp8_quantize", "append", "hot_plan",
                "hot_fetch", "other")
HOT_MAX_SLOTS = 16384

STATUS_NAMES = {0: "DSA_OK", 1: "DSA_ERR_INVALID_ARG", 2: "DSA_ERR_UNSUPPORTED",
                3: "DSA_ERR_WORKSPACE", 4: "DSA_ERR_CUDA", 5: "DSA_ERR_TIMEOUT",
                6: "DSA_ERR_DEVICE_INDEX", 7: "DSA_ERR_HOT_OVERFLOW"}


class DsaError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} {detail}".strip())


class _Batch(ctypes.Structure):
    _fields_ = [("num_seqs", c_int32), ("num_q", c_int32), ("max_q", c_int32),
                ("max_len", c_int32), ("q_start", c_void_p), ("q_pos", c_void_p),
                ("seq_row0", c_void_p), ("block_table", c_void_p), ("block_rows", c_int32),
                ("blocks_per_seq", c_int32)]


_PP = POINTER(c_void_p)


class _Group(ctypes.Structure):
    _fields_ = [("layer_types", c_char_p), ("heads", c_int32), ("k", c_int32),
                ("scale", c_float), ("idx_dtype", c_int), ("kv_rows", c_int64),
                ("k_rows", c_int64), ("q_lat", _PP), ("q_rope", _PP), ("kv", _PP), ("out", _PP),
                ("lse", _PP), ("q_idx", _PP), ("q_scale", _PP), ("w", _PP), ("k_idx", _PP),
                ("k_scale", _PP), ("kv_dtype", c_int)]


class _Hot(ctypes.Structure):
    _fields_ = [("hot_slots", c_int32), ("max_pos", c_int32), ("slot_pos", c_void_p),
                ("slot_stamp", c_void_p), ("pos_slot", c_void_p), ("fetch_pos", c_void_p),
                ("fetch_slot", c_void_p), ("fetch_count", c_void_p)]


class _HotGroup(ctypes.Structure):
    _fields_ = [("spans", POINTER(_Hot)), ("n_spans", c_int32), ("cold_kv", _PP),
                ("cold_rows", c_int64), ("step", c_int32), ("rows", c_void_p)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it first (python dsa_indexer_indexshare_gb300/_build.py)")
    L = ctypes.CDLL(LIB_PATH)
    B = POINTER(_Batch)
    st = c_int
    sig = {
        "dsa_last_error_string": (c_char_p, []),
        "dsa_status_bytes": (c_size_t, []),
        "dsa_workspace_init": (st, [c_void_p, c_size_t, c_void_p]),
        "dsa_status_fetch": (st, [c_void_p, c_void_p, POINTER(c_int32)]),
        "dsa_launch_counts": (c_int, [POINTER(c_uint64), c_int]),
        "dsa_launch_counts_reset": (None, []),
        "dsa_set_wait_timeout_ns": (None, [c_uint64]),
        "dsa_set_mla_persistent": (None, [c_int]),
        "dsa_profile_enable": (None, [c_int]),
        "dsa_profile_collect": (c_int, [POINTER(ctypes.c_double), POINTER(c_uint64), c_int]),
        "dsa_selftest_wait_timeout": (st, [c_void_p, c_size_t, c_void_p]),
        "dsa_indexer_workspace_size": (c_size_t, [B]),
        "dsa_indexer_scores": (st, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int64,
                                    c_int, B, c_void_p, c_void_p, c_size_t, c_void_p]),
        "dsa_topk_workspace_size": (c_size_t, [B, c_int32]),
        "dsa_topk": (st, [c_void_p, B, c_int32, c_void_p, c_void_p, c_size_t, c_void_p]),
        "dsa_sparse_mla_workspace_size": (c_size_t, [B, c_int32, c_int32]),
        "dsa_sparse_mla_attn": (st, [c_void_p, c_void_p, c_void_p, c_int64, c_void_p, c_int32,
                                     c_int32, c_float, B, c_void_p, c_void_p, c_void_p, c_size_t,
                                     c_void_p]),
        "dsa_group_workspace_size": (c_size_t, [POINTER(_Group), B]),
        "indexshare_group_forward": (st, [POINTER(_Group), B, c_void_p, c_void_p, c_size_t,
                                          c_void_p]),
        "dsa_fp8_quantize": (st, [c_void_p, c_int64, c_void_p, c_void_p, c_void_p]),
        "dsa_kv_fp8_quantize": (st, [c_void_p, c_int64, c_void_p, c_void_p]),
        "dsa_sparse_mla_attn_fp8kv": (st, [c_void_p, c_void_p, c_void_p, c_int64, c_void_p,
                                           c_int32, c_int32, c_float, B, c_void_p, c_void_p,
                                           c_void_p, c_size_t, c_void_p]),
        "dsa_indexer_append_keys": (st, [c_void_p, c_void_p, c_void_p, c_int32, B, c_int,
                                         c_void_p, c_void_p, c_void_p, c_int64, c_void_p,
                                         c_size_t, c_void_p]),
        "dsa_indexer_prepare_queries": (st, [c_void_p, B, c_int, c_void_p, c_void_p, c_void_p,
                                             c_void_p, c_size_t, c_void_p]),
        "dsa_hot_plan": (st, [c_void_p, c_int32, B, POINTER(_Hot), c_int32, c_void_p, c_void_p,
                              c_size_t, c_void_p]),
        "dsa_hot_fetch": (st, [POINTER(_Hot), B, c_int32, _PP, c_int64, _PP, c_int64, c_int,
                               c_void_p, c_size_t, c_void_p]),
        "dsa_hot_touch": (st, [c_int32, _PP, c_int64, c_int64, c_void_p]),
        "dsa_sparse_mla_attn_rows": (st, [c_void_p, c_void_p, c_void_p, c_int64, c_int, c_void_p,
                                          c_int32, c_int32, c_float, B, c_void_p, c_void_p,
                                          c_void_p, c_size_t, c_void_p]),
        "indexshare_group_forward_hot": (st, [POINTER(_Group), B, POINTER(_HotGroup), c_void_p,
                                              c_void_p, c_size_t, c_void_p]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


lib = _load()


# ---------------------------------------------------------------- helpers
def _ptr(t):
    return None if t is None else c_void_p(t.data_ptr())


def _stream(stream, device):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return c_void_p(s.cuda_stream)


def _check(status: int, where: str):
    if status != DSA_OK:
        raise DsaError(status, where, lib.dsa_last_error_string().decode())


def _need(t, name, dtype=None, device=None, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError(f"{name} has dtype {t.dtype}, want {dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, want {device}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, want {tuple(shape)}")
    return t


class Batch:
    """Batch layout (dsa_batch_t): query rows of sequence b are
    [q_start[b], q_start[b+1]); query t sits at position q_pos[t]; position s
    of sequence b is row seq_row0[b] + s of every per-layer cache, or, with a
    block table [num_seqs, blocks_per_seq] (paged caches), row
    block_table[b, s // block_rows] * block_rows + s % block_rows."""

    def __init__(self, q_start, q_pos, seq_row0, max_len: int, device="cuda", *,
                 block_table=None, block_rows: int = 0):
        import numpy as np
        qs = np.asarray(q_start, np.int64)
        self.num_seqs = int(qs.size - 1)
        self.num_q = int(np.asarray(q_pos).size)
        self.max_q = int(np.diff(qs).max(initial=0)) if qs.size > 1 else 0
        self.max_len = int(max_len)
        dev = torch.device(device)
        self.device = dev
        self.q_start = torch.as_tensor(np.asarray(q_start, np.int32), device=dev)
        self.q_pos = torch.as_tensor(np.asarray(q_pos, np.int32), device=dev)
        self.seq_row0 = (torch.as_tensor(np.asarray(seq_row0, np.int64), device=dev)
                         if seq_row0 is not None else None)
        if block_table is not None:
            bt = np.asarray(block_table, np.int32)
            if bt.ndim != 2 or bt.shape[0] != self.num_seqs:
                raise ValueError("block_table must be [num_seqs, blocks_per_seq]")
            self.block_table = torch.as_tensor(np.ascontiguousarray(bt), device=dev)
            self.block_rows, self.blocks_per_seq = int(block_rows), int(bt.shape[1])
        else:
            self.block_table, self.block_rows, self.blocks_per_seq = None, 0, 0
        self._c = _Batch(self.num_seqs, self.num_q, self.max_q, self.max_len,
                         _ptr(self.q_start), _ptr(self.q_pos),
                         _ptr(self.seq_row0) if self.seq_row0 is not None else None,
                         _ptr(self.block_table) if self.block_table is not None else None,
                         self.block_rows, self.blocks_per_seq)

    @property
    def c(self):
        return ctypes.byref(self._c)


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A zeroed device workspace (status block included)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def status_fetch(ws: torch.Tensor, stream=None):
    """Synchronise, read and clear the device status of a workspace; raise on error."""
    bits = c_int32(0)
    s = lib.dsa_status_fetch(_ptr(ws), _stream(stream, ws.device), ctypes.byref(bits))
    _check(s, "device status")
    return bits.value


def launch_counts() -> dict:
    arr = (c_uint64 * len(LAUNCH_KINDS))()
    lib.dsa_launch_counts(arr, len(LAUNCH_KINDS))
    return dict(zip(LAUNCH_KINDS, list(arr)))


def launch_counts_reset():
    lib.dsa_launch_counts_reset()


def dsa_profile_enable(on: bool = True):
    lib.dsa_profile_enable(1 if on else 0)


def dsa_profile_collect() -> dict:
    """{kind: (total_ms, launches)} of the launches recorded since the last collect."""
    n = len(LAUNCH_KINDS)
    ms = (ctypes.c_double * n)()
    cnt = (c_uint64 * n)()
    if lib.dsa_profile_collect(ms, cnt, n) < 0:
        raise DsaError(DSA_ERR_CUDA, "dsa_profile_collect")
    return {k: (ms[i], int(cnt[i])) for i, k in enumerate(LAUNCH_KINDS)}


def set_wait_timeout_ns(ns: int):
    lib.dsa_set_wait_timeout_ns(int(ns))


def set_mla_persistent(on: bool):
    """Sparse attention over many tokens on a persistent grid (default) or one
    CTA per token; both give bit-identical results."""
    lib.dsa_set_mla_persistent(1 if on else 0)


def dsa_selftest_wait_timeout(ws: torch.Tensor, stream=None):
    _check(lib.dsa_selftest_wait_timeout(_ptr(ws), ws.numel(), _stream(stream, ws.device)),
           "dsa_selftest_wait_timeout")


def _idx_dtype(t):
    if t.dtype == torch.bfloat16:
        return DSA_BF16
    if t.dtype in (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8)):
        return DSA_FP8_E4M3
    raise ValueError(f"indexer tensors must be bfloat16 or E4M3 codes, got {t.dtype}")


# ---------------------------------------------------------------- entry points
def dsa_indexer_scores(q_idx, w, k_idx, batch: Batch, scores=None, *, q_scale=None,
                       k_scale=None, ws=None, stream=None):
    """Indexer scores [num_q, max_len] fp32 (-inf beyond each query's position)."""
    dev = batch.device
    dt = _idx_dtype(q_idx)
    _need(q_idx, "q_idx", device=dev, shape=(batch.num_q, INDEX_HEADS, INDEX_DIM))
    _need(w, "w", torch.float32, dev, (batch.num_q, INDEX_HEADS))
    _need(k_idx, "k_idx", q_idx.dtype, dev)
    if k_idx.dim() != 2 or k_idx.shape[1] != INDEX_DIM:
        raise ValueError("k_idx must be [rows, 128]")
    if dt == DSA_FP8_E4M3:
        _need(q_scale, "q_scale", torch.float32, dev, (batch.num_q, INDEX_HEADS))
        _need(k_scale, "k_scale", torch.float32, dev, (k_idx.shape[0],))
    if scores is None:
        scores = torch.empty((batch.num_q, batch.max_len), dtype=torch.float32, device=dev)
    _need(scores, "scores", torch.float32, dev, (batch.num_q, batch.max_len))
    if ws is None:
        ws = workspace(lib.dsa_indexer_workspace_size(batch.c), dev)
    _check(lib.dsa_indexer_scores(_ptr(q_idx), _ptr(q_scale), _ptr(w), _ptr(k_idx), _ptr(k_scale),
                                  k_idx.shape[0], dt, batch.c, _ptr(scores), _ptr(ws), ws.numel(),
                                  _stream(stream, dev)), "dsa_indexer_scores")
    return scores


def dsa_topk(scores, batch: Batch, k: int, idx=None, *, ws=None, stream=None):
    """Top-k positions per query (ascending, ties to the lower position, -1 padded)."""
    dev = batch.device
    _need(scores, "scores", torch.float32, dev, (batch.num_q, batch.max_len))
    if idx is None:
        idx = torch.empty((batch.num_q, k), dtype=torch.int32, device=dev)
    _need(idx, "idx", torch.int32, dev, (batch.num_q, k))
    if ws is None:
        ws = workspace(lib.dsa_topk_workspace_size(batch.c, k), dev)
    _check(lib.dsa_topk(_ptr(scores), batch.c, k, _ptr(idx), _ptr(ws), ws.numel(),
                        _stream(stream, dev)), "dsa_topk")
    return idx


def dsa_sparse_mla_attn(q_lat, q_rope, kv, idx, batch: Batch, *, scale: float, out=None,
                        lse=None, with_lse=True, ws=None, stream=None):
    """Sparse absorbed-MLA attention: (out [num_q, H, 512] bf16, lse [num_q, H] fp32).
    kv: bf16 [rows, 576], or FP8 rows uint8 [rows, 656] (dsa_kv_fp8_quantize)."""
    dev = batch.device
    H = q_lat.shape[1]
    _need(q_lat, "q_lat", torch.bfloat16, dev, (batch.num_q, H, LATENT))
    _need(q_rope, "q_rope", torch.bfloat16, dev, (batch.num_q, H, ROPE))
    _need(kv, "kv", (torch.bfloat16, torch.uint8), dev)
    kv_fp8 = kv.dtype == torch.uint8
    if kv.dim() != 2 or kv.shape[1] != (KV_ROW_FP8 if kv_fp8 else KV_ROW):
        raise ValueError("kv must be bf16 [rows, 576] or uint8 [rows, 656]")
    _need(idx, "idx", torch.int32, dev)
    k = idx.shape[1]
    if out is None:
        out = torch.empty((batch.num_q, H, LATENT), dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, dev, (batch.num_q, H, LATENT))
    if lse is None and with_lse:
        lse = torch.empty((batch.num_q, H), dtype=torch.float32, device=dev)
    if ws is None:
        ws = workspace(lib.dsa_sparse_mla_workspace_size(batch.c, H, k), dev)
    fn = lib.dsa_sparse_mla_attn_fp8kv if kv_fp8 else lib.dsa_sparse_mla_attn
    _check(fn(_ptr(q_lat), _ptr(q_rope), _ptr(kv), kv.shape[0], _ptr(idx), k, H, float(scale),
              batch.c, _ptr(out), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream, dev)),
           "dsa_sparse_mla_attn")
    return out, lse


def dsa_kv_fp8_quantize(kv, out=None, *, stream=None):
    """bf16 KV rows [rows, 576] -> FP8 KV rows uint8 [rows, 656] (four E4M3
    groups of 128 latent dims with fp32 scales, then the bf16 RoPE key)."""
    _need(kv, "kv", torch.bfloat16)
    if kv.dim() != 2 or kv.shape[1] != KV_ROW:
        raise ValueError("kv must be [rows, 576]")
    if out is None:
        out = torch.empty((kv.shape[0], KV_ROW_FP8), dtype=torch.uint8, device=kv.device)
    _need(out, "out", torch.uint8, kv.device, (kv.shape[0], KV_ROW_FP8))
    _check(lib.dsa_kv_fp8_quantize(_ptr(kv), kv.shape[0], _ptr(out), _stream(stream, kv.device)),
           "dsa_kv_fp8_quantize")
    return out


class Group:
    """Host-side description of one layer group (dsa_group_t).  layers[l] is a
    dict of device tensors: q_lat, q_rope, kv, and on F layers q_idx, w, k_idx
    (+ q_scale, k_scale for the FP8 indexer)."""

    def __init__(self, layer_types: str, layers, *, k: int, scale: float, outs=None,
                 with_lse=False):
        self.layer_types = layer_types
        self.layers = layers
        nl = len(layer_types)
        if len(layers) != nl:
            raise ValueError("one layer dict per layer type")
        first = layers[0]
        dev = first["q_lat"].device
        num_q, H = first["q_lat"].shape[0], first["q_lat"].shape[1]
        fl = [l for l, c in enumerate(layer_types) if c == "F"]
        idx_t = layers[fl[0]]["q_idx"] if fl else None
        self.idx_dtype = _idx_dtype(idx_t) if idx_t is not None else DSA_BF16
        for l, L in enumerate(layers):
            _need(L["q_lat"], f"q_lat[{l}]", torch.bfloat16, dev, (num_q, H, LATENT))
            _need(L["q_rope"], f"q_rope[{l}]", torch.bfloat16, dev, (num_q, H, ROPE))
            kv_fp8 = first["kv"].dtype == torch.uint8
            _need(L["kv"], f"kv[{l}]", torch.uint8 if kv_fp8 else torch.bfloat16, dev,
                  (first["kv"].shape[0], KV_ROW_FP8 if kv_fp8 else KV_ROW))
            if layer_types[l] == "F":
                _need(L["q_idx"], f"q_idx[{l}]", idx_t.dtype, dev, (num_q, INDEX_HEADS, INDEX_DIM))
                _need(L["w"], f"w[{l}]", torch.float32, dev, (num_q, INDEX_HEADS))
                _need(L["k_idx"], f"k_idx[{l}]", idx_t.dtype, dev,
                      (layers[fl[0]]["k_idx"].shape[0], INDEX_DIM))
                if self.idx_dtype == DSA_FP8_E4M3:
                    _need(L["q_scale"], f"q_scale[{l}]", torch.float32, dev, (num_q, INDEX_HEADS))
                    _need(L["k_scale"], f"k_scale[{l}]", torch.float32, dev)
        self.outs = outs if outs is not None else [
            torch.empty((num_q, H, LATENT), dtype=torch.bfloat16, device=dev) for _ in range(nl)]
        self.lses = [torch.empty((num_q, H), dtype=torch.float32, device=dev)
                     for _ in range(nl)] if with_lse else None

        def arr(key):
            return (c_void_p * nl)(*[layers[l][key].data_ptr() if layers[l].get(key) is not None
                                     else None for l in range(nl)])

        self._arrays = {k_: arr(k_) for k_ in ("q_lat", "q_rope", "kv", "q_idx", "q_scale", "w",
                                              "k_idx", "k_scale")}
        self._arrays["out"] = (c_void_p * nl)(*[o.data_ptr() for o in self.outs])
        self._arrays["lse"] = ((c_void_p * nl)(*[o.data_ptr() for o in self.lses])
                               if self.lses else None)
        self._types = layer_types.encode()
        kv_rows = first["kv"].shape[0]
        k_rows = layers[fl[0]]["k_idx"].shape[0] if fl else 0
        a = self._arrays
        cast = lambda x: ctypes.cast(x, _PP) if x is not None else None
        self._c = _Group(self._types, H, k, float(scale), self.idx_dtype, kv_rows, k_rows,
                         cast(a["q_lat"]), cast(a["q_rope"]), cast(a["kv"]), cast(a["out"]),
                         cast(a["lse"]), cast(a["q_idx"]), cast(a["q_scale"]), cast(a["w"]),
                         cast(a["k_idx"]), cast(a["k_scale"]),
                         DSA_FP8_E4M3 if first["kv"].dtype == torch.uint8 else DSA_BF16)
        self.k = k
        self.device = dev
        self.num_q = num_q

    @property
    def c(self):
        return ctypes.byref(self._c)

    def workspace_size(self, batch: Batch) -> int:
        return lib.dsa_group_workspace_size(self.c, batch.c)


def indexshare_group_forward(group: Group, batch: Batch, idx_buf=None, *, ws=None, stream=None):
    """Run one layer group; returns (outs, lses, idx_buf).  outs[l] is the
    layer's [num_q, H, 512] bf16 output; idx_buf holds the last F layer's
    indices."""
    dev = batch.device
    if idx_buf is None:
        idx_buf = torch.empty((batch.num_q, group.k), dtype=torch.int32, device=dev)
    _need(idx_buf, "idx_buf", torch.int32, dev, (batch.num_q, group.k))
    if ws is None:
        ws = workspace(group.workspace_size(batch), dev)
    _check(lib.indexshare_group_forward(group.c, batch.c, _ptr(idx_buf), _ptr(ws), ws.numel(),
                                        _stream(stream, dev)), "indexshare_group_forward")
    return group.outs, group.lses, idx_buf


def dsa_fp8_quantize(x, codes=None, scale=None, *, stream=None):
    """Hadamard-rotate and E4M3-quantise rows of 128 bf16 values:
    returns (codes uint8 [..., 128], scale fp32 [rows])."""
    _need(x, "x", torch.bfloat16)
    if x.shape[-1] != 128:
        raise ValueError("last dimension must be 128")
    rows = x.numel() // 128
    if codes is None:
        codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    _need(codes, "codes", torch.uint8, x.device)
    _need(scale, "scale", torch.float32, x.device)
    _check(lib.dsa_fp8_quantize(_ptr(x), rows, _ptr(codes), _ptr(scale), _stream(stream, x.device)),
           "dsa_fp8_quantize")
    return codes, scale


def _freq(inv_freq):
    f = (ctypes.c_double * 32)(*[float(v) for v in list(inv_freq)[:32]])
    if len(list(inv_freq)) < 32:
        raise ValueError("inv_freq needs 32 entries")
    return f


def dsa_indexer_append_keys(k_new, k_seq, k_pos, batch: Batch, k_cache, inv_freq, *,
                            k_scale=None, ws=None, stream=None):
    """RoPE (+ Hadamard + FP8 when k_cache is uint8) of new indexer keys
    k_new bf16 [n, 128], written at the cache rows of (k_seq, k_pos) in the
    batch layout.  inv_freq: 32 rotary frequencies (host sequence)."""
    dev = batch.device
    _need(k_new, "k_new", torch.bfloat16, dev)
    n = k_new.numel() // 128
    _need(k_seq, "k_seq", torch.int32, dev, (n,))
    _need(k_pos, "k_pos", torch.int32, dev, (n,))
    _need(k_cache, "k_cache", (torch.bfloat16, torch.uint8), dev)
    fp8 = k_cache.dtype == torch.uint8
    if fp8:
        _need(k_scale, "k_scale", torch.float32, dev, (k_cache.shape[0],))
    if ws is None:
        ws = workspace(STATUS_BYTES, dev)
    _check(lib.dsa_indexer_append_keys(_ptr(k_new), _ptr(k_seq), _ptr(k_pos), n, batch.c,
                                       DSA_FP8_E4M3 if fp8 else DSA_BF16, _freq(inv_freq),
                                       _ptr(k_cache), _ptr(k_scale) if fp8 else None,
                                       k_cache.shape[0], _ptr(ws), ws.numel(),
                                       _stream(stream, dev)), "dsa_indexer_append_keys")
    return k_cache


def dsa_indexer_prepare_queries(q_new, batch: Batch, inv_freq, *, fp8=False, q_out=None,
                                q_scale=None, ws=None, stream=None):
    """RoPE (+ Hadamard + FP8) of the batch's indexer queries q_new bf16
    [num_q, 32, 128] at q_pos: returns q_out (bf16, or uint8 codes with
    q_scale fp32 [num_q, 32])."""
    dev = batch.device
    _need(q_new, "q_new", torch.bfloat16, dev, (batch.num_q, INDEX_HEADS, INDEX_DIM))
    if q_out is None:
        q_out = torch.empty(q_new.shape, dtype=torch.uint8 if fp8 else torch.bfloat16, device=dev)
    if fp8 and q_scale is None:
        q_scale = torch.empty((batch.num_q, INDEX_HEADS), dtype=torch.float32, device=dev)
    _need(q_out, "q_out", torch.uint8 if fp8 else torch.bfloat16, dev, tuple(q_new.shape))
    if ws is None:
        ws = workspace(STATUS_BYTES, dev)
    _check(lib.dsa_indexer_prepare_queries(_ptr(q_new), batch.c, DSA_FP8_E4M3 if fp8 else DSA_BF16,
                                           _freq(inv_freq), _ptr(q_out),
                                           _ptr(q_scale) if fp8 else None, _ptr(ws), ws.numel(),
                                           _stream(stream, dev)), "dsa_indexer_prepare_queries")
    return (q_out, q_scale) if fp8 else q_out


# ---------------------------------------------------------------- hot / cold KV
def _cold(t, name):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError(f"{name} must be page-locked host memory (pin_memory) or a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


class HotState:
    """Hot-buffer state of one index span (dsa_hot_t) on the device: slot ->
    position, slot stamps, position -> slot for positions < max_pos, and the
    last plan's fetch lists."""

    def __init__(self, num_seqs: int, hot_slots: int, max_pos: int, device="cuda"):
        dev = torch.device(device)
        i32 = dict(dtype=torch.int32, device=dev)
        self.num_seqs, self.hot_slots, self.max_pos, self.device = num_seqs, hot_slots, max_pos, dev
        self.slot_pos = torch.full((num_seqs, hot_slots), -1, **i32)
        self.slot_stamp = torch.full((num_seqs, hot_slots), -1, **i32)
        self.pos_slot = torch.full((num_seqs, max_pos), -1, **i32)
        self.fetch_pos = torch.zeros((num_seqs, hot_slots), **i32)
        self.fetch_slot = torch.zeros((num_seqs, hot_slots), **i32)
        self.fetch_count = torch.zeros((num_seqs,), **i32)
        self._c = _Hot(hot_slots, max_pos, *[_ptr(t) for t in (
            self.slot_pos, self.slot_stamp, self.pos_slot, self.fetch_pos, self.fetch_slot,
            self.fetch_count)])

    @property
    def c(self):
        return ctypes.byref(self._c)

    def fetch_lists(self):
        """[(position, slot), ...] per sequence of the last plan (host copy)."""
        n = self.fetch_count.cpu().tolist()
        fp, fs = self.fetch_pos.cpu(), self.fetch_slot.cpu()
        return [list(zip(fp[b, :n[b]].tolist(), fs[b, :n[b]].tolist())) for b in range(self.num_seqs)]


def dsa_hot_plan(idx, batch: Batch, state: HotState, step: int, rows=None, *, ws=None, stream=None):
    """One step of the hot buffer: returns rows int32 [num_q, k], the hot row
    of every valid index entry (-1 elsewhere); the state's fetch lists name
    the rows to swap in."""
    dev = batch.device
    _need(idx, "idx", torch.int32, dev)
    k = idx.shape[1]
    if rows is None:
        rows = torch.empty((batch.num_q, k), dtype=torch.int32, device=dev)
    _need(rows, "rows", torch.int32, dev, (batch.num_q, k))
    if ws is None:
        ws = workspace(STATUS_BYTES, dev)
    _check(lib.dsa_hot_plan(_ptr(idx), k, batch.c, state.c, int(step), _ptr(rows), _ptr(ws),
                            ws.numel(), _stream(stream, dev)), "dsa_hot_plan")
    return rows


def dsa_hot_fetch(state: HotState, batch: Batch, cold_kv, hot_kv, *, ws=None, stream=None):
    """Swap in the last plan's rows for every layer: hot_kv[l] (device, bf16
    [num_seqs * hot_slots, 576] or uint8 [.., 656]) from cold_kv[l] (pinned host
    memory, the batch's cache layout)."""
    dev = batch.device
    n = len(cold_kv)
    if len(hot_kv) != n:
        raise ValueError("one hot array per cold cache")
    fp8 = cold_kv[0].dtype == torch.uint8
    row = KV_ROW_FP8 if fp8 else KV_ROW
    for l in range(n):
        _cold(cold_kv[l], f"cold_kv[{l}]")
        _need(hot_kv[l], f"hot_kv[{l}]", cold_kv[0].dtype, dev,
              (state.num_seqs * state.hot_slots, row))
        if cold_kv[l].dtype != cold_kv[0].dtype or tuple(cold_kv[l].shape) != tuple(cold_kv[0].shape):
            raise ValueError("cold caches must share dtype and shape")
    if ws is None:
        ws = workspace(STATUS_BYTES, dev)
    cold = (c_void_p * n)(*[t.data_ptr() for t in cold_kv])
    hot = (c_void_p * n)(*[t.data_ptr() for t in hot_kv])
    _check(lib.dsa_hot_fetch(state.c, batch.c, n, ctypes.cast(cold, _PP), cold_kv[0].shape[0],
                             ctypes.cast(hot, _PP), hot_kv[0].shape[0],
                             DSA_FP8_E4M3 if fp8 else DSA_BF16, _ptr(ws), ws.numel(),
                             _stream(stream, dev)), "dsa_hot_fetch")
    return hot_kv


def dsa_hot_touch(cold_kv, *, stride: int = 65536, stream=None, device="cuda"):
    """Read every host page of the cold caches once from the device (one
    read per `stride` bytes), so that later swap-ins find their translations."""
    n = len(cold_kv)
    for l, t in enumerate(cold_kv):
        _cold(t, f"cold_kv[{l}]")
    if n == 0:
        return
    nbytes = cold_kv[0].numel() * cold_kv[0].element_size()
    if any(t.numel() * t.element_size() != nbytes for t in cold_kv):
        raise ValueError("cold caches must have the same size")
    cold = (c_void_p * n)(*[t.data_ptr() for t in cold_kv])
    _check(lib.dsa_hot_touch(n, ctypes.cast(cold, _PP), nbytes, int(stride),
                             _stream(stream, torch.device(device))), "dsa_hot_touch")


def dsa_sparse_mla_attn_rows(q_lat, q_rope, kv, rows, batch: Batch, *, scale: float, out=None,
                             lse=None, with_lse=True, ws=None, stream=None):
    """dsa_sparse_mla_attn whose index entries are absolute kv rows (e.g. the
    hot rows of dsa_hot_plan)."""
    dev = batch.device
    H = q_lat.shape[1]
    _need(q_lat, "q_lat", torch.bfloat16, dev, (batch.num_q, H, LATENT))
    _need(q_rope, "q_rope", torch.bfloat16, dev, (batch.num_q, H, ROPE))
    _need(kv, "kv", (torch.bfloat16, torch.uint8), dev)
    fp8 = kv.dtype == torch.uint8
    if kv.dim() != 2 or kv.shape[1] != (KV_ROW_FP8 if fp8 else KV_ROW):
        raise ValueError("kv must be bf16 [rows, 576] or uint8 [rows, 656]")
    _need(rows, "rows", torch.int32, dev)
    k = rows.shape[1]
    if out is None:
        out = torch.empty((batch.num_q, H, LATENT), dtype=torch.bfloat16, device=dev)
    if lse is None and with_lse:
        lse = torch.empty((batch.num_q, H), dtype=torch.float32, device=dev)
    if ws is None:
        ws = workspace(lib.dsa_sparse_mla_workspace_size(batch.c, H, k), dev)
    _check(lib.dsa_sparse_mla_attn_rows(_ptr(q_lat), _ptr(q_rope), _ptr(kv), kv.shape[0],
                                        DSA_FP8_E4M3 if fp8 else DSA_BF16, _ptr(rows), k, H,
                                        float(scale), batch.c, _ptr(out), _ptr(lse), _ptr(ws),
                                        ws.numel(), _stream(stream, dev)), "dsa_sparse_mla_attn_rows")
    return out, lse


class HotGroup:
    """Hot / cold arguments of indexshare_group_forward_hot (dsa_hot_group_t):
    one HotState per F layer, the layers' cold caches in pinned host memory
    (the group's layers[l]["kv"] are then the hot arrays)."""

    def __init__(self, spans, cold_kv, *, num_q: int, k: int, device="cuda"):
        self.spans = list(spans)
        self.cold_kv = list(cold_kv)
        for l, t in enumerate(self.cold_kv):
            _cold(t, f"cold_kv[{l}]")
        self.rows = torch.empty((num_q, k), dtype=torch.int32, device=device)
        self._spans = (_Hot * len(self.spans))(*[s._c for s in self.spans])
        self._cold = (c_void_p * len(self.cold_kv))(*[t.data_ptr() for t in self.cold_kv])
        self._c = _HotGroup(ctypes.cast(self._spans, POINTER(_Hot)), len(self.spans),
                            ctypes.cast(self._cold, _PP), self.cold_kv[0].shape[0], 0,
                            _ptr(self.rows))


def indexshare_group_forward_hot(group: Group, batch: Batch, hot: HotGroup, step: int,
                                 idx_buf=None, *, ws=None, stream=None):
    """indexshare_group_forward over hot buffers: per F layer, select, plan the
    span's hot buffer, swap in its missing rows for every layer of the span,
    and attend over hot rows.  Returns (outs, lses, idx_buf)."""
    dev = batch.device
    nl = len(group.layer_types)
    if len(hot.cold_kv) != nl:
        raise ValueError(f"{len(hot.cold_kv)} cold caches for {nl} layers")
    if len(hot.spans) != group.layer_types.count("F"):
        raise ValueError("one HotState per F layer")
    for l in range(nl):
        hk, ck = group.layers[l]["kv"], hot.cold_kv[l]
        if hk.dtype != ck.dtype or hk.shape[1] != ck.shape[1]:
            raise ValueError(f"layer {l}: hot and cold rows differ in dtype or width")
    if idx_buf is None:
        idx_buf = torch.empty((batch.num_q, group.k), dtype=torch.int32, device=dev)
    _need(idx_buf, "idx_buf", torch.int32, dev, (batch.num_q, group.k))
    _need(hot.rows, "hot.rows", torch.int32, dev, (batch.num_q, group.k))
    if ws is None:
        ws = workspace(group.workspace_size(batch), dev)
    hot._c.step = int(step)
    _check(lib.indexshare_group_forward_hot(group.c, batch.c, ctypes.byref(hot._c), _ptr(idx_buf),
                                            _ptr(ws), ws.numel(), _stream(stream, dev)),
           "indexshare_group_forward_hot")
    return group.outs, group.lses, idx_buf
