"""Seeded synthetic inputs for the DSA layer group with IndexShare.

This module draws random tensors shaped like the workloads of the GLM-5.2
pages and holds none of the method's arithmetic; both the oracle (through
host copies) and the CUDA path consume exactly the tensors it returns.

Workloads (all seeded):

* ``tiny``      prefill of one 512-token sequence, H=16 MLA heads, K=64;
                every tensor integer-valued in [-3, 3], head weights in
                {-1, 0, 1, 2}, so indexer scores are exact in fp32.
* ``prefill8k`` one 8192-token causal prefill, H=64, K=2048.
* ``decode64``  64 sequences, one query each, context ~ U[98304, 131072].
* ``chunked``   4096 new queries after a 131072-token cached prefix, 8 layers.
* ``decode1m``  4 sequences of 1,048,576 positions, FP8 indexer keys.
* ``prefill2k`` / ``decode8`` / ``chunked1k``: the same shapes at 2560 tokens /
  8 sequences / 1024 new queries (4 layers), small enough for profiler captures.

Gaussian workloads draw each vector as N(0, 1)/sqrt(d) with d its own width
(128 for indexer q/k, 512 for latent parts, 64 for RoPE parts) and head
weights as N(0, 1)/sqrt(32); values are rounded to bf16 (round to nearest
even).  RoPE is not applied: a rotation of i.i.d. isotropic Gaussian pairs
leaves their joint distribution unchanged, so drawing the post-RoPE values
directly gives inputs with the same statistics.

Layout: query-major rows, sequences packed back to back.
  q_idx [num_q, 32, 128], w [num_q, 32] fp32, k_idx [rows, 128]
  q_lat [num_q, H, 512], q_rope [num_q, H, 64], kv [rows, 576]
  q_start [num_seqs+1] int32, q_pos [num_q] int32, seq_row0 [num_seqs] int64
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

HI, DI, DL, DR = 32, 128, 512, 64

WORKLOADS = {
    "tiny": dict(kind="prefill", T=512, H=16, K=64, layers="FSSS", ints=True),
    "prefill8k": dict(kind="prefill", T=8192, H=64, K=2048, layers="FSSS"),
    "decode64": dict(kind="decode", B=64, lo=98304, hi=131072, H=64, K=2048, layers="FSSS"),
    "chunked": dict(kind="chunked", prefix=131072, Tq=4096, H=64, K=2048, layers="FSSSFSSS"),
    "decode1m": dict(kind="decode", B=4, lo=1048576, hi=1048576, H=64, K=2048, layers="FSSS",
                     fp8=True),
    # smaller cases of the same kernels, sized for profiler captures
    "prefill2k": dict(kind="prefill", T=2560, H=64, K=2048, layers="FSSS"),
    "decode8": dict(kind="decode", B=8, lo=98304, hi=131072, H=64, K=2048, layers="FSSS"),
    "chunked1k": dict(kind="chunked", prefix=131072, Tq=1024, H=64, K=2048, layers="FSSS"),
}


def round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


@dataclasses.dataclass
class Layout:
    """Batch layout: which query rows belong to which sequence and where."""
    num_seqs: int
    num_q: int
    max_q: int
    max_len: int          # capacity of a score row, multiple of 128
    rows: int             # cache rows per layer
    q_start: np.ndarray   # int32 [num_seqs + 1]
    q_pos: np.ndarray     # int32 [num_q]
    seq_row0: np.ndarray  # int64 [num_seqs]
    seq_len: np.ndarray   # int64 [num_seqs] cached positions per sequence


def make_layout(seq_lens, q_counts) -> Layout:
    """Each sequence b has seq_lens[b] cached positions and its q_counts[b]
    queries sit at the last q_counts[b] positions."""
    seq_lens = np.asarray(seq_lens, np.int64)
    q_counts = np.asarray(q_counts, np.int64)
    assert (q_counts <= seq_lens).all() and (q_counts >= 0).all()
    B = seq_lens.size
    q_start = np.zeros(B + 1, np.int32)
    q_start[1:] = np.cumsum(q_counts)
    seq_row0 = np.zeros(B, np.int64)
    seq_row0[1:] = np.cumsum(seq_lens)[:-1]
    q_pos = np.concatenate([np.arange(L - n, L) for L, n in zip(seq_lens, q_counts)]
                           ).astype(np.int32) if q_counts.sum() else np.zeros(0, np.int32)
    return Layout(num_seqs=B, num_q=int(q_counts.sum()), max_q=int(q_counts.max(initial=0)),
                  max_len=round_up(int(seq_lens.max(initial=1)), 128), rows=int(seq_lens.sum()),
                  q_start=q_start, q_pos=q_pos, seq_row0=seq_row0, seq_len=seq_lens)


def workload_layout(name: str, seed: int = 0) -> Layout:
    cfg = WORKLOADS[name]
    if cfg["kind"] == "prefill":
        return make_layout([cfg["T"]], [cfg["T"]])
    if cfg["kind"] == "chunked":
        L = cfg["prefix"] + cfg["Tq"]
        return make_layout([L], [cfg["Tq"]])
    rng = np.random.Generator(np.random.PCG64(10_000 + seed))
    lens = rng.integers(cfg["lo"], cfg["hi"], size=cfg["B"], endpoint=True)
    return make_layout(lens, np.ones(cfg["B"], np.int64))


# ---------------------------------------------------------------- host (numpy)
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


class HostGen:
    """numpy PCG64 stream per (seed, tensor id)."""

    def __init__(self, seed: int):
        self.seed = seed

    def rng(self, tid: int):
        return np.random.Generator(np.random.PCG64(self.seed * 1000 + tid))

    def gauss_bf16(self, tid, shape, width):
        x = self.rng(tid).standard_normal(shape, dtype=np.float32) / np.float32(math.sqrt(width))
        return f32_to_bf16_bits(x)

    def int_bf16(self, tid, shape, lo=-3, hi=3):
        x = self.rng(tid).integers(lo, hi, size=shape, endpoint=True).astype(np.float32)
        return f32_to_bf16_bits(x)

    def gauss_f32(self, tid, shape, width):
        return (self.rng(tid).standard_normal(shape, dtype=np.float32)
                / np.float32(math.sqrt(width))).astype(np.float32)

    def int_w(self, tid, shape):
        return self.rng(tid).choice(np.array([-1, 0, 1, 2], np.float32), size=shape)


def host_layers(layout: Layout, layer_types: str, H: int, *, ints: bool, seed: int = 0):
    """Per-layer host tensors (numpy; bf16 as uint16 bit patterns)."""
    g = HostGen(seed)
    nq, rows = layout.num_q, layout.rows
    layers = []
    for l, t in enumerate(layer_types):
        base = 100 * (l + 1)
        if ints:
            L = dict(q_lat=g.int_bf16(base + 0, (nq, H, DL)), q_rope=g.int_bf16(base + 1, (nq, H, DR)),
                     kv=g.int_bf16(base + 2, (rows, DL + DR)))
        else:
            kv = np.empty((rows, DL + DR), np.uint16)
            kv[:, :DL] = g.gauss_bf16(base + 2, (rows, DL), DL)
            kv[:, DL:] = g.gauss_bf16(base + 3, (rows, DR), DR)
            L = dict(q_lat=g.gauss_bf16(base + 0, (nq, H, DL), DL),
                     q_rope=g.gauss_bf16(base + 1, (nq, H, DR), DR), kv=kv)
        if t == "F":
            if ints:
                L.update(q_idx=g.int_bf16(base + 10, (nq, HI, DI)), w=g.int_w(base + 11, (nq, HI)),
                         k_idx=g.int_bf16(base + 12, (rows, DI)))
            else:
                L.update(q_idx=g.gauss_bf16(base + 10, (nq, HI, DI), DI),
                         w=g.gauss_f32(base + 11, (nq, HI), HI),
                         k_idx=g.gauss_bf16(base + 12, (rows, DI), DI))
        layers.append(L)
    return layers


def planted_host_layers(layout: Layout, layer_types: str, H: int, *, m: int, seed: int = 0,
                        latent_gain: float = 4.0):
    """Gaussian layers as host_layers, plus a planted set of m relevant
    positions per sequence (drawn among the positions every query of the
    sequence sees): their indexer keys lie along a direction u_b that every
    indexer head of the sequence's queries also points along (with positive
    head weights), and their latent rows along a direction v_b shared by the
    queries' latent parts, scaled so that those positions lead both the
    indexer ranking and the attention (latent_gain sets the attention's margin:
    a planted key's score exceeds a random one's by about latent_gain^2 / 16
    in the softmax exponent).  Returns (layers,
    planted positions per sequence).  The premise of sparse attention made
    explicit, for tolerance checks of quantised indexers."""
    layers = host_layers(layout, layer_types, H, ints=False, seed=seed)
    planted = []
    for b, (qs, qe, pos, u, v) in enumerate(_planted_draws(layout, m, seed)):
        planted.append(pos)
        if qe == qs:
            continue
        rows = int(layout.seq_row0[b]) + pos
        for l, t in enumerate(layer_types):
            L = layers[l]
            lat = bf16_bits_to_f32(L["kv"][rows, :DL])
            L["kv"][rows, :DL] = f32_to_bf16_bits((lat + latent_gain * v).astype(np.float32))
            ql = bf16_bits_to_f32(L["q_lat"][qs:qe])
            L["q_lat"][qs:qe] = f32_to_bf16_bits((ql + latent_gain * v).astype(np.float32))
            if t == "F":
                k = bf16_bits_to_f32(L["k_idx"][rows])
                L["k_idx"][rows] = f32_to_bf16_bits((k + u).astype(np.float32))
                q = bf16_bits_to_f32(L["q_idx"][qs:qe])
                L["q_idx"][qs:qe] = f32_to_bf16_bits((q + u).astype(np.float32))
                L["w"][qs:qe] = np.abs(L["w"][qs:qe])
    return layers, planted


def _planted_draws(layout: Layout, m: int, seed: int):
    """Per sequence: (query rows [qs, qe), planted positions, u [128], v [512])
    drawn from the seeded host stream shared by both planting functions."""
    g = HostGen(seed + 7919)
    out = []
    for b in range(layout.num_seqs):
        qs, qe = int(layout.q_start[b]), int(layout.q_start[b + 1])
        if qe == qs:
            out.append((qs, qe, np.zeros(0, np.int64), None, None))
            continue
        first = int(layout.q_pos[qs:qe].min()) + 1       # positions every query sees
        r = g.rng(10 * b)
        pos = np.sort(r.choice(first, size=min(m, first), replace=False)).astype(np.int64)
        u = r.standard_normal(DI)
        u /= np.linalg.norm(u)
        v = r.standard_normal(DL)
        v /= np.linalg.norm(v)
        out.append((qs, qe, pos, u, v))
    return out


def plant_device(layers, layout: Layout, layer_types: str, *, m: int, seed: int = 0,
                 latent_gain: float = 4.0):
    """The planted relevant set of planted_host_layers, applied in place to
    device layers (torch tensors from device_layers), for workloads too large
    to draw on the host: the same positions and directions for the same
    layout, m and seed, and the same arithmetic (fp64 sum, rounded to fp32,
    then to bf16).  Returns the planted positions per sequence."""
    import torch

    planted = []
    for b, (qs, qe, pos, u, v) in enumerate(_planted_draws(layout, m, seed)):
        planted.append(pos)
        if qe == qs:
            continue
        dev = layers[0]["kv"].device
        rows = torch.as_tensor(int(layout.seq_row0[b]) + pos, device=dev)
        uu = torch.as_tensor(u, dtype=torch.float64, device=dev)
        vv = torch.as_tensor(latent_gain * v, dtype=torch.float64, device=dev)
        add = lambda t, d: (t.double() + d).float().to(torch.bfloat16)
        for l, t in enumerate(layer_types):
            L = layers[l]
            L["kv"][rows, :DL] = add(L["kv"][rows, :DL], vv)
            L["q_lat"][qs:qe] = add(L["q_lat"][qs:qe], vv)
            if t == "F":
                L["k_idx"][rows] = add(L["k_idx"][rows], uu)
                L["q_idx"][qs:qe] = add(L["q_idx"][qs:qe], uu)
                L["w"][qs:qe] = L["w"][qs:qe].abs()
    return planted


# ---------------------------------------------------------------- device (torch)
def device_layers(layout: Layout, layer_types: str, H: int, *, device, seed: int = 0,
                  ints: bool = False):
    """Per-layer device tensors drawn with torch's seeded generator on
    `device` (for workloads too large to draw on the host).  bf16 tensors are
    torch.bfloat16; w is float32."""
    import torch

    gen = torch.Generator(device=device)
    nq, rows = layout.num_q, layout.rows

    def gauss(tid, shape, width):
        gen.manual_seed(seed * 1000 + tid)
        x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
        return x.mul_(1.0 / math.sqrt(width)).to(torch.bfloat16)

    def ints_(tid, shape):
        gen.manual_seed(seed * 1000 + tid)
        return torch.randint(-3, 4, shape, generator=gen, device=device).to(torch.bfloat16)

    layers = []
    for l, t in enumerate(layer_types):
        base = 100 * (l + 1)
        if ints:
            L = dict(q_lat=ints_(base, (nq, H, DL)), q_rope=ints_(base + 1, (nq, H, DR)),
                     kv=ints_(base + 2, (rows, DL + DR)))
        else:
            kv = torch.empty((rows, DL + DR), dtype=torch.bfloat16, device=device)
            kv[:, :DL] = gauss(base + 2, (rows, DL), DL)
            kv[:, DL:] = gauss(base + 3, (rows, DR), DR)
            L = dict(q_lat=gauss(base, (nq, H, DL), DL), q_rope=gauss(base + 1, (nq, H, DR), DR),
                     kv=kv)
        if t == "F":
            if ints:
                gen.manual_seed(seed * 1000 + base + 11)
                wv = torch.tensor([-1.0, 0.0, 1.0, 2.0], device=device)
                w = wv[torch.randint(0, 4, (nq, HI), generator=gen, device=device)]
                L.update(q_idx=ints_(base + 10, (nq, HI, DI)), w=w,
                         k_idx=ints_(base + 12, (rows, DI)))
            else:
                gen.manual_seed(seed * 1000 + base + 11)
                w = torch.randn((nq, HI), generator=gen, device=device) * (1.0 / math.sqrt(HI))
                L.update(q_idx=gauss(base + 10, (nq, HI, DI), DI), w=w.float(),
                         k_idx=gauss(base + 12, (rows, DI), DI))
        layers.append(L)
    return layers
