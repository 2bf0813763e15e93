"""Seeded synthetic inputs for the decode path (shared by tests, benchmark and smoke check).

Holds no arithmetic of the method: it only draws Q, K, V from fixed seeds, with the
shapes and value distributions of the workloads the pages measure (the 10-layer,
2-KV-head, D=256 hybrid model of "kv: 8-bit KV cache as a bolt-tier long-context decode
lever"; the 48-layer, 8-KV-head, D=128 dense model of "HAL #582 -- per-layer KV
compression study").  No dataset or trained weights are involved.

Recipe: Q, V ~ N(0, 1); K ~ N(0, 1) with, per (layer, KV head), 4 distinct outlier
channels (a seeded permutation of the head dimension) multiplied by 10 for every row.
Rows are drawn in fixed chunks of 4096 positions, each chunk from its own seed, so any
row range of any (layer, sequence, head) can be regenerated on its own.  Generation runs
on the GPU (torch's CUDA generator); CPU-side consumers copy the tensors to the host.
"""
from __future__ import annotations

import dataclasses
import math

import torch

CHUNK = 4096
_MASK = (1 << 64) - 1


def mix(*parts: int) -> int:
    """splitmix64-style hash of integers -> a 63-bit seed."""
    h = 0x9E3779B97F4A7C15
    for p in parts:
        h = (h ^ (int(p) & _MASK)) & _MASK
        h = (h + 0x9E3779B97F4A7C15) & _MASK
        z = h
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK
        h = z ^ (z >> 31)
    return h & ((1 << 63) - 1)


KIND_K, KIND_V, KIND_Q, KIND_NEWK, KIND_NEWV, KIND_PERM = 1, 2, 3, 4, 5, 6


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    layers: int
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    type_k: str
    type_v: str
    lengths: tuple          # per-sequence context length
    outliers: int = 4       # outlier channels per (layer, KV head) in K
    outlier_scale: float = 10.0
    seed: int = 1234

    @property
    def G(self):
        return self.n_q_heads // self.n_kv_heads

    @property
    def scale(self):
        return float(torch.tensor(1.0 / math.sqrt(self.head_dim), dtype=torch.float32))


def _normal(shape, seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def outlier_channels(wl: Workload, layer: int, h: int):
    if wl.outliers <= 0:
        return []
    g = torch.Generator(device="cpu")
    g.manual_seed(mix(wl.seed, KIND_PERM, layer, h))
    return torch.randperm(wl.head_dim, generator=g)[: wl.outliers].tolist()


def kv_rows(wl: Workload, kind: int, layer: int, b: int, h: int, t0: int, n: int, device="cuda"):
    """Rows [t0, t0+n) of K (kind=KIND_K) or V (KIND_V) for (layer, sequence b, KV head h)."""
    D = wl.head_dim
    out = torch.empty((n, D), dtype=torch.float32, device=device)
    c0, c1 = t0 // CHUNK, (t0 + n + CHUNK - 1) // CHUNK
    for c in range(c0, c1):
        blk = _normal((CHUNK, D), mix(wl.seed, kind, layer, b, h, c), device)
        lo, hi = max(t0, c * CHUNK), min(t0 + n, (c + 1) * CHUNK)
        out[lo - t0:hi - t0] = blk[lo - c * CHUNK:hi - c * CHUNK]
    if kind == KIND_K and wl.outliers > 0:
        out[:, outlier_channels(wl, layer, h)] *= wl.outlier_scale
    return out


def layer_kv(wl: Workload, layer: int, kind: int, n_rows: int, device="cuda", b_range=None):
    """K or V of one layer as [nb, Hkv, n_rows, D] (rows [0, n_rows) of each sequence)."""
    bs = range(wl.batch) if b_range is None else b_range
    out = torch.empty((len(bs), wl.n_kv_heads, n_rows, wl.head_dim), dtype=torch.float32, device=device)
    for i, b in enumerate(bs):
        for h in range(wl.n_kv_heads):
            out[i, h] = kv_rows(wl, kind, layer, b, h, 0, n_rows, device)
    return out


def queries(wl: Workload, layer: int, step: int = 0, device="cuda"):
    """Q [B, Hq, D] for one decode step of one layer."""
    return _normal((wl.batch, wl.n_q_heads, wl.head_dim), mix(wl.seed, KIND_Q, layer, step), device)


def new_rows(wl: Workload, layer: int, step: int, device="cuda"):
    """The K and V rows [B, Hkv, 1, D] a decode step appends (K keeps its outlier channels)."""
    k = _normal((wl.batch, wl.n_kv_heads, 1, wl.head_dim), mix(wl.seed, KIND_NEWK, layer, step), device)
    v = _normal((wl.batch, wl.n_kv_heads, 1, wl.head_dim), mix(wl.seed, KIND_NEWV, layer, step), device)
    for h in range(wl.n_kv_heads):
        ch = outlier_channels(wl, layer, h)
        if ch:
            k[:, h, :, ch] *= wl.outlier_scale
    return k, v


def session_lengths(seed: int, n: int, lo: int, hi: int):
    """n integer context lengths uniform in [lo, hi] (inclusive), from a seed."""
    g = torch.Generator(device="cpu")
    g.manual_seed(mix(seed, 77))
    return tuple(int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g))


# ---- the workloads (sizes and distributions of the pages' models) ----

def tiny():
    """1 layer, batch 1, ctx 512, Hkv 2, Hq 4, D 128, q8_0 K and V, Q/K/V ~ N(0,1)."""
    return Workload("tiny-q8_0-q8_0-ctx512", 1, 1, 4, 2, 128, "q8_0", "q8_0", (512,), outliers=0)


def hybrid(ctx: int, type_k="q8_0", type_v="q8_0"):
    """10 full-attention layers, batch 1, Hkv 2, Hq 16, D 256 (qwisp #168 hybrid model)."""
    return Workload(f"hybrid-10L-{type_k}-{type_v}-ctx{ctx}", 10, 1, 16, 2, 256, type_k, type_v, (ctx,))


def dense14b(ctx: int, type_k="q8_0", type_v="q4_0"):
    """48 layers, batch 1, Hkv 8, Hq 40, D 128 (HAL #582 14B model)."""
    return Workload(f"dense-48L-{type_k}-{type_v}-ctx{ctx}", 48, 1, 40, 8, 128, type_k, type_v, (ctx,))


def multi_session(type_k="q8_0", type_v="q4_0", n=16, lo=8192, hi=65536, seed=1234):
    """48 layers, 16 sequences with ctx uniform in [8K, 64K] from the seed, Hkv 8, Hq 40, D 128."""
    return Workload(f"multi-session-48L-{n}seq-{type_k}-{type_v}", 48, n, 40, 8, 128, type_k, type_v,
                    session_lengths(seed, n, lo, hi), seed=seed)
