"""CPU oracle for the block-quantised KV decode path (numpy + a plain C library).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path (the
CUDA library and its Python binding) never imports, links or calls it, and the two
share no code: this side works on natural row-major layouts, quantises with the
plain fp32 rules and attends in fp64.

Definitions restated (sources named per function in ``kvq_oracle.c``):
  * q8_0 / q4_0 blocks of 32 values with one f16 scale, f16 control arm -- sized by
    "HAL #582 -- per-layer KV compression study", section 1 (size model table);
  * exact softmax attention ("logit-identical", same study, sections 3b and 5 P0);
  * exact merge of split softmax triples (same study, section 5 P2 read path).

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, brute force over codes, exact rational arithmetic, invariants and
library routines); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libkvq_oracle.so")

TYPES = {"f16": 0, "q8_0": 1, "q4_0": 2, "q4_1": 3, "q5_0": 4, "q5_1": 5}
QK = 32


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (no fused multiply-add, IEEE semantics)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-std=c11", "-o", _LIB_PATH + ".tmp", _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.kvqo_quantize_rows.argtypes = [i32, vp, i64, i32, vp, vp, i32]
        L.kvqo_quantize_rows.restype = None
        L.kvqo_dequantize_rows.argtypes = [i32, vp, vp, i64, i32, vp]
        L.kvqo_dequantize_rows.restype = None
        L.kvqo_attention.argtypes = [i32, vp, vp, i32, vp, vp, i32, i64, i64, i32, vp, i32,
                                     ctypes.c_float, vp, vp, i32]
        L.kvqo_attention.restype = None
        L.kvqo_attention_partials.argtypes = [i32, vp, vp, i32, vp, vp, i32, i64, i32, vp, i32,
                                              ctypes.c_float, vp, i32, vp, vp, vp]
        L.kvqo_attention_partials.restype = None
        L.kvqo_combine.argtypes = [vp, vp, vp, i64, i32, i32, vp, vp]
        L.kvqo_combine.restype = None
        L.kvqo_code_row_bytes.argtypes = [i32, i32]
        L.kvqo_code_row_bytes.restype = i64
        _lib = L
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def code_dtype(kv_type: str):
    return {"f16": np.uint16, "q8_0": np.int8}.get(kv_type, np.uint8)


def code_row_len(kv_type: str, D: int) -> int:
    """Number of code elements per row (f16: D halves, q8_0: D bytes, q4_0: D/2 packed
    bytes, q4_1 / q5_0 / q5_1: D codes, one per byte)."""
    return D // 2 if kv_type == "q4_0" else D


def scales_per_block(kv_type: str) -> int:
    """f16 scale values per 32-value block: 0 (f16), 2 for the types with a minimum (d, lo), else 1."""
    return 0 if kv_type == "f16" else (2 if kv_type in ("q4_1", "q5_1") else 1)


def quantize(kv_type: str, x: np.ndarray, n_threads: int = 1):
    """Quantise fp32 rows ``x[..., D]``.  Returns (codes, scales) in natural layout:
    codes ``[..., code_row_len]`` (f16 bits / int8 / packed uint8 / uint8 codes), scales
    f16 bits ``[..., D/32 * scales_per_block]`` ((d, lo) pairs for q4_1 / q5_1; an empty
    trailing axis for f16)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    D = x.shape[-1]
    assert D % QK == 0
    rows = int(np.prod(x.shape[:-1])) if x.ndim > 1 else 1
    codes = np.empty(x.shape[:-1] + (code_row_len(kv_type, D),), dtype=code_dtype(kv_type))
    nsc = scales_per_block(kv_type) * (D // QK)
    scales = np.empty(x.shape[:-1] + (nsc,), dtype=np.uint16)
    lib().kvqo_quantize_rows(TYPES[kv_type], _ptr(x), rows, D, _ptr(codes), _ptr(scales), n_threads)
    return codes, scales


def dequantize(kv_type: str, codes: np.ndarray, scales: np.ndarray, D: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    rows = int(np.prod(codes.shape[:-1])) if codes.ndim > 1 else 1
    out = np.empty(codes.shape[:-1] + (D,), dtype=np.float64)
    lib().kvqo_dequantize_rows(TYPES[kv_type], _ptr(codes), _ptr(scales), rows, D, _ptr(out))
    return out


def attention(type_k: str, k_codes, k_scales, type_v: str, v_codes, v_scales, n: int,
              q: np.ndarray, scale: float, n_threads: int = 1):
    """Decode attention of one sequence.  ``k_codes [Hkv, cap, row]``, ``k_scales
    [Hkv, cap, D/32]`` (same for V), ``q [Hq, D]`` fp32; attends over rows ``[0, n)``.
    Returns (out fp64 [Hq, D], lse fp64 [Hq])."""
    q = np.ascontiguousarray(q, dtype=np.float32)
    Hq, D = q.shape
    Hkv, cap = k_codes.shape[0], k_codes.shape[1]
    assert Hq % Hkv == 0 and n <= cap
    kc, ks = np.ascontiguousarray(k_codes), np.ascontiguousarray(k_scales, dtype=np.uint16)
    vc, vs = np.ascontiguousarray(v_codes), np.ascontiguousarray(v_scales, dtype=np.uint16)
    out = np.empty((Hq, D), dtype=np.float64)
    lse = np.empty((Hq,), dtype=np.float64)
    lib().kvqo_attention(TYPES[type_k], _ptr(kc), _ptr(ks), TYPES[type_v], _ptr(vc), _ptr(vs),
                         Hkv, cap, n, D, _ptr(q), Hq, ctypes.c_float(scale), _ptr(out), _ptr(lse),
                         n_threads)
    return out, lse


def attention_partials(type_k: str, k_codes, k_scales, type_v: str, v_codes, v_scales,
                       bounds, q: np.ndarray, scale: float):
    """Unnormalised split triples over key ranges ``[bounds[s], bounds[s+1])``.
    Returns (o [Hq, S, D], m [Hq, S], l [Hq, S]) in fp64, natural-log units."""
    q = np.ascontiguousarray(q, dtype=np.float32)
    Hq, D = q.shape
    Hkv, cap = k_codes.shape[0], k_codes.shape[1]
    b = np.ascontiguousarray(np.asarray(bounds, dtype=np.int64))
    S = len(b) - 1
    kc, ks = np.ascontiguousarray(k_codes), np.ascontiguousarray(k_scales, dtype=np.uint16)
    vc, vs = np.ascontiguousarray(v_codes), np.ascontiguousarray(v_scales, dtype=np.uint16)
    o = np.empty((Hq, S, D), dtype=np.float64)
    m = np.empty((Hq, S), dtype=np.float64)
    l = np.empty((Hq, S), dtype=np.float64)
    lib().kvqo_attention_partials(TYPES[type_k], _ptr(kc), _ptr(ks), TYPES[type_v], _ptr(vc),
                                  _ptr(vs), Hkv, cap, D, _ptr(q), Hq, ctypes.c_float(scale),
                                  _ptr(b), S, _ptr(o), _ptr(m), _ptr(l))
    return o, m, l


def combine(part_o: np.ndarray, part_m: np.ndarray, part_l: np.ndarray):
    """Merge split triples: ``part_o [R, S, D]``, ``part_m/part_l [R, S]`` -> (out [R, D], lse [R])."""
    po = np.ascontiguousarray(part_o, dtype=np.float64)
    pm = np.ascontiguousarray(part_m, dtype=np.float64)
    pl = np.ascontiguousarray(part_l, dtype=np.float64)
    R, S, D = po.shape
    out = np.empty((R, D), dtype=np.float64)
    lse = np.empty((R,), dtype=np.float64)
    lib().kvqo_combine(_ptr(po), _ptr(pm), _ptr(pl), R, S, D, _ptr(out), _ptr(lse))
    return out, lse


# Bits of one stored code of each type (f16: the value itself).
CODE_BITS = {"f16": 16, "q8_0": 8, "q4_0": 4, "q4_1": 4, "q5_0": 5, "q5_1": 5}


def block_storage_bytes(kv_type: str) -> int:
    """Packed storage of one 32-value block: 32 codes of CODE_BITS bits plus its f16 scale
    values (d, and lo for the types with a minimum).  The natural layouts returned by
    ``quantize`` keep 5-bit and q4_1 codes one per byte, so their arrays are larger."""
    return QK * CODE_BITS[kv_type] // 8 + 2 * scales_per_block(kv_type)


# Bytes of one 32-value block, pinned by the pages: f16, q8_0, q5_0, q4_0 by the size model
# table of "HAL #582 -- per-layer KV compression study", section 1 (192 / 102 / 66 / 54
# KiB per token of the 14B shape); q5_1 by the section 5 P1 validation (q5_1 K + q4_0 V =
# 2016 MiB at 32768 cells, i.e. 63 KiB per token, of which q4_0 V is 27).  q4_1 is not
# printed on the pages (its 20 bytes follow from block_storage_bytes alone).
BLOCK_BYTES = {t: block_storage_bytes(t) for t in ("f16", "q8_0", "q4_0", "q5_0", "q5_1")}
TIER_LADDER = [("f16", "f16"), ("q8_0", "q8_0"), ("q8_0", "q4_0"), ("q5_1", "q4_0")]


def kv_cache_bytes(cells: int, n_layers: int, n_kv_heads: int, head_dim: int, type_k: str, type_v: str) -> int:
    """Whole-cache bytes: every cell stores head_dim values per KV head per layer, for K and V."""
    blocks = cells * n_layers * n_kv_heads * (head_dim // QK)
    return blocks * (BLOCK_BYTES[type_k] + BLOCK_BYTES[type_v])


def select_tier(cells: int, n_layers: int, n_kv_heads: int, head_dim: int, budget_bytes: int) -> dict:
    """Automatic KV tier (same study, section 5 P1): walk the ladder f16 -> q8/q8 -> q8K/q4V ->
    q5_1K/q4V and take the first (least compressing) rung whose whole cache fits the budget;
    if none fits, take the last rung and report that it does not fit."""
    for rung, (tk, tv) in enumerate(TIER_LADDER):
        size = kv_cache_bytes(cells, n_layers, n_kv_heads, head_dim, tk, tv)
        last = rung == len(TIER_LADDER) - 1
        if size <= budget_bytes or last:
            return {"rung": rung, "type_k": tk, "type_v": tv, "fits": size <= budget_bytes, "bytes": size}


def f16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
