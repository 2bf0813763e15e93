"""Host-side checks of the C ABI that need no GPU: the library loads, exports every entry
point the header declares, reproduces the pages' cache sizes, and rejects bad input."""
import ctypes
import os
import subprocess

import pytest

import quantised_kv_long_gb300 as kvq
from tests import kvq_layout

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_library_exports_every_header_symbol():
    names = kvq.header_functions()
    assert len(names) >= 15
    out = subprocess.run(["nm", "-D", "--defined-only", kvq.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    for n in names:
        assert n in exported, n
        assert hasattr(kvq.lib, n)
    assert kvq.lib.kvq_abi_version() == 4


def test_status_strings():
    for code in range(7):
        assert kvq.lib.kvq_status_string(code)
    assert kvq.lib.kvq_status_string(3) == b"append exceeds cache capacity"


def _golden_rows():
    rows = []
    with open(os.path.join(GOLDEN, "size_model.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                src, L, H, D, tk, tv, ctx, val, unit = [t.strip() for t in line.split("|")]
                rows.append((src, int(L), int(H), int(D), tk, tv, int(ctx), float(val), unit))
    return rows


@pytest.mark.parametrize("row", _golden_rows(), ids=lambda r: f"{r[0]}-{r[4]}-{r[5]}-{r[6]}")
def test_cache_size_matches_pages(row):
    """kvq_cache_size of one layer x layers reproduces every size the pages print."""
    src, L, H, D, tk, tv, ctx, val, unit = row
    cap = ctx if ctx % 16 == 0 else 16
    kb, vb, sb = kvq.cache_size(1, H, D, cap, tk, tv)
    per_tok = L * (kb + vb) / cap
    if unit == "KiB_per_token":
        assert per_tok / 1024 == val
    elif unit == "MiB":
        assert L * (kb + vb) / 2**20 == val
    else:
        assert per_tok == val
    assert sb % 16 == 0 and sb >= 4 * 3


def test_cache_size_hybrid_examples():
    # qwisp #168 Observation table: f16 KV of the hybrid model, 160 MB at 8K and 5.0 GB at 262,144
    kb, vb, _ = kvq.cache_size(1, 2, 256, 8192, "f16", "f16")
    assert 10 * (kb + vb) == 160 * 2**20
    kb, vb, _ = kvq.cache_size(1, 2, 256, 262144, "f16", "f16")
    assert 10 * (kb + vb) == 5 * 2**30
    # "8-bit saves" column: q8_0 is 8.5 bits per value, so the saving is 15/32 of f16
    kq, vq, _ = kvq.cache_size(1, 2, 256, 8192, "q8_0", "q8_0")
    assert (kb + vb) * 8192 // 262144 - (kq + vq) == (kb + vb) * 8192 // 262144 * 15 // 32


@pytest.mark.parametrize("desc,status", [
    ((0, 8, 128, 64, "q8_0", "q8_0"), 1),      # batch 0
    ((1, 0, 128, 64, "q8_0", "q8_0"), 1),      # no heads
    ((1, 8, 128, 40, "q8_0", "q8_0"), 1),      # capacity not a multiple of 16
    ((1, 8, 128, 0, "q8_0", "q8_0"), 1),       # zero capacity
    ((1, 8, 64, 64, "q8_0", "q8_0"), 2),       # head_dim 64 unsupported
    ((1, 8, 96, 64, "q8_0", "q8_0"), 2),       # head_dim not a multiple of 128
    ((1, 8, 128, 64, 7, "q8_0"), 2),           # unknown type
])
def test_bad_descriptors_rejected(desc, status):
    with pytest.raises(kvq.KvqError) as e:
        kvq.cache_size(*desc)
    assert e.value.status == status


def test_null_pointers_rejected_without_cuda():
    d = kvq.Desc(1, 2, 128, 64, 1, 1)
    h = ctypes.c_void_p()
    assert kvq.lib.kvq_cache_create(ctypes.byref(d), None, None, None, None, ctypes.byref(h)) == 1
    assert kvq.lib.kvq_cache_size(None, None, None, None) == 1
    assert kvq.lib.kvq_cache_destroy(None) == 1
    assert kvq.lib.kvq_quantize_append(None, None, None, 0, 1, 1, None) == 1
    assert kvq.lib.kvq_decode_attention(None, None, 4, ctypes.c_float(1.0), 0, None, None, None, None) == 1
    assert kvq.lib.kvq_combine(None, None, None, 1, 1, 128, None, None, None) == 1
    f1 = ctypes.c_float(1.0)
    assert kvq.lib.kvq_window_append(None, None, None, None, None) == 1
    assert kvq.lib.kvq_window_decode(None, None, None, 4, f1, None, None, None, None) == 1
    assert kvq.lib.kvq_window_append_decode(None, None, None, None, None, 4, f1, None, None, None, None) == 1
    # misaligned pointers are refused before any CUDA call
    fake = ctypes.c_void_p(0x1000)
    bad = ctypes.c_void_p(0x1004)
    assert kvq.lib.kvq_cache_create(ctypes.byref(d), bad, fake, fake, None, ctypes.byref(h)) == 4
    assert kvq.lib.kvq_combine(bad, fake, fake, 1, 1, 128, fake, None, None) == 4
    assert kvq.lib.kvq_combine(fake, fake, fake, 1, 0, 128, fake, None, None) == 1
    assert kvq.lib.kvq_combine(fake, fake, fake, 1, 1, 130, fake, None, None) == 1


def test_layout_is_a_bijection():
    kvq_layout.check_bijective()


def test_block_bytes():
    assert [kvq.block_bytes(t) for t in ("f16", "q8_0", "q4_0", "q5_1")] == [64, 34, 18, 24]
    assert kvq.lib.kvq_block_bytes(9) == 0


def test_select_tier_matches_oracle():
    import oracle
    shapes = [(32768, 48, 8, 128), (65536, 10, 2, 256), (262144, 48, 8, 128), (1, 1, 1, 32), (0, 4, 4, 64)]
    for cells, L, H, D in shapes:
        sizes = [oracle.kv_cache_bytes(cells, L, H, D, tk, tv) for tk, tv in oracle.TIER_LADDER]
        budgets = {0, 1} | {s + d for s in sizes for d in (-1, 0, 1) if s + d >= 0}
        for budget in sorted(budgets):
            assert kvq.select_tier(cells, L, H, D, budget) == oracle.select_tier(cells, L, H, D, budget), \
                (cells, L, H, D, budget)


def test_select_tier_rejects_bad_arguments():
    c = kvq.TierChoice()
    for args in [(-1, 48, 8, 128), (1, 0, 8, 128), (1, 48, 0, 128), (1, 48, 8, 100), (1, 48, 8, 0),
                 (1 << 62, 1 << 20, 1 << 10, 1 << 20)]:
        assert kvq.lib.kvq_select_tier(*args, 1 << 30, ctypes.byref(c)) == 1, args
    assert kvq.lib.kvq_select_tier(1, 48, 8, 128, 1 << 30, None) == 1


def test_cache_size_of_further_types_is_the_block_footprint():
    """Plane sizes of the further types against the oracle's packed block sizes (q5_0 and
    q5_1 pinned there by the pages' 66 KiB/token and 2016 MiB rows), not the library's own."""
    import oracle
    for tk, tv in [("q8_0", "q5_0"), ("q5_0", "q5_0"), ("q5_1", "q5_1"), ("q4_1", "q4_1"), ("q5_1", "q4_0")]:
        for D in (128, 256):
            kb, vb, _ = kvq.cache_size(2, 3, D, 64, tk, tv)
            blocks = 2 * 3 * 64 * D // 32
            assert kb == blocks * oracle.block_storage_bytes(tk), (tk, tv, D)
            assert vb == blocks * oracle.block_storage_bytes(tv), (tk, tv, D)
            assert kvq.block_bytes(tk) == oracle.block_storage_bytes(tk)
    # pairs outside the supported set are refused
    d = kvq.Desc(1, 2, 128, 64, kvq.Q5_1, kvq.Q8_0)
    kb, vb, sb = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    assert kvq.lib.kvq_cache_size(ctypes.byref(d), ctypes.byref(kb), ctypes.byref(vb), ctypes.byref(sb)) == 2
