"""Test-side reader of the cache layout documented in include/kvq.h.

Turns the raw K/V planes of a cache (uint8 arrays copied to the host) back into the
natural row-major codes and scales the oracle produces, using only the byte-offset
formulas printed in the header.  Shares nothing with the CUDA path.
"""
import numpy as np

CODE_TILE = {"f16": 4096, "q8_0": 2048, "q4_0": 1024, "q4_1": 1024, "q5_0": 1280, "q5_1": 1280}
SCALE_TILE = {"f16": 0, "q8_0": 128, "q4_0": 128, "q4_1": 256, "q5_0": 128, "q5_1": 256}
NIBBLE = ("q4_0", "q4_1", "q5_0", "q5_1")


def _pair(kt):
    kt = np.asarray(kt)
    j = np.where(kt < 8, kt // 2, (kt - 8) // 2)
    pos = np.where(kt < 8, kt % 2, 2 + kt % 2)
    return j, pos


def _q_of_pos(pos):  # A,B,C,D -> byte 0,2,1,3 of a V word
    return np.array([0, 2, 1, 3])[pos]


def tile_offsets(kv_type: str, is_v: bool):
    """(off[16,128], nibble[16,128]) byte offset of (row kt, value dd) inside one
    (tile, slice) of codes, and 0/1 for the low/high nibble (q4_0) or -1."""
    kt, dd = np.meshgrid(np.arange(16), np.arange(128), indexing="ij")
    n, st = kt % 8, kt // 8
    b, i = dd // 32, dd % 32
    j, pos = _pair(kt)
    nib = np.full(kt.shape, -1)
    if not is_v:
        if kv_type == "q8_0":
            off = b * 512 + (4 * n + (dd % 16) // 4) * 16 + (2 * st + i // 16) * 4 + dd % 4
        elif kv_type in NIBBLE:
            off = (b // 2) * 512 + (4 * n + (i % 16) // 4) * 16 + (2 * (b % 2) + st) * 4 + (i % 16) % 4
            nib = (i >= 16).astype(int)
        else:
            P = np.array([0, 2, 1, 3])[dd % 4]
            off = (2 * b + st) * 512 + (4 * n + (dd % 16) // 4) * 16 + (i // 16) * 8 + P * 2
    else:
        r, hv = i % 16, i // 16
        n2 = r // 2
        if kv_type == "q8_0":
            off = b * 512 + (4 * n2 + j) * 16 + ((r % 2) + 2 * hv) * 4 + _q_of_pos(pos)
        elif kv_type in NIBBLE:
            off = (b // 2) * 512 + (4 * n2 + j) * 16 + (2 * (b % 2) + r % 2) * 4 + _q_of_pos(pos)
            nib = (i >= 16).astype(int)
        else:
            off = (2 * b + hv) * 512 + (4 * n2 + j) * 16 + (r % 2) * 8 + pos * 2
    return off, nib


def scale_offsets():
    """off[16, 4]: byte offset of the f16 scale of (row kt, block b) inside one (tile, slice)."""
    kt, b = np.meshgrid(np.arange(16), np.arange(4), indexing="ij")
    j, pos = _pair(kt)
    return j * 32 + b * 8 + pos * 2


def decode_plane(codes_plane: np.ndarray, scales_plane: np.ndarray, kv_type: str, is_v: bool,
                 B: int, Hkv: int, cap: int, D: int):
    """Raw plane bytes -> (codes, scales) in the oracle's natural layout:
    codes [B, Hkv, cap, row] (f16 bits uint16 / int8 / packed uint8), scales uint16 [B, Hkv, cap, D/32]."""
    NS = D // 128
    T = cap // 16
    ct = CODE_TILE[kv_type]
    raw = np.asarray(codes_plane, dtype=np.uint8).reshape(B, Hkv, T, NS, ct)
    off, nib = tile_offsets(kv_type, is_v)
    if kv_type == "f16":
        lo = raw[..., off]          # [B,Hkv,T,NS,16,128]
        hi = raw[..., off + 1]
        vals = lo.astype(np.uint16) | (hi.astype(np.uint16) << 8)
        codes = vals.transpose(0, 1, 2, 4, 3, 5).reshape(B, Hkv, cap, D)
        scales = np.zeros((B, Hkv, cap, 0), np.uint16)
        return codes, scales
    byte = raw[..., off]
    if kv_type == "q8_0":
        # stored as a sign-magnitude byte
        mag = (byte & np.uint8(0x7F)).astype(np.int16)
        q = np.where(byte & np.uint8(0x80), -mag, mag).astype(np.int8)
        codes = q.transpose(0, 1, 2, 4, 3, 5).reshape(B, Hkv, cap, D)
    else:
        c = np.where(nib == 1, byte >> 4, byte & 0x0F).astype(np.uint8)   # [B,Hkv,T,NS,16,128]
        if kv_type in ("q5_0", "q5_1"):
            # fifth bits: 32-bit word of lane L = (off % 512) // 16 in the plane after the
            # nibbles (128 B per 512-B chunk); bit 8e + 4 + wi (low nibble) or 8e + wi (high
            # nibble), e = byte of the nibble word, wi = word of the lane
            lane = (off % 512) // 16
            wi, e = (off % 16) // 4, off % 4
            woff = 1024 + (off // 512) * 128 + lane * 4
            words = (raw[..., woff].astype(np.uint32) | (raw[..., woff + 1].astype(np.uint32) << 8) |
                     (raw[..., woff + 2].astype(np.uint32) << 16) | (raw[..., woff + 3].astype(np.uint32) << 24))
            bit = np.where(nib == 1, 8 * e + wi, 8 * e + 4 + wi)
            c = (c | (((words >> bit.astype(np.uint32)) & 1) << 4)).astype(np.uint8)
        c = c.transpose(0, 1, 2, 4, 3, 5).reshape(B, Hkv, cap, D // 32, 32)
        if kv_type == "q4_0":
            codes = (c[..., :16] | (c[..., 16:] << 4)).astype(np.uint8).reshape(B, Hkv, cap, D // 2)
        else:
            codes = c.reshape(B, Hkv, cap, D)
    sraw = np.asarray(scales_plane, dtype=np.uint8).reshape(B, Hkv, T, NS, SCALE_TILE[kv_type])
    so = scale_offsets()
    s = sraw[..., so].astype(np.uint16) | (sraw[..., so + 1].astype(np.uint16) << 8)  # [B,Hkv,T,NS,16,4]
    scales = s.transpose(0, 1, 2, 4, 3, 5).reshape(B, Hkv, cap, D // 32)
    if kv_type in ("q4_1", "q5_1"):  # lo after d, interleaved as (d, lo) per block
        s2 = sraw[..., so + 128].astype(np.uint16) | (sraw[..., so + 129].astype(np.uint16) << 8)
        lo = s2.transpose(0, 1, 2, 4, 3, 5).reshape(B, Hkv, cap, D // 32)
        scales = np.stack([scales, lo], -1).reshape(B, Hkv, cap, D // 16)
    return codes, scales


def check_bijective():
    """Every layout maps the 16x128 (row, value) slots onto distinct bytes/nibbles."""
    for t in ("f16", "q8_0", "q4_0", "q4_1", "q5_0", "q5_1"):
        for is_v in (False, True):
            off, nib = tile_offsets(t, is_v)
            if t == "f16":
                keys = np.concatenate([off.ravel(), off.ravel() + 1])
                assert len(set(keys.tolist())) == 2 * 16 * 128 and keys.max() < CODE_TILE[t]
            elif t == "q8_0":
                assert len(set(off.ravel().tolist())) == 16 * 128 and off.max() < CODE_TILE[t]
            else:
                keys = off.ravel() * 2 + nib.ravel()
                assert len(set(keys.tolist())) == 16 * 128 and off.max() < 1024
                if t in ("q5_0", "q5_1"):  # fifth-bit (word, bit) places are distinct too
                    woff = 1024 + (off // 512) * 128 + ((off % 512) // 16) * 4
                    bit = np.where(nib == 1, 8 * (off % 4) + (off % 16) // 4, 8 * (off % 4) + 4 + (off % 16) // 4)
                    fb = (woff * 32 + bit).ravel()
                    assert len(set(fb.tolist())) == 16 * 128 and woff.max() + 4 <= CODE_TILE[t]
    so = scale_offsets()
    assert len(set(so.ravel().tolist())) == 64 and so.max() < 128
