"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

* Quantised codes and f16 scales: bit-exact, read back through the layout documented in
  include/kvq.h (tests/kvq_layout.py).
* Attention outputs: max abs error <= 1e-3 (fp32 out) against the fp64 oracle, which
  quantises the same fp32 rows itself.  lse is checked to the same tolerance.
All inputs are seeded; the oracle never sees a value produced by the CUDA path.
"""
import math
import zlib

import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from tests import kvq_layout

pytestmark = pytest.mark.gpu

TOL = 1e-3
PAIRS = [("q8_0", "q8_0"), ("q8_0", "q4_0"), ("q4_0", "q4_0"), ("f16", "f16"),
         ("f16", "q4_0"), ("q4_0", "q8_0"), ("q8_0", "f16"), ("q4_0", "f16"), ("f16", "q8_0")]


@pytest.fixture(scope="module")
def kvq():
    import quantised_kv_long_gb300 as m
    return m


def host_planes(cache):
    kc, ks, vc, vs = (t.cpu().numpy() for t in cache.planes())
    return kc, ks, vc, vs


def read_natural(cache):
    """(k_codes, k_scales, v_codes, v_scales) of the whole cache in natural layout."""
    kc, ks, vc, vs = host_planes(cache)
    B, H, cap, D = cache.batch, cache.n_kv_heads, cache.capacity, cache.head_dim
    k = kvq_layout.decode_plane(kc, ks, cache.type_k, False, B, H, cap, D)
    v = kvq_layout.decode_plane(vc, vs, cache.type_v, True, B, H, cap, D)
    return k + v


def crafted_rows(n, D, rng):
    """Rows that hit the quantisers' corner cases, block by block."""
    x = rng.standard_normal((n, D)).astype(np.float32)
    blocks = x.reshape(n, D // 32, 32)
    for r in range(n):
        for b in range(D // 32):
            kind = (r * 7 + b) % 10
            blk = blocks[r, b]
            if kind == 0:
                blk[:] = 0.0                                   # zero block
            elif kind == 1:
                blk[:] = 0.0
                blk[5] = -3.0                                  # single value
            elif kind == 2:
                blk[:] = np.arange(32) - 16.0
                blk[0] = 127.0                                 # d = 1: exact codes
                blk[1:6] = [2.5, -2.5, 0.5, -0.5, 0.49999997]  # halves and a just-below-half
            elif kind == 3:
                blk[:] = 1e-7 * rng.standard_normal(32)        # f16-subnormal scale
            elif kind == 4:
                blk[:] = 0.0
                blk[3], blk[7] = 2.0, -2.0                     # q4 tie: first index wins, clip
            elif kind == 5:
                blk[:] = 0.375                                 # all equal
            elif kind == 6:
                blk[:] = rng.standard_normal(32) * 3e4         # large values
            elif kind == 7:
                blk[0], blk[1] = 1.0, -0.999                   # q4 clip case
    return x


@pytest.mark.parametrize("tk,tv", [("q8_0", "q4_0"), ("f16", "q8_0"), ("q4_0", "f16")])
@pytest.mark.parametrize("start", [0, 1, 7, 15])
def test_bulk_append_tile_edges(kvq, tk, tv, start):
    """Appends of 16 rows or more (assembled tile by tile) starting at every kind of offset
    inside a tile, with lengths that end anywhere in a tile: the codes of the whole prefix
    stay bit-exact (rows written before are kept) and lengths advance."""
    H, D = 2, 128
    rng = np.random.default_rng(start * 7 + len(tk))
    cache = kvq.KVCache(1, H, D, 16 * 24, tk, tv)
    chunks = [start, 16, 17, 31, 32, 47, 1, 63]
    K = crafted_rows(H * sum(chunks), D, rng).reshape(H, sum(chunks), D)
    V = crafted_rows(H * sum(chunks), D, rng).reshape(H, sum(chunks), D)
    t = 0
    for n in chunks:
        if n:
            cache.append(torch.from_numpy(K[None, :, t:t + n].copy()).cuda(),
                         torch.from_numpy(V[None, :, t:t + n].copy()).cuda())
        t += n
    torch.cuda.synchronize()
    assert cache.sync_lengths() == [t] and cache.read_error() == 0
    kc, ksc, vc, vsc = read_natural(cache)
    ok_c, ok_s = oracle.quantize(tk, K)
    ov_c, ov_s = oracle.quantize(tv, V)
    assert np.array_equal(kc[0, :, :t], ok_c) and np.array_equal(ksc[0, :, :t], ok_s)
    assert np.array_equal(vc[0, :, :t], ov_c) and np.array_equal(vsc[0, :, :t], ov_s)


@pytest.mark.parametrize("tk,tv", PAIRS)
@pytest.mark.parametrize("D", [128, 256])
def test_append_codes_bit_exact(kvq, tk, tv, D):
    B, H, cap = 3, 2, 96
    rng = np.random.default_rng(zlib.crc32(f"{tk}-{tv}-{D}".encode()))
    cache = kvq.KVCache(B, H, D, cap, tk, tv)
    rows = {b: [] for b in range(B)}
    # ragged appends that start and end inside tiles, one call covering several sequences
    for b0, nb, n_new in [(0, 3, 5), (1, 1, 1), (0, 2, 16), (2, 1, 20), (0, 3, 11), (1, 2, 33)]:
        kx = crafted_rows(nb * H * n_new, D, rng).reshape(nb, H, n_new, D)
        vx = crafted_rows(nb * H * n_new, D, rng).reshape(nb, H, n_new, D)
        cache.append(torch.from_numpy(kx).cuda(), torch.from_numpy(vx).cuda(), b0=b0)
        for i in range(nb):
            rows[b0 + i].append((kx[i], vx[i]))
    torch.cuda.synchronize()
    lens = cache.sync_lengths()
    assert lens == [sum(r[0].shape[1] for r in rows[b]) for b in range(B)]
    assert cache.read_error() == 0
    kc, ksc, vc, vsc = read_natural(cache)
    for b in range(B):
        K = np.concatenate([r[0] for r in rows[b]], axis=1)   # [H, len, D]
        V = np.concatenate([r[1] for r in rows[b]], axis=1)
        n = K.shape[1]
        ok_c, ok_s = oracle.quantize(tk, K)
        ov_c, ov_s = oracle.quantize(tv, V)
        assert np.array_equal(kc[b, :, :n], ok_c), f"K codes differ (b={b})"
        assert np.array_equal(ksc[b, :, :n], ok_s), f"K scales differ (b={b})"
        assert np.array_equal(vc[b, :, :n], ov_c), f"V codes differ (b={b})"
        assert np.array_equal(vsc[b, :, :n], ov_s), f"V scales differ (b={b})"


def run_case(kvq, tk, tv, D, Hkv, G, lens, cap, n_splits, seed=0, scale=None, append_chunks=(None,)):
    """Fill a cache from seeded rows, decode, and compare with the oracle."""
    B = len(lens)
    Hq = Hkv * G
    wl = syn.Workload("case", 1, B, Hq, Hkv, D, tk, tv, tuple(lens), outliers=4, seed=seed)
    cache = kvq.KVCache(B, Hkv, D, cap, tk, tv)
    Ks, Vs = [], []
    for b in range(B):
        K = torch.stack([syn.kv_rows(wl, syn.KIND_K, 0, b, h, 0, lens[b]) for h in range(Hkv)])
        V = torch.stack([syn.kv_rows(wl, syn.KIND_V, 0, b, h, 0, lens[b]) for h in range(Hkv)])
        Ks.append(K)
        Vs.append(V)
        # append in a few ragged pieces
        t = 0
        step = max(1, lens[b] // 3 + 7)
        while t < lens[b]:
            n = min(step, lens[b] - t)
            cache.append(K[None, :, t:t + n].contiguous(), V[None, :, t:t + n].contiguous(), b0=b)
            t += n
    q = syn.queries(wl, 0)
    scale = wl.scale if scale is None else scale
    out, lse = cache.decode(q, scale=scale, n_splits=n_splits)
    torch.cuda.synchronize()
    assert cache.read_error() == 0
    out, lse, qh = out.cpu().numpy(), lse.cpu().numpy(), q.cpu().numpy()
    worst = 0.0
    for b in range(B):
        kc, ks = oracle.quantize(tk, Ks[b].cpu().numpy())
        vc, vs = oracle.quantize(tv, Vs[b].cpu().numpy())
        ref, ref_lse = oracle.attention(tk, kc, ks, tv, vc, vs, lens[b], qh[b], scale, n_threads=0)
        err = np.abs(out[b] - ref).max()
        worst = max(worst, err)
        assert err <= TOL, f"b={b} max abs err {err}"
        if lens[b] == 0:
            assert np.isneginf(lse[b]).all() and (out[b] == 0).all()
        else:
            assert np.abs(lse[b] - ref_lse).max() <= TOL
    return worst


def test_tiny_config(kvq):
    """1 layer, batch 1, ctx 512, Hkv 2, Hq 4, D 128, q8_0 K and V; all 512 rows quantised, one decode."""
    wl = syn.tiny()
    cache = kvq.KVCache(1, 2, 128, 512, "q8_0", "q8_0")
    K = syn.layer_kv(wl, 0, syn.KIND_K, 512)
    V = syn.layer_kv(wl, 0, syn.KIND_V, 512)
    cache.append(K, V)
    q = syn.queries(wl, 0)
    out, lse = cache.decode(q, scale=wl.scale)
    torch.cuda.synchronize()
    kc, ks = oracle.quantize("q8_0", K[0].cpu().numpy())
    vc, vs = oracle.quantize("q8_0", V[0].cpu().numpy())
    gk, gks, gv, gvs = read_natural(cache)
    assert np.array_equal(gk[0], kc) and np.array_equal(gks[0], ks)
    assert np.array_equal(gv[0], vc) and np.array_equal(gvs[0], vs)
    ref, ref_lse = oracle.attention("q8_0", kc, ks, "q8_0", vc, vs, 512, q[0].cpu().numpy(), wl.scale)
    assert np.abs(out[0].cpu().numpy() - ref).max() <= TOL
    assert np.abs(lse[0].cpu().numpy() - ref_lse).max() <= TOL


@pytest.mark.parametrize("tk,tv", PAIRS)
@pytest.mark.parametrize("D,G", [(128, 5), (256, 8), (128, 1), (256, 2)])
def test_decode_pairs(kvq, tk, tv, D, G):
    run_case(kvq, tk, tv, D, Hkv=2, G=G, lens=[700], cap=768, n_splits=0, seed=G + D)


@pytest.mark.parametrize("n_splits", [1, 2, 3, 0, 64, 1024])
@pytest.mark.parametrize("lens", [[1], [15], [16], [17], [511], [2049], [0], [33, 0, 300, 1]])
def test_decode_lengths_and_splits(kvq, lens, n_splits):
    run_case(kvq, "q8_0", "q4_0", 128, Hkv=2, G=4, lens=lens, cap=2064, n_splits=n_splits, seed=len(lens))


@pytest.mark.parametrize("tk,tv", [("q8_0", "q8_0"), ("q4_0", "q4_0"), ("q8_0", "q4_0")])
@pytest.mark.parametrize("n_splits", [4, 7, 13])
def test_decode_d256_split_tile_counts(kvq, tk, tv, n_splits):
    """Head dim 256 (two slice-warps per tile pair) with 33, 19 and 10 tiles per split: the
    last stage of a split is partial, sometimes with an odd tile count, so the second tile
    of a pair lies in a ring slot that holds stale or never-written bytes."""
    run_case(kvq, tk, tv, 256, Hkv=2, G=8, lens=[2049], cap=2064, n_splits=n_splits, seed=n_splits)


@pytest.mark.parametrize("tk,tv", [("q8_0", "q8_0"), ("q4_0", "q4_0"), ("q8_0", "q4_0"), ("q5_1", "q5_1")])
@pytest.mark.parametrize("big_slice", [0, 1])
def test_decode_large_v_scales_in_one_slice(kvq, tk, tv, big_slice):
    """V blocks with |scale| >= 256 in one 128-value half of a 256-wide head only (every
    other tile).  The f16 overflow guard then fires for one slice-warp of each tile pair and
    not the other; both must still move their running maximum together, or the merge
    combines accumulators taken against different maxima."""
    B, H, G, D, L = 1, 2, 8, 256, 700
    wl = syn.Workload("bigv", 1, B, H * G, H, D, tk, tv, (L,), seed=31 + big_slice)
    cache = kvq.KVCache(B, H, D, 704, tk, tv)
    K = torch.stack([syn.kv_rows(wl, syn.KIND_K, 0, 0, h, 0, L) for h in range(H)])
    V = torch.stack([syn.kv_rows(wl, syn.KIND_V, 0, 0, h, 0, L) for h in range(H)])
    # scale d = amax / 127 (q8_0) or amax / 8 (4- and 5-bit types) reaches 256 and more
    factor = 1.0e4 if tv == "q8_0" else 2.0e3
    big = torch.zeros(L, dtype=torch.bool, device=V.device)
    big[(torch.arange(L, device=V.device) // 16) % 2 == 1] = True
    lo, hi = big_slice * 128, big_slice * 128 + 128
    V[:, big, lo:hi] *= factor
    cache.append(K[None].contiguous(), V[None].contiguous())
    q = syn.queries(wl, 0)
    out, lse = cache.decode(q, scale=wl.scale, n_splits=2)
    torch.cuda.synchronize()
    assert cache.read_error() == 0
    kc, ks = oracle.quantize(tk, K.cpu().numpy())
    vc, vs = oracle.quantize(tv, V.cpu().numpy())
    spb = oracle.scales_per_block(tv)
    d = vs.view(np.float16).astype(np.float64)[..., ::spb]  # the block scales d (not the minima)
    assert np.abs(d[:, :, lo // 32:hi // 32]).max() >= 256  # the guard's threshold is reached
    assert np.abs(d[:, :, (128 - lo) // 32:(256 - lo) // 32]).max() < 256
    ref, ref_lse = oracle.attention(tk, kc, ks, tv, vc, vs, L, q[0].cpu().numpy(), wl.scale)
    o = out[0].cpu().numpy()
    other = slice(128 - lo, 256 - lo) if big_slice == 0 else slice(0, 128)
    assert np.abs(o[:, other] - ref[:, other]).max() <= TOL
    # the large half: f32 accumulation of values up to about 4 x factor
    assert np.abs(o[:, lo:hi] - ref[:, lo:hi]).max() <= TOL + 1e-5 * factor
    assert np.abs(lse[0].cpu().numpy() - ref_lse).max() <= TOL


@pytest.mark.parametrize("G", [9, 16, 12])
def test_decode_wide_groups(kvq, G):
    """More than 8 query heads per KV head: several row groups per KV head."""
    run_case(kvq, "q4_0", "q4_0", 128, Hkv=2, G=G, lens=[257, 40], cap=272, n_splits=0, seed=G)


def test_decode_capacity_full(kvq):
    run_case(kvq, "q8_0", "q8_0", 256, Hkv=1, G=8, lens=[4096], cap=4096, n_splits=0, seed=5)


def test_decode_concentrated_attention(kvq):
    """One dominant key (scores far apart): exercises the f16 hi+lo split of P and Q."""
    for scale in (1.0, 4.0):
        run_case(kvq, "q8_0", "q4_0", 128, Hkv=2, G=5, lens=[1000], cap=1008, n_splits=0, seed=9, scale=scale)


def test_decode_identical_keys_mean_of_v(kvq):
    """All keys equal -> the output is the mean of the dequantised V rows."""
    B, H, D, n = 1, 2, 128, 333
    cache = kvq.KVCache(B, H, D, 336, "q4_0", "q8_0")
    rng = np.random.default_rng(3)
    K = np.broadcast_to(rng.standard_normal((1, H, 1, D)), (1, H, n, D)).astype(np.float32).copy()
    V = rng.standard_normal((1, H, n, D)).astype(np.float32)
    cache.append(torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda())
    q = torch.from_numpy(rng.standard_normal((1, 2 * H, D)).astype(np.float32)).cuda()
    out, _ = cache.decode(q)
    vc, vs = oracle.quantize("q8_0", V[0])
    mean = oracle.dequantize("q8_0", vc, vs, D).mean(axis=1)   # [H, D]
    o = out[0].cpu().numpy()
    for hq in range(2 * H):
        assert np.abs(o[hq] - mean[hq // 2]).max() <= 1e-5


@pytest.mark.parametrize("tk,tv", [("q8_0", "q4_0"), ("f16", "f16"), ("q4_0", "q4_0")])
def test_partials_and_combine(kvq, tk, tv):
    """kvq_decode_partials equals the oracle's split triples over the documented ranges,
    and kvq_combine of them equals the unsplit attention."""
    B, H, D, G, S = 2, 2, 128, 3, 5
    lens = [203, 64]
    wl = syn.Workload("p", 1, B, H * G, H, D, tk, tv, tuple(lens), seed=17)
    cache = kvq.KVCache(B, H, D, 208, tk, tv)
    Ks = [torch.stack([syn.kv_rows(wl, syn.KIND_K, 0, b, h, 0, lens[b]) for h in range(H)]) for b in range(B)]
    Vs = [torch.stack([syn.kv_rows(wl, syn.KIND_V, 0, b, h, 0, lens[b]) for h in range(H)]) for b in range(B)]
    for b in range(B):
        cache.append(Ks[b][None].contiguous(), Vs[b][None].contiguous(), b0=b)
    q = syn.queries(wl, 0)
    po, pm, pl = cache.decode_partials(q, S, scale=wl.scale)
    out, lse = kvq.combine(po, pm, pl)
    torch.cuda.synchronize()
    po, pm, pl = po.cpu().numpy(), pm.cpu().numpy(), pl.cpu().numpy()
    qh = q.cpu().numpy()
    for b in range(B):
        T = (lens[b] + 15) // 16
        ns = max(1, min(S, T))
        c = (T + ns - 1) // ns
        bounds = [min(lens[b], min(T, s * c) * 16) for s in range(S + 1)]
        kc, ks = oracle.quantize(tk, Ks[b].cpu().numpy())
        vc, vs = oracle.quantize(tv, Vs[b].cpu().numpy())
        o_ref, m_ref, l_ref = oracle.attention_partials(tk, kc, ks, tv, vc, vs, bounds, qh[b], wl.scale)
        for hq in range(H * G):
            for s in range(S):
                if np.isneginf(m_ref[hq, s]):
                    assert np.isneginf(pm[b, hq, s]) and pl[b, hq, s] == 0 and (po[b, hq, s] == 0).all()
                    continue
                assert abs(pm[b, hq, s] - m_ref[hq, s]) <= 1e-4
                assert abs(pl[b, hq, s] - l_ref[hq, s]) <= 1e-4 * max(1.0, l_ref[hq, s])
                assert np.abs(po[b, hq, s] - o_ref[hq, s]).max() <= TOL * max(1.0, l_ref[hq, s])
        ref, ref_lse = oracle.attention(tk, kc, ks, tv, vc, vs, lens[b], qh[b], wl.scale)
        assert np.abs(out[b].cpu().numpy() - ref).max() <= TOL
        assert np.abs(lse[b].cpu().numpy() - ref_lse).max() <= TOL


def test_combine_against_oracle(kvq):
    rng = np.random.default_rng(2)
    R, S, D = 37, 19, 128
    po = rng.standard_normal((R, S, D))
    pm = rng.standard_normal((R, S)) * 5
    pl = rng.uniform(0.5, 20, (R, S))
    pm[3, :] = -np.inf
    pl[3, :] = 0
    po[3] = 0
    pm[5, 4:9] = -np.inf
    pl[5, 4:9] = 0
    po[5, 4:9] = 0
    out, lse = kvq.combine(*(torch.tensor(a, dtype=torch.float32).cuda() for a in (po, pm, pl)))
    ref, ref_lse = oracle.combine(po.astype(np.float32), pm.astype(np.float32), pl.astype(np.float32))
    assert np.abs(out.cpu().numpy() - ref).max() <= 1e-5
    o = lse.cpu().numpy()
    assert np.isneginf(o[3]) and np.isneginf(ref_lse[3])
    fin = np.isfinite(ref_lse)
    assert np.abs(o[fin] - ref_lse[fin]).max() <= 1e-5


def test_graph_capture_append_then_decode(kvq):
    """Append (advancing len on the device) + decode captured once, replayed three times."""
    H, D, G = 2, 128, 4
    wl = syn.Workload("g", 1, 1, H * G, H, D, "q8_0", "q4_0", (100,), seed=4)
    cache = kvq.KVCache(1, H, D, 128, "q8_0", "q4_0")
    K = torch.stack([syn.kv_rows(wl, syn.KIND_K, 0, 0, h, 0, 103) for h in range(H)])[None].contiguous()
    V = torch.stack([syn.kv_rows(wl, syn.KIND_V, 0, 0, h, 0, 103) for h in range(H)])[None].contiguous()
    cache.append(K[:, :, :100].contiguous(), V[:, :, :100].contiguous())
    q = syn.queries(wl, 0)
    knew = torch.empty((1, H, 1, D), device="cuda")
    vnew = torch.empty((1, H, 1, D), device="cuda")
    n_splits = cache.auto_splits(H * G)
    ws = cache.workspace(H * G, n_splits)
    out = torch.empty_like(q)
    lse = torch.empty((1, H * G), device="cuda")
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        cache.append(knew, vnew, stream=s)
        cache.decode(q, n_splits=n_splits, out=out, lse=lse, workspace=ws, stream=s)
    torch.cuda.synchronize()
    # the capture itself enqueued nothing: length still 100 on the device
    assert cache.sync_lengths() == [100]
    qh = q.cpu().numpy()
    for step in range(3):
        knew.copy_(K[:, :, 100 + step:101 + step])
        vnew.copy_(V[:, :, 100 + step:101 + step])
        g.replay()
        torch.cuda.synchronize()
        n = 101 + step
        assert cache.sync_lengths() == [n]
        kc, ks = oracle.quantize("q8_0", K[0, :, :n].cpu().numpy())
        vc, vs = oracle.quantize("q4_0", V[0, :, :n].cpu().numpy())
        ref, _ = oracle.attention("q8_0", kc, ks, "q4_0", vc, vs, n, qh[0], wl.scale)
        assert np.abs(out[0].cpu().numpy() - ref).max() <= TOL


def test_error_paths(kvq):
    cache = kvq.KVCache(2, 2, 128, 32, "q8_0", "q8_0")
    x = torch.zeros((1, 2, 33, 128), device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        cache.append(x, x)                       # 33 rows > capacity 32
    assert e.value.status == 3
    assert cache.sync_lengths() == [0, 0]        # nothing written
    x = torch.zeros((1, 2, 20, 128), device="cuda")
    cache.append(x, x, b0=1)
    with pytest.raises(kvq.KvqError) as e:
        cache.append(x, x, b0=1)                 # 40 > 32
    assert e.value.status == 3
    assert cache.sync_lengths() == [0, 20]
    with pytest.raises(kvq.KvqError) as e:
        cache.append(x, x, b0=2)                 # sequence out of range
    assert e.value.status == 1
    q = torch.zeros((2, 6, 128), device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        cache.decode(q[:, :5].contiguous())      # Hq not a multiple of Hkv
    assert e.value.status == 1
    buf = torch.zeros(2 * 6 * 128 + 1, device="cuda")
    qmis = buf[1:].view(2, 6, 128)               # 4-byte aligned, not 16
    with pytest.raises(kvq.KvqError) as e:
        cache.decode(qmis)
    assert e.value.status == 4
    # a device-side capacity overflow (lengths changed behind the host mirror)
    cache.state[1] = 30
    cache.append(x[:, :, :5].contiguous(), x[:, :, :5].contiguous(), b0=1)  # mirror says 20 + 5 <= 32
    torch.cuda.synchronize()
    assert cache.read_error() == kvq.DEVERR_CAPACITY
    assert cache.sync_lengths() == [0, 30]       # the device refused to advance
    assert cache.read_error() == 0


@pytest.mark.parametrize("which", ["hybrid-64K-q8", "hybrid-64K-f16", "dense-131072-q8q4", "long-262144-q4q4",
                                   "long-262144-q8q8", "multi-session"])
def test_full_size_sampled(kvq, which):
    """One layer at the benchmark's full sizes and launch configuration (auto splits),
    checked on sampled query heads against the oracle."""
    if which.startswith("hybrid"):
        wl = syn.hybrid(65536, *(("q8_0", "q8_0") if which.endswith("q8") else ("f16", "f16")))
    elif which.startswith("dense"):
        wl = syn.dense14b(131072, "q8_0", "q4_0")
    elif which == "long-262144-q4q4":
        wl = syn.dense14b(262144, "q4_0", "q4_0")
    elif which == "long-262144-q8q8":
        wl = syn.dense14b(262144, "q8_0", "q8_0")
    else:
        wl = syn.multi_session()
    layer = 3 if wl.layers > 3 else 0
    cap = (max(wl.lengths) + 16 + 15) // 16 * 16
    cache = kvq.KVCache(wl.batch, wl.n_kv_heads, wl.head_dim, cap, wl.type_k, wl.type_v)
    for b in range(wl.batch):
        K = torch.stack([syn.kv_rows(wl, syn.KIND_K, layer, b, h, 0, wl.lengths[b]) for h in range(wl.n_kv_heads)])
        V = torch.stack([syn.kv_rows(wl, syn.KIND_V, layer, b, h, 0, wl.lengths[b]) for h in range(wl.n_kv_heads)])
        cache.append(K[None], V[None], b0=b)
        del K, V
    q = syn.queries(wl, layer)
    out, lse = cache.decode(q, scale=wl.scale)
    torch.cuda.synchronize()
    assert cache.read_error() == 0
    rng = np.random.default_rng(len(which))
    samples = [(int(rng.integers(wl.batch)), int(rng.integers(wl.n_q_heads))) for _ in range(3)]
    qh = q.cpu().numpy()
    for b, hq in samples:
        h = hq // wl.G
        n = wl.lengths[b]
        K = syn.kv_rows(wl, syn.KIND_K, layer, b, h, 0, n).cpu().numpy()[None]
        V = syn.kv_rows(wl, syn.KIND_V, layer, b, h, 0, n).cpu().numpy()[None]
        kc, ks = oracle.quantize(wl.type_k, K, n_threads=0)
        vc, vs = oracle.quantize(wl.type_v, V, n_threads=0)
        ref, ref_lse = oracle.attention(wl.type_k, kc, ks, wl.type_v, vc, vs, n, qh[b, hq:hq + 1], wl.scale)
        err = np.abs(out[b, hq].cpu().numpy() - ref[0]).max()
        assert err <= TOL, (b, hq, err)
        assert abs(float(lse[b, hq]) - ref_lse[0]) <= TOL


@pytest.mark.parametrize("tk,tv", [("q8_0", "q8_0"), ("q8_0", "q4_0"), ("q4_0", "q4_0"), ("f16", "f16"), ("f16", "q4_0")])
@pytest.mark.parametrize("D,G", [(128, 5), (256, 8), (128, 12)])
def test_append_decode_fused_steps(kvq, tk, tv, D, G):
    """kvq_append_decode: one launch appends one row per sequence and attends over it.
    Codes of every row (old and appended) are bit-exact; outputs match the oracle."""
    H = 2
    lens = [300, 17, 48]
    B = len(lens)
    wl = syn.Workload("fused", 1, B, H * G, H, D, tk, tv, tuple(lens), seed=G + D)
    steps = 3
    cap = 320
    cache = kvq.KVCache(B, H, D, cap, tk, tv)
    Ks = [torch.stack([syn.kv_rows(wl, syn.KIND_K, 0, b, h, 0, lens[b] + steps) for h in range(H)]) for b in range(B)]
    Vs = [torch.stack([syn.kv_rows(wl, syn.KIND_V, 0, b, h, 0, lens[b] + steps) for h in range(H)]) for b in range(B)]
    for b in range(B):
        cache.append(Ks[b][None, :, :lens[b]].contiguous(), Vs[b][None, :, :lens[b]].contiguous(), b0=b)
    for step in range(steps):
        kn = torch.stack([Ks[b][:, lens[b] + step] for b in range(B)])[:, :, None].contiguous()
        vn = torch.stack([Vs[b][:, lens[b] + step] for b in range(B)])[:, :, None].contiguous()
        q = syn.queries(wl, 0, step=step)
        out, lse = cache.append_decode(kn, vn, q, scale=wl.scale)
        torch.cuda.synchronize()
        assert cache.lengths() == [n + step + 1 for n in lens]
        qh = q.cpu().numpy()
        for b in range(B):
            n = lens[b] + step + 1
            kc, ks = oracle.quantize(tk, Ks[b][:, :n].cpu().numpy())
            vc, vs = oracle.quantize(tv, Vs[b][:, :n].cpu().numpy())
            ref, ref_lse = oracle.attention(tk, kc, ks, tv, vc, vs, n, qh[b], wl.scale)
            assert np.abs(out[b].cpu().numpy() - ref).max() <= TOL, (step, b)
            assert np.abs(lse[b].cpu().numpy() - ref_lse).max() <= TOL
    assert cache.sync_lengths() == [n + steps for n in lens]
    assert cache.read_error() == 0
    kc, ksc, vc, vsc = read_natural(cache)
    for b in range(B):
        n = lens[b] + steps
        ok_c, ok_s = oracle.quantize(tk, Ks[b][:, :n].cpu().numpy())
        ov_c, ov_s = oracle.quantize(tv, Vs[b][:, :n].cpu().numpy())
        assert np.array_equal(kc[b, :, :n], ok_c) and np.array_equal(ksc[b, :, :n], ok_s)
        assert np.array_equal(vc[b, :, :n], ov_c) and np.array_equal(vsc[b, :, :n], ov_s)


def test_append_decode_capacity(kvq):
    H, D, G = 2, 128, 4
    cache = kvq.KVCache(2, H, D, 32, "q8_0", "q4_0")
    x = torch.randn((1, H, 32, D), device="cuda")
    cache.append(x, x, b0=0)                               # sequence 0 is full
    cache.append(x[:, :, :5].contiguous(), x[:, :, :5].contiguous(), b0=1)
    kn = torch.randn((2, H, 1, D), device="cuda")
    q = torch.randn((2, H * G, D), device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        cache.append_decode(kn, kn, q)
    assert e.value.status == 3
    assert cache.sync_lengths() == [32, 5]
    # full only on the device: that sequence is attended without the new row and not advanced
    cache.state[0] = 31
    cache.sync_lengths()
    cache.state[0] = 32
    out, _ = cache.append_decode(kn, kn, q)
    torch.cuda.synchronize()
    assert cache.read_error() == kvq.DEVERR_CAPACITY
    assert cache.sync_lengths() == [32, 6]


def test_append_decode_graph_replay(kvq):
    H, D, G = 2, 256, 8
    wl = syn.Workload("gf", 1, 1, H * G, H, D, "q8_0", "q8_0", (200,), seed=8)
    cache = kvq.KVCache(1, H, D, 224, "q8_0", "q8_0")
    K = torch.stack([syn.kv_rows(wl, syn.KIND_K, 0, 0, h, 0, 204) for h in range(H)])[None].contiguous()
    V = torch.stack([syn.kv_rows(wl, syn.KIND_V, 0, 0, h, 0, 204) for h in range(H)])[None].contiguous()
    cache.append(K[:, :, :200].contiguous(), V[:, :, :200].contiguous())
    q = syn.queries(wl, 0)
    kn = torch.empty((1, H, 1, D), device="cuda")
    vn = torch.empty((1, H, 1, D), device="cuda")
    S = cache.auto_splits(H * G)
    ws = cache.workspace(H * G, S)
    out = torch.empty_like(q)
    lse = torch.empty((1, H * G), device="cuda")
    st = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        cache.append_decode(kn, vn, q, n_splits=S, out=out, lse=lse, workspace=ws, stream=st)
    torch.cuda.synchronize()
    assert cache.sync_lengths() == [200]
    qh = q.cpu().numpy()
    for step in range(4):
        kn.copy_(K[:, :, 200 + step:201 + step])
        vn.copy_(V[:, :, 200 + step:201 + step])
        g.replay()
        torch.cuda.synchronize()
        n = 201 + step
        assert cache.sync_lengths() == [n]
        kc, ks = oracle.quantize("q8_0", K[0, :, :n].cpu().numpy())
        vc, vs = oracle.quantize("q8_0", V[0, :, :n].cpu().numpy())
        ref, _ = oracle.attention("q8_0", kc, ks, "q8_0", vc, vs, n, qh[0], wl.scale)
        assert np.abs(out[0].cpu().numpy() - ref).max() <= TOL


@pytest.mark.parametrize("order", ["layers", "same_cache", "mixed"])
def test_back_to_back_launches_without_sync(kvq, order):
    """Launches queued back to back with no synchronisation in between, as a model's decode
    step issues them.  A decode launch may start while the previous kernel of the stream is
    still running and then reads its cache's lengths and tiles early unless that kernel
    wrote the cache; these orders cover both cases (other caches before it, the same cache
    before it, a bulk append of the same cache just before it, a plain decode between)."""
    H, D, G, tk, tv = 2, 128, 5, "q8_0", "q4_0"
    lens = [700, 333]
    B = len(lens)
    n_layers = 1 if order == "same_cache" else 3
    steps = 6 if order == "same_cache" else 4
    wl = syn.Workload("b2b", n_layers, B, H * G, H, D, tk, tv, tuple(lens), seed=77)
    cap = 736
    caches = [kvq.KVCache(B, H, D, cap, tk, tv) for _ in range(n_layers)]
    rows = {}
    for l in range(n_layers):
        for kind in (syn.KIND_K, syn.KIND_V):
            rows[l, kind] = [torch.stack([syn.kv_rows(wl, kind, l, b, h, 0, lens[b] + steps + 1) for h in range(H)])
                             for b in range(B)]
    ops = []
    if order == "mixed":
        # layer 0 is filled right before its first fused step; layer 1 gets a plain decode
        # between fused steps; layer 2 follows a bulk append of itself
        ops += [("prefill", 1), ("prefill", 2)]
        for s in range(steps):
            if s == 0:
                ops.append(("prefill", 0))
            ops += [("step", 0, s), ("decode", 1), ("step", 1, s), ("step", 2, s)]
    else:
        ops += [("prefill", l) for l in range(n_layers)]
        ops += [("step", l, s) for s in range(steps) for l in range(n_layers)]
    # every input is made before the first launch, so that the library's launches follow
    # one another on the stream with no other kernel between them
    n_now = [list(lens) for _ in range(n_layers)]
    plan = []
    for i, op in enumerate(ops):
        l = op[1]
        if op[0] == "prefill":
            plan.append((op[0], l, [rows[l, syn.KIND_K][b][None, :, :lens[b]].contiguous() for b in range(B)],
                         [rows[l, syn.KIND_V][b][None, :, :lens[b]].contiguous() for b in range(B)], None))
            continue
        q = syn.queries(wl, l, step=i)
        kn = vn = None
        if op[0] == "step":
            kn = torch.stack([rows[l, syn.KIND_K][b][:, n_now[l][b]] for b in range(B)])[:, :, None].contiguous()
            vn = torch.stack([rows[l, syn.KIND_V][b][:, n_now[l][b]] for b in range(B)])[:, :, None].contiguous()
            n_now[l] = [n + 1 for n in n_now[l]]
        plan.append((op[0], l, kn, vn, q, list(n_now[l]),
                     torch.empty_like(q), torch.empty((B, H * G), device="cuda")))
    ws = caches[0].workspace(H * G, 0)  # one workspace shared by every launch
    torch.cuda.synchronize()
    expect = []
    for item in plan:
        kind, l = item[0], item[1]
        c = caches[l]
        if kind == "prefill":
            for b in range(B):
                c.append(item[2][b], item[3][b], b0=b)
            continue
        _, _, kn, vn, q, ns, out, lse = item
        if kind == "step":
            c.append_decode(kn, vn, q, scale=wl.scale, out=out, lse=lse, workspace=ws)
        else:
            c.decode(q, scale=wl.scale, out=out, lse=lse, workspace=ws)
        expect.append((l, ns, q, out, lse))
    torch.cuda.synchronize()
    for l in range(n_layers):
        assert caches[l].sync_lengths() == n_now[l]
        assert caches[l].read_error() == 0
    for l, ns, q, out, lse in expect:
        qh = q.cpu().numpy()
        for b in range(B):
            n = ns[b]
            kc, ks = oracle.quantize(tk, rows[l, syn.KIND_K][b][:, :n].cpu().numpy())
            vc, vs = oracle.quantize(tv, rows[l, syn.KIND_V][b][:, :n].cpu().numpy())
            ref, ref_lse = oracle.attention(tk, kc, ks, tv, vc, vs, n, qh[b], wl.scale)
            assert np.abs(out[b].cpu().numpy() - ref).max() <= TOL, (l, n, b)
            assert np.abs(lse[b].cpu().numpy() - ref_lse).max() <= TOL


def test_one_workspace_serves_every_split_count(kvq):
    """The workspace's arrival counters sit at places that do not depend on n_splits, so one
    workspace zeroed once serves decodes with different split counts in turn: 3 splits (one
    merge level), then 64 (8192 CTAs: the two-level merge), then 3 again (16 sequences, 8 KV
    heads, G 5)."""
    B, Hkv, G, D = 16, 8, 5, 128
    lens = tuple(300 + 97 * b for b in range(B))
    wl = syn.Workload("ws-reuse", 1, B, Hkv * G, Hkv, D, "q8_0", "q4_0", lens, seed=71)
    cache = kvq.KVCache(B, Hkv, D, (max(lens) + 31) // 16 * 16, "q8_0", "q4_0")
    Ks, Vs = [], []
    for b in range(B):
        K = torch.stack([syn.kv_rows(wl, syn.KIND_K, 0, b, h, 0, lens[b]) for h in range(Hkv)])
        V = torch.stack([syn.kv_rows(wl, syn.KIND_V, 0, b, h, 0, lens[b]) for h in range(Hkv)])
        cache.append(K[None].contiguous(), V[None].contiguous(), b0=b)
        Ks.append(K.cpu().numpy())
        Vs.append(V.cpu().numpy())
    ws = torch.zeros(max(cache.workspace_bytes(wl.n_q_heads, s) for s in (3, 64)), dtype=torch.uint8,
                     device="cuda")
    refs = []
    for step in range(3):
        q = syn.queries(wl, 0, step=step)
        qh = q.cpu().numpy()
        r = []
        for b in range(B):
            kc, ks = oracle.quantize("q8_0", Ks[b])
            vc, vs = oracle.quantize("q4_0", Vs[b])
            r.append(oracle.attention("q8_0", kc, ks, "q4_0", vc, vs, lens[b], qh[b], wl.scale, n_threads=0))
        refs.append((q, r))
    for (q, r), splits in zip(refs, (3, 64, 3)):
        out, lse = cache.decode(q, scale=wl.scale, n_splits=splits, workspace=ws)
        torch.cuda.synchronize()
        assert cache.read_error() == 0
        for b in range(B):
            assert np.abs(out[b].cpu().numpy() - r[b][0]).max() <= TOL, (splits, b)
            assert np.abs(lse[b].cpu().numpy() - r[b][1]).max() <= TOL, (splits, b)
