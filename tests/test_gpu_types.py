"""GPU parity of the further scalar types (q4_1, q5_0, q5_1) in the supported pairs
(q8_0/q5_0, q5_0/q5_0, q5_1/q5_1, q4_1/q4_1, q5_1/q4_0): codes (with their fifth bits)
and scales bit-exact against the oracle's quantisers after appends of many rows in one
launch, and decode attention within 1e-3 of the oracle's exact attention."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from tests import kvq_layout
from tests.test_gpu_parity import crafted_rows

pytestmark = pytest.mark.gpu

TOL = 1e-3
PAIRS = [("q8_0", "q5_0"), ("q5_0", "q5_0"), ("q5_1", "q5_1"), ("q4_1", "q4_1"), ("q5_1", "q4_0")]


@pytest.fixture(scope="module")
def kvq():
    import quantised_kv_long_gb300 as m
    return m


def natural(cache):
    kc, ks, vc, vs = (t.cpu().numpy() for t in cache.planes())
    B, H, cap, D = cache.batch, cache.n_kv_heads, cache.capacity, cache.head_dim
    return (kvq_layout.decode_plane(kc, ks, cache.type_k, False, B, H, cap, D) +
            kvq_layout.decode_plane(vc, vs, cache.type_v, True, B, H, cap, D))


@pytest.mark.parametrize("tk,tv", PAIRS)
@pytest.mark.parametrize("D", [128, 256])
def test_further_types_codes_bit_exact(kvq, tk, tv, D):
    rng = np.random.default_rng(D + len(tk + tv))
    B, H = 2, 2
    lens = [45, 70]
    cache = kvq.KVCache(B, H, D, 80, tk, tv)
    X = {}
    for b in range(B):
        # two appends per sequence (a ragged first one, so rows of one tile come from both)
        xk = np.stack([crafted_rows(lens[b], D, rng) for _ in range(H)])
        xv = np.stack([crafted_rows(lens[b], D, rng) for _ in range(H)])
        X[b] = (xk, xv)
        cut = 13 + b
        for s0, s1 in ((0, cut), (cut, lens[b])):
            cache.append(torch.from_numpy(xk[None, :, s0:s1]).cuda().contiguous(),
                         torch.from_numpy(xv[None, :, s0:s1]).cuda().contiguous(), b0=b)
    torch.cuda.synchronize()
    kc, ks, vc, vs = natural(cache)
    for b in range(B):
        n = lens[b]
        ok, osk = oracle.quantize(tk, X[b][0])
        ov, osv = oracle.quantize(tv, X[b][1])
        assert np.array_equal(kc[b, :, :n], ok) and np.array_equal(ks[b, :, :n], osk), b
        assert np.array_equal(vc[b, :, :n], ov) and np.array_equal(vs[b, :, :n], osv), b


@pytest.mark.parametrize("tk,tv", PAIRS)
@pytest.mark.parametrize("D,G,lens,splits", [(128, 5, (1, 500), 0), (256, 8, (2049,), 0), (128, 8, (17, 301, 64), 7),
                                             (256, 2, (777,), 64)])
def test_further_types_decode(kvq, tk, tv, D, G, lens, splits):
    B, H = len(lens), 2
    wl = syn.Workload("types", 1, B, H * G, H, D, tk, tv, tuple(lens), seed=D + G + sum(lens))
    cache = kvq.KVCache(B, H, D, (max(lens) + 15) // 16 * 16, tk, tv)
    K, V = [], []
    for b in range(B):
        k = torch.stack([syn.kv_rows(wl, syn.KIND_K, 0, b, h, 0, lens[b]) for h in range(H)])
        v = torch.stack([syn.kv_rows(wl, syn.KIND_V, 0, b, h, 0, lens[b]) for h in range(H)])
        cache.append(k[None].contiguous(), v[None].contiguous(), b0=b)
        K.append(k.cpu().numpy())
        V.append(v.cpu().numpy())
    q = syn.queries(wl, 0)
    out, lse = cache.decode(q, scale=wl.scale, n_splits=splits)
    torch.cuda.synchronize()
    qh = q.cpu().numpy()
    for b in range(B):
        kc, ks = oracle.quantize(tk, K[b])
        vc, vs = oracle.quantize(tv, V[b])
        ref, ref_lse = oracle.attention(tk, kc, ks, tv, vc, vs, lens[b], qh[b], wl.scale)
        assert np.abs(out[b].cpu().numpy() - ref).max() <= TOL, b
        assert np.abs(lse[b].cpu().numpy() - ref_lse).max() <= TOL, b
    assert cache.read_error() == 0


def test_further_types_fused_append_decode(kvq):
    tk, tv, H, D, G = "q5_1", "q4_0", 2, 128, 5
    lens = [300, 33]
    B, steps = len(lens), 3
    wl = syn.Workload("types_fused", 1, B, H * G, H, D, tk, tv, tuple(lens), seed=21)
    cache = kvq.KVCache(B, H, D, 352, tk, tv)
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
        qh = q.cpu().numpy()
        for b in range(B):
            n = lens[b] + step + 1
            kc, ks = oracle.quantize(tk, Ks[b][:, :n].cpu().numpy())
            vc, vs = oracle.quantize(tv, Vs[b][:, :n].cpu().numpy())
            ref, _ = oracle.attention(tk, kc, ks, tv, vc, vs, n, qh[b], wl.scale)
            assert np.abs(out[b].cpu().numpy() - ref).max() <= TOL, (step, b)
    assert cache.read_error() == 0


def test_further_types_rejected_where_unsupported(kvq):
    cache = kvq.KVCache(1, 2, 128, 64, "q5_0", "q5_0")
    b = __import__("ctypes").c_size_t()
    q = torch.zeros((1, 2, 10, 128), device="cuda")
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    assert kvq.lib.kvq_decode_verify(cache.handle, q.data_ptr(), 2, 10, 0.1, 0, ws.data_ptr(), q.data_ptr(),
                                     None, None) == 2
    with pytest.raises(kvq.KvqError):
        kvq.KVCache(1, 2, 128, 64, "q4_1", "q8_0")
