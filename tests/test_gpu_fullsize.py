"""GPU parity at the benchmark's full sizes, beyond the sampled decode checks of
test_gpu_parity.py:

* every code and scale of a whole-layer cache fill of the headline shape (hybrid: 65,536
  positions x 2 KV heads x 256 values, q8_0 / q8_0) and of one 4,096-row prefill chunk of
  the 14B shape (8 KV heads x 128 values, q8_0 K / q4_0 V, written behind 13 earlier rows so
  that its first and last tiles are partial), bit-exact against the oracle's quantisers;
* draft verify at full size in the benchmark's launch configuration: 16 draft queries on
  the hybrid shape (the 128-row tensor-memory tile) and 4 on the 14B shape at 131,072 (the
  8-row groups), sampled (query, head) rows against the oracle within 1e-3.
Inputs are the seeded synthetic workloads; the oracle quantises the same fp32 rows itself.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from tests import kvq_layout

pytestmark = pytest.mark.gpu

TOL = 1e-3


@pytest.fixture(scope="module")
def kvq():
    import quantised_kv_long_gb300 as m
    m.set_verify_path(0)
    return m


def natural(cache):
    """(k_codes, k_scales, v_codes, v_scales) of the whole cache in the oracle's layout."""
    kc, ks, vc, vs = (t.cpu().numpy() for t in cache.planes())
    B, H, cap, D = cache.batch, cache.n_kv_heads, cache.capacity, cache.head_dim
    return (kvq_layout.decode_plane(kc, ks, cache.type_k, False, B, H, cap, D) +
            kvq_layout.decode_plane(vc, vs, cache.type_v, True, B, H, cap, D))


def layer_rows(wl, kind, layer, n):
    return torch.stack([syn.kv_rows(wl, kind, layer, 0, h, 0, n) for h in range(wl.n_kv_heads)])


def test_headline_cache_fill_bit_exact(kvq):
    wl = syn.hybrid(65536, "q8_0", "q8_0")
    n = wl.lengths[0]
    cache = kvq.KVCache(1, wl.n_kv_heads, wl.head_dim, n, wl.type_k, wl.type_v)
    K, V = layer_rows(wl, syn.KIND_K, 0, n), layer_rows(wl, syn.KIND_V, 0, n)
    cache.append(K[None].contiguous(), V[None].contiguous())
    torch.cuda.synchronize()
    assert cache.sync_lengths() == [n] and cache.read_error() == 0
    kc, ks, vc, vs = natural(cache)
    ok_c, ok_s = oracle.quantize(wl.type_k, K.cpu().numpy(), n_threads=0)
    ov_c, ov_s = oracle.quantize(wl.type_v, V.cpu().numpy(), n_threads=0)
    assert np.array_equal(kc[0], ok_c) and np.array_equal(ks[0], ok_s)
    assert np.array_equal(vc[0], ov_c) and np.array_equal(vs[0], ov_s)


def test_prefill_chunk_bit_exact(kvq):
    wl = syn.multi_session()  # the 14B shape: Hkv 8, D 128, q8_0 K / q4_0 V
    lead, n = 13, 4096
    cap = (lead + n + 15) // 16 * 16
    K, V = layer_rows(wl, syn.KIND_K, 0, lead + n), layer_rows(wl, syn.KIND_V, 0, lead + n)
    cache = kvq.KVCache(1, wl.n_kv_heads, wl.head_dim, cap, wl.type_k, wl.type_v)
    cache.append(K[None, :, :lead].contiguous(), V[None, :, :lead].contiguous())
    cache.append(K[None, :, lead:].contiguous(), V[None, :, lead:].contiguous())
    torch.cuda.synchronize()
    assert cache.sync_lengths() == [lead + n] and cache.read_error() == 0
    kc, ks, vc, vs = natural(cache)
    ok_c, ok_s = oracle.quantize(wl.type_k, K.cpu().numpy(), n_threads=0)
    ov_c, ov_s = oracle.quantize(wl.type_v, V.cpu().numpy(), n_threads=0)
    m = lead + n
    assert np.array_equal(kc[0, :, :m], ok_c) and np.array_equal(ks[0, :, :m], ok_s)
    assert np.array_equal(vc[0, :, :m], ov_c) and np.array_equal(vs[0, :, :m], ov_s)


@pytest.mark.parametrize("which", ["hybrid-65536-nq16", "dense-131072-nq4"])
def test_verify_full_size_sampled(kvq, which):
    if which.startswith("hybrid"):
        wl, n_q = syn.hybrid(65536, "q8_0", "q8_0"), 16
    else:
        wl, n_q = syn.dense14b(131072, "q8_0", "q4_0"), 4
    L = wl.lengths[0]
    cache = kvq.KVCache(1, wl.n_kv_heads, wl.head_dim, L, wl.type_k, wl.type_v)
    K, V = layer_rows(wl, syn.KIND_K, 0, L), layer_rows(wl, syn.KIND_V, 0, L)
    cache.append(K[None].contiguous(), V[None].contiguous())
    del K, V
    torch.cuda.synchronize()
    assert cache.sync_lengths() == [L]
    q = torch.randn((1, n_q, wl.n_q_heads, wl.head_dim), generator=torch.Generator(device="cuda").manual_seed(n_q),
                    device="cuda")
    out, lse = cache.verify(q, scale=wl.scale)
    torch.cuda.synchronize()
    assert cache.read_error() == 0
    rng = np.random.default_rng(len(which))
    qh = q.cpu().numpy()
    heads = sorted({int(x) for x in rng.integers(wl.n_kv_heads, size=2)})
    for h in heads:
        K = syn.kv_rows(wl, syn.KIND_K, 0, 0, h, 0, L).cpu().numpy()[None]
        V = syn.kv_rows(wl, syn.KIND_V, 0, 0, h, 0, L).cpu().numpy()[None]
        kc, ks = oracle.quantize(wl.type_k, K, n_threads=0)
        vc, vs = oracle.quantize(wl.type_v, V, n_threads=0)
        for i in (0, n_q - 1, int(rng.integers(n_q))):
            hq = h * wl.G + int(rng.integers(wl.G))
            n = L - n_q + i + 1
            ref, ref_lse = oracle.attention(wl.type_k, kc, ks, wl.type_v, vc, vs, n, qh[0, i, hq:hq + 1], wl.scale,
                                            n_threads=0)
            assert np.abs(out[0, i, hq].cpu().numpy() - ref[0]).max() <= TOL, (h, i, hq)
            assert abs(float(lse[0, i, hq]) - ref_lse[0]) <= TOL, (h, i, hq)
