"""GPU parity of draft verify (kvq_decode_verify): n_q queries per sequence, the last n_q
cache rows being the draft, query i attending to positions [0, len - n_q + i]
("HAL #582 -- per-layer KV compression study", section 5 P0: decode batches of up to 16
query rows through the same typed readers).  Every (sequence, query, head) is checked
against the oracle's exact attention over its own prefix, within 1e-3."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn

pytestmark = pytest.mark.gpu

TOL = 1e-3


@pytest.fixture(scope="module")
def kvq():
    import quantised_kv_long_gb300 as m
    yield m
    m.set_verify_path(0)


def filled(kvq, wl, cap):
    cache = kvq.KVCache(wl.batch, wl.n_kv_heads, wl.head_dim, cap, wl.type_k, wl.type_v)
    K, V = [], []
    for b in range(wl.batch):
        k = torch.stack([syn.kv_rows(wl, syn.KIND_K, 0, b, h, 0, wl.lengths[b]) for h in range(wl.n_kv_heads)])
        v = torch.stack([syn.kv_rows(wl, syn.KIND_V, 0, b, h, 0, wl.lengths[b]) for h in range(wl.n_kv_heads)])
        if wl.lengths[b]:
            cache.append(k[None].contiguous(), v[None].contiguous(), b0=b)
        K.append(k.cpu().numpy())
        V.append(v.cpu().numpy())
    return cache, K, V


def check(wl, K, V, q, out, lse, n_q):
    qh, oh, lh = q.cpu().numpy(), out.cpu().numpy(), lse.cpu().numpy()
    for b in range(wl.batch):
        L = wl.lengths[b]
        kc, ks = oracle.quantize(wl.type_k, K[b])
        vc, vs = oracle.quantize(wl.type_v, V[b])
        for i in range(n_q):
            n = min(L, max(0, L - n_q + i + 1))
            ref, ref_lse = oracle.attention(wl.type_k, kc, ks, wl.type_v, vc, vs, n, qh[b, i], wl.scale)
            if n == 0:
                assert np.all(oh[b, i] == 0) and np.all(np.isneginf(lh[b, i])), (b, i)
                continue
            assert np.abs(oh[b, i] - ref).max() <= TOL, (b, i, n)
            assert np.abs(lh[b, i] - ref_lse).max() <= TOL, (b, i, n)


@pytest.mark.parametrize("shape", [
    # (B, Hkv, G, D, K type, V type, lengths, n_q, splits)
    (2, 2, 5, 128, "q8_0", "q4_0", (300, 1000), 4, 0),
    (2, 2, 5, 128, "q8_0", "q4_0", (300, 1000), 16, 0),
    (1, 2, 8, 256, "q8_0", "q8_0", (2049,), 16, 0),
    (1, 2, 8, 256, "q8_0", "q8_0", (2049,), 3, 7),
    (2, 1, 4, 128, "q4_0", "q4_0", (777, 64), 9, 64),
    (1, 2, 6, 128, "f16", "f16", (513,), 5, 1),
    (3, 2, 2, 128, "q4_0", "q8_0", (5, 17, 40), 8, 0),     # a sequence shorter than the draft
    (1, 2, 5, 128, "q8_0", "q4_0", (1,), 1, 0),
])
@pytest.mark.parametrize("path", [0, 1, 2])
def test_verify_matches_oracle(kvq, shape, path):
    """Every verify kernel: automatic choice (0), groups of 8 rows on the register-operand
    MMA (1), one 128-row tile on the tensor cores with tensor memory (2)."""
    kvq.set_verify_path(path)
    B, H, G, D, tk, tv, lens, n_q, splits = shape
    wl = syn.Workload("verify", 1, B, H * G, H, D, tk, tv, tuple(lens), seed=sum(lens) + n_q)
    cache, K, V = filled(kvq, wl, (max(lens) + 15) // 16 * 16 + 16)
    gen = torch.Generator(device="cuda").manual_seed(n_q * 1000 + D)
    q = torch.randn((B, n_q, H * G, D), generator=gen, device="cuda")
    out, lse = cache.verify(q, scale=wl.scale, n_splits=splits)
    torch.cuda.synchronize()
    check(wl, K, V, q, out, lse, n_q)
    assert cache.read_error() == 0


def test_verify_one_query_equals_decode(kvq):
    wl = syn.Workload("verify1", 1, 2, 16, 2, 256, "q8_0", "q8_0", (3000, 1234), seed=5)
    cache, _, _ = filled(kvq, wl, 3008)
    q = syn.queries(wl, 0)
    ref, ref_lse = cache.decode(q, scale=wl.scale)
    out, lse = cache.verify(q[:, None].contiguous(), scale=wl.scale)
    torch.cuda.synchronize()
    assert float((out[:, 0] - ref).abs().max()) <= 1e-5
    assert float((lse[:, 0] - ref_lse).abs().max()) <= 1e-5


def test_verify_rejects_bad_arguments(kvq):
    cache = kvq.KVCache(1, 2, 128, 64, "q8_0", "q8_0")
    b = __import__("ctypes").c_size_t()
    assert kvq.lib.kvq_verify_workspace_size(cache.handle, 0, 8, 0, __import__("ctypes").byref(b)) == 1
    assert kvq.lib.kvq_verify_workspace_size(cache.handle, 17, 8, 0, __import__("ctypes").byref(b)) == 1
    assert kvq.lib.kvq_verify_workspace_size(cache.handle, 16, 8, 0, __import__("ctypes").byref(b)) == 0


@pytest.mark.parametrize("tk,tv", [("q8_0", "q8_0"), ("q4_0", "q4_0"), ("q8_0", "q4_0"), ("q4_0", "q8_0")])
@pytest.mark.parametrize("D", [128, 256])
def test_verify_tensor_tile_large_values(kvq, tk, tv, D):
    """The 128-row tensor-memory kernel carries dequantised values as f16 hi + lo times a
    per-chunk power of two; blocks of values up to ~1e5 (scales near the f16 range) beside
    ordinary ones must stay exact.  Outputs of rows that attend to a huge V block are of
    that size, so the output check is relative to the row's largest reference value."""
    kvq.set_verify_path(2)
    B, H, G, n_q, L = 1, 2, 8, 16, 700
    rng = np.random.default_rng(D + len(tk + tv))
    K = rng.standard_normal((H, L, D)).astype(np.float32)
    V = rng.standard_normal((H, L, D)).astype(np.float32)
    for h in range(H):  # a few rows with huge blocks, spread over the chunks
        for r in range(3, L, 97):
            K[h, r, 32:64] *= 3e4
            V[h, r, 64:96] *= 3e4
            V[h, r + 1, :32] *= 9e4 if tv != "q4_0" else 1.0
    cache = kvq.KVCache(B, H, D, (L + 15) // 16 * 16, tk, tv)
    cache.append(torch.from_numpy(K[None]).cuda(), torch.from_numpy(V[None]).cuda())
    # the huge K block (values 32..63) changes the chunks' exponent but not the scores: Q has
    # no weight there, so scores stay O(1) and lse keeps its absolute tolerance
    qn = rng.standard_normal((B, n_q, H * G, D)).astype(np.float32)
    qn[..., 32:64] = 0.0
    q = torch.from_numpy(qn).cuda()
    scale = 1.0 / np.sqrt(D)
    out, lse = cache.verify(q, scale=scale)
    torch.cuda.synchronize()
    assert cache.read_error() == 0
    kc, ks = oracle.quantize(tk, K)
    vc, vs = oracle.quantize(tv, V)
    qh, oh, lh = q.cpu().numpy(), out.cpu().numpy(), lse.cpu().numpy()
    for i in range(n_q):
        n = L - n_q + i + 1
        ref, ref_lse = oracle.attention(tk, kc, ks, tv, vc, vs, n, qh[0, i], scale)
        err = np.abs(oh[0, i] - ref).max() / max(1.0, np.abs(ref).max())
        assert err <= TOL, (i, err)
        assert np.abs(lh[0, i] - ref_lse).max() <= TOL, i
