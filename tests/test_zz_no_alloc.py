"""kvq_decode_attention_noalloc: decode without a caller workspace.

Some callers cannot allocate device memory where they decode (a plugin that is handed
only input and output pointers, a server whose allocator has reserved all of HBM for
cache pages, code that must not allocate during graph capture).  For them the library
keeps a fixed scratch array of its own.  These checks call the entry point through the
C ABI and compare it with the CPU oracle (fp64 attention over the oracle's own
quantisation of the same rows) and with kvq_decode_attention (caller workspace) on the
same inputs, for two calls in a row, and check that an oversized request is refused.
This file is named to be collected last.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn

pytestmark = pytest.mark.gpu

TOL = 1e-3  # the attention tolerance of the parity tests


@pytest.fixture(scope="module")
def kvq():
    import quantised_kv_long_gb300 as m
    return m


def filled_cache(kvq, wl):
    cache = kvq.KVCache(wl.batch, wl.n_kv_heads, wl.head_dim, (max(wl.lengths) + 31) // 16 * 16,
                        wl.type_k, wl.type_v)
    for b in range(wl.batch):
        K = torch.stack([syn.kv_rows(wl, syn.KIND_K, 0, b, h, 0, wl.lengths[b]) for h in range(wl.n_kv_heads)])
        V = torch.stack([syn.kv_rows(wl, syn.KIND_V, 0, b, h, 0, wl.lengths[b]) for h in range(wl.n_kv_heads)])
        cache.append(K[None].contiguous(), V[None].contiguous(), b0=b)
    return cache


def oracle_reference(wl, q):
    """fp64 attention of every sequence by the CPU oracle, which quantises the same seeded
    fp32 rows itself: (out [B, Hq, D], lse [B, Hq])."""
    qh = q.cpu().numpy()
    outs, lses = [], []
    for b in range(wl.batch):
        n = wl.lengths[b]
        K = torch.stack([syn.kv_rows(wl, syn.KIND_K, 0, b, h, 0, n) for h in range(wl.n_kv_heads)]).cpu().numpy()
        V = torch.stack([syn.kv_rows(wl, syn.KIND_V, 0, b, h, 0, n) for h in range(wl.n_kv_heads)]).cpu().numpy()
        kc, ks = oracle.quantize(wl.type_k, K, n_threads=0)
        vc, vs = oracle.quantize(wl.type_v, V, n_threads=0)
        o, l = oracle.attention(wl.type_k, kc, ks, wl.type_v, vc, vs, n, qh[b], wl.scale, n_threads=0)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)


def assert_close_to_oracle(out, lse, ref, ref_lse, what):
    err = float(np.abs(out.cpu().numpy() - ref).max())
    lerr = float(np.abs(lse.cpu().numpy() - ref_lse).max())
    assert err <= TOL and lerr <= TOL, (what, err, lerr)


@pytest.mark.parametrize("shape", [
    # (batch, Hq, Hkv, D, K type, V type, lengths)
    (1, 16, 2, 256, "q8_0", "q8_0", (3001,)),
    (2, 40, 8, 128, "q8_0", "q4_0", (2500, 777)),
    (1, 8, 2, 128, "f16", "f16", (40,)),
])
def test_noalloc_matches_workspace_decode_twice(kvq, shape):
    B, Hq, Hkv, D, tk, tv, lens = shape
    wl = syn.Workload("noalloc", 1, B, Hq, Hkv, D, tk, tv, lens, seed=31)
    cache = filled_cache(kvq, wl)
    q = syn.queries(wl, 0)
    ws_out, ws_lse = cache.decode(q, scale=wl.scale)
    torch.cuda.synchronize()
    ref, ref_lse = oracle_reference(wl, q)
    assert_close_to_oracle(ws_out, ws_lse, ref, ref_lse, "workspace entry point")
    for call in range(2):
        out, lse = cache.decode_noalloc(q, scale=wl.scale)
        torch.cuda.synchronize()
        assert_close_to_oracle(out, lse, ref, ref_lse, f"no-allocation call {call}")
        err = float((out - ws_out).abs().max())
        lerr = float((lse - ws_lse).abs().max())
        assert err <= TOL and lerr <= TOL, (call, err, lerr)
    assert cache.read_error() == 0


def test_noalloc_explicit_splits_and_new_queries(kvq):
    """Two consecutive calls with different split counts and queries (the scratch keeps
    the previous call's contents; each call must not depend on them)."""
    wl = syn.Workload("noalloc2", 1, 1, 10, 2, 128, "q4_0", "q4_0", (1999,), seed=32)
    cache = filled_cache(kvq, wl)
    for call, (splits, step) in enumerate([(64, 0), (7, 1), (300, 2)]):
        q = syn.queries(wl, 0, step=step)
        ref, ref_lse = oracle_reference(wl, q)
        ws_out, ws_lse = cache.decode(q, scale=wl.scale, n_splits=splits)
        out, lse = cache.decode_noalloc(q, scale=wl.scale, n_splits=splits)
        torch.cuda.synchronize()
        assert_close_to_oracle(out, lse, ref, ref_lse, call)
        assert float((out - ws_out).abs().max()) <= TOL, call
        assert float((lse - ws_lse).abs().max()) <= TOL, call


def test_noalloc_after_a_larger_shape(kvq):
    """A call whose counter region is smaller than the previous call's: the array's front is
    still zero from the previous call (its counters ended at zero), so the clear is skipped;
    then a larger one again, which must clear the previous call's split partials first."""
    shapes = [(16, 40, 8, 128, "q8_0", "q4_0", tuple(300 + 37 * b for b in range(16))),
              (1, 4, 2, 128, "q8_0", "q8_0", (900,)),
              (4, 40, 8, 128, "q4_0", "q4_0", (1000, 17, 600, 2049))]
    for i, (B, Hq, Hkv, D, tk, tv, lens) in enumerate(shapes):
        wl = syn.Workload(f"noalloc4-{i}", 1, B, Hq, Hkv, D, tk, tv, lens, seed=40 + i)
        cache = filled_cache(kvq, wl)
        q = syn.queries(wl, 0)
        out, lse = cache.decode_noalloc(q, scale=wl.scale)
        torch.cuda.synchronize()
        ref, ref_lse = oracle_reference(wl, q)
        assert_close_to_oracle(out, lse, ref, ref_lse, i)
        assert cache.read_error() == 0


def test_noalloc_rejects_oversized_request(kvq):
    wl = syn.Workload("noalloc3", 1, 2, 16, 2, 128, "q8_0", "q8_0", (64, 64), seed=33)
    cache = filled_cache(kvq, wl)
    q = syn.queries(wl, 0)
    # 2 sequences x 16 heads x 1024 splits x 128 values x 4 B of partials alone is 16 MiB
    assert cache.workspace_bytes(16, 1024) > 8 << 20
    out = torch.full_like(q, 7.0)
    with pytest.raises(kvq.KvqError) as e:
        cache.decode_noalloc(q, n_splits=1024, out=out)
    assert e.value.status == 7
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())  # nothing was launched
    assert kvq.lib.kvq_status_string(7).startswith(b"decode needs more scratch")
