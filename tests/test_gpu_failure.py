"""Failure handling of the decode kernels on the GPU, without faulting or hanging it.

Every pipeline and merge wait in the decode kernels is bounded (about two seconds).
kvq_set_wait_limit sets the time after which a wait is reported (here a few dozen SM
cycles, so that waits on a healthy GPU exceed it): the kernel must then return, set
KVQ_DEVERR_TIMEOUT in the cache's error word, and leave the workspace's arrival counters
at zero, so that the next call on the same workspace (with the default limit restored)
matches the oracle again.  Each merge form is covered: one split, the last arrival merging
all splits, the column merge of a grid that is resident at once, and the two-level merge
of a larger grid.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn

pytestmark = pytest.mark.gpu

TOL = 1e-3
SHORT_LIMIT = 64  # SM cycles: far below the latency of a copy from HBM


@pytest.fixture(scope="module")
def kvq():
    import quantised_kv_long_gb300 as m
    yield m
    m.set_wait_limit(0)


def filled(kvq, wl):
    cache = kvq.KVCache(wl.batch, wl.n_kv_heads, wl.head_dim, (max(wl.lengths) + 31) // 16 * 16,
                        wl.type_k, wl.type_v)
    for b in range(wl.batch):
        K = torch.stack([syn.kv_rows(wl, syn.KIND_K, 0, b, h, 0, wl.lengths[b]) for h in range(wl.n_kv_heads)])
        V = torch.stack([syn.kv_rows(wl, syn.KIND_V, 0, b, h, 0, wl.lengths[b]) for h in range(wl.n_kv_heads)])
        cache.append(K[None].contiguous(), V[None].contiguous(), b0=b)
        del K, V
    return cache


def counter_bytes(wl):
    """Bytes of the workspace's arrival counters (front of the workspace, include/kvq.h):
    one int32 per (sequence, KV head, row group), then 33 first-level group counters each,
    each region rounded up to 256 bytes."""
    qg = (wl.G + 7) // 8
    units = wl.batch * wl.n_kv_heads * qg
    a256 = lambda x: (x + 255) // 256 * 256
    return a256(units * 4) + a256(units * 33 * 4)


def check_sequences(wl, q, out, lse, seqs):
    qh = q.cpu().numpy()
    for b in seqs:
        n = wl.lengths[b]
        K = torch.stack([syn.kv_rows(wl, syn.KIND_K, 0, b, h, 0, n) for h in range(wl.n_kv_heads)]).cpu().numpy()
        V = torch.stack([syn.kv_rows(wl, syn.KIND_V, 0, b, h, 0, n) for h in range(wl.n_kv_heads)]).cpu().numpy()
        kc, ks = oracle.quantize(wl.type_k, K, n_threads=0)
        vc, vs = oracle.quantize(wl.type_v, V, n_threads=0)
        ref, ref_lse = oracle.attention(wl.type_k, kc, ks, wl.type_v, vc, vs, n, qh[b], wl.scale, n_threads=0)
        assert np.abs(out[b].cpu().numpy() - ref).max() <= TOL, b
        assert np.abs(lse[b].cpu().numpy() - ref_lse).max() <= TOL, b


CASES = {
    # name: (batch, Hq, Hkv, D, K type, V type, lengths, n_splits)
    "one-split": (1, 8, 2, 128, "q8_0", "q4_0", (20000,), 1),
    "last-arrival": (1, 8, 2, 128, "q8_0", "q4_0", (20000,), 4),  # 8 KB of triples: one CTA merges
    "column-merge": (1, 16, 2, 256, "q8_0", "q8_0", (65536,), 0),
    "two-level": (4, 40, 8, 128, "q8_0", "q4_0", (45000, 44000, 43000, 46000), 40),
}


@pytest.mark.parametrize("name", list(CASES))
def test_wait_timeout_reported_and_recovered(kvq, name):
    B, Hq, Hkv, D, tk, tv, lens, splits = CASES[name]
    wl = syn.Workload(f"timeout-{name}", 1, B, Hq, Hkv, D, tk, tv, lens, seed=61)
    cache = filled(kvq, wl)
    q = syn.queries(wl, 0)
    ws = cache.workspace(Hq, splits)
    out = torch.full_like(q, 7.0)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    torch.cuda.synchronize()
    assert cache.read_error() == 0
    kvq.set_wait_limit(SHORT_LIMIT)
    try:
        cache.decode(q, scale=wl.scale, n_splits=splits, out=out, lse=lse, workspace=ws)
    finally:
        kvq.set_wait_limit(0)
    torch.cuda.synchronize()  # the kernel returned
    err = cache.read_error()
    assert err == kvq.DEVERR_TIMEOUT, err
    # every CTA took its arrivals: the arrival counts (low 16 bits of each counter; a wide
    # merge keeps a launch epoch above them) are back at zero
    counts = ws[:counter_bytes(wl)].view(torch.int32) & 0xffff
    assert int(counts.count_nonzero()) == 0
    # the next call on the same workspace, with the default limit, is exact again
    out2, lse2 = cache.decode(q, scale=wl.scale, n_splits=splits, workspace=ws)
    torch.cuda.synchronize()
    assert cache.read_error() == 0
    check_sequences(wl, q, out2, lse2, range(B) if B <= 2 else (0, B - 1))


def test_wait_limit_arguments(kvq):
    with pytest.raises(kvq.KvqError):
        kvq.set_wait_limit(-1)
    kvq.set_wait_limit(0)
