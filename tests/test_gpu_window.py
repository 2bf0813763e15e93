"""GPU parity of the position-axis mixed cache: an f16 window of the most recent tokens in
front of a quantised tail ("HAL #582 -- per-layer KV compression study", section 5 P2).

* Write path: every token quantised into the tail on eviction is bit-exact against the
  oracle quantising the same token's f16 value; the window holds the f16 values of the
  last W tokens, each in ring slot t mod W.
* Read path: decode over both regions matches the oracle's two-region result (split
  triples of each region, merged by the oracle's exact combine) within 1e-3, through the
  one-launch form (both regions' splits in one grid and one merge) at D = 128 and 256.
* One step in one launch (kvq_window_append_decode): bit-identical to the separate append
  and decode, the same pins as above, graph replay across the window's fill and first
  evictions, capacity refusal, and slow waits reported without losing exactness.
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
    return m


def natural(cache):
    kc, ks, vc, vs = (t.cpu().numpy() for t in cache.planes())
    B, H, cap, D = cache.batch, cache.n_kv_heads, cache.capacity, cache.head_dim
    return (kvq_layout.decode_plane(kc, ks, cache.type_k, False, B, H, cap, D) +
            kvq_layout.decode_plane(vc, vs, cache.type_v, True, B, H, cap, D))


def f16_round(x):
    return x.astype(np.float16).astype(np.float32)


def reference(tk, tv, Xk, Xv, n, W, q, scale):
    """Oracle decode over window (last min(n, W) tokens, f16) + tail (older tokens quantised
    from their f16 values), for one sequence: Xk, Xv [H, N, D], q [Hq, D]."""
    w = min(n, W)
    kw = oracle.quantize("f16", Xk[:, n - w:n])
    vw = oracle.quantize("f16", Xv[:, n - w:n])
    kt = oracle.quantize(tk, f16_round(Xk[:, :n - w]))
    vt = oracle.quantize(tv, f16_round(Xv[:, :n - w]))
    ow, mw, lw = oracle.attention_partials("f16", *kw, "f16", *vw, [0, w], q, scale)
    ot, mt, lt = oracle.attention_partials(tk, *kt, tv, *vt, [0, n - w], q, scale)
    return oracle.combine(np.concatenate([ow, ot], 1), np.concatenate([mw, mt], 1), np.concatenate([lw, lt], 1))


@pytest.mark.parametrize("tk,tv,D,G", [("q8_0", "q4_0", 128, 5), ("q8_0", "q8_0", 256, 8), ("q4_0", "q4_0", 128, 4),
                                    ("q4_0", "q8_0", 256, 2), ("f16", "q4_0", 256, 5)])
def test_window_evicts_bit_exact_and_decodes(kvq, tk, tv, D, G):
    B, H, W, N = 2, 2, 32, 90
    wl = syn.Workload("window", 1, B, H * G, H, D, tk, tv, (N, N), seed=40 + D + G)
    Xk = torch.stack([torch.stack([syn.kv_rows(wl, syn.KIND_K, 0, b, h, 0, N) for h in range(H)]) for b in range(B)])
    Xv = torch.stack([torch.stack([syn.kv_rows(wl, syn.KIND_V, 0, b, h, 0, N) for h in range(H)]) for b in range(B)])
    cache = kvq.WindowedCache(B, H, D, W, 96, tk, tv)
    Xk_h, Xv_h = Xk.cpu().numpy(), Xv.cpu().numpy()
    checkpoints = {1, 17, W, W + 1, 63, N}
    for t in range(N):
        cache.append(Xk[:, :, t].contiguous(), Xv[:, :, t].contiguous())
        n = t + 1
        if n not in checkpoints:
            continue
        q = syn.queries(wl, 0, step=n)
        out, lse = cache.decode(q, scale=wl.scale)
        torch.cuda.synchronize()
        assert cache.lengths() == ([min(n, W)] * B, [max(0, n - W)] * B)
        qh = q.cpu().numpy()
        for b in range(B):
            ref, ref_lse = reference(tk, tv, Xk_h[b], Xv_h[b], n, W, qh[b], wl.scale)
            assert np.abs(out[b].cpu().numpy() - ref).max() <= TOL, (n, b)
            assert np.abs(lse[b].cpu().numpy() - ref_lse).max() <= TOL, (n, b)
    assert cache.window.sync_lengths() == [W] * B and cache.tail.sync_lengths() == [N - W] * B
    assert cache.window.read_error() == 0 and cache.tail.read_error() == 0
    # tail: tokens 0 .. N-W-1, quantised from their f16 values, in order
    tkc, tks, tvc, tvs = natural(cache.tail)
    ok, osk = oracle.quantize(tk, f16_round(Xk_h[:, :, :N - W]))
    ov, osv = oracle.quantize(tv, f16_round(Xv_h[:, :, :N - W]))
    assert np.array_equal(tkc[:, :, :N - W], ok) and np.array_equal(tks[:, :, :N - W], osk)
    assert np.array_equal(tvc[:, :, :N - W], ov) and np.array_equal(tvs[:, :, :N - W], osv)
    # window: token t in slot t mod W
    wkc, _, wvc, _ = natural(cache.window)
    for t in range(N - W, N):
        s = t % W
        assert np.array_equal(wkc[:, :, s], oracle.quantize("f16", Xk_h[:, :, t])[0])
        assert np.array_equal(wvc[:, :, s], oracle.quantize("f16", Xv_h[:, :, t])[0])


def test_window_capacity_and_arguments(kvq):
    B, H, D, W = 1, 2, 128, 16
    cache = kvq.WindowedCache(B, H, D, W, 16, "q8_0", "q8_0")
    x = torch.randn((B, H, D), device="cuda")
    for _ in range(2 * W):
        cache.append(x, x)
    with pytest.raises(kvq.KvqError) as e:      # a full window would evict into a full tail
        cache.append(x, x)
    assert e.value.status == 3
    assert cache.lengths() == ([W], [16])
    bad = kvq.KVCache(B, H, D, 32, "q8_0", "q8_0")  # the window must be f16
    assert kvq.lib.kvq_window_append(bad.handle, cache.tail.handle, x.data_ptr(), x.data_ptr(), None) == 2
    other = kvq.KVCache(B, H, 256, 32, "q8_0", "q8_0")  # shapes differ
    assert kvq.lib.kvq_window_append(cache.window.handle, other.handle, x.data_ptr(), x.data_ptr(), None) == 1
    assert kvq.lib.kvq_window_append(cache.window.handle, cache.window.handle, x.data_ptr(), x.data_ptr(), None) == 1
    torch.cuda.synchronize()


def test_window_graph_replay(kvq):
    """Append + decode captured once and replayed: the ring slot and the lengths advance on
    the device."""
    B, H, D, G, W = 1, 2, 128, 4, 32
    N0, steps = 40, 6
    wl = syn.Workload("windowg", 1, B, H * G, H, D, "q8_0", "q4_0", (N0 + steps,), seed=7)
    Xk = torch.stack([syn.kv_rows(wl, syn.KIND_K, 0, 0, h, 0, N0 + steps) for h in range(H)])[None]
    Xv = torch.stack([syn.kv_rows(wl, syn.KIND_V, 0, 0, h, 0, N0 + steps) for h in range(H)])[None]
    cache = kvq.WindowedCache(B, H, D, W, 64, "q8_0", "q4_0")
    for t in range(N0):
        cache.append(Xk[:, :, t].contiguous(), Xv[:, :, t].contiguous())
    kn = torch.empty((B, H, D), device="cuda")
    vn = torch.empty((B, H, D), device="cuda")
    q = syn.queries(wl, 0)
    out = torch.empty_like(q)
    lse = torch.empty((B, H * G), device="cuda")
    ws = cache.workspace(H * G)
    st = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        cache.append(kn, vn, stream=st)
        cache.decode(q, scale=wl.scale, out=out, lse=lse, workspace=ws, stream=st)
    torch.cuda.synchronize()
    cache.window.sync_lengths()
    cache.tail.sync_lengths()
    Xk_h, Xv_h, qh = Xk.cpu().numpy(), Xv.cpu().numpy(), q.cpu().numpy()
    for s in range(steps):
        kn.copy_(Xk[:, :, N0 + s])
        vn.copy_(Xv[:, :, N0 + s])
        g.replay()
        torch.cuda.synchronize()
        n = N0 + s + 1
        assert cache.window.sync_lengths() == [W] and cache.tail.sync_lengths() == [n - W]
        ref, _ = reference("q8_0", "q4_0", Xk_h[0], Xv_h[0], n, W, qh[0], wl.scale)
        assert np.abs(out[0].cpu().numpy() - ref).max() <= TOL, s


def rows_of(wl, kind, B, H, N):
    return torch.stack([torch.stack([syn.kv_rows(wl, kind, 0, b, h, 0, N) for h in range(H)]) for b in range(B)])


@pytest.mark.parametrize("tk,tv,D,G", [("q8_0", "q4_0", 128, 5), ("q8_0", "q8_0", 256, 8), ("q4_0", "q4_0", 128, 4),
                                    ("f16", "q4_0", 256, 2), ("q4_0", "q8_0", 256, 12)])
def test_window_append_decode_one_step(kvq, tk, tv, D, G):
    """kvq_window_append_decode: the write path and the read path of one token in one launch
    (G <= 8; G = 12 takes the two-launch form).  Every step's output equals, bit for bit,
    that of a second pair driven by the separate append and decode calls, and matches the
    oracle at checkpoints; the tail's codes are bit-exact and the window holds token t in
    slot t mod W."""
    B, H, W, N = 2, 2, 32, 90
    wl = syn.Workload("window1", 1, B, H * G, H, D, tk, tv, (N, N), seed=70 + D + G)
    Xk, Xv = rows_of(wl, syn.KIND_K, B, H, N), rows_of(wl, syn.KIND_V, B, H, N)
    fused = kvq.WindowedCache(B, H, D, W, 96, tk, tv)
    split = kvq.WindowedCache(B, H, D, W, 96, tk, tv)
    ws = fused.workspace(H * G)
    Xk_h, Xv_h = Xk.cpu().numpy(), Xv.cpu().numpy()
    checkpoints = {1, 17, W, W + 1, 63, N}
    for t in range(N):
        n = t + 1
        q = syn.queries(wl, 0, step=n)
        out, lse = fused.append_decode(Xk[:, :, t].contiguous(), Xv[:, :, t].contiguous(), q, scale=wl.scale,
                                       workspace=ws)
        split.append(Xk[:, :, t].contiguous(), Xv[:, :, t].contiguous())
        out2, lse2 = split.decode(q, scale=wl.scale)
        torch.cuda.synchronize()
        assert torch.equal(out, out2) and torch.equal(lse, lse2), n
        assert fused.lengths() == ([min(n, W)] * B, [max(0, n - W)] * B)
        if n not in checkpoints:
            continue
        assert fused.window.sync_lengths() == [min(n, W)] * B and fused.tail.sync_lengths() == [max(0, n - W)] * B
        qh = q.cpu().numpy()
        for b in range(B):
            ref, ref_lse = reference(tk, tv, Xk_h[b], Xv_h[b], n, W, qh[b], wl.scale)
            assert np.abs(out[b].cpu().numpy() - ref).max() <= TOL, (n, b)
            assert np.abs(lse[b].cpu().numpy() - ref_lse).max() <= TOL, (n, b)
    assert fused.window.read_error() == 0 and fused.tail.read_error() == 0
    assert torch.count_nonzero(ws[-256:]) == 0  # the eviction flags are left at zero
    tkc, tks, tvc, tvs = natural(fused.tail)
    ok, osk = oracle.quantize(tk, f16_round(Xk_h[:, :, :N - W]))
    ov, osv = oracle.quantize(tv, f16_round(Xv_h[:, :, :N - W]))
    assert np.array_equal(tkc[:, :, :N - W], ok) and np.array_equal(tks[:, :, :N - W], osk)
    assert np.array_equal(tvc[:, :, :N - W], ov) and np.array_equal(tvs[:, :, :N - W], osv)
    wkc, _, wvc, _ = natural(fused.window)
    for t in range(N - W, N):
        assert np.array_equal(wkc[:, :, t % W], oracle.quantize("f16", Xk_h[:, :, t])[0])
        assert np.array_equal(wvc[:, :, t % W], oracle.quantize("f16", Xv_h[:, :, t])[0])


def test_window_append_decode_graph_replay(kvq):
    """The one-launch step captured once and replayed across the window's fill and its
    first evictions: lengths, ring slot and eviction flags advance on the device."""
    B, H, D, G, W = 1, 2, 256, 8, 32
    N0, steps = 20, 30
    wl = syn.Workload("window1g", 1, B, H * G, H, D, "q8_0", "q8_0", (N0 + steps,), seed=9)
    Xk, Xv = rows_of(wl, syn.KIND_K, B, H, N0 + steps), rows_of(wl, syn.KIND_V, B, H, N0 + steps)
    cache = kvq.WindowedCache(B, H, D, W, 64, "q8_0", "q8_0")
    for t in range(N0):
        cache.append(Xk[:, :, t].contiguous(), Xv[:, :, t].contiguous())
    kn = torch.empty((B, H, D), device="cuda")
    vn = torch.empty((B, H, D), device="cuda")
    q = syn.queries(wl, 0)
    out = torch.empty_like(q)
    lse = torch.empty((B, H * G), device="cuda")
    ws = cache.workspace(H * G)
    st = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        cache.append_decode(kn, vn, q, scale=wl.scale, out=out, lse=lse, workspace=ws, stream=st)
    torch.cuda.synchronize()
    cache.window.sync_lengths()
    cache.tail.sync_lengths()
    Xk_h, Xv_h, qh = Xk.cpu().numpy(), Xv.cpu().numpy(), q.cpu().numpy()
    for s in range(steps):
        kn.copy_(Xk[:, :, N0 + s])
        vn.copy_(Xv[:, :, N0 + s])
        g.replay()
        torch.cuda.synchronize()
        n = N0 + s + 1
        assert cache.window.sync_lengths() == [min(n, W)] and cache.tail.sync_lengths() == [max(0, n - W)]
        ref, ref_lse = reference("q8_0", "q8_0", Xk_h[0], Xv_h[0], n, W, qh[0], wl.scale)
        assert np.abs(out[0].cpu().numpy() - ref).max() <= TOL, s
        assert np.abs(lse[0].cpu().numpy() - ref_lse).max() <= TOL, s
    assert cache.window.read_error() == 0 and cache.tail.read_error() == 0


def test_window_append_decode_capacity(kvq):
    """A full window with a full tail: refused on the host, nothing written."""
    B, H, D, W = 1, 2, 128, 16
    cache = kvq.WindowedCache(B, H, D, W, 32, "q8_0", "q8_0")
    x = torch.randn((B, H, D), device="cuda")
    q = torch.randn((B, 2 * H, D), device="cuda")
    for _ in range(W + 32):
        cache.append_decode(x, x, q)
    with pytest.raises(kvq.KvqError) as e:
        cache.append_decode(x, x, q)
    assert e.value.status == 3
    assert cache.lengths() == ([W], [32])
    torch.cuda.synchronize()
    assert cache.window.read_error() == 0 and cache.tail.read_error() == 0


def test_window_append_decode_wait_reported(kvq):
    """With a wait limit far below a copy's latency every slow wait of the one-launch step
    (ring waits, the merge, the window CTA's wait for the evicted row) is reported as
    KVQ_DEVERR_TIMEOUT and then completed: the step's result is still exact, the lengths
    advance, the eviction flags end at zero, and the next step with the default limit
    reports nothing."""
    B, H, D, G, W, N = 1, 2, 256, 8, 32, 192  # N a multiple of W: the window's slot 0 holds its oldest token
    wl = syn.Workload("window-timeout", 1, B, H * G, H, D, "q8_0", "q8_0", (N + 2,), seed=62)
    Xk, Xv = rows_of(wl, syn.KIND_K, B, H, N + 2), rows_of(wl, syn.KIND_V, B, H, N + 2)
    cache = kvq.WindowedCache(B, H, D, W, 256, "q8_0", "q8_0")
    # the tail holds evicted tokens, quantised from their f16 values
    cache.tail.append(Xk[:, :, :N - W].half().float().contiguous(), Xv[:, :, :N - W].half().float().contiguous())
    cache.window.append(Xk[:, :, N - W:N].contiguous(), Xv[:, :, N - W:N].contiguous())
    ws = cache.workspace(H * G)
    q = syn.queries(wl, 0)
    torch.cuda.synchronize()
    assert cache.window.read_error() == 0 and cache.tail.read_error() == 0
    Xk_h, Xv_h, qh = Xk.cpu().numpy(), Xv.cpu().numpy(), q.cpu().numpy()
    kvq.set_wait_limit(64)
    try:
        out, lse = cache.append_decode(Xk[:, :, N].contiguous(), Xv[:, :, N].contiguous(), q, scale=wl.scale,
                                       workspace=ws)
    finally:
        kvq.set_wait_limit(0)
    torch.cuda.synchronize()
    assert cache.window.read_error() == kvq.DEVERR_TIMEOUT
    assert cache.tail.read_error() in (0, kvq.DEVERR_TIMEOUT)
    assert torch.count_nonzero(ws[-256:]) == 0
    assert cache.window.sync_lengths() == [W] and cache.tail.sync_lengths() == [N - W + 1]
    ref, ref_lse = reference("q8_0", "q8_0", Xk_h[0], Xv_h[0], N + 1, W, qh[0], wl.scale)
    assert np.abs(out[0].cpu().numpy() - ref).max() <= TOL
    assert np.abs(lse[0].cpu().numpy() - ref_lse).max() <= TOL
    out, lse = cache.append_decode(Xk[:, :, N + 1].contiguous(), Xv[:, :, N + 1].contiguous(), q, scale=wl.scale,
                                   workspace=ws)
    torch.cuda.synchronize()
    assert cache.window.read_error() == 0 and cache.tail.read_error() == 0
    ref, ref_lse = reference("q8_0", "q8_0", Xk_h[0], Xv_h[0], N + 2, W, qh[0], wl.scale)
    assert np.abs(out[0].cpu().numpy() - ref).max() <= TOL
    assert np.abs(lse[0].cpu().numpy() - ref_lse).max() <= TOL


def test_window_append_decode_large_grid_two_launches(kvq):
    """A batch whose two-region grid is larger than one resident wave (8 sequences x 8 KV
    heads x the tail's splits): the launcher refuses the one-launch form and the call runs
    the append and the decode as two launches, with the same results and lengths."""
    B, H, D, G, W, N = 8, 8, 128, 5, 16, 40
    wl = syn.Workload("window-wide", 1, B, H * G, H, D, "q8_0", "q4_0", (N,) * B, seed=77)
    Xk, Xv = rows_of(wl, syn.KIND_K, B, H, N), rows_of(wl, syn.KIND_V, B, H, N)
    fused = kvq.WindowedCache(B, H, D, W, 160, "q8_0", "q4_0")
    split = kvq.WindowedCache(B, H, D, W, 160, "q8_0", "q4_0")
    assert fused.tail.auto_splits(H * G) * H * B > 152  # more CTAs than one CTA per SM
    ws = fused.workspace(H * G)
    Xk_h, Xv_h = Xk.cpu().numpy(), Xv.cpu().numpy()
    for t in range(N):
        q = syn.queries(wl, 0, step=t + 1)
        out, lse = fused.append_decode(Xk[:, :, t].contiguous(), Xv[:, :, t].contiguous(), q, scale=wl.scale,
                                       workspace=ws)
        split.append(Xk[:, :, t].contiguous(), Xv[:, :, t].contiguous())
        out2, lse2 = split.decode(q, scale=wl.scale)
        torch.cuda.synchronize()
        assert torch.equal(out, out2) and torch.equal(lse, lse2), t
    assert fused.window.sync_lengths() == [W] * B and fused.tail.sync_lengths() == [N - W] * B
    assert fused.window.read_error() == 0 and fused.tail.read_error() == 0
    qh = q.cpu().numpy()
    for b in (0, B - 1):
        ref, ref_lse = reference("q8_0", "q4_0", Xk_h[b], Xv_h[b], N, W, qh[b], wl.scale)
        assert np.abs(out[b].cpu().numpy() - ref).max() <= TOL, b
        assert np.abs(lse[b].cpu().numpy() - ref_lse).max() <= TOL, b
