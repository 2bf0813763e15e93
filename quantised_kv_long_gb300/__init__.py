"""Python binding of libkvq (include/kvq.h): block-quantised KV cache for GB300.

Argument marshalling only.  Every step of the path -- quantise-on-append, split-K
decode attention, split merge -- runs in the CUDA kernels of ``libkvq.so``.  PyTorch
is used for device memory and streams; there is no CPU or PyTorch fallback: if the
library is missing, importing the binding raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvq.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "kvq.h")

F16, Q8_0, Q4_0 = 0, 1, 2
Q4_1, Q5_0, Q5_1 = 3, 4, 5
TYPE_IDS = {"f16": F16, "q8_0": Q8_0, "q4_0": Q4_0, "q4_1": Q4_1, "q5_0": Q5_0, "q5_1": Q5_1}
# bytes per 16-row x 128-value tile slice: codes, scales
CODE_TILE = {F16: 4096, Q8_0: 2048, Q4_0: 1024, Q4_1: 1024, Q5_0: 1280, Q5_1: 1280}
TYPE_NAMES = {v: k for k, v in TYPE_IDS.items()}
STATUS = {0: "KVQ_OK", 1: "KVQ_ERR_INVALID_ARG", 2: "KVQ_ERR_UNSUPPORTED", 3: "KVQ_ERR_CAPACITY",
          4: "KVQ_ERR_ALIGNMENT", 5: "KVQ_ERR_CUDA", 6: "KVQ_ERR_DEVICE", 7: "KVQ_ERR_SCRATCH"}
DEVERR_CAPACITY, DEVERR_TIMEOUT = 0x1, 0x2


class KvqError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}")


class TierChoice(ctypes.Structure):
    _fields_ = [("rung", ctypes.c_int32), ("type_k", ctypes.c_int32), ("type_v", ctypes.c_int32),
                ("fits", ctypes.c_int32), ("bytes", ctypes.c_uint64)]


class Desc(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("capacity", ctypes.c_int32), ("type_k", ctypes.c_int32), ("type_v", ctypes.c_int32)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libkvq.so not built ({LIB_PATH}); run `python quantised_kv_long_gb300/build.py` or __graft_entry__.build()")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    pdesc = ctypes.POINTER(Desc)
    sigs = {
        "kvq_cache_size": [pdesc, ctypes.POINTER(sz), ctypes.POINTER(sz), ctypes.POINTER(sz)],
        "kvq_cache_create": [pdesc, vp, vp, vp, vp, ctypes.POINTER(vp)],
        "kvq_cache_destroy": [vp],
        "kvq_cache_lengths": [vp, vp],
        "kvq_cache_set_lengths": [vp, vp, vp],
        "kvq_cache_sync_lengths": [vp, vp],
        "kvq_cache_read_error": [vp, vp, ctypes.POINTER(i32)],
        "kvq_quantize_append": [vp, vp, vp, i32, i32, i32, vp],
        "kvq_decode_auto_splits": [vp, i32, ctypes.POINTER(i32)],
        "kvq_decode_workspace_size": [vp, i32, i32, ctypes.POINTER(sz)],
        "kvq_decode_attention": [vp, vp, i32, ctypes.c_float, i32, vp, vp, vp, vp],
        "kvq_decode_partials": [vp, vp, i32, ctypes.c_float, i32, vp, vp, vp, vp],
        "kvq_combine": [vp, vp, vp, i32, i32, i32, vp, vp, vp],
        "kvq_decode_attention_noalloc": [vp, vp, i32, ctypes.c_float, i32, vp, vp, vp],
        "kvq_append_decode": [vp, vp, vp, vp, i32, ctypes.c_float, i32, vp, vp, vp, vp],
        "kvq_window_append": [vp, vp, vp, vp, vp],
        "kvq_verify_workspace_size": [vp, i32, i32, i32, ctypes.POINTER(sz)],
        "kvq_decode_verify": [vp, vp, i32, i32, ctypes.c_float, i32, vp, vp, vp, vp],
        "kvq_window_workspace_size": [vp, vp, i32, ctypes.POINTER(sz)],
        "kvq_window_decode": [vp, vp, vp, i32, ctypes.c_float, vp, vp, vp, vp],
        "kvq_window_append_decode": [vp, vp, vp, vp, vp, i32, ctypes.c_float, vp, vp, vp, vp],
    }
    for name, args in sigs.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    L.kvq_set_wait_limit.argtypes = [ctypes.c_int64]
    L.kvq_set_wait_limit.restype = ctypes.c_int
    L.kvq_set_verify_path.argtypes = [i32]
    L.kvq_set_verify_path.restype = ctypes.c_int
    L.kvq_set_launch_stamps.argtypes = [vp, i32, i32]
    L.kvq_set_launch_stamps.restype = ctypes.c_int
    L.kvq_select_tier.argtypes = [ctypes.c_int64, i32, i32, i32, ctypes.c_uint64, ctypes.POINTER(TierChoice)]
    L.kvq_select_tier.restype = ctypes.c_int
    L.kvq_block_bytes.argtypes = [ctypes.c_int]
    L.kvq_block_bytes.restype = ctypes.c_int32
    L.kvq_status_string.argtypes = [ctypes.c_int]
    L.kvq_status_string.restype = ctypes.c_char_p
    L.kvq_abi_version.argtypes = []
    L.kvq_abi_version.restype = ctypes.c_int32
    return L


lib = _load()


def header_functions() -> list[str]:
    """Names of the entry points declared in include/kvq.h."""
    with open(HEADER) as f:
        text = f.read()
    return re.findall(r"^KVQ_API\s+[^(]*?\b(kvq_\w+)\s*\(", text, flags=re.M)


def _check(status: int, what: str):
    if status != 0:
        raise KvqError(status, what)


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def cache_size(batch, n_kv_heads, head_dim, capacity, type_k, type_v):
    """(k_bytes, v_bytes, state_bytes) for a cache descriptor; pure host arithmetic."""
    d = Desc(batch, n_kv_heads, head_dim, capacity, _tid(type_k), _tid(type_v))
    kb, vb, sb = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib.kvq_cache_size(ctypes.byref(d), ctypes.byref(kb), ctypes.byref(vb), ctypes.byref(sb)),
           "kvq_cache_size")
    return kb.value, vb.value, sb.value


class WindowedCache:
    """A rolling f16 window of the most recent `window` tokens in front of a quantised tail
    (kvq_window_append / kvq_window_decode).  `window` must be a multiple of 16."""

    def __init__(self, batch, n_kv_heads, head_dim, window, tail_capacity, type_k="q8_0", type_v="q8_0",
                 device=None, stream=None):
        self.window = KVCache(batch, n_kv_heads, head_dim, window, "f16", "f16", device=device, stream=stream)
        self.tail = KVCache(batch, n_kv_heads, head_dim, tail_capacity, type_k, type_v, device=device, stream=stream)
        self.batch, self.n_kv_heads, self.head_dim = batch, n_kv_heads, head_dim

    def append(self, k, v, stream=None):
        """One new row per sequence: k, v fp32 [B, Hkv, D] (or [B, Hkv, 1, D])."""
        for t in (k, v):
            assert t.dtype == torch.float32 and t.is_contiguous()
            assert t.numel() == self.batch * self.n_kv_heads * self.head_dim
        _check(lib.kvq_window_append(self.window.handle, self.tail.handle, _ptr(k), _ptr(v), _stream(stream)),
               "kvq_window_append")

    def workspace_bytes(self, n_q_heads) -> int:
        b = ctypes.c_size_t()
        _check(lib.kvq_window_workspace_size(self.window.handle, self.tail.handle, n_q_heads, ctypes.byref(b)),
               "kvq_window_workspace_size")
        return b.value

    def workspace(self, n_q_heads):
        return torch.zeros(self.workspace_bytes(n_q_heads), dtype=torch.uint8, device=self.window.device)

    def decode(self, q, scale=None, out=None, lse=None, workspace=None, stream=None):
        assert q.dtype == torch.float32 and q.is_contiguous() and q.dim() == 3
        B, Hq, D = q.shape
        assert B == self.batch and D == self.head_dim
        scale = 1.0 / math.sqrt(D) if scale is None else scale
        out = torch.empty_like(q) if out is None else out
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device) if lse is None else lse
        ws = self.workspace(Hq) if workspace is None else workspace
        _check(lib.kvq_window_decode(self.window.handle, self.tail.handle, _ptr(q), Hq, scale, _ptr(ws), _ptr(out),
                                     _ptr(lse), _stream(stream)), "kvq_window_decode")
        return out, lse

    def append_decode(self, k, v, q, scale=None, out=None, lse=None, workspace=None, stream=None):
        """append(k, v) then decode(q) as one step (kvq_window_append_decode): one launch
        where the two-region grid is resident at once."""
        for t in (k, v):
            assert t.dtype == torch.float32 and t.is_contiguous()
            assert t.numel() == self.batch * self.n_kv_heads * self.head_dim
        assert q.dtype == torch.float32 and q.is_contiguous() and q.dim() == 3
        B, Hq, D = q.shape
        assert B == self.batch and D == self.head_dim
        scale = 1.0 / math.sqrt(D) if scale is None else scale
        out = torch.empty_like(q) if out is None else out
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device) if lse is None else lse
        ws = self.workspace(Hq) if workspace is None else workspace
        _check(lib.kvq_window_append_decode(self.window.handle, self.tail.handle, _ptr(k), _ptr(v), _ptr(q), Hq, scale,
                                            _ptr(ws), _ptr(out), _ptr(lse), _stream(stream)), "kvq_window_append_decode")
        return out, lse

    def lengths(self):
        """(window lengths, tail lengths) from the host mirrors."""
        return self.window.lengths(), self.tail.lengths()


def set_wait_limit(cycles: int = 0):
    """Wait limit (SM clock cycles) of later decode launches' pipeline and merge waits
    (kvq_set_wait_limit); 0 restores the default of about two seconds."""
    _check(lib.kvq_set_wait_limit(int(cycles)), "kvq_set_wait_limit")


def set_verify_path(path: int = 0):
    """Kernel of kvq_decode_verify (kvq_set_verify_path): 0 automatic, 1 groups of 8 rows on
    the register-operand MMA, 2 one 128-row tile on the tensor cores with tensor memory."""
    _check(lib.kvq_set_verify_path(int(path)), "kvq_set_verify_path")


def set_launch_stamps(buf=None, n_slots: int = 0, ctas_per_slot: int = 0):
    """Per-CTA start/exit timer stamps of later decode launches (kvq_set_launch_stamps):
    buf a uint64/int64 device tensor of n_slots * ctas_per_slot * 2 elements, or None to stop."""
    if buf is not None:
        assert buf.numel() >= n_slots * ctas_per_slot * 2 and buf.element_size() == 8 and buf.is_cuda
    _check(lib.kvq_set_launch_stamps(_ptr(buf), n_slots, ctas_per_slot), "kvq_set_launch_stamps")


def block_bytes(kv_type) -> int:
    """Bytes of one 32-value block of a storage type (kvq_block_bytes)."""
    return int(lib.kvq_block_bytes(_tid(kv_type)))


def select_tier(cells, n_layers, n_kv_heads, head_dim, budget_bytes) -> dict:
    """KV tier ladder choice (kvq_select_tier): rung, K/V type names, fits, whole-cache bytes."""
    c = TierChoice()
    _check(lib.kvq_select_tier(cells, n_layers, n_kv_heads, head_dim, budget_bytes, ctypes.byref(c)),
           "kvq_select_tier")
    return {"rung": c.rung, "type_k": TYPE_NAMES[c.type_k], "type_v": TYPE_NAMES[c.type_v], "fits": bool(c.fits),
            "bytes": int(c.bytes)}


def _tid(t):
    return TYPE_IDS[t] if isinstance(t, str) else int(t)


class KVCache:
    """One layer's cache [B, Hkv, capacity, D] over caller-side torch allocations."""

    def __init__(self, batch, n_kv_heads, head_dim, capacity, type_k="q8_0", type_v="q8_0", device=None,
                 lengths=None, stream=None):
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        self.batch, self.n_kv_heads, self.head_dim, self.capacity = batch, n_kv_heads, head_dim, capacity
        self.type_k, self.type_v = type_k, type_v
        kb, vb, sb = cache_size(batch, n_kv_heads, head_dim, capacity, type_k, type_v)
        self.k_mem = torch.empty(kb, dtype=torch.uint8, device=self.device)
        self.v_mem = torch.empty(vb, dtype=torch.uint8, device=self.device)
        self.state = torch.zeros(sb // 4, dtype=torch.int32, device=self.device)
        if lengths is not None:
            self.state[:batch] = torch.as_tensor(lengths, dtype=torch.int32, device=self.device)
        self.desc = Desc(batch, n_kv_heads, head_dim, capacity, _tid(type_k), _tid(type_v))
        h = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            _check(lib.kvq_cache_create(ctypes.byref(self.desc), _ptr(self.k_mem), _ptr(self.v_mem),
                                        _ptr(self.state), _stream(stream), ctypes.byref(h)), "kvq_cache_create")
        self.handle = h
        self._ws = {}

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value:
            lib.kvq_cache_destroy(h)
            self.handle = None

    # ---- raw planes (for tests and checkpointing) ----
    def planes(self):
        """(k_codes, k_scales, v_codes, v_scales) uint8 views of the caller-owned planes."""
        ns = self.head_dim // 128
        tiles = self.batch * self.n_kv_heads * (self.capacity // 16)
        kc = tiles * ns * CODE_TILE[_tid(self.type_k)]
        vc = tiles * ns * CODE_TILE[_tid(self.type_v)]
        return self.k_mem[:kc], self.k_mem[kc:], self.v_mem[:vc], self.v_mem[vc:]

    def lengths(self):
        out = (ctypes.c_int32 * self.batch)()
        _check(lib.kvq_cache_lengths(self.handle, ctypes.cast(out, ctypes.c_void_p)), "kvq_cache_lengths")
        return list(out)

    def set_lengths(self, lengths, stream=None):
        arr = (ctypes.c_int32 * self.batch)(*[int(x) for x in lengths])
        _check(lib.kvq_cache_set_lengths(self.handle, ctypes.cast(arr, ctypes.c_void_p), _stream(stream)),
               "kvq_cache_set_lengths")

    def sync_lengths(self, stream=None):
        _check(lib.kvq_cache_sync_lengths(self.handle, _stream(stream)), "kvq_cache_sync_lengths")
        return self.lengths()

    def read_error(self, stream=None) -> int:
        e = ctypes.c_int32()
        _check(lib.kvq_cache_read_error(self.handle, _stream(stream), ctypes.byref(e)), "kvq_cache_read_error")
        return e.value

    # ---- hot path ----
    def append(self, k, v, b0=0, stream=None):
        """Quantise fp32 rows k, v [nb, Hkv, n_new, D] into sequences b0..b0+nb-1."""
        assert k.dtype == torch.float32 and v.dtype == torch.float32 and k.is_contiguous() and v.is_contiguous()
        assert k.shape == v.shape and k.dim() == 4 and k.shape[1] == self.n_kv_heads and k.shape[3] == self.head_dim
        _check(lib.kvq_quantize_append(self.handle, _ptr(k), _ptr(v), b0, k.shape[0], k.shape[2], _stream(stream)),
               "kvq_quantize_append")

    def auto_splits(self, n_q_heads) -> int:
        s = ctypes.c_int32()
        _check(lib.kvq_decode_auto_splits(self.handle, n_q_heads, ctypes.byref(s)), "kvq_decode_auto_splits")
        return s.value

    def workspace_bytes(self, n_q_heads, n_splits=0) -> int:
        b = ctypes.c_size_t()
        _check(lib.kvq_decode_workspace_size(self.handle, n_q_heads, n_splits, ctypes.byref(b)),
               "kvq_decode_workspace_size")
        return b.value

    def workspace(self, n_q_heads, n_splits=0):
        """A zeroed workspace for (n_q_heads, n_splits), cached on the cache object."""
        key = (n_q_heads, n_splits)
        ws = self._ws.get(key)
        if ws is None:
            ws = torch.zeros(self.workspace_bytes(n_q_heads, n_splits), dtype=torch.uint8, device=self.device)
            self._ws[key] = ws
        return ws

    def decode(self, q, scale=None, n_splits=0, out=None, lse=None, workspace=None, stream=None):
        """Decode attention: q fp32 [B, Hq, D] -> (out fp32 [B, Hq, D], lse fp32 [B, Hq])."""
        assert q.dtype == torch.float32 and q.is_contiguous() and q.dim() == 3
        B, Hq, D = q.shape
        assert B == self.batch and D == self.head_dim
        scale = 1.0 / math.sqrt(D) if scale is None else scale
        out = torch.empty_like(q) if out is None else out
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device) if lse is None else lse
        ws = self.workspace(Hq, n_splits) if workspace is None else workspace
        _check(lib.kvq_decode_attention(self.handle, _ptr(q), Hq, scale, n_splits, _ptr(ws), _ptr(out), _ptr(lse),
                                        _stream(stream)), "kvq_decode_attention")
        return out, lse

    def append_decode(self, k_new, v_new, q, scale=None, n_splits=0, out=None, lse=None, workspace=None,
                      stream=None):
        """One decode step: quantise-append k_new, v_new fp32 [B, Hkv, 1, D] (one row per
        sequence), then attend q fp32 [B, Hq, D] over the cache including them."""
        for t in (k_new, v_new, q):
            assert t.dtype == torch.float32 and t.is_contiguous()
        assert k_new.shape == v_new.shape and k_new.numel() == self.batch * self.n_kv_heads * self.head_dim
        B, Hq, D = q.shape
        assert B == self.batch and D == self.head_dim
        scale = 1.0 / math.sqrt(D) if scale is None else scale
        out = torch.empty_like(q) if out is None else out
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device) if lse is None else lse
        ws = self.workspace(Hq, n_splits) if workspace is None else workspace
        _check(lib.kvq_append_decode(self.handle, _ptr(k_new), _ptr(v_new), _ptr(q), Hq, scale, n_splits, _ptr(ws),
                                     _ptr(out), _ptr(lse), _stream(stream)), "kvq_append_decode")
        return out, lse

    def verify(self, q, scale=None, n_splits=0, out=None, lse=None, workspace=None, stream=None):
        """Draft verify: q fp32 [B, n_q, Hq, D], the last n_q cache rows being the draft;
        query i attends to positions [0, len - n_q + i].  Returns (out [B, n_q, Hq, D],
        lse [B, n_q, Hq])."""
        assert q.dtype == torch.float32 and q.is_contiguous() and q.dim() == 4
        B, n_q, Hq, D = q.shape
        assert B == self.batch and D == self.head_dim
        scale = 1.0 / math.sqrt(D) if scale is None else scale
        out = torch.empty_like(q) if out is None else out
        lse = torch.empty((B, n_q, Hq), dtype=torch.float32, device=q.device) if lse is None else lse
        if workspace is None:
            b = ctypes.c_size_t()
            _check(lib.kvq_verify_workspace_size(self.handle, n_q, Hq, n_splits, ctypes.byref(b)),
                   "kvq_verify_workspace_size")
            workspace = torch.zeros(b.value, dtype=torch.uint8, device=self.device)
        _check(lib.kvq_decode_verify(self.handle, _ptr(q), n_q, Hq, scale, n_splits, _ptr(workspace), _ptr(out),
                                     _ptr(lse), _stream(stream)), "kvq_decode_verify")
        return out, lse

    def decode_noalloc(self, q, scale=None, n_splits=0, out=None, lse=None, stream=None):
        """Decode through kvq_decode_attention_noalloc: no workspace argument; the library's
        built-in scratch array is used (see include/kvq.h for its limits)."""
        assert q.dtype == torch.float32 and q.is_contiguous() and q.dim() == 3
        B, Hq, D = q.shape
        assert B == self.batch and D == self.head_dim
        scale = 1.0 / math.sqrt(D) if scale is None else scale
        out = torch.empty_like(q) if out is None else out
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device) if lse is None else lse
        _check(lib.kvq_decode_attention_noalloc(self.handle, _ptr(q), Hq, scale, n_splits, _ptr(out), _ptr(lse),
                                                _stream(stream)), "kvq_decode_attention_noalloc")
        return out, lse

    def decode_partials(self, q, n_splits, scale=None, stream=None):
        """Split triples (o [B,Hq,S,D], m [B,Hq,S], l [B,Hq,S]) without the merge."""
        B, Hq, D = q.shape
        scale = 1.0 / math.sqrt(D) if scale is None else scale
        po = torch.empty((B, Hq, n_splits, D), dtype=torch.float32, device=q.device)
        pm = torch.empty((B, Hq, n_splits), dtype=torch.float32, device=q.device)
        pl = torch.empty((B, Hq, n_splits), dtype=torch.float32, device=q.device)
        _check(lib.kvq_decode_partials(self.handle, _ptr(q), Hq, scale, n_splits, _ptr(po), _ptr(pm), _ptr(pl),
                                       _stream(stream)), "kvq_decode_partials")
        return po, pm, pl


def combine(part_o, part_m, part_l, out=None, lse=None, stream=None):
    """Merge split triples: part_o [..., S, D], part_m/part_l [..., S] -> (out [..., D], lse [...])."""
    S, D = part_o.shape[-2], part_o.shape[-1]
    lead = part_o.shape[:-2]
    rows = int(math.prod(lead))
    out = torch.empty(lead + (D,), dtype=torch.float32, device=part_o.device) if out is None else out
    lse = torch.empty(lead, dtype=torch.float32, device=part_o.device) if lse is None else lse
    _check(lib.kvq_combine(_ptr(part_o), _ptr(part_m), _ptr(part_l), rows, S, D, _ptr(out), _ptr(lse),
                           _stream(stream)), "kvq_combine")
    return out, lse
