"""ctypes binding of libkvq.so (include/kvq.h): argument marshalling only.

Every step of the decode path runs in the library's CUDA kernels; torch only
provides device memory and the stream handle.  Importing this module does not
load the library; the first call does, and raises if libkvq.so is missing --
there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading
from ctypes import POINTER, c_float, c_int32, c_size_t, c_void_p

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkvq.so")

KVQ_OK = 0
KVQ_ERR_INVALID_ARG = 1
KVQ_ERR_UNSUPPORTED = 2
KVQ_ERR_CAPACITY = 3
KVQ_ERR_WORKSPACE = 4
KVQ_ERR_CUDA = 5
KVQ_ERR_TIMEOUT = 6
V_Q4_0 = 0
V_Q8_0 = 1
K_I8 = 0    # K: int8 codes + fp16 scale per 32 (query quantized the same way)
K_F16 = 1   # K: fp16 values (query unquantized)
LAYOUT_TILES = 0   # segment code bytes in 16-token tiles, fragment order
LAYOUT_ROWS = 1    # one row per token in element order
HEAD_DIM = 128
SEG_ALIGN = 64
QBLOCK = 32

EXPORTED = ("kvq_append", "kvq_decode_attn", "kvq_decode_workspace_size", "kvq_decode_attn_multi",
            "kvq_decode_multi_workspace_size", "kvq_decode_attn_noalloc", "kvq_wait_timeouts",
            "kvq_reset_wait_timeouts", "kvq_status_string", "kvq_debug_qk", "kvq_debug_lose_stage",
            "kvq_debug_plan", "kvq_layout_model_default", "kvq_layout_cost", "kvq_choose_layout")
MAX_CALLS = 16
MAX_T_Q = 4096
MAX_T_Q_APPEND = 8
NOALLOC_SCRATCH_BYTES = 32 << 20


class KvqSegment(ctypes.Structure):
    _fields_ = [("k_q", c_void_p), ("k_s", c_void_p), ("v_q", c_void_p), ("v_s", c_void_p),
                ("cap", c_int32), ("len", c_int32), ("pos0", c_int32), ("layout", c_int32)]


class KvqCache(ctypes.Structure):
    _fields_ = [("n_seqs", c_int32), ("n_kv_heads", c_int32), ("head_dim", c_int32),
                ("v_type", c_int32), ("max_segs", c_int32), ("n_segs", POINTER(c_int32)),
                ("segs", POINTER(KvqSegment)), ("k_type", c_int32), ("reserved", c_int32)]


class KvqDecodeDesc(ctypes.Structure):
    _fields_ = [("cache", POINTER(KvqCache)), ("q16", c_void_p), ("n_q_heads", c_int32), ("t_q", c_int32),
                ("causal_tail", c_int32), ("seq_lens", c_void_p), ("max_len", c_int32),
                ("head_map", POINTER(c_int32)), ("sm_scale", c_float), ("out", c_void_p), ("lse", c_void_p),
                ("k16_new", c_void_p), ("v16_new", c_void_p)]


class KvqLayoutModel(ctypes.Structure):
    _fields_ = [("us_per_byte", ctypes.c_double), ("us_per_op", ctypes.c_double),
                ("ops_rows_per_tile", ctypes.c_double)]


class KvqPlanLaunch(ctypes.Structure):
    _fields_ = [("kernel", c_int32), ("n_tiles8", c_int32), ("warps", c_int32), ("chunk", c_int32),
                ("chunk0", c_int32), ("n_ctas", c_int32), ("n_rows", c_int32)]


class KvqError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s failed: %s (%d)" % (what, status_string(status), status))


_lib = None
_lock = threading.Lock()


def load():
    """Load libkvq.so (built by ``__graft_entry__.build()``)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError("libkvq.so is not built (%s); run __graft_entry__.build()" % LIB_PATH)
            lib = ctypes.CDLL(LIB_PATH)
            lib.kvq_status_string.restype = ctypes.c_char_p
            lib.kvq_status_string.argtypes = [c_int32]
            lib.kvq_append.restype = c_int32
            lib.kvq_append.argtypes = [POINTER(KvqCache), c_int32, POINTER(c_int32), POINTER(c_int32),
                                       c_void_p, c_void_p, c_void_p]
            lib.kvq_decode_attn.restype = c_int32
            lib.kvq_decode_attn.argtypes = [POINTER(KvqCache), c_void_p, c_int32, c_int32, c_int32, c_void_p,
                                            c_int32, POINTER(c_int32), c_float, c_void_p, c_void_p, c_void_p,
                                            c_size_t, c_void_p]
            lib.kvq_decode_workspace_size.restype = c_int32
            lib.kvq_decode_workspace_size.argtypes = [POINTER(KvqCache), c_int32, c_int32, c_int32,
                                                      POINTER(c_int32), POINTER(c_size_t)]
            lib.kvq_decode_attn_multi.restype = c_int32
            lib.kvq_decode_attn_multi.argtypes = [c_int32, POINTER(KvqDecodeDesc), c_void_p, c_size_t, c_void_p]
            lib.kvq_decode_multi_workspace_size.restype = c_int32
            lib.kvq_decode_multi_workspace_size.argtypes = [c_int32, POINTER(KvqDecodeDesc), POINTER(c_size_t)]
            lib.kvq_decode_attn_noalloc.restype = c_int32
            lib.kvq_decode_attn_noalloc.argtypes = [POINTER(KvqCache), c_void_p, c_int32, c_int32, c_int32,
                                                    c_void_p, c_int32, POINTER(c_int32), c_float, c_void_p,
                                                    c_void_p, c_void_p]
            lib.kvq_wait_timeouts.restype = c_int32
            lib.kvq_wait_timeouts.argtypes = [POINTER(ctypes.c_uint32)]
            lib.kvq_reset_wait_timeouts.restype = c_int32
            lib.kvq_reset_wait_timeouts.argtypes = []
            lib.kvq_layout_model_default.restype = c_int32
            lib.kvq_layout_model_default.argtypes = [POINTER(KvqLayoutModel)]
            lib.kvq_layout_cost.restype = c_int32
            lib.kvq_layout_cost.argtypes = [c_int32, c_int32, c_int32, POINTER(KvqLayoutModel),
                                            POINTER(ctypes.c_double)]
            lib.kvq_choose_layout.restype = c_int32
            lib.kvq_choose_layout.argtypes = [c_int32, c_int32, c_int32, POINTER(KvqLayoutModel), POINTER(c_int32)]
            lib.kvq_debug_lose_stage.restype = c_int32
            lib.kvq_debug_lose_stage.argtypes = lib.kvq_decode_attn.argtypes
            lib.kvq_debug_qk.restype = c_int32
            lib.kvq_debug_qk.argtypes = [POINTER(KvqCache), c_void_p, c_int32, c_int32, c_void_p, c_int32,
                                         POINTER(c_int32), c_void_p, c_void_p, c_void_p, POINTER(c_int32),
                                         c_void_p]
            lib.kvq_debug_plan.restype = c_int32
            lib.kvq_debug_plan.argtypes = [c_int32, POINTER(KvqDecodeDesc), c_int32, POINTER(c_int32),
                                           POINTER(KvqPlanLaunch), c_int32, POINTER(c_int32), POINTER(c_size_t),
                                           POINTER(c_int32)]
            _lib = lib
    return _lib


def status_string(s: int) -> str:
    return load().kvq_status_string(int(s)).decode()


def _ptr(t):
    return None if t is None else c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _i32(vals):
    vals = [int(v) for v in vals]
    return (c_int32 * max(1, len(vals)))(*vals)


class Cache:
    """A batch of append-only segmented caches (device memory from torch).

    Holds the host descriptor of include/kvq.h and keeps the segment tensors
    alive.  Segment arrays are allocated with the byte layout of kvq_segment.
    """

    def __init__(self, n_seqs: int, n_kv_heads: int, v_type: int, max_segs: int = 8,
                 head_dim: int = HEAD_DIM, device=None, k_type: int = K_I8):
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.n_seqs, self.n_kv_heads, self.v_type, self.head_dim = n_seqs, n_kv_heads, v_type, head_dim
        self.k_type = k_type
        self.max_segs = max_segs
        self._segs = (KvqSegment * max(1, n_seqs * max_segs))()
        self._nsegs = (c_int32 * max(1, n_seqs))()
        self.desc = KvqCache(n_seqs, n_kv_heads, head_dim, v_type, max_segs,
                             ctypes.cast(self._nsegs, POINTER(c_int32)),
                             ctypes.cast(self._segs, POINTER(KvqSegment)), k_type, 0)
        self.tensors = [[] for _ in range(n_seqs)]

    def seg(self, b: int, k: int) -> KvqSegment:
        return self._segs[b * self.max_segs + k]

    def n_segs(self, b: int) -> int:
        return self._nsegs[b]

    def add_segment(self, b: int, cap: int, layout=LAYOUT_TILES):
        """Open a new segment of `cap` tokens (rounded up to 64) for sequence b,
        its code bytes in `layout` (LAYOUT_TILES, LAYOUT_ROWS, or "auto": the
        layout kvq_choose_layout picks for `cap` expected tokens)."""
        if layout == "auto":
            layout = choose_layout(self.k_type, self.v_type, max(1, int(cap)))
        ns = self._nsegs[b]
        if ns >= self.max_segs:
            raise ValueError("sequence %d already has max_segs segments" % b)
        cap = max(SEG_ALIGN, (int(cap) + SEG_ALIGN - 1) // SEG_ALIGN * SEG_ALIGN)
        H, D = self.n_kv_heads, self.head_dim
        vb = D // 2 if self.v_type == V_Q4_0 else D
        f16k = self.k_type == K_F16
        t = dict(k_q=torch.empty((H, cap, D), dtype=torch.int16 if f16k else torch.int8, device=self.device),
                 k_s=None if f16k else torch.empty((H, cap, D // QBLOCK), dtype=torch.int16, device=self.device),
                 v_q=torch.empty((H, cap, vb), dtype=torch.uint8, device=self.device),
                 v_s=torch.empty((H, cap, D // QBLOCK), dtype=torch.int16, device=self.device))
        pos0 = 0
        if ns:
            prev = self.seg(b, ns - 1)
            pos0 = prev.pos0 + prev.len
        s = self.seg(b, ns)
        s.k_q, s.k_s, s.v_q, s.v_s = (0 if t[n] is None else t[n].data_ptr() for n in ("k_q", "k_s", "v_q", "v_s"))
        s.cap, s.len, s.pos0, s.layout = cap, 0, pos0, int(layout)
        self.tensors[b].append(t)
        self._nsegs[b] = ns + 1
        return t

    def length(self, b: int) -> int:
        ns = self._nsegs[b]
        if not ns:
            return 0
        s = self.seg(b, ns - 1)
        return s.pos0 + s.len

    def lengths(self):
        return [self.length(b) for b in range(self.n_seqs)]

    def export(self, b: int, raw: bool = False):
        """Sequence b copied to host numpy arrays.  raw=False: the filled
        positions, [H][L][row] per array in logical row order.  raw=True: one
        dict per segment with the whole arrays as stored ([H][cap][row], code
        bytes in their in-tile order for tile-layout segments) plus its "len"
        and "layout".  F16 K caches give "k16" (fp16 bits) instead of "kq" and
        "ks"."""
        import numpy as np
        f16k = self.k_type == K_F16
        arrays = ((("k16", "k_q", np.uint16),) if f16k else (("kq", "k_q", np.uint8), ("ks", "k_s", np.uint16))) + \
            (("vq", "v_q", np.uint8), ("vs", "v_s", np.uint16))
        parts = {n: [] for n, _, _ in arrays}
        segs = []
        for k in range(self._nsegs[b]):
            s, t = self.seg(b, k), self.tensors[b][k]
            seg = {"len": s.len, "layout": s.layout}
            for name, key, view in arrays:
                a = t[key].cpu().numpy().view(view)
                seg[name] = a
                if not raw and name in ("kq", "vq", "k16") and s.layout == LAYOUT_TILES:
                    a = untile_codes(a, name, self.v_type)
                parts[name].append(a[:, :s.len])
            segs.append(seg)
        if raw:
            return segs
        return {n: np.concatenate(v, axis=1) for n, v in parts.items()}


def _tile_index(name: str, v_type: int):
    """idx[u, j] = in-tile offset of byte j of the tile's token u (the tile
    layout of include/kvq.h, head_dim 128)."""
    import numpy as np
    u = np.arange(16)[:, None]
    sub, gu, e = u // 8, u % 8, u % 2
    cu = gu // 2
    if name == "k16":   # fp16 elements (offsets in 2-byte units)
        j = np.arange(128)[None, :]
        return ((j // 16) * 512 + (4 * gu + (j % 8) // 2) * 16 + 4 * (sub + 2 * ((j % 16) // 8)) + 2 * (j % 2)) // 2
    if name == "kq":
        j = np.arange(128)[None, :]
        return ((2 * sub + j // 64) * 32 + 4 * gu + (j % 32) // 8) * 16 + 8 * ((j // 32) % 2) + j % 8
    if v_type == V_Q4_0:
        j = np.arange(64)[None, :]
        return (sub * 32 + 4 * ((j % 16) // 2) + cu) * 16 + 4 * (j // 16) + 2 * e + j % 2
    j = np.arange(128)[None, :]
    return (((2 * sub + j // 64) * 32 + 4 * ((j % 32) // 4) + cu) * 16 + 8 * ((j // 32) % 2)
            + 4 * ((j % 4) // 2) + 2 * (j % 2) + e)


def untile_codes(a, name: str, v_type: int):
    """Stored code bytes [H][cap][row] -> logical row order (cap % 16 == 0)."""
    H, cap, row = a.shape
    idx = _tile_index(name, v_type)
    tiles = a.reshape(H, cap // 16, 16 * row)
    return tiles[:, :, idx].reshape(H, cap, row)


def kvq_append(cache: Cache, seq_ids, n_new, k16: torch.Tensor, v16: torch.Tensor, stream=None) -> None:
    """kvq_append of include/kvq.h.  k16/v16: fp16 [sum(n_new)][Hkv][D] on the device."""
    ids, nn = list(seq_ids), list(n_new)
    st = load().kvq_append(ctypes.byref(cache.desc), len(ids), _i32(ids), _i32(nn), _ptr(k16), _ptr(v16),
                           _stream(stream))
    if st:
        raise KvqError(st, "kvq_append")


def kvq_decode_workspace_size(cache: Cache, n_q_heads: int, t_q: int, max_len: int, head_map=None) -> int:
    """Bytes of workspace kvq_decode_attn needs for these arguments."""
    size = c_size_t(0)
    hm = None if head_map is None else _i32(head_map)
    st = load().kvq_decode_workspace_size(ctypes.byref(cache.desc), n_q_heads, t_q, max_len, hm,
                                          ctypes.byref(size))
    if st:
        raise KvqError(st, "kvq_decode_workspace_size")
    return size.value


def kvq_decode_attn(cache: Cache, q16: torch.Tensor, n_q_heads: int, t_q: int, causal_tail: bool,
                    seq_lens: torch.Tensor, max_len: int, head_map, sm_scale: float, out: torch.Tensor,
                    lse: torch.Tensor, workspace: torch.Tensor | None, stream=None) -> None:
    """kvq_decode_attn of include/kvq.h (workspace: a uint8 device tensor of at
    least kvq_decode_workspace_size() bytes, or None when that size is 0)."""
    hm = None if head_map is None else _i32(head_map)
    st = load().kvq_decode_attn(ctypes.byref(cache.desc), _ptr(q16), n_q_heads, t_q, int(causal_tail),
                                _ptr(seq_lens), max_len, hm, float(sm_scale), _ptr(out), _ptr(lse),
                                _ptr(workspace), 0 if workspace is None else workspace.numel(),
                                _stream(stream))
    if st:
        raise KvqError(st, "kvq_decode_attn")


def _descs(calls):
    """calls: sequence of dicts with the per-cache arguments of kvq_decode_attn
    (cache, q16, n_q_heads, t_q, causal_tail, seq_lens, max_len, head_map,
    sm_scale, out, lse) and optionally k16_new / v16_new (fused append);
    tensors may be None for a size query."""
    arr = (KvqDecodeDesc * max(1, len(calls)))()
    keep = []
    for i, c in enumerate(calls):
        hm = c.get("head_map")
        hm_arr = None if hm is None else _i32(hm)
        keep.append(hm_arr)
        arr[i] = KvqDecodeDesc(ctypes.pointer(c["cache"].desc), _ptr(c.get("q16")), c["n_q_heads"], c["t_q"],
                               int(c.get("causal_tail", False)), _ptr(c.get("seq_lens")), c["max_len"],
                               ctypes.cast(hm_arr, POINTER(c_int32)) if hm_arr is not None else None,
                               float(c.get("sm_scale", 1.0)), _ptr(c.get("out")), _ptr(c.get("lse")),
                               _ptr(c.get("k16_new")), _ptr(c.get("v16_new")))
    return arr, keep


def kvq_decode_multi_workspace_size(calls) -> int:
    """Bytes of workspace kvq_decode_attn_multi needs for these calls."""
    arr, keep = _descs(calls)
    size = c_size_t(0)
    st = load().kvq_decode_multi_workspace_size(len(calls), arr, ctypes.byref(size))
    if st:
        raise KvqError(st, "kvq_decode_multi_workspace_size")
    return int(size.value)


def kvq_decode_attn_multi(calls, workspace, stream=None) -> None:
    """kvq_decode_attn_multi of include/kvq.h: several decode calls (list of
    dicts, see _descs) in one launch."""
    arr, keep = _descs(calls)
    st = load().kvq_decode_attn_multi(len(calls), arr, _ptr(workspace), 0 if workspace is None else workspace.numel(),
                                      _stream(stream))
    if st:
        raise KvqError(st, "kvq_decode_attn_multi")


class MultiCall:
    """A prepared kvq_decode_attn_multi: the descriptor array is built once and
    each call only passes the stream (the caches' host tables are read at call
    time, so appends between calls are seen)."""

    def __init__(self, calls, workspace=None):
        self.calls = list(calls)
        self.arr, self._keep = _descs(self.calls)
        self.ws = workspace

    def workspace_size(self) -> int:
        size = c_size_t(0)
        st = load().kvq_decode_multi_workspace_size(len(self.calls), self.arr, ctypes.byref(size))
        if st:
            raise KvqError(st, "kvq_decode_multi_workspace_size")
        return int(size.value)

    def __call__(self, stream=None):
        ws = self.ws
        st = load().kvq_decode_attn_multi(len(self.calls), self.arr, _ptr(ws), 0 if ws is None else ws.numel(),
                                          _stream(stream))
        if st:
            raise KvqError(st, "kvq_decode_attn_multi")


def kvq_decode_attn_noalloc(cache: Cache, q16: torch.Tensor, n_q_heads: int, t_q: int, causal_tail: bool,
                            seq_lens: torch.Tensor, max_len: int, head_map, sm_scale: float, out: torch.Tensor,
                            lse: torch.Tensor, stream=None) -> None:
    """kvq_decode_attn_noalloc of include/kvq.h: no workspace argument; the split
    partials use the library's fixed device scratch (see the header for the
    size limit, the first-call set-up and the no-overlap rule)."""
    hm = None if head_map is None else _i32(head_map)
    st = load().kvq_decode_attn_noalloc(ctypes.byref(cache.desc), _ptr(q16), n_q_heads, t_q, int(causal_tail),
                                        _ptr(seq_lens), max_len, hm, float(sm_scale), _ptr(out), _ptr(lse),
                                        _stream(stream))
    if st:
        raise KvqError(st, "kvq_decode_attn_noalloc")


DUMP_KERNELS = ("split", "tcgen05")


def kvq_debug_qk(cache: Cache, q16, n_q_heads, t_q, seq_lens, max_len, head_map, q_codes, q_scales, scores,
                 stream=None) -> str:
    """kvq_debug_qk test hook of include/kvq.h; returns the kernel that
    produced the dumps ("split" or "tcgen05")."""
    hm = None if head_map is None else _i32(head_map)
    kern = c_int32(-1)
    st = load().kvq_debug_qk(ctypes.byref(cache.desc), _ptr(q16), n_q_heads, t_q, _ptr(seq_lens), max_len, hm,
                             _ptr(q_codes), _ptr(q_scales), _ptr(scores), ctypes.byref(kern), _stream(stream))
    if st:
        raise KvqError(st, "kvq_debug_qk")
    return DUMP_KERNELS[kern.value]


def kvq_wait_timeouts() -> int:
    """kvq_wait_timeouts of include/kvq.h: the device's count of attention-kernel
    copy waits that gave up (0 in every correct run)."""
    n = ctypes.c_uint32(0)
    st = load().kvq_wait_timeouts(ctypes.byref(n))
    if st not in (0, KVQ_ERR_TIMEOUT):
        raise KvqError(st, "kvq_wait_timeouts")
    return int(n.value)


def layout_model_default() -> KvqLayoutModel:
    """kvq_layout_model_default of include/kvq.h."""
    m = KvqLayoutModel()
    st = load().kvq_layout_model_default(ctypes.byref(m))
    if st:
        raise KvqError(st, "kvq_layout_model_default")
    return m


def layout_cost(layout: int, v_type: int, n_tokens: int, model: KvqLayoutModel | None = None) -> float:
    """kvq_layout_cost of include/kvq.h (microseconds per kv head)."""
    c = ctypes.c_double(0.0)
    st = load().kvq_layout_cost(layout, v_type, n_tokens, None if model is None else ctypes.byref(model),
                                ctypes.byref(c))
    if st:
        raise KvqError(st, "kvq_layout_cost")
    return c.value


def choose_layout(k_type: int, v_type: int, n_tokens: int, model: KvqLayoutModel | None = None) -> int:
    """kvq_choose_layout of include/kvq.h."""
    out = c_int32(-1)
    st = load().kvq_choose_layout(k_type, v_type, n_tokens, None if model is None else ctypes.byref(model),
                                  ctypes.byref(out))
    if st:
        raise KvqError(st, "kvq_choose_layout")
    return out.value


def kvq_reset_wait_timeouts() -> None:
    """kvq_reset_wait_timeouts of include/kvq.h."""
    st = load().kvq_reset_wait_timeouts()
    if st:
        raise KvqError(st, "kvq_reset_wait_timeouts")


def kvq_debug_lose_stage(cache: Cache, q16: torch.Tensor, n_q_heads: int, t_q: int, causal_tail: bool,
                         seq_lens: torch.Tensor, max_len: int, head_map, sm_scale: float, out: torch.Tensor,
                         lse: torch.Tensor, workspace: torch.Tensor | None, stream=None) -> None:
    """kvq_debug_lose_stage test hook of include/kvq.h (arguments as
    kvq_decode_attn)."""
    hm = None if head_map is None else _i32(head_map)
    st = load().kvq_debug_lose_stage(ctypes.byref(cache.desc), _ptr(q16), n_q_heads, t_q, int(causal_tail),
                                     _ptr(seq_lens), max_len, hm, float(sm_scale), _ptr(out), _ptr(lse),
                                     _ptr(workspace), 0 if workspace is None else workspace.numel(),
                                     _stream(stream))
    if st:
        raise KvqError(st, "kvq_debug_lose_stage")


PLAN_KERNELS = ("split", "prefill")


def kvq_debug_plan(calls, n_sms: int, ctas_per_sm=(1, 2, 2, 2), max_out: int = 64):
    """kvq_debug_plan of include/kvq.h (test hook): the launches the decode
    call would make for `calls` (dicts as for kvq_decode_attn_multi; only the
    caches' host descriptors are read) on a described device.  Returns
    (launches as dicts, workspace bytes); the calls whose step tokens get an
    append launch of their own first are in kvq_debug_plan.n_pre_appends."""
    arr, keep = _descs(calls)
    ctas = _i32(ctas_per_sm)
    out = (KvqPlanLaunch * max(1, max_out))()
    n_out, ws, n_pre = c_int32(0), c_size_t(0), c_int32(0)
    st = load().kvq_debug_plan(len(calls), arr, int(n_sms), ctas, out, max_out, ctypes.byref(n_out),
                               ctypes.byref(ws), ctypes.byref(n_pre))
    kvq_debug_plan.n_pre_appends = int(n_pre.value)
    if st:
        raise KvqError(st, "kvq_debug_plan")
    launches = [dict(kernel=PLAN_KERNELS[r.kernel], n_tiles8=r.n_tiles8, warps=r.warps, chunk=r.chunk,
                     chunk0=r.chunk0, n_ctas=r.n_ctas, n_rows=r.n_rows) for r in out[:min(n_out.value, max_out)]]
    return launches, int(ws.value)
