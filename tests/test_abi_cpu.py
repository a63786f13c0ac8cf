"""The C ABI without a GPU: the library builds, loads, exports every function
include/kvq.h declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

from quantized_kv_cache_03_gb300 import build as B
from quantized_kv_cache_03_gb300 import kvq

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "kvq.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return kvq.load()


def declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s*(kvq_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_api():
    assert declared() == sorted(kvq.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in declared():
        assert hasattr(lib, name), name
    assert kvq.status_string(kvq.KVQ_ERR_CAPACITY) == "segment capacity exceeded"


def _fake_cache(n_seqs=2, H=2, vt=0, cap=128, lens=(100, 64), head_dim=128, max_segs=2, addr=0x10000):
    segs = (kvq.KvqSegment * (n_seqs * max_segs))()
    ns = (ctypes.c_int32 * n_seqs)()
    for b in range(n_seqs):
        ns[b] = 1
        s = segs[b * max_segs]
        s.k_q = s.k_s = s.v_q = s.v_s = addr
        s.cap, s.len, s.pos0 = cap, lens[b], 0
    c = kvq.KvqCache(n_seqs, H, head_dim, vt, max_segs, ctypes.cast(ns, ctypes.POINTER(ctypes.c_int32)),
                     ctypes.cast(segs, ctypes.POINTER(kvq.KvqSegment)))
    c._keep = (segs, ns)
    return c


def _decode(lib, c, Hq=4, t_q=1, head_map=None, max_len=128, ws=0):
    hm = None if head_map is None else (ctypes.c_int32 * len(head_map))(*head_map)
    return lib.kvq_decode_attn(ctypes.byref(c), ctypes.c_void_p(0x20000), Hq, t_q, 0, ctypes.c_void_p(0x30000),
                               max_len, hm, 0.1, ctypes.c_void_p(0x40000), ctypes.c_void_p(0x50000), None, ws, None)


def _append(lib, c, ids, nn):
    a = (ctypes.c_int32 * len(ids))(*ids)
    n = (ctypes.c_int32 * len(nn))(*nn)
    return lib.kvq_append(ctypes.byref(c), len(ids), a, n, ctypes.c_void_p(0x60000), ctypes.c_void_p(0x70000), None)


def test_decode_argument_errors(lib):
    assert lib.kvq_decode_attn(None, None, 4, 1, 0, None, 1, None, 0.1, None, None, None, 0, None) == kvq.KVQ_ERR_INVALID_ARG
    assert _decode(lib, _fake_cache(head_dim=64)) == kvq.KVQ_ERR_UNSUPPORTED
    assert _decode(lib, _fake_cache(head_dim=100)) == kvq.KVQ_ERR_INVALID_ARG
    assert _decode(lib, _fake_cache(cap=100)) == kvq.KVQ_ERR_INVALID_ARG          # cap not a multiple of 64
    assert _decode(lib, _fake_cache(lens=(200, 1))) == kvq.KVQ_ERR_INVALID_ARG    # len > cap
    assert _decode(lib, _fake_cache(addr=0x10008)) == kvq.KVQ_ERR_INVALID_ARG     # misaligned segment
    assert _decode(lib, _fake_cache(vt=7)) == kvq.KVQ_ERR_INVALID_ARG
    c = _fake_cache()
    assert _decode(lib, c, t_q=0) == kvq.KVQ_ERR_INVALID_ARG
    assert _decode(lib, c, t_q=kvq.MAX_T_Q + 1) == kvq.KVQ_ERR_INVALID_ARG
    assert _decode(lib, c, Hq=5) == kvq.KVQ_ERR_INVALID_ARG                       # 5 % 2 != 0 without a map
    assert _decode(lib, c, Hq=3, head_map=[0, 2, 1]) == kvq.KVQ_ERR_INVALID_ARG   # kv head out of range
    assert _decode(lib, c, max_len=-1) == kvq.KVQ_ERR_INVALID_ARG


def test_pos0_chain_is_checked(lib):
    c = _fake_cache(n_seqs=1, max_segs=2)
    ns = c._keep[1]
    segs = c._keep[0]
    ns[0] = 2
    segs[1].k_q = segs[1].k_s = segs[1].v_q = segs[1].v_s = 0x10000
    segs[1].cap, segs[1].len, segs[1].pos0 = 64, 3, 99                          # should be 100
    assert _decode(lib, c) == kvq.KVQ_ERR_INVALID_ARG
    segs[1].pos0 = 100
    st = _decode(lib, c)
    assert st in (kvq.KVQ_ERR_UNSUPPORTED, kvq.KVQ_OK)


def test_append_errors_leave_state_unchanged(lib):
    c = _fake_cache()
    segs = c._keep[0]
    assert _append(lib, c, [0], [29]) == kvq.KVQ_ERR_CAPACITY                   # 100 + 29 > 128
    assert _append(lib, c, [0, 0], [1, 1]) == kvq.KVQ_ERR_INVALID_ARG            # duplicate sequence
    assert _append(lib, c, [2], [1]) == kvq.KVQ_ERR_INVALID_ARG                  # no such sequence
    assert _append(lib, c, [1], [-1]) == kvq.KVQ_ERR_INVALID_ARG
    assert _append(lib, c, [0, 1], [0, 0]) == kvq.KVQ_OK                         # nothing to do
    assert segs[0].len == 100 and segs[2].len == 64


@pytest.mark.skipif(os.path.exists("/dev/nvidia0"), reason="checks the no-GPU path")
def test_no_device_is_reported(lib):
    c = _fake_cache()
    assert _decode(lib, c) == kvq.KVQ_ERR_UNSUPPORTED
    assert _append(lib, c, [0], [1]) == kvq.KVQ_ERR_UNSUPPORTED
    assert c._keep[0][0].len == 100


def _desc(c, Hq=4, t_q=1, max_len=128):
    return kvq.KvqDecodeDesc(ctypes.pointer(c), ctypes.c_void_p(0x20000), Hq, t_q, 0, ctypes.c_void_p(0x30000),
                             max_len, None, 0.1, ctypes.c_void_p(0x40000), ctypes.c_void_p(0x50000))


def test_multi_argument_errors(lib):
    c1, c2 = _fake_cache(), _fake_cache(H=4)
    arr = (kvq.KvqDecodeDesc * 2)(_desc(c1), _desc(c2, Hq=6))                  # 6 % 4 != 0 without a map
    assert lib.kvq_decode_attn_multi(2, arr, None, 0, None) == kvq.KVQ_ERR_INVALID_ARG
    assert lib.kvq_decode_attn_multi(-1, arr, None, 0, None) == kvq.KVQ_ERR_INVALID_ARG
    assert lib.kvq_decode_attn_multi(kvq.MAX_CALLS + 1, arr, None, 0, None) == kvq.KVQ_ERR_INVALID_ARG
    assert lib.kvq_decode_attn_multi(1, None, None, 0, None) == kvq.KVQ_ERR_INVALID_ARG
    assert lib.kvq_decode_attn_multi(0, None, None, 0, None) == kvq.KVQ_OK   # nothing to do
    size = ctypes.c_size_t(7)
    assert lib.kvq_decode_multi_workspace_size(2, arr, None) == kvq.KVQ_ERR_INVALID_ARG
    assert lib.kvq_decode_multi_workspace_size(2, arr, ctypes.byref(size)) == kvq.KVQ_ERR_INVALID_ARG
    arr[1].t_q = kvq.MAX_T_Q + 1
    arr[1].n_q_heads = 8
    assert lib.kvq_decode_attn_multi(2, arr, None, 0, None) == kvq.KVQ_ERR_INVALID_ARG


def test_multi_rejects_a_cache_that_receives_tokens_twice(lib):
    c = _fake_cache()
    d0, d1 = _desc(c), _desc(c)
    d1.k16_new = d1.v16_new = 0x60000
    arr = (kvq.KvqDecodeDesc * 2)(d0, d1)
    assert lib.kvq_decode_attn_multi(2, arr, None, 0, None) == kvq.KVQ_ERR_INVALID_ARG
    d1.v16_new = None                                  # k without v
    arr = (kvq.KvqDecodeDesc * 1)(d1)
    assert lib.kvq_decode_attn_multi(1, arr, None, 0, None) == kvq.KVQ_ERR_INVALID_ARG
