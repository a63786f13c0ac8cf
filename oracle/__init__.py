"""Plain fp64 CPU oracle for decode attention over a quantized KV cache.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the CUDA product path
never does, and this package imports nothing from it.

The arithmetic lives in ``kvq_oracle.c`` (plain C99, fp64, optional OpenMP over
independent query rows).  This module only compiles it with gcc and marshals
numpy arrays through ctypes.  Each function below names the passage of the
pages it follows; the C file's header states the rules and the byte layouts.

Pinned by ``tests/test_oracle_*.py`` (fp16 against numpy's correctly rounded
conversion, hand-worked quantizer blocks under ``tests/golden/``, brute-force
nearest-code search, exact integer dots, textbook fp64 softmax attention and
its special cases).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_kvq.so")
_lock = threading.Lock()
_lib = None

VT_Q4_0 = 0
VT_Q8_0 = 1
KT_I8 = 0    # K: int8 codes + fp16 scale per 32
KT_F16 = 1   # K: the fp16 values (F16 K)
QBLK = 32


def build(force: bool = False) -> str:
    """Compile kvq_oracle.c into liboracle_kvq.so next to it (gcc, -O2, OpenMP)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-fopenmp", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32 = ctypes.c_int
            lib.orc_f16_to_f64.restype = ctypes.c_double
            lib.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.orc_f64_to_f16.restype = ctypes.c_uint16
            lib.orc_f64_to_f16.argtypes = [ctypes.c_double]
            lib.orc_quant_i8_block.restype = None
            lib.orc_quant_i8_block.argtypes = [P, P, P]
            lib.orc_quant_q4_0_block.restype = None
            lib.orc_quant_q4_0_block.argtypes = [P, P, P]
            lib.orc_quantize_kv.restype = i32
            lib.orc_quantize_kv.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P]
            lib.orc_decode_seq.restype = i32
            lib.orc_decode_seq.argtypes = [
                i32, i32, i32, i32, P, P, P, P,
                i32, i32, P, i32, ctypes.c_double, P,
                P, P, P, P, P, P, i32]
            lib.orc_decode_seq_f16k.argtypes = [
                i32, i32, i32, i32, P, P, P,
                i32, i32, P, i32, ctypes.c_double, P,
                P, P, P, i32]
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------- fp16 --

def f16_to_f64(bits: int) -> float:
    """IEEE-754 binary16 bit pattern -> exact double."""
    return _load().orc_f16_to_f64(int(bits) & 0xFFFF)


def f64_to_f16(x: float) -> int:
    """double -> binary16 bit pattern, round to nearest even."""
    return int(_load().orc_f64_to_f16(float(x)))


# --------------------------------------------------------------- quantizers --

def quant_i8_block(x16: np.ndarray):
    """One 32-element fp16 block -> (int8 codes[32], fp16 scale bits).

    K payload + fp16 scale ("Flash Attention for llama.cpp on RDNA3", first
    paragraph); scale absmax/127, codes rounded half away from zero.
    """
    x = _c(x16, np.uint16)
    assert x.shape == (QBLK,)
    codes = np.zeros(QBLK, np.int8)
    scale = np.zeros(1, np.uint16)
    _load().orc_quant_i8_block(_ptr(x), _ptr(codes), _ptr(scale))
    return codes, int(scale[0])


def quant_q4_0_block(x16: np.ndarray):
    """One 32-element fp16 block -> (16 packed q4_0 bytes, fp16 scale bits).

    q4_0 V (VRAM and KLD tables of the RDNA3 page): d = absmax/8,
    q = round(x/d) + 8 clamped to [0, 15]; byte j = q[j] | q[j+16] << 4.
    """
    x = _c(x16, np.uint16)
    assert x.shape == (QBLK,)
    packed = np.zeros(QBLK // 2, np.uint8)
    scale = np.zeros(1, np.uint16)
    _load().orc_quant_q4_0_block(_ptr(x), _ptr(packed), _ptr(scale))
    return packed, int(scale[0])


def quantize_kv(k16: np.ndarray, v16: np.ndarray, v_type: int, k_type: int = KT_I8):
    """Quantize token-major fp16 K, V [n_tok][n_kv_heads][head_dim] (uint16 bit
    patterns or float16) into the head-major cache layout.

    Returns dict(kq int8 [H][n][D], ks uint16 [H][n][D/32],
                 vq uint8 [H][n][D/2 or D], vs uint16 [H][n][D/32]); with
    k_type KT_F16 ("F16 K" of the RDNA3 page's title and KLD tables) K is kept
    as its fp16 bits, k16 uint16 [H][n][D], instead of kq / ks.
    """
    k = _c(np.asarray(k16).view(np.uint16), np.uint16)
    v = _c(np.asarray(v16).view(np.uint16), np.uint16)
    n, H, D = k.shape
    assert v.shape == k.shape
    vb = D // 2 if v_type == VT_Q4_0 else D
    out = dict(kq=np.zeros((H, n, D), np.int8), ks=np.zeros((H, n, D // QBLK), np.uint16),
               vq=np.zeros((H, n, vb), np.uint8), vs=np.zeros((H, n, D // QBLK), np.uint16))
    rc = _load().orc_quantize_kv(n, H, D, v_type, _ptr(k), _ptr(v), _ptr(out["kq"]),
                                 _ptr(out["ks"]), _ptr(out["vq"]), _ptr(out["vs"]))
    if rc:
        raise ValueError("orc_quantize_kv failed (%d)" % rc)
    if k_type == KT_F16:
        del out["kq"], out["ks"]
        out["k16"] = np.ascontiguousarray(k.transpose(1, 0, 2))
    return out


def decode_seq(cache: dict, q16: np.ndarray, head_map, causal: bool, sm_scale: float,
               v_type: int, want_codes: bool = False, want_scores: bool = False,
               row_mask=None, n_threads: int = 1):
    """Decode attention of one sequence over its quantized cache.

    ``cache`` holds the arrays of :func:`quantize_kv` for positions 0..L-1;
    ``q16`` is [t_q][n_q_heads][head_dim] fp16 (bits or float16).  Returns
    dict(out fp64 [t_q][Hq][D], lse fp64 [t_q][Hq]) plus, on request, the Q
    codes/scales and the exact per-block integer scores I [t_q][Hq][L][D/32].
    """
    if "k16" in cache:
        if want_codes or want_scores:
            raise ValueError("an F16-K cache has no Q codes or integer block scores")
        return _decode_seq_f16k(cache, q16, head_map, causal, sm_scale, v_type, row_mask, n_threads)
    kq, ks, vq, vs = (_c(cache["kq"], np.int8), _c(cache["ks"], np.uint16),
                      _c(cache["vq"], np.uint8), _c(cache["vs"], np.uint16))
    H, L, D = kq.shape
    q = _c(np.asarray(q16).view(np.uint16), np.uint16)
    t_q, Hq, Dq = q.shape
    assert Dq == D
    hm = _c(head_map, np.int32)
    nb = D // QBLK
    res = dict(out=np.zeros((t_q, Hq, D), np.float64), lse=np.zeros((t_q, Hq), np.float64))
    qc = qs = sc = None
    if want_codes:
        qc = res["q_codes"] = np.zeros((t_q, Hq, D), np.int8)
        qs = res["q_scales"] = np.zeros((t_q, Hq, nb), np.uint16)
    if want_scores:
        sc = res["scores"] = np.zeros((t_q, Hq, L, nb), np.int64)
    rm = None if row_mask is None else _c(row_mask, np.uint8)
    rc = _load().orc_decode_seq(L, H, D, v_type, _ptr(kq), _ptr(ks), _ptr(vq), _ptr(vs),
                                t_q, Hq, _ptr(hm), int(bool(causal)), float(sm_scale), _ptr(q),
                                _ptr(res["out"]), _ptr(res["lse"]), _ptr(qc), _ptr(qs), _ptr(sc),
                                _ptr(rm), int(n_threads))
    if rc:
        raise ValueError("orc_decode_seq failed (%d)" % rc)
    return res


def _decode_seq_f16k(cache, q16, head_map, causal, sm_scale, v_type, row_mask, n_threads):
    """Decode attention over an F16-K cache (quantize_kv with KT_F16): the
    score is sm_scale * q.k over the fp16 values, Q not quantized."""
    k, vq, vs = _c(cache["k16"], np.uint16), _c(cache["vq"], np.uint8), _c(cache["vs"], np.uint16)
    H, L, D = k.shape
    q = _c(np.asarray(q16).view(np.uint16), np.uint16)
    t_q, Hq, Dq = q.shape
    assert Dq == D
    hm = _c(head_map, np.int32)
    res = dict(out=np.zeros((t_q, Hq, D), np.float64), lse=np.zeros((t_q, Hq), np.float64))
    rm = None if row_mask is None else _c(row_mask, np.uint8)
    rc = _load().orc_decode_seq_f16k(L, H, D, v_type, _ptr(k), _ptr(vq), _ptr(vs), t_q, Hq, _ptr(hm),
                                     int(bool(causal)), float(sm_scale), _ptr(q), _ptr(res["out"]),
                                     _ptr(res["lse"]), _ptr(rm), int(n_threads))
    if rc:
        raise ValueError("orc_decode_seq_f16k failed (%d)" % rc)
    return res


def default_head_map(n_q_heads: int, n_kv_heads: int) -> np.ndarray:
    """Contiguous GQA groups: query head h reads kv head h // (Hq/Hkv)."""
    g = n_q_heads // n_kv_heads
    return (np.arange(n_q_heads) // g).astype(np.int32)


def bytes_per_token_head(head_dim: int, v_type: int) -> dict:
    """Stored bytes per (token, kv head): 8-bit K payload + fp16 scale per 32,
    and the V block format (q4_0: 16 B + 2 B per 32; q8_0: 32 B + 2 B per 32)."""
    nb = head_dim // QBLK
    k = head_dim + 2 * nb
    v = (head_dim // 2 if v_type == VT_Q4_0 else head_dim) + 2 * nb
    return dict(k=k, v=v, total=k + v)
