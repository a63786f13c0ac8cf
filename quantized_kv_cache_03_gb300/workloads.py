"""Seeded synthetic workloads for decode attention over a quantized KV cache.

This module only draws inputs: fp16 Q, K and V, sequence lengths and segment
cut points.  It holds none of the method's arithmetic (no quantization, no
attention), so both the CUDA path and the CPU oracle can be fed from it.

Recipes (all draws from numpy's PCG64, seeded per stream so that any one
sequence can be regenerated on its own):

* ``tiny``     batch 1, 1 kv head, 4 query heads, head_dim 128, 256 positions,
               1 query token, V q8_0, Q/K/V ~ N(0,1), seed 0.
* ``single``   batch 1, 32 query / 8 kv heads, 8192 positions, 1 query token,
               V q4_0; 4 distinct channels per kv head drawn from the seed have
               K and V multiplied by 10 (Q unscaled), seed 1.
* ``long``     two independent caches decoded in the same step (main + draft):
               main 40 query / 8 kv heads (seed 2), draft 16 query / 4 kv heads
               (seed 3); 131072 positions each, built in 4 append-only segments
               whose 3 cut points are distinct integers uniform in [1, L-1];
               V q4_0, N(0,1), 1 query token.
* ``batched``  64 sequences, lengths uniform integers in [1024, 32768] (seed 4),
               32 query / 8 kv heads, 1 query token, V q8_0, 4 outlier
               channels per kv head x10 on K and V.
* ``verify``   16 sequences x 4 query tokens with a causal mask among the 4
               newest positions, 32768 positions each, 64 query / 8 kv heads
               (32 query rows per kv head), V q4_0, N(0,1), seed 5.
* ``long_f16k`` the ``long`` pair (same seeds and inputs) with K kept as fp16
               values (the F16 K / q4_0 V configuration).
* ``prefill``  one chunk of chunked prefill: 1 sequence of 32768 positions whose
               last 512 are the chunk's tokens (causal among themselves), the
               earlier ones cached in 2 segments (one cut uniform in [1, L-1]
               with at least 512 positions after it); 32 query / 8 kv heads
               (2048 query rows per kv head), V q4_0, N(0,1), seed 6.

Every sequence's last ``t_q`` positions are the step's new tokens: the cache is
built from the first ``L - t_q`` tokens and the step appends the rest.
"""
from __future__ import annotations

import dataclasses
from typing import List

import numpy as np

V_Q4_0 = 0
V_Q8_0 = 1
K_I8 = 0
K_F16 = 1

CONFIG_NAMES = ("tiny", "single", "long", "batched", "verify", "prefill", "long_f16k")


@dataclasses.dataclass
class CacheSpec:
    """One KV cache of a workload (a workload may decode several per step)."""
    name: str
    seed: int
    n_seqs: int
    n_kv_heads: int
    n_q_heads: int
    head_dim: int
    t_q: int
    causal: bool
    v_type: int
    lengths: np.ndarray            # [n_seqs] positions incl. the t_q new tokens
    segments: List[np.ndarray]     # per sequence: segment lengths, sum = length
    outlier_channels: int = 0      # per kv head, K and V x10
    k_type: int = K_I8             # K_F16: K kept as fp16 values

    @property
    def max_len(self) -> int:
        return int(self.lengths.max()) if self.n_seqs else 0

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    def rng(self, *stream) -> np.random.Generator:
        return np.random.Generator(np.random.PCG64(np.random.SeedSequence([self.seed, *stream])))


def _cuts(rng: np.random.Generator, L: int, n_seg: int, min_last: int) -> np.ndarray:
    """n_seg segment lengths summing to L from n_seg-1 distinct sorted cut points
    uniform in [1, L-1]; redrawn until the last segment holds >= min_last."""
    if n_seg <= 1 or L < n_seg:
        return np.array([L], np.int64)
    while True:
        pts = np.sort(rng.choice(np.arange(1, L), size=n_seg - 1, replace=False))
        seg = np.diff(np.concatenate([[0], pts, [L]]))
        if seg[-1] >= min_last:
            return seg.astype(np.int64)


def make_spec(name: str, ctx: int | None = None, n_seqs: int | None = None,
              seed: int | None = None, **over) -> List[CacheSpec]:
    """The caches of workload ``name``.  ``ctx`` shrinks the context (the
    length range of ``batched`` scales with it) and ``n_seqs`` the batch, for
    parity cases the oracle finishes quickly; the structure is kept."""
    if name == "tiny":
        base = [dict(seed=0, n_seqs=1, n_kv_heads=1, n_q_heads=4, ctx=256, t_q=1, causal=False,
                     v_type=V_Q8_0, n_seg=1, outliers=0)]
    elif name == "single":
        base = [dict(seed=1, n_seqs=1, n_kv_heads=8, n_q_heads=32, ctx=8192, t_q=1, causal=False,
                     v_type=V_Q4_0, n_seg=1, outliers=4)]
    elif name == "long":
        base = [dict(seed=2, n_seqs=1, n_kv_heads=8, n_q_heads=40, ctx=131072, t_q=1, causal=False,
                     v_type=V_Q4_0, n_seg=4, outliers=0, tag="main"),
                dict(seed=3, n_seqs=1, n_kv_heads=4, n_q_heads=16, ctx=131072, t_q=1, causal=False,
                     v_type=V_Q4_0, n_seg=4, outliers=0, tag="draft")]
    elif name == "batched":
        base = [dict(seed=4, n_seqs=64, n_kv_heads=8, n_q_heads=32, ctx=32768, lo=1024, t_q=1,
                     causal=False, v_type=V_Q8_0, n_seg=1, outliers=4)]
    elif name == "verify":
        base = [dict(seed=5, n_seqs=16, n_kv_heads=8, n_q_heads=64, ctx=32768, t_q=4, causal=True,
                     v_type=V_Q4_0, n_seg=1, outliers=0)]
    elif name == "long_f16k":   # the long-context pair with F16 K (q4_0 V), seeds as "long"
        base = [dict(seed=2, n_seqs=1, n_kv_heads=8, n_q_heads=40, ctx=131072, t_q=1, causal=False,
                     v_type=V_Q4_0, n_seg=4, outliers=0, tag="main", k_type=K_F16),
                dict(seed=3, n_seqs=1, n_kv_heads=4, n_q_heads=16, ctx=131072, t_q=1, causal=False,
                     v_type=V_Q4_0, n_seg=4, outliers=0, tag="draft", k_type=K_F16)]
    elif name == "prefill":
        base = [dict(seed=6, n_seqs=1, n_kv_heads=8, n_q_heads=32, ctx=32768, t_q=512, causal=True,
                     v_type=V_Q4_0, n_seg=2, outliers=0)]
    else:
        raise KeyError(name)
    specs = []
    for b in base:
        b = dict(b)
        b.update(over)
        full_ctx = b["ctx"]
        c = int(ctx) if ctx is not None else full_ctx
        B = int(n_seqs) if n_seqs is not None else b["n_seqs"]
        s = int(seed) if seed is not None else b["seed"]
        meta = np.random.Generator(np.random.PCG64(np.random.SeedSequence([s, 0])))
        if "lo" in b:
            lo = max(b["t_q"], int(round(b["lo"] * c / full_ctx)))
            lengths = meta.integers(lo, c, size=B, endpoint=True).astype(np.int64)
        else:
            lengths = np.full(B, c, np.int64)
        segs = [_cuts(meta, int(L), b["n_seg"], b["t_q"]) for L in lengths]
        tag = b.get("tag")
        specs.append(CacheSpec(name=name if tag is None else "%s/%s" % (name, tag), seed=s,
                               n_seqs=B, n_kv_heads=b["n_kv_heads"], n_q_heads=b["n_q_heads"],
                               head_dim=b.get("head_dim", 128), t_q=b["t_q"], causal=b["causal"],
                               v_type=b["v_type"], lengths=lengths, segments=segs,
                               outlier_channels=b["outliers"], k_type=b.get("k_type", K_I8)))
    return specs


def outlier_channels(spec: CacheSpec) -> np.ndarray:
    """[n_kv_heads][outlier_channels] distinct channel indices per kv head."""
    rng = spec.rng(0, 1)
    return np.stack([rng.choice(spec.head_dim, size=spec.outlier_channels, replace=False)
                     for _ in range(spec.n_kv_heads)]) if spec.outlier_channels else \
        np.zeros((spec.n_kv_heads, 0), np.int64)


def gen_kv(spec: CacheSpec, seq: int, lo: int = 0, hi: int | None = None):
    """fp16 K and V of sequence ``seq`` for positions [lo, hi), token-major
    [n][n_kv_heads][head_dim].  Positions are drawn in chunks of 4096 so any
    range regenerates the same values."""
    L = int(spec.lengths[seq])
    hi = L if hi is None else min(int(hi), L)
    lo = max(0, int(lo))
    H, D = spec.n_kv_heads, spec.head_dim
    n = max(0, hi - lo)
    k = np.empty((n, H, D), np.float16)
    v = np.empty((n, H, D), np.float16)
    if n == 0:
        return k, v
    och = outlier_channels(spec)
    CH = 4096
    for c0 in range((lo // CH) * CH, hi, CH):
        c1 = min(c0 + CH, L)
        rk = spec.rng(1, seq, c0 // CH)
        rv = spec.rng(2, seq, c0 // CH)
        kk = rk.standard_normal((c1 - c0, H, D), dtype=np.float32)
        vv = rv.standard_normal((c1 - c0, H, D), dtype=np.float32)
        for h in range(H):
            if och.shape[1]:
                kk[:, h, och[h]] *= 10.0
                vv[:, h, och[h]] *= 10.0
        a, b = max(lo, c0), min(hi, c1)
        k[a - lo:b - lo] = kk[a - c0:b - c0].astype(np.float16)
        v[a - lo:b - lo] = vv[a - c0:b - c0].astype(np.float16)
    return k, v


def gen_q(spec: CacheSpec) -> np.ndarray:
    """fp16 Q [n_seqs][t_q][n_q_heads][head_dim], N(0,1)."""
    r = spec.rng(3)
    return r.standard_normal((spec.n_seqs, spec.t_q, spec.n_q_heads, spec.head_dim),
                             dtype=np.float32).astype(np.float16)


def kv_bytes_per_token_head(head_dim: int, v_type: int, k_type: int = K_I8) -> int:
    """Stored bytes read per (position, kv head): int8 K + fp16 scale per 32
    (F16 K: 2 bytes per element), plus the V block bytes (q4_0 18 B / q8_0
    34 B per 32)."""
    nb = head_dim // 32
    k = 2 * head_dim if k_type == K_F16 else head_dim + 2 * nb
    return k + (head_dim // 2 if v_type == V_Q4_0 else head_dim) + 2 * nb


def step_kv_bytes(specs: List[CacheSpec]) -> int:
    """Algorithmic KV bytes one decode step reads over all caches."""
    return int(sum(int(s.lengths.sum()) * s.n_kv_heads * kv_bytes_per_token_head(s.head_dim, s.v_type, s.k_type)
                   for s in specs))


def step_attn_flops(specs: List[CacheSpec]) -> int:
    """Algorithmic multiply-add FLOPs of one step's attention over all caches:
    per (query head, visible position) 2 x head_dim for q.k and 2 x head_dim
    for p.v; a query token i of t_q sees L - t_q + i + 1 positions under the
    causal tail, else all L."""
    total = 0
    for s in specs:
        for L in s.lengths:
            L, t = int(L), s.t_q
            vis = (t * (L - t) + t * (t + 1) // 2) if s.causal else t * L
            total += 4 * s.head_dim * s.n_q_heads * vis
    return int(total)
