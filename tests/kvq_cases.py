"""Shared helpers of the GPU tests: build a segmented cache from a workload
spec through kvq_append, run one decode step, and compute the oracle's answer
on the same seeded inputs."""
import numpy as np
import torch

import oracle
from quantized_kv_cache_03_gb300 import kvq
from quantized_kv_cache_03_gb300 import workloads as W

SM_SCALE = 1.0 / np.sqrt(128.0)
OUT_TOL = 2e-3
LSE_TOL = 1e-4


def dev():
    return torch.device("cuda", 0)


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


class Case:
    """One cache of a workload: inputs, the GPU cache after the step's append,
    and the oracle's cache."""

    def __init__(self, spec, kv=None, q=None):
        self.spec = spec
        self.B, self.tq, self.Hq = spec.n_seqs, spec.t_q, spec.n_q_heads
        self.kv = kv if kv is not None else [W.gen_kv(spec, b) for b in range(self.B)]
        self.q = q if q is not None else W.gen_q(spec)
        self.lens = [int(x) for x in spec.lengths]
        self.max_len = max(self.lens) if self.lens else 0
        self.cache = None

    def build(self, append_step=True, layout_of=None):
        """layout_of(b, k, n) -> kvq.LAYOUT_* of segment k (n tokens) of
        sequence b (default: every segment in tiles)."""
        s = self.spec
        self.cache = kvq.Cache(self.B, s.n_kv_heads, s.v_type, max_segs=max(len(x) for x in s.segments),
                               k_type=s.k_type)
        for b in range(self.B):
            if self.lens[b] == 0:
                continue
            k, v = self.kv[b]
            pos = 0
            segs = s.segments[b]
            for j, n in enumerate(segs):
                n = int(n)
                self.cache.add_segment(b, n, kvq.LAYOUT_TILES if layout_of is None else layout_of(b, j, n))
                nb = n - (self.tq if j == len(segs) - 1 else 0)
                if nb > 0:
                    kvq.kvq_append(self.cache, [b], [nb], to_dev(k[pos:pos + nb]), to_dev(v[pos:pos + nb]))
                pos += n
        if append_step:
            self.append_step()
        return self

    def append_step(self):
        ids = [b for b in range(self.B) if self.lens[b] > 0]
        ks = np.concatenate([self.kv[b][0][self.lens[b] - self.tq:] for b in ids])
        vs = np.concatenate([self.kv[b][1][self.lens[b] - self.tq:] for b in ids])
        kvq.kvq_append(self.cache, ids, [self.tq] * len(ids), to_dev(ks), to_dev(vs))

    def decode(self, head_map=None, stream=None):
        s = self.spec
        q16 = to_dev(self.q)
        lens = torch.tensor(self.lens, dtype=torch.int32, device=dev())
        out = torch.full((self.B, self.tq, self.Hq, 128), float("nan"), dtype=torch.float32, device=dev())
        lse = torch.full((self.B, self.tq, self.Hq), float("nan"), dtype=torch.float32, device=dev())
        n = kvq.kvq_decode_workspace_size(self.cache, self.Hq, self.tq, self.max_len, head_map)
        ws = torch.empty(n, dtype=torch.uint8, device=dev()) if n else None
        kvq.kvq_decode_attn(self.cache, q16, self.Hq, self.tq, s.causal, lens, self.max_len, head_map, SM_SCALE,
                            out, lse, ws, stream)
        torch.cuda.synchronize()
        return out.cpu().numpy(), lse.cpu().numpy()

    def debug_qk(self, head_map=None):
        q16 = to_dev(self.q)
        lens = torch.tensor(self.lens, dtype=torch.int32, device=dev())
        qc = torch.zeros((self.B, self.tq, self.Hq, 128), dtype=torch.int8, device=dev())
        qs = torch.zeros((self.B, self.tq, self.Hq, 4), dtype=torch.int16, device=dev())
        sc = torch.zeros((self.B, self.tq, self.Hq, self.max_len, 4), dtype=torch.int32, device=dev())
        self.dump_kernel = kvq.kvq_debug_qk(self.cache, q16, self.Hq, self.tq, lens, self.max_len, head_map, qc,
                                            qs, sc)
        torch.cuda.synchronize()
        return qc.cpu().numpy(), qs.cpu().numpy().view(np.uint16), sc.cpu().numpy()

    def oracle_cache(self, b):
        k, v = self.kv[b]
        return oracle.quantize_kv(k, v, self.spec.v_type, k_type=self.spec.k_type)

    def oracle_decode(self, b, head_map=None, row_mask=None, want_scores=False, threads=8, causal=None):
        s = self.spec
        hm = oracle.default_head_map(s.n_q_heads, s.n_kv_heads) if head_map is None else np.asarray(head_map)
        causal = s.causal if causal is None else causal
        return oracle.decode_seq(self.oracle_cache(b), self.q[b], hm, causal, SM_SCALE, s.v_type,
                                 want_codes=want_scores, want_scores=want_scores, row_mask=row_mask,
                                 n_threads=threads)


def lane_view_index(name, v_type):
    """(stored offset, token u, logical byte j) of every code byte of a 16-token
    tile, enumerated the way the attention kernel reads a stage: 16-byte load i
    of lane = 4g + c, byte q of that load.
      K:    load i = 2 sub + hb: token 8 sub + g, codes 8c..8c+7 of block 2hb
            (bytes 0..7) and of block 2hb + 1 (bytes 8..15).
      q4_0: load i = sub, word bb = block bb: bytes 2g, 2g+1 of token t, then of
            token t + 1, t = 8 sub + 2c.
      q8_0: load i = 2 sub + hb, bytes 0..7 block 2hb, 8..15 block 2hb + 1; in
            each half word 0 holds dims 4g, 4g+1 and word 1 dims 4g+2, 4g+3,
            each as (t, t+1, t, t+1)."""
    rows = []
    if name == "k16":
        # F16 K (2-byte elements): the mma A fragment of k16 step ks for lane
        # 4g + c is four registers a0 (row g, k 2c, 2c+1), a1 (row g + 8, same
        # k), a2 (row g, k 2c + 8, 2c + 9), a3 (row g + 8, same), stored as
        # the 16-byte word ks * 512 + lane * 16
        for ks in range(8):
            for lane in range(32):
                g, c = lane // 4, lane % 4
                for reg in range(4):
                    for half in range(2):
                        u = g + 8 * (reg % 2)
                        kk = 2 * c + 8 * (reg // 2) + half
                        rows.append((ks * 256 + lane * 8 + reg * 2 + half, u, 16 * ks + kk))
        return np.array(rows, dtype=np.int64)
    for lane in range(32):
        g, c = lane // 4, lane % 4
        for q in range(16):
            if name == "kq":
                for i in range(4):
                    sub, hb = i // 2, i % 2
                    bb = 2 * hb + q // 8
                    rows.append((i * 512 + lane * 16 + q, 8 * sub + g, 32 * bb + 8 * c + q % 8))
            elif v_type == kvq.V_Q4_0:
                for i in range(2):
                    bb, w = q // 4, q % 4
                    rows.append((i * 512 + lane * 16 + q, 8 * i + 2 * c + w // 2, 16 * bb + 2 * g + w % 2))
            else:
                for i in range(4):
                    sub, hb = i // 2, i % 2
                    bb, r = 2 * hb + q // 8, q % 8
                    wd, y = r // 4, r % 4
                    rows.append((i * 512 + lane * 16 + q, 8 * sub + 2 * c + y % 2, 32 * bb + 4 * g + 2 * wd + y // 2))
    return np.array(rows, dtype=np.int64)


def logical_codes(stored, name, v_type):
    """Stored codes [H][cap][row] (tile order) -> logical [H][cap][row]."""
    H, cap, row = stored.shape
    idx = lane_view_index(name, v_type)
    assert len(idx) == 16 * row and len(np.unique(idx[:, 0])) == 16 * row
    tiles = stored.reshape(H, cap // 16, 16 * row)
    out = np.empty((H, cap // 16, 16, row), dtype=stored.dtype)
    out[:, :, idx[:, 1], idx[:, 2]] = tiles[:, :, idx[:, 0]]
    return out.reshape(H, cap, row)


def export_logical(cache, b):
    """Sequence b's filled positions in logical order, un-tiled by the lane view
    above (independently of the library's own untile helper)."""
    names = ("k16", "vq", "vs") if cache.k_type == kvq.K_F16 else ("kq", "ks", "vq", "vs")
    parts = {n: [] for n in names}
    for seg in cache.export(b, raw=True):
        n = seg["len"]
        for name in parts:
            a = seg[name]
            if name in ("kq", "vq") and seg["layout"] == kvq.LAYOUT_ROWS:
                a = a.view(np.uint8)                  # rows layout: element order as stored
            elif name in ("kq", "vq"):
                a = logical_codes(a.view(np.uint8), name, cache.v_type)
            elif name == "k16":
                a = logical_codes(a.view(np.uint16), name, cache.v_type)
            parts[name].append(a[:, :n])
    return {k: np.concatenate(v, axis=1) for k, v in parts.items()}


def assert_cache_bytes(case, b, oc=None):
    oc = case.oracle_cache(b) if oc is None else oc
    got = export_logical(case.cache, b)
    for name in oc:
        g, o = got[name].view(np.uint8), oc[name].view(np.uint8)
        assert g.shape == o.shape, (name, g.shape, o.shape)
        if not np.array_equal(g, o):
            bad = np.argwhere(g != o)
            raise AssertionError("cache bytes %s differ at %d places, first %s" % (name, len(bad), bad[:5]))


def assert_close(out, lse, ref, rows=None, what=""):
    o, l = out, lse
    ro, rl = ref["out"], ref["lse"]
    if rows is not None:
        o, l = o.reshape(-1, 128)[rows], l.reshape(-1)[rows]
        ro, rl = ro.reshape(-1, 128)[rows], rl.reshape(-1)[rows]
    both_inf = np.isneginf(l) & np.isneginf(rl)
    assert np.array_equal(np.isneginf(l), np.isneginf(rl)), what + " -inf lse mismatch"
    eo = float(np.abs(o - ro).max()) if o.size else 0.0
    el = float(np.abs(l[~both_inf] - rl[~both_inf]).max()) if (~both_inf).any() else 0.0
    assert eo <= OUT_TOL, "%s max|out-oracle| = %.3e" % (what, eo)
    assert el <= LSE_TOL, "%s max|lse-oracle| = %.3e" % (what, el)
    return eo, el
