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

    def build(self, append_step=True):
        s = self.spec
        self.cache = kvq.Cache(self.B, s.n_kv_heads, s.v_type, max_segs=max(len(x) for x in s.segments))
        for b in range(self.B):
            if self.lens[b] == 0:
                continue
            k, v = self.kv[b]
            pos = 0
            segs = s.segments[b]
            for j, n in enumerate(segs):
                n = int(n)
                self.cache.add_segment(b, n)
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
        kvq.kvq_debug_qk(self.cache, q16, self.Hq, self.tq, lens, self.max_len, head_map, qc, qs, sc)
        torch.cuda.synchronize()
        return qc.cpu().numpy(), qs.cpu().numpy().view(np.uint16), sc.cpu().numpy()

    def oracle_cache(self, b):
        k, v = self.kv[b]
        return oracle.quantize_kv(k, v, self.spec.v_type)

    def oracle_decode(self, b, head_map=None, row_mask=None, want_scores=False, threads=8):
        s = self.spec
        hm = oracle.default_head_map(s.n_q_heads, s.n_kv_heads) if head_map is None else np.asarray(head_map)
        return oracle.decode_seq(self.oracle_cache(b), self.q[b], hm, s.causal, SM_SCALE, s.v_type,
                                 want_codes=want_scores, want_scores=want_scores, row_mask=row_mask,
                                 n_threads=threads)


def assert_cache_bytes(case, b, oc=None):
    oc = case.oracle_cache(b) if oc is None else oc
    got = case.cache.export(b)
    for name in ("kq", "ks", "vq", "vs"):
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
