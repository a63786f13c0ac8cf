"""Device-side setup of a workload for repeated decode steps, using only the
public API (kvq_append / kvq_decode_attn) and the seeded generator.

A *step* is one pass of the decode path over one batch: append the t_q newest
tokens of every sequence into its open segment, then decode attention for all
query rows.  ``DecodeSet.rewind()`` moves the host length bookkeeping back by
t_q so the same step can be replayed (the append rewrites identical bytes).
"""
from __future__ import annotations

import numpy as np
import torch

from . import kvq
from . import workloads as W

SM_SCALE = 1.0 / float(np.sqrt(128.0))


class HostData:
    """fp16 inputs of one cache spec, drawn once (host numpy)."""

    def __init__(self, spec: W.CacheSpec):
        self.spec = spec
        self.kv = [W.gen_kv(spec, b) for b in range(spec.n_seqs)]
        self.q = W.gen_q(spec)


class DecodeSet:
    def __init__(self, data: HostData, device=None, staging=None, layout="auto"):
        s = self.spec = data.spec
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.B, self.tq, self.Hq = s.n_seqs, s.t_q, s.n_q_heads
        self.lens_host = [int(x) for x in s.lengths]
        self.max_len = max(self.lens_host) if self.lens_host else 0
        self.cache = kvq.Cache(self.B, s.n_kv_heads, s.v_type, max_segs=max(len(x) for x in s.segments),
                               k_type=s.k_type)
        # device staging of every sequence's fp16 K/V (shared between copies)
        if staging is None:
            staging = [(torch.from_numpy(k).to(self.device), torch.from_numpy(v).to(self.device))
                       for k, v in data.kv]
        self.staging = staging
        for b in range(self.B):
            k, v = staging[b]
            pos = 0
            segs = s.segments[b]
            for j, n in enumerate(segs):
                n = int(n)
                self.cache.add_segment(b, n, layout)
                nb = n - (self.tq if j == len(segs) - 1 else 0)
                if nb > 0:
                    kvq.kvq_append(self.cache, [b], [nb], k[pos:pos + nb], v[pos:pos + nb])
                pos += n
        L = self.lens_host
        self.k_new = torch.cat([staging[b][0][L[b] - self.tq:L[b]] for b in range(self.B)]).contiguous()
        self.v_new = torch.cat([staging[b][1][L[b] - self.tq:L[b]] for b in range(self.B)]).contiguous()
        self.q16 = torch.from_numpy(data.q).to(self.device)
        self.lens = torch.tensor(self.lens_host, dtype=torch.int32, device=self.device)
        self.out = torch.empty((self.B, self.tq, self.Hq, 128), dtype=torch.float32, device=self.device)
        self.lse = torch.empty((self.B, self.tq, self.Hq), dtype=torch.float32, device=self.device)
        self.ws_bytes = kvq.kvq_decode_workspace_size(self.cache, self.Hq, self.tq, self.max_len)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.device) if self.ws_bytes else None
        self.seq_ids = list(range(self.B))

    def kv_bytes(self) -> int:
        """Algorithmic KV bytes one step reads (packed codes + scales)."""
        return W.step_kv_bytes([self.spec])

    def append_step(self, k_new=None, v_new=None, stream=None):
        kvq.kvq_append(self.cache, self.seq_ids, [self.tq] * self.B, self.k_new if k_new is None else k_new,
                       self.v_new if v_new is None else v_new, stream)

    def decode(self, q16=None, stream=None, out=None, lse=None):
        kvq.kvq_decode_attn(self.cache, self.q16 if q16 is None else q16, self.Hq, self.tq, self.spec.causal,
                            self.lens, self.max_len, None, SM_SCALE, self.out if out is None else out,
                            self.lse if lse is None else lse, self.ws, stream)

    def rewind(self):
        for b in range(self.B):
            self.cache.seg(b, self.cache.n_segs(b) - 1).len -= self.tq

    def launches_per_step(self) -> int:
        """Kernels one step launches: one append, one split kernel per group of
        up to 64 sequences, and a combine per group when sequences are split."""
        groups = (self.B + 63) // 64
        return 1 + groups * (2 if self.ws_bytes else 1)


class StepSet:
    """Every cache of one workload copy decoded by one kvq_decode_attn_multi
    call (one split launch and one combine for all of them).  With append=True
    the call also appends each cache's step tokens (fused append), so a step is
    that one call; else the caller runs kvq_append first."""

    def __init__(self, sets, q16=None, append=False, kv_new=None, outs=None):
        self.sets = list(sets)
        self.append = append
        self.calls = []
        for i, ds in enumerate(self.sets):
            out, lse = (ds.out, ds.lse) if outs is None else outs[i]
            c = dict(cache=ds.cache, q16=ds.q16 if q16 is None else q16[i], n_q_heads=ds.Hq, t_q=ds.tq,
                     causal_tail=ds.spec.causal, seq_lens=ds.lens, max_len=ds.max_len, head_map=None,
                     sm_scale=SM_SCALE, out=out, lse=lse)
            if append:
                k, v = (ds.k_new, ds.v_new) if kv_new is None else kv_new[i]
                c.update(k16_new=k, v16_new=v)
            self.calls.append(c)
        self.call = kvq.MultiCall(self.calls)
        n = self.call.workspace_size()
        self.call.ws = torch.empty(n, dtype=torch.uint8, device=self.sets[0].device) if n else None

    def decode(self, stream=None):
        self.call(stream)
