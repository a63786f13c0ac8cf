"""The split planner on the host (kvq_debug_plan, no GPU): which kernel, CTA
form, chunk and CTA count each bench workload gets on a 152-SM GB300, and how
the environment knobs steer it.  The expected plans are the ones measured best
on the GPU (split-chunk sweeps, 8- vs 16-warp CTAs)."""
import ctypes

import pytest

from quantized_kv_cache_03_gb300 import build as B
from quantized_kv_cache_03_gb300 import kvq
from quantized_kv_cache_03_gb300 import workloads as W

N_SMS = 152
# resident CTAs per SM: <= 8 rows with 16 warps, the same with 8 warps, 16-row and 32-row tiles
CTAS = (1, 2, 2, 2)
ADDR = 0x100000   # never dereferenced by the planner


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    kvq.load()


@pytest.fixture(autouse=True)
def _clean_env(monkeypatch):
    for k in ("KVQ_SPLIT", "KVQ_SPLIT_WARPS", "KVQ_ROW_TILE", "KVQ_PREFILL", "KVQ_TC_ROWS"):
        monkeypatch.delenv(k, raising=False)


class HostCache:
    """The host descriptor of a cache built as the bench builds it (segments
    of the spec, capacities rounded to 64), with fake device addresses."""

    def __init__(self, spec, fused):
        S = max(len(x) for x in spec.segments)
        self.segs = (kvq.KvqSegment * (spec.n_seqs * S))()
        self.ns = (ctypes.c_int32 * spec.n_seqs)()
        for b in range(spec.n_seqs):
            pos = 0
            lens = [int(n) for n in spec.segments[b]]
            for j, n in enumerate(lens):
                s = self.segs[b * S + j]
                s.k_q = s.k_s = s.v_q = s.v_s = ADDR
                s.cap = -(-n // kvq.SEG_ALIGN) * kvq.SEG_ALIGN
                s.len = n - (spec.t_q if fused and j == len(lens) - 1 else 0)
                s.pos0 = pos
                pos += n
            self.ns[b] = len(lens)
        self.desc = kvq.KvqCache(spec.n_seqs, spec.n_kv_heads, spec.head_dim, spec.v_type, S,
                                 ctypes.cast(self.ns, ctypes.POINTER(ctypes.c_int32)),
                                 ctypes.cast(self.segs, ctypes.POINTER(kvq.KvqSegment)), spec.k_type, 0)


class FakePtr:
    """Stands in for a tensor: only its address is passed on."""

    def data_ptr(self):
        return ADDR


def calls_of(name, fused, **kw):
    specs = W.make_spec(name, **kw)
    calls = []
    for spec in specs:
        c = dict(cache=HostCache(spec, fused), n_q_heads=spec.n_q_heads, t_q=spec.t_q, causal_tail=spec.causal,
                 max_len=spec.max_len, sm_scale=0.088)
        if fused:
            c.update(k16_new=FakePtr(), v16_new=FakePtr())
        calls.append(c)
    return specs, calls


def plan(calls):
    return kvq.kvq_debug_plan(calls, N_SMS, CTAS)


def test_long_pair_fused_is_one_wave_of_16_warp_ctas():
    """Both caches in one launch: 12 splits of 11008 positions per kv head,
    (8 + 4) x 12 = 144 CTAs, one combine over the 40 + 16 query rows."""
    _, calls = calls_of("long", fused=True)
    lns, ws = plan(calls)
    assert lns == [dict(kernel="split", n_tiles8=1, warps=16, chunk=11008, chunk0=11008, n_ctas=144, n_rows=56)]
    assert ws > 0


def test_long_caches_one_call_each():
    """Per cache, as the per-cache variant of the bench launches them: the
    main cache fills the 152 SMs with 19 splits, the draft 148 with 37."""
    _, calls = calls_of("long", fused=False)
    main, _ = plan(calls[:1])
    draft, _ = plan(calls[1:])
    assert (main[0]["warps"], main[0]["n_ctas"], main[0]["n_rows"]) == (16, 152, 40)
    assert (draft[0]["warps"], draft[0]["n_ctas"], draft[0]["n_rows"]) == (16, 148, 16)


def test_batched_takes_the_8_warp_form():
    """64 sequences x 8 kv heads need more than one wave of 16-warp CTAs, so
    the 8-warp form (two per SM) runs, with chunks in its 128-position granule."""
    specs, calls = calls_of("batched", fused=True)
    lns, _ = plan(calls)
    assert len(lns) == 1
    ln = lns[0]
    assert ln["kernel"] == "split" and ln["n_tiles8"] == 1 and ln["warps"] == 8
    assert ln["chunk"] % 128 == 0 and ln["n_ctas"] > N_SMS * CTAS[0]
    assert ln["n_rows"] == specs[0].n_seqs * specs[0].n_q_heads


def test_split_knobs(monkeypatch):
    """KVQ_SPLIT forces the chunk and keeps 16 warps; KVQ_SPLIT_WARPS forces
    the form either way."""
    _, calls = calls_of("batched", fused=True)
    monkeypatch.setenv("KVQ_SPLIT", "4096")
    ln = plan(calls)[0][0]
    assert (ln["warps"], ln["chunk"]) == (16, 4096)
    monkeypatch.setenv("KVQ_SPLIT_WARPS", "8")
    ln = plan(calls)[0][0]
    assert (ln["warps"], ln["chunk"]) == (8, 4096)
    monkeypatch.delenv("KVQ_SPLIT")
    monkeypatch.setenv("KVQ_SPLIT_WARPS", "16")
    assert plan(calls)[0][0]["warps"] == 16
    # a one-wave launch forced onto the 8-warp form
    _, calls = calls_of("long", fused=True)
    monkeypatch.setenv("KVQ_SPLIT_WARPS", "8")
    ln = plan(calls)[0][0]
    assert ln["warps"] == 8 and ln["n_ctas"] <= N_SMS * CTAS[1]


def test_single_and_tiny():
    """single: 16 splits of 512 positions (128 CTAs, the best of the chunk
    sweep); tiny: one split, so no combine launch and no workspace."""
    _, calls = calls_of("single", fused=True)
    lns, ws = plan(calls)
    assert lns == [dict(kernel="split", n_tiles8=1, warps=16, chunk=512, chunk0=512, n_ctas=128, n_rows=32)]
    _, calls = calls_of("tiny", fused=True)
    lns, ws = plan(calls)
    assert len(lns) == 1 and lns[0]["n_ctas"] == 1 and lns[0]["n_rows"] == 0 and ws == 0


def test_verify_shape(monkeypatch):
    """32 query rows per kv head: the 32-row tiles by default; KVQ_ROW_TILE=16
    doubles the CTAs with 16-row tiles."""
    specs, calls = calls_of("verify", fused=True)
    ln = plan(calls)[0][0]
    assert (ln["kernel"], ln["n_tiles8"], ln["warps"]) == ("split", 4, 4)
    monkeypatch.setenv("KVQ_ROW_TILE", "16")
    ln16 = plan(calls)[0][0]
    assert (ln16["n_tiles8"], ln16["warps"]) == (2, 4)
    monkeypatch.delenv("KVQ_ROW_TILE")
    assert kvq.kvq_debug_plan.n_pre_appends == 0
    # KVQ_TC_ROWS=17: the tcgen05 kernel, its step tokens through an append launch first
    # (128 one-tile units on 152 SMs: split unevenly in two)
    monkeypatch.setenv("KVQ_TC_ROWS", "17")
    ln = plan(calls)[0][0]
    assert ln["kernel"] == "prefill" and ln["n_ctas"] == 2 * 16 * 8 and kvq.kvq_debug_plan.n_pre_appends == 1
    assert ln["n_rows"] == 16 * 4 * 64


def test_prefill_chunk(monkeypatch):
    """A 512-token chunk (2048 rows per kv head) runs on the tcgen05 prefill
    kernel.  Its 128 units (8 kv heads x 16 row tiles) on 152 SMs would leave 24
    SMs idle, so every unit is split unevenly: 128 large CTAs [0, chunk0), then
    128 small ones [chunk0, reach) that the 24 spare SMs take six at a time, and
    a combine over all 16384 rows.  chunk0 balances one large CTA against six
    small ones (256 positions of fixed cost each).  KVQ_PREFILL_BALANCE=0 keeps
    one split on 128 CTAs; KVQ_PREFILL=0 sends the chunk to the split kernel's
    32-row tiles."""
    specs, calls = calls_of("prefill", fused=False)
    reach = max(specs[0].lengths)
    lns, ws = plan(calls)
    assert len(lns) == 1 and lns[0]["kernel"] == "prefill" and lns[0]["n_ctas"] == 256
    ln = lns[0]
    c0, c1 = ln["chunk0"], ln["chunk"]
    assert c0 % 64 == 0 and c1 % 64 == 0 and c0 < reach <= c0 + c1 < reach + 64
    k, o = 6, 256
    assert k * (reach - c0 + o) <= c0 + o < k * (reach - c0 + o) + (k + 1) * 64
    assert ln["n_rows"] == 512 * 32 and ws == (512 * 32 * 2 * 129 * 4 + 255) // 256 * 256
    monkeypatch.setenv("KVQ_PREFILL_BALANCE", "3")
    ln3 = plan(calls)[0][0]
    assert ln3["n_ctas"] == 256 and ln3["chunk0"] < c0 and 3 * (reach - ln3["chunk0"] + o) <= ln3["chunk0"] + o
    monkeypatch.setenv("KVQ_PREFILL_BALANCE", "0")
    lns, ws = plan(calls)
    assert lns[0]["n_ctas"] == 128 and lns[0]["chunk0"] == lns[0]["chunk"] and lns[0]["n_rows"] == 0 and ws == 0
    monkeypatch.delenv("KVQ_PREFILL_BALANCE")
    monkeypatch.setenv("KVQ_SPLIT", "8192")   # a forced chunk keeps even splits
    ln = plan(calls)[0][0]
    assert ln["chunk0"] == ln["chunk"] == 8192 and ln["n_ctas"] == 128 * ((reach + 8191) // 8192)
    monkeypatch.delenv("KVQ_SPLIT")
    monkeypatch.setenv("KVQ_PREFILL", "0")
    ln = plan(calls)[0][0]
    assert (ln["kernel"], ln["n_tiles8"]) == ("split", 4)


def test_uneven_split_only_for_one_partial_wave_of_one_group():
    """The uneven split applies to a one-group tcgen05 launch whose units fill
    more than half but not all of the SMs.  At most half (4 kv heads x 16 row
    tiles = 64 units) the even split already fills the machine (2 x 64 CTAs);
    more units than SMs (10 kv heads: 160) take even splits over several
    waves; two calls in one launch (two work groups) keep even splits too."""
    for kw, units in ((dict(n_q_heads=16, n_kv_heads=4), 64), (dict(n_q_heads=40, n_kv_heads=10), 160)):
        _, calls = calls_of("prefill", fused=False, **kw)
        ln = plan(calls)[0][0]
        assert ln["kernel"] == "prefill" and ln["chunk0"] == ln["chunk"], kw
        assert ln["n_ctas"] % units == 0 and ln["n_ctas"] > units, kw
    _, calls = calls_of("prefill", fused=False)
    ln = plan(calls + calls)[0][0]
    assert ln["kernel"] == "prefill" and ln["chunk0"] == ln["chunk"] and ln["n_ctas"] % 256 == 0


def test_bad_arguments():
    _, calls = calls_of("tiny", fused=True)
    with pytest.raises(kvq.KvqError):
        kvq.kvq_debug_plan(calls, 0, CTAS)
    with pytest.raises(kvq.KvqError):
        kvq.kvq_debug_plan(calls, N_SMS, (1, 0, 2, 2))
    # F16 K takes no fused append
    _, f16 = calls_of("long_f16k", fused=True)
    with pytest.raises(kvq.KvqError):
        plan(f16)


def test_workspace_is_the_split_partials():
    """The workspace holds, per unit with more than one split, every query
    row's per-split partial output and lse (128 + 1 floats), each unit's block
    rounded up to 256 bytes."""
    specs, calls = calls_of("long", fused=True)
    lns, ws = plan(calls)
    n_split = -(-131072 // lns[0]["chunk"])
    want = sum(-(-(s.n_seqs * s.t_q * s.n_q_heads * n_split * 129 * 4) // 256) * 256 for s in specs)
    assert ws == want


def test_more_than_64_sequences_take_several_launches():
    """A launch's tables hold at most 64 sequences: a 100-sequence batch runs
    as a launch of 64 and one of 36, each planned on its own (the second fits
    one wave of 8-warp CTAs unsplit, so it needs no combine)."""
    specs, calls = calls_of("batched", fused=True, ctx=4096, n_seqs=100)
    lns, _ = plan(calls)
    H, Hq = specs[0].n_kv_heads, specs[0].n_q_heads
    assert len(lns) == 2 and all(ln["kernel"] == "split" for ln in lns)
    for ln, nb in zip(lns, (64, 36)):
        assert ln["n_ctas"] % (nb * H) == 0
        n_split = ln["n_ctas"] // (nb * H)
        assert ln["n_rows"] == (nb * Hq if n_split > 1 else 0)
    assert lns[1]["n_ctas"] == 36 * H and lns[1]["warps"] == 8


def test_f16k_pair_without_fused_append():
    """F16 K decodes on the same split kernel (its own K format) once the
    step's tokens went in through kvq_append: one launch for both caches."""
    _, calls = calls_of("long_f16k", fused=False)
    lns, _ = plan(calls)
    assert len(lns) == 1 and lns[0]["kernel"] == "split" and lns[0]["n_rows"] == 56


def test_rows_segments_route_long_chunks_to_the_row_tiles():
    """The tcgen05 prefill kernel reads tile-layout segments only: a chunk over
    a cache with a rows-layout segment plans on the split kernel's 32-row
    tiles; decode calls keep their plan."""
    _, calls = calls_of("prefill", fused=False)
    assert plan(calls)[0][0]["kernel"] == "prefill"
    calls[0]["cache"].segs[1].layout = kvq.LAYOUT_ROWS
    ln = plan(calls)[0][0]
    assert (ln["kernel"], ln["n_tiles8"]) == ("split", 4)
    _, dec = calls_of("long", fused=True)
    before = plan(dec)
    dec[0]["cache"].segs[2].layout = kvq.LAYOUT_ROWS
    assert plan(dec) == before


def test_segment_layout_is_checked():
    _, calls = calls_of("long", fused=False)
    calls[0]["cache"].segs[0].layout = 2
    with pytest.raises(kvq.KvqError) as e:
        plan(calls)
    assert e.value.status == kvq.KVQ_ERR_INVALID_ARG
    _, f16 = calls_of("long_f16k", fused=False)
    f16[0]["cache"].segs[0].layout = kvq.LAYOUT_ROWS      # rows layout: int8 K only
    with pytest.raises(kvq.KvqError) as e:
        plan(f16)
    assert e.value.status == kvq.KVQ_ERR_UNSUPPORTED
