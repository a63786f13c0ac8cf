"""GPU vs oracle on the same seeded inputs, through the C ABI.

Bar: cache bytes, query codes/scales and per-block int32 scores bit-exact;
out within 2e-3 and lse within 1e-4 (max abs)."""
import numpy as np
import pytest

import oracle
from quantized_kv_cache_03_gb300 import workloads as W

from kvq_cases import Case, assert_cache_bytes, assert_close

pytestmark = pytest.mark.gpu

SMALL = {
    "tiny": dict(),                               # 256 positions, GQA 4, q8_0
    "single": dict(),                             # 8192 positions, outliers, q4_0
    "long": dict(ctx=5000),                       # 4 segments, GQA 5 main + GQA 4 draft
    "batched": dict(ctx=4096, n_seqs=6),          # ragged lengths, q8_0, outliers
    "verify": dict(ctx=3000, n_seqs=2),           # t_q = 4 causal, 32 rows per kv head
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("name", list(SMALL))
def test_config_parity(name):
    for spec in W.make_spec(name, **SMALL[name]):
        case = Case(spec).build()
        out, lse = case.decode()
        for b in range(case.B):
            oc = case.oracle_cache(b)
            assert_cache_bytes(case, b, oc)
            ref = case.oracle_decode(b, want_scores=True)
            assert_close(out[b], lse[b], ref, what="%s seq %d" % (spec.name, b))
        qc, qs, sc = case.debug_qk()
        for b in range(case.B):
            ref = case.oracle_decode(b, want_scores=True)
            assert np.array_equal(qc[b], ref["q_codes"]), "query codes"
            assert np.array_equal(qs[b], ref["q_scales"]), "query scales"
            L = case.lens[b]
            for i in range(case.tq):
                vis = L - case.tq + i + 1 if spec.causal else L
                assert np.array_equal(sc[b, i, :, :vis], ref["scores"][i, :, :vis]), "int32 block scores"


@pytest.mark.parametrize("name,kw", [("verify", dict(ctx=3000, n_seqs=2)), ("prefill", dict(ctx=1500, t_q=40))])
def test_sixteen_row_tiles(name, kw, monkeypatch):
    """KVQ_ROW_TILE=16 takes a kv head's 32 (verify) or more (a 40-token
    chunk) query rows with several CTAs of the 16-row kernel that stream the
    same positions, each under its own causal limit; KVQ_PREFILL=0 keeps the
    chunk off the tcgen05 kernel."""
    monkeypatch.setenv("KVQ_ROW_TILE", "16")
    monkeypatch.setenv("KVQ_PREFILL", "0")
    for spec in W.make_spec(name, **kw):
        case = Case(spec).build()
        out, lse = case.decode()
        for b in range(case.B):
            ref = case.oracle_decode(b)
            assert_close(out[b], lse[b], ref, what="%s seq %d (16-row tiles)" % (spec.name, b))


def test_half_warp_ctas(monkeypatch):
    """The 8-row kernel also runs with half its warps (two CTAs per SM).  The
    planner takes it when full CTAs would need more than one wave: a batch of 24
    sequences x 8 kv heads is at least 192 CTAs on 152 SMs.  Both forms match
    the oracle, the automatic choice is bitwise the forced half-warp result
    there, and bitwise the forced full-warp result for a call that fits one
    wave (the main cache of the long pair)."""
    def run(case, force):
        if force is None:
            monkeypatch.delenv("KVQ_SPLIT_WARPS", raising=False)
        else:
            monkeypatch.setenv("KVQ_SPLIT_WARPS", force)
        return case.decode()

    spec = W.make_spec("batched", ctx=4096, n_seqs=24)[0]
    case = Case(spec).build()
    res = {f: run(case, f) for f in (None, "8", "16")}
    for f in ("8", "16"):
        out, lse = res[f]
        for b in range(case.B):
            ref = case.oracle_decode(b)
            assert_close(out[b], lse[b], ref, what="batched seq %d (%s warps)" % (b, f))
    assert np.array_equal(res[None][0], res["8"][0]) and np.array_equal(res[None][1], res["8"][1])

    spec = W.make_spec("long", ctx=5000)[0]
    case = Case(spec).build()
    res = {f: run(case, f) for f in (None, "8", "16")}
    for f in ("8", "16"):
        out, lse = res[f]
        ref = case.oracle_decode(0)
        assert_close(out[0], lse[0], ref, what="long main (%s warps)" % f)
    assert np.array_equal(res[None][0], res["16"][0]) and np.array_equal(res[None][1], res["16"][1])
