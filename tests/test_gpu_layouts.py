"""The rows segment layout (KVQ_LAYOUT_ROWS: one row per token in element
order, copied row by row and permuted into the tile order in shared memory)
next to the default tiles, on the GPU against the oracle: cache bytes
bit-exact (the rows layout stores exactly the oracle's rows), out within 2e-3,
lse within 1e-4, int32 block scores bit-exact.  Segments of one sequence mix
the layouts; short segments put copies that start and end inside a tile; the
step's tokens are appended, separately and fused, into a rows segment; long
chunks over rows segments run on the split kernel's row tiles."""
import numpy as np
import pytest
import torch

from quantized_kv_cache_03_gb300 import kvq
from quantized_kv_cache_03_gb300 import workloads as W

from kvq_cases import SM_SCALE, Case, assert_cache_bytes, assert_close, dev, to_dev

pytestmark = pytest.mark.gpu

ROWS, TILES = kvq.LAYOUT_ROWS, kvq.LAYOUT_TILES
SHAPES = {
    "tiny": dict(),
    "single": dict(ctx=3000),                     # outlier channels x10, q4_0
    "long": dict(ctx=5000),                       # 4 segments, main + draft
    "batched": dict(ctx=4096, n_seqs=6),          # ragged lengths, q8_0
    "verify": dict(ctx=3000, n_seqs=2),           # t_q = 4 causal, 32 rows per kv head
    "prefill": dict(ctx=1500, t_q=40),            # 160 rows per kv head: row tiles over rows segments
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _check(case):
    out, lse = case.decode()
    for b in range(case.B):
        if case.lens[b] > 0:
            assert_cache_bytes(case, b)
        assert_close(out[b], lse[b], case.oracle_decode(b), what="%s seq %d" % (case.spec.name, b))
    assert kvq.kvq_wait_timeouts() == 0


@pytest.mark.parametrize("name", sorted(SHAPES))
@pytest.mark.parametrize("mix", ["all_rows", "alternate"])
def test_shapes_with_rows_segments(name, mix):
    lay = (lambda b, k, n: ROWS) if mix == "all_rows" else (lambda b, k, n: ROWS if (b + k) % 2 else TILES)
    for spec in W.make_spec(name, **SHAPES[name]):
        _check(Case(spec).build(layout_of=lay))


@pytest.mark.parametrize("vt", [0, 1])
def test_many_short_rows_segments(vt, monkeypatch):
    """One sequence of 40 segments of 1 to 37 tokens in the rows layout (and a
    tiles prefix), with splits of 64 positions: copies that start and end
    anywhere inside a tile, pieces of one token, odd scale-row counts."""
    monkeypatch.setenv("KVQ_SPLIT", "64")
    rng = np.random.default_rng(11)
    lens = [300] + [int(x) for x in rng.integers(1, 38, 39)]
    spec = W.make_spec("single", ctx=sum(lens), v_type=vt, n_seg=1)[0]
    spec.segments[0] = np.array(lens, np.int64)
    case = Case(spec).build(layout_of=lambda b, k, n: TILES if k == 0 else ROWS)
    _check(case)


def test_fused_append_into_a_rows_segment():
    cases = [Case(s).build(append_step=False, layout_of=lambda b, k, n: ROWS if k >= 2 else TILES)
             for s in W.make_spec("long", ctx=4000)]
    calls = []
    for case in cases:
        L = case.lens[0]
        calls.append(dict(cache=case.cache, q16=to_dev(case.q), n_q_heads=case.Hq, t_q=1, causal_tail=False,
                          seq_lens=torch.tensor(case.lens, dtype=torch.int32, device=dev()), max_len=L,
                          head_map=None, sm_scale=SM_SCALE,
                          out=torch.full((1, 1, case.Hq, 128), float("nan"), device=dev()),
                          lse=torch.full((1, 1, case.Hq), float("nan"), device=dev()),
                          k16_new=to_dev(case.kv[0][0][L - 1:]), v16_new=to_dev(case.kv[0][1][L - 1:])))
    n = kvq.kvq_decode_multi_workspace_size(calls)
    kvq.kvq_decode_attn_multi(calls, torch.empty(n, dtype=torch.uint8, device=dev()) if n else None)
    torch.cuda.synchronize()
    for case, call in zip(cases, calls):
        assert case.cache.lengths() == case.lens
        assert_cache_bytes(case, 0)
        assert_close(call["out"][0].cpu().numpy(), call["lse"][0].cpu().numpy(), case.oracle_decode(0))


@pytest.mark.parametrize("vt", [0, 1])
def test_scores_bit_exact_over_rows_segments(vt):
    spec = W.make_spec("single", ctx=2000, v_type=vt, n_seg=3)[0]
    case = Case(spec).build(layout_of=lambda b, k, n: ROWS if k != 1 else TILES)
    qc, qs, sc = case.debug_qk()
    ref = case.oracle_decode(0, want_scores=True)
    assert np.array_equal(qc[0], ref["q_codes"]) and np.array_equal(qs[0], ref["q_scales"])
    assert np.array_equal(sc[0, 0, :, :case.lens[0]], ref["scores"][0])


def test_prefill_over_rows_segments_takes_the_row_tiles():
    spec = W.make_spec("prefill", ctx=1500, t_q=64)[0]
    case = Case(spec).build(layout_of=lambda b, k, n: ROWS)
    call = dict(cache=case.cache, n_q_heads=case.Hq, t_q=case.tq, causal_tail=True, max_len=case.max_len,
                head_map=None, sm_scale=SM_SCALE)
    lns, _ = kvq.kvq_debug_plan([call], 152)
    assert [ln["kernel"] for ln in lns] == ["split"]
    _check(case)


def test_repeats_and_pdl_on_off_bitwise_equal(monkeypatch):
    monkeypatch.setenv("KVQ_SPLIT", "256")
    spec = W.make_spec("long", ctx=3000)[0]
    case = Case(spec).build(layout_of=lambda b, k, n: ROWS if k % 2 else TILES)
    monkeypatch.setenv("KVQ_PDL", "1")
    runs = [case.decode() for _ in range(3)]
    monkeypatch.setenv("KVQ_PDL", "0")
    runs += [case.decode() for _ in range(2)]
    for o, l in runs[1:]:
        assert np.array_equal(o, runs[0][0]) and np.array_equal(l, runs[0][1])
