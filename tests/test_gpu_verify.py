"""Multi-token verify over the quantized cache: calls with 9 to 32 query rows
per kv head (t_q query tokens x the kv head's query heads).  They run on the
split kernel's 16- and 32-row tiles.  The cases cover row counts that are not
multiples of 8, ragged and short contexts (tiles cut by segment ends, by the
sequence length and by the causal tail), several splits merged by the combine,
q8_0 V with x10 outlier channels, a non-causal call, uneven head maps, the
step's tokens passed to the call (fused append), and a launch that mixes
verify and decode calls.  With KVQ_TC_ROWS=17 the same calls run on the
tcgen05 kernel (one 128-row tile whose idle lane quarters keep only the
barrier phases, the step's tokens appended by a launch of their own first);
the tests marked below run both ways.  All against the oracle on the same seeded inputs:
cache bytes bit-exact, out within 2e-3 and lse within 1e-4."""

import numpy as np
import pytest
import torch

from quantized_kv_cache_03_gb300 import kvq
from quantized_kv_cache_03_gb300 import workloads as W

from kvq_cases import SM_SCALE, Case, assert_cache_bytes, assert_close, dev, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.fixture(params=["rowtile", "tcgen05"])
def route(request, monkeypatch):
    if request.param == "tcgen05":
        monkeypatch.setenv("KVQ_TC_ROWS", "17")
    return request.param


def _check_all(case, head_map=None):
    out, lse = case.decode(head_map=head_map)
    for b in range(case.B):
        assert_cache_bytes(case, b)
        ref = case.oracle_decode(b, head_map=head_map)
        assert_close(out[b], lse[b], ref, what="seq %d" % b)
    assert kvq.kvq_wait_timeouts() == 0
    return out, lse


@pytest.mark.parametrize("vt", [0, 1])
def test_verify_shape_two_sequences(vt, route):
    # 4 causal tokens x 8 query heads = 32 rows per kv head, 3000 positions
    spec = W.make_spec("verify", ctx=3000, n_seqs=2, v_type=vt)[0]
    _check_all(Case(spec).build())


@pytest.mark.parametrize("tq,hq,hkv", [(3, 20, 4), (5, 12, 4), (2, 40, 8), (9, 24, 8)])
def test_row_counts_not_multiples_of_eight(tq, hq, hkv):
    # 15, 15, 10 and 27 rows per kv head
    spec = W.make_spec("verify", ctx=1700, n_seqs=1, t_q=tq, n_q_heads=hq, n_kv_heads=hkv)[0]
    _check_all(Case(spec).build())


def test_ragged_short_contexts_and_segments(route):
    """Four sequences of very different lengths (one shorter than a KV tile),
    three segments each: KV tiles cut by segment ends and sequence lengths."""
    spec = W.make_spec("verify", ctx=2600, n_seqs=4, n_seg=3, v_type=1, outliers=4)[0]
    spec.lengths[:] = [2600, 37, 611, 1290]
    spec.segments[:] = [W._cuts(spec.rng(9, b), int(L), 3, spec.t_q) for b, L in enumerate(spec.lengths)]
    _check_all(Case(spec).build())


def test_context_of_the_step_tokens_only():
    # the cache holds only the 4 tokens being verified
    spec = W.make_spec("verify", ctx=4, n_seqs=2, n_seg=1)[0]
    out, lse = _check_all(Case(spec).build())
    assert np.all(np.isfinite(lse))


@pytest.mark.parametrize("split", [128, 640])
def test_several_splits_and_the_combine(split, monkeypatch):
    monkeypatch.setenv("KVQ_SPLIT", str(split))
    spec = W.make_spec("verify", ctx=2900, n_seqs=2, v_type=1, outliers=4)[0]
    _check_all(Case(spec).build())


def test_non_causal_rows():
    spec = W.make_spec("verify", ctx=1500, n_seqs=1, causal=False)[0]
    _check_all(Case(spec).build())


def test_uneven_head_map():
    # kv head 0 takes 7 query heads (28 rows), kv head 3 two (8 rows)
    spec = W.make_spec("verify", ctx=1800, n_seqs=1, n_q_heads=16, n_kv_heads=4)[0]
    hm = [0] * 7 + [1, 1, 1, 1, 2, 2, 2, 3, 3]
    assert len(hm) == 16
    _check_all(Case(spec).build(), head_map=hm)


def test_step_tokens_passed_to_the_call(route):
    """k16_new / v16_new with a verify call: the tokens are appended (cache
    bytes as kvq_append writes them), the host lengths advance, and the
    attention sees them."""
    spec = W.make_spec("verify", ctx=1500, n_seqs=3, v_type=0)[0]
    case = Case(spec).build(append_step=False)
    ids = list(range(case.B))
    ks = np.concatenate([case.kv[b][0][case.lens[b] - case.tq:] for b in ids])
    vs = np.concatenate([case.kv[b][1][case.lens[b] - case.tq:] for b in ids])
    before = case.cache.lengths()
    call = dict(cache=case.cache, q16=to_dev(case.q), n_q_heads=case.Hq, t_q=case.tq, causal_tail=True,
                seq_lens=torch.tensor(case.lens, dtype=torch.int32, device=dev()), max_len=case.max_len,
                head_map=None, sm_scale=SM_SCALE,
                out=torch.full((case.B, case.tq, case.Hq, 128), float("nan"), device=dev()),
                lse=torch.full((case.B, case.tq, case.Hq), float("nan"), device=dev()),
                k16_new=to_dev(ks), v16_new=to_dev(vs))
    n = kvq.kvq_decode_multi_workspace_size([call])
    kvq.kvq_decode_attn_multi([call], torch.empty(n, dtype=torch.uint8, device=dev()) if n else None)
    torch.cuda.synchronize()
    assert case.cache.lengths() == [x + case.tq for x in before]
    for b in range(case.B):
        assert_cache_bytes(case, b)
        assert_close(call["out"][b].cpu().numpy(), call["lse"][b].cpu().numpy(), case.oracle_decode(b),
                     what="seq %d" % b)


def test_verify_and_decode_calls_in_one_launch():
    """A verify call and a single-token decode of another cache in one
    kvq_decode_attn_multi call (two launches of different kernels)."""
    ver = Case(W.make_spec("verify", ctx=1200, n_seqs=2)[0]).build()
    dec = Case(W.make_spec("long", ctx=2000)[0]).build()
    calls = []
    for case in (ver, dec):
        calls.append(dict(cache=case.cache, q16=to_dev(case.q), n_q_heads=case.Hq, t_q=case.tq,
                          causal_tail=case.spec.causal,
                          seq_lens=torch.tensor(case.lens, dtype=torch.int32, device=dev()),
                          max_len=case.max_len, head_map=None, sm_scale=SM_SCALE,
                          out=torch.full((case.B, case.tq, case.Hq, 128), float("nan"), device=dev()),
                          lse=torch.full((case.B, case.tq, case.Hq), float("nan"), device=dev())))
    n = kvq.kvq_decode_multi_workspace_size(calls)
    kvq.kvq_decode_attn_multi(calls, torch.empty(n, dtype=torch.uint8, device=dev()) if n else None)
    torch.cuda.synchronize()
    for case, call in zip((ver, dec), calls):
        for b in range(case.B):
            assert_close(call["out"][b].cpu().numpy(), call["lse"][b].cpu().numpy(), case.oracle_decode(b),
                         what="%s seq %d" % (case.spec.name, b))


def test_full_size_sampled_rows():
    """The verify workload at full size (16 sequences x 4 causal tokens over
    32768 positions, 64/8 heads), in the benchmark's launch configuration:
    sampled query rows of the first and last sequence against the oracle."""
    spec = W.make_spec("verify")[0]
    case = Case(spec).build()
    out, lse = case.decode()
    rng = np.random.default_rng(3)
    nr = case.tq * case.Hq
    for b in (0, case.B - 1):
        rows = np.unique(np.concatenate([[0, nr - 1], rng.integers(0, nr, 6)]))
        mask = np.zeros(nr, np.uint8)
        mask[rows] = 1
        ref = case.oracle_decode(b, row_mask=mask)
        assert_close(out[b], lse[b], ref, rows=rows, what="seq %d" % b)
    assert kvq.kvq_wait_timeouts() == 0


def test_repeats_and_pdl_on_off_bitwise_equal(monkeypatch, route):
    """Five runs with programmatic dependent launch and three without give
    identical bits (fixed-order reductions), with a forced split so the
    combine runs too."""
    monkeypatch.setenv("KVQ_SPLIT", "1024")
    spec = W.make_spec("verify", ctx=4000, n_seqs=2, v_type=1, outliers=4)[0]
    case = Case(spec).build()
    monkeypatch.setenv("KVQ_PDL", "1")
    runs = [case.decode() for _ in range(5)]
    monkeypatch.setenv("KVQ_PDL", "0")
    runs += [case.decode() for _ in range(3)]
    for o, l in runs[1:]:
        assert np.array_equal(o, runs[0][0]) and np.array_equal(l, runs[0][1])
    for b in range(case.B):
        assert_close(runs[0][0][b], runs[0][1][b], case.oracle_decode(b), what="seq %d" % b)
