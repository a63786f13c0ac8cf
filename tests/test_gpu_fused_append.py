"""kvq_decode_attn_multi with k16_new / v16_new: the step's new tokens are
appended inside the attention kernel.  The cache bytes must then be exactly
the oracle's (as after kvq_append), the host lengths must grow by t_q, and the
decode must see the new tokens (out / lse vs the oracle)."""
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


def _new_tokens(case):
    ks = np.concatenate([case.kv[b][0][case.lens[b] - case.tq:case.lens[b]] for b in range(case.B)])
    vs = np.concatenate([case.kv[b][1][case.lens[b] - case.tq:case.lens[b]] for b in range(case.B)])
    return to_dev(ks), to_dev(vs)


def _call(case):
    k, v = _new_tokens(case)
    return dict(cache=case.cache, q16=to_dev(case.q), n_q_heads=case.Hq, t_q=case.tq,
                causal_tail=case.spec.causal, seq_lens=torch.tensor(case.lens, dtype=torch.int32, device=dev()),
                max_len=case.max_len, head_map=None, sm_scale=SM_SCALE,
                out=torch.full((case.B, case.tq, case.Hq, 128), float("nan"), device=dev()),
                lse=torch.full((case.B, case.tq, case.Hq), float("nan"), device=dev()), k16_new=k, v16_new=v)


def _run_and_check(cases):
    calls = [_call(c) for c in cases]
    n = kvq.kvq_decode_multi_workspace_size(calls)
    ws = torch.empty(n, dtype=torch.uint8, device=dev()) if n else None
    kvq.kvq_decode_attn_multi(calls, ws)
    torch.cuda.synchronize()
    for case, call in zip(cases, calls):
        assert case.cache.lengths() == case.lens
        o, l = call["out"].cpu().numpy(), call["lse"].cpu().numpy()
        for b in range(case.B):
            assert_cache_bytes(case, b)
            assert_close(o[b], l[b], case.oracle_decode(b), what="%s seq %d" % (case.spec.name, b))


@pytest.mark.parametrize("name,over", [("long", dict(ctx=5000)), ("tiny", dict()),
                                       ("verify", dict(ctx=1538, n_seqs=2)),
                                       ("batched", dict(ctx=3000, n_seqs=5))])
def test_fused_append_matches_the_oracle(name, over):
    _run_and_check([Case(s).build(append_step=False) for s in W.make_spec(name, **over)])


def test_new_tokens_across_split_and_warp_edges(monkeypatch):
    # chunk 64: the 4 new tokens of the 1538-position sequences straddle the
    # split boundary at 1536, and several warps' sub-ranges
    monkeypatch.setenv("KVQ_SPLIT", "64")
    _run_and_check([Case(s).build(append_step=False) for s in W.make_spec("verify", ctx=1538, n_seqs=2)])


def test_full_open_segment_is_rejected():
    case = Case(W.make_spec("long", ctx=640)[1]).build(append_step=True)   # open segment holds its len
    seg = case.cache.seg(0, case.cache.n_segs(0) - 1)
    seg.len = seg.cap                                                        # no room left
    before = case.cache.lengths()
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_decode_attn_multi([_call(case)], None)
    assert e.value.status == kvq.KVQ_ERR_CAPACITY
    assert case.cache.lengths() == before


def test_fused_append_max_tokens_with_a_head_map(monkeypatch):
    # t_q = 8 (the limit), 4 query heads per kv head -> 32 rows, several segments,
    # an uneven explicit head map, splits forced small so the tokens cross splits
    monkeypatch.setenv("KVQ_SPLIT", "128")
    spec = W.make_spec("verify", ctx=1300, n_seqs=2, t_q=8, n_q_heads=24, n_seg=3)[0]
    case = Case(spec).build(append_step=False)
    counts = [4, 4, 4, 4, 4, 2, 1, 1]                       # query heads per kv head
    hm = [k for k, n in enumerate(counts) for _ in range(n)]
    hm = [hm[(7 * h) % case.Hq] for h in range(case.Hq)]    # interleaved
    assert sorted(hm.count(k) for k in range(8)) == sorted(counts)
    call = _call(case)
    call["head_map"] = hm
    kvq.kvq_decode_attn_multi([call], torch.zeros(kvq.kvq_decode_multi_workspace_size([call]), dtype=torch.uint8, device=dev()))
    torch.cuda.synchronize()
    assert case.cache.lengths() == case.lens
    o, l = call["out"].cpu().numpy(), call["lse"].cpu().numpy()
    for b in range(case.B):
        assert_cache_bytes(case, b)
        assert_close(o[b], l[b], case.oracle_decode(b, head_map=hm), what="seq %d" % b)


@pytest.mark.parametrize("split", [None, "64"])
def test_fused_append_on_sixteen_row_tiles(split, monkeypatch):
    """KVQ_ROW_TILE=16: the verify shape's 32 rows per kv head go to two
    16-row CTAs that stream the same positions; only the tile holding the kv
    head's last query token stores the appended tokens, and both see them
    (with 64-position splits the new tokens straddle split edges too)."""
    monkeypatch.setenv("KVQ_ROW_TILE", "16")
    if split:
        monkeypatch.setenv("KVQ_SPLIT", split)
    _run_and_check([Case(s).build(append_step=False) for s in W.make_spec("verify", ctx=1538, n_seqs=2)])
