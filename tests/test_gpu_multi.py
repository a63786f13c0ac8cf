"""kvq_decode_attn_multi: several caches' decode calls in one launch plan must
give, for every call, what the oracle gives for that cache alone (same
tolerances as the single-call parity tests)."""
import numpy as np
import pytest
import torch

from quantized_kv_cache_03_gb300 import kvq
from quantized_kv_cache_03_gb300 import workloads as W

from kvq_cases import SM_SCALE, Case, assert_close, dev, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _call(case, out=None, lse=None, head_map=None):
    s = case.spec
    out = torch.full((case.B, case.tq, case.Hq, 128), float("nan"), dtype=torch.float32, device=dev()) if out is None else out
    lse = torch.full((case.B, case.tq, case.Hq), float("nan"), dtype=torch.float32, device=dev()) if lse is None else lse
    return dict(cache=case.cache, q16=to_dev(case.q), n_q_heads=case.Hq, t_q=case.tq, causal_tail=s.causal,
                seq_lens=torch.tensor(case.lens, dtype=torch.int32, device=dev()), max_len=case.max_len,
                head_map=head_map, sm_scale=SM_SCALE, out=out, lse=lse)


def _run(calls):
    n = kvq.kvq_decode_multi_workspace_size(calls)
    ws = torch.empty(n, dtype=torch.uint8, device=dev()) if n else None
    kvq.kvq_decode_attn_multi(calls, ws)
    torch.cuda.synchronize()


def _check(case, call, head_map=None):
    o, l = call["out"].cpu().numpy(), call["lse"].cpu().numpy()
    for b in range(case.B):
        ref = case.oracle_decode(b, head_map=head_map)
        assert_close(o[b], l[b], ref, what="%s seq %d" % (case.spec.name, b))


def test_main_and_draft_in_one_launch():
    cases = [Case(s).build() for s in W.make_spec("long", ctx=6000)]
    calls = [_call(c) for c in cases]
    _run(calls)
    for c, call in zip(cases, calls):
        _check(c, call)


def test_mixed_formats_shapes_and_head_maps():
    # q4_0 causal t_q = 4 with an uneven head map, q4_0 single and q8_0 tiny: two
    # V formats -> two launches, three head tables
    ver = Case(W.make_spec("verify", ctx=1500, n_seqs=2)[0]).build()
    hm = [(3 * h) % 8 for h in range(ver.Hq)]
    hm = [min(x, 7) for x in hm]
    sgl = Case(W.make_spec("single", ctx=3000)[0]).build()
    tny = Case(W.make_spec("tiny")[0]).build()
    calls = [_call(ver, head_map=hm), _call(sgl), _call(tny)]
    _run(calls)
    _check(ver, calls[0], head_map=hm)
    _check(sgl, calls[1])
    _check(tny, calls[2])


def test_multi_matches_single_calls_with_forced_splits(monkeypatch):
    monkeypatch.setenv("KVQ_SPLIT", "192")
    cases = [Case(s).build() for s in W.make_spec("long", ctx=2500)]
    calls = [_call(c) for c in cases]
    _run(calls)
    for c, call in zip(cases, calls):
        o, l = c.decode()
        assert np.array_equal(call["out"].cpu().numpy(), o)   # same chunk -> same splits and order
        assert np.array_equal(call["lse"].cpu().numpy(), l)
        _check(c, call)


def test_multi_rejects_a_bad_call_before_enqueueing():
    cases = [Case(s).build() for s in W.make_spec("long", ctx=1000)]
    calls = [_call(c) for c in cases]
    calls[1]["n_q_heads"] = 15                      # not a multiple of 4 kv heads, no head map
    with pytest.raises(kvq.KvqError) as e:
        _run(calls)
    assert e.value.status == kvq.KVQ_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.isnan(calls[0]["out"]).all()        # the valid call did not run either
    kvq.kvq_decode_attn_multi([], None)              # n = 0 is a no-op
