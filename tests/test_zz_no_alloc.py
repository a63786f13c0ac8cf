"""kvq_decode_attn_noalloc: the decode entry point for callers that cannot
allocate device memory (graph-recorded or latency-critical loops where
cudaMalloc is not allowed, runtimes whose allocator owns all device memory).

It must give the same results as kvq_decode_attn with a caller workspace, on
two calls in a row (the second call runs over whatever the first left in the
shared scratch), and reject a call whose partials would not fit the scratch.
This file is collected last on purpose."""
import numpy as np
import pytest
import torch

from quantized_kv_cache_03_gb300 import kvq
from quantized_kv_cache_03_gb300 import workloads as W

from kvq_cases import SM_SCALE, Case, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _enqueue_noalloc(case):
    """Enqueue one kvq_decode_attn_noalloc call on the current stream; returns
    its (out, lse) device tensors (and keeps its inputs alive with them)."""
    s = case.spec
    dev = torch.device("cuda", 0)
    q16 = torch.from_numpy(case.q).to(dev)
    lens = torch.tensor(case.lens, dtype=torch.int32, device=dev)
    out = torch.full((case.B, case.tq, case.Hq, 128), float("nan"), dtype=torch.float32, device=dev)
    lse = torch.full((case.B, case.tq, case.Hq), float("nan"), dtype=torch.float32, device=dev)
    kvq.kvq_decode_attn_noalloc(case.cache, q16, case.Hq, case.tq, s.causal, lens, case.max_len, None, SM_SCALE,
                                out, lse)
    return out, lse, (q16, lens)


def _noalloc(case):
    out, lse, _ = _enqueue_noalloc(case)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy()


def _same_as_workspace_entry(case, o, l, what):
    o_ref, l_ref = case.decode()
    for b in range(case.B):
        assert_close(o[b], l[b], {"out": o_ref[b].astype(np.float64), "lse": l_ref[b].astype(np.float64)},
                     what="%s, seq %d" % (what, b))


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row():
    # two different caches back to back: the second call reuses the scratch
    # the first one filled
    cases = [Case(W.make_spec("long", ctx=6000)[0]).build(),
             Case(W.make_spec("batched", ctx=3000, n_seqs=5)[0]).build()]
    for case in cases:
        assert kvq.kvq_decode_workspace_size(case.cache, case.Hq, case.tq, case.max_len) > 0  # uses scratch
        o_ref, l_ref = case.decode()
        o, l = _noalloc(case)
        for b in range(case.B):
            assert_close(o[b], l[b], {"out": o_ref[b].astype(np.float64), "lse": l_ref[b].astype(np.float64)},
                         what="noalloc vs workspace, seq %d" % b)
        ref = case.oracle_decode(0)
        assert_close(o[0], l[0], ref, what="noalloc vs oracle")


@pytest.mark.parametrize("pdl", ["1", "0"])
def test_noalloc_two_calls_enqueued_back_to_back(pdl, monkeypatch):
    """Two noalloc calls on one stream with no synchronization between them
    (different caches, their own out / lse), with and without programmatic
    dependent launch.  With it, the second call's split kernel may start
    while the first call's combine still reads the shared scratch, so this
    checks that no kernel writes the scratch before its wait on the kernel
    before it.  One synchronize at the end; both results against the
    workspace entry point."""
    monkeypatch.setenv("KVQ_PDL", pdl)
    main, draft = W.make_spec("long", ctx=6000)
    cases = [Case(main).build(), Case(W.make_spec("long", ctx=5000, seed=7)[1]).build()]
    for case in cases:
        assert kvq.kvq_decode_workspace_size(case.cache, case.Hq, case.tq, case.max_len) > 0  # uses scratch
    torch.cuda.synchronize()
    pending = [_enqueue_noalloc(case) for case in cases]
    torch.cuda.synchronize()
    for case, (out, lse, _) in zip(cases, pending):
        _same_as_workspace_entry(case, out.cpu().numpy(), lse.cpu().numpy(), "back-to-back noalloc")


def test_noalloc_rejects_partials_beyond_the_scratch(monkeypatch):
    monkeypatch.setenv("KVQ_SPLIT", "64")    # many splits -> partials above 32 MiB
    spec = W.make_spec("verify", ctx=8192, n_seqs=4)[0]
    case = Case(spec).build()
    need = kvq.kvq_decode_workspace_size(case.cache, case.Hq, case.tq, case.max_len)
    assert need > kvq.NOALLOC_SCRATCH_BYTES
    with pytest.raises(kvq.KvqError) as e:
        _noalloc(case)
    assert e.value.status == kvq.KVQ_ERR_WORKSPACE


def test_no_copy_wait_gave_up():
    # collected last: no attention kernel of the whole GPU suite lost a stage
    assert kvq.kvq_wait_timeouts() == 0
