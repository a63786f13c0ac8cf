"""The attention kernel's bounded copy waits, driven to run out on purpose.

kvq_debug_lose_stage runs the decode call on a test flavour of the split-KV
kernel in which warp 0 of the first CTA arms one copy stage's barrier without
issuing the stage's copies.  That wait (given a short limit) gives up; the warp
then waits, with the normal limit, for every copy it did issue, the CTA writes
NaN for its query rows and the per-device wait counter grows by one.  No
kernel faults or waits without a limit.  The test checks the counter and the
status of kvq_wait_timeouts, the NaN rows (kv head 0's query rows, whose first
split that CTA is), every other row against the oracle, the counter reset,
and that a normal decode on the same device is correct afterwards."""
import ctypes

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


@pytest.mark.parametrize("ctx", [6000, 16000, 28000])
def test_a_lost_stage_gives_up_poisons_its_rows_and_counts(ctx, monkeypatch):
    # 2048-position splits of 16 warps: warp 0 of each CTA streams 128
    # positions, four copy stages, so its second stage exists.  3 splits per
    # kv head at 6000 positions and 8 at 16000 (the combine's row-per-warp
    # form with 4 and with 12 slots), 14 at 28000 (one CTA per row): every
    # form must carry the poisoned partial into NaN.
    monkeypatch.setenv("KVQ_SPLIT", "2048")
    spec = W.make_spec("long", ctx=ctx)[0]           # 40 query / 8 kv heads, q4_0 V, 4 segments
    case = Case(spec).build()
    call = dict(cache=case.cache, n_q_heads=case.Hq, t_q=1, causal_tail=False, max_len=case.max_len,
                head_map=None, sm_scale=SM_SCALE)
    (ln,), ws_bytes = kvq.kvq_debug_plan([call], 152)
    assert (ln["kernel"], ln["n_tiles8"], ln["warps"], ln["chunk"]) == ("split", 1, 16, 2048)
    torch.cuda.synchronize()
    kvq.kvq_reset_wait_timeouts()
    assert kvq.kvq_wait_timeouts() == 0
    lens = torch.tensor(case.lens, dtype=torch.int32, device=dev())
    out = torch.zeros((1, 1, case.Hq, 128), dtype=torch.float32, device=dev())
    lse = torch.zeros((1, 1, case.Hq), dtype=torch.float32, device=dev())
    n = kvq.kvq_decode_workspace_size(case.cache, case.Hq, 1, case.max_len)
    ws = torch.empty(n, dtype=torch.uint8, device=dev())
    try:
        kvq.kvq_debug_lose_stage(case.cache, to_dev(case.q), case.Hq, 1, False, lens, case.max_len, None,
                                 SM_SCALE, out, lse, ws)
        torch.cuda.synchronize()
        count = ctypes.c_uint32(0)
        st = kvq.load().kvq_wait_timeouts(ctypes.byref(count))
        assert st == kvq.KVQ_ERR_TIMEOUT and count.value == 1, "status %d, count %d" % (st, count.value)
    finally:
        torch.cuda.synchronize()
        kvq.kvq_reset_wait_timeouts()
    o, l = out.cpu().numpy()[0, 0], lse.cpu().numpy()[0, 0]
    group = case.Hq // spec.n_kv_heads
    lost = np.arange(case.Hq) < group                  # the query heads of kv head 0
    assert np.all(np.isnan(o[lost])) and np.all(np.isnan(l[lost]))
    ref = case.oracle_decode(0)
    assert_close(o[~lost][None], l[~lost][None], {"out": ref["out"][0][~lost][None], "lse": ref["lse"][0][~lost][None]},
                 what="rows of the other kv heads")
    kvq.kvq_reset_wait_timeouts()
    assert kvq.kvq_wait_timeouts() == 0
    # the device stays usable: the normal decode is correct and counts nothing
    o2, l2 = case.decode()
    assert_close(o2[0], l2[0], ref, what="decode after the lost stage")
    assert kvq.kvq_wait_timeouts() == 0


def test_lose_stage_refuses_other_kernel_forms():
    # 32 query rows per kv head plan on the 32-row tiles: no test flavour there
    spec = W.make_spec("verify", ctx=600, n_seqs=1)[0]
    case = Case(spec).build()
    lens = torch.tensor(case.lens, dtype=torch.int32, device=dev())
    out = torch.zeros((1, case.tq, case.Hq, 128), dtype=torch.float32, device=dev())
    lse = torch.zeros((1, case.tq, case.Hq), dtype=torch.float32, device=dev())
    n = kvq.kvq_decode_workspace_size(case.cache, case.Hq, case.tq, case.max_len)
    ws = torch.empty(n, dtype=torch.uint8, device=dev()) if n else None
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_debug_lose_stage(case.cache, to_dev(case.q), case.Hq, case.tq, True, lens, case.max_len, None,
                                 SM_SCALE, out, lse, ws)
    assert e.value.status == kvq.KVQ_ERR_UNSUPPORTED
    assert kvq.kvq_wait_timeouts() == 0
