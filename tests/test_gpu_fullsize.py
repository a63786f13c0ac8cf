"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times (default split policy): cache bytes of sampled positions,
sampled query rows' out/lse, and sampled int32 block scores, each against the
oracle on the same seeded inputs."""
import numpy as np
import pytest

import oracle
from quantized_kv_cache_03_gb300 import workloads as W

from kvq_cases import Case, assert_close, export_logical

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _sample_check(case, seqs, n_rows=6, seed=0):
    rng = np.random.default_rng(seed)
    out, lse = case.decode()
    qc, qs, sc = case.debug_qk()
    for b in seqs:
        L = case.lens[b]
        oc = case.oracle_cache(b)
        got = export_logical(case.cache, b)
        pos = np.unique(np.concatenate([np.arange(min(L, 300)), np.arange(max(0, L - 300), L),
                                        rng.integers(0, L, 2000)]))
        for name in ("kq", "ks", "vq", "vs"):
            assert np.array_equal(got[name].view(np.uint8)[:, pos], oc[name].view(np.uint8)[:, pos]), name
        nr = case.tq * case.Hq
        rows = np.unique(np.concatenate([[0, nr - 1], rng.integers(0, nr, n_rows)]))
        mask = np.zeros(nr, np.uint8)
        mask[rows] = 1
        ref = case.oracle_decode(b, row_mask=mask, want_scores=True)
        assert_close(out[b], lse[b], ref, rows=rows, what="seq %d" % b)
        for r in rows:
            i, h = divmod(int(r), case.Hq)
            vis = L - case.tq + i + 1 if case.spec.causal else L
            assert np.array_equal(sc[b, i, h, :vis], ref["scores"][i, h, :vis]), "scores row %d" % r
            assert np.array_equal(qc[b, i, h], ref["q_codes"][i, h])


def test_long_context_main_and_draft_full_size():
    for spec in W.make_spec("long"):
        case = Case(spec).build()
        _sample_check(case, [0])


def test_batched_full_size():
    spec = W.make_spec("batched")[0]
    case = Case(spec).build()
    lens = np.array(case.lens)
    _sample_check(case, [int(lens.argmax()), int(lens.argmin()), 17], n_rows=4)


def test_verify_full_size():
    spec = W.make_spec("verify")[0]
    case = Case(spec).build()
    _sample_check(case, [0, 15], n_rows=6)


def test_single_full_size_all_rows():
    spec = W.make_spec("single")[0]
    case = Case(spec).build()
    out, lse = case.decode()
    assert_close(out[0], lse[0], case.oracle_decode(0))


def test_long_context_step_as_bench_runs_it():
    """The bench's launch configuration: both full-size caches (131072
    positions, 4 segments each) decoded by one kvq_decode_attn_multi call that
    also appends the step's token (fused append); sampled rows and cache
    positions against the oracle, the appended token's bytes in full."""
    import torch
    from quantized_kv_cache_03_gb300 import kvq
    from kvq_cases import SM_SCALE, dev, to_dev

    rng = np.random.default_rng(1)
    cases = [Case(s).build(append_step=False) for s in W.make_spec("long")]
    calls = []
    for case in cases:
        L = case.lens[0]
        calls.append(dict(cache=case.cache, q16=to_dev(case.q), n_q_heads=case.Hq, t_q=case.tq,
                          causal_tail=case.spec.causal, seq_lens=torch.tensor(case.lens, dtype=torch.int32, device=dev()),
                          max_len=case.max_len, head_map=None, sm_scale=SM_SCALE,
                          out=torch.full((1, case.tq, case.Hq, 128), float("nan"), device=dev()),
                          lse=torch.full((1, case.tq, case.Hq), float("nan"), device=dev()),
                          k16_new=to_dev(case.kv[0][0][L - case.tq:L]), v16_new=to_dev(case.kv[0][1][L - case.tq:L])))
    n = kvq.kvq_decode_multi_workspace_size(calls)
    kvq.kvq_decode_attn_multi(calls, torch.empty(n, dtype=torch.uint8, device=dev()) if n else None)
    torch.cuda.synchronize()
    for case, call in zip(cases, calls):
        L = case.lens[0]
        assert case.cache.lengths() == case.lens
        oc = case.oracle_cache(0)
        got = export_logical(case.cache, 0)
        pos = np.unique(np.concatenate([np.arange(L - 64, L), rng.integers(0, L, 2000)]))
        for name in ("kq", "ks", "vq", "vs"):
            assert np.array_equal(got[name].view(np.uint8)[:, pos], oc[name].view(np.uint8)[:, pos]), name
        nr = case.tq * case.Hq
        rows = np.unique(np.concatenate([[0, nr - 1], rng.integers(0, nr, 5)]))
        mask = np.zeros(nr, np.uint8)
        mask[rows] = 1
        ref = case.oracle_decode(0, row_mask=mask)
        assert_close(call["out"][0].cpu().numpy(), call["lse"][0].cpu().numpy(), ref, rows=rows,
                     what=case.spec.name)
