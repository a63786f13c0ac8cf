"""F16 K (K kept as fp16 values, the query unquantized; the F16 K / q4_0 V
configuration of the RDNA3 page's title and KLD tables) on the GPU against the
oracle's F16-K path on the same seeded inputs: cache bytes bit-exact (fp16 K in
its fragment-order tile, V as on the int8 path), out within 2e-3 and lse within
1e-4.  Covers every workload shape at reduced size, long query chunks (32-row
tiles), a launch mixing F16-K and int8-K caches, the full-size long context,
and the calls F16 K does not support."""
import numpy as np
import pytest
import torch

from quantized_kv_cache_03_gb300 import kvq
from quantized_kv_cache_03_gb300 import workloads as W

from kvq_cases import SM_SCALE, Case, assert_cache_bytes, assert_close, dev, export_logical, to_dev

pytestmark = pytest.mark.gpu

SMALL = {
    "tiny": dict(),
    "single": dict(ctx=3000),                     # outlier channels x10 on K and V
    "long": dict(ctx=5000),                       # 4 segments, main + draft
    "batched": dict(ctx=4096, n_seqs=6),          # ragged lengths, q8_0 V
    "verify": dict(ctx=3000, n_seqs=2),           # t_q = 4 causal, 32 rows per kv head
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _check(case, head_map=None):
    out, lse = case.decode(head_map=head_map)
    for b in range(case.B):
        if case.lens[b] > 0:
            assert_cache_bytes(case, b)
        assert_close(out[b], lse[b], case.oracle_decode(b, head_map=head_map), what="seq %d" % b)


@pytest.mark.parametrize("name", list(SMALL))
def test_config_parity(name):
    for spec in W.make_spec(name, k_type=W.K_F16, **SMALL[name]):
        _check(Case(spec).build())


@pytest.mark.parametrize("vt", [0, 1])
def test_long_chunk_on_row_tiles(vt):
    # 64 causal tokens x 4 query heads: 8 tiles of 32 rows on the split kernel
    spec = W.make_spec("prefill", ctx=900, t_q=64, v_type=vt, k_type=W.K_F16)[0]
    _check(Case(spec).build())


def test_uneven_head_map_and_forced_splits(monkeypatch):
    monkeypatch.setenv("KVQ_SPLIT", "192")
    spec = W.make_spec("verify", ctx=1500, n_seqs=2, t_q=3, n_q_heads=24, k_type=W.K_F16)[0]
    hm = [0] * 7 + [1, 1, 2, 2, 3, 3, 3, 4, 4, 5, 5, 6, 6, 7, 7, 7, 7]
    assert len(hm) == 24
    _check(Case(spec).build(), head_map=hm)


def test_f16_and_int8_caches_in_one_call():
    """One kvq_decode_attn_multi call over an F16-K and an int8-K cache (the
    planner puts them in separate launches)."""
    cf = Case(W.make_spec("long", ctx=2500, k_type=W.K_F16)[0]).build()
    ci = Case(W.make_spec("long", ctx=2500)[1]).build()
    calls = []
    for case in (cf, ci):
        calls.append(dict(cache=case.cache, q16=to_dev(case.q), n_q_heads=case.Hq, t_q=case.tq,
                          causal_tail=case.spec.causal,
                          seq_lens=torch.tensor(case.lens, dtype=torch.int32, device=dev()),
                          max_len=case.max_len, head_map=None, sm_scale=SM_SCALE,
                          out=torch.full((case.B, case.tq, case.Hq, 128), float("nan"), device=dev()),
                          lse=torch.full((case.B, case.tq, case.Hq), float("nan"), device=dev())))
    n = kvq.kvq_decode_multi_workspace_size(calls)
    kvq.kvq_decode_attn_multi(calls, torch.empty(n, dtype=torch.uint8, device=dev()) if n else None)
    torch.cuda.synchronize()
    for case, call in zip((cf, ci), calls):
        assert_close(call["out"][0].cpu().numpy(), call["lse"][0].cpu().numpy(), case.oracle_decode(0),
                     what=case.spec.name)


def test_unsupported_calls_change_nothing():
    case = Case(W.make_spec("long", ctx=700, k_type=W.K_F16)[1]).build(append_step=False)
    L = case.lens[0]
    call = dict(cache=case.cache, q16=to_dev(case.q), n_q_heads=case.Hq, t_q=case.tq, causal_tail=False,
                seq_lens=torch.tensor(case.lens, dtype=torch.int32, device=dev()), max_len=L, head_map=None,
                sm_scale=SM_SCALE, out=torch.empty((1, 1, case.Hq, 128), device=dev()),
                lse=torch.empty((1, 1, case.Hq), device=dev()),
                k16_new=to_dev(case.kv[0][0][L - 1:]), v16_new=to_dev(case.kv[0][1][L - 1:]))
    with pytest.raises(kvq.KvqError) as ei:
        kvq.kvq_decode_attn_multi([call], None)
    assert ei.value.status == kvq.KVQ_ERR_UNSUPPORTED
    assert case.cache.lengths() == [L - 1]
    case.append_step()
    with pytest.raises(kvq.KvqError) as ei:
        case.debug_qk()
    assert ei.value.status == kvq.KVQ_ERR_UNSUPPORTED


def test_long_context_full_size_sampled():
    """Both full-size long-context caches (131072 positions, 4 segments) with
    F16 K: sampled cache positions and query rows against the oracle."""
    rng = np.random.default_rng(3)
    for spec in W.make_spec("long", k_type=W.K_F16):
        case = Case(spec).build()
        out, lse = case.decode()
        L = case.lens[0]
        oc = case.oracle_cache(0)
        got = export_logical(case.cache, 0)
        pos = np.unique(np.concatenate([np.arange(L - 64, L), rng.integers(0, L, 2000)]))
        for name in oc:
            assert np.array_equal(got[name].view(np.uint8)[:, pos] if name != "k16" else got[name][:, pos],
                                  oc[name].view(np.uint8)[:, pos] if name != "k16" else oc[name][:, pos]), name
        nr = case.tq * case.Hq
        rows = np.unique(np.concatenate([[0, nr - 1], rng.integers(0, nr, 6)]))
        mask = np.zeros(nr, np.uint8)
        mask[rows] = 1
        assert_close(out[0], lse[0], case.oracle_decode(0, row_mask=mask), rows=rows, what=spec.name)
