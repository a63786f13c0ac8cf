"""Chunked prefill over the quantized cache: many query tokens per sequence
(t_q up to 4096), the chunk causal among its own tokens.  Calls with more than
32 query rows per kv head run on the tcgen05 kernel (128-row tiles, TMEM
accumulators); KVQ_PREFILL=0 sends them to the split kernel's 32-row tiles, and
every case below runs on both.  The cases span several row tiles with a ragged
last one, splits that lie wholly past a tile's causal limit, uneven head maps
(tiles past a small group's rows), an empty context, a non-causal chunk and a
mixed launch with a decode call, all against the oracle on the same seeded
inputs: cache bytes bit-exact, out within 2e-3 and lse within 1e-4.

The raw int32 block scores and the query codes are compared bit for bit with
the oracle through the kvq_debug_qk hook, which runs the kernel the decode call
picks and reports which one ran: the tests assert that it is the tcgen05
kernel (its scores are the TMEM accumulators of its fp16 MMAs on exact integer
operands) or the split kernel, as the fixture selects."""

import numpy as np
import pytest
import torch

from quantized_kv_cache_03_gb300 import kvq
from quantized_kv_cache_03_gb300 import workloads as W

import oracle

from kvq_cases import SM_SCALE, Case, assert_cache_bytes, assert_close, dev, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.fixture(params=["tcgen05", "rowtile"], autouse=True)
def kernel(request, monkeypatch):
    monkeypatch.setenv("KVQ_PREFILL", "1" if request.param == "tcgen05" else "0")
    return request.param


def _check_all(case, head_map=None, scores=False):
    out, lse = case.decode(head_map=head_map)
    for b in range(case.B):
        assert_cache_bytes(case, b)
        ref = case.oracle_decode(b, head_map=head_map, want_scores=scores)
        assert_close(out[b], lse[b], ref, what="seq %d" % b)
    return out, lse


def _plan_kernel(case):
    call = dict(cache=case.cache, n_q_heads=case.Hq, t_q=case.tq, causal_tail=case.spec.causal,
                max_len=case.max_len, head_map=None, sm_scale=SM_SCALE)
    lns, _ = kvq.kvq_debug_plan([call], 152)
    return {ln["kernel"] for ln in lns}


def _check_scores(case, kernel, rows=None):
    """Query codes / scales and every position's int32 block scores of the
    dump against the oracle (causal mask off: the hook dumps every position
    below the sequence length), on the kernel the fixture selects."""
    want = "tcgen05" if kernel == "tcgen05" else "split"
    assert _plan_kernel(case) == {"prefill" if kernel == "tcgen05" else "split"}
    qc, qs, sc = case.debug_qk()
    assert case.dump_kernel == want, "the dump ran on the %s kernel" % case.dump_kernel
    for b in range(case.B):
        L = case.lens[b]
        ref = case.oracle_decode(b, want_scores=True, causal=False)
        assert np.array_equal(qc[b], ref["q_codes"]), "query codes, seq %d" % b
        assert np.array_equal(qs[b], ref["q_scales"]), "query scales, seq %d" % b
        got, exp = sc[b, :, :, :L], ref["scores"]
        if not np.array_equal(got, exp):
            bad = np.argwhere(got != exp)
            raise AssertionError("int32 block scores differ at %d places, first (token, head, pos, block) %s"
                                 % (len(bad), bad[:5].tolist()))


@pytest.mark.parametrize("vt", [0, 1])
def test_chunk_of_64_tokens_all_rows_and_scores(vt, kernel):
    # 64 tokens x 4 query heads = 256 rows per kv head: 2 tcgen05 row tiles (8 of 32 rows)
    spec = W.make_spec("prefill", ctx=1000, t_q=64, v_type=vt)[0]
    case = Case(spec).build()
    _check_all(case)
    _check_scores(case, kernel)


@pytest.mark.parametrize("split", [192, 640])
def test_scores_over_splits_ragged_tiles_and_segments(split, kernel, monkeypatch):
    """Two sequences, three segments each, 40 tokens x 6 heads (240 rows per kv
    head: a ragged second 128-row tile), positions split in chunks that cut
    KV tiles at split and segment edges."""
    monkeypatch.setenv("KVQ_SPLIT", str(split))
    spec = W.make_spec("prefill", ctx=1500, t_q=40, n_seqs=2, n_seg=3, n_q_heads=48, n_kv_heads=8, v_type=1)[0]
    spec.lengths[:] = [1500, 777]
    spec.segments[:] = [W._cuts(spec.rng(9, b), int(L), 3, 40) for b, L in enumerate(spec.lengths)]
    case = Case(spec).build()
    _check_all(case)
    _check_scores(case, kernel)


def test_chunk_full_size_sampled_scores(kernel):
    """The 512-token chunk over 32768 positions as the benchmark runs it: the
    dump of every row (8.6 GB of int32 scores on the device), compared on
    sampled rows (first and last of the chunk, random ones) at every position."""
    if kernel != "tcgen05":
        pytest.skip("the split kernel's dump at full size is covered by the decode workloads")
    spec = W.make_spec("prefill")[0]
    case = Case(spec).build()
    assert _plan_kernel(case) == {"prefill"}
    L, tq, Hq = case.lens[0], case.tq, case.Hq
    q16 = to_dev(case.q)
    lens = torch.tensor(case.lens, dtype=torch.int32, device=dev())
    qc = torch.zeros((1, tq, Hq, 128), dtype=torch.int8, device=dev())
    qs = torch.zeros((1, tq, Hq, 4), dtype=torch.int16, device=dev())
    sc = torch.zeros((1, tq, Hq, L, 4), dtype=torch.int32, device=dev())
    assert kvq.kvq_debug_qk(case.cache, q16, Hq, tq, lens, L, None, qc, qs, sc) == "tcgen05"
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    nr = tq * Hq
    rows = np.unique(np.concatenate([[0, 1, Hq - 1, nr - Hq, nr - 1], rng.integers(0, nr, 11)]))
    # the oracle on just these rows: one query token whose heads are the sampled (token, head) rows
    hm_full = np.arange(Hq) // (Hq // spec.n_kv_heads)
    q_sub = case.q[0].reshape(nr, 128)[rows][None]
    ref = oracle.decode_seq(case.oracle_cache(0), q_sub, hm_full[rows % Hq].astype(np.int32), False, SM_SCALE,
                            spec.v_type, want_codes=True, want_scores=True, n_threads=8)
    got_sc = sc.view(nr, L, 4)[torch.as_tensor(rows, device=dev())].cpu().numpy()
    assert np.array_equal(qc.view(nr, 128).cpu().numpy()[rows], ref["q_codes"][0])
    assert np.array_equal(qs.view(nr, 4).cpu().numpy().view(np.uint16)[rows], ref["q_scales"][0])
    if not np.array_equal(got_sc, ref["scores"][0]):
        bad = np.argwhere(got_sc != ref["scores"][0])
        raise AssertionError("int32 block scores differ at %d places, first %s" % (len(bad), bad[:5].tolist()))
    del sc


def test_splits_past_a_row_tiles_causal_limit(monkeypatch):
    # context of 100 positions, chunk of 600: the first row tiles see ~100
    # positions, so with 64-position splits most of their splits hold nothing
    monkeypatch.setenv("KVQ_SPLIT", "64")
    spec = W.make_spec("prefill", ctx=700, t_q=600, n_q_heads=8, n_kv_heads=2, v_type=0)[0]
    _check_all(Case(spec).build())


@pytest.mark.parametrize("vt", [0, 1])
def test_prefill_of_an_empty_context(vt):
    # the whole sequence is the chunk; 300 x 4 = 1200 rows: 37.5 row tiles
    spec = W.make_spec("prefill", ctx=300, t_q=300, n_seg=1, n_q_heads=16, n_kv_heads=4, v_type=vt)[0]
    out, lse = _check_all(Case(spec).build())
    assert np.all(np.isfinite(lse))


def test_uneven_head_map_ragged_row_tiles():
    # kv head 0 takes 9 query heads (360 rows, 12 tiles), kv head 7 one (40 rows)
    spec = W.make_spec("prefill", ctx=1500, t_q=40, n_q_heads=24, v_type=1)[0]
    hm = [0] * 9 + [1, 1, 1, 2, 2, 2, 3, 3, 4, 4, 5, 5, 6, 6, 7]
    assert len(hm) == 24
    _check_all(Case(spec).build(), head_map=hm)


def test_batched_chunks_of_ragged_contexts():
    """Three sequences, each with its own context length, one 80-token chunk
    each, in one call (one work group of three sequences)."""
    spec = W.make_spec("prefill", ctx=1400, t_q=80, n_seqs=3, v_type=1)[0]
    spec.lengths[:] = [1400, 333, 980]
    spec.segments[:] = [W._cuts(spec.rng(9, b), int(L), 2, 80) for b, L in enumerate(spec.lengths)]
    _check_all(Case(spec).build())


def test_non_causal_chunk():
    spec = W.make_spec("prefill", ctx=2000, t_q=100, causal=False, v_type=0)[0]
    _check_all(Case(spec).build())


def test_chunk_and_decode_calls_in_one_launch():
    """A prefill chunk and a decode step of another cache fused in one
    kvq_decode_attn_multi call (one launch at the chunk's row-tile size)."""
    pre = Case(W.make_spec("prefill", ctx=1200, t_q=48, v_type=0)[0]).build()
    dec = Case(W.make_spec("long", ctx=2000)[0]).build()
    calls = []
    for case in (pre, dec):
        calls.append(dict(cache=case.cache, q16=to_dev(case.q), n_q_heads=case.Hq, t_q=case.tq,
                          causal_tail=case.spec.causal,
                          seq_lens=torch.tensor(case.lens, dtype=torch.int32, device=dev()),
                          max_len=case.max_len, head_map=None, sm_scale=SM_SCALE,
                          out=torch.full((case.B, case.tq, case.Hq, 128), float("nan"), device=dev()),
                          lse=torch.full((case.B, case.tq, case.Hq), float("nan"), device=dev())))
    n = kvq.kvq_decode_multi_workspace_size(calls)
    kvq.kvq_decode_attn_multi(calls, torch.empty(n, dtype=torch.uint8, device=dev()) if n else None)
    torch.cuda.synchronize()
    for case, call in zip((pre, dec), calls):
        assert_close(call["out"][0].cpu().numpy(), call["lse"][0].cpu().numpy(), case.oracle_decode(0),
                     what=case.spec.name)


def test_fused_append_is_limited_to_short_chunks():
    spec = W.make_spec("prefill", ctx=640, t_q=kvq.MAX_T_Q_APPEND + 1, v_type=0)[0]
    case = Case(spec).build(append_step=False)
    L = case.lens[0]
    call = dict(cache=case.cache, q16=to_dev(case.q), n_q_heads=case.Hq, t_q=case.tq, causal_tail=True,
                seq_lens=torch.tensor(case.lens, dtype=torch.int32, device=dev()), max_len=L, head_map=None,
                sm_scale=SM_SCALE, out=torch.empty((1, case.tq, case.Hq, 128), device=dev()),
                lse=torch.empty((1, case.tq, case.Hq), device=dev()),
                k16_new=to_dev(case.kv[0][0][L - case.tq:]), v16_new=to_dev(case.kv[0][1][L - case.tq:]))
    with pytest.raises(kvq.KvqError) as ei:
        kvq.kvq_decode_attn_multi([call], None)
    assert ei.value.status == kvq.KVQ_ERR_UNSUPPORTED
    assert case.cache.lengths() == [L - case.tq]


def test_chunk_full_size_sampled_rows():
    """The 512-token chunk over 32768 positions as the benchmark runs it:
    sampled rows (first, last, random) and cache positions against the oracle."""
    spec = W.make_spec("prefill")[0]
    case = Case(spec).build()
    out, lse = case.decode()
    rng = np.random.default_rng(0)
    L = case.lens[0]
    oc = case.oracle_cache(0)
    from kvq_cases import export_logical
    got = export_logical(case.cache, 0)
    pos = np.unique(np.concatenate([np.arange(L - 600, L), rng.integers(0, L, 2000)]))
    for name in ("kq", "ks", "vq", "vs"):
        assert np.array_equal(got[name].view(np.uint8)[:, pos], oc[name].view(np.uint8)[:, pos]), name
    nr = case.tq * case.Hq
    rows = np.unique(np.concatenate([[0, 1, 31, 32, nr - 1], rng.integers(0, nr, 24)]))
    mask = np.zeros(nr, np.uint8)
    mask[rows] = 1
    ref = case.oracle_decode(0, row_mask=mask)
    assert_close(out[0], lse[0], ref, rows=rows, what="prefill full size")


def test_uneven_split_of_a_one_wave_launch(kernel, monkeypatch):
    """A 512-token chunk over 3000 positions, 8 kv heads x 16 row tiles: 128
    units on 152 SMs, so the launch splits every unit unevenly (large pieces
    first, small ones on the spare SMs, then the combine).  The first row
    tiles' causal limit falls before the split point, so their small pieces see
    nothing.  Sampled rows of every row tile against the oracle, the int32 block
    scores of the same rows bit for bit, and the same rows with the split off
    (KVQ_PREFILL_BALANCE=0) also within the tolerance."""
    if kernel != "tcgen05":
        pytest.skip("the uneven split is a tcgen05 launch policy")
    spec = W.make_spec("prefill", ctx=3000, v_type=1)[0]
    case = Case(spec).build()
    call = dict(cache=case.cache, n_q_heads=case.Hq, t_q=case.tq, causal_tail=True, max_len=case.max_len,
                head_map=None, sm_scale=SM_SCALE)
    ln = kvq.kvq_debug_plan([call], 152)[0][0]
    L, tq, Hq = case.lens[0], case.tq, case.Hq
    assert ln["kernel"] == "prefill" and ln["n_ctas"] == 256 and ln["chunk0"] < L
    assert ln["chunk0"] > L - tq + 32   # row tile 0 (tokens 0-31) ends before the split point
    nr = tq * Hq
    rng = np.random.default_rng(3)
    # rows of every row tile (128 rows = 32 tokens x 4 heads per kv head)
    rows = np.unique(np.concatenate([[0, 1, nr - 1], (np.arange(16) * 32 + 31) * Hq + 5, rng.integers(0, nr, 40)]))
    mask = np.zeros(nr, np.uint8)
    mask[rows] = 1
    ref = case.oracle_decode(0, row_mask=mask)
    out, lse = case.decode()
    assert_close(out[0], lse[0], ref, rows=rows, what="uneven split")
    # the dump runs on the same plan: int32 block scores of the sampled rows
    q16 = to_dev(case.q)
    lens = torch.tensor(case.lens, dtype=torch.int32, device=dev())
    qc = torch.zeros((1, tq, Hq, 128), dtype=torch.int8, device=dev())
    qs = torch.zeros((1, tq, Hq, 4), dtype=torch.int16, device=dev())
    sc = torch.zeros((1, tq, Hq, L, 4), dtype=torch.int32, device=dev())
    assert kvq.kvq_debug_qk(case.cache, q16, Hq, tq, lens, L, None, qc, qs, sc) == "tcgen05"
    torch.cuda.synchronize()
    hm_full = np.arange(Hq) // (Hq // spec.n_kv_heads)
    q_sub = case.q[0].reshape(nr, 128)[rows][None]
    refs = oracle.decode_seq(case.oracle_cache(0), q_sub, hm_full[rows % Hq].astype(np.int32), False, SM_SCALE,
                             spec.v_type, want_scores=True, n_threads=8)
    got_sc = sc.view(nr, L, 4)[torch.as_tensor(rows, device=dev())].cpu().numpy()
    assert np.array_equal(got_sc, refs["scores"][0])
    # the split-major CTA order and the two-partial combine repeat bit for
    # bit, with and without programmatic dependent launch
    again = [case.decode() for _ in range(2)]
    monkeypatch.setenv("KVQ_PDL", "0")
    again.append(case.decode())
    monkeypatch.delenv("KVQ_PDL")
    for o2, l2 in again:
        assert np.array_equal(o2, out) and np.array_equal(l2, lse)
    monkeypatch.setenv("KVQ_PREFILL_BALANCE", "0")
    assert kvq.kvq_debug_plan([call], 152)[0][0]["n_ctas"] == 128
    out0, lse0 = case.decode()
    assert_close(out0[0], lse0[0], ref, rows=rows, what="one split")


def test_repeats_and_pdl_on_off_bitwise_equal(monkeypatch):
    """Five runs with programmatic dependent launch and three without give
    identical bits: every reduction has a fixed order, so a stale read through
    a mis-ordered barrier phase or buffer reuse would show as a difference."""
    spec = W.make_spec("prefill", ctx=3000, t_q=96, v_type=0)[0]
    case = Case(spec).build()
    monkeypatch.setenv("KVQ_PDL", "1")
    runs = [case.decode() for _ in range(5)]
    monkeypatch.setenv("KVQ_PDL", "0")
    runs += [case.decode() for _ in range(3)]
    for o, l in runs[1:]:
        assert np.array_equal(o, runs[0][0]) and np.array_equal(l, runs[0][1])
    assert_close(runs[0][0][0], runs[0][1][0], case.oracle_decode(0))
