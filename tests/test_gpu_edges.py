"""Edge cases of the decode path on the GPU against the oracle: a one-position
context, zero and extreme-valued blocks, causal rows that see nothing in a
split or at all, uneven explicit head maps, many short segments, several
launch groups, empty sequences, forced split sizes and PDL on/off equality."""
import os

import numpy as np
import pytest

from quantized_kv_cache_03_gb300 import workloads as W

from kvq_cases import LSE_TOL, OUT_TOL, Case, assert_cache_bytes, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.fixture
def env(monkeypatch):
    return monkeypatch


def _check(case, head_map=None, scores=True):
    out, lse = case.decode(head_map=head_map)
    for b in range(case.B):
        if case.lens[b] > 0:
            assert_cache_bytes(case, b)
        ref = case.oracle_decode(b, head_map=head_map, want_scores=scores)
        assert_close(out[b], lse[b], ref, what="seq %d" % b)
    return out, lse


def _spec(name="single", **kw):
    return W.make_spec(name, **kw)[0]


@pytest.mark.parametrize("vt", [0, 1])
def test_one_position_context_with_outliers(vt):
    spec = _spec("single", ctx=1, v_type=vt)
    case = Case(spec).build()
    out, lse = _check(case)
    assert np.all(np.isfinite(out))


@pytest.mark.parametrize("vt", [0, 1])
def test_zero_and_extreme_blocks(vt):
    spec = _spec("single", ctx=700, v_type=vt)
    k, v = W.gen_kv(spec, 0)
    k[10:20, :, 0:32] = 0                          # all-zero blocks -> scale 0
    v[30:40, :, 32:64] = 0
    k[50, 0, :] = np.float16(65504)                # largest fp16
    k[51, 1, ::2] = np.float16(-65504)
    v[52, 2, 64:96] = np.float16(-65504)
    v[53, 3, :] = np.float16(2.0 ** -24)           # smallest subnormal
    k[54, 4, :] = np.float16(6.1e-5)
    v[60:64] = np.float16(1000.0)
    case = Case(spec, kv=[(k, v)]).build()
    for b in range(case.B):
        assert_cache_bytes(case, b)
    qc, qs, sc = case.debug_qk()
    ref = case.oracle_decode(0, want_scores=True)
    assert np.array_equal(sc[0, 0, :, :case.lens[0]], ref["scores"][0])
    out, lse = case.decode()
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    # out at the usual bar; the +-65504 keys make some rows' softmax one-hot
    # with scores near 1e5..1e6, where one fp32 ulp (0.008..0.06) exceeds the
    # absolute lse bar of 1e-4, so lse is held to 1e-4 absolute where
    # |lse| <= 1 and to 1e-5 relative above (a few hundred ulps of the
    # four-term fp32 score sum and the log)
    eo = float(np.abs(out[0] - ref["out"]).max())
    assert eo <= OUT_TOL, "max|out-oracle| = %.3e" % eo
    rel = np.abs(lse[0] - ref["lse"]) / np.maximum(1.0, np.abs(ref["lse"]))
    assert rel.max() < 1e-5
    small = np.abs(ref["lse"]) <= 1.0
    assert np.all(np.abs(lse[0] - ref["lse"])[small] <= LSE_TOL)


def test_causal_tail_rows_seeing_nothing_in_a_split(env):
    env.setenv("KVQ_SPLIT", "64")
    spec = _spec("verify", ctx=130, n_seqs=2)      # split edge at 128 inside the 4-token tail
    case = Case(spec).build()
    _check(case)


def test_causal_query_seeing_only_position_zero():
    spec = _spec("verify", ctx=4, n_seqs=1)
    case = Case(spec).build()
    out, lse = _check(case)


def test_uneven_explicit_head_map():
    spec = _spec("single", ctx=999)
    spec.n_q_heads = 12                             # 12 query heads over 8 kv heads, groups 0..3 wide
    hm = [7, 0, 0, 3, 7, 7, 1, 0, 3, 5, 7, 1]
    q = np.random.default_rng(4).standard_normal((1, 1, 12, 128)).astype(np.float16)
    case = Case(spec, q=q).build()
    _check(case, head_map=hm)
    qc, qs, sc = case.debug_qk(head_map=hm)
    ref = case.oracle_decode(0, head_map=hm, want_scores=True)
    assert np.array_equal(qc[0], ref["q_codes"])
    assert np.array_equal(sc[0, 0, :, :999], ref["scores"][0])


def test_many_short_segments():
    spec = _spec("long", ctx=2500)
    spec.segments = [np.array([1, 63, 64, 65, 7, 300, 1000, 1, 999], np.int64)]
    assert spec.segments[0].sum() == 2500
    case = Case(spec).build()
    _check(case)


def test_two_launch_groups_and_an_empty_sequence():
    spec = _spec("batched", ctx=600, n_seqs=70)     # > 64 sequences -> two launch groups
    spec.lengths[5] = 0                              # a sequence without any segment
    spec.segments[5] = np.array([0], np.int64)
    case = Case(spec)
    case.build()
    _check(case, scores=False)


def test_forced_splits_match_unsplit(env):
    spec = W.make_spec("long", ctx=3000)[1]
    case = Case(spec).build()
    env.setenv("KVQ_SPLIT", "100000")
    o1, l1 = case.decode()
    env.setenv("KVQ_SPLIT", "64")
    o2, l2 = case.decode()
    ref = case.oracle_decode(0)
    assert_close(o1[0], l1[0], ref, what="one split")
    assert_close(o2[0], l2[0], ref, what="47 splits")


def test_pdl_on_off_bitwise_equal(env):
    spec = W.make_spec("long", ctx=20000)[0]
    case = Case(spec).build()
    env.setenv("KVQ_PDL", "1")
    runs = [case.decode() for _ in range(5)]
    env.setenv("KVQ_PDL", "0")
    runs += [case.decode() for _ in range(3)]
    for o, l in runs[1:]:
        assert np.array_equal(o, runs[0][0]) and np.array_equal(l, runs[0][1])
