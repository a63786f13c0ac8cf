"""Pins for the oracle's decode attention.

* exact integer block dots against numpy int64 products of the codes;
* textbook softmax attention (numpy matmul + scipy logsumexp) over the
  dequantized Q, K, V;
* special cases: a one-position context returns its dequantized V, identical
  keys return the mean of dequantized V, t_q = 1 causal equals non-causal,
  splitting the positions and merging the parts by log-sum-exp equals the
  unsplit result, and an online (running-max) softmax equals the two-pass one;
* a row that sees no position returns out = 0, lse = -inf;
* the F16-K variant: on integer K and Q with block absmax 127 (int8 scales
  exactly 1, codes equal to the values) it agrees bit for bit with the int8
  path; identical keys give the mean of V with lse = s + ln n; a dominant key
  selects its V row; K is stored unchanged and V as on the int8 path.
"""
import numpy as np
import pytest
from scipy.special import logsumexp

from quantized_kv_cache_03_gb300 import workloads as W


def _deq_k(c, orc):
    s = c["ks"].view(np.float16).astype(np.float64)
    return c["kq"].astype(np.float64) * np.repeat(s, 32, axis=-1)


def _deq_v(c, vt, orc):
    s = np.repeat(c["vs"].view(np.float16).astype(np.float64), 32, axis=-1)
    if vt == orc.VT_Q8_0:
        return c["vq"].view(np.int8).astype(np.float64) * s
    H, n, half = c["vq"].shape
    blk = c["vq"].reshape(H, n, half // 16, 16).astype(np.int64)
    q = np.concatenate([blk & 0xF, blk >> 4], axis=-1).reshape(H, n, half * 2)
    return (q - 8).astype(np.float64) * s


def _textbook(c, q16, head_map, causal, sm_scale, vt, orc, res):
    """softmax(q_deq k_deq^T * sm_scale) v_deq in fp64, from the oracle's Q codes."""
    K, V = _deq_k(c, orc), _deq_v(c, vt, orc)
    t_q, Hq, D = q16.shape
    L = K.shape[1]
    qs = np.repeat(res["q_scales"].view(np.float16).astype(np.float64), 32, axis=-1)
    Qd = res["q_codes"].astype(np.float64) * qs
    out = np.zeros((t_q, Hq, D))
    lse = np.zeros((t_q, Hq))
    for i in range(t_q):
        n = L - t_q + i + 1 if causal else L
        for h in range(Hq):
            kv = head_map[h]
            s = (K[kv, :n] @ Qd[i, h]) * sm_scale
            lse[i, h] = logsumexp(s)
            out[i, h] = np.exp(s - lse[i, h]) @ V[kv, :n]
    return out, lse


def _case(seed, n, Hkv, Hq, D, t_q, vt, scale_k=1.0):
    rng = np.random.default_rng(seed)
    k = (rng.standard_normal((n, Hkv, D)) * scale_k).astype(np.float16)
    v = rng.standard_normal((n, Hkv, D)).astype(np.float16)
    q = rng.standard_normal((t_q, Hq, D)).astype(np.float16)
    return k, v, q


@pytest.mark.parametrize("vt", [0, 1])
@pytest.mark.parametrize("causal,t_q", [(False, 1), (True, 4), (False, 3)])
def test_against_textbook_and_int_dots(orc, vt, causal, t_q):
    n, Hkv, Hq, D = 77, 2, 6, 64
    k, v, q = _case(11 + vt + t_q, n, Hkv, Hq, D, t_q, vt, scale_k=3.0)
    c = orc.quantize_kv(k, v, vt)
    hm = orc.default_head_map(Hq, Hkv)
    res = orc.decode_seq(c, q, hm, causal, 1 / np.sqrt(D), vt, want_codes=True, want_scores=True)
    # exact integer dots per 32-block
    for i in range(t_q):
        nvis = n - t_q + i + 1 if causal else n
        for h in range(Hq):
            prod = (c["kq"][hm[h], :nvis].astype(np.int64).reshape(nvis, D // 32, 32)
                    * res["q_codes"][i, h].astype(np.int64).reshape(1, D // 32, 32)).sum(-1)
            assert np.array_equal(res["scores"][i, h, :nvis], prod)
    out, lse = _textbook(c, q, hm, causal, 1 / np.sqrt(D), vt, orc, res)
    assert np.max(np.abs(res["out"] - out)) < 1e-12
    assert np.max(np.abs(res["lse"] - lse)) < 1e-12
    # the Q codes follow the K rule
    for i in range(t_q):
        for h in range(Hq):
            for b in range(D // 32):
                cc, s = orc.quant_i8_block(q[i, h, 32 * b:32 * b + 32].view(np.uint16))
                assert np.array_equal(res["q_codes"][i, h, 32 * b:32 * b + 32], cc)
                assert res["q_scales"][i, h, b] == s


@pytest.mark.parametrize("vt", [0, 1])
def test_one_position_returns_deq_v(orc, vt):
    k, v, q = _case(5, 1, 1, 4, 128, 1, vt)
    c = orc.quantize_kv(k, v, vt)
    res = orc.decode_seq(c, q, np.zeros(4, np.int32), False, 0.1, vt, want_scores=True)
    dv = _deq_v(c, vt, orc)[0, 0]
    for h in range(4):
        assert np.array_equal(res["out"][0, h], dv)


@pytest.mark.parametrize("vt", [0, 1])
def test_identical_keys_give_mean_v(orc, vt):
    n = 300
    k, v, q = _case(6, n, 1, 4, 128, 1, vt)
    k[:] = k[0]
    c = orc.quantize_kv(k, v, vt)
    res = orc.decode_seq(c, q, np.zeros(4, np.int32), False, 1 / np.sqrt(128), vt)
    mean = _deq_v(c, vt, orc)[0].mean(axis=0)
    assert np.max(np.abs(res["out"][0] - mean[None])) < 1e-12


def test_causal_single_token_equals_plain(orc):
    k, v, q = _case(7, 50, 2, 4, 64, 1, 0)
    c = orc.quantize_kv(k, v, 0)
    hm = orc.default_head_map(4, 2)
    a = orc.decode_seq(c, q, hm, True, 0.2, 0)
    b = orc.decode_seq(c, q, hm, False, 0.2, 0)
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["lse"], b["lse"])


@pytest.mark.parametrize("cuts", [[1], [64, 65], [10, 200, 201, 390]])
def test_split_and_lse_merge_equals_unsplit(orc, cuts):
    n = 400
    k, v, q = _case(8, n, 2, 10, 128, 1, 1)
    c = orc.quantize_kv(k, v, 1)
    hm = orc.default_head_map(10, 2)
    full = orc.decode_seq(c, q, hm, False, 1 / np.sqrt(128), 1)
    edges = [0] + list(cuts) + [n]
    parts = []
    for a, b in zip(edges[:-1], edges[1:]):
        sub = {kk: vv[:, a:b] for kk, vv in c.items()}
        parts.append(orc.decode_seq(sub, q, hm, False, 1 / np.sqrt(128), 1))
    lses = np.stack([p["lse"] for p in parts])
    M = lses.max(axis=0)
    w = np.exp(lses - M)
    out = sum(p["out"] * w[j][..., None] for j, p in enumerate(parts)) / w.sum(0)[..., None]
    assert np.max(np.abs(out - full["out"])) < 1e-12
    assert np.max(np.abs(M + np.log(w.sum(0)) - full["lse"])) < 1e-12


def test_online_softmax_equals_two_pass(orc):
    n = 257
    k, v, q = _case(9, n, 1, 2, 128, 1, 0, scale_k=4.0)
    c = orc.quantize_kv(k, v, 0)
    sm = 1 / np.sqrt(128)
    res = orc.decode_seq(c, q, np.zeros(2, np.int32), False, sm, 0, want_codes=True, want_scores=True)
    sk = c["ks"].view(np.float16).astype(np.float64)[0]
    V = _deq_v(c, 0, orc)[0]
    for h in range(2):
        sq = res["q_scales"][0, h].view(np.float16).astype(np.float64)
        m, l, o = -np.inf, 0.0, np.zeros(128)
        for t0 in range(0, n, 16):                # running max over chunks
            I = res["scores"][0, h, t0:t0 + 16].astype(np.float64)
            s = sm * (I * sq[None] * sk[t0:t0 + 16]).sum(-1)
            m2 = max(m, s.max())
            a = np.exp(m - m2)
            p = np.exp(s - m2)
            l = l * a + p.sum()
            o = o * a + p @ V[t0:t0 + 16]
            m = m2
        assert np.max(np.abs(o / l - res["out"][0, h])) < 1e-12
        assert abs(m + np.log(l) - res["lse"][0, h]) < 1e-12


def test_no_visible_position(orc):
    k, v, q = _case(10, 3, 1, 2, 64, 4, 0)
    c = orc.quantize_kv(k, v, 0)
    res = orc.decode_seq(c, q, np.zeros(2, np.int32), True, 0.1, 0)
    # L=3, t_q=4: query 0 sees positions 0..-1 (none)
    assert np.all(res["out"][0] == 0) and np.all(np.isneginf(res["lse"][0]))
    assert np.all(np.isfinite(res["lse"][1:]))


def test_row_mask_and_threads(orc):
    k, v, q = _case(12, 90, 2, 8, 128, 2, 0)
    c = orc.quantize_kv(k, v, 0)
    hm = orc.default_head_map(8, 2)
    a = orc.decode_seq(c, q, hm, True, 0.1, 0, n_threads=1)
    mask = np.zeros(16, np.uint8)
    mask[[0, 5, 11]] = 1
    b = orc.decode_seq(c, q, hm, True, 0.1, 0, row_mask=mask, n_threads=4)
    ao, bo = a["out"].reshape(16, -1), b["out"].reshape(16, -1)
    assert np.array_equal(ao[mask == 1], bo[mask == 1])


def test_workload_recipe_runs_through_oracle(orc):
    """A shrunken 'single' workload (outlier channels, GQA 4, q4_0) end to end."""
    spec = W.make_spec("single", ctx=300)[0]
    k, v = W.gen_kv(spec, 0)
    q = W.gen_q(spec)
    c = orc.quantize_kv(k, v, spec.v_type)
    res = orc.decode_seq(c, q[0], orc.default_head_map(spec.n_q_heads, spec.n_kv_heads),
                         spec.causal, 1 / np.sqrt(128), spec.v_type, want_codes=True)
    out, lse = _textbook(c, q[0], orc.default_head_map(spec.n_q_heads, spec.n_kv_heads),
                         spec.causal, 1 / np.sqrt(128), spec.v_type, orc, res)
    assert np.max(np.abs(res["out"] - out)) < 1e-11


# ---------------------------------------------------------------- F16 K --
# The F16-K variant ("Flash Attention for llama.cpp on RDNA3", title and KLD
# tables: F16 K with q4_0 V) keeps K as fp16 values and does not quantize Q.

def _integer_case(seed, n, Hkv, Hq, D, t_q):
    """K and Q integers in [-127, 127] with every 32-block's absmax exactly
    127: the int8 rule then gives scale 1 and codes equal to the values."""
    rng = np.random.default_rng(seed)

    def ints(shape):
        x = rng.integers(-126, 127, size=shape).astype(np.float64)
        xb = x.reshape(shape[:-1] + (shape[-1] // 32, 32))
        xb[..., 0] = np.where(rng.integers(0, 2, size=xb.shape[:-1]) == 0, 127.0, -127.0)
        return xb.reshape(shape).astype(np.float16)

    k = ints((n, Hkv, D))
    q = ints((t_q, Hq, D))
    v = rng.standard_normal((n, Hkv, D)).astype(np.float16)
    return k, v, q


@pytest.mark.parametrize("vt", [0, 1])
def test_f16k_equals_int8_path_on_integer_inputs(vt):
    """On integer K and Q with block absmax 127 both K paths compute the same
    exact scores, so out and lse agree bit for bit."""
    import oracle
    k, v, q = _integer_case(11, 70, 2, 6, 128, 3)
    ci = oracle.quantize_kv(k, v, vt)
    assert np.array_equal(ci["ks"].view(np.float16).astype(np.float64), np.ones_like(ci["ks"], np.float64))
    assert np.array_equal(ci["kq"].astype(np.float64), k.astype(np.float64).transpose(1, 0, 2))
    cf = oracle.quantize_kv(k, v, vt, k_type=oracle.KT_F16)
    hm = oracle.default_head_map(6, 2)
    for causal in (False, True):
        a = oracle.decode_seq(ci, q, hm, causal, 0.01, vt)
        b = oracle.decode_seq(cf, q, hm, causal, 0.01, vt)
        assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["lse"], b["lse"])


def test_f16k_stores_k_unchanged_and_v_as_the_int8_path():
    import oracle
    k, v, q = _case(12, 40, 2, 4, 128, 1, 0)
    ci = oracle.quantize_kv(k, v, 0)
    cf = oracle.quantize_kv(k, v, 0, k_type=oracle.KT_F16)
    assert np.array_equal(cf["k16"], k.view(np.uint16).transpose(1, 0, 2))
    assert np.array_equal(cf["vq"], ci["vq"]) and np.array_equal(cf["vs"], ci["vs"])
    with pytest.raises(ValueError):
        oracle.decode_seq(cf, q, oracle.default_head_map(4, 2), False, 0.1, 0, want_scores=True)


@pytest.mark.parametrize("vt", [0, 1])
def test_f16k_identical_keys_give_the_mean_of_v(vt):
    """All keys equal: every visible position scores the same, so out is the
    mean of the dequantized V rows a query token sees and lse = s + ln n,
    with s = sm_scale * q.k over the fp16 values (Q unquantized)."""
    import oracle
    rng = np.random.default_rng(13)
    n, D, t_q = 37, 128, 4
    key = rng.standard_normal(D).astype(np.float16)
    k = np.broadcast_to(key, (n, 1, D)).copy()
    v = rng.standard_normal((n, 1, D)).astype(np.float16)
    q = rng.standard_normal((t_q, 3, D)).astype(np.float16)
    c = oracle.quantize_kv(k, v, vt, k_type=oracle.KT_F16)
    V = _deq_v(oracle.quantize_kv(k, v, vt), vt, oracle)[0]
    res = oracle.decode_seq(c, q, np.zeros(3, np.int32), True, 0.125, vt)
    for i in range(t_q):
        m = n - t_q + i + 1
        for h in range(3):
            s = 0.125 * float(np.dot(q[i, h].astype(np.float64), key.astype(np.float64)))
            np.testing.assert_allclose(res["out"][i, h], V[:m].mean(axis=0), rtol=0, atol=1e-12)
            assert abs(res["lse"][i, h] - (s + np.log(m))) < 1e-12


def test_f16k_dominant_key_selects_its_value():
    """One key aligned with the query at a large scale: the softmax puts all
    its weight there, out equals that position's dequantized V row."""
    import oracle
    rng = np.random.default_rng(14)
    n, D = 50, 128
    q = rng.standard_normal((1, 1, D)).astype(np.float16)
    k = (rng.standard_normal((n, 1, D)) * 0.01).astype(np.float16)
    k[17, 0] = (q[0, 0].astype(np.float32) * 4).astype(np.float16)
    v = rng.standard_normal((n, 1, D)).astype(np.float16)
    c = oracle.quantize_kv(k, v, 1, k_type=oracle.KT_F16)
    V = _deq_v(oracle.quantize_kv(k, v, 1), 1, oracle)[0]
    res = oracle.decode_seq(c, q, np.zeros(1, np.int32), False, 1.0, 1)
    np.testing.assert_allclose(res["out"][0, 0], V[17], rtol=0, atol=1e-9)
