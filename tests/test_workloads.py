"""The seeded input generator: determinism, shapes and the workload recipes."""
import numpy as np

from quantized_kv_cache_03_gb300 import workloads as W


def test_recipes_full_size_metadata():
    tiny = W.make_spec("tiny")[0]
    assert (tiny.n_seqs, tiny.n_kv_heads, tiny.n_q_heads, tiny.max_len, tiny.v_type) == (1, 1, 4, 256, W.V_Q8_0)
    single = W.make_spec("single")[0]
    assert (single.n_q_heads, single.n_kv_heads, single.max_len, single.outlier_channels) == (32, 8, 8192, 4)
    main, draft = W.make_spec("long")
    assert (main.n_q_heads, main.n_kv_heads, draft.n_q_heads, draft.n_kv_heads) == (40, 8, 16, 4)
    for s in (main, draft):
        assert s.max_len == 131072 and len(s.segments[0]) == 4
        assert s.segments[0].sum() == 131072 and s.segments[0].min() >= 1
    assert not np.array_equal(main.segments[0], draft.segments[0])
    bat = W.make_spec("batched")[0]
    assert bat.n_seqs == 64 and bat.lengths.min() >= 1024 and bat.lengths.max() <= 32768
    assert len(np.unique(bat.lengths)) > 50 and bat.v_type == W.V_Q8_0
    ver = W.make_spec("verify")[0]
    assert (ver.n_seqs, ver.t_q, ver.causal, ver.group * ver.t_q) == (16, 4, True, 32)
    # algorithmic bytes of the long-context step: (8 + 4) heads * 131072 * 208 B
    assert W.step_kv_bytes([main, draft]) == 327155712


def test_generator_deterministic_and_sliceable():
    spec = W.make_spec("single", ctx=9000)[0]
    k1, v1 = W.gen_kv(spec, 0)
    k2, v2 = W.gen_kv(spec, 0, 4000, 8500)
    assert np.array_equal(k1[4000:8500], k2) and np.array_equal(v1[4000:8500], v2)
    och = W.outlier_channels(spec)
    assert och.shape == (8, 4)
    for h in range(8):
        big = np.abs(k1[:, h].astype(np.float32)).mean(0)
        assert set(np.argsort(big)[-4:]) == set(och[h].tolist())
    q = W.gen_q(spec)
    assert q.shape == (1, 1, 32, 128) and q.dtype == np.float16
    assert np.array_equal(q, W.gen_q(W.make_spec("single", ctx=9000)[0]))
