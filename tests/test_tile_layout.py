"""The in-tile order of the cache's code bytes (include/kvq.h, "Tiles"): the
library's untile helper, written from the header's offset formulas, must agree
with the lane-by-lane view of what the attention kernel reads (tests/kvq_cases),
and both must be permutations of a tile."""
import numpy as np
import pytest

from quantized_kv_cache_03_gb300 import kvq
from kvq_cases import lane_view_index, logical_codes

CASES = [("kq", kvq.V_Q4_0, 128), ("vq", kvq.V_Q4_0, 64), ("vq", kvq.V_Q8_0, 128),
         ("k16", kvq.V_Q4_0, 128)]   # F16 K: 128 two-byte elements per row


@pytest.mark.parametrize("name,vt,row", CASES)
def test_lane_view_is_a_permutation(name, vt, row):
    idx = lane_view_index(name, vt)
    assert len(idx) == 16 * row
    assert sorted(idx[:, 0]) == list(range(16 * row))
    assert len({(u, j) for _, u, j in idx}) == 16 * row
    assert idx[:, 1].min() == 0 and idx[:, 1].max() == 15 and idx[:, 2].max() == row - 1


@pytest.mark.parametrize("name,vt,row", CASES)
def test_header_formula_matches_lane_view(name, vt, row):
    rng = np.random.default_rng(7)
    dt = np.uint16 if name == "k16" else np.uint8
    stored = rng.integers(0, np.iinfo(dt).max + 1, size=(3, 64, row), dtype=dt)
    assert np.array_equal(kvq.untile_codes(stored, name, vt), logical_codes(stored, name, vt))


def test_f16_k_fragment_words():
    # F16 K: the 16-byte word of k16 step ks for lane (g, c) holds (u, j) =
    # (g, 16ks+2c), (g, 16ks+2c+1), (g+8, ...), (g+8, ...), (g, 16ks+2c+8), ...
    idx = {int(o): (int(u), int(j)) for o, u, j in lane_view_index("k16", kvq.V_Q4_0)}
    ks, g, c = 5, 6, 1
    base = ks * 256 + (4 * g + c) * 8
    k0 = 16 * ks + 2 * c
    assert [idx[base + k] for k in range(8)] == [(g, k0), (g, k0 + 1), (g + 8, k0), (g + 8, k0 + 1),
                                                 (g, k0 + 8), (g, k0 + 9), (g + 8, k0 + 8), (g + 8, k0 + 9)]


def test_q4_0_word_pairs_positions():
    # word bb of lane (g, c)'s q4_0 load: bytes (2g, 2g+1) of token t then of t+1
    idx = {(int(o)): (int(u), int(j)) for o, u, j in lane_view_index("vq", kvq.V_Q4_0)}
    g, c, bb = 3, 2, 1
    lane = 4 * g + c
    base = 0 * 512 + lane * 16 + 4 * bb
    t = 2 * c
    assert [idx[base + k] for k in range(4)] == [(t, 16 * bb + 2 * g), (t, 16 * bb + 2 * g + 1),
                                                 (t + 1, 16 * bb + 2 * g), (t + 1, 16 * bb + 2 * g + 1)]
