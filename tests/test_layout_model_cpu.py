"""The per-segment layout cost model (kvq_layout_cost / kvq_choose_layout)
on the host, pinned to the calibration record layout_model.json (decode times
measured on a GB300 for segments of n tokens in both layouts): the library's
default coefficients are the record's fit, its cost terms follow the byte and
unpack counts written out here from the layouts' definitions, the modelled
ranking matches the measured one at every calibration point, and the choice
for new segments follows from it (tiles at every length on this GPU; rows
where a model with cheaper unpacking makes the saved bytes worth it)."""
import json
import os

import pytest

from quantized_kv_cache_03_gb300 import build as B
from quantized_kv_cache_03_gb300 import kvq

RECORD = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "quantized_kv_cache_03_gb300",
                      "layout_model.json")


@pytest.fixture(scope="module")
def rec():
    B.build()
    kvq.load()
    with open(RECORD) as f:
        return json.load(f)


def _bytes(layout, v_type, n):
    code = 128 + (64 if v_type == kvq.V_Q4_0 else 128)    # K codes + V codes per row
    if layout == kvq.LAYOUT_TILES:
        return -(-n // 16) * 16 * (code + 16)             # whole 16-token tiles, scales included
    return n * code + (n + n % 2) * 16                    # exact rows, scale rows in pairs


def test_default_coefficients_are_the_recorded_fit(rec):
    m = kvq.layout_model_default()
    assert m.us_per_byte == pytest.approx(rec["us_per_byte"], rel=1e-12)
    assert m.us_per_op == pytest.approx(rec["us_per_op"], rel=1e-12)
    assert m.ops_rows_per_tile == pytest.approx(rec["ops_rows_per_tile"], rel=1e-12)


@pytest.mark.parametrize("v_type", [kvq.V_Q4_0, kvq.V_Q8_0])
@pytest.mark.parametrize("n", [1, 2, 7, 15, 16, 17, 31, 32, 100, 4097])
def test_cost_terms(v_type, n, rec):
    m = kvq.KvqLayoutModel(1.0, 0.0, 0.0)                 # bytes only
    assert kvq.layout_cost(kvq.LAYOUT_TILES, v_type, n, m) == _bytes(kvq.LAYOUT_TILES, v_type, n)
    assert kvq.layout_cost(kvq.LAYOUT_ROWS, v_type, n, m) == _bytes(kvq.LAYOUT_ROWS, v_type, n)
    m = kvq.KvqLayoutModel(0.0, 1.0, 134.0)               # unpack only
    assert kvq.layout_cost(kvq.LAYOUT_TILES, v_type, n, m) == 0.0
    assert kvq.layout_cost(kvq.LAYOUT_ROWS, v_type, n, m) == 134.0 * -(-n // 16)


def test_record_points_and_the_modelled_ranking(rec):
    """Each recorded point's bytes and unpack ops are the model's terms for
    its configuration (256 kv heads x 60 segments); the model ranks the two
    layouts as the measurement did at every segment length."""
    H, S, vt = rec["heads"], rec["segments"], rec["v_type"]
    pts = {(p["n"], p["layout"]): p for p in rec["points"]}
    for (n, lay), p in pts.items():
        assert p["bytes"] == H * S * _bytes(lay, vt, n)
        assert p["unpack_ops"] == pytest.approx(H * S * -(-n // 16) * (rec["ops_rows_per_tile"] if lay else 0.0))
    for n in sorted({n for n, _ in pts}):
        measured_rows_faster = pts[(n, kvq.LAYOUT_ROWS)]["us"] < pts[(n, kvq.LAYOUT_TILES)]["us"]
        model_rows_cheaper = kvq.layout_cost(kvq.LAYOUT_ROWS, vt, n) < kvq.layout_cost(kvq.LAYOUT_TILES, vt, n)
        assert measured_rows_faster == model_rows_cheaper, n
        assert kvq.choose_layout(kvq.K_I8, vt, n) == (kvq.LAYOUT_ROWS if model_rows_cheaper else kvq.LAYOUT_TILES)


def test_fit_reproduces_the_measured_times(rec):
    """The least-squares fit explains the recorded times within 20 % (the
    offset t0 is the layout-independent part the cost leaves out)."""
    for p in rec["points"]:
        model = rec["t0_us"] + rec["us_per_byte"] * p["bytes"] + rec["us_per_op"] * p["unpack_ops"]
        assert model == pytest.approx(p["us"], rel=0.2), p


def test_choice_follows_the_weights():
    # on the recorded GB300 weights the tiles win everywhere, for both V formats
    for vt in (kvq.V_Q4_0, kvq.V_Q8_0):
        assert {kvq.choose_layout(kvq.K_I8, vt, n) for n in range(1, 300)} == {kvq.LAYOUT_TILES}
    # a GPU where unpacking is cheap relative to bytes: short ragged segments go to rows
    cheap = kvq.KvqLayoutModel(1.0, 1.0, 10.0)
    assert kvq.choose_layout(kvq.K_I8, kvq.V_Q4_0, 1, cheap) == kvq.LAYOUT_ROWS
    assert kvq.choose_layout(kvq.K_I8, kvq.V_Q4_0, 16, cheap) == kvq.LAYOUT_TILES
    assert kvq.choose_layout(kvq.K_F16, kvq.V_Q4_0, 1, cheap) == kvq.LAYOUT_TILES   # rows: int8 K only
    with pytest.raises(kvq.KvqError):
        kvq.layout_cost(kvq.LAYOUT_ROWS, kvq.V_Q4_0, 0)
    with pytest.raises(kvq.KvqError):
        kvq.layout_cost(2, kvq.V_Q4_0, 5)
