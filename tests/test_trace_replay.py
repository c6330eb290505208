"""The dispatch model of the trace tool's --replay (host arithmetic only)."""

import numpy as np

from paged_kv_cache_217_gb300 import trace as T


def test_modelled_span_fills_slots_in_row_order():
    # 4 one-tile sequences of one CTA each through 2 slots, life 1 + 0 x tiles
    assert T.modelled_span([0, 1, 2, 3], np.ones(4, np.int64), 1, 2, 1.0, 0.0) == 2.0
    # a long sequence dispatched last ends last: 1 + 1 (wait for a slot) + 10
    tiles = np.array([1, 1, 1, 10])
    assert T.modelled_span([0, 1, 2, 3], tiles, 1, 2, 0.0, 1.0) == 11.0
    # dispatched first, it overlaps the short ones
    assert T.modelled_span([3, 0, 1, 2], tiles, 1, 2, 0.0, 1.0) == 10.0
    # every head of a row's sequence takes a slot
    assert T.modelled_span([0], np.array([3]), 4, 2, 0.0, 1.0) == 6.0


def test_replay_orders_and_buckets(capsys):
    # lengths with one long (>= 2x the mean tile count) and short (<= 5/8) ones
    lens = np.array([16 * 20, 16, 16, 16 * 4, 16 * 4, 16 * 4], np.int32)
    tiles = np.array([1, 2, 4, 8, 20])
    life = 2.0 + 0.5 * tiles
    T.replay(tiles, life, lens, 2, 3)
    out = capsys.readouterr().out
    assert "life = 2.00 + 0.500 x tiles" in out
    spans = {ln.split("modelled span")[0].strip(): float(ln.split("modelled span")[1].split("us")[0])
             for ln in out.splitlines() if "modelled span" in ln}
    assert set(spans) == {"natural", "long first", "long first, short last", "descending"}
    assert spans["long first"] <= spans["natural"]


def test_replay_and_order_test_use_the_library_thresholds():
    # the replay (and the GPU test of the ordering kernel) restate the bucket
    # rule; their thresholds must be the defaults compiled into the library
    import os
    import re
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    with open(os.path.join(root, "paged_kv_cache_217_gb300", "csrc", "decode.cuh")) as f:
        src = f.read()
    defaults = dict(re.findall(r"constexpr long long (kLongFirstX2|kShortLastX8) = (\d+);", src))
    assert int(defaults["kLongFirstX2"]) == T.LONG_FIRST_X2
    assert int(defaults["kShortLastX8"]) == T.SHORT_LAST_X8
    with open(os.path.join(root, "tests", "test_gpu_decode.py")) as f:
        gpu_test = f.read()
    assert f"2 * t[s] * S >= {T.LONG_FIRST_X2} * total" in gpu_test
    assert f"8 * t[s] * S <= {T.SHORT_LAST_X8} * total" in gpu_test
