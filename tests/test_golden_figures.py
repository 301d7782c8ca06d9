"""Pins on the figures the pages print (tests/golden/page_figures.json)."""
import json
import os

import gen

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")))


def test_layer_schedule_matches_the_page():
    s = GOLDEN["layer_schedule"]
    assert tuple(s["full_layer_ids"]) == gen.EMBLA_FULL_LAYERS
    assert len(gen.EMBLA_WINDOW_LAYERS) == s["window_layers"]
    sparse = [l for ls in gen.EMBLA_SPARSE_OF.values() for l in ls]
    assert len(sparse) == s["sparse_layers"]
    assert len(gen.EMBLA_FULL_LAYERS) == s["full_layers"]
    every = sorted(list(gen.EMBLA_WINDOW_LAYERS) + list(gen.EMBLA_FULL_LAYERS) + sparse)
    assert every == list(range(s["layers"]))
    # second half: blocks of four, a full layer followed by its three sparse layers
    for f in range(s["blocks_of_four_from"], s["layers"], 4):
        assert f in gen.EMBLA_FULL_LAYERS and gen.EMBLA_SPARSE_OF[f] == (f + 1, f + 2, f + 3)
    assert gen.EMBLA_SPARSE_OF[7] == ()
    assert gen.HQ * gen.HEAD_DIM == s["width"]


def test_selection_and_window_sizes():
    assert GOLDEN["selection"]["topk"] == 1024 and GOLDEN["selection"]["recent"] == 128
    assert GOLDEN["window"]["keys"] == gen.WINDOW
