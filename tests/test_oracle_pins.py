"""The oracle against facts fixed by the pages and by mathematics (CPU only)."""
import pytest

import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(oracle_lib, pin):
    pin(oracle_lib)


def test_golden_fixtures_cite_a_page():
    import glob
    import json
    import os
    files = glob.glob(os.path.join(pins.GOLDEN, "*.json"))
    assert len(files) >= 4
    for f in files:
        with open(f) as fh:
            g = json.load(fh)
        assert g.get("source"), f"{f} has no citation"


def test_diagram_tiles_match_the_caption():
    # the ragged tail of the caption: 10 keys in tiles of 4 -> last tile holds
    # positions 8 and 9, and 10 and 11 fall past the history
    d = pins.golden("fused_kernel_diagram.json")
    S, T = d["history"], d["tile"]
    tiles = [list(range(t, min(t + T, S))) for t in range(0, S, T)]
    assert tiles == d["tiles"]
    last_tile_end = ((S + T - 1) // T) * T
    assert list(range(S, last_tile_end)) == d["masked_positions"]
