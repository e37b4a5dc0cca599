"""The tensor-core schedule as include/smla.h states it (tests/smla_testlib.
tc_schedule, which the GPU tests check the kernels' partials against):
coverage of every tile by exactly one CTA, the partial-slot rule, and the
tile counts per CTA that the half-tile slots of the native-fp8 kernel give."""

import numpy as np
import pytest

from smla_testlib import tc_schedule


def per_cta_tiles(parts, G, tile):
    n = np.zeros(G, dtype=np.int64)
    for pl in parts.values():
        for c, _, lo, hi in pl:
            n[c] += -(-(hi - lo) // tile) if hi > lo else 1  # (an empty row's tile still counts)
    return n


@pytest.mark.parametrize("start,per_tile", [(2, 1), (1, 2), (3, 2), (0, 2), (2, 4)])
def test_every_tile_belongs_to_exactly_one_cta(start, per_tile):
    rng = np.random.default_rng(start * 10 + per_tile)
    for _ in range(200):
        tile = int(rng.choice([64, 128]))
        lens = [int(x) for x in rng.choice([0, 1, 63, 64, 65, 500, 2048, 4097], size=int(rng.integers(1, 12)))]
        G = int(rng.integers(1, 40))
        parts = tc_schedule(lens, G, tile=tile, start_slots=start, tile_slots=per_tile)
        for r, L in enumerate(lens):
            spans = sorted((lo, hi) for _, _, lo, hi in parts[r])
            # the parts tile the row's positions in order, without gaps or overlaps
            assert spans[0][0] == 0 and spans[-1][1] == L
            for (lo0, hi0), (lo1, _) in zip(spans, spans[1:]):
                assert hi0 == lo1 and lo1 % tile == 0
            ctas = [c for c, _, _, _ in parts[r]]
            assert ctas == sorted(ctas) and len(set(ctas)) == len(ctas)
            # partial slot 2 c + 1 for the part that begins the row (its first
            # tile lies in CTA c's range), 2 c for a part that continues it
            for k, (c, slot, _, _) in enumerate(parts[r]):
                assert slot == 2 * c + (1 if k == 0 else 0)


def test_half_tile_slots_balance_decode_64x16():
    """decode_64x16_k2048 over 152 CTAs: with two slots per 128-key tile and one
    per row start (the native-fp8 kernel) every CTA holds 6 or 7 tiles; with
    one slot per tile and two per row start it held 5 to 8."""
    lens = [2048] * 64
    fp8 = per_cta_tiles(tc_schedule(lens, 152, tile=128, start_slots=1, tile_slots=2), 152, 128)
    assert fp8.sum() == 64 * 16 and fp8.min() == 6 and fp8.max() == 7
    whole = per_cta_tiles(tc_schedule(lens, 152, tile=128, start_slots=2, tile_slots=1), 152, 128)
    assert whole.sum() == 64 * 16 and whole.min() == 5 and whole.max() == 8
